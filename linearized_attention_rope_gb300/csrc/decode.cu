// Decode: one token per sequence per step, with the fixed-budget cache of
// "迈向线性的关键：分析驱动的 Transformer 线性化", section 填补近似缺口的实用设计
// (8 sinks + a sliding window keep exact attention; the GDN state absorbs the
// non-sink token that leaves the window, GDN equation of section
// 线性注意力替换机制).  The decode state is caller-owned (see hla.h); this
// file also writes it at the end of a prefill.
#include "hla_common.cuh"

namespace hla {

__device__ __forceinline__ int64_t ring_slot(int64_t p, int n_sinks, int window) {
    return p < n_sinks ? p : n_sinks + (p - n_sinks) % window;
}

// RoPE'd channel c of row x (d channels) at position p.
template <typename T>
__device__ __forceinline__ float rope_channel(const T* __restrict__ x, int c, int D, int64_t p,
                                              const LayerDims& L) {
    const int half = D / 2, i = c % half;
    float cs, sn;
    rope_cs_exact(p, L.theta[i], &cs, &sn);
    float x1 = to_f32(x[i]), x2 = to_f32(x[i + half]);
    return c < half ? x1 * cs - x2 * sn : x2 * cs + x1 * sn;
}

// ---------------------------------------------------------------------------
// Prefill -> decode state.  CTA (q-head h, sequence n); the first q-head of
// each kv group also writes that kv-head's ring, pending k/v and conv caches.
template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(128)
state_fill_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                  const Tin* __restrict__ v, const float* __restrict__ g,
                  const float* __restrict__ beta, const Tf* __restrict__ khat,
                  const Tf* __restrict__ vhat, const int32_t* __restrict__ cu, hla_state s) {
    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G;
    const bool leader = (h % L.G) == 0;
    const int ns = L.n_sinks, W = L.window, R = ns + W, P = W + 1;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t pend_lo = len - W > ns ? len - W : ns;  // tokens still waiting to be absorbed

    for (int idx = threadIdx.x; idx < kConvHalo * D; idx += blockDim.x) {
        int m = idx / D, c = idx % D;
        int64_t pp = len - kConvHalo + m;
        float val = 0.f;
        if (pp >= 0) val = rope_channel(q + ((size_t)(start + pp) * L.Hq + h) * D, c, D, pp, L);
        s.conv_q[(((size_t)n * kConvHalo + m) * L.Hq + h) * D + c] = val;
    }
    for (int64_t pp = pend_lo + threadIdx.x; pp < len; pp += blockDim.x) {
        size_t slot = ((size_t)n * L.Hq + h) * P + (size_t)(pp % P);
        s.pend_g[slot] = g[(size_t)(start + pp) * L.Hq + h];
        s.pend_beta[slot] = beta[(size_t)(start + pp) * L.Hq + h];
    }
    if (leader) {
        Tin* kring = static_cast<Tin*>(s.k_ring);
        Tin* vring = static_cast<Tin*>(s.v_ring);
        const int64_t n_sink_rows = len < ns ? len : ns;
        const int64_t n_win_rows = len - pend_lo > 0 ? len - pend_lo : 0;
        for (int64_t idx = threadIdx.x; idx < (n_sink_rows + n_win_rows) * D; idx += blockDim.x) {
            int64_t r = idx / D;
            int c = (int)(idx % D);
            int64_t pp = r < n_sink_rows ? r : pend_lo + (r - n_sink_rows);
            size_t row = (size_t)(start + pp) * L.Hkv + kv;
            size_t dst = (((size_t)n * L.Hkv + kv) * R + ring_slot(pp, ns, W)) * D + c;
            kring[dst] = from_f32<Tin>(rope_channel(k + row * D, c, D, pp, L));
            vring[dst] = v[row * D + c];
        }
        for (int64_t idx = threadIdx.x; idx < n_win_rows * D; idx += blockDim.x) {
            int64_t pp = pend_lo + idx / D;
            int c = (int)(idx % D);
            size_t row = (size_t)(start + pp) * L.Hkv + kv;
            size_t dst = (((size_t)n * L.Hkv + kv) * P + (size_t)(pp % P)) * D + c;
            s.pend_k[dst] = to_f32(khat[row * D + c]);
            s.pend_v[dst] = to_f32(vhat[row * D + c]);
        }
        for (int idx = threadIdx.x; idx < kConvHalo * D; idx += blockDim.x) {
            int m = idx / D, c = idx % D;
            int64_t pp = len - kConvHalo + m;
            float kval = 0.f, vval = 0.f;
            if (pp >= 0) {
                size_t row = (size_t)(start + pp) * L.Hkv + kv;
                kval = rope_channel(k + row * D, c, D, pp, L);
                vval = to_f32(v[row * D + c]);
            }
            size_t dst = (((size_t)n * kConvHalo + m) * L.Hkv + kv) * D + c;
            s.conv_k[dst] = kval;
            s.conv_v[dst] = vval;
        }
    }
    if (h == 0 && threadIdx.x == 0) s.pos[n] = len;
}

template <typename Tin, typename Tf>
cudaError_t launch_state_fill(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                              const float* g, const float* beta, const Tf* khat, const Tf* vhat,
                              const int32_t* cu, const hla_state& s, cudaStream_t st) {
    dim3 grid(L.Hq, L.n_seqs);
    if (L.d == 128)
        state_fill_kernel<Tin, Tf, 128><<<grid, 128, 0, st>>>(L, q, k, v, g, beta, khat, vhat, cu, s);
    else
        state_fill_kernel<Tin, Tf, 64><<<grid, 128, 0, st>>>(L, q, k, v, g, beta, khat, vhat, cu, s);
    return cudaGetLastError();
}

template cudaError_t launch_state_fill<float, float>(const LayerDims&, const float*, const float*,
                                                     const float*, const float*, const float*,
                                                     const float*, const float*, const int32_t*,
                                                     const hla_state&, cudaStream_t);
template cudaError_t launch_state_fill<__nv_bfloat16, __half>(
    const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, const float*,
    const float*, const __half*, const __half*, const int32_t*, const hla_state&, cudaStream_t);

// ---------------------------------------------------------------------------
// One decode step.  CTA (kv head, sequence n), 256 threads, owning the G
// query heads of the group, so the new token's key/value features, the ring
// and the pending ring are touched by one CTA only:
//  1. RoPE q, k of the new token p; short conv of q (G heads), k and v with
//     their histories; L2 norms -> qhat (G heads), khat.  The new token is
//     written into the KV ring (slot p, or n_sinks + (p - n_sinks) % W) and
//     into the pending ring (slot p % (W + 1)) with each head's g and beta.
//  2. If token j = p - W is not a sink it leaves the window now.  Per head,
//     the d x d state is read once into registers: x = khat_j^T S and
//     y = qhat_p^T S; then S <- alpha S + khat_j u^T with u = beta (vhat_j -
//     alpha x) is written back, and o_lin = alpha y + (qhat_p . khat_j) u.
//  3. Softmax over the ring (sinks + window, the new token included), in
//     tiles of up to kTile keys: logits of all G heads per key row (8 lanes
//     per row), per-head max and sum, then P V with the value rows read
//     coalesced; tiles are merged with a running max.
//  4. o = o_sm + lambda_h o_lin.
constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxG = 8;
constexpr int kTile = 1024;
constexpr int kUnrollK = 4;   // key rows in flight per lane (logits)
constexpr int kUnrollV = 8;   // value rows in flight per thread (P V)

template <typename Tin, int D>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_step_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                   const Tin* __restrict__ v, const float* __restrict__ g,
                   const float* __restrict__ beta, const float* __restrict__ lambda,
                   const float* __restrict__ wq, const float* __restrict__ wk,
                   const float* __restrict__ wv, hla_state s, Tin* __restrict__ out) {
    constexpr int HALF = D / 2;
    constexpr int CG = D / 4;              // float4 column groups of S
    constexpr int RG = kDecThreads / CG;   // row groups
    constexpr int RPT = D / RG;            // rows of S per thread
    constexpr int DL = D / 8;              // channels per lane in the 8-lane key groups
    constexpr int NKS = kDecThreads / CG;  // key subsets in P V
    extern __shared__ __align__(16) float dyn[];  // logits [G][kTile], later P V partials [NKS][G][D]
    __shared__ __align__(16) float qrot_s[kMaxG][D], qhat_s[kMaxG][D], olin_s[kMaxG][D];
    __shared__ __align__(16) float krot_s[D], vraw_s[D], khat_s[D], kj_s[D], vj_s[D];
    __shared__ __align__(16) float redx[RG][D], redy[RG][D];
    __shared__ float cs_s[HALF], sn_s[HALF];
    __shared__ float alpha_s[kMaxG], b_s[kMaxG], cdot_s[kMaxG], inv_s[kMaxG + 1];
    __shared__ float m_s[kMaxG], l_s[kMaxG], corr_s[kMaxG];

    const int kv = blockIdx.x, n = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = L.G, ns = L.n_sinks, W = L.window, R = ns + W, P = W + 1;
    const int64_t p = s.pos[n];
    Tin* kring = static_cast<Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    Tin* vring = static_cast<Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    const size_t kvrow = ((size_t)n * L.Hkv + kv) * D;

    // ---- 1. features of the new token
    if (tid < HALF) {
        float c, sn;
        rope_cs_exact(p, L.theta[tid], &c, &sn);
        cs_s[tid] = c;
        sn_s[tid] = sn;
    }
    __syncthreads();
    auto rot = [&](const Tin* x, int c) {
        const int i = c % HALF;
        const float x1 = to_f32(x[i]), x2 = to_f32(x[i + HALF]);
        return c < HALF ? x1 * cs_s[i] - x2 * sn_s[i] : x2 * cs_s[i] + x1 * sn_s[i];
    };
    if (tid < 2 * D) {  // k channels, then v channels
        const bool is_k = tid < D;
        const int c = is_k ? tid : tid - D;
        const float xr = is_k ? rot(k + kvrow, c) : to_f32(v[kvrow + c]);
        float* hist = (is_k ? s.conv_k : s.conv_v) + ((size_t)n * kConvHalo * L.Hkv + kv) * D + c;
        const size_t step = (size_t)L.Hkv * D;
        const float* w = (is_k ? wk : wv) + ((size_t)kv * D + c) * kConvWidth;
        float hst[kConvHalo];
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) hst[m] = hist[m * step];
        float acc = w[kConvHalo] * xr;
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) acc = fmaf(w[m], hst[m], acc);
#pragma unroll
        for (int m = 0; m + 1 < kConvHalo; ++m) hist[m * step] = hst[m + 1];
        hist[(kConvHalo - 1) * step] = xr;
        if (is_k) { krot_s[c] = xr; khat_s[c] = acc; }
        else { vraw_s[c] = xr; vj_s[c] = acc; }  // vj_s holds vhat_p until phase 2
    }
    for (int e = tid; e < G * D; e += kDecThreads) {
        const int gg = e / D, c = e % D, h = kv * G + gg;
        const float xr = rot(q + ((size_t)n * L.Hq + h) * D, c);
        float* hist = s.conv_q + ((size_t)n * kConvHalo * L.Hq + h) * D + c;
        const size_t step = (size_t)L.Hq * D;
        const float* w = wq + ((size_t)h * D + c) * kConvWidth;
        float hst[kConvHalo];
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) hst[m] = hist[m * step];
        float acc = w[kConvHalo] * xr;
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) acc = fmaf(w[m], hst[m], acc);
#pragma unroll
        for (int m = 0; m + 1 < kConvHalo; ++m) hist[m * step] = hst[m + 1];
        hist[(kConvHalo - 1) * step] = xr;
        qrot_s[gg][c] = xr;
        qhat_s[gg][c] = acc;
    }
    __syncthreads();
    // L2 norms: job gg < G is q-head gg, job G is the key
    for (int job = warp; job <= G; job += kDecWarps) {
        const float* x = job < G ? qhat_s[job] : khat_s;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) inv_s[job] = (job == G || (L.flags & HLA_FLAG_L2NORM_Q)) ? rsqrtf(ss + 1e-6f) : 1.f;
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += kDecThreads) qhat_s[e / D][e % D] *= inv_s[e / D];
    const size_t pslot = (size_t)(p % P);
    if (tid < D) {
        const float kh = khat_s[tid] * inv_s[G];
        const size_t slot = (size_t)ring_slot(p, ns, W) * D + tid;
        kring[slot] = from_f32<Tin>(krot_s[tid]);
        vring[slot] = from_f32<Tin>(vraw_s[tid]);
        const size_t ps = (((size_t)n * L.Hkv + kv) * P + pslot) * D + tid;
        s.pend_k[ps] = kh;
        s.pend_v[ps] = vj_s[tid];
    }
    const int64_t j = p - W;  // the token leaving the window
    const bool absorb = j >= ns;
    const size_t jslot = absorb ? (size_t)(j % P) : 0;
    if (tid < G) {
        const size_t gs = ((size_t)n * L.Hq + kv * G + tid) * P;
        if (absorb) {
            alpha_s[tid] = expf(s.pend_g[gs + jslot]);
            b_s[tid] = s.pend_beta[gs + jslot];
        }
        s.pend_g[gs + pslot] = g[(size_t)n * L.Hq + kv * G + tid];
        s.pend_beta[gs + pslot] = beta[(size_t)n * L.Hq + kv * G + tid];
    }
    __syncthreads();  // ring slot p, pending slot p written; vj_s free

    // ---- 2. absorb token j and read the state out, one head at a time
    if (absorb) {
        if (tid < D) {
            const size_t ps = (((size_t)n * L.Hkv + kv) * P + jslot) * D + tid;
            kj_s[tid] = s.pend_k[ps];
            vj_s[tid] = s.pend_v[ps];
        }
        __syncthreads();
        for (int job = warp; job < G; job += kDecWarps) {
            float d = 0.f;
            for (int c = lane; c < D; c += 32) d += qhat_s[job][c] * kj_s[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) cdot_s[job] = d;
        }
        const int cg = tid % CG, rg = tid / CG;
        for (int gg = 0; gg < G; ++gg) {
            float4* S4 = reinterpret_cast<float4*>(s.S + ((size_t)n * L.Hq + kv * G + gg) * D * D);
            float4 Sr[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) Sr[r] = S4[(size_t)(rg * RPT + r) * CG + cg];
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float kk = kj_s[rg * RPT + r], qq = qhat_s[gg][rg * RPT + r];
                x.x = fmaf(kk, Sr[r].x, x.x); x.y = fmaf(kk, Sr[r].y, x.y);
                x.z = fmaf(kk, Sr[r].z, x.z); x.w = fmaf(kk, Sr[r].w, x.w);
                y.x = fmaf(qq, Sr[r].x, y.x); y.y = fmaf(qq, Sr[r].y, y.y);
                y.z = fmaf(qq, Sr[r].z, y.z); y.w = fmaf(qq, Sr[r].w, y.w);
            }
            reinterpret_cast<float4*>(redx[rg])[cg] = x;
            reinterpret_cast<float4*>(redy[rg])[cg] = y;
            __syncthreads();
            const float alpha = alpha_s[gg], b = b_s[gg], cdot = cdot_s[gg];
            float u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = 4 * cg + e;
                float xs = 0.f, ys = 0.f;
#pragma unroll
                for (int r = 0; r < RG; ++r) { xs += redx[r][col]; ys += redy[r][col]; }
                u[e] = b * (vj_s[col] - alpha * xs);
                if (rg == 0) olin_s[gg][col] = fmaf(alpha, ys, cdot * u[e]);
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float kk = kj_s[rg * RPT + r];
                float4 o;
                o.x = fmaf(alpha, Sr[r].x, kk * u[0]);
                o.y = fmaf(alpha, Sr[r].y, kk * u[1]);
                o.z = fmaf(alpha, Sr[r].z, kk * u[2]);
                o.w = fmaf(alpha, Sr[r].w, kk * u[3]);
                S4[(size_t)(rg * RPT + r) * CG + cg] = o;
            }
            __syncthreads();  // redx/redy reused by the next head
        }
    } else {
        // nothing has been absorbed yet: the state is still empty
        for (int e = tid; e < G * D; e += kDecThreads) olin_s[e / D][e % D] = 0.f;
    }

    // ---- 3. softmax over the ring: sinks j < min(ns, p + 1), window [w_lo, p]
    const int64_t nsk = p + 1 < ns ? p + 1 : ns;
    const int64_t w_lo = (p - W + 1) > ns ? (p - W + 1) : ns;
    const int64_t n_win = p >= w_lo ? p - w_lo + 1 : 0;
    const int64_t n_keys = nsk + n_win;
    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
    float* logit = dyn;  // [G][kTile]
    const int l8 = tid & 7, grp8 = tid >> 3;
    const int cg4 = tid % CG, ks = tid / CG;
    float acc[kMaxG][4];
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[gg][e] = 0.f;
    if (tid < G) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }
    for (int64_t t0 = 0; t0 < n_keys; t0 += kTile) {
        const int nt = (int)min((int64_t)kTile, n_keys - t0);
        __syncthreads();  // logits of the previous tile consumed
        // logits: 8 lanes per key row, DL channels per lane, kUnrollK rows in
        // flight per lane.  The trip count is the same for the whole warp (the
        // shuffles run with every lane present); tail rows are predicated.
        for (int i0 = 0; i0 < nt; i0 += (kDecThreads / 8) * kUnrollK) {
            float kx[kUnrollK][DL];
#pragma unroll
            for (int u = 0; u < kUnrollK; ++u) {
                const int i = i0 + grp8 + (kDecThreads / 8) * u;
                if (i < nt) {
                    const int64_t ii = t0 + i;
                    const int64_t jj = ii < nsk ? ii : w_lo + (ii - nsk);
                    const Tin* kr = kring + (size_t)ring_slot(jj, ns, W) * D + DL * l8;
#pragma unroll
                    for (int e = 0; e < DL; e += 4) load_vec<4>(kr + e, kx[u] + e);
                } else {
#pragma unroll
                    for (int e = 0; e < DL; ++e) kx[u][e] = 0.f;
                }
            }
            for (int gg = 0; gg < G; ++gg) {
                float part[kUnrollK];
#pragma unroll
                for (int u = 0; u < kUnrollK; ++u) {
                    part[u] = 0.f;
#pragma unroll
                    for (int e = 0; e < DL; ++e) part[u] = fmaf(qrot_s[gg][DL * l8 + e], kx[u][e], part[u]);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1)
#pragma unroll
                    for (int u = 0; u < kUnrollK; ++u) part[u] += __shfl_xor_sync(0xffffffffu, part[u], o);
#pragma unroll
                for (int u = 0; u < kUnrollK; ++u) {
                    const int i = i0 + grp8 + (kDecThreads / 8) * u;
                    if (i < nt && l8 == 0) logit[gg * kTile + i] = part[u] * qscale;
                }
            }
        }
        __syncthreads();
        // per-head running max and sum; logits -> probabilities
        for (int gg = warp; gg < G; gg += kDecWarps) {
            float mx = -INFINITY;
            for (int i = lane; i < nt; i += 32) mx = fmaxf(mx, logit[gg * kTile + i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = m_s[gg], m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int i = lane; i < nt; i += 32) {
                const float e = exp2f(logit[gg * kTile + i] - m_new);
                logit[gg * kTile + i] = e;
                sum += e;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) {
                const float corr = exp2f(m_old - m_new);  // 0 on the first tile
                corr_s[gg] = corr;
                l_s[gg] = l_s[gg] * corr + sum;
                m_s[gg] = m_new;
            }
        }
        __syncthreads();
        // P V: thread (key subset ks, 4 channels cg4), value rows read coalesced
#pragma unroll
        for (int gg = 0; gg < kMaxG; ++gg)
            if (gg < G) {
                const float c = corr_s[gg];
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[gg][e] *= c;
            }
        for (int i0 = ks; i0 < nt; i0 += NKS * kUnrollV) {
            float vx[kUnrollV][4];
#pragma unroll
            for (int u = 0; u < kUnrollV; ++u) {
                const int i = i0 + NKS * u;
                if (i < nt) {
                    const int64_t ii = t0 + i;
                    const int64_t jj = ii < nsk ? ii : w_lo + (ii - nsk);
                    load_vec<4>(vring + (size_t)ring_slot(jj, ns, W) * D + 4 * cg4, vx[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) vx[u][e] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnrollV; ++u) {
                const int i = min(i0 + NKS * u, nt - 1);  // rows past the tail carry zero values
#pragma unroll
                for (int gg = 0; gg < kMaxG; ++gg)
                    if (gg < G) {
                        const float pr = logit[gg * kTile + i];
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[gg][e] = fmaf(pr, vx[u][e], acc[gg][e]);
                    }
            }
        }
    }
    __syncthreads();
    float* part = dyn;  // [NKS][G][D]
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg)
        if (gg < G)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[((size_t)ks * G + gg) * D + 4 * cg4 + e] = acc[gg][e];
    __syncthreads();

    // ---- 4. combine
    for (int e = tid; e < G * D; e += kDecThreads) {
        const int gg = e / D, c = e % D, h = kv * G + gg;
        float o = 0.f;
        for (int r = 0; r < NKS; ++r) o += part[((size_t)r * G + gg) * D + c];
        o = (L.flags & HLA_FLAG_SOFTMAX_OFF) ? 0.f : o / l_s[gg];
        if (!(L.flags & HLA_FLAG_LINEAR_OFF)) o = fmaf(__ldg(lambda + h), olin_s[gg][c], o);
        out[((size_t)n * L.Hq + h) * D + c] = from_f32<Tin>(o);
    }
}

__global__ void advance_pos_kernel(int64_t* pos, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) pos[i] += 1;
}

template <int D>
constexpr size_t decode_dyn_smem() {
    return sizeof(float) * (size_t)(kMaxG * kTile > (kDecThreads / (D / 4)) * kMaxG * D
                                         ? kMaxG * kTile
                                         : (kDecThreads / (D / 4)) * kMaxG * D);
}

template <typename Tin>
cudaError_t launch_decode_step(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                               const float* g, const float* beta, const float* lambda,
                               const float* wq, const float* wk, const float* wv,
                               const hla_state& s, Tin* out, cudaStream_t st) {
    if (L.G > kMaxG) return cudaErrorInvalidValue;
    dim3 grid(L.Hkv, L.n_seqs);
    if (L.d == 128) {
        constexpr size_t dyn = decode_dyn_smem<128>();
        cudaFuncSetAttribute(decode_step_kernel<Tin, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        decode_step_kernel<Tin, 128><<<grid, kDecThreads, dyn, st>>>(L, q, k, v, g, beta, lambda, wq, wk, wv, s, out);
    } else {
        constexpr size_t dyn = decode_dyn_smem<64>();
        cudaFuncSetAttribute(decode_step_kernel<Tin, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        decode_step_kernel<Tin, 64><<<grid, kDecThreads, dyn, st>>>(L, q, k, v, g, beta, lambda, wq, wk, wv, s, out);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    advance_pos_kernel<<<(L.n_seqs + 255) / 256, 256, 0, st>>>(s.pos, L.n_seqs);
    return cudaGetLastError();
}

template cudaError_t launch_decode_step<float>(const LayerDims&, const float*, const float*,
                                               const float*, const float*, const float*,
                                               const float*, const float*, const float*,
                                               const float*, const hla_state&, float*, cudaStream_t);
template cudaError_t launch_decode_step<__nv_bfloat16>(
    const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, const float*,
    const float*, const float*, const float*, const float*, const float*, const hla_state&,
    __nv_bfloat16*, cudaStream_t);

}  // namespace hla
