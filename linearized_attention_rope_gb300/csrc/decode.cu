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
// One decode step.  CTA (q-head h, sequence n), 256 threads.
//  1. RoPE q, k of the new token p; short conv of q with the q conv cache,
//     L2 norm -> qhat.  The first q-head of the kv group also convolves k, v,
//     writes the new token into the KV ring and the pending ring, and shifts
//     the k/v conv caches; no other CTA reads those slots in this step.
//  2. If token j = p - W is not a sink it leaves the window now: the 128x128
//     state is streamed through registers once, giving x = khat_j^T S and
//     y = qhat_p^T S; then S <- alpha S + khat_j u^T with u = beta (vhat_j -
//     alpha x), and o_lin = alpha y + (qhat_p . khat_j) u.
//  3. Softmax over the ring (sinks + window) and the new token; combine.
constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) t += red[w];
    return t;
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kDecThreads)
decode_step_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                   const Tin* __restrict__ v, const float* __restrict__ g,
                   const float* __restrict__ beta, const float* __restrict__ lambda,
                   const float* __restrict__ wq, const float* __restrict__ wk,
                   const float* __restrict__ wv, hla_state s, Tin* __restrict__ out) {
    constexpr int E = D / 32;
    constexpr int CG = D / 4;               // float4 column groups of S
    constexpr int RG = kDecThreads / CG;    // row groups
    constexpr int RPT = D / RG;             // rows of S per thread
    __shared__ __align__(16) float qrot_s[D], qhat_s[D], krot_s[D], vraw_s[D];
    __shared__ __align__(16) float kj_s[D], vj_s[D], olin_s[D];
    __shared__ __align__(16) float redx[RG][D], redy[RG][D];
    __shared__ float acc_w[kDecWarps][D], m_w[kDecWarps], l_w[kDecWarps], red[kDecWarps];

    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G, tid = threadIdx.x;
    const bool leader = (h % L.G) == 0;
    const int ns = L.n_sinks, W = L.window, R = ns + W, P = W + 1;
    const int64_t p = s.pos[n];
    Tin* kring = static_cast<Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    Tin* vring = static_cast<Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;

    // ---- 1. features of the new token
    float qt = 0.f, kt = 0.f, vt = 0.f;
    if (tid < D) {
        const int c = tid;
        const size_t qrow = ((size_t)n * L.Hq + h) * D, krow = ((size_t)n * L.Hkv + kv) * D;
        const float qr = rope_channel(q + qrow, c, D, p, L);
        const float kr = rope_channel(k + krow, c, D, p, L);
        const float vr = to_f32(v[krow + c]);
        qrot_s[c] = qr;
        krot_s[c] = kr;
        vraw_s[c] = vr;
        float* cq = s.conv_q + ((size_t)n * kConvHalo * L.Hq + h) * D + c;
        const size_t cq_step = (size_t)L.Hq * D;
        const float* w = wq + ((size_t)h * D + c) * kConvWidth;
        float hist[kConvHalo];
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) hist[m] = cq[m * cq_step];
        qt = w[kConvHalo] * qr;
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) qt = fmaf(w[m], hist[m], qt);
#pragma unroll
        for (int m = 0; m + 1 < kConvHalo; ++m) cq[m * cq_step] = hist[m + 1];
        cq[(kConvHalo - 1) * cq_step] = qr;
        if (leader) {
            float* ck = s.conv_k + ((size_t)n * kConvHalo * L.Hkv + kv) * D + c;
            float* cv = s.conv_v + ((size_t)n * kConvHalo * L.Hkv + kv) * D + c;
            const size_t ck_step = (size_t)L.Hkv * D;
            const float* w_k = wk + ((size_t)kv * D + c) * kConvWidth;
            const float* w_v = wv + ((size_t)kv * D + c) * kConvWidth;
            float hk[kConvHalo], hv[kConvHalo];
#pragma unroll
            for (int m = 0; m < kConvHalo; ++m) { hk[m] = ck[m * ck_step]; hv[m] = cv[m * ck_step]; }
            kt = w_k[kConvHalo] * kr;
            vt = w_v[kConvHalo] * vr;
#pragma unroll
            for (int m = 0; m < kConvHalo; ++m) { kt = fmaf(w_k[m], hk[m], kt); vt = fmaf(w_v[m], hv[m], vt); }
#pragma unroll
            for (int m = 0; m + 1 < kConvHalo; ++m) { ck[m * ck_step] = hk[m + 1]; cv[m * ck_step] = hv[m + 1]; }
            ck[(kConvHalo - 1) * ck_step] = kr;
            cv[(kConvHalo - 1) * ck_step] = vr;
        }
    }
    float qss = block_sum(qt * qt, red);
    if (tid < D) qhat_s[tid] = (L.flags & HLA_FLAG_L2NORM_Q) ? qt * rsqrtf(qss + 1e-6f) : qt;
    if (leader) {
        float kss = block_sum(kt * kt, red);
        if (tid < D) {
            const size_t slot = (size_t)ring_slot(p, ns, W) * D + tid;
            kring[slot] = from_f32<Tin>(krot_s[tid]);
            vring[slot] = from_f32<Tin>(vraw_s[tid]);
            const size_t ps = (((size_t)n * L.Hkv + kv) * P + (size_t)(p % P)) * D + tid;
            s.pend_k[ps] = kt * rsqrtf(kss + 1e-6f);
            s.pend_v[ps] = vt;
        }
    }
    const size_t gslot = ((size_t)n * L.Hq + h) * P;

    // ---- 2. absorb the token leaving the window; linear read-out
    const int64_t j = p - W;
    if (j >= ns) {
        const size_t js = (size_t)(j % P);
        const float alpha = expf(s.pend_g[gslot + js]);
        const float b = s.pend_beta[gslot + js];
        if (tid < D) {
            const size_t ps = (((size_t)n * L.Hkv + kv) * P + js) * D + tid;
            kj_s[tid] = s.pend_k[ps];
            vj_s[tid] = s.pend_v[ps];
        }
        __syncthreads();
        const float cdot = block_sum(tid < D ? qhat_s[tid] * kj_s[tid] : 0.f, red);
        const int cg = tid % CG, rg = tid / CG;
        float4* S4 = reinterpret_cast<float4*>(s.S + ((size_t)n * L.Hq + h) * D * D);
        float4 Sr[RPT];
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
        for (int r = 0; r < RPT; ++r) Sr[r] = S4[(size_t)(rg * RPT + r) * CG + cg];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const float kk = kj_s[rg * RPT + r], qq = qhat_s[rg * RPT + r];
            x.x = fmaf(kk, Sr[r].x, x.x); x.y = fmaf(kk, Sr[r].y, x.y);
            x.z = fmaf(kk, Sr[r].z, x.z); x.w = fmaf(kk, Sr[r].w, x.w);
            y.x = fmaf(qq, Sr[r].x, y.x); y.y = fmaf(qq, Sr[r].y, y.y);
            y.z = fmaf(qq, Sr[r].z, y.z); y.w = fmaf(qq, Sr[r].w, y.w);
        }
        reinterpret_cast<float4*>(redx[rg])[cg] = x;
        reinterpret_cast<float4*>(redy[rg])[cg] = y;
        __syncthreads();
        float u[4], ol[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = 4 * cg + e;
            float xs = 0.f, ys = 0.f;
#pragma unroll
            for (int r = 0; r < RG; ++r) { xs += redx[r][col]; ys += redy[r][col]; }
            u[e] = b * (vj_s[col] - alpha * xs);
            ol[e] = fmaf(alpha, ys, cdot * u[e]);
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
        if (rg == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) olin_s[4 * cg + e] = ol[e];
        }
    } else if (tid < D) {
        olin_s[tid] = 0.f;  // nothing absorbed yet: the state is still empty
    }
    if (tid == 0) {
        s.pend_g[gslot + (size_t)(p % P)] = g[(size_t)n * L.Hq + h];
        s.pend_beta[gslot + (size_t)(p % P)] = beta[(size_t)n * L.Hq + h];
    }
    __syncthreads();

    // ---- 3. softmax over sinks + window (ring) and the new token
    const int lane = tid & 31, warp = tid >> 5, c0 = lane * E;
    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
    float qv[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) { qv[e] = qrot_s[c0 + e] * qscale; acc[e] = 0.f; }
    float m = -INFINITY, l = 0.f;
    if (warp == 0) {  // the new token itself
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(qv[e], krot_s[c0 + e], part);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        m = part;
        l = 1.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = vraw_s[c0 + e];
    }
    const int64_t n_sink_keys = p < ns ? p : ns;  // sinks strictly before p
    const int64_t w_lo = (p - W + 1) > ns ? (p - W + 1) : ns;
    const int64_t n_win = p - w_lo > 0 ? p - w_lo : 0;  // window keys strictly before p
    const int64_t n_keys = n_sink_keys + n_win;
    for (int64_t i0 = (int64_t)warp * 4; i0 < n_keys; i0 += kDecWarps * 4) {
        float sc[4];
        int64_t sl[4];
#pragma unroll
        for (int u2 = 0; u2 < 4; ++u2) {
            const int64_t i = i0 + u2;
            const int64_t jj = i < n_sink_keys ? i : w_lo + (i - n_sink_keys);
            sl[u2] = ring_slot(jj, ns, W);
            float part = 0.f;
            if (i < n_keys) {
                float kx[E];
                load_vec<E>(kring + (size_t)sl[u2] * D + c0, kx);
#pragma unroll
                for (int e = 0; e < E; ++e) part = fmaf(qv[e], kx[e], part);
            }
            sc[u2] = part;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) sc[u2] += __shfl_xor_sync(0xffffffffu, sc[u2], o);
        }
        float mx = m;
#pragma unroll
        for (int u2 = 0; u2 < 4; ++u2) {
            if (i0 + u2 >= n_keys) sc[u2] = -INFINITY;
            mx = fmaxf(mx, sc[u2]);
        }
        const float corr = exp2f(m - mx);
        l *= corr;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
        for (int u2 = 0; u2 < 4; ++u2) {
            if (i0 + u2 < n_keys) {
                const float pu = exp2f(sc[u2] - mx);
                l += pu;
                float vx[E];
                load_vec<E>(vring + (size_t)sl[u2] * D + c0, vx);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(pu, vx[e], acc[e]);
            }
        }
        m = mx;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) acc_w[warp][c0 + e] = acc[e];
    if (lane == 0) { m_w[warp] = m; l_w[warp] = l; }
    __syncthreads();
    if (tid < D) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, m_w[w]);
        float Ls = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float f = exp2f(m_w[w] - M);  // 0 for warps that saw no key
            Ls = fmaf(l_w[w], f, Ls);
            A = fmaf(acc_w[w][tid], f, A);
        }
        float o = (L.flags & HLA_FLAG_SOFTMAX_OFF) ? 0.f : A / Ls;
        if (!(L.flags & HLA_FLAG_LINEAR_OFF)) o = fmaf(__ldg(lambda + h), olin_s[tid], o);
        out[((size_t)n * L.Hq + h) * D + tid] = from_f32<Tin>(o);
    }
}

__global__ void advance_pos_kernel(int64_t* pos, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) pos[i] += 1;
}

template <typename Tin>
cudaError_t launch_decode_step(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                               const float* g, const float* beta, const float* lambda,
                               const float* wq, const float* wk, const float* wv,
                               const hla_state& s, Tin* out, cudaStream_t st) {
    dim3 grid(L.Hq, L.n_seqs);
    if (L.d == 128)
        decode_step_kernel<Tin, 128><<<grid, kDecThreads, 0, st>>>(L, q, k, v, g, beta, lambda, wq, wk, wv, s, out);
    else
        decode_step_kernel<Tin, 64><<<grid, kDecThreads, 0, st>>>(L, q, k, v, g, beta, lambda, wq, wk, wv, s, out);
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
