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
// One decode step, in three launches over per-step scratch (hla_state.scratch):
//  1. features (CTA per kv head and sequence): RoPE q, k of the new token p;
//     short conv of q (the G heads of the group), k and v with their
//     histories; L2 norms.  The new token goes into the KV ring (slot p, or
//     n_sinks + (p - n_sinks) % W) and the pending ring (slot p % (W + 1))
//     with each head's g and beta; RoPE'd q and qhat go to scratch.
//  2. state (CTA per q-head, half of the value columns and sequence): if token
//     j = p - W is not a sink it leaves the window now: the half's 32 KiB of
//     the state are read once into registers, x = khat_j^T S and
//     y = qhat_p^T S (the half's columns) are reduced across the CTA, and
//     S <- alpha S + khat_j u^T with u = beta (vhat_j - alpha x) is written
//     back; o_lin = alpha y + (qhat_p . khat_j) u.  Otherwise o_lin = 0.
//  3. softmax (CTA per kv head, key split and sequence): the ring's valid slots
//     are [0, min(n_sinks, p + 1)) and [n_sinks, n_sinks + n_window) (the
//     window fills its slots in order, then stays full), so a split is a
//     plain range of slots; per head of the group a running max, sum and P V
//     over its keys go to scratch.
//  4. combine (CTA per q-head and sequence): splits merged by their maxima,
//     o = o_sm + lambda_h o_lin; then pos += 1.
// Steps 2 and 3 stream the state and the ring, the step's bulk traffic; they
// run as one launch whose CTAs are state units and softmax splits in turn, so
// both streams share every wave.
constexpr int kMaxG = kMaxDecodeGroup;
constexpr int kFeatThreads = 256;
constexpr int kStateThreads = 128;
constexpr int kSmThreads = 128;
constexpr int kSplitKeys = 64;    // key slots per softmax split (at most)

// Per-step scratch layout (floats): qrot, qhat, olin [N, Hq, D]; pm, pl [N, Hq, splits];
// pacc [N, Hq, splits, D].
struct DecScratch {
    float *qrot, *qhat, *olin, *pm, *pl, *pacc;
    int splits;
};
__host__ __device__ inline int decode_splits(int n_sinks, int window) {
    return (n_sinks + window + kSplitKeys - 1) / kSplitKeys;
}
inline DecScratch dec_scratch(float* base, int n_seqs, int Hq, int D, int splits) {
    DecScratch d;
    const size_t nh = (size_t)n_seqs * Hq;
    d.qrot = base;
    d.qhat = d.qrot + nh * D;
    d.olin = d.qhat + nh * D;
    d.pm = d.olin + nh * D;
    d.pl = d.pm + nh * splits;
    d.pacc = d.pl + nh * splits;
    d.splits = splits;
    return d;
}
size_t decode_scratch_bytes(int n_seqs, int Hq, int D, int n_sinks, int window) {
    const size_t nh = (size_t)n_seqs * Hq, sp = (size_t)decode_splits(n_sinks, window);
    return sizeof(float) * (3 * nh * D + 2 * nh * sp + nh * sp * D);
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kFeatThreads)
decode_features_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                       const Tin* __restrict__ v, const float* __restrict__ g,
                       const float* __restrict__ beta, const float* __restrict__ wq,
                       const float* __restrict__ wk, const float* __restrict__ wv, hla_state s, DecScratch sc) {
    constexpr int HALF = D / 2;
    __shared__ __align__(16) float qhat_s[kMaxG][D];
    __shared__ __align__(16) float krot_s[D], vraw_s[D], khat_s[D], vhat_s[D];
    __shared__ float cs_s[HALF], sn_s[HALF], inv_s[kMaxG + 1];
    // Launched with programmatic stream serialization: wait for the launch before this one (the previous
    // step's combine, which advanced pos) to complete before any read, then let the next launch place its
    // CTAs (it waits the same way).  No effect on a plain launch.
    pdl_wait();
    pdl_trigger();
    const int kv = blockIdx.x, n = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = L.G, ns = L.n_sinks, W = L.window, R = ns + W, P = W + 1;
    const int64_t p = s.pos[n];
    if (p < 0) {  // not a position a prefill or a decode step can leave: flag it, touch nothing
        if (tid == 0) atomicExch(s.err, kErrState);
        return;
    }
    const size_t kvrow = ((size_t)n * L.Hkv + kv) * D;

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
    // short conv with the history; tap 7 on the new token
    auto conv = [&](float xr, float* hist, size_t step, const float* w) {
        float hst[kConvHalo];
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) hst[m] = hist[m * step];
        float acc = w[kConvHalo] * xr;
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) acc = fmaf(w[m], hst[m], acc);
#pragma unroll
        for (int m = 0; m + 1 < kConvHalo; ++m) hist[m * step] = hst[m + 1];
        hist[(kConvHalo - 1) * step] = xr;
        return acc;
    };
    if (tid < 2 * D) {  // k channels, then v channels
        const bool is_k = tid < D;
        const int c = is_k ? tid : tid - D;
        const float xr = is_k ? rot(k + kvrow, c) : to_f32(v[kvrow + c]);
        const float acc = conv(xr, (is_k ? s.conv_k : s.conv_v) + ((size_t)n * kConvHalo * L.Hkv + kv) * D + c,
                               (size_t)L.Hkv * D, (is_k ? wk : wv) + ((size_t)kv * D + c) * kConvWidth);
        if (is_k) { krot_s[c] = xr; khat_s[c] = acc; }
        else { vraw_s[c] = xr; vhat_s[c] = acc; }
    }
    for (int e = tid; e < G * D; e += kFeatThreads) {
        const int gg = e / D, c = e % D, h = kv * G + gg;
        const float xr = rot(q + ((size_t)n * L.Hq + h) * D, c);
        qhat_s[gg][c] = conv(xr, s.conv_q + ((size_t)n * kConvHalo * L.Hq + h) * D + c, (size_t)L.Hq * D,
                             wq + ((size_t)h * D + c) * kConvWidth);
        sc.qrot[((size_t)n * L.Hq + h) * D + c] = xr;
    }
    __syncthreads();
    // L2 norms: job gg < G is q-head gg, job G is the key
    for (int job = warp; job <= G; job += kFeatThreads / 32) {
        const float* x = job < G ? qhat_s[job] : khat_s;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) inv_s[job] = (job == G || (L.flags & HLA_FLAG_L2NORM_Q)) ? rsqrtf(ss + 1e-6f) : 1.f;
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += kFeatThreads)
        sc.qhat[((size_t)n * L.Hq + kv * G) * D + e] = qhat_s[e / D][e % D] * inv_s[e / D];
    const size_t pslot = (size_t)(p % P);
    if (tid < D) {
        Tin* kring = static_cast<Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
        Tin* vring = static_cast<Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;
        const size_t slot = (size_t)ring_slot(p, ns, W) * D + tid;
        kring[slot] = from_f32<Tin>(krot_s[tid]);
        vring[slot] = from_f32<Tin>(vraw_s[tid]);
        const size_t ps = (((size_t)n * L.Hkv + kv) * P + pslot) * D + tid;
        s.pend_k[ps] = khat_s[tid] * inv_s[G];
        s.pend_v[ps] = vhat_s[tid];
    }
    if (tid < G) {
        const size_t gs = ((size_t)n * L.Hq + kv * G + tid) * P;
        s.pend_g[gs + pslot] = g[(size_t)n * L.Hq + kv * G + tid];
        s.pend_beta[gs + pslot] = beta[(size_t)n * L.Hq + kv * G + tid];
    }
}

// State unit (q-head h, sequence n, value-column half hf), one CTA: the state's columns never mix, so
// each half of a head's state is its own unit.  Thread t owns column group t % (D/8) (four value dims,
// float4) of the half's columns, rows (t / (D/8)) * RPT .. + RPT - 1; the half's 32 KiB are read once into
// registers and written back once.
template <int D>
__device__ __forceinline__ void decode_state_unit(const LayerDims& L, const hla_state& s, const DecScratch& sc,
                                                  int h, int n, int hf) {
    constexpr int NC = D / 2, CG = NC / 4, RG = kStateThreads / CG, RPT = D / RG;
    __shared__ __align__(16) float kj_s[D], vj_s[NC], qh_s[D];
    __shared__ __align__(16) float redx[RG][NC], redy[RG][NC];
    __shared__ float cdot_s;
    const int tid = threadIdx.x, kv = h / L.G, c0 = hf * NC;
    const int ns = L.n_sinks, W = L.window, P = W + 1;
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    const int64_t p = s.pos[n], j = p - W;  // the token leaving the window
    float* olin = sc.olin + ((size_t)n * L.Hq + h) * D + c0;
    if (j < ns) {  // nothing leaves the window into the state this step
        for (int c = tid; c < NC; c += kStateThreads) olin[c] = 0.f;
        return;
    }
    const size_t jslot = (size_t)(j % P);
    const size_t gs = ((size_t)n * L.Hq + h) * P + jslot;
    const float alpha = expf(s.pend_g[gs]), b = s.pend_beta[gs];
    const int cg = tid % CG, rg = tid / CG;
    float4* S4 = reinterpret_cast<float4*>(s.S + ((size_t)n * L.Hq + h) * D * D + c0);
    float4 Sr[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) Sr[r] = S4[(size_t)(rg * RPT + r) * (D / 4) + cg];
    for (int c = tid; c < D; c += kStateThreads) {
        const size_t ps = (((size_t)n * L.Hkv + kv) * P + jslot) * D + c;
        kj_s[c] = s.pend_k[ps];
        if (c < NC) vj_s[c] = s.pend_v[ps + c0];
        qh_s[c] = sc.qhat[((size_t)n * L.Hq + h) * D + c];
    }
    __syncthreads();
    if (tid < 32) {
        float d = 0.f;
        for (int c = tid; c < D; c += 32) d += qh_s[c] * kj_s[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        if (tid == 0) cdot_s = d;
    }
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float kk = kj_s[rg * RPT + r], qq = qh_s[rg * RPT + r];
        x.x = fmaf(kk, Sr[r].x, x.x); x.y = fmaf(kk, Sr[r].y, x.y);
        x.z = fmaf(kk, Sr[r].z, x.z); x.w = fmaf(kk, Sr[r].w, x.w);
        y.x = fmaf(qq, Sr[r].x, y.x); y.y = fmaf(qq, Sr[r].y, y.y);
        y.z = fmaf(qq, Sr[r].z, y.z); y.w = fmaf(qq, Sr[r].w, y.w);
    }
    reinterpret_cast<float4*>(redx[rg])[cg] = x;
    reinterpret_cast<float4*>(redy[rg])[cg] = y;
    __syncthreads();
    float u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int col = 4 * cg + e;
        float xs = 0.f, ys = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) { xs += redx[r][col]; ys += redy[r][col]; }
        u[e] = gla ? vj_s[col] : b * (vj_s[col] - alpha * xs);  // GLA: no erase, write gain 1
        if (rg == 0) olin[col] = fmaf(alpha, ys, cdot_s * u[e]);
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float kk = kj_s[rg * RPT + r];
        float4 o;
        o.x = fmaf(alpha, Sr[r].x, kk * u[0]);
        o.y = fmaf(alpha, Sr[r].y, kk * u[1]);
        o.z = fmaf(alpha, Sr[r].z, kk * u[2]);
        o.w = fmaf(alpha, Sr[r].w, kk * u[3]);
        S4[(size_t)(rg * RPT + r) * (D / 4) + cg] = o;
    }
}

// The 16 / sizeof(T) values of a 16-byte chunk as fp32 pairs.
template <typename T> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
    static constexpr int kPairs = 4;
    static __device__ __forceinline__ void unpack(uint4 u, float2* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) f[k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    }
};
template <> struct Chunk<float> {
    static constexpr int kPairs = 2;
    static __device__ __forceinline__ void unpack(uint4 u, float2* f) {
        f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
};

// CTA (kv head x split, sequence n): softmax partials of the G <= GM heads of
// the group over key slots [split * KS, (split + 1) * KS) of the valid-slot
// list.  No shared-memory staging of the ring: every thread loads, straight
// into registers with 16-byte loads issued up front, exactly the key and value
// chunks it uses.  Logits: lane pairs per key (adjacent chunks, so a warp's
// load covers whole 32-byte sectors), q broadcast from shared memory, one
// shuffle per head.  P V: thread (value chunk, key subset), packed FMAs,
// subsets summed through shared memory.
template <typename Tin, int D, int GM>
struct DecSm {
    static constexpr int kEpc = 16 / (int)sizeof(Tin);  // values per chunk
    static constexpr int kCh = D / kEpc;                // chunks per row
    static constexpr int kKc = kCh / 2;                 // key chunks per thread (two lanes per key)
    static constexpr int kNks = kSmThreads / kCh;       // key subsets in P V
    static constexpr int kKpt = kSplitKeys / kNks;      // value rows per thread
    // shared memory (floats): q [GM][D], logits [GM][keys], P [keys][GM], P V partials [kNks][GM][D]
    static constexpr int kQ = 0, kLg = kQ + GM * D, kP = kLg + GM * kSplitKeys, kPart = kP + kSplitKeys * GM;
    static constexpr size_t kSmemBytes = sizeof(float) * (size_t)(kPart + kNks * GM * D);
    static_assert(kSmThreads == 2 * kSplitKeys, "two lanes per key");
    static_assert(kCh % 2 == 0 && kSmThreads % kCh == 0 && kSplitKeys % kNks == 0, "mapping");
};

template <typename Tin, int D, int GM>
__device__ __forceinline__ void decode_softmax_unit(const LayerDims& L, const hla_state& s, const DecScratch& sc,
                                                    int split, int kv, int n, float* fsm) {
    using P = DecSm<Tin, D, GM>;
    using C = Chunk<Tin>;
    constexpr int NP = C::kPairs;
    float* q_s = fsm + P::kQ;
    float* lg_s = fsm + P::kLg;
    float* p_s = fsm + P::kP;
    float* part_s = fsm + P::kPart;
    __shared__ float m_s[GM], l_s[GM];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = L.G, ns = L.n_sinks, W = L.window, R = ns + W;
    const int64_t p = s.pos[n];
    const int nsk = (int)(p + 1 < ns ? p + 1 : ns);
    const int n_win = p >= ns ? (int)min((int64_t)W, p - ns + 1) : 0;
    const int n_keys = nsk + n_win;
    const int KS = (R + sc.splits - 1) / sc.splits;
    const int k0 = split * KS, nt = max(0, min(KS, n_keys - k0));
    const uint4* kring = reinterpret_cast<const uint4*>(static_cast<const Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D);
    const uint4* vring = reinterpret_cast<const uint4*>(static_cast<const Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D);
    auto slot_of = [&](int i) { return i < nsk ? i : ns + (i - nsk); };  // valid-slot list entry -> ring slot

    // loads first: this thread's key chunks (key ki, chunks 2c + kh) and value chunks (chunk vc of
    // rows vk + kNks r); rows past the split's keys read as zero
    const int ki = tid >> 1, kh = tid & 1;
    const int vc = tid % P::kCh, vk = tid / P::kCh;
    uint4 kraw[P::kKc], vraw[P::kKpt];
    {
        const uint4* kr = kring + (size_t)slot_of(k0 + min(ki, max(nt - 1, 0))) * P::kCh;
#pragma unroll
        for (int c = 0; c < P::kKc; ++c) kraw[c] = ki < nt ? __ldg(kr + 2 * c + kh) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < P::kKpt; ++r) {
            const int i = vk + P::kNks * r;
            vraw[r] = i < nt ? __ldg(vring + (size_t)slot_of(k0 + i) * P::kCh + vc) : make_uint4(0, 0, 0, 0);
        }
    }
    for (int e = tid; e < G * D; e += kSmThreads) q_s[e] = sc.qrot[((size_t)n * L.Hq + kv * G) * D + e];
    __syncthreads();

    // logits of key ki: this lane's half of the dot products, then the pair's sum
    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
    {
        float2 acc[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < P::kKc; ++c) {
            float2 kf[NP];
            C::unpack(kraw[c], kf);
            const int d0 = (2 * c + kh) * P::kEpc;
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g < G) {
#pragma unroll
                    for (int e = 0; e < NP; e += 2) {
                        const float4 qv = *reinterpret_cast<const float4*>(q_s + g * D + d0 + 2 * e);
                        acc[g] = ffma2(make_float2(qv.x, qv.y), kf[e], acc[g]);
                        acc[g] = ffma2(make_float2(qv.z, qv.w), kf[e + 1], acc[g]);
                    }
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            float t = acc[g].x + acc[g].y;
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            if (g < G && kh == 0) lg_s[g * kSplitKeys + ki] = t * qscale;
        }
    }
    __syncthreads();
    for (int g = warp; g < G; g += kSmThreads / 32) {  // per-head max and sum; P into [key][head]
        float mx = -INFINITY;
        for (int i = lane; i < nt; i += 32) mx = fmaxf(mx, lg_s[g * kSplitKeys + i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int i = lane; i < kSplitKeys; i += 32) {
            const float e = i < nt ? exp2f(lg_s[g * kSplitKeys + i] - mx) : 0.f;
            p_s[i * GM + g] = e;
            sum += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) { m_s[g] = mx; l_s[g] = sum; }
    }
    __syncthreads();

    // P V over this thread's value rows, then the key subsets summed
    {
        float2 acc[GM][NP];
#pragma unroll
        for (int g = 0; g < GM; ++g)
#pragma unroll
            for (int e = 0; e < NP; ++e) acc[g][e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < P::kKpt; ++r) {
            const int i = vk + P::kNks * r;
            float2 vf[NP];
            C::unpack(vraw[r], vf);
            float pr[GM];
#pragma unroll
            for (int g = 0; g < GM; g += 4) {
                if constexpr (GM >= 4) {
                    const float4 p4 = *reinterpret_cast<const float4*>(p_s + i * GM + g);
                    pr[g] = p4.x; pr[g + 1] = p4.y; pr[g + 2] = p4.z; pr[g + 3] = p4.w;
                } else {
#pragma unroll
                    for (int u = 0; u < GM; ++u) pr[u] = p_s[i * GM + u];
                }
            }
#pragma unroll
            for (int g = 0; g < GM; ++g)
                if (g < G)
#pragma unroll
                    for (int e = 0; e < NP; ++e) acc[g][e] = ffma2(make_float2(pr[g], pr[g]), vf[e], acc[g][e]);
        }
#pragma unroll
        for (int g = 0; g < GM; ++g)
            if (g < G)
#pragma unroll
                for (int e = 0; e < NP; ++e)
                    *reinterpret_cast<float2*>(part_s + (vk * GM + g) * D + vc * P::kEpc + 2 * e) = acc[g][e];
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += kSmThreads) {
        const int g = e / D, c = e % D;
        float o = 0.f;
#pragma unroll
        for (int r = 0; r < P::kNks; ++r) o += part_s[(r * GM + g) * D + c];
        const size_t hs = ((size_t)n * L.Hq + kv * G + g) * sc.splits + split;
        sc.pacc[hs * D + c] = o;
        if (c == 0) {
            sc.pm[hs] = nt > 0 ? m_s[g] : -INFINITY;
            sc.pl[hs] = nt > 0 ? l_s[g] : 0.f;
        }
    }
}

// One launch for the step's two streams over HBM: per (kv head, sequence) a
// run of 2G state units (the two value-column halves of each of the group's
// heads) followed by the softmax splits, so the state updates and the ring
// reads share every wave of CTAs.  Half-head state units keep 64 floats of
// state per thread, which lets five CTAs share an SM (bf16 rings; fp32 rings
// need the registers of three) and so keeps more of the stream in flight.
template <typename Tin, int D, int GM>
__global__ void __launch_bounds__(kSmThreads, sizeof(Tin) == 2 ? 5 : 3)
decode_attn_state_kernel(LayerDims L, hla_state s, DecScratch sc) {
    static_assert(kStateThreads == kSmThreads, "one CTA shape for both units");
    extern __shared__ __align__(16) float fsm[];
    pdl_wait();  // the features launch has completed (see decode_features_kernel)
    pdl_trigger();
    const int run = 2 * L.G + sc.splits, kv = blockIdx.x / run, r = blockIdx.x % run, n = blockIdx.y;
    if (r < 2 * L.G) decode_state_unit<D>(L, s, sc, kv * L.G + (r >> 1), n, r & 1);
    else decode_softmax_unit<Tin, D, GM>(L, s, sc, r - 2 * L.G, kv, n, fsm);
}

// CTA per (q-head, sequence), thread per channel: splits merged by their
// maxima (read sixteen at a time, so their loads overlap: one batch for an
// 896-slot ring), o = o_sm + lambda_h o_lin; then the sequence's position
// advances (CTA of head 0: no CTA of this launch reads it).
// Merge of the softmax splits of (q-head h, sequence n): warp 0 forms the splits' weights
// 2^(m_r - M) (M the largest split maximum, splits without keys weighted 0) and the normaliser
// sum_r 2^(m_r - M) l_r once, a tile of kCombineTile weights at a time in shared memory; every thread then
// sums its value dim over the splits' partial outputs.  Then + lambda_h o_lin, and pos advances.
constexpr int kCombineTile = 256;
template <typename Tin, int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(LayerDims L, DecScratch sc, const float* __restrict__ lambda, Tin* __restrict__ out,
                      int64_t* __restrict__ pos) {
    // (a negative position was flagged by the features launch; it is left as it is)
    __shared__ float w_s[kCombineTile];
    __shared__ float mx_s, inv_s;
    pdl_wait();  // the state + softmax launch has completed (see decode_features_kernel)
    pdl_trigger();
    const int h = blockIdx.x, n = blockIdx.y, c = threadIdx.x, lane = c & 31;
    const size_t hs = ((size_t)n * L.Hq + h) * sc.splits;
    if (c < 32) {
        float m = -INFINITY;
        for (int r = lane; r < sc.splits; r += 32)
            if (sc.pl[hs + r] > 0.f) m = fmaxf(m, sc.pm[hs + r]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        if (m != -INFINITY)
            for (int r = lane; r < sc.splits; r += 32) {
                const float pl = sc.pl[hs + r];
                if (pl > 0.f) l = fmaf(pl, exp2f(sc.pm[hs + r] - m), l);
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            mx_s = m;
            inv_s = l > 0.f ? 1.f / l : 0.f;
        }
    }
    __syncthreads();
    const float m = mx_s;
    float o0 = 0.f, o1 = 0.f;  // two chains
    for (int r0 = 0; r0 < sc.splits && m != -INFINITY; r0 += kCombineTile) {
        const int nr = min(kCombineTile, sc.splits - r0);
        __syncthreads();  // the previous tile's weights are no longer read
        for (int r = c; r < nr; r += D) {
            const float pl = sc.pl[hs + r0 + r];
            w_s[r] = pl > 0.f ? exp2f(sc.pm[hs + r0 + r] - m) : 0.f;
        }
        __syncthreads();
        const float* pa = sc.pacc + (hs + r0) * D + c;
        int r = 0;
        for (; r + 1 < nr; r += 2) {
            o0 = fmaf(w_s[r], pa[(size_t)r * D], o0);
            o1 = fmaf(w_s[r + 1], pa[(size_t)(r + 1) * D], o1);
        }
        if (r < nr) o0 = fmaf(w_s[r], pa[(size_t)r * D], o0);
    }
    float o = (L.flags & HLA_FLAG_SOFTMAX_OFF) ? 0.f : (o0 + o1) * inv_s;
    if (!(L.flags & HLA_FLAG_LINEAR_OFF)) o = fmaf(__ldg(lambda + h), sc.olin[((size_t)n * L.Hq + h) * D + c], o);
    out[((size_t)n * L.Hq + h) * D + c] = from_f32<Tin>(o);
    if (h == 0 && c == 0 && pos[n] >= 0) pos[n] += 1;
}

template <typename Tin, int D, int GM>
cudaError_t launch_decode_attn_state(const LayerDims& L, const hla_state& s, const DecScratch& sc, cudaStream_t st) {
    using P = DecSm<Tin, D, GM>;
    static DeviceCache cache;  // the shared-memory attribute, per device and instantiation
    cudaError_t e = device_cached(cache, nullptr, [](int, int*) {
        return cudaFuncSetAttribute(decode_attn_state_kernel<Tin, D, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)P::kSmemBytes);
    });
    if (e != cudaSuccess) return e;
    LaunchCfg lc(dim3(L.Hkv * (2 * L.G + sc.splits), L.n_seqs), dim3(kSmThreads), P::kSmemBytes, st, true);
    return cudaLaunchKernelEx(&lc.cfg, decode_attn_state_kernel<Tin, D, GM>, L, s, sc);
}

template <typename Tin, int D>
cudaError_t decode_kernels(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* g,
                           const float* beta, const float* lambda, const float* wq, const float* wk,
                           const float* wv, const hla_state& s, Tin* out, cudaStream_t st) {
    const DecScratch sc = dec_scratch(static_cast<float*>(s.scratch), L.n_seqs, L.Hq, D, decode_splits(L.n_sinks, L.window));
    // three launches, each placed while the one before it finishes (programmatic dependent launch; every
    // kernel waits for its predecessor to complete before its first read)
    {
        LaunchCfg lc(dim3(L.Hkv, L.n_seqs), dim3(kFeatThreads), 0, st, true);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, decode_features_kernel<Tin, D>, L, q, k, v, g, beta, wq, wk, wv, s,
                                           sc);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e0 = L.G <= 1 ? launch_decode_attn_state<Tin, D, 1>(L, s, sc, st)
                   : L.G <= 2 ? launch_decode_attn_state<Tin, D, 2>(L, s, sc, st)
                   : L.G <= 4 ? launch_decode_attn_state<Tin, D, 4>(L, s, sc, st)
                              : launch_decode_attn_state<Tin, D, 8>(L, s, sc, st);
    if (e0 != cudaSuccess) return e0;
    LaunchCfg lc(dim3(L.Hq, L.n_seqs), dim3(D), 0, st, true);
    return cudaLaunchKernelEx(&lc.cfg, decode_combine_kernel<Tin, D>, L, sc, lambda, out, s.pos);
}

template <typename Tin>
cudaError_t launch_decode_step(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                               const float* g, const float* beta, const float* lambda,
                               const float* wq, const float* wk, const float* wv,
                               const hla_state& s, Tin* out, cudaStream_t st) {
    if (L.G > kMaxG) return cudaErrorInvalidValue;
    if (L.n_seqs <= 0) return cudaSuccess;
    cudaError_t e = L.d == 128 ? decode_kernels<Tin, 128>(L, q, k, v, g, beta, lambda, wq, wk, wv, s, out, st)
                               : decode_kernels<Tin, 64>(L, q, k, v, g, beta, lambda, wq, wk, wv, s, out, st);
    return e;
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
