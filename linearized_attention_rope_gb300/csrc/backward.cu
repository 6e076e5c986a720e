// Backward of the hybrid layer: the gradients of L = sum(dO . o) with respect
// to q, k, v, the gates g, beta, the branch weight lambda and the conv
// filters, for the layer of "迈向线性的关键：分析驱动的 Transformer 线性化"
// (RoPE -> short conv -> L2 norm feature path of section 实践建议 item 3, the
// delayed GDN of sections 线性注意力替换机制 and 填补近似缺口的实用设计, the
// sink + window softmax) combined as o = o_sm + lambda_h o_lin ("Untangling
// Component Imbalance in Hybrid Linear Attention Conversion", 关键设计 (1)).
//
// fp32 throughout, on the CUDA cores; every reduction has a fixed order (no
// atomics).  Launches, in order:
//  0. the 64-row block table of the sequences (and a check of cu_seqlens);
//  1. rope: RoPE'd q and k rows (fp32) for every token and head;
//  2. conv: q~, k~ (and their L2-normalised qhat, khat) and vhat = conv(v);
//  3. GDN, a cluster of 8 CTAs per (sequence, q-head) splitting the value
//     columns: a forward pass that keeps the state every 64 absorptions (and
//     lambda's partial sum), then per 64-absorption block, last first, the
//     states every 8 (d 128) or 16 (d 64) absorptions, and per such stage the
//     states in registers and the read-out and absorption steps differentiated
//     in reverse (dqhat, and per head dkhat, dvhat, dg, dbeta);
//  4. softmax: per 64-query block the rows' max, sum and D = dO . o_sm and dq;
//     per 64-key block dk, dv of its non-sink keys; the sink keys' sums over
//     the query blocks' partials;
//  5. feature backward of q (L2, conv, RoPE); of k and v after the per-head
//     gradients of each kv group are summed;
//  6. the conv filters' gradients (per token block, then over the blocks);
//  7. lambda's gradient over the sequences.
#include "hla_common.cuh"

namespace hla {

namespace {

constexpr int kWB = 256;    // tokens per block of the conv-filter reduction

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// sum over the CTA of v, for every thread (red: 32 floats)
__device__ __forceinline__ float cta_sum_f(float v, float* red) {
    v = warp_sum_f(v);
    const int nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    __syncthreads();
    return t;
}
// ---- 1. RoPE'd rows: row r < Hq is q-head r, else k-head r - Hq; thread per channel
template <typename Tin>
__global__ void bwd_rope_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                                const int32_t* __restrict__ cu, float* __restrict__ qr, float* __restrict__ kr,
                                int32_t* __restrict__ err) {
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d, half = D / 2;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    // a token outside every sequence: cu_seqlens is not a monotone table from 0 to total
    if ((p < 0 || p >= len) && r == 0 && c == 0) atomicExch(err, kErrSeqlens);
    const bool isq = r < L.Hq;
    const int hh = isq ? r : r - L.Hq, H = isq ? L.Hq : L.Hkv;
    const Tin* x = (isq ? q : k) + ((size_t)t * H + hh) * D;
    const int i = c % half;
    float cs, sn;
    rope_cs_exact(p, L.theta[i], &cs, &sn);
    const float x1 = to_f32(x[i]), x2 = to_f32(x[i + half]);
    (isq ? qr : kr)[((size_t)t * H + hh) * D + c] = c < half ? x1 * cs - x2 * sn : x2 * cs + x1 * sn;
}

// ---- 2. conv (+ L2): rows r < Hq: q-heads, < Hq + Hkv: k-heads, else v-heads; thread per channel
template <typename Tin>
__global__ void bwd_conv_kernel(LayerDims L, const Tin* __restrict__ v, const float* __restrict__ wq,
                                const float* __restrict__ wk, const float* __restrict__ wv,
                                const int32_t* __restrict__ cu, const float* __restrict__ qr,
                                const float* __restrict__ kr, float* __restrict__ qt, float* __restrict__ qh,
                                float* __restrict__ kt, float* __restrict__ kh, float* __restrict__ vh) {
    __shared__ float red[32];
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* w = (kind == 0 ? wq : kind == 1 ? wk : wv) + ((size_t)hh * D + c) * kConvWidth;
    float acc = 0.f;
    for (int m = 0; m < kConvWidth; ++m) {
        const int64_t pp = p - (kConvWidth - 1) + m;
        if (pp < 0) continue;
        const size_t row = ((size_t)(start + pp) * H + hh) * D + c;
        const float x = kind == 0 ? qr[row] : kind == 1 ? kr[row] : to_f32(v[row]);
        acc = fmaf(w[m], x, acc);
    }
    const size_t o = ((size_t)t * H + hh) * D + c;
    if (kind == 2) {
        vh[o] = acc;
        return;
    }
    const bool norm = kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q);
    const float inv = norm ? rsqrtf(cta_sum_f(acc * acc, red) + 1e-6f) : 1.f;
    (kind == 0 ? qt : kt)[o] = acc;
    (kind == 0 ? qh : kh)[o] = acc * inv;
}

// ---- 3. GDN backward: a cluster of kCl CTAs per (q-head, sequence), each CTA D / kCl value columns of S
// (the columns of the recurrence are independent: only the gradients of q, k, alpha and beta sum over
// them).  A warp holds CPW columns, lane l rows l, l + 32, ... of each, in registers.  Three passes over
// the absorptions, all fed by one schedule of K-token stages loaded ahead with cp.async:
//   0: forward: S every 64 absorptions to the global checkpoints; lambda's gradient sum(dO . o_lin);
//   1: per 64-absorption block, last block first: from its checkpoint, S every K absorptions to a
//      per-(sequence, head) scratch (stays in L2);
//   2: the same block's K-stages, last first: the K + 1 states from the scratch state, in registers; then
//      the read-out and absorption steps differentiated in reverse.  Per stage the warps' contributions
//      to dq, dk, dalpha, dbeta are summed in the CTA, then over the cluster's CTAs through distributed
//      shared memory (one cluster barrier per stage, double-buffered); dv is per column.
constexpr int kCl = 8;      // CTAs per cluster
constexpr int kGW = 8;      // warps per CTA
constexpr int kGT = kGW * 32;
constexpr int kCkB = 64;    // absorptions per global checkpoint
constexpr int kRing = 3;    // stages in flight
template <int D> struct GdnB {
    static constexpr int K = D == 128 ? 8 : 16;  // absorptions per stage (the states of one stage in registers)
    static constexpr int E = D / 32, CPC = D / kCl, CPW = CPC / kGW, SPB = kCkB / K;
    // shared memory (floats): warp partials, cluster exchange (2 buffers), stage ring, dv of a stage, sums
    static constexpr int PART = K * 2 * kGW * D, SPART = K * 2 * kGW, XCH = 2 * K * 2 * D, XS = 2 * K * 2;
    static constexpr int SLOT = 2 * K * D + 2 * K * CPC + 2 * K;
    static constexpr size_t BYTES = (size_t)(PART + SPART + XCH + XS + kRing * SLOT + K * CPC + kGW + 4) * 4;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the float at the same shared-memory offset as `local` in CTA `rank` of the cluster
__device__ __forceinline__ float ld_cluster(const float* local, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}
__device__ __forceinline__ void cp_async(void* dst, const void* src, int bytes16or4) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    if (bytes16or4 == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_ring() { asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory"); }

template <int N>
__device__ __forceinline__ void warp_sum_n(float (&x)[N]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kGT, 2)
bwd_gdn_kernel(LayerDims L, const float* __restrict__ g, const float* __restrict__ beta,
               const float* __restrict__ lambda, const Tin* __restrict__ dout, const int32_t* __restrict__ cu,
               const float* __restrict__ qh, const float* __restrict__ kh, const float* __restrict__ vh,
               float* __restrict__ ckpt, float* __restrict__ sub, float* __restrict__ dqh,
               float* __restrict__ dkh_h, float* __restrict__ dvh_h, float* __restrict__ dg,
               float* __restrict__ dbeta, float* __restrict__ dlam_part) {
    using B = GdnB<D>;
    constexpr int K = B::K, E = B::E, CPC = B::CPC, CPW = B::CPW, SPB = B::SPB;
    extern __shared__ __align__(16) float smem[];
    float* part = smem;                 // [K][2][kGW][D]: dq (0), dk (1) of each warp's columns
    float* spart = part + B::PART;      // [K][2][kGW]: dalpha, dbeta
    float* xch = spart + B::SPART;      // [2][K][2][D]: the CTA's sums
    float* xs = xch + B::XCH;           // [2][K][2]
    float* ring = xs + B::XS;           // kRing stage slots
    float* dv_s = ring + kRing * B::SLOT;  // [K][CPC]
    float* red = dv_s + K * CPC;        // [kGW] + 1
    const uint32_t rank = cluster_rank();
    const int h = blockIdx.x / kCl, n = blockIdx.y, kv = h / L.G, tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const int ns = L.n_sinks, W = L.window;
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    if (L.flags & HLA_FLAG_LINEAR_OFF) {  // o does not depend on the linear branch (the whole cluster leaves)
        if (rank == 0 && tid == 0) dlam_part[(size_t)n * L.Hq + h] = 0.f;
        return;
    }
    const float lam = lambda[h];
    const int64_t n_abs = max((int64_t)0, len - W - ns);
    const int n_st = (int)((n_abs + K - 1) / K);          // stages
    const int n_blk = (n_st + SPB - 1) / SPB;             // checkpoint blocks
    const int last_nb = n_st - (n_blk - 1) * SPB;         // stages of the last block
    const int n_sched = 3 * n_st;
    const size_t DD = (size_t)D * D;
    const int64_t ck0 = start / kCkB + n;                 // the sequence's first global checkpoint slot
    float* my_sub = sub + ((size_t)n * L.Hq + h) * SPB * DD;
    auto colg = [&](int cw) { return (int)rank * CPC + w * CPW + cw; };  // global column of (warp, cw)
    auto ck_col = [&](int blk, int cw) { return ckpt + ((size_t)(ck0 + blk) * L.Hq + h) * DD + (size_t)colg(cw) * D; };
    auto sub_col = [&](int si, int cw) { return my_sub + (size_t)si * DD + (size_t)colg(cw) * D; };

    // schedule entry i -> (phase, stage)
    auto sched = [&](int i, int* phase, int* s) {
        if (i < n_st) {
            *phase = 0;
            *s = i;
            return;
        }
        int r = i - n_st, blk, loc, nb;
        if (r < 2 * last_nb) {
            blk = n_blk - 1;
            loc = r;
            nb = last_nb;
        } else {
            r -= 2 * last_nb;
            blk = n_blk - 2 - r / (2 * SPB);
            loc = r % (2 * SPB);
            nb = SPB;
        }
        *phase = loc < nb ? 1 : 2;
        *s = blk * SPB + (loc < nb ? loc : 2 * nb - 1 - loc);
    };
    // slot layout: k [K][D], q [K][D], v [K][CPC], dO [K][CPC] (Tin), g [K], beta [K]
    auto slot_k = [&](int sl) { return ring + sl * B::SLOT; };
    auto slot_q = [&](int sl) { return ring + sl * B::SLOT + K * D; };
    auto slot_v = [&](int sl) { return ring + sl * B::SLOT + 2 * K * D; };
    auto slot_o = [&](int sl) { return reinterpret_cast<Tin*>(ring + sl * B::SLOT + 2 * K * D + K * CPC); };
    auto slot_g = [&](int sl) { return ring + sl * B::SLOT + 2 * K * D + 2 * K * CPC; };
    auto slot_b = [&](int sl) { return ring + sl * B::SLOT + 2 * K * D + 2 * K * CPC + K; };
    auto issue = [&](int i) {
        if (i < n_sched) {
            int phase, s;
            sched(i, &phase, &s);
            const int sl = i % kRing;
            const int64_t m0 = (int64_t)s * K;
            const int cnt = (int)min((int64_t)K, n_abs - m0);
            for (int idx = tid; idx < K * (D / 4); idx += kGT) {
                const int t = idx / (D / 4), c = (idx % (D / 4)) * 4;
                if (t < cnt) {
                    const int64_t j = ns + m0 + t, p = j + W;
                    cp_async(slot_k(sl) + t * D + c, kh + ((size_t)(start + j) * L.Hkv + kv) * D + c, 16);
                    cp_async(slot_q(sl) + t * D + c, qh + ((size_t)(start + p) * L.Hq + h) * D + c, 16);
                }
            }
            for (int idx = tid; idx < K * (CPC / 4); idx += kGT) {
                const int t = idx / (CPC / 4), c = (idx % (CPC / 4)) * 4;
                if (t < cnt) {
                    const int64_t j = ns + m0 + t;
                    cp_async(slot_v(sl) + t * CPC + c, vh + ((size_t)(start + j) * L.Hkv + kv) * D + rank * CPC + c, 16);
                }
            }
            constexpr int OCH = CPC * (int)sizeof(Tin) / 16;  // 16-byte chunks of a dO row slice
            for (int idx = tid; idx < K * OCH; idx += kGT) {
                const int t = idx / OCH, c = (idx % OCH) * (16 / (int)sizeof(Tin));
                if (t < cnt) {
                    const int64_t p = ns + m0 + t + W;
                    cp_async(slot_o(sl) + t * CPC + c, dout + ((size_t)(start + p) * L.Hq + h) * D + rank * CPC + c, 16);
                }
            }
            if (tid < cnt) {
                const int64_t j = ns + m0 + tid;
                cp_async(slot_g(sl) + tid, g + (size_t)(start + j) * L.Hq + h, 4);
                cp_async(slot_b(sl) + tid, beta + (size_t)(start + j) * L.Hq + h, 4);
            }
        }
        cp_async_commit();
    };
    // one absorption of stage token t into S (registers)
    auto absorb = [&](float (&S)[CPW][E], int sl, int t) {
        const float* kr = slot_k(sl) + t * D;
        float k[E];
#pragma unroll
        for (int e = 0; e < E; ++e) k[e] = kr[lane + 32 * e];
        float x[CPW];
#pragma unroll
        for (int cw = 0; cw < CPW; ++cw) {
            x[cw] = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) x[cw] = fmaf(k[e], S[cw][e], x[cw]);
        }
        warp_sum_n<CPW>(x);
        const float a = expf(slot_g(sl)[t]), b = slot_b(sl)[t];
#pragma unroll
        for (int cw = 0; cw < CPW; ++cw) {
            const float vv = slot_v(sl)[t * CPC + w * CPW + cw];
            const float u = gla ? vv : b * (vv - a * x[cw]);
#pragma unroll
            for (int e = 0; e < E; ++e) S[cw][e] = fmaf(a, S[cw][e], k[e] * u);
        }
    };

    float S[CPW][E];
#pragma unroll
    for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
        for (int e = 0; e < E; ++e) S[cw][e] = 0.f;
    float dS[CPW][E];
#pragma unroll
    for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
        for (int e = 0; e < E; ++e) dS[cw][e] = 0.f;
    float dl = 0.f;
    int buf = 0;
    for (int i = 0; i < kRing; ++i) issue(i);
    for (int i = 0; i < n_sched; ++i) {
        cp_async_wait_ring();
        __syncthreads();
        int phase, s;
        sched(i, &phase, &s);
        const int sl = i % kRing;
        const int64_t m0 = (int64_t)s * K;
        const int cnt = (int)min((int64_t)K, n_abs - m0);
        const int blk = s / SPB, si = s % SPB;
        if (phase == 0) {
            if (si == 0) {
#pragma unroll
                for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                    for (int e = 0; e < E; ++e) ck_col(blk, cw)[lane + 32 * e] = S[cw][e];
            }
#pragma unroll
            for (int t = 0; t < K; ++t) {
                if (t < cnt) {
                    absorb(S, sl, t);
                    // read-out at p = j + W for lambda's gradient
                    const float* qr = slot_q(sl) + t * D;
                    float o[CPW];
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw) {
                        o[cw] = 0.f;
#pragma unroll
                        for (int e = 0; e < E; ++e) o[cw] = fmaf(qr[lane + 32 * e], S[cw][e], o[cw]);
                    }
                    warp_sum_n<CPW>(o);
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw) dl = fmaf(to_f32(slot_o(sl)[t * CPC + w * CPW + cw]), o[cw], dl);
                }
            }
        } else if (phase == 1) {
            if (si == 0) {
#pragma unroll
                for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                    for (int e = 0; e < E; ++e) S[cw][e] = ck_col(blk, cw)[lane + 32 * e];
            }
#pragma unroll
            for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                for (int e = 0; e < E; ++e) sub_col(si, cw)[lane + 32 * e] = S[cw][e];
#pragma unroll
            for (int t = 0; t < K; ++t)
                if (t < cnt) absorb(S, sl, t);
        } else {
            // the stage's states S_{m0} .. S_{m0 + cnt}
            float St[K + 1][CPW][E];
#pragma unroll
            for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                for (int e = 0; e < E; ++e) St[0][cw][e] = sub_col(si, cw)[lane + 32 * e];
#pragma unroll
            for (int t = 0; t < K; ++t) {
#pragma unroll
                for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                    for (int e = 0; e < E; ++e) St[t + 1][cw][e] = St[t][cw][e];
                if (t < cnt) absorb(St[t + 1], sl, t);
            }
#pragma unroll
            for (int tt = 0; tt < K; ++tt) {
                const int t = K - 1 - tt;
                if (t < cnt) {
                    const float* kr = slot_k(sl) + t * D;
                    const float* qr = slot_q(sl) + t * D;
                    float k[E], q[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        k[e] = kr[lane + 32 * e];
                        q[e] = qr[lane + 32 * e];
                    }
                    float ldo[CPW], vv[CPW];
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw) {
                        ldo[cw] = lam * to_f32(slot_o(sl)[t * CPC + w * CPW + cw]);
                        vv[cw] = slot_v(sl)[t * CPC + w * CPW + cw];
                    }
                    // read-out at p: o_lin = S_{m+1}^T qhat -> dqhat += S_{m+1} dO_lin, dS += qhat dO_lin^T
                    float* pq = part + ((t * 2 + 0) * kGW + w) * D;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        float acc = 0.f;
#pragma unroll
                        for (int cw = 0; cw < CPW; ++cw) acc = fmaf(St[t + 1][cw][e], ldo[cw], acc);
                        pq[lane + 32 * e] = acc;
                    }
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                        for (int e = 0; e < E; ++e) dS[cw][e] = fmaf(q[e], ldo[cw], dS[cw][e]);
                    // absorption of token j from S_prev = S_m
                    float red3[3 * CPW];
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw) {
                        float x = 0.f, du = 0.f, gs = 0.f;
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            x = fmaf(k[e], St[t][cw][e], x);
                            du = fmaf(k[e], dS[cw][e], du);
                            gs = fmaf(dS[cw][e], St[t][cw][e], gs);
                        }
                        red3[3 * cw] = x;
                        red3[3 * cw + 1] = du;
                        red3[3 * cw + 2] = gs;
                    }
                    warp_sum_n<3 * CPW>(red3);
                    const float a = expf(slot_g(sl)[t]), b = slot_b(sl)[t];
                    float da = 0.f, db = 0.f, u[CPW], du[CPW];
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw) {
                        const float x = red3[3 * cw];
                        du[cw] = red3[3 * cw + 1];
                        u[cw] = gla ? vv[cw] : b * (vv[cw] - a * x);
                        if (lane == 0) dv_s[t * CPC + w * CPW + cw] = gla ? du[cw] : b * du[cw];
                        db += gla ? 0.f : du[cw] * (vv[cw] - a * x);
                        da += red3[3 * cw + 2] - (gla ? 0.f : b * du[cw] * x);
                    }
                    if (lane == 0) {
                        spart[(t * 2 + 0) * kGW + w] = da;
                        spart[(t * 2 + 1) * kGW + w] = db;
                    }
                    // dk = dS u - a b S_prev du (GLA: dS v); dS_prev = a (dS - b k du^T) (GLA: a dS)
                    float* pk = part + ((t * 2 + 1) * kGW + w) * D;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        float acc = 0.f;
#pragma unroll
                        for (int cw = 0; cw < CPW; ++cw) {
                            acc = fmaf(dS[cw][e], u[cw], acc);
                            if (!gla) acc = fmaf(-a * b * St[t][cw][e], du[cw], acc);
                        }
                        pk[lane + 32 * e] = acc;
                    }
#pragma unroll
                    for (int cw = 0; cw < CPW; ++cw)
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            dS[cw][e] = gla ? a * dS[cw][e] : a * fmaf(-b * k[e], du[cw], dS[cw][e]);
                }
            }
            __syncthreads();
            // the CTA's sums over its warps
            float* xb = xch + buf * (K * 2 * D);
            float* xsb = xs + buf * (K * 2);
            for (int idx = tid; idx < K * 2 * D; idx += kGT) {
                const int tq = idx / D, r = idx % D;
                float acc = 0.f;
#pragma unroll
                for (int ww = 0; ww < kGW; ++ww) acc += part[(tq * kGW + ww) * D + r];
                xb[idx] = acc;
            }
            if (tid < K * 2) {
                float acc = 0.f;
#pragma unroll
                for (int ww = 0; ww < kGW; ++ww) acc += spart[tid * kGW + ww];
                xsb[tid] = acc;
            }
            cluster_sync_all();
            // over the cluster: this CTA finishes rows [rank D / kCl, (rank + 1) D / kCl) of dq and dk
            constexpr int RS = D / kCl;
            for (int idx = tid; idx < K * 2 * RS; idx += kGT) {
                const int tq = idx / RS, t = tq / 2, r = (int)rank * RS + idx % RS;
                if (t < cnt) {
                    float acc = 0.f;
#pragma unroll
                    for (int rr = 0; rr < kCl; ++rr) acc += ld_cluster(xb + tq * D + r, rr);
                    const int64_t j = ns + m0 + t;
                    if (tq % 2 == 0)
                        dqh[((size_t)(start + j + W) * L.Hq + h) * D + r] = acc;
                    else
                        dkh_h[((size_t)(start + j) * L.Hq + h) * D + r] = acc;
                }
            }
            if (rank == 0 && tid < K * 2) {
                const int t = tid / 2;
                if (t < cnt) {
                    float acc = 0.f;
#pragma unroll
                    for (int rr = 0; rr < kCl; ++rr) acc += ld_cluster(xsb + tid, rr);
                    const size_t o = (size_t)(start + ns + m0 + t) * L.Hq + h;
                    if (tid % 2 == 0)
                        dg[o] = acc * expf(slot_g(sl)[t]);
                    else
                        dbeta[o] = acc;
                }
            }
            for (int idx = tid; idx < K * CPC; idx += kGT) {
                const int t = idx / CPC, c = idx % CPC;
                if (t < cnt) dvh_h[((size_t)(start + ns + m0 + t) * L.Hq + h) * D + rank * CPC + c] = dv_s[idx];
            }
            buf ^= 1;
        }
        __syncthreads();
        issue(i + kRing);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // lambda's gradient: over the warps, then over the cluster
    if (lane == 0) red[w] = dl;
    __syncthreads();
    if (tid == 0) {
        float acc = 0.f;
        for (int ww = 0; ww < kGW; ++ww) acc += red[ww];
        red[kGW] = acc;
    }
    cluster_sync_all();
    if (rank == 0 && tid == 0) {
        float acc = 0.f;
        for (int rr = 0; rr < kCl; ++rr) acc += ld_cluster(red + kGW, rr);
        dlam_part[(size_t)n * L.Hq + h] = acc;
    }
    cluster_sync_all();  // every CTA's shared memory stays until rank 0 has read it
}

// ---- 4. softmax backward: 64 x 64 fp32 tiles in shared memory, on the CUDA cores.
// Per 64-query block (query-centric): the row max m, sum l and o_sm (online, over the visible key tiles),
// D = dO . o_sm / l, then dq = scale sum_j P (dP - D) k_j over the tiles again; the sink keys' dk, dv
// partial sums of the block go to a per-block buffer.  Per 64-key block (key-centric): dk, dv of its
// non-sink keys from the queries that see them (at most 63 + W of them), with P, dS from the rows' m, l, D.
// Last, per (sequence, head) the sink keys' partials are summed over the query blocks.
constexpr int kSB = 64;          // queries or keys per tile
constexpr int kSmThreads = 256;  // 16 x 16: a thread holds rows ty + 16 i, columns tx + 16 j of a 64 x 64 tile
constexpr int kLP = kSB + 4;     // row pitch (floats) of the 64 x 64 tiles

template <int D> constexpr size_t sm_smem_bytes(int n_tiles64) {
    return (size_t)(4 * kSB * (D + 4) + n_tiles64 * kSB * kLP + 3 * kSB) * sizeof(float);
}

// acc[i][j] += sum_k A[ty + 16 i][k] B[tx + 16 j][k] (row pitch D + 4, 16-byte rows)
template <int D>
__device__ __forceinline__ void mm_abT(const float* __restrict__ A, const float* __restrict__ B, int ty, int tx,
                                       float acc[4][4]) {
    constexpr int LD = D + 4;
#pragma unroll 2
    for (int k = 0; k < D; k += 4) {
        float4 a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (ty + 16 * i) * LD + k);
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(B + (tx + 16 * j) * LD + k);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][j] = fmaf(a[i].x, b[j].x, acc[i][j]);
                acc[i][j] = fmaf(a[i].y, b[j].y, acc[i][j]);
                acc[i][j] = fmaf(a[i].z, b[j].z, acc[i][j]);
                acc[i][j] = fmaf(a[i].w, b[j].w, acc[i][j]);
            }
    }
}

// Column c of a thread's D / 16 output columns: tx * 4 + (c % 4) + 64 (c / 4).
__device__ __forceinline__ int sm_col(int tx, int c) { return tx * 4 + (c & 3) + 64 * (c >> 2); }

// acc[i][c] += sum_j P[ty + 16 i][j] X[j][sm_col(tx, c)], j < 64 (P pitch kLP, X pitch D + 4)
template <int D>
__device__ __forceinline__ void mm_ab(const float* __restrict__ P, const float* __restrict__ X, int ty, int tx,
                                      float acc[4][D / 16]) {
    constexpr int LD = D + 4, CC = D / 64;
#pragma unroll 2
    for (int j = 0; j < kSB; j += 4) {
        float4 p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = *reinterpret_cast<const float4*>(P + (ty + 16 * i) * kLP + j);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            float4 x[CC];
#pragma unroll
            for (int cc = 0; cc < CC; ++cc) x[cc] = *reinterpret_cast<const float4*>(X + (j + jj) * LD + tx * 4 + 64 * cc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float pv = jj == 0 ? p[i].x : jj == 1 ? p[i].y : jj == 2 ? p[i].z : p[i].w;
#pragma unroll
                for (int cc = 0; cc < CC; ++cc) {
                    acc[i][4 * cc + 0] = fmaf(pv, x[cc].x, acc[i][4 * cc + 0]);
                    acc[i][4 * cc + 1] = fmaf(pv, x[cc].y, acc[i][4 * cc + 1]);
                    acc[i][4 * cc + 2] = fmaf(pv, x[cc].z, acc[i][4 * cc + 2]);
                    acc[i][4 * cc + 3] = fmaf(pv, x[cc].w, acc[i][4 * cc + 3]);
                }
            }
        }
    }
}

// rows [0, n) of a 64-row tile from global rows src + r * stride (fp32 copy), zeros below
template <int D, typename T>
__device__ __forceinline__ void load_tile(float* __restrict__ dst, const T* __restrict__ src, size_t stride, int n) {
    constexpr int LD = D + 4, V = D / 4;
    for (int idx = threadIdx.x; idx < kSB * V; idx += kSmThreads) {
        const int r = idx / V, c4 = (idx % V) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < n) {
            const T* s = src + (size_t)r * stride + c4;
            x = make_float4(to_f32(s[0]), to_f32(s[1]), to_f32(s[2]), to_f32(s[3]));
        }
        *reinterpret_cast<float4*>(dst + r * LD + c4) = x;
    }
}

__device__ __forceinline__ float max16(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// sequence of row block b: largest n with base[n] <= b
__device__ __forceinline__ int block_seq(const int32_t* __restrict__ base, int n_seqs, int b) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(base + mid) <= b) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// base[n] = sum over sequences i < n of ceil(len_i / 64); base[N] = the total.  One CTA of 1024 threads.
// Also checks cu_seqlens: 0 first, non-decreasing, total last (else kErrSeqlens).
__global__ void __launch_bounds__(1024) bwd_blocks_kernel(LayerDims L, const int32_t* __restrict__ cu,
                                                          int32_t* __restrict__ base, int32_t* __restrict__ err) {
    __shared__ int32_t part[1024];
    const int N = L.n_seqs, tid = threadIdx.x, per = (N + 1023) / 1024;
    const int lo = min(N, tid * per), hi = min(N, lo + per);
    int32_t s = 0;
    for (int i = lo; i < hi; ++i) {
        int64_t a, len;
        seq_range(cu, i, L.total, &a, &len);
        s += (int32_t)((len + kSB - 1) / kSB);
        if (__ldg(cu + i) > __ldg(cu + i + 1)) atomicExch(err, kErrSeqlens);
    }
    if (tid == 0 && (__ldg(cu) != 0 || (int64_t)__ldg(cu + N) != L.total)) atomicExch(err, kErrSeqlens);
    part[tid] = s;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const int32_t add = tid >= o ? part[tid - o] : 0;
        __syncthreads();
        part[tid] += add;
        __syncthreads();
    }
    int32_t run = tid > 0 ? part[tid - 1] : 0;
    for (int i = lo; i < hi; ++i) {
        base[i] = run;
        int64_t a, len;
        seq_range(cu, i, L.total, &a, &len);
        run += (int32_t)((len + kSB - 1) / kSB);
    }
    if (tid == 1023) base[N] = part[1023];
}

// Query-centric pass: CTA per (64-query block, q-head).  stats[(t Hq + h) 3 + {0, 1, 2}] = m, l, D of query t;
// dqr[t][h] = the softmax branch's gradient of the RoPE'd query; sink_k / sink_v[(b Hq + h) ns + j] = the
// block's partial dk (scaled) and dv of sink key j (rows j <= the block's last query).
template <typename Tin, int D>
__global__ void __launch_bounds__(kSmThreads)
bwd_sm_query_kernel(LayerDims L, const Tin* __restrict__ v, const Tin* __restrict__ dout,
                    const int32_t* __restrict__ cu, const int32_t* __restrict__ base, const float* __restrict__ qr,
                    const float* __restrict__ kr, float* __restrict__ stats, float* __restrict__ dqr,
                    float* __restrict__ sink_k, float* __restrict__ sink_v) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LD = D + 4, NC = D / 16;
    float* Qs = smem;
    float* dOs = Qs + kSB * LD;
    float* Ks = dOs + kSB * LD;
    float* Vs = Ks + kSB * LD;
    float* Ps = Vs + kSB * LD;   // P row-major (first pass); P^T of a sink tile (second pass)
    float* dSs = Ps + kSB * kLP; // dS row-major
    float* Ts = dSs + kSB * kLP; // dS^T of a sink tile
    const int b = blockIdx.x, h = blockIdx.y, kv = h / L.G, tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    if (b >= __ldg(base + L.n_seqs)) return;
    const int n = block_seq(base, L.n_seqs, b);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p0 = (int64_t)(b - __ldg(base + n)) * kSB;
    const int nq = (int)max((int64_t)0, min((int64_t)kSB, len - p0));
    if (nq == 0) return;
    const int ns = L.n_sinks, W = L.window;
    const float scale = rsqrtf((float)D);
    const bool sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF);
    const size_t qstride = (size_t)L.Hq * D, kstride = (size_t)L.Hkv * D;
    load_tile<D>(Qs, qr + ((size_t)(start + p0) * L.Hq + h) * D, qstride, nq);
    load_tile<D>(dOs, dout + ((size_t)(start + p0) * L.Hq + h) * D, qstride, nq);
    const int64_t p_last = p0 + nq - 1;
    const int64_t s_end = min((int64_t)ns, p_last + 1);
    const int64_t w_lo = max((int64_t)ns, p0 - W + 1), w_end = p_last + 1;
    const int n_sink_tiles = (int)((s_end + kSB - 1) / kSB);
    const int n_tiles = n_sink_tiles + (w_end > w_lo ? (int)((w_end - w_lo + kSB - 1) / kSB) : 0);
    auto tile = [&](int t, int64_t* j0, int* nk) {
        if (t < n_sink_tiles) {
            *j0 = (int64_t)t * kSB;
            *nk = (int)min((int64_t)kSB, s_end - *j0);
        } else {
            *j0 = w_lo + (int64_t)(t - n_sink_tiles) * kSB;
            *nk = (int)min((int64_t)kSB, w_end - *j0);
        }
    };
    auto visible = [&](int row, int col, int64_t j0, int nk) {
        const int64_t p = p0 + row, j = j0 + col;
        return row < nq && col < nk && j <= p && (j < ns || j >= p - W + 1);
    };
    auto load_kv = [&](int64_t j0, int nk) {
        __syncthreads();
        load_tile<D>(Ks, kr + ((size_t)(start + j0) * L.Hkv + kv) * D, kstride, nk);
        load_tile<D>(Vs, v + ((size_t)(start + j0) * L.Hkv + kv) * D, kstride, nk);
        __syncthreads();
    };

    // ---- first pass: m, l, o_sm (unnormalised) per row
    float m[4], l[4], O[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) O[i][c] = 0.f;
    }
    for (int t = 0; t < n_tiles; ++t) {
        int64_t j0;
        int nk;
        tile(t, &j0, &nk);
        load_kv(j0, nk);
        float s[4][4] = {};
        mm_abT<D>(Qs, Ks, ty, tx, s);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                s[i][j] = visible(ty + 16 * i, tx + 16 * j, j0, nk) ? s[i][j] * scale : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
            mx = max16(mx);
            const float mn = fmaxf(m[i], mx);
            const float basev = mn == -INFINITY ? 0.f : mn;
            const float r = m[i] == -INFINITY ? 0.f : expf(m[i] - basev);
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float e = expf(s[i][j] - basev);
                sum += e;
                Ps[(ty + 16 * i) * kLP + tx + 16 * j] = e;
            }
            l[i] = l[i] * r + sum16(sum);
            m[i] = mn;
#pragma unroll
            for (int c = 0; c < NC; ++c) O[i][c] *= r;
        }
        __syncthreads();
        mm_ab<D>(Ps, Vs, ty, tx, O);
    }
    float Dp[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) dot = fmaf(dOs[(ty + 16 * i) * LD + sm_col(tx, c)], O[i][c], dot);
        dot = sum16(dot);
        Dp[i] = l[i] > 0.f ? dot / l[i] : 0.f;
        const int row = ty + 16 * i;
        if (tx == 0 && row < nq) {
            float* st = stats + ((size_t)(start + p0 + row) * L.Hq + h) * 3;
            st[0] = m[i];
            st[1] = l[i];
            st[2] = Dp[i];
        }
    }
    // ---- second pass: dS = P (dP - D); dq += dS K; sink tiles: the block's dk = dS^T Q, dv = P^T dO
    float dq[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) dq[i][c] = 0.f;
    for (int t = 0; t < n_tiles; ++t) {
        int64_t j0;
        int nk;
        tile(t, &j0, &nk);
        const bool sink = t < n_sink_tiles;
        load_kv(j0, nk);
        float s[4][4] = {}, dp[4][4] = {};
        mm_abT<D>(Qs, Ks, ty, tx, s);
        mm_abT<D>(dOs, Vs, ty, tx, dp);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = ty + 16 * i, col = tx + 16 * j;
                const bool vis = sm_on && visible(row, col, j0, nk);
                const float P = vis ? expf(s[i][j] * scale - m[i]) / l[i] : 0.f;
                const float ds = P * (dp[i][j] - Dp[i]);
                dSs[row * kLP + col] = ds;
                if (sink) {
                    Ps[col * kLP + row] = P;
                    Ts[col * kLP + row] = ds;
                }
            }
        __syncthreads();
        mm_ab<D>(dSs, Ks, ty, tx, dq);
        if (sink) {
            float pk[4][NC], pv[4][NC];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < NC; ++c) pk[i][c] = pv[i][c] = 0.f;
            mm_ab<D>(Ts, Qs, ty, tx, pk);
            mm_ab<D>(Ps, dOs, ty, tx, pv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int key = ty + 16 * i;
                if (key < nk) {
                    const size_t o = (((size_t)b * L.Hq + h) * ns + j0 + key) * D;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        sink_k[o + sm_col(tx, c)] = pk[i][c] * scale;
                        sink_v[o + sm_col(tx, c)] = pv[i][c];
                    }
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = ty + 16 * i;
        if (row < nq) {
            float* o = dqr + ((size_t)(start + p0 + row) * L.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < NC; ++c) o[sm_col(tx, c)] = dq[i][c] * scale;
        }
    }
}

// Key-centric pass: CTA per (64-key block, q-head), the block's non-sink keys j; the queries that see j are
// p in [j, j + W - 1].  dkr_h[j][h] = scale sum_p dS_pj qr_p, dv_h[j][h] = sum_p P_pj dO_p.
template <typename Tin, int D>
__global__ void __launch_bounds__(kSmThreads)
bwd_sm_key_kernel(LayerDims L, const Tin* __restrict__ v, const Tin* __restrict__ dout,
                  const int32_t* __restrict__ cu, const int32_t* __restrict__ base, const float* __restrict__ qr,
                  const float* __restrict__ kr, const float* __restrict__ stats, float* __restrict__ dkr_h,
                  float* __restrict__ dv_h) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LD = D + 4, NC = D / 16;
    float* Ks = smem;
    float* Vs = Ks + kSB * LD;
    float* Qs = Vs + kSB * LD;
    float* dOs = Qs + kSB * LD;
    float* PT = dOs + kSB * LD;
    float* dST = PT + kSB * kLP;
    float* ms = dST + kSB * kLP;
    float* ls = ms + kSB;
    float* Ds = ls + kSB;
    const int b = blockIdx.x, h = blockIdx.y, kv = h / L.G, tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    if (b >= __ldg(base + L.n_seqs)) return;
    const int n = block_seq(base, L.n_seqs, b);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t k0 = (int64_t)(b - __ldg(base + n)) * kSB;
    const int nk = (int)max((int64_t)0, min((int64_t)kSB, len - k0));
    const int ns = L.n_sinks, W = L.window;
    const int64_t q_lo = max(k0, (int64_t)ns), q_hi = min(len, k0 + nk - 1 + W);
    if (q_lo >= k0 + nk) return;  // sink keys only: their sums come from the query blocks' partials
    const float scale = rsqrtf((float)D);
    const bool sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF);
    const size_t qstride = (size_t)L.Hq * D, kstride = (size_t)L.Hkv * D;
    load_tile<D>(Ks, kr + ((size_t)(start + k0) * L.Hkv + kv) * D, kstride, nk);
    load_tile<D>(Vs, v + ((size_t)(start + k0) * L.Hkv + kv) * D, kstride, nk);
    float dK[4][NC], dV[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) dK[i][c] = dV[i][c] = 0.f;
    for (int64_t q0 = q_lo; q0 < q_hi; q0 += kSB) {
        const int nq = (int)min((int64_t)kSB, q_hi - q0);
        __syncthreads();
        load_tile<D>(Qs, qr + ((size_t)(start + q0) * L.Hq + h) * D, qstride, nq);
        load_tile<D>(dOs, dout + ((size_t)(start + q0) * L.Hq + h) * D, qstride, nq);
        if (tid < kSB) {
            const bool ok = tid < nq;
            const float* st = stats + ((size_t)(start + q0 + (ok ? tid : 0)) * L.Hq + h) * 3;
            ms[tid] = ok ? st[0] : 0.f;
            ls[tid] = ok ? st[1] : 1.f;
            Ds[tid] = ok ? st[2] : 0.f;
        }
        __syncthreads();
        float s[4][4] = {}, dp[4][4] = {};
        mm_abT<D>(Qs, Ks, ty, tx, s);
        mm_abT<D>(dOs, Vs, ty, tx, dp);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = ty + 16 * i, col = tx + 16 * j;
                const int64_t p = q0 + row, key = k0 + col;
                const bool vis = sm_on && row < nq && col < nk && key >= ns && key <= p && p <= key + W - 1;
                const float P = vis ? expf(s[i][j] * scale - ms[row]) / ls[row] : 0.f;
                PT[col * kLP + row] = P;
                dST[col * kLP + row] = P * (dp[i][j] - Ds[row]);
            }
        __syncthreads();
        mm_ab<D>(dST, Qs, ty, tx, dK);
        mm_ab<D>(PT, dOs, ty, tx, dV);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = ty + 16 * i;
        const int64_t key = k0 + row;
        if (row < nk && key >= ns) {
            const size_t o = ((size_t)(start + key) * L.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                dkr_h[o + sm_col(tx, c)] = dK[i][c] * scale;
                dv_h[o + sm_col(tx, c)] = dV[i][c];
            }
        }
    }
}

// Sink keys: CTA per (sequence, q-head), thread per channel; the sums over the sequence's query blocks
// (those whose last query is at or after the key) of the partials.
__global__ void bwd_sm_sink_kernel(LayerDims L, const int32_t* __restrict__ cu, const int32_t* __restrict__ base,
                                   int n_blk, const float* __restrict__ sink_k, const float* __restrict__ sink_v,
                                   float* __restrict__ dkr_h, float* __restrict__ dv_h) {
    const int n = blockIdx.x, h = blockIdx.y, c = threadIdx.x, D = L.d, ns = L.n_sinks;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int b0 = __ldg(base + n), nb = (int)((len + kSB - 1) / kSB);
    for (int64_t j = 0; j < min((int64_t)ns, len); ++j) {
        float sk = 0.f, sv = 0.f;
        for (int qb = 0; qb < nb && b0 + qb < n_blk; ++qb) {
            if (j > min(len, (int64_t)(qb + 1) * kSB) - 1) continue;
            const size_t o = (((size_t)(b0 + qb) * L.Hq + h) * ns + j) * D + c;
            sk += sink_k[o];
            sv += sink_v[o];
        }
        const size_t o = ((size_t)(start + j) * L.Hq + h) * D + c;
        dkr_h[o] = sk;
        dv_h[o] = sv;
    }
}

// ---- 5. feature backward: rows r < Hq are q-heads, < Hq + Hkv k-heads, else v-heads; thread per channel.
// First the L2 backward into d(pre-norm) (kind-specific inputs), written over dpre; the conv and RoPE
// backward then run in bwd_feat_out_kernel.
__global__ void bwd_l2_kernel(LayerDims L, const int32_t* __restrict__ cu, const float* __restrict__ qt,
                              const float* __restrict__ kt, const float* __restrict__ dqh,
                              const float* __restrict__ dkh_h, const float* __restrict__ dvh_h,
                              float* __restrict__ dqt, float* __restrict__ dkt, float* __restrict__ dvt) {
    __shared__ float red[32];
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    if (kind == 2) {  // vhat = conv(v): the per-head gradients of the group summed
        float s = 0.f;
        for (int gq = 0; gq < L.G; ++gq) s += dvh_h[((size_t)t * L.Hq + hh * L.G + gq) * D + c];
        dvt[((size_t)t * L.Hkv + hh) * D + c] = s;
        return;
    }
    float dyh;
    const float* pre;
    if (kind == 0) {
        dyh = dqh[((size_t)t * L.Hq + hh) * D + c];
        pre = qt + ((size_t)t * L.Hq + hh) * D;
    } else {
        dyh = 0.f;
        for (int gq = 0; gq < L.G; ++gq) dyh += dkh_h[((size_t)t * L.Hq + hh * L.G + gq) * D + c];
        pre = kt + ((size_t)t * L.Hkv + hh) * D;
    }
    const bool norm = kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q);
    float dx = dyh;
    if (norm) {  // y = x / nrm, nrm = sqrt(|x|^2 + eps): dx = (dy - x (x . dy) / nrm^2) / nrm
        const float x = pre[c];
        const float n2 = cta_sum_f(x * x, red) + 1e-6f;
        const float xd = cta_sum_f(x * dyh, red);
        dx = (dyh - x * xd / n2) * rsqrtf(n2);
    }
    (kind == 0 ? dqt : dkt)[((size_t)t * (kind == 0 ? L.Hq : L.Hkv) + hh) * D + c] = dx;
}

// conv backward (the taps that read position p, from the later positions of the same sequence),
// plus the softmax branch's gradient, then RoPE's transpose; writes dq, dk, dv
__global__ void bwd_feat_out_kernel(LayerDims L, const int32_t* __restrict__ cu, const float* __restrict__ wq,
                                    const float* __restrict__ wk, const float* __restrict__ wv,
                                    const float* __restrict__ dqt, const float* __restrict__ dkt,
                                    const float* __restrict__ dvt, const float* __restrict__ dqr_sm,
                                    const float* __restrict__ dkr_h, const float* __restrict__ dv_h,
                                    float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv) {
    __shared__ float gx[128];
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d, half = D / 2;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* w = (kind == 0 ? wq : kind == 1 ? wk : wv) + ((size_t)hh * D + c) * kConvWidth;
    const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
    // x_p feeds y_{p + 7 - m} through tap m
    float acc = 0.f;
    for (int m = 0; m < kConvWidth; ++m) {
        const int64_t pp = p + (kConvWidth - 1) - m;
        if (pp >= len) continue;
        acc = fmaf(w[m], dy[((size_t)(start + pp) * H + hh) * D + c], acc);
    }
    // the softmax branch's gradient of the RoPE'd row (q, k) or of raw v, summed over the group for k, v
    if (kind == 0) {
        acc += dqr_sm[((size_t)t * L.Hq + hh) * D + c];
    } else {
        for (int gq = 0; gq < L.G; ++gq) acc += (kind == 1 ? dkr_h : dv_h)[((size_t)t * L.Hq + hh * L.G + gq) * D + c];
    }
    if (kind == 2) {
        dv[((size_t)t * L.Hkv + hh) * D + c] = acc;
        return;
    }
    // RoPE's transpose: rotate the pair (i, i + D/2) back by the angle p theta_i
    gx[c] = acc;
    __syncthreads();
    const int i = c % half;
    float cs, sn;
    rope_cs_exact(p, L.theta[i], &cs, &sn);
    const float g1 = gx[i], g2 = gx[i + half];
    (kind == 0 ? dq : dk)[((size_t)t * H + hh) * D + c] = c < half ? g1 * cs + g2 * sn : g2 * cs - g1 * sn;
}

// ---- 6. conv filters: partial sums over a block of kWB tokens, per (row, channel, tap); then the blocks
template <typename Tin>
__global__ void bwd_convw_part_kernel(LayerDims L, const Tin* __restrict__ v, const int32_t* __restrict__ cu,
                                      const float* __restrict__ qr, const float* __restrict__ kr,
                                      const float* __restrict__ dqt, const float* __restrict__ dkt,
                                      const float* __restrict__ dvt, float* __restrict__ part) {
    const int blk = blockIdx.x, r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
    float acc[kConvWidth];
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) acc[m] = 0.f;
    const int64_t t0 = (int64_t)blk * kWB, t1 = min(L.total, t0 + kWB);
    for (int64_t t = t0; t < t1; ++t) {
        const int n = seq_of_token(cu, L.n_seqs, t);
        int64_t start, len;
        seq_range(cu, n, L.total, &start, &len);
        const int64_t p = t - start;
        const float d_y = dy[((size_t)t * H + hh) * D + c];
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) {
            const int64_t pp = p - (kConvWidth - 1) + m;
            if (pp < 0) continue;
            const size_t row = ((size_t)(start + pp) * H + hh) * D + c;
            const float x = kind == 0 ? qr[row] : kind == 1 ? kr[row] : to_f32(v[row]);
            acc[m] = fmaf(d_y, x, acc[m]);
        }
    }
    const int rows = L.Hq + 2 * L.Hkv;
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) part[(((size_t)blk * rows + r) * D + c) * kConvWidth + m] = acc[m];
}

__global__ void bwd_convw_sum_kernel(LayerDims L, int n_blocks, const float* __restrict__ part,
                                     float* __restrict__ dwq, float* __restrict__ dwk, float* __restrict__ dwv) {
    const int r = blockIdx.x, c = threadIdx.x, D = L.d, rows = L.Hq + 2 * L.Hkv;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    float* dw = (kind == 0 ? dwq : kind == 1 ? dwk : dwv) + ((size_t)hh * D + c) * kConvWidth;
    for (int m = 0; m < kConvWidth; ++m) {
        float s = 0.f;
        for (int b = 0; b < n_blocks; ++b) s += part[(((size_t)b * rows + r) * D + c) * kConvWidth + m];
        dw[m] = s;
    }
}

// ---- 7. lambda: partial sums over the sequences
__global__ void bwd_lambda_kernel(LayerDims L, const float* __restrict__ part, float* __restrict__ dlam) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= L.Hq) return;
    float s = 0.f;
    for (int n = 0; n < L.n_seqs; ++n) s += part[(size_t)n * L.Hq + h];
    dlam[h] = s;
}

}  // namespace

BwdLayout bwd_layout(const LayerDims& L) {
    BwdLayout b;
    const size_t T = (size_t)L.total, Hq = (size_t)L.Hq, Hkv = (size_t)L.Hkv, D = (size_t)L.d, N = (size_t)L.n_seqs;
    const size_t rows = Hq + 2 * Hkv, nblk = (T + kWB - 1) / kWB;
    const size_t spb = (size_t)kCkB / (L.d == 128 ? GdnB<128>::K : GdnB<64>::K);
    size_t off = 256;  // bytes 0..15: the device error word
    b.err = 0;
    auto take = [&](size_t floats) {
        const size_t o = off;
        off = (off + floats * sizeof(float) + 255) / 256 * 256;
        return o;
    };
    b.qr = take(T * Hq * D);
    b.kr = take(T * Hkv * D);
    b.qt = take(T * Hq * D);
    b.qh = take(T * Hq * D);
    b.kt = take(T * Hkv * D);
    b.kh = take(T * Hkv * D);
    b.vh = take(T * Hkv * D);
    b.dqh = take(T * Hq * D);
    b.dkh_h = take(T * Hq * D);
    b.dvh_h = take(T * Hq * D);
    b.dqr_sm = take(T * Hq * D);
    b.dkr_h = take(T * Hq * D);
    b.dv_h = take(T * Hq * D);
    b.dqt = take(T * Hq * D);
    b.dkt = take(T * Hkv * D);
    b.dvt = take(T * Hkv * D);
    b.stats = take(T * Hq * 3);
    b.ckpt = take((T / kCkB + N + 1) * Hq * D * D);  // S every 64 absorptions of every sequence and q-head
    b.sub = take(N * Hq * spb * D * D);               // S every stage of one 64-absorption block
    b.dlam_part = take(N * Hq);
    b.convw_part = take(nblk * rows * D * kConvWidth);
    b.n_blocks = (int)nblk;
    b.n_sm_blocks = (int)(T / kSB + N);                // bounds the 64-row softmax blocks of all sequences
    b.sm_base = take(N + 1);                           // int32
    b.sink_k = take((size_t)b.n_sm_blocks * Hq * (size_t)L.n_sinks * D);
    b.sink_v = take((size_t)b.n_sm_blocks * Hq * (size_t)L.n_sinks * D);
    b.total = off;
    return b;
}

template <typename Tin, int D>
cudaError_t launch_gdn_bwd(const LayerDims& L, const float* g, const float* beta, const float* lambda,
                           const Tin* dout, const int32_t* cu, const float* qh, const float* kh, const float* vh,
                           float* ckpt, float* sub, float* dqh, float* dkh_h, float* dvh_h, float* dg, float* dbeta,
                           float* dlam_part, cudaStream_t st) {
    static DeviceCache cache;  // the shared-memory attribute, per device
    const size_t bytes = GdnB<D>::BYTES;
    cudaError_t e = device_cached(cache, nullptr, [&](int, int*) {
        return cudaFuncSetAttribute(bwd_gdn_kernel<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCl * L.Hq, L.n_seqs);
    cfg.blockDim = dim3(kGT);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_gdn_kernel<Tin, D>, L, g, beta, lambda, dout, cu, qh, kh, vh, ckpt, sub, dqh,
                              dkh_h, dvh_h, dg, dbeta, dlam_part);
}

template <typename Tin, int D>
cudaError_t launch_sm_bwd(const LayerDims& L, const Tin* v, const Tin* dout, const int32_t* cu, const int32_t* base,
                          int n_blk, const float* qr, const float* kr, float* stats, float* dqr, float* dkr_h,
                          float* dv_h, float* sink_k, float* sink_v, cudaStream_t st) {
    static DeviceCache cache;  // the shared-memory attributes, per device
    const size_t bq = sm_smem_bytes<D>(3), bk = sm_smem_bytes<D>(2);
    cudaError_t e = device_cached(cache, nullptr, [&](int, int*) {
        cudaError_t r = cudaFuncSetAttribute(bwd_sm_query_kernel<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bq);
        if (r != cudaSuccess) return r;
        return cudaFuncSetAttribute(bwd_sm_key_kernel<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bk);
    });
    if (e != cudaSuccess) return e;
    bwd_sm_query_kernel<Tin, D><<<dim3(n_blk, L.Hq), kSmThreads, bq, st>>>(L, v, dout, cu, base, qr, kr, stats, dqr,
                                                                           sink_k, sink_v);
    bwd_sm_key_kernel<Tin, D><<<dim3(n_blk, L.Hq), kSmThreads, bk, st>>>(L, v, dout, cu, base, qr, kr, stats, dkr_h,
                                                                         dv_h);
    if (L.n_sinks > 0)
        bwd_sm_sink_kernel<<<dim3(L.n_seqs, L.Hq), D, 0, st>>>(L, cu, base, n_blk, sink_k, sink_v, dkr_h, dv_h);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_backward(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* g,
                            const float* beta, const float* lambda, const float* wq, const float* wk, const float* wv,
                            const int32_t* cu, const Tin* dout, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, float* dlam, float* dwq, float* dwk, float* dwv, char* ws,
                            const BwdLayout& b, const cudaEvent_t* marks, int n_marks, cudaStream_t st) {
    auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    auto mark = [&](int i) { return i < n_marks && marks[i] ? cudaEventRecord(marks[i], st) : cudaSuccess; };
    const size_t T = (size_t)L.total;
    const int D = L.d, rows = L.Hq + 2 * L.Hkv;
    cudaError_t e;
    // tokens that no state absorbs keep zero gradients of g, beta, khat, vhat
    if ((e = cudaMemsetAsync(dg, 0, T * L.Hq * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dbeta, 0, T * L.Hq * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(F(b.dkh_h), 0, T * L.Hq * D * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(F(b.dvh_h), 0, T * L.Hq * D * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(F(b.dqh), 0, T * L.Hq * D * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(ws + b.err, 0, 16, st)) != cudaSuccess) return e;
    if ((e = mark(0)) != cudaSuccess) return e;
    int32_t* sm_base = reinterpret_cast<int32_t*>(ws + b.sm_base);
    bwd_blocks_kernel<<<1, 1024, 0, st>>>(L, cu, sm_base, reinterpret_cast<int32_t*>(ws + b.err));
    bwd_rope_kernel<Tin><<<dim3((unsigned)T, L.Hq + L.Hkv), D, 0, st>>>(L, q, k, cu, F(b.qr), F(b.kr),
                                                                        reinterpret_cast<int32_t*>(ws + b.err));
    if ((e = mark(1)) != cudaSuccess) return e;
    bwd_conv_kernel<Tin><<<dim3((unsigned)T, rows), D, 0, st>>>(L, v, wq, wk, wv, cu, F(b.qr), F(b.kr), F(b.qt), F(b.qh),
                                                                F(b.kt), F(b.kh), F(b.vh));
    if ((e = mark(2)) != cudaSuccess) return e;
    e = D == 128 ? launch_gdn_bwd<Tin, 128>(L, g, beta, lambda, dout, cu, F(b.qh), F(b.kh), F(b.vh), F(b.ckpt),
                                            F(b.sub), F(b.dqh), F(b.dkh_h), F(b.dvh_h), dg, dbeta, F(b.dlam_part), st)
                 : launch_gdn_bwd<Tin, 64>(L, g, beta, lambda, dout, cu, F(b.qh), F(b.kh), F(b.vh), F(b.ckpt),
                                           F(b.sub), F(b.dqh), F(b.dkh_h), F(b.dvh_h), dg, dbeta, F(b.dlam_part), st);
    if (e != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    e = D == 128 ? launch_sm_bwd<Tin, 128>(L, v, dout, cu, sm_base, b.n_sm_blocks, F(b.qr), F(b.kr), F(b.stats),
                                           F(b.dqr_sm), F(b.dkr_h), F(b.dv_h), F(b.sink_k), F(b.sink_v), st)
                 : launch_sm_bwd<Tin, 64>(L, v, dout, cu, sm_base, b.n_sm_blocks, F(b.qr), F(b.kr), F(b.stats),
                                          F(b.dqr_sm), F(b.dkr_h), F(b.dv_h), F(b.sink_k), F(b.sink_v), st);
    if (e != cudaSuccess) return e;
    if ((e = mark(4)) != cudaSuccess) return e;
    bwd_l2_kernel<<<dim3((unsigned)T, rows), D, 0, st>>>(L, cu, F(b.qt), F(b.kt), F(b.dqh), F(b.dkh_h), F(b.dvh_h),
                                                         F(b.dqt), F(b.dkt), F(b.dvt));
    if ((e = mark(5)) != cudaSuccess) return e;
    bwd_feat_out_kernel<<<dim3((unsigned)T, rows), D, 0, st>>>(L, cu, wq, wk, wv, F(b.dqt), F(b.dkt), F(b.dvt),
                                                               F(b.dqr_sm), F(b.dkr_h), F(b.dv_h), dq, dk, dv);
    if ((e = mark(6)) != cudaSuccess) return e;
    bwd_convw_part_kernel<Tin><<<dim3(b.n_blocks, rows), D, 0, st>>>(L, v, cu, F(b.qr), F(b.kr), F(b.dqt), F(b.dkt),
                                                                      F(b.dvt), F(b.convw_part));
    bwd_convw_sum_kernel<<<rows, D, 0, st>>>(L, b.n_blocks, F(b.convw_part), dwq, dwk, dwv);
    if ((e = mark(7)) != cudaSuccess) return e;
    bwd_lambda_kernel<<<(L.Hq + 127) / 128, 128, 0, st>>>(L, F(b.dlam_part), dlam);
    if ((e = mark(8)) != cudaSuccess) return e;
    return cudaGetLastError();
}

template cudaError_t launch_backward<float>(const LayerDims&, const float*, const float*, const float*, const float*,
                                            const float*, const float*, const float*, const float*, const float*,
                                            const int32_t*, const float*, float*, float*, float*, float*, float*,
                                            float*, float*, float*, float*, char*, const BwdLayout&, const cudaEvent_t*, int,
                                            cudaStream_t);
template cudaError_t launch_backward<__nv_bfloat16>(const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*,
                                                    const __nv_bfloat16*, const float*, const float*, const float*,
                                                    const float*, const float*, const float*, const int32_t*,
                                                    const __nv_bfloat16*, float*, float*, float*, float*, float*,
                                                    float*, float*, float*, float*, char*, const BwdLayout&,
                                                    const cudaEvent_t*, int, cudaStream_t);

}  // namespace hla
