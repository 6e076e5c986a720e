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
//  1. rope: RoPE'd q and k rows (fp32) for every token and head; alpha = e^g;
//  2. conv: q~, k~ (and their L2-normalised qhat, khat) and vhat = conv(v);
//  3. GDN, a cluster of 8 CTAs per (sequence, q-head) splitting the value
//     columns: a forward pass that keeps the state every 64 absorptions, then
//     per 64-absorption block, last first, the states every 4 (d 128) or 8
//     (d 64) absorptions, and per such stage the states in registers and the
//     read-out and absorption steps differentiated in reverse (dqhat, lambda's
//     partial sum, and per head dkhat, dvhat, dg, dbeta);
//  4. softmax: per 64-query block the rows' max, sum and D = dO . o_sm and dq;
//     per 64-key block dk, dv of its non-sink keys; the sink keys' sums over
//     the query blocks' partials;
//  5. feature backward of q (L2, conv, RoPE); of k and v after the per-head
//     gradients of each kv group are summed;
//  6. the conv filters' gradients (per token block, then over the blocks);
//  7. lambda's gradient over the sequences.
#include <type_traits>

#include "hla_common.cuh"

namespace hla {

namespace {

constexpr int kWB = 64;     // tokens per block of the conv-filter reduction

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// cos/sin of p theta_i, i < d / 2, for one position, into shared memory (threads < d / 2)
__device__ __forceinline__ void angles(const LayerDims& L, int64_t p, float* cs, float* sn) {
    if ((int)threadIdx.x < L.d / 2) rope_cs_exact(p, L.theta[threadIdx.x], &cs[threadIdx.x], &sn[threadIdx.x]);
    __syncthreads();
}

// ---- 1. RoPE'd rows: CTA per token; rows r < Hq are q-heads, the rest k-heads; a thread per channel pair
constexpr int kRowThreads = 256;
template <typename Tin>
__global__ void __launch_bounds__(kRowThreads)
bwd_rope_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k, const float* __restrict__ g,
                const int32_t* __restrict__ cu, float* __restrict__ qr, float* __restrict__ kr,
                float* __restrict__ alpha, int32_t* __restrict__ err) {
    __shared__ float cs[64], sn[64];
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x, D = L.d, half = D / 2;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    // a token outside every sequence: cu_seqlens is not a monotone table from 0 to total
    if ((p < 0 || p >= len) && tid == 0) atomicExch(err, kErrSeqlens);
    for (int h = tid; h < L.Hq; h += kRowThreads) alpha[t * L.Hq + h] = expf(g[t * L.Hq + h]);  // alpha = e^g
    angles(L, p, cs, sn);
    for (int idx = tid; idx < (L.Hq + L.Hkv) * half; idx += kRowThreads) {
        const int r = idx / half, i = idx % half;
        const bool isq = r < L.Hq;
        const size_t row = isq ? (size_t)t * L.Hq + r : (size_t)t * L.Hkv + (r - L.Hq);
        const Tin* x = (isq ? q : k) + row * D;
        float* y = (isq ? qr : kr) + row * D;
        const float x1 = to_f32(x[i]), x2 = to_f32(x[i + half]);
        y[i] = x1 * cs[i] - x2 * sn[i];
        y[i + half] = x2 * cs[i] + x1 * sn[i];
    }
}

// ---- 2. conv (+ L2): CTA per token, a warp per row (rows r < Hq: q-heads, < Hq + Hkv: k-heads, else
// v-heads), lane l holding channels l + 32 e
template <typename Tin, int D>
__global__ void __launch_bounds__(kRowThreads)
bwd_conv_kernel(LayerDims L, const Tin* __restrict__ v, const float* __restrict__ wq, const float* __restrict__ wk,
                const float* __restrict__ wv, const int32_t* __restrict__ cu, const float* __restrict__ qr,
                const float* __restrict__ kr, float* __restrict__ qt, float* __restrict__ qh,
                float* __restrict__ kt, float* __restrict__ kh, float* __restrict__ vh) {
    constexpr int E = D / 32;
    const int64_t t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    for (int r = warp; r < L.Hq + 2 * L.Hkv; r += kRowThreads / 32) {
        const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
        const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
        const int H = kind == 0 ? L.Hq : L.Hkv;
        const float* w = (kind == 0 ? wq : kind == 1 ? wk : wv) + (size_t)hh * D * kConvWidth;
        float acc[E], wt[E][kConvWidth];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            acc[e] = 0.f;
            const float4* w4 = reinterpret_cast<const float4*>(w + (size_t)(lane + 32 * e) * kConvWidth);
            const float4 a = w4[0], b = w4[1];
            wt[e][0] = a.x; wt[e][1] = a.y; wt[e][2] = a.z; wt[e][3] = a.w;
            wt[e][4] = b.x; wt[e][5] = b.y; wt[e][6] = b.z; wt[e][7] = b.w;
        }
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) {
            const int64_t pp = p - (kConvWidth - 1) + m;
            if (pp < 0) continue;
            const size_t row = ((size_t)(start + pp) * H + hh) * D;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int c = lane + 32 * e;
                const float x = kind == 0 ? qr[row + c] : kind == 1 ? kr[row + c] : to_f32(v[row + c]);
                acc[e] = fmaf(wt[e][m], x, acc[e]);
            }
        }
        const size_t o = ((size_t)t * H + hh) * D;
        if (kind == 2) {
#pragma unroll
            for (int e = 0; e < E; ++e) vh[o + lane + 32 * e] = acc[e];
            continue;
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(acc[e], acc[e], ss);
        const bool norm = kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q);
        const float inv = norm ? rsqrtf(warp_sum_f(ss) + 1e-6f) : 1.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            (kind == 0 ? qt : kt)[o + lane + 32 * e] = acc[e];
            (kind == 0 ? qh : kh)[o + lane + 32 * e] = acc[e] * inv;
        }
    }
}

// ---- 3. GDN backward: a cluster of kCl CTAs per (q-head, sequence), each CTA D / kCl value columns of S
// (the columns of the recurrence are independent: only the gradients of q, k, alpha and beta sum over
// them).  Eight lanes share a column, lane l holding rows 32 e + 4 (l % 8) + i (i < 4) of it in registers,
// so a dot product over the key dim ends in three shuffle rounds that serve the warp's four columns at
// once.  Three passes over the absorptions, all fed by one schedule of K-token stages loaded ahead with
// cp.async:
//   0: forward: S every 64 absorptions to the global checkpoints;
//   1: per 64-absorption block, last block first: from its checkpoint, S every K absorptions to a
//      per-(sequence, head) scratch (stays in L2);
//   2: the same block's stages, last first: the K + 1 states from the scratch state, in registers; then
//      the read-out and absorption steps differentiated in reverse.  Per stage the columns' contributions
//      to dq, dk, dalpha, dbeta are summed in the CTA, then over the cluster's CTAs through distributed
//      shared memory (one cluster barrier per stage, double-buffered); dv is per column.  lambda's
//      gradient sum_p dO_p . o_lin,p is sum_p qhat_p . (S_p dO_p), from the same sums.
constexpr int kCl = 8;      // CTAs per cluster
constexpr int kCkB = 64;    // absorptions per global checkpoint
constexpr int kRing = 3;    // stages in flight
constexpr int kXB = 4;      // stages per cluster exchange
template <int D> struct GdnB {
    static constexpr int LPC = 8, E = D / LPC, CPW = 32 / LPC;  // lanes per column, rows per lane, columns per warp
    static constexpr int CPC = D / kCl, NW = CPC / CPW, NT = NW * 32;
    static constexpr int K = D == 128 ? 4 : 8;  // absorptions per stage (the states of one stage in registers)
    static constexpr int SPB = kCkB / K;
    // shared memory (floats): column partials, cluster exchange (2 buffers), stage ring, dv of a stage, sums
    static constexpr int PART = K * 2 * CPC * D, SPART = K * 2 * CPC;
    static constexpr int XCH = 2 * kXB * K * 2 * D, XS = 2 * kXB * K * 2, XM = 2 * kXB * 2;
    static constexpr int SLOT = 2 * K * D + 2 * K * CPC + 2 * K;  // k, q rows; v, dO columns; alpha, beta
    static constexpr size_t BYTES =
        (size_t)(PART + SPART + XCH + XS + XM + kRing * SLOT + K * CPC + NW + 4) * 4;
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

// the sum over the 8 lanes of a column (lanes differing in bits 0-2), for N values at once
template <int N>
__device__ __forceinline__ void col_sum(float (&x)[N]) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
}
// this lane's E rows of a D-vector in shared memory: rows 32 e + 4 lr + i
template <int D>
__device__ __forceinline__ void lane_rows(const float* __restrict__ src, int lr, float* x) {
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
        const float4 v = *reinterpret_cast<const float4*>(src + 32 * e + 4 * lr);
        x[4 * e] = v.x;
        x[4 * e + 1] = v.y;
        x[4 * e + 2] = v.z;
        x[4 * e + 3] = v.w;
    }
}
template <int D>
__device__ __forceinline__ void lane_rows_store(float* __restrict__ dst, int lr, const float* x) {
#pragma unroll
    for (int e = 0; e < D / 32; ++e)
        *reinterpret_cast<float4*>(dst + 32 * e + 4 * lr) = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
}

template <typename Tin, int D>
__global__ void __launch_bounds__(GdnB<D>::NT)
bwd_gdn_kernel(LayerDims L, const float* __restrict__ alpha, const float* __restrict__ beta,
               const float* __restrict__ lambda, const Tin* __restrict__ dout, const int32_t* __restrict__ cu,
               const float* __restrict__ qh, const float* __restrict__ kh, const float* __restrict__ vh,
               float* __restrict__ ckpt, float* __restrict__ sub, float* __restrict__ dqh,
               float* __restrict__ dkh_h, float* __restrict__ dvh_h, float* __restrict__ dg,
               float* __restrict__ dbeta, float* __restrict__ dlam_part) {
    using B = GdnB<D>;
    constexpr int K = B::K, E = B::E, CPC = B::CPC, SPB = B::SPB, NT = B::NT, NW = B::NW;
    extern __shared__ __align__(16) float smem[];
    float* part = smem;                 // [K][2][CPC][D]: dq (S dO, unscaled) and dk contributions per column
    float* spart = part + B::PART;      // [K][2][CPC]: dalpha, dbeta
    float* xch = spart + B::SPART;      // [2][kXB][K][2][D]: the CTA's sums of up to kXB stages
    float* xs = xch + B::XCH;           // [2][kXB][K][2]: dg (alpha applied), dbeta
    int* xm = reinterpret_cast<int*>(xs + B::XS);  // [2][kXB][2]: each stage's first absorption and count
    float* ring = xs + B::XS + B::XM;   // kRing stage slots
    float* dv_s = ring + kRing * B::SLOT;  // [K][CPC]
    float* red = dv_s + K * CPC;        // [NW] + 1
    const uint32_t rank = cluster_rank();
    const int h = blockIdx.x / kCl, n = blockIdx.y, kv = h / L.G, tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31, lr = lane & 7;
    const int colL = w * B::CPW + (lane >> 3);            // this lane's column in the CTA
    const int col = (int)rank * CPC + colL;               // and in S
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
    float* ck_col_base = ckpt + (size_t)col * D;
    auto ck_col = [&](int blk) { return ck_col_base + ((size_t)(ck0 + blk) * L.Hq + h) * DD; };
    auto sub_col = [&](int si) { return my_sub + (size_t)si * DD + (size_t)col * D; };

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
    // slot layout: k [K][D], q [K][D], v [K][CPC], dO [K][CPC] (Tin), alpha [K], beta [K]
    auto slot_k = [&](int sl) { return ring + sl * B::SLOT; };
    auto slot_q = [&](int sl) { return ring + sl * B::SLOT + K * D; };
    auto slot_v = [&](int sl) { return ring + sl * B::SLOT + 2 * K * D; };
    auto slot_o = [&](int sl) { return reinterpret_cast<Tin*>(ring + sl * B::SLOT + 2 * K * D + K * CPC); };
    auto slot_a = [&](int sl) { return ring + sl * B::SLOT + 2 * K * D + 2 * K * CPC; };
    auto slot_b = [&](int sl) { return ring + sl * B::SLOT + 2 * K * D + 2 * K * CPC + K; };
    auto issue = [&](int i) {
        if (i < n_sched) {
            int phase, s;
            sched(i, &phase, &s);
            const int sl = i % kRing;
            const int64_t m0 = (int64_t)s * K;
            const int cnt = (int)min((int64_t)K, n_abs - m0);
            const int64_t j0 = start + ns + m0;  // global row of the stage's first absorbed token
            for (int idx = tid; idx < K * (D / 4); idx += NT) {
                const int t = idx / (D / 4), c = (idx % (D / 4)) * 4;
                if (t < cnt) {
                    cp_async(slot_k(sl) + t * D + c, kh + ((size_t)(j0 + t) * L.Hkv + kv) * D + c, 16);
                    if (phase == 2)
                        cp_async(slot_q(sl) + t * D + c, qh + ((size_t)(j0 + t + W) * L.Hq + h) * D + c, 16);
                }
            }
            for (int idx = tid; idx < K * (CPC / 4); idx += NT) {
                const int t = idx / (CPC / 4), c = (idx % (CPC / 4)) * 4;
                if (t < cnt)
                    cp_async(slot_v(sl) + t * CPC + c, vh + ((size_t)(j0 + t) * L.Hkv + kv) * D + rank * CPC + c, 16);
            }
            constexpr int OCH = CPC * (int)sizeof(Tin) / 16;  // 16-byte chunks of a dO row slice
            if (phase == 2) {
                for (int idx = tid; idx < K * OCH; idx += NT) {
                    const int t = idx / OCH, c = (idx % OCH) * (16 / (int)sizeof(Tin));
                    if (t < cnt)
                        cp_async(slot_o(sl) + t * CPC + c, dout + ((size_t)(j0 + t + W) * L.Hq + h) * D + rank * CPC + c,
                                 16);
                }
            }
            if (tid < cnt) {
                cp_async(slot_a(sl) + tid, alpha + (size_t)(j0 + tid) * L.Hq + h, 4);
                cp_async(slot_b(sl) + tid, beta + (size_t)(j0 + tid) * L.Hq + h, 4);
            }
        }
        cp_async_commit();
    };
    // one absorption of stage token t into S (registers)
    auto absorb = [&](float (&S)[E], int sl, int t) {
        float k[E];
        lane_rows<D>(slot_k(sl) + t * D, lr, k);
        float xp[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < E; ++e) xp[e & 1] = fmaf(k[e], S[e], xp[e & 1]);
        float x[1] = {xp[0] + xp[1]};
        col_sum<1>(x);
        const float a = slot_a(sl)[t], b = slot_b(sl)[t], vv = slot_v(sl)[t * CPC + colL];
        const float u = gla ? vv : b * (vv - a * x[0]);
#pragma unroll
        for (int e = 0; e < E; ++e) S[e] = fmaf(a, S[e], k[e] * u);
    };

    float S[E], dS[E];
#pragma unroll
    for (int e = 0; e < E; ++e) S[e] = dS[e] = 0.f;
    float dl = 0.f;
    int buf = 0, nx = 0;  // exchange buffer, stages in it
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
        // a full stage (cnt == K, all but a sequence's last) runs without per-token tests, so that the
        // compiler can overlap one token's loads with the previous token's chain

        // the stage's states S_{m0} .. S_{m0 + cnt}, then the read-out and absorption steps in reverse
        auto reverse_stage = [&](auto full) {
            constexpr bool FULL = decltype(full)::value;
            float St[K + 1][E];
            lane_rows<D>(sub_col(si), lr, St[0]);
#pragma unroll
            for (int t = 0; t < K; ++t) {
#pragma unroll
                for (int e = 0; e < E; ++e) St[t + 1][e] = St[t][e];
                if (FULL || t < cnt) absorb(St[t + 1], sl, t);
            }
#pragma unroll
            for (int tt = 0; tt < K; ++tt) {
                const int t = K - 1 - tt;
                if (FULL || t < cnt) {
                    float k[E], q[E];
                    lane_rows<D>(slot_k(sl) + t * D, lr, k);
                    lane_rows<D>(slot_q(sl) + t * D, lr, q);
                    const float dor = to_f32(slot_o(sl)[t * CPC + colL]), ldo = lam * dor;
                    const float vv = slot_v(sl)[t * CPC + colL];
                    const float a = slot_a(sl)[t], b = slot_b(sl)[t];
                    // read-out at p: o_lin = S_{m+1}^T qhat -> (S_{m+1} dO) to the partials, dS += qhat lambda dO^T
                    float pq[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) pq[e] = St[t + 1][e] * dor;
                    lane_rows_store<D>(part + ((t * 2 + 0) * CPC + colL) * D, lr, pq);
#pragma unroll
                    for (int e = 0; e < E; ++e) dS[e] = fmaf(q[e], ldo, dS[e]);
                    // absorption of token j from S_prev = S_m
                    float r6[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        r6[(e & 1)] = fmaf(k[e], St[t][e], r6[(e & 1)]);
                        r6[2 + (e & 1)] = fmaf(k[e], dS[e], r6[2 + (e & 1)]);
                        r6[4 + (e & 1)] = fmaf(dS[e], St[t][e], r6[4 + (e & 1)]);
                    }
                    float r3[3] = {r6[0] + r6[1], r6[2] + r6[3], r6[4] + r6[5]};
                    col_sum<3>(r3);
                    const float x = r3[0], du = r3[1], gs = r3[2];
                    const float u = gla ? vv : b * (vv - a * x);
                    if (lr == 0) {
                        dv_s[t * CPC + colL] = gla ? du : b * du;
                        spart[(t * 2 + 0) * CPC + colL] = gs - (gla ? 0.f : b * du * x);
                        spart[(t * 2 + 1) * CPC + colL] = gla ? 0.f : du * (vv - a * x);
                    }
                    // dk = dS u - a b S_prev du (GLA: dS v); dS_prev = a (dS - b k du^T) (GLA: a dS)
                    float pk[E];
                    const float abdu = gla ? 0.f : -a * b * du;
#pragma unroll
                    for (int e = 0; e < E; ++e) pk[e] = fmaf(dS[e], u, abdu * St[t][e]);
                    lane_rows_store<D>(part + ((t * 2 + 1) * CPC + colL) * D, lr, pk);
                    const float bdu = gla ? 0.f : -b * du;
#pragma unroll
                    for (int e = 0; e < E; ++e) dS[e] = a * fmaf(bdu, k[e], dS[e]);
                }
            }
        };
        if (phase < 2) {
            if (phase == 0 && si == 0) lane_rows_store<D>(ck_col(blk), lr, S);
            if (phase == 1) {
                if (si == 0) lane_rows<D>(ck_col(blk), lr, S);
                lane_rows_store<D>(sub_col(si), lr, S);
            }
            if (cnt == K) {
#pragma unroll
                for (int t = 0; t < K; ++t) absorb(S, sl, t);
            } else {
#pragma unroll
                for (int t = 0; t < K; ++t)
                    if (t < cnt) absorb(S, sl, t);
            }
        } else {
            if (cnt == K) reverse_stage(std::true_type{}); else reverse_stage(std::false_type{});
            __syncthreads();
            // dv of the stage (this CTA's columns are final)
            for (int idx = tid; idx < K * CPC; idx += NT) {
                const int t = idx / CPC, c = idx % CPC;
                if (t < cnt) dvh_h[((size_t)(start + ns + m0 + t) * L.Hq + h) * D + rank * CPC + c] = dv_s[idx];
            }
            // the CTA's sums over its columns into exchange slot nx; lambda's gradient from the dq rows
            // (sum_p qhat_p . S_p dO_p), alpha applied to dalpha
            float* xb = xch + (buf * kXB + nx) * (K * 2 * D);
            float* xsb = xs + (buf * kXB + nx) * (K * 2);
            for (int idx = tid; idx < K * 2 * (D / 4); idx += NT) {
                const int tq = idx / (D / 4), r = (idx % (D / 4)) * 4;
                float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
                for (int c = 0; c < CPC; c += 2) {
                    const float4 u0 = *reinterpret_cast<const float4*>(part + (tq * CPC + c) * D + r);
                    const float4 u1 = *reinterpret_cast<const float4*>(part + (tq * CPC + c + 1) * D + r);
                    a0.x += u0.x; a0.y += u0.y; a0.z += u0.z; a0.w += u0.w;
                    a1.x += u1.x; a1.y += u1.y; a1.z += u1.z; a1.w += u1.w;
                }
                const float4 sum = make_float4(a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w);
                *reinterpret_cast<float4*>(xb + tq * D + r) = sum;
                if (tq % 2 == 0 && tq / 2 < cnt) {
                    const float4 qv = *reinterpret_cast<const float4*>(slot_q(sl) + (tq / 2) * D + r);
                    dl = fmaf(qv.x, sum.x, fmaf(qv.y, sum.y, fmaf(qv.z, sum.z, fmaf(qv.w, sum.w, dl))));
                }
            }
            for (int idx = tid; idx < K * 2; idx += NT) {
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < CPC; ++c) acc += spart[idx * CPC + c];
                xsb[idx] = idx % 2 == 0 && idx / 2 < cnt ? acc * slot_a(sl)[idx / 2] : acc;
            }
            if (tid == 0) {
                xm[(buf * kXB + nx) * 2] = (int)m0;
                xm[(buf * kXB + nx) * 2 + 1] = cnt;
            }
            ++nx;
            if (nx == kXB || si == 0) {  // exchange: a full buffer, or the block's last stage
                cluster_sync_all();
                // over the cluster: this CTA finishes rows [rank D / kCl, (rank + 1) D / kCl) of dq and dk
                constexpr int RS = D / kCl;
                const float* xbb = xch + buf * kXB * (K * 2 * D);
                const int* xmb = xm + buf * kXB * 2;
                for (int idx = tid; idx < nx * K * 2 * RS; idx += NT) {
                    const int sx = idx / (K * 2 * RS), rem = idx % (K * 2 * RS);
                    const int tq = rem / RS, t = tq / 2, r = (int)rank * RS + rem % RS;
                    if (t < xmb[sx * 2 + 1]) {
                        float acc = 0.f;
#pragma unroll
                        for (int rr = 0; rr < kCl; ++rr) acc += ld_cluster(xbb + (sx * K * 2 + tq) * D + r, rr);
                        const int64_t j = start + ns + xmb[sx * 2] + t;
                        if (tq % 2 == 0)
                            dqh[((size_t)(j + W) * L.Hq + h) * D + r] = lam * acc;
                        else
                            dkh_h[((size_t)j * L.Hq + h) * D + r] = acc;
                    }
                }
                if (rank == 0) {
                    const float* xsx = xs + buf * kXB * (K * 2);
                    for (int idx = tid; idx < nx * K * 2; idx += NT) {
                        const int sx = idx / (K * 2), t = (idx % (K * 2)) / 2;
                        if (t < xmb[sx * 2 + 1]) {
                            float acc = 0.f;
#pragma unroll
                            for (int rr = 0; rr < kCl; ++rr) acc += ld_cluster(xsx + idx, rr);
                            const size_t o = (size_t)(start + ns + xmb[sx * 2] + t) * L.Hq + h;
                            (idx % 2 == 0 ? dg : dbeta)[o] = acc;
                        }
                    }
                }
                buf ^= 1;
                nx = 0;
            }
        }
        __syncthreads();
        issue(i + kRing);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // lambda's gradient: over the CTA, then over the cluster
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
    if (lane == 0) red[w] = dl;
    __syncthreads();
    if (tid == 0) {
        float acc = 0.f;
        for (int ww = 0; ww < NW; ++ww) acc += red[ww];
        red[NW] = acc;
    }
    cluster_sync_all();
    if (rank == 0 && tid == 0) {
        float acc = 0.f;
        for (int rr = 0; rr < kCl; ++rr) acc += ld_cluster(red + NW, rr);
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

// acc[i][j] += sum_k A[ty + 16 i][k] B[tx + 16 j][k], j < NJ (row pitch D + 4, 16-byte rows)
template <int D, int NJ = 4>
__device__ __forceinline__ void mm_abT(const float* __restrict__ A, const float* __restrict__ B, int ty, int tx,
                                       float acc[4][4]) {
    constexpr int LD = D + 4;
#pragma unroll 2
    for (int k = 0; k < D; k += 4) {
        float4 a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (ty + 16 * i) * LD + k);
#pragma unroll
        for (int j = 0; j < NJ; ++j) b[j] = *reinterpret_cast<const float4*>(B + (tx + 16 * j) * LD + k);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                acc[i][j] = fmaf(a[i].x, b[j].x, acc[i][j]);
                acc[i][j] = fmaf(a[i].y, b[j].y, acc[i][j]);
                acc[i][j] = fmaf(a[i].z, b[j].z, acc[i][j]);
                acc[i][j] = fmaf(a[i].w, b[j].w, acc[i][j]);
            }
    }
}

// Column c of a thread's D / 16 output columns: tx * 4 + (c % 4) + 64 (c / 4).
__device__ __forceinline__ int sm_col(int tx, int c) { return tx * 4 + (c & 3) + 64 * (c >> 2); }

// acc[i][c] += sum_j P[ty + 16 i][j] X[j][sm_col(tx, c)], j < JB, i < NI (P pitch kLP, X pitch D + 4)
template <int D, int JB = kSB, int NI = 4>
__device__ __forceinline__ void mm_ab(const float* __restrict__ P, const float* __restrict__ X, int ty, int tx,
                                      float acc[4][D / 16]) {
    constexpr int LD = D + 4, CC = D / 64;
#pragma unroll 2
    for (int j = 0; j < JB; j += 4) {
        float4 p[4];
#pragma unroll
        for (int i = 0; i < NI; ++i) p[i] = *reinterpret_cast<const float4*>(P + (ty + 16 * i) * kLP + j);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            float4 x[CC];
#pragma unroll
            for (int cc = 0; cc < CC; ++cc) x[cc] = *reinterpret_cast<const float4*>(X + (j + jj) * LD + tx * 4 + 64 * cc);
#pragma unroll
            for (int i = 0; i < NI; ++i) {
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
    // a tile of at most 16 keys (the sinks) runs on the first 16 columns only (NJ = 1)
    auto pass1 = [&](auto nj, int64_t j0, int nk) {
        constexpr int NJ = decltype(nj)::value;
        float s[4][4] = {};
        mm_abT<D, NJ>(Qs, Ks, ty, tx, s);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                s[i][j] = visible(ty + 16 * i, tx + 16 * j, j0, nk) ? s[i][j] * scale : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
            mx = max16(mx);
            const float mn = fmaxf(m[i], mx);
            const float basev = mn == -INFINITY ? 0.f : mn;
            const float r = m[i] == -INFINITY ? 0.f : expf(m[i] - basev);
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
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
        mm_ab<D, 16 * NJ>(Ps, Vs, ty, tx, O);
    };
    for (int t = 0; t < n_tiles; ++t) {
        int64_t j0;
        int nk;
        tile(t, &j0, &nk);
        load_kv(j0, nk);
        if (nk <= 16)
            pass1(std::integral_constant<int, 1>{}, j0, nk);
        else
            pass1(std::integral_constant<int, 4>{}, j0, nk);
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
    auto pass2 = [&](auto nj, int64_t j0, int nk, bool sink) {
        constexpr int NJ = decltype(nj)::value;
        float s[4][4] = {}, dp[4][4] = {};
        mm_abT<D, NJ>(Qs, Ks, ty, tx, s);
        mm_abT<D, NJ>(dOs, Vs, ty, tx, dp);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
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
        mm_ab<D, 16 * NJ>(dSs, Ks, ty, tx, dq);
        if (sink) {  // the block's partial sums for the sink keys (rows of the transposed tiles)
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                float acc[4][NC];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;
                mm_ab<D, kSB, NJ>(which ? Ps : Ts, which ? dOs : Qs, ty, tx, acc);
                float* dst = which ? sink_v : sink_k;
                const float f = which ? 1.f : scale;
#pragma unroll
                for (int i = 0; i < NJ; ++i) {
                    const int key = ty + 16 * i;
                    if (key < nk) {
                        const size_t o = (((size_t)b * L.Hq + h) * ns + j0 + key) * D;
#pragma unroll
                        for (int c = 0; c < NC; ++c) dst[o + sm_col(tx, c)] = acc[i][c] * f;
                    }
                }
            }
        }
    };
    for (int t = 0; t < n_tiles; ++t) {
        int64_t j0;
        int nk;
        tile(t, &j0, &nk);
        load_kv(j0, nk);
        if (nk <= 16)
            pass2(std::integral_constant<int, 1>{}, j0, nk, t < n_sink_tiles);
        else
            pass2(std::integral_constant<int, 4>{}, j0, nk, t < n_sink_tiles);
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

// Sink keys: CTA per (sequence, q-head, sink key), thread per channel; the sums over the sequence's query
// blocks (those whose last query is at or after the key) of the partials, in four interleaved chains.
__global__ void bwd_sm_sink_kernel(LayerDims L, const int32_t* __restrict__ cu, const int32_t* __restrict__ base,
                                   int n_blk, const float* __restrict__ sink_k, const float* __restrict__ sink_v,
                                   float* __restrict__ dkr_h, float* __restrict__ dv_h) {
    const int n = blockIdx.x, h = blockIdx.y, c = threadIdx.x, D = L.d, ns = L.n_sinks;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int b0 = __ldg(base + n), nb = (int)((len + kSB - 1) / kSB);
    for (int j = blockIdx.z; j < min((int64_t)ns, len); j += gridDim.z) {
        const int qb_lo = j / kSB;  // blocks whose last query is before key j see nothing of it
        const int qb_hi = min(nb, n_blk - b0);
        float sk[4] = {0.f, 0.f, 0.f, 0.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
        for (int qb = qb_lo; qb < qb_hi; ++qb) {
            const size_t o = (((size_t)(b0 + qb) * L.Hq + h) * ns + j) * D + c;
            sk[qb & 3] += sink_k[o];
            sv[qb & 3] += sink_v[o];
        }
        const size_t o = ((size_t)(start + j) * L.Hq + h) * D + c;
        dkr_h[o] = (sk[0] + sk[1]) + (sk[2] + sk[3]);
        dv_h[o] = (sv[0] + sv[1]) + (sv[2] + sv[3]);
    }
}

// ---- 5. feature backward: first the L2 backward into the gradient of the pre-norm rows (q-heads, then
// k-heads with the group's per-head gradients summed) and the group sums of the v rows; the conv and RoPE
// backward then run in bwd_feat_out_kernel.  CTA per token, a warp per row, lane l channels l + 32 e.
template <int D>
__global__ void __launch_bounds__(kRowThreads)
bwd_l2_kernel(LayerDims L, const float* __restrict__ qt, const float* __restrict__ kt,
              const float* __restrict__ dqh, const float* __restrict__ dkh_h, const float* __restrict__ dvh_h,
              float* __restrict__ dqt, float* __restrict__ dkt, float* __restrict__ dvt) {
    constexpr int E = D / 32;
    const int64_t t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < L.Hq + 2 * L.Hkv; r += kRowThreads / 32) {
        const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
        const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
        float dy[E];
#pragma unroll
        for (int e = 0; e < E; ++e) dy[e] = 0.f;
        if (kind == 0) {
#pragma unroll
            for (int e = 0; e < E; ++e) dy[e] = dqh[((size_t)t * L.Hq + hh) * D + lane + 32 * e];
        } else {
            const float* src = kind == 1 ? dkh_h : dvh_h;
            for (int gq = 0; gq < L.G; ++gq)
#pragma unroll
                for (int e = 0; e < E; ++e) dy[e] += src[((size_t)t * L.Hq + hh * L.G + gq) * D + lane + 32 * e];
        }
        if (kind == 2) {  // vhat = conv(v): no norm
#pragma unroll
            for (int e = 0; e < E; ++e) dvt[((size_t)t * L.Hkv + hh) * D + lane + 32 * e] = dy[e];
            continue;
        }
        const float* pre = kind == 0 ? qt + ((size_t)t * L.Hq + hh) * D : kt + ((size_t)t * L.Hkv + hh) * D;
        float* dst = kind == 0 ? dqt + ((size_t)t * L.Hq + hh) * D : dkt + ((size_t)t * L.Hkv + hh) * D;
        if (kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q)) {
            // y = x / nrm, nrm = sqrt(|x|^2 + eps): dx = (dy - x (x . dy) / nrm^2) / nrm
            float x[E], n2 = 0.f, xd = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                x[e] = pre[lane + 32 * e];
                n2 = fmaf(x[e], x[e], n2);
                xd = fmaf(x[e], dy[e], xd);
            }
            n2 = warp_sum_f(n2) + 1e-6f;
            xd = warp_sum_f(xd);
            const float inv = rsqrtf(n2);
#pragma unroll
            for (int e = 0; e < E; ++e) dst[lane + 32 * e] = (dy[e] - x[e] * xd / n2) * inv;
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) dst[lane + 32 * e] = dy[e];
        }
    }
}

// conv backward (the taps that read position p, from the later positions of the same sequence), plus the
// softmax branch's gradient, then RoPE's transpose; writes dq, dk, dv.  CTA per token; rows r < Hq are
// q-heads, < Hq + Hkv k-heads, else v-heads; a thread per channel pair (i, i + d / 2).
__global__ void __launch_bounds__(kRowThreads)
bwd_feat_out_kernel(LayerDims L, const int32_t* __restrict__ cu, const float* __restrict__ wq,
                    const float* __restrict__ wk, const float* __restrict__ wv, const float* __restrict__ dqt,
                    const float* __restrict__ dkt, const float* __restrict__ dvt, const float* __restrict__ dqr_sm,
                    const float* __restrict__ dkr_h, const float* __restrict__ dv_h, float* __restrict__ dq,
                    float* __restrict__ dk, float* __restrict__ dv) {
    __shared__ float cs[64], sn[64];
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x, D = L.d, half = D / 2;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    angles(L, p, cs, sn);
    for (int idx = tid; idx < (L.Hq + 2 * L.Hkv) * half; idx += kRowThreads) {
        const int r = idx / half, i = idx % half;
        const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
        const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
        const int H = kind == 0 ? L.Hq : L.Hkv;
        const float* w = kind == 0 ? wq : kind == 1 ? wk : wv;
        const float4* w1 = reinterpret_cast<const float4*>(w + ((size_t)hh * D + i) * kConvWidth);
        const float4* w2 = reinterpret_cast<const float4*>(w + ((size_t)hh * D + i + half) * kConvWidth);
        const float4 w1a = w1[0], w1b = w1[1], w2a = w2[0], w2b = w2[1];
        const float t1[kConvWidth] = {w1a.x, w1a.y, w1a.z, w1a.w, w1b.x, w1b.y, w1b.z, w1b.w};
        const float t2[kConvWidth] = {w2a.x, w2a.y, w2a.z, w2a.w, w2b.x, w2b.y, w2b.z, w2b.w};
        const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
        // x_p feeds y_{p + 7 - m} through tap m
        float a1 = 0.f, a2 = 0.f;
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) {
            const int64_t pp = p + (kConvWidth - 1) - m;
            if (pp >= len) continue;
            const float* yr = dy + ((size_t)(start + pp) * H + hh) * D;
            a1 = fmaf(t1[m], yr[i], a1);
            a2 = fmaf(t2[m], yr[i + half], a2);
        }
        // the softmax branch's gradient of the RoPE'd row (q, k) or of raw v, summed over the group for k, v
        if (kind == 0) {
            const float* sg = dqr_sm + ((size_t)t * L.Hq + hh) * D;
            a1 += sg[i];
            a2 += sg[i + half];
        } else {
            for (int gq = 0; gq < L.G; ++gq) {
                const float* sg = (kind == 1 ? dkr_h : dv_h) + ((size_t)t * L.Hq + hh * L.G + gq) * D;
                a1 += sg[i];
                a2 += sg[i + half];
            }
        }
        if (kind == 2) {
            float* o = dv + ((size_t)t * L.Hkv + hh) * D;
            o[i] = a1;
            o[i + half] = a2;
        } else {  // RoPE's transpose: rotate the pair back by the angle p theta_i
            float* o = (kind == 0 ? dq : dk) + ((size_t)t * H + hh) * D;
            o[i] = a1 * cs[i] + a2 * sn[i];
            o[i + half] = a2 * cs[i] - a1 * sn[i];
        }
    }
}

// ---- 6. conv filters: partial sums over a block of kWB tokens, per (row, channel, tap); then the blocks.
// A thread walks its channel through the block's tokens with the last 8 inputs of the sequence in
// registers (zeros before the sequence start), so every input is read once.
template <typename Tin>
__global__ void bwd_convw_part_kernel(LayerDims L, const Tin* __restrict__ v, const int32_t* __restrict__ cu,
                                      const float* __restrict__ qr, const float* __restrict__ kr,
                                      const float* __restrict__ dqt, const float* __restrict__ dkt,
                                      const float* __restrict__ dvt, float* __restrict__ part) {
    __shared__ int32_t pos_s[kWB];  // position of each token of the block in its sequence
    const int blk = blockIdx.x, r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
    const int64_t t0 = (int64_t)blk * kWB, t1 = min(L.total, t0 + kWB);
    for (int64_t t = t0 + c; t < t1; t += blockDim.x) {
        int64_t start, len;
        seq_range(cu, seq_of_token(cu, L.n_seqs, t), L.total, &start, &len);
        pos_s[t - t0] = (int32_t)min(t - start, (int64_t)INT32_MAX);
    }
    __syncthreads();
    auto input = [&](int64_t t) {
        const size_t row = ((size_t)t * H + hh) * D + c;
        return kind == 0 ? qr[row] : kind == 1 ? kr[row] : to_f32(v[row]);
    };
    float acc[kConvWidth], win[kConvWidth];  // win[m]: the input at position p - 7 + m
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) acc[m] = win[m] = 0.f;
    // the window before the block's first token
    if (t1 > t0) {
        const int p0 = pos_s[0];
#pragma unroll
        for (int m = 1; m < kConvWidth; ++m) {
            const int back = kConvWidth - m;  // position p0 - back sits at win[m - 1] before the shift
            win[m] = back <= p0 ? input(t0 - back) : 0.f;
        }
    }
    for (int64_t t = t0; t < t1; ++t) {
        const int p = pos_s[t - t0];
        if (p == 0) {  // a sequence starts: nothing before it
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) win[m] = 0.f;
        } else {
#pragma unroll
            for (int m = 0; m + 1 < kConvWidth; ++m) win[m] = win[m + 1];
        }
        win[kConvWidth - 1] = input(t);
        const float d_y = dy[((size_t)t * H + hh) * D + c];
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) acc[m] = fmaf(d_y, win[m], acc[m]);
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
    b.alpha = take(T * Hq);
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
cudaError_t launch_gdn_bwd(const LayerDims& L, const float* alpha, const float* beta, const float* lambda,
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
    cfg.blockDim = dim3(GdnB<D>::NT);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_gdn_kernel<Tin, D>, L, alpha, beta, lambda, dout, cu, qh, kh, vh, ckpt, sub, dqh,
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
        bwd_sm_sink_kernel<<<dim3(L.n_seqs, L.Hq, min(L.n_sinks, 64)), D, 0, st>>>(L, cu, base, n_blk, sink_k, sink_v,
                                                                                 dkr_h, dv_h);
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
    bwd_rope_kernel<Tin><<<(unsigned)T, kRowThreads, 0, st>>>(L, q, k, g, cu, F(b.qr), F(b.kr), F(b.alpha),
                                                                        reinterpret_cast<int32_t*>(ws + b.err));
    if ((e = mark(1)) != cudaSuccess) return e;
    if (D == 128)
        bwd_conv_kernel<Tin, 128><<<(unsigned)T, kRowThreads, 0, st>>>(L, v, wq, wk, wv, cu, F(b.qr), F(b.kr), F(b.qt),
                                                                       F(b.qh), F(b.kt), F(b.kh), F(b.vh));
    else
        bwd_conv_kernel<Tin, 64><<<(unsigned)T, kRowThreads, 0, st>>>(L, v, wq, wk, wv, cu, F(b.qr), F(b.kr), F(b.qt),
                                                                      F(b.qh), F(b.kt), F(b.kh), F(b.vh));
    if ((e = mark(2)) != cudaSuccess) return e;
    e = D == 128 ? launch_gdn_bwd<Tin, 128>(L, F(b.alpha), beta, lambda, dout, cu, F(b.qh), F(b.kh), F(b.vh), F(b.ckpt),
                                            F(b.sub), F(b.dqh), F(b.dkh_h), F(b.dvh_h), dg, dbeta, F(b.dlam_part), st)
                 : launch_gdn_bwd<Tin, 64>(L, F(b.alpha), beta, lambda, dout, cu, F(b.qh), F(b.kh), F(b.vh), F(b.ckpt),
                                           F(b.sub), F(b.dqh), F(b.dkh_h), F(b.dvh_h), dg, dbeta, F(b.dlam_part), st);
    if (e != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    e = D == 128 ? launch_sm_bwd<Tin, 128>(L, v, dout, cu, sm_base, b.n_sm_blocks, F(b.qr), F(b.kr), F(b.stats),
                                           F(b.dqr_sm), F(b.dkr_h), F(b.dv_h), F(b.sink_k), F(b.sink_v), st)
                 : launch_sm_bwd<Tin, 64>(L, v, dout, cu, sm_base, b.n_sm_blocks, F(b.qr), F(b.kr), F(b.stats),
                                          F(b.dqr_sm), F(b.dkr_h), F(b.dv_h), F(b.sink_k), F(b.sink_v), st);
    if (e != cudaSuccess) return e;
    if ((e = mark(4)) != cudaSuccess) return e;
    if (D == 128)
        bwd_l2_kernel<128><<<(unsigned)T, kRowThreads, 0, st>>>(L, F(b.qt), F(b.kt), F(b.dqh), F(b.dkh_h), F(b.dvh_h),
                                                                F(b.dqt), F(b.dkt), F(b.dvt));
    else
        bwd_l2_kernel<64><<<(unsigned)T, kRowThreads, 0, st>>>(L, F(b.qt), F(b.kt), F(b.dqh), F(b.dkh_h), F(b.dvh_h),
                                                               F(b.dqt), F(b.dkt), F(b.dvt));
    if ((e = mark(5)) != cudaSuccess) return e;
    bwd_feat_out_kernel<<<(unsigned)T, kRowThreads, 0, st>>>(L, cu, wq, wk, wv, F(b.dqt), F(b.dkt), F(b.dvt),
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
