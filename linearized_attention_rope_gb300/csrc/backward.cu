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
//  1. rope: RoPE'd q and k rows (fp32) for every token and head, the angle
//     table; alpha = e^g;
//  2. conv: q~, k~ (and their L2-normalised qhat, khat) and vhat = conv(v),
//     a warp per (row, span of tokens) with the conv window in registers;
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
//     gradients of each kv group are summed; one launch, streaming like 2;
//  6. the conv filters' gradients (per span of tokens, then over the spans);
//  7. lambda's gradient over the sequences.
#include <type_traits>

#include "hla_common.cuh"

namespace hla {

namespace {

constexpr int kWB = 64;  // the shortest span of the conv-filter partial sums (at most ceil(T / 64) of them)

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
                float* __restrict__ alpha, float2* __restrict__ ang, int32_t* __restrict__ err) {
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
    if (tid < half) ang[(size_t)t * half + tid] = make_float2(cs[tid], sn[tid]);  // for the RoPE backward
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

// Sums of eight per-lane values over a warp, reduced together: the lanes exchange halves of the set in three
// butterfly steps and then add across 8 and 16 lanes, so lane l returns the sum of v[red8_slot(l)] (lanes l,
// l ^ 8, l ^ 16 and l ^ 24 alike); 9 shuffles in place of 40.
__device__ __forceinline__ int red8_slot(int lane) { return ((lane & 1) << 2) | (lane & 2) | ((lane >> 2) & 1); }
__device__ __forceinline__ float warp_reduce8(const float (&v)[8], int lane) {
    const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
    float a[4], b[2];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        a[j] = (b0 ? v[4 + j] : v[j]) + __shfl_xor_sync(0xffffffffu, b0 ? v[j] : v[4 + j], 1);
#pragma unroll
    for (int j = 0; j < 2; ++j)
        b[j] = (b1 ? a[2 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, b1 ? a[j] : a[2 + j], 2);
    float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, b2 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xffffffffu, c, 8);
    return c + __shfl_xor_sync(0xffffffffu, c, 16);
}
// Rows of one tensor laid out [token][head][D] for a CTA of D threads: the rows of head hh at tokens
// tb .. tb + 7 into dst[8][D] by 16-byte cp.async (rows at or past t_end zero-filled, read from token 0's
// row, which exists whenever there are tokens).
template <typename T, int D>
__device__ __forceinline__ void stage_rows8(T* dst, const T* __restrict__ src, int64_t tb, int64_t t_end, int H,
                                            int hh) {
    constexpr int CPR = D * (int)sizeof(T) / 16;  // 16-byte pieces per row
    constexpr int PER = 8 * CPR / D;              // pieces per thread
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int j = (int)threadIdx.x + D * i, u = j / CPR, piece = j % CPR;
        const int64_t t = tb + u;
        const bool in = t < t_end;
        const char* g = reinterpret_cast<const char*>(src + ((size_t)(in ? t : 0) * H + hh) * D) + 16 * piece;
        const uint32_t d = (uint32_t)__cvta_generic_to_shared(reinterpret_cast<char*>(dst + u * D) + 16 * piece);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(g), "r"(in ? 16 : 0) : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---- 2. conv (+ L2): a CTA per (row, span of tokens) with a thread per channel; rows r < Hq are q-heads,
// < Hq + Hkv k-heads, else v-heads.  The CTA streams its span's input rows through a shared-memory ring of
// kCvRing blocks of 8 tokens (cp.async, kCvRing - 1 blocks in flight) and keeps the last 8 inputs of each
// channel in a register ring (token t in slot (t - span start) mod 8), zeroed where a sequence starts so
// that the taps before a sequence's first token read zero.  Every input row is read once (the 7 rows before
// a span twice).  One CTA barrier per block: it makes the block's rows visible, frees the slot the next copy
// refills, and closes the previous block's L2 row sums, whose outputs are written then.
constexpr int kCvRing = 4;
template <typename Tin, int D>
__global__ void __launch_bounds__(D)
bwd_conv_kernel(LayerDims L, const Tin* __restrict__ v, const float* __restrict__ wq, const float* __restrict__ wk,
                const float* __restrict__ wv, const int32_t* __restrict__ cu, const float* __restrict__ qr,
                const float* __restrict__ kr, float* __restrict__ qt, float* __restrict__ qh,
                float* __restrict__ kt, float* __restrict__ kh, float* __restrict__ vh, int64_t span) {
    constexpr int B = kConvWidth;
    __shared__ __align__(16) float ring_f[kCvRing][B][D];  // q, k rows (v rows use the first half, as Tin)
    __shared__ float part[2][B][D / 32];
    const int c = threadIdx.x, r = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * span;
    if (t0 >= L.total) return;  // whole CTA
    const int64_t t1 = min(L.total, t0 + span);
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const bool norm = kind == 1 || (kind == 0 && (L.flags & HLA_FLAG_L2NORM_Q));  // uniform over the CTA
    const float* src = kind == 0 ? qr : kr;
    auto issue = [&](int64_t tb, int slot) {
        if (kind == 2)
            stage_rows8<Tin, D>(reinterpret_cast<Tin*>(&ring_f[slot][0][0]), v, tb, t1, H, hh);
        else
            stage_rows8<float, D>(&ring_f[slot][0][0], src, tb, t1, H, hh);
        cp_async_commit_group();
    };
    auto staged = [&](int slot, int u) {
        return kind == 2 ? to_f32(reinterpret_cast<const Tin*>(&ring_f[slot][0][0])[u * D + c]) : ring_f[slot][u][c];
    };
    const int64_t n_blk = (t1 - t0 + B - 1) / B;
#pragma unroll
    for (int i = 0; i < kCvRing - 1; ++i) {
        if (i < n_blk) {
            issue(t0 + (int64_t)B * i, i);
        } else {
            cp_async_commit_group();  // empty groups keep the count per block uniform
        }
    }
    float wt[kConvWidth];
    {
        const float4* w4 = reinterpret_cast<const float4*>((kind == 0 ? wq : kind == 1 ? wk : wv) +
                                                           ((size_t)hh * D + c) * kConvWidth);
        const float4 a = w4[0], b = w4[1];
        wt[0] = a.x; wt[1] = a.y; wt[2] = a.z; wt[3] = a.w;
        wt[4] = b.x; wt[5] = b.y; wt[6] = b.z; wt[7] = b.w;
    }
    int s = seq_of_token(cu, L.n_seqs, t0);
    int64_t s_start, s_len;
    seq_range(cu, s, L.total, &s_start, &s_len);
    float ring[B];
    ring[0] = 0.f;
#pragma unroll
    for (int m = 0; m < B - 1; ++m) {  // tokens t0 - 7 .. t0 - 1 in slots 1..7: those of t0's sequence
        const int64_t t = t0 - (B - 1) + m;
        const size_t i = ((size_t)t * H + hh) * D + c;
        ring[m + 1] = t >= s_start && t >= 0 ? (kind == 2 ? to_f32(v[i]) : src[i]) : 0.f;
    }
    float* out_t = kind == 0 ? qt : kind == 1 ? kt : vh;
    float* out_h = kind == 0 ? qh : kh;
    float y[B];  // the previous block's conv outputs, written after the next barrier
    // the outputs of block tb (its row sums in part[p] for the normalised rows)
    auto finish = [&](int64_t tb, int p) {
        float inv[B];
        if (norm) {
#pragma unroll
            for (int u = 0; u < B; ++u) {
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < D / 32; ++k) acc += part[p][u][k];
                inv[u] = rsqrtf(acc + 1e-6f);
            }
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t t = tb + u;
            if (t >= t1) break;
            const size_t o = ((size_t)t * H + hh) * D + c;
            out_t[o] = y[u];
            if (kind != 2) out_h[o] = norm ? y[u] * inv[u] : y[u];
        }
    };
#pragma unroll 1
    for (int64_t b = 0; b < n_blk; ++b) {
        const int64_t tb = t0 + B * b;
        cp_async_wait_group<kCvRing - 2>();
        __syncthreads();
        if (b > 0) finish(tb - B, (int)((b - 1) & 1));
        if (b + kCvRing - 1 < n_blk) {
            issue(tb + (int64_t)B * (kCvRing - 1), (int)((b + kCvRing - 1) % kCvRing));
        } else {
            cp_async_commit_group();
        }
        const int slot = (int)(b % kCvRing);
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t t = tb + u;
            while (t >= s_start + s_len && s + 1 < L.n_seqs) {  // uniform over the CTA
                ++s;
                seq_range(cu, s, L.total, &s_start, &s_len);
            }
            if (t == s_start) {  // a sequence starts here: nothing before it feeds the conv
#pragma unroll
                for (int m = 0; m < B; ++m) ring[m] = 0.f;
            }
            ring[u] = staged(slot, u);
            // tap m reads token t - 7 + m: slot (u + 1 + m) mod 8
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) acc = fmaf(wt[m], ring[(u + 1 + m) & (B - 1)], acc);
            y[u] = acc;
        }
        if (norm) {
            float sq[B];
#pragma unroll
            for (int u = 0; u < B; ++u) sq[u] = y[u] * y[u];
            const int lane = c & 31;
            const float w = warp_reduce8(sq, lane);
            if (lane < 8) part[b & 1][red8_slot(lane)][c >> 5] = w;
        }
    }
    __syncthreads();
    if (n_blk > 0) finish(t0 + B * (n_blk - 1), (int)((n_blk - 1) & 1));
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

// Row y of a grid over sequences takes the sequence of rank y by length, longest first (ties in index order),
// so that with sequences of mixed lengths the longest chains start in the first wave of CTAs (the rows are
// placed in order); more than kMaxRankedSeqs sequences keep index order.  Reads only cu_seqlens; every
// thread of the CTA calls it (one CTA barrier); `slot` is a shared int.
constexpr int kMaxRankedSeqs = 64;
__device__ __forceinline__ int ranked_seq(const LayerDims& L, const int32_t* __restrict__ cu, int y, int* slot) {
    if (L.n_seqs > kMaxRankedSeqs) return y;
    for (int q = threadIdx.x; q < L.n_seqs; q += blockDim.x) {
        int64_t qs, ql;
        seq_range(cu, q, L.total, &qs, &ql);
        int r = 0;
        for (int o = 0; o < L.n_seqs; ++o) {
            int64_t os, ol;
            seq_range(cu, o, L.total, &os, &ol);
            r += (ol > ql || (ol == ql && o < q)) ? 1 : 0;
        }
        if (r == y) *slot = q;  // exactly one sequence has each rank
    }
    __syncthreads();
    return *slot;
}

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
    float* red = dv_s + K * CPC;        // [NW] + 1, then the CTA's sequence (an int)
    const uint32_t rank = cluster_rank();
    const int h = blockIdx.x / kCl, kv = h / L.G, tid = threadIdx.x;
    const int n = ranked_seq(L, cu, (int)blockIdx.y, reinterpret_cast<int*>(red + NW + 1));
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

// ---- 5. feature backward, a CTA per (row, span of tokens) with a thread per channel, as in the conv above.
// Per token t' of the row the L2 backward gives y(t'), the gradient of the conv output (q-heads: from dqhat;
// k-heads: from the sum of the group's per-head dkhat; v-heads: the sum of the group's per-head dvhat, no
// norm), kept for the filter gradients; the conv's transpose then gives the input's gradient,
// dx(t) = sum_m w_m y(t + 7 - m) over the t + 7 - m inside t's sequence, to which the softmax branch's
// gradient of the same row is added (summed over the group for k and v) before RoPE's transpose (q, k),
// which pairs channel i with i + d / 2.  Walking the span in blocks of 8 tokens, the CTA holds y of the
// current block and the next one, and per block forms y of the block after those and dx of the current one.
// Its rows stream through a shared-memory ring of kFoRing units (cp.async, kFoRing - 1 in flight); a unit
// holds, for one head g of the row's group (one head for q), 8 rows of y's source for a later block and of
// the softmax gradient for the current one, and with g = 0 also the 8 pre-norm rows and RoPE angles.  The
// first 2 units per head carry y's sources of the span's first two blocks.  One CTA barrier per unit; the
// row sums of the L2 backward and the RoPE partners cross the CTA in shared memory (double-buffered by block
// parity) and are read after the next unit's barrier.  The 15 rows of y past the span are formed again by
// the next span's CTA, which writes them.
struct FeatOutArgs {
    const int32_t* cu;
    const float *wq, *wk, *wv, *qt, *kt, *dqh, *dkh_h, *dvh_h, *dqr_sm, *dkr_h, *dv_h;
    const float2* ang;
    float *dqt, *dkt, *dvt, *dq, *dk, *dv;
};
constexpr int kFoRing = 4;
template <int D>
constexpr size_t feat_out_smem() {  // the unit ring, then part[2][2][8][D / 32], dxs[2][8][D]
    return ((size_t)kFoRing * 4 * kConvWidth * D + 2 * 2 * kConvWidth * (D / 32) + 2 * kConvWidth * D) * sizeof(float);
}

template <int D>
__global__ void __launch_bounds__(D, 512 / D)
bwd_feat_out_kernel(LayerDims L, FeatOutArgs A, int64_t span) {
    constexpr int B = kConvWidth, half = D / 2, NW = D / 32, SLOT = 4 * B * D;
    extern __shared__ __align__(16) float fo_smem[];
    float* slots = fo_smem;
    float (*part)[2][B][NW] = reinterpret_cast<float (*)[2][B][NW]>(fo_smem + kFoRing * SLOT);
    float (*dxs)[B][D] = reinterpret_cast<float (*)[B][D]>(fo_smem + kFoRing * SLOT + 2 * 2 * B * NW);
    const int c = threadIdx.x, r = blockIdx.y, lane = c & 31, warp = c >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * span;
    if (t0 >= L.total) return;  // whole CTA
    const int64_t t1 = min(L.total, t0 + span);
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const int U = kind == 0 ? 1 : L.G;  // heads summed per row: units per block
    const bool norm = kind == 1 || (kind == 0 && (L.flags & HLA_FLAG_L2NORM_Q));  // uniform over the CTA
    const float* ysrc = kind == 0 ? A.dqh : kind == 1 ? A.dkh_h : A.dvh_h;
    const float* gsrc = kind == 0 ? A.dqr_sm : kind == 1 ? A.dkr_h : A.dv_h;
    const float* pre = kind == 0 ? A.qt : A.kt;
    float* ydst = kind == 0 ? A.dqt : kind == 1 ? A.dkt : A.dvt;
    float* dst = kind == 0 ? A.dq : kind == 1 ? A.dk : A.dv;
    const int64_t n_blk = (t1 - t0 + B - 1) / B;
    const int64_t n_units = (2 + n_blk) * U;
    // unit n: n < 2U carries y's sources of block n / U (head n % U); after those, unit (b + 2) U + g carries
    // y's sources of block b + 2 and the softmax gradient and angles of block b (head g)
    auto issue = [&](int64_t n) {
        if (n < n_units) {
            float* sl = slots + (size_t)(n % kFoRing) * SLOT;
            const int64_t j = n / U;
            const int g = (int)(n % U);
            const int64_t ty = t0 + B * j;  // y's block: j
            stage_rows8<float, D>(sl, ysrc, ty, L.total, L.Hq, hh * U + g);
            if (g == 0 && norm) stage_rows8<float, D>(sl + 2 * B * D, pre, ty, L.total, H, hh);
            if (j >= 2) {
                const int64_t tb = t0 + B * (j - 2);
                stage_rows8<float, D>(sl + B * D, gsrc, tb, t1, L.Hq, hh * U + g);
                if (g == 0 && kind != 2)
                    stage_rows8<float, D>(sl + 3 * B * D, reinterpret_cast<const float*>(A.ang), tb, t1, 1, 0);
            }
        }
        cp_async_commit_group();  // (empty past the last unit: the count per unit stays uniform)
    };
    float wt[kConvWidth];
    {
        const float4* w4 = reinterpret_cast<const float4*>((kind == 0 ? A.wq : kind == 1 ? A.wk : A.wv) +
                                                           ((size_t)hh * D + c) * kConvWidth);
        const float4 a = w4[0], b = w4[1];
        wt[0] = a.x; wt[1] = a.y; wt[2] = a.z; wt[3] = a.w;
        wt[4] = b.x; wt[5] = b.y; wt[6] = b.z; wt[7] = b.w;
    }
    for (int i = 0; i < kFoRing - 1; ++i) issue(i);
    int s = seq_of_token(A.cu, L.n_seqs, t0);
    int64_t s_start, s_len;
    seq_range(A.cu, s, L.total, &s_start, &s_len);
    float y0[B], y1[B];     // y of the current block and the next one
    float ya[B], xa[B];     // y's source summed over the heads so far, and the pre-norm rows, of the block in hand
    float sa[B], dx[B];     // the softmax gradient summed over the heads so far; dx of the current block
    float2 an[B];           // RoPE cos / sin of the current block's tokens at this thread's channel pair
#pragma unroll
    for (int u = 0; u < B; ++u) ya[u] = xa[u] = sa[u] = 0.f;
    // the block of y whose row sums are in part[jp & 1] (pending after its last unit), and the block whose dx
    // waits for its RoPE partners in dxs
    int64_t y_pending = -1, dx_pending = -1;
    auto finish_y = [&](int64_t j, float (&y)[B]) {
        if (norm) {
#pragma unroll
            for (int u = 0; u < B; ++u) {
                float n2 = 0.f, xd = 0.f;
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    n2 += part[j & 1][0][u][k];
                    xd += part[j & 1][1][u][k];
                }
                n2 += 1e-6f;
                // y = x / nrm, nrm = sqrt(|x|^2 + eps): dx = (dy - x (x . dy) / nrm^2) / nrm
                y[u] = (ya[u] - xa[u] * xd / n2) * rsqrtf(n2);
            }
        } else {
#pragma unroll
            for (int u = 0; u < B; ++u) y[u] = ya[u];
        }
        const int64_t tb = t0 + B * j;
#pragma unroll
        for (int u = 0; u < B; ++u) {
            if (tb + u < t1) ydst[((size_t)(tb + u) * H + hh) * D + c] = y[u];
            ya[u] = xa[u] = 0.f;
        }
    };
    auto finish_dx = [&](int64_t b) {
        const int64_t tb = t0 + B * b;
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t t = tb + u;
            if (t >= t1) break;
            const float other = dxs[b & 1][u][c ^ half];
            dst[((size_t)t * H + hh) * D + c] = c < half ? dx[u] * an[u].x + other * an[u].y
                                                         : dx[u] * an[u].x - other * an[u].y;
        }
    };
#pragma unroll 1
    for (int64_t n = 0; n < n_units; ++n) {
        cp_async_wait_group<kFoRing - 2>();
        __syncthreads();
        issue(n + kFoRing - 1);
        // work whose shared sums were written before this barrier
        if (y_pending >= 0) {
            if (y_pending == 0) {
                finish_y(0, y0);
            } else if (y_pending == 1) {
                finish_y(1, y1);
            } else {
                float y2[B];
                finish_y(y_pending, y2);
#pragma unroll
                for (int u = 0; u < B; ++u) {
                    y0[u] = y1[u];
                    y1[u] = y2[u];
                }
            }
            y_pending = -1;
        }
        if (dx_pending >= 0) {
            finish_dx(dx_pending);
            dx_pending = -1;
        }
        // this unit
        const float* sl = slots + (size_t)(n % kFoRing) * SLOT;
        const int64_t j = n / U;
        const int g = (int)(n % U);
#pragma unroll
        for (int u = 0; u < B; ++u) ya[u] += sl[u * D + c];
        if (g == 0 && norm) {
#pragma unroll
            for (int u = 0; u < B; ++u) xa[u] = sl[2 * B * D + u * D + c];
        }
        if (j >= 2) {
#pragma unroll
            for (int u = 0; u < B; ++u) sa[u] += sl[B * D + u * D + c];
            if (g == 0 && kind != 2) {
#pragma unroll
                for (int u = 0; u < B; ++u)
                    an[u] = reinterpret_cast<const float2*>(sl + 3 * B * D + u * D)[c & (half - 1)];
            }
        }
        if (g != U - 1) continue;
        // the block's last unit: y's row sums to part, then (main units) dx of block j - 2
        if (norm) {
            float n2[B], xd[B];
#pragma unroll
            for (int u = 0; u < B; ++u) {
                n2[u] = xa[u] * xa[u];
                xd[u] = xa[u] * ya[u];
            }
            const float wn = warp_reduce8(n2, lane), wd = warp_reduce8(xd, lane);
            if (lane < 8) {
                part[j & 1][0][red8_slot(lane)][warp] = wn;
                part[j & 1][1][red8_slot(lane)][warp] = wd;
            }
        }
        y_pending = j;
        if (j < 2) continue;
        const int64_t b = j - 2, tb = t0 + B * b;
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t t = tb + u;
            while (t >= s_start + s_len && s + 1 < L.n_seqs) {  // uniform over the CTA
                ++s;
                seq_range(A.cu, s, L.total, &s_start, &s_len);
            }
            const int64_t s_end = s_start + s_len;
            float acc = 0.f;
            // x_t feeds the conv output at t + 7 - m through tap m
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) {
                const int jj = u + (kConvWidth - 1) - m;
                if (tb + jj < s_end) acc = fmaf(wt[m], jj < B ? y0[jj] : y1[jj - B], acc);
            }
            dx[u] = acc + sa[u];
            sa[u] = 0.f;
        }
        if (kind == 2) {
#pragma unroll
            for (int u = 0; u < B; ++u)
                if (tb + u < t1) dst[((size_t)(tb + u) * H + hh) * D + c] = dx[u];
        } else {
#pragma unroll
            for (int u = 0; u < B; ++u) dxs[b & 1][u][c] = dx[u];
            dx_pending = b;
        }
    }
    __syncthreads();
    if (y_pending >= 0) {  // the last unit's block of y: past the span, nothing to write
        float y2[B];
        finish_y(y_pending, y2);
    }
    if (dx_pending >= 0) finish_dx(dx_pending);
}

// ---- 6. conv filters: partial sums over a span of tokens per (row, channel, tap), then over the spans.
// A CTA per (row, span of at least kWB tokens) with a thread per channel streams the span's conv inputs and
// the gradients y of the conv outputs through a shared-memory ring as in the conv launch, with the last 8
// inputs of each channel in registers (zeros before a sequence's start), so every row is read once.
template <typename Tin, int D>
__global__ void __launch_bounds__(D)
bwd_convw_part_kernel(LayerDims L, const Tin* __restrict__ v, const int32_t* __restrict__ cu,
                      const float* __restrict__ qr, const float* __restrict__ kr, const float* __restrict__ dqt,
                      const float* __restrict__ dkt, const float* __restrict__ dvt, float* __restrict__ part,
                      int64_t span) {
    constexpr int B = kConvWidth;
    __shared__ __align__(16) float xs[kCvRing][B][D];  // conv inputs (v rows use the first half, as Tin)
    __shared__ __align__(16) float ys[kCvRing][B][D];  // gradients of the conv outputs
    const int c = threadIdx.x, r = blockIdx.y, rows = L.Hq + 2 * L.Hkv;
    const int64_t t0 = (int64_t)blockIdx.x * span;
    if (t0 >= L.total) return;  // whole CTA
    const int64_t t1 = min(L.total, t0 + span);
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* src = kind == 0 ? qr : kr;
    const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
    auto issue = [&](int64_t tb, int slot) {
        if (kind == 2)
            stage_rows8<Tin, D>(reinterpret_cast<Tin*>(&xs[slot][0][0]), v, tb, t1, H, hh);
        else
            stage_rows8<float, D>(&xs[slot][0][0], src, tb, t1, H, hh);
        stage_rows8<float, D>(&ys[slot][0][0], dy, tb, t1, H, hh);
        cp_async_commit_group();
    };
    const int64_t n_blk = (t1 - t0 + B - 1) / B;
#pragma unroll
    for (int i = 0; i < kCvRing - 1; ++i) {
        if (i < n_blk) {
            issue(t0 + (int64_t)B * i, i);
        } else {
            cp_async_commit_group();
        }
    }
    int s = seq_of_token(cu, L.n_seqs, t0);
    int64_t s_start, s_len;
    seq_range(cu, s, L.total, &s_start, &s_len);
    float ring[B], acc[kConvWidth];
    ring[0] = 0.f;
#pragma unroll
    for (int m = 0; m < B - 1; ++m) {  // tokens t0 - 7 .. t0 - 1 in slots 1..7: those of t0's sequence
        const int64_t t = t0 - (B - 1) + m;
        const size_t i = ((size_t)t * H + hh) * D + c;
        ring[m + 1] = t >= s_start && t >= 0 ? (kind == 2 ? to_f32(v[i]) : src[i]) : 0.f;
    }
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) acc[m] = 0.f;
#pragma unroll 1
    for (int64_t b = 0; b < n_blk; ++b) {
        const int64_t tb = t0 + B * b;
        cp_async_wait_group<kCvRing - 2>();
        __syncthreads();
        if (b + kCvRing - 1 < n_blk) {
            issue(tb + (int64_t)B * (kCvRing - 1), (int)((b + kCvRing - 1) % kCvRing));
        } else {
            cp_async_commit_group();
        }
        const int slot = (int)(b % kCvRing);
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t t = tb + u;
            while (t >= s_start + s_len && s + 1 < L.n_seqs) {  // uniform over the CTA
                ++s;
                seq_range(cu, s, L.total, &s_start, &s_len);
            }
            if (t == s_start) {  // a sequence starts here: nothing before it
#pragma unroll
                for (int m = 0; m < B; ++m) ring[m] = 0.f;
            }
            ring[u] = kind == 2 ? to_f32(reinterpret_cast<const Tin*>(&xs[slot][0][0])[u * D + c]) : xs[slot][u][c];
            const float d_y = ys[slot][u][c];  // zero past the span
            // tap m multiplies the input at t - 7 + m: slot (u + 1 + m) mod 8
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) acc[m] = fmaf(d_y, ring[(u + 1 + m) & (B - 1)], acc[m]);
        }
    }
    float4* o = reinterpret_cast<float4*>(part + (((size_t)blockIdx.x * rows + r) * D + c) * kConvWidth);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// the sum of the spans' partial sums, in span order; a thread per (row, channel, tap) of the filters
constexpr int kWsThreads = 256;
__global__ void __launch_bounds__(kWsThreads)
bwd_convw_sum_kernel(LayerDims L, int n_spans, const float* __restrict__ part, float* __restrict__ dwq,
                     float* __restrict__ dwk, float* __restrict__ dwv) {
    const int r = blockIdx.x, f = blockIdx.y * kWsThreads + threadIdx.x, D = L.d, rows = L.Hq + 2 * L.Hkv;
    if (f >= D * kConvWidth) return;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const size_t stride = (size_t)rows * D * kConvWidth;
    const float* p = part + (size_t)r * D * kConvWidth + f;
    float s = 0.f;
    int b = 0;
    for (; b + 8 <= n_spans; b += 8) {
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = p[(size_t)(b + k) * stride];
#pragma unroll
        for (int k = 0; k < 8; ++k) s += x[k];
    }
    for (; b < n_spans; ++b) s += p[(size_t)b * stride];
    (kind == 0 ? dwq : kind == 1 ? dwk : dwv)[(size_t)hh * D * kConvWidth + f] = s;
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
    b.convw_part = take(nblk * rows * D * kConvWidth);  // per span of at least kWB tokens
    b.n_blocks = (int)nblk;
    b.n_sm_blocks = (int)(T / kSB + N);                // bounds the 64-row softmax blocks of all sequences
    b.sm_base = take(N + 1);                           // int32
    b.sink_k = take((size_t)b.n_sm_blocks * Hq * (size_t)L.n_sinks * D);
    b.sink_v = take((size_t)b.n_sm_blocks * Hq * (size_t)L.n_sinks * D);
    take(T * D);  // the RoPE angle table, the last region (bwd_ang_offset)
    b.total = off;
    return b;
}

namespace {
// The RoPE cos/sin of every token, a float2 per channel pair (written by the RoPE launch, read by the RoPE
// backward): the last region of the workspace
size_t bwd_ang_offset(const LayerDims& L, const BwdLayout& b) {
    return b.total - ((size_t)L.total * L.d * sizeof(float) + 255) / 256 * 256;
}

// Token spans of a launch with a CTA of `threads` (and smem bytes of dynamic shared memory) per (row, span of
// tokens): the smallest multiple of 8 tokens
// (at least min_span, itself a multiple of 8) for which the grid (spans x rows) is one wave of the CTAs the
// device holds at once
template <class K>
cudaError_t row_span_grid(DeviceCache& cache, K kernel, int threads, size_t smem, int64_t min_span,
                          const LayerDims& L, int64_t* span, dim3* grid) {
    int resident = 0;
    cudaError_t e = device_cached(cache, &resident, [kernel, threads, smem](int dev, int* val) {
        int n_sm = 0, per_sm = 0;
        cudaError_t r = sm_count(dev, &n_sm);
        if (r == cudaSuccess && smem > 48 * 1024)
            r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (r == cudaSuccess) r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
        *val = std::max(1, n_sm * std::max(1, per_sm));
        return r;
    });
    if (e != cudaSuccess) return e;
    const int rows = L.Hq + 2 * L.Hkv;
    const int64_t spans = std::max<int64_t>(1, resident / rows);
    *span = std::max<int64_t>(min_span, ((L.total + spans - 1) / spans + kConvWidth - 1) / kConvWidth * kConvWidth);
    *grid = dim3((unsigned)((L.total + *span - 1) / *span), (unsigned)rows);
    return cudaSuccess;
}
}  // namespace

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
    const size_t T = (size_t)L.total;  // > 0: with no tokens hla_backward returns before the launches
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
    bwd_rope_kernel<Tin><<<(unsigned)T, kRowThreads, 0, st>>>(
        L, q, k, g, cu, F(b.qr), F(b.kr), F(b.alpha), reinterpret_cast<float2*>(ws + bwd_ang_offset(L, b)),
        reinterpret_cast<int32_t*>(ws + b.err));
    if ((e = mark(1)) != cudaSuccess) return e;
    {
        int64_t span = 0;
        dim3 grid;
        if (D == 128) {
            static DeviceCache cache;
            if ((e = row_span_grid(cache, bwd_conv_kernel<Tin, 128>, 128, 0, kConvWidth, L, &span, &grid)) !=
                cudaSuccess)
                return e;
            bwd_conv_kernel<Tin, 128><<<grid, 128, 0, st>>>(L, v, wq, wk, wv, cu, F(b.qr), F(b.kr), F(b.qt),
                                                                     F(b.qh), F(b.kt), F(b.kh), F(b.vh), span);
        } else {
            static DeviceCache cache;
            if ((e = row_span_grid(cache, bwd_conv_kernel<Tin, 64>, 64, 0, kConvWidth, L, &span, &grid)) !=
                cudaSuccess)
                return e;
            bwd_conv_kernel<Tin, 64><<<grid, 64, 0, st>>>(L, v, wq, wk, wv, cu, F(b.qr), F(b.kr), F(b.qt),
                                                                    F(b.qh), F(b.kt), F(b.kh), F(b.vh), span);
        }
    }
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
    if ((e = mark(5)) != cudaSuccess) return e;  // the L2 backward runs inside the next launch
    {
        const FeatOutArgs A{cu,        wq,         wk,         wv,          F(b.qt),    F(b.kt),
                            F(b.dqh),  F(b.dkh_h), F(b.dvh_h), F(b.dqr_sm), F(b.dkr_h), F(b.dv_h),
                            reinterpret_cast<const float2*>(ws + bwd_ang_offset(L, b)),
                            F(b.dqt),  F(b.dkt),   F(b.dvt),   dq,          dk,         dv};
        int64_t span = 0;
        dim3 grid;
        if (D == 128) {
            static DeviceCache cache;
            if ((e = row_span_grid(cache, bwd_feat_out_kernel<128>, 128, feat_out_smem<128>(), kConvWidth, L, &span,
                                   &grid)) != cudaSuccess)
                return e;
            bwd_feat_out_kernel<128><<<grid, 128, feat_out_smem<128>(), st>>>(L, A, span);
        } else {
            static DeviceCache cache;
            if ((e = row_span_grid(cache, bwd_feat_out_kernel<64>, 64, feat_out_smem<64>(), kConvWidth, L, &span,
                                   &grid)) != cudaSuccess)
                return e;
            bwd_feat_out_kernel<64><<<grid, 64, feat_out_smem<64>(), st>>>(L, A, span);
        }
    }
    if ((e = mark(6)) != cudaSuccess) return e;
    {
        int64_t span = 0;
        dim3 grid;  // spans of at least kWB tokens: at most b.n_blocks partial sums
        if (D == 128) {
            static DeviceCache cache;
            if ((e = row_span_grid(cache, bwd_convw_part_kernel<Tin, 128>, 128, 0, kWB, L, &span, &grid)) != cudaSuccess)
                return e;
            bwd_convw_part_kernel<Tin, 128><<<grid, 128, 0, st>>>(L, v, cu, F(b.qr), F(b.kr), F(b.dqt), F(b.dkt),
                                                                   F(b.dvt), F(b.convw_part), span);
        } else {
            static DeviceCache cache;
            if ((e = row_span_grid(cache, bwd_convw_part_kernel<Tin, 64>, 64, 0, kWB, L, &span, &grid)) != cudaSuccess)
                return e;
            bwd_convw_part_kernel<Tin, 64><<<grid, 64, 0, st>>>(L, v, cu, F(b.qr), F(b.kr), F(b.dqt), F(b.dkt),
                                                                 F(b.dvt), F(b.convw_part), span);
        }
        bwd_convw_sum_kernel<<<dim3(rows, (D * kConvWidth + kWsThreads - 1) / kWsThreads), kWsThreads, 0, st>>>(
            L, (int)grid.x, F(b.convw_part), dwq, dwk, dwv);
    }
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
