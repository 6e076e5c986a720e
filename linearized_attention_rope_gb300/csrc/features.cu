// Feature path of the linear branch: RoPE -> causal depthwise short conv
// (width 8) -> L2 norm, on q and k; short conv alone on v.
// Source: "迈向线性的关键：分析驱动的 Transformer 线性化", section 实践建议,
// item 3 (a kernel-8 short convolution after RoPE and before L2
// normalisation).  The RoPE'd q and k are also written out: the exact
// softmax branch reads them (frozen-backbone attention).
#include <algorithm>

#include "hla_common.cuh"

namespace hla {

// RoPE angles at position p = 64 a + b come from two small tables and the
// angle-addition identities, so the per-token work is fp32 only while every
// table entry is formed and range-reduced in double precision.  The same
// launch clears the error word and the item counters and writes the
// per-sequence work tables of the softmax and chunked-GDN kernels, which all
// depend on cu_seqlens alone: one launch ahead of the feature path instead of
// four small ones spread over the step.
__global__ void prefill_tables_kernel(LayerDims L, float2* __restrict__ fine, float2* __restrict__ coarse,
                                      int n_coarse, PrefillTables t) {
    const int half = L.d / 2;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n_fine = 64 * half;
    float c, s;
    if (idx < n_fine) {
        int b = (int)(idx / half), i = (int)(idx % half);
        rope_cs_exact(b, L.theta[i], &c, &s);
        fine[idx] = make_float2(c, s);
    } else if (idx < n_fine + (int64_t)n_coarse * half) {
        int64_t j = idx - n_fine;
        int64_t a = j / half;
        int i = (int)(j % half);
        rope_cs_exact(64 * a, L.theta[i], &c, &s);
        coarse[j] = make_float2(c, s);
    }
    pdl_trigger();  // the features launch may start; it waits for this grid before reading
    if (blockIdx.x != 0) return;
    if (threadIdx.x < 4) t.err[threadIdx.x] = 0;
    if (threadIdx.x < t.n_counters) t.counters[threadIdx.x] = 0;
    if (threadIdx.x == 96 && t.st_pos) {  // the state to fill must be fresh (every position 0)
        bool fresh = true;
        for (int q = 0; q < L.n_seqs; ++q) fresh = fresh && t.st_pos[q] == 0;
        if (!fresh) atomicExch(t.st_err, kErrState);
    }
    // Work tables: base[s] = items of the sequences before s, base[n_seqs] = all.
    int32_t* base = nullptr;
    int per = 1;
    int64_t skip = 0;
    if (threadIdx.x == 32) base = t.blk_base, per = t.blk_rows;                                 // row blocks
    if (threadIdx.x == 64) base = t.chunk_base, per = t.chunk_rows, skip = L.window + L.n_sinks;  // chunks
    if (threadIdx.x == 128) base = t.part_base, per = t.part_rows, skip = L.window + L.n_sinks;   // parts
    if (!base) return;
    int32_t acc = 0;
    for (int q = 0; q < L.n_seqs; ++q) {
        base[q] = acc;
        int64_t start, len;
        seq_range(t.cu, q, L.total, &start, &len);
        const int64_t m = len - skip;
        acc += m > 0 ? (int32_t)((m + per - 1) / per) : 0;
    }
    base[L.n_seqs] = acc;
}

cudaError_t launch_prefill_tables(const LayerDims& L, float2* fine, float2* coarse, int n_coarse,
                                  const PrefillTables& t, cudaStream_t st) {
    if (t.n_counters < 0 || t.n_counters > 32 || (t.blk_base && t.blk_rows <= 0) ||
        (t.chunk_base && t.chunk_rows <= 0) || (t.part_base && t.part_rows <= 0))
        return cudaErrorInvalidValue;
    int64_t n = (int64_t)(64 + n_coarse) * (L.d / 2);
    int blocks = (int)std::max<int64_t>(1, (n + 255) / 256);
    prefill_tables_kernel<<<blocks, 256, 0, st>>>(L, fine, coarse, n_coarse, t);
    return cudaGetLastError();
}

constexpr int kFeatWarps = 4;     // feature rows (q, k or v heads) per CTA, one per warp
constexpr int kBlk = 8;           // tokens per unrolled step = conv width (the window is a ring of 8)
constexpr int kRing = 4;          // steps of input rows in flight per warp (shared-memory ring)

// NP consecutive elements of one lane, as fp32 (loads of the layer's input
// type, stores and rounding of the feature type).
template <typename T, int NP> struct LaneIO;
template <> struct LaneIO<__nv_bfloat16, 2> {
    __device__ static void read(const __nv_bfloat16* p, float* x) {  // shared memory
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        x[0] = f.x; x[1] = f.y;
    }
};
template <> struct LaneIO<__nv_bfloat16, 1> {
    __device__ static void read(const __nv_bfloat16* p, float* x) { x[0] = __bfloat162float(*p); }
};
template <> struct LaneIO<float, 2> {
    __device__ static void read(const float* p, float* x) {
        const float2 f = *reinterpret_cast<const float2*>(p);
        x[0] = f.x; x[1] = f.y;
    }
    __device__ static void store(float* p, const float* x) { *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]); }
    __device__ static void round(float*) {}
};
template <> struct LaneIO<float, 1> {
    __device__ static void read(const float* p, float* x) { x[0] = *p; }
    __device__ static void store(float* p, const float* x) { *p = x[0]; }
    __device__ static void round(float*) {}
};
template <> struct LaneIO<__half, 2> {
    __device__ static void store(__half* p, const float* x) {
        *reinterpret_cast<__half2*>(p) = __floats2half2_rn(x[0], x[1]);
    }
    __device__ static void round(float* x) {
        const float2 f = __half22float2(__floats2half2_rn(x[0], x[1]));
        x[0] = f.x; x[1] = f.y;
    }
};
template <> struct LaneIO<__half, 1> {
    __device__ static void store(__half* p, const float* x) { *p = __float2half_rn(x[0]); }
    __device__ static void round(float* x) { x[0] = __half2float(__float2half_rn(x[0])); }
};

// Per-warp state of one feature row (see features_kernel).
template <typename Tin, typename Tf, int D>
struct FeatRow {
    static constexpr int NP = D / 64, HALF = D / 2, NC = 2 * NP;  // RoPE pairs and channels per lane
    const float2* fine;
    const float2* coarse;
    Tf* rot;       // RoPE'd rows (q and k), lane's first pair already added
    Tf* hat;       // conv (+ norm) rows, lane offset added
    size_t rowstride;  // elements between consecutive tokens of one head
    float2 w[NC / 2][kConvWidth];  // conv taps of channel pairs (2j, 2j + 1) of the lane
    float2 ring[kBlk][NC / 2];      // the last 8 inputs, same pairing
    float2 step1[NP];  // (cos, sin) of one position step for the lane's pairs
};

// Eight tokens t_first .. + 7 of one step, the inputs read from the warp's
// shared-memory slot `rows` (lane offset added).  CHECK = false is the fast
// path: every token has a position p0 + u >= 7 in one sequence and lies
// inside the tensor, so the step is straight-line code the compiler can
// interleave across tokens; CHECK = true tracks sequences token by token,
// masks the conv taps before a sequence's first token and skips the outputs
// of tokens outside every sequence.  OUT = false only fills the ring.
template <typename Tin, typename Tf, int D, bool ROPE, bool NORM, bool CHECK, bool OUT>
__device__ __forceinline__ void feat_step(FeatRow<Tin, Tf, D>& fr, const Tin* rows, int64_t t_first, int p0,
                                          const LayerDims& L, const int32_t* cu, int& s, int64_t& s_start,
                                          int64_t& s_len, int32_t* err, int lane) {
    using Row = FeatRow<Tin, Tf, D>;
    constexpr int NP = Row::NP, HALF = Row::HALF, NC = Row::NC;
    using In = LaneIO<Tin, NP>;
    using Out = LaneIO<Tf, NP>;
    float2 cs_run[NP];  // fast path: (cos, sin) at p0 + u, advanced by one position step per token
#pragma unroll
    for (int u = 0; u < kBlk; ++u) {
        const int64_t t = t_first + u;
        int p = p0 + u;
        if constexpr (CHECK) {  // position in its sequence (-1: outside every sequence); warp-uniform
            p = -1;
            if (t >= 0 && t < L.total) {
                while (t >= s_start + s_len && s + 1 < L.n_seqs) {
                    ++s;
                    seq_range(cu, s, L.total, &s_start, &s_len);
                }
                if (t >= s_start && t < s_start + s_len) p = (int)(t - s_start);
                else if (err && blockIdx.y == 0 && lane == 0) atomicExch(err, kErrSeqlens);
            }
        }
        float x[NC];
        In::read(rows + u * D, x);
        In::read(rows + u * D + HALF, x + NP);
        if constexpr (ROPE) {
            if (!CHECK || p >= 0) {
                float2 csn[NP];
                if (CHECK || u == 0) {  // from the tables (angle addition of two reduced entries)
                    float2 f[NP], g[NP];
                    if constexpr (NP == 2) {  // both pairs' table entries in one 16-byte load per table
                        const float4 fa = __ldg(reinterpret_cast<const float4*>(fr.fine + (p & 63) * HALF + 2 * lane));
                        const float4 ga = __ldg(reinterpret_cast<const float4*>(fr.coarse + (p >> 6) * HALF + 2 * lane));
                        f[0] = make_float2(fa.x, fa.y); f[1] = make_float2(fa.z, fa.w);
                        g[0] = make_float2(ga.x, ga.y); g[1] = make_float2(ga.z, ga.w);
                    } else {
                        f[0] = __ldg(fr.fine + (p & 63) * HALF + lane);
                        g[0] = __ldg(fr.coarse + (p >> 6) * HALF + lane);
                    }
#pragma unroll
                    for (int c = 0; c < NP; ++c)
                        csn[c] = make_float2(g[c].x * f[c].x - g[c].y * f[c].y, g[c].y * f[c].x + g[c].x * f[c].y);
                } else {  // the previous token's angle plus one step (at most 7 steps from a table value)
#pragma unroll
                    for (int c = 0; c < NP; ++c)
                        csn[c] = make_float2(cs_run[c].x * fr.step1[c].x - cs_run[c].y * fr.step1[c].y,
                                             cs_run[c].y * fr.step1[c].x + cs_run[c].x * fr.step1[c].y);
                }
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    cs_run[c] = csn[c];
                    const float a = x[c], b = x[NP + c];
                    x[c] = a * csn[c].x - b * csn[c].y;
                    x[NP + c] = b * csn[c].x + a * csn[c].y;
                }
            }
        }
        Out::round(x);
        Out::round(x + NP);
        const bool out_tok = OUT && (!CHECK || (t < L.total && p >= 0));
        if constexpr (ROPE && OUT) {
            if (out_tok) {
                Tf* dst = fr.rot + (size_t)t * fr.rowstride;
                Out::store(dst, x);
                Out::store(dst + HALF, x + NP);
            }
        }
#pragma unroll
        for (int j = 0; j < NC / 2; ++j) fr.ring[u][j] = make_float2(x[2 * j], x[2 * j + 1]);
        if constexpr (OUT) {
            // tap m reads token t - 7 + m (ring slot (u + 1 + m) mod 8); none before the sequence start;
            // two channels per packed FMA
            float2 y2[NC / 2];
#pragma unroll
            for (int j = 0; j < NC / 2; ++j) y2[j] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) {
                if (CHECK && m < kConvHalo - p) continue;
#pragma unroll
                for (int j = 0; j < NC / 2; ++j) y2[j] = ffma2(fr.w[j][m], fr.ring[(u + 1 + m) & (kBlk - 1)][j], y2[j]);
            }
            float y[NC];
#pragma unroll
            for (int j = 0; j < NC / 2; ++j) { y[2 * j] = y2[j].x; y[2 * j + 1] = y2[j].y; }
            if constexpr (NORM) {
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < NC; ++c) ss = fmaf(y[c], y[c], ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float rs = rsqrtf(ss + 1e-6f);
#pragma unroll
                for (int c = 0; c < NC; ++c) y[c] *= rs;
            }
            if (out_tok) {
                Tf* dst = fr.hat + (size_t)t * fr.rowstride;
                Out::store(dst, y);
                Out::store(dst + HALF, y + NP);
            }
        }
    }
}

// One warp = one feature row (a q, k or v head) over a span of `span` tokens
// (a multiple of 8, chosen by the launcher so the grid is one wave), streamed
// in token order.  Lane l owns the RoPE pairs i = NP l .. NP l + NP - 1 (channels
// i and D/2 + i), so every token row is read and written as coalesced lines
// and the rotation needs no exchange.  Each token is rotated (q and k; cos/sin
// from the fine and coarse tables by angle addition, both reduced in double
// precision), rounded to the feature type and written out as the RoPE'd row,
// then enters a ring of the last 8 inputs held in registers; the width-8
// causal conv of the token is 8 FMAs per channel over the ring, and the L2
// norm a warp reduction.  The warp starts 8 tokens early to fill the ring;
// taps before a sequence's first token read as zero.  Input rows arrive by
// cp.async in steps of 8 tokens, kRing steps in flight per warp, each warp
// with its own slice of shared memory (no CTA-wide barrier).
template <typename Tin, typename Tf, int D, bool ROPE, bool NORM>
__device__ __forceinline__ void feat_row(FeatRow<Tin, Tf, D>& fr, const Tin* src, unsigned char* wring, int64_t tb,
                                         int span, const LayerDims& L, const int32_t* cu, int32_t* err, int lane) {
    constexpr int ROWB = D * (int)sizeof(Tin), STEPB = kBlk * ROWB, CPT = ROWB / 16;  // 16-byte chunks per row
    const int kSteps = span / kBlk + 1;  // the first step only fills the ring
    constexpr int NP = FeatRow<Tin, Tf, D>::NP;
    const size_t H = fr.rowstride / D;
    // sequence of the first token the warp touches (positions advance by one per token)
    int s = seq_of_token(cu, L.n_seqs, tb < 0 ? 0 : tb);
    int64_t s_start, s_len;
    seq_range(cu, s, L.total, &s_start, &s_len);

    // the rows of step `st` into ring slot st % kRing, one commit group per step (empty past the end)
    auto issue = [&](int st) {
        if (st < kSteps) {
            unsigned char* dst = wring + (size_t)(st % kRing) * STEPB;
#pragma unroll
            for (int e = lane; e < kBlk * CPT; e += 32) {
                const int u = e / CPT, ch = e % CPT;
                const int64_t t = tb + (int64_t)kBlk * st + u;
                const bool in = t >= 0 && t < L.total;
                const Tin* gp = src + (size_t)(in ? t : 0) * H * D + ch * (16 / (int)sizeof(Tin));
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                                 (uint32_t)__cvta_generic_to_shared(dst + u * ROWB + ch * 16)),
                             "l"(gp), "r"(in ? 16u : 0u)
                             : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int st = 0; st < kRing - 1; ++st) issue(st);

#pragma unroll 1
    for (int step = 0; step < kSteps; ++step) {
        const int64_t t_first = tb + (int64_t)kBlk * step;
        issue(step + kRing - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
        __syncwarp();
        const Tin* rows = reinterpret_cast<const Tin*>(wring + (size_t)(step % kRing) * STEPB) + NP * lane;
        if (step == 0) {
            feat_step<Tin, Tf, D, ROPE, NORM, true, false>(fr, rows, t_first, 0, L, cu, s, s_start, s_len, err, lane);
        } else {
            // the step's sequence: advance past sequences that end before it
            while (t_first >= s_start + s_len && s + 1 < L.n_seqs) {
                ++s;
                seq_range(cu, s, L.total, &s_start, &s_len);
            }
            const bool fast = t_first >= s_start + kConvHalo && t_first + kBlk <= s_start + s_len &&
                              t_first + kBlk <= L.total;
            if (fast)
                feat_step<Tin, Tf, D, ROPE, NORM, false, true>(fr, rows, t_first, (int)(t_first - s_start), L, cu, s,
                                                               s_start, s_len, err, lane);
            else
                feat_step<Tin, Tf, D, ROPE, NORM, true, true>(fr, rows, t_first, 0, L, cu, s, s_start, s_len, err,
                                                              lane);
        }
        __syncwarp();  // the slot is refilled by the next step's issue
    }
}

template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(32 * kFeatWarps, 4)
features_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                const Tin* __restrict__ v, const float* __restrict__ wq,
                const float* __restrict__ wk, const float* __restrict__ wv,
                const int32_t* __restrict__ cu, const float2* __restrict__ fine,
                const float2* __restrict__ coarse, Tf* __restrict__ qr, Tf* __restrict__ kr,
                Tf* __restrict__ qhat, Tf* __restrict__ khat, Tf* __restrict__ vhat,
                int32_t* __restrict__ err, int span) {
    using Row = FeatRow<Tin, Tf, D>;
    constexpr int NP = Row::NP, HALF = Row::HALF, NC = Row::NC;
    constexpr int STEPB = kBlk * D * (int)sizeof(Tin);
    extern __shared__ __align__(16) unsigned char ring_s[];  // [warp][kRing][kBlk tokens][D]
    pdl_trigger();  // the softmax launch may set up beside this one; it waits for this grid before reading
    pdl_wait();     // after the table launch (no effect on a plain launch)
    const int lane = threadIdx.x & 31;
    unsigned char* wring = ring_s + (size_t)(threadIdx.x >> 5) * kRing * STEPB;
    int hr = blockIdx.y * kFeatWarps + (threadIdx.x >> 5);
    if (hr >= L.Hq + 2 * L.Hkv) return;  // whole warp; no CTA-wide barrier below
    int kind = 0;
    if (hr >= L.Hq + L.Hkv) { kind = 2; hr -= L.Hq + L.Hkv; }
    else if (hr >= L.Hq) { kind = 1; hr -= L.Hq; }
    const int head = hr;
    const size_t H = kind == 0 ? L.Hq : L.Hkv;
    const Tin* src = (kind == 0 ? q : (kind == 1 ? k : v)) + (size_t)head * D;

    Row fr;
    fr.fine = fine;
    fr.coarse = coarse;
#pragma unroll
    for (int c = 0; c < NP; ++c) fr.step1[c] = __ldg(fine + HALF + NP * lane + c);  // angle of position 1
    fr.rowstride = H * D;
    fr.rot = (kind == 0 ? qr : kr) + (size_t)head * D + NP * lane;
    fr.hat = (kind == 0 ? qhat : (kind == 1 ? khat : vhat)) + (size_t)head * D + NP * lane;
    {  // conv weights of the lane's channels: c < NP -> channel NP lane + c, else HALF + NP lane + c - NP
        const float* wb = (kind == 0 ? wq : (kind == 1 ? wk : wv)) + (size_t)head * D * kConvWidth;
        float wc[NC][kConvWidth];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int ch = (c < NP ? 0 : HALF) + NP * lane + (c % NP);
            const float4 a = __ldg(reinterpret_cast<const float4*>(wb + (size_t)ch * kConvWidth));
            const float4 b = __ldg(reinterpret_cast<const float4*>(wb + (size_t)ch * kConvWidth + 4));
            wc[c][0] = a.x; wc[c][1] = a.y; wc[c][2] = a.z; wc[c][3] = a.w;
            wc[c][4] = b.x; wc[c][5] = b.y; wc[c][6] = b.z; wc[c][7] = b.w;
        }
#pragma unroll
        for (int j = 0; j < NC / 2; ++j)
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) fr.w[j][m] = make_float2(wc[2 * j][m], wc[2 * j + 1][m]);
    }
#pragma unroll
    for (int u = 0; u < kBlk; ++u)
#pragma unroll
        for (int j = 0; j < NC / 2; ++j) fr.ring[u][j] = make_float2(0.f, 0.f);

    const int64_t tb = (int64_t)blockIdx.x * span - kBlk;
    if (kind == 2)
        feat_row<Tin, Tf, D, false, false>(fr, src, wring, tb, span, L, cu, err, lane);
    else if (kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q))
        feat_row<Tin, Tf, D, true, true>(fr, src, wring, tb, span, L, cu, err, lane);
    else
        feat_row<Tin, Tf, D, true, false>(fr, src, wring, tb, span, L, cu, err, lane);
}

// Token span per warp: the smallest multiple of 8 for which the whole grid
// (row groups x spans CTAs) fits in one wave of resident CTAs.
static int64_t feature_span(int64_t total, int row_groups, int resident_ctas) {
    const int64_t spans = std::max<int64_t>(1, resident_ctas / std::max(1, row_groups));
    const int64_t span = (total + spans - 1) / spans;
    return std::max<int64_t>(kBlk, (span + kBlk - 1) / kBlk * kBlk);
}

template <typename Tin, typename Tf, int D>
static cudaError_t launch_features_d(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* wq,
                                     const float* wk, const float* wv, const int32_t* cu, const float2* fine,
                                     const float2* coarse, Tf* qr, Tf* kr, Tf* qhat, Tf* khat, Tf* vhat,
                                     int32_t* err, bool after_prior, cudaStream_t st) {
    const size_t smem = (size_t)kFeatWarps * kRing * kBlk * D * sizeof(Tin);
    static DeviceCache cache;  // CTAs resident on the device at once, per device and instantiation
    int resident = 0;
    cudaError_t e = device_cached(cache, &resident, [smem](int dev, int* v) {
        int n_sm = 0, per_sm = 0;
        cudaError_t r = cudaFuncSetAttribute(features_kernel<Tin, Tf, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (r == cudaSuccess) r = sm_count(dev, &n_sm);
        if (r == cudaSuccess)
            r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, features_kernel<Tin, Tf, D>, 32 * kFeatWarps,
                                                              smem);
        *v = std::max(1, n_sm * std::max(1, per_sm));
        return r;
    });
    if (e != cudaSuccess) return e;
    const int row_groups = (L.Hq + 2 * L.Hkv + kFeatWarps - 1) / kFeatWarps;
    const int64_t span = feature_span(L.total, row_groups, resident);
    LaunchCfg lc(dim3((unsigned)((L.total + span - 1) / span), (unsigned)row_groups), dim3(32 * kFeatWarps), smem,
                 st, after_prior);
    return cudaLaunchKernelEx(&lc.cfg, features_kernel<Tin, Tf, D>, L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr,
                              qhat, khat, vhat, err, (int)span);
}

template <typename Tin, typename Tf>
cudaError_t launch_features(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                            const float* wq, const float* wk, const float* wv, const int32_t* cu,
                            const float2* fine, const float2* coarse, Tf* qr, Tf* kr, Tf* qhat,
                            Tf* khat, Tf* vhat, int32_t* err, bool after_prior, cudaStream_t st) {
    if (L.total <= 0) return cudaSuccess;
    if (L.d == 128)
        return launch_features_d<Tin, Tf, 128>(L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr, qhat, khat, vhat,
                                               err, after_prior, st);
    return launch_features_d<Tin, Tf, 64>(L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr, qhat, khat, vhat, err,
                                          after_prior, st);
}

template cudaError_t launch_features<float, float>(const LayerDims&, const float*, const float*,
                                                   const float*, const float*, const float*,
                                                   const float*, const int32_t*, const float2*,
                                                   const float2*, float*, float*, float*, float*,
                                                   float*, int32_t*, bool, cudaStream_t);
template cudaError_t launch_features<__nv_bfloat16, __half>(
    const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*,
    const float*, const float*, const float*, const int32_t*, const float2*, const float2*, __half*,
    __half*, __half*, __half*, __half*, int32_t*, bool, cudaStream_t);

}  // namespace hla
