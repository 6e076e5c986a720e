// Prefill that continues from a decode state, on the tensor-core path (bf16 layer, head_dim 128): the
// throughput form of appending a prompt to live sequences.
//
// The cache of "迈向线性的关键：分析驱动的 Transformer 线性化" (section 填补近似缺口的实用设计) keeps, of
// the context before position pos, only the n_s sinks and the last W positions (the KV ring), their
// features while they wait to be absorbed (the pending ring) and the GDN state S that absorbed the rest
// (section 线性注意力替换机制).  Laid out in front of the new tokens, with the positions between the sinks
// and the window left out, they form an extended sequence of n_old + len rows, n_old = min(pos,
// n_s + W), on which the window rule (sinks, and the W rows before a row) and the delayed absorption
// (row j enters the state W rows after it) hold row for row: a cached row i >= n_s is a token still
// waiting, absorbed W rows later, at a new position.  So the prefill's softmax and chunked GDN kernels
// run unchanged on the extended rows, the GDN starting from the cached S, and the new rows of their
// output are the continuation's output.  Launches:
//  1. the extended sequence table (positions < 0 and overlapping sequences flagged in the state's error
//     word);
//  2. the prefill's work tables on it; rows past the last sequence (up to the workspace's bound) zeroed, the
//     new tokens' gates placed on their rows and their RoPE angles tabulated;
//  3. the cached rows: RoPE'd keys and values from the ring, khat, vhat, g and beta from the pending ring;
//  4. the new rows: RoPE at the true position, the short conv fed by the state's conv histories, L2;
//  5. softmax, chunk-local GDN and GDN state + combine (the prefill's kernels, S from the state);
//  6. the new rows of the output into out;
//  7. the state: ring, pending ring, conv histories (S was written by 5);
//  8. pos += len.
#include <algorithm>

#include "hla_common.cuh"

namespace hla {

namespace {

constexpr int kCD = 128;  // head dim of the tensor-core path
constexpr int kCT = 256;  // threads of the row kernels

__device__ __forceinline__ int64_t cont_ring_slot(int64_t p, int ns, int W) { return p < ns ? p : ns + (p - ns) % W; }
// cached rows in front of the new tokens
__device__ __forceinline__ int64_t cont_n_old(int64_t pos, int ns, int W) {
    return pos < 0 ? 0 : min(pos, (int64_t)ns + W);
}
// true position of cached row i
__device__ __forceinline__ int64_t cont_old_pos(int64_t pos, int64_t i, int ns, int W) {
    return pos <= ns + W || i < ns ? i : pos - W + (i - ns);
}

// 1. ext_cu[n] = the extended rows of the sequences before n (a sequence with pos < 0 has none and is
// flagged; so is a table whose sequences overlap).  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) cont_ext_table_kernel(LayerDims L, const int32_t* __restrict__ cu, hla_state s,
                                                              int32_t* __restrict__ ext_cu) {
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    __shared__ int32_t part[1024];
    const int N = L.n_seqs, tid = threadIdx.x, per = (N + 1023) / 1024;
    const int lo = min(N, tid * per), hi = min(N, lo + per);
    auto rows = [&](int i) -> int32_t {
        int64_t a, len;
        seq_range(cu, i, L.total, &a, &len);
        const int64_t p = s.pos[i];
        return p < 0 ? 0 : (int32_t)(cont_n_old(p, L.n_sinks, L.window) + len);
    };
    // sequences must not overlap (cu non-decreasing once clamped into [0, total]): otherwise their extended
    // rows could add up past the workspace's bound, so the table is flagged and every sequence given ext_cu = 0
    // (the extended rows then overlap, but every row a kernel below forms stays below the bound)
    bool bad = false;
    for (int i = lo; i < hi; ++i) bad = bad || clamp_i64(__ldg(cu + i + 1), 0, L.total) < clamp_i64(__ldg(cu + i), 0, L.total);
    if (__syncthreads_or(bad)) {
        if (tid == 0) atomicExch(s.err, kErrSeqlens);
        for (int i = tid; i <= N; i += 1024) ext_cu[i] = 0;
        return;
    }
    int32_t sum = 0;
    for (int i = lo; i < hi; ++i) {
        if (s.pos[i] < 0) atomicExch(s.err, kErrState);
        sum += rows(i);
    }
    part[tid] = sum;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const int32_t add = tid >= o ? part[tid - o] : 0;
        __syncthreads();
        part[tid] += add;
        __syncthreads();
    }
    int32_t run = tid > 0 ? part[tid - 1] : 0;
    for (int i = lo; i < hi; ++i) {
        ext_cu[i] = run;
        run += rows(i);
    }
    if (tid == 1023) ext_cu[N] = part[1023];
}

// 2b. (i) rows past the last extended row, up to the workspace's bound: zero.  The tensor-core kernels read
// whole tiles, and a tile that runs past a sequence's end must meet finite rows (masked rows are multiplied
// by zero, and zero times a stale non-finite value would not vanish).  (ii) g and beta of every new token onto
// its extended row.  (iii) ang[t][i] = (cos, sin) of p theta_i for every new token t at its true position p
// (angle formed and reduced in double precision), and ang[total][i] that of one position step, read by the
// feature kernel.
__global__ void __launch_bounds__(kCT)
cont_prep_kernel(LayerDims L, LayerDims Lx, const int32_t* __restrict__ cu, hla_state s,
                 const int32_t* __restrict__ ext_cu, __half* __restrict__ qr, __half* __restrict__ kr,
                 __half* __restrict__ qh, __half* __restrict__ kh, __half* __restrict__ vh,
                 __nv_bfloat16* __restrict__ ev, float* __restrict__ eg, float* __restrict__ eb,
                 const float* __restrict__ g, const float* __restrict__ beta, float2* __restrict__ ang) {
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    const int64_t first = __ldg(ext_cu + Lx.n_seqs);
    const int D = kCD, HALF = kCD / 2;
    for (int64_t r = first + blockIdx.x; r < Lx.total; r += gridDim.x) {
        for (int idx = threadIdx.x; idx < Lx.Hq * D; idx += kCT) {
            qr[r * Lx.Hq * D + idx] = __float2half_rn(0.f);
            qh[r * Lx.Hq * D + idx] = __float2half_rn(0.f);
        }
        for (int idx = threadIdx.x; idx < Lx.Hkv * D; idx += kCT) {
            kr[r * Lx.Hkv * D + idx] = __float2half_rn(0.f);
            kh[r * Lx.Hkv * D + idx] = __float2half_rn(0.f);
            vh[r * Lx.Hkv * D + idx] = __float2half_rn(0.f);
            ev[r * Lx.Hkv * D + idx] = __float2bfloat16_rn(0.f);
        }
        for (int h = threadIdx.x; h < Lx.Hq; h += kCT) {
            eg[r * Lx.Hq + h] = 0.f;
            eb[r * Lx.Hq + h] = 0.f;
        }
    }
    const int64_t stride = (int64_t)gridDim.x * kCT, id = (int64_t)blockIdx.x * kCT + threadIdx.x;
    // (token, item) pairs: the 64 angles of a token are two whole warps, the gates of a token one warp when
    // Hq = 32, so the sequence lookup is warp-uniform there
    for (int64_t idx = id; idx < (L.total + 1) * HALF; idx += stride) {
        const int64_t t = idx / HALF;
        const int i = (int)(idx % HALF);
        int64_t p = 1;
        if (t < L.total) {
            const int n = seq_of_token(cu, L.n_seqs, t);
            int64_t start, len;
            seq_range(cu, n, L.total, &start, &len);
            const int64_t pos = s.pos[n];
            p = pos >= 0 && t >= start && t < start + len ? pos + (t - start) : 0;
        }
        float c, sv;
        rope_cs_exact(p, L.theta[i], &c, &sv);
        ang[idx] = make_float2(c, sv);
    }
    for (int64_t idx = id; idx < L.total * L.Hq; idx += stride) {
        const int64_t t = idx / L.Hq;
        const int h = (int)(idx % L.Hq);
        const int n = seq_of_token(cu, L.n_seqs, t);
        int64_t start, len;
        seq_range(cu, n, L.total, &start, &len);
        const int64_t pos = s.pos[n];
        if (pos < 0 || t < start || t >= start + len) continue;
        const size_t e = (size_t)__ldg(ext_cu + n) + (size_t)cont_n_old(pos, L.n_sinks, L.window) + (size_t)(t - start);
        eg[e * L.Hq + h] = g[idx];
        eb[e * L.Hq + h] = beta[idx];
    }
}

// 3. the cached rows: CTA per (cached row i, sequence)
__global__ void __launch_bounds__(kCT)
cont_gather_kernel(LayerDims L, hla_state s, const int32_t* __restrict__ ext_cu, __half* __restrict__ qr,
                   __half* __restrict__ kr, __half* __restrict__ qh, __half* __restrict__ kh, __half* __restrict__ vh,
                   __nv_bfloat16* __restrict__ ev, float* __restrict__ eg, float* __restrict__ eb) {
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    const int i = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
    const int ns = L.n_sinks, W = L.window, P = W + 1, R = ns + W, D = kCD;
    const int64_t pos = s.pos[n];
    if (pos < 0 || i >= cont_n_old(pos, ns, W)) return;
    const int64_t tp = cont_old_pos(pos, i, ns, W);
    const size_t e = (size_t)__ldg(ext_cu + n) + i, slot = (size_t)cont_ring_slot(tp, ns, W);
    // every cached non-sink token is still waiting to be absorbed (it sits in the last W positions, or
    // the window has never filled)
    const bool pend = tp >= ns;
    const size_t pslot = (size_t)(tp % P);
    const __nv_bfloat16* kring = static_cast<const __nv_bfloat16*>(s.k_ring) + (size_t)n * L.Hkv * R * D;
    const __nv_bfloat16* vring = static_cast<const __nv_bfloat16*>(s.v_ring) + (size_t)n * L.Hkv * R * D;
    for (int idx = tid; idx < L.Hkv * D; idx += kCT) {
        const int kv = idx / D, c = idx % D;
        const size_t o = (e * L.Hkv + kv) * D + c, r = ((size_t)kv * R + slot) * D + c;
        kr[o] = __float2half_rn(__bfloat162float(kring[r]));
        ev[o] = vring[r];
        const size_t ps = (((size_t)n * L.Hkv + kv) * P + pslot) * D + c;
        kh[o] = __float2half_rn(pend ? s.pend_k[ps] : 0.f);
        vh[o] = __float2half_rn(pend ? s.pend_v[ps] : 0.f);
    }
    for (int idx = tid; idx < L.Hq * D; idx += kCT) {  // the cached rows' queries are never read out
        qr[e * L.Hq * D + idx] = __float2half_rn(0.f);
        qh[e * L.Hq * D + idx] = __float2half_rn(0.f);
    }
    for (int h = tid; h < L.Hq; h += kCT) {
        const size_t gs = ((size_t)n * L.Hq + h) * P + pslot;
        eg[e * L.Hq + h] = pend ? s.pend_g[gs] : 0.f;
        eb[e * L.Hq + h] = pend ? s.pend_beta[gs] : 0.f;
    }
}

// 4. the new rows.  A warp per (feature row, span of new tokens): q-heads, then k-heads, then v-heads, 4 rows
// to a CTA, the span a multiple of 8 tokens chosen so that the grid is one wave.  Lane l owns the RoPE pairs
// 2l and 2l + 1 (channels 2l, 2l + 1, 64 + 2l, 64 + 2l + 1), so every row is read and written as whole lines.
// The warp walks its span in steps of 8 tokens, the input rows of 4 steps in flight by cp.async in the warp's
// slice of shared memory (no CTA-wide barrier).  Each token is rotated at its true position (the angle from
// the table at a step's first token, then advanced by one position step per token), stored as the RoPE'd row,
// and enters a register ring of the last 8 inputs; the width-8 causal conv reads the ring, except for the
// taps of a sequence's first 7 new tokens that fall before the call, which read the state's conv history of
// that sequence (the roped inputs of positions pos - 7 .. pos - 1; none before position 0).  The conv of q
// and k is L2-normalised (q only under HLA_FLAG_L2NORM_Q); the v rows also keep the raw value for the softmax.
// Every output lands on the token's extended row, t + (ext_cu[n] + n_old - start of n) for its sequence n.
constexpr int kFW = 4;     // feature rows (warps) per CTA
constexpr int kFB = 8;     // tokens per step = conv width
constexpr int kFRing = 4;  // steps of input rows in flight per warp
constexpr size_t kFeatSmem = (size_t)kFW * kFRing * kFB * kCD * sizeof(__nv_bfloat16);

struct ContSeq {  // the sequence a warp is in (token indices fit the int32 sequence table)
    int n, start, len;
    int pos7;  // its position before the call, clamped to [-1, 7] (-1: not live; 7: no tap reaches position 0)
    int off;   // extended row minus token index
};
__device__ __forceinline__ void cont_seq_at(const LayerDims& L, const int32_t* cu, const hla_state& s,
                                            const int32_t* ext_cu, int n, ContSeq& q) {
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t pos = s.pos[n];
    q.n = n;
    q.start = (int)start;
    q.len = (int)len;
    q.pos7 = pos < 0 ? -1 : (int)min(pos, (int64_t)kConvHalo);
    q.off = pos < 0 ? 0 : (int)((int64_t)__ldg(ext_cu + n) + cont_n_old(pos, L.n_sinks, L.window) - start);
}

struct ContRow {
    const float2* ang;   // angle table, lane's first pair added
    const float* hist;   // conv history of the row (n = 0, m = 0), lane's first channel added
    size_t hstride;      // floats between consecutive (n, m) entries of the history
    __half* rot;         // RoPE'd rows (q, k), head and lane offsets added
    __half* hat;         // conv (+ norm) rows
    __nv_bfloat16* raw;  // v: the raw rows
    size_t rowstride;    // elements between consecutive rows of one head
    float2 w[2][kConvWidth];   // taps of the channel pairs (2l, 2l + 1) and (64 + 2l, 64 + 2l + 1)
    float2 ring[kFB][2];       // the last 8 inputs, same pairing
    float2 step1[2];           // (cos, sin) of one position step for the lane's pairs
};

// Eight tokens t_first .. + 7, the inputs in the warp's slot `rows` (lane offset added).  CHECK = false: every
// token lies in one live sequence at index >= 7 (straight-line code); CHECK = true follows the sequences token
// by token, skips tokens of no live sequence and feeds the early taps from the history.  OUT = false only
// fills the ring.
template <bool ROPE, bool NORM, bool CHECK, bool OUT>
__device__ __forceinline__ void cont_feat_step(ContRow& fr, const __nv_bfloat16* rows, int64_t t_first, ContSeq& sq,
                                               const LayerDims& L, const int32_t* cu, const hla_state& s,
                                               const int32_t* ext_cu) {
    constexpr int HALF = kCD / 2;
    float2 cs_run[2];
#pragma unroll
    for (int u = 0; u < kFB; ++u) {
        const int64_t t = t_first + u;
        bool live = true;
        if constexpr (CHECK) {  // warp-uniform
            live = false;
            if (t >= 0 && t < L.total) {
                while (t >= sq.start + sq.len && sq.n + 1 < L.n_seqs) cont_seq_at(L, cu, s, ext_cu, sq.n + 1, sq);
                live = sq.pos7 >= 0 && t >= sq.start && t < sq.start + sq.len;
            }
        }
        const __nv_bfloat162 r0 = *reinterpret_cast<const __nv_bfloat162*>(rows + u * kCD);
        const __nv_bfloat162 r1 = *reinterpret_cast<const __nv_bfloat162*>(rows + u * kCD + HALF);
        const float2 a0 = __bfloat1622float2(r0), a1 = __bfloat1622float2(r1);
        float x[4] = {a0.x, a0.y, a1.x, a1.y};  // channels 2l, 2l + 1, 64 + 2l, 64 + 2l + 1
        if constexpr (ROPE) {
            if (live) {
                float2 csn[2];
                if (CHECK || u == 0) {
                    const float4 f = __ldg(reinterpret_cast<const float4*>(fr.ang + (size_t)t * HALF));
                    csn[0] = make_float2(f.x, f.y);
                    csn[1] = make_float2(f.z, f.w);
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        csn[c] = make_float2(cs_run[c].x * fr.step1[c].x - cs_run[c].y * fr.step1[c].y,
                                             cs_run[c].y * fr.step1[c].x + cs_run[c].x * fr.step1[c].y);
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    cs_run[c] = csn[c];
                    const float p1 = x[c], p2 = x[2 + c];
                    x[c] = p1 * csn[c].x - p2 * csn[c].y;
                    x[2 + c] = p2 * csn[c].x + p1 * csn[c].y;
                }
            }
        }
        fr.ring[u][0] = make_float2(x[0], x[1]);
        fr.ring[u][1] = make_float2(x[2], x[3]);
        if constexpr (OUT) {
            if (!live) continue;
            // tap m reads token t - 7 + m (ring slot (u + 1 + m) mod 8); in CHECK mode, taps before the
            // sequence's first new token read the history entry i + m (position pos - 7 + i + m)
            const int64_t i = t - sq.start;
            float2 y2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) {
                float2 in0 = fr.ring[(u + 1 + m) & (kFB - 1)][0], in1 = fr.ring[(u + 1 + m) & (kFB - 1)][1];
                if (CHECK && i + m < kConvHalo) {
                    if (sq.pos7 + i - kConvHalo + m < 0) {
                        in0 = in1 = make_float2(0.f, 0.f);
                    } else {
                        const float* h = fr.hist + ((size_t)sq.n * kConvHalo + (size_t)(i + m)) * fr.hstride;
                        in0 = *reinterpret_cast<const float2*>(h);
                        in1 = *reinterpret_cast<const float2*>(h + HALF);
                    }
                }
                y2[0] = ffma2(fr.w[0][m], in0, y2[0]);
                y2[1] = ffma2(fr.w[1][m], in1, y2[1]);
            }
            if constexpr (NORM) {
                float ss = y2[0].x * y2[0].x;
                ss = fmaf(y2[0].y, y2[0].y, ss);
                ss = fmaf(y2[1].x, y2[1].x, ss);
                ss = fmaf(y2[1].y, y2[1].y, ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float rs = rsqrtf(ss + 1e-6f);
                y2[0].x *= rs; y2[0].y *= rs; y2[1].x *= rs; y2[1].y *= rs;
            }
            const size_t o = (size_t)(t + sq.off) * fr.rowstride;
            *reinterpret_cast<__half2*>(fr.hat + o) = __floats2half2_rn(y2[0].x, y2[0].y);
            *reinterpret_cast<__half2*>(fr.hat + o + HALF) = __floats2half2_rn(y2[1].x, y2[1].y);
            if constexpr (ROPE) {
                *reinterpret_cast<__half2*>(fr.rot + o) = __floats2half2_rn(x[0], x[1]);
                *reinterpret_cast<__half2*>(fr.rot + o + HALF) = __floats2half2_rn(x[2], x[3]);
            } else {
                *reinterpret_cast<__nv_bfloat162*>(fr.raw + o) = r0;
                *reinterpret_cast<__nv_bfloat162*>(fr.raw + o + HALF) = r1;
            }
        }
    }
}

template <bool ROPE, bool NORM>
__device__ __forceinline__ void cont_feat_row(ContRow& fr, const __nv_bfloat16* src, size_t H, unsigned char* wring,
                                              int64_t tb, int span, const LayerDims& L, const int32_t* cu,
                                              const hla_state& s, const int32_t* ext_cu, int lane) {
    constexpr int ROWB = kCD * (int)sizeof(__nv_bfloat16), STEPB = kFB * ROWB, CPT = ROWB / 16;
    const int n_steps = span / kFB + 1;  // the first step only fills the ring
    ContSeq sq;
    cont_seq_at(L, cu, s, ext_cu, seq_of_token(cu, L.n_seqs, tb < 0 ? 0 : tb), sq);
    // the rows of step `st` into slot st % kFRing, one commit group per step (empty past the end)
    auto issue = [&](int st) {
        if (st < n_steps) {
            unsigned char* dst = wring + (size_t)(st % kFRing) * STEPB;
#pragma unroll
            for (int e = lane; e < kFB * CPT; e += 32) {
                const int u = e / CPT, ch = e % CPT;
                const int64_t t = tb + (int64_t)kFB * st + u;
                const bool in = t >= 0 && t < L.total;
                const __nv_bfloat16* gp = src + (size_t)(in ? t : 0) * H * kCD + ch * 8;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                                 (uint32_t)__cvta_generic_to_shared(dst + u * ROWB + ch * 16)),
                             "l"(gp), "r"(in ? 16u : 0u)
                             : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int st = 0; st < kFRing - 1; ++st) issue(st);
#pragma unroll 1
    for (int step = 0; step < n_steps; ++step) {
        const int64_t t_first = tb + (int64_t)kFB * step;
        issue(step + kFRing - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(kFRing - 1) : "memory");
        __syncwarp();
        const __nv_bfloat16* rows = reinterpret_cast<const __nv_bfloat16*>(wring + (size_t)(step % kFRing) * STEPB) +
                                    2 * lane;
        if (step == 0) {
            cont_feat_step<ROPE, NORM, true, false>(fr, rows, t_first, sq, L, cu, s, ext_cu);
        } else {
            while (t_first >= sq.start + sq.len && sq.n + 1 < L.n_seqs) cont_seq_at(L, cu, s, ext_cu, sq.n + 1, sq);
            const bool fast = sq.pos7 >= 0 && t_first >= sq.start + kConvHalo && t_first + kFB <= sq.start + sq.len &&
                              t_first + kFB <= L.total;
            if (fast)
                cont_feat_step<ROPE, NORM, false, true>(fr, rows, t_first, sq, L, cu, s, ext_cu);
            else
                cont_feat_step<ROPE, NORM, true, true>(fr, rows, t_first, sq, L, cu, s, ext_cu);
        }
        __syncwarp();  // the slot is refilled by the next step's issue
    }
}

__global__ void __launch_bounds__(32 * kFW, 4)
cont_features_kernel(LayerDims L, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     const __nv_bfloat16* __restrict__ v, const float* __restrict__ wq, const float* __restrict__ wk,
                     const float* __restrict__ wv, const int32_t* __restrict__ cu, hla_state s,
                     const int32_t* __restrict__ ext_cu, const float2* __restrict__ ang, __half* __restrict__ qr,
                     __half* __restrict__ kr, __half* __restrict__ qh, __half* __restrict__ kh,
                     __half* __restrict__ vh, __nv_bfloat16* __restrict__ ev, int span) {
    constexpr int D = kCD, HALF = D / 2;
    extern __shared__ __align__(16) unsigned char ring_s[];  // [warp][kFRing][kFB tokens][D]
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    unsigned char* wring = ring_s + (size_t)(threadIdx.x >> 5) * kFRing * kFB * D * sizeof(__nv_bfloat16);
    int head = blockIdx.y * kFW + (threadIdx.x >> 5);
    if (head >= L.Hq + 2 * L.Hkv) return;  // whole warp; no CTA-wide barrier below
    int kind = 0;
    if (head >= L.Hq + L.Hkv) { kind = 2; head -= L.Hq + L.Hkv; }
    else if (head >= L.Hq) { kind = 1; head -= L.Hq; }
    const size_t H = kind == 0 ? L.Hq : L.Hkv;
    const __nv_bfloat16* src = (kind == 0 ? q : (kind == 1 ? k : v)) + (size_t)head * D;
    ContRow fr;
    fr.ang = ang + 2 * lane;
    fr.hist = (kind == 0 ? s.conv_q : (kind == 1 ? s.conv_k : s.conv_v)) + (size_t)head * D + 2 * lane;
    fr.hstride = H * D;
    fr.rowstride = H * D;
    fr.rot = (kind == 0 ? qr : kr) + (size_t)head * D + 2 * lane;
    fr.hat = (kind == 0 ? qh : (kind == 1 ? kh : vh)) + (size_t)head * D + 2 * lane;
    fr.raw = ev + (size_t)head * D + 2 * lane;
    {
        const float4 f = __ldg(reinterpret_cast<const float4*>(fr.ang + (size_t)L.total * HALF));
        fr.step1[0] = make_float2(f.x, f.y);
        fr.step1[1] = make_float2(f.z, f.w);
    }
    {  // conv taps: pair j = 0 -> channels 2l, 2l + 1; j = 1 -> 64 + 2l, 64 + 2l + 1
        const float* wb = (kind == 0 ? wq : (kind == 1 ? wk : wv)) + (size_t)head * D * kConvWidth;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float wc[2][kConvWidth];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float4* w4 = reinterpret_cast<const float4*>(wb + (size_t)(j * HALF + 2 * lane + c) * kConvWidth);
                const float4 a = __ldg(w4), b = __ldg(w4 + 1);
                wc[c][0] = a.x; wc[c][1] = a.y; wc[c][2] = a.z; wc[c][3] = a.w;
                wc[c][4] = b.x; wc[c][5] = b.y; wc[c][6] = b.z; wc[c][7] = b.w;
            }
#pragma unroll
            for (int m = 0; m < kConvWidth; ++m) fr.w[j][m] = make_float2(wc[0][m], wc[1][m]);
        }
    }
#pragma unroll
    for (int u = 0; u < kFB; ++u) fr.ring[u][0] = fr.ring[u][1] = make_float2(0.f, 0.f);
    const int64_t tb = (int64_t)blockIdx.x * span - kFB;
    if (kind == 2)
        cont_feat_row<false, false>(fr, src, H, wring, tb, span, L, cu, s, ext_cu, lane);
    else if (kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q))
        cont_feat_row<true, true>(fr, src, H, wring, tb, span, L, cu, s, ext_cu, lane);
    else
        cont_feat_row<true, false>(fr, src, H, wring, tb, span, L, cu, s, ext_cu, lane);
}

// 6. the new rows of the extended output into out (16-byte copies)
__global__ void __launch_bounds__(kCT)
cont_out_kernel(LayerDims L, const int32_t* __restrict__ cu, hla_state s, const int32_t* __restrict__ ext_cu,
                const __nv_bfloat16* __restrict__ eo, __nv_bfloat16* __restrict__ out) {
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    const int64_t t = blockIdx.x;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t pos = s.pos[n];
    if (pos < 0 || t < start || t >= start + len) return;
    const size_t e = (size_t)__ldg(ext_cu + n) + (size_t)cont_n_old(pos, L.n_sinks, L.window) + (size_t)(t - start);
    const uint4* src = reinterpret_cast<const uint4*>(eo + e * L.Hq * kCD);
    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)t * L.Hq * kCD);
    for (int idx = threadIdx.x; idx < L.Hq * kCD / 8; idx += kCT) dst[idx] = src[idx];
}

// 7. the state after the call.  CTA per (sequence, y): y = 0: the pending gates; y = 1 + h: q-head h's conv
// history; y = 1 + Hq + kv: kv head kv's k and v conv histories; y = 1 + Hq + Hkv + kStGroups kv + j: group j
// of the new rows of kv head kv that stay in the ring (new sinks and the final window) and in the pending
// ring.  RoPE angles of new tokens come from the table of step 2.  Loads are issued in batches ahead of their
// stores.
constexpr int kStGroups = 8;
template <typename Tin>
__global__ void __launch_bounds__(kCT)
cont_state_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta, const int32_t* __restrict__ cu,
                  hla_state s, const int32_t* __restrict__ ext_cu, const __half* __restrict__ kh,
                  const __half* __restrict__ vh, const float2* __restrict__ ang) {
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    constexpr int D = kCD, HALF = D / 2;
    const int n = blockIdx.x, y = blockIdx.y, tid = threadIdx.x;
    const int ns = L.n_sinks, W = L.window, P = W + 1, R = ns + W;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t pos = s.pos[n];
    if (pos < 0 || len == 0) return;
    const int64_t p_end = pos + len;
    // channel c of new token i, RoPE'd (c and c +- d/2 form a pair; the angle from the table)
    auto rope = [&](const Tin* row, int c, int64_t i) {
        const int ii = c % HALF;
        const float2 cs = __ldg(ang + (size_t)(start + i) * HALF + ii);
        const float x1 = to_f32(row[ii]), x2 = to_f32(row[ii + HALF]);
        return c < HALF ? x1 * cs.x - x2 * cs.y : x2 * cs.x + x1 * cs.y;
    };
    // conv history of a row (H heads, head hh): entry m <- position p_end - 7 + m; the values are all read
    // (old entries from m + len) before any is written
    auto advance_history = [&](float* hist, const Tin* src, int H, int hh, bool rotate) {
        constexpr int PER = (kConvHalo * D + kCT - 1) / kCT;
        float val[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int idx = tid + u * kCT, m = idx / D, c = idx % D;
            val[u] = 0.f;
            if (idx >= kConvHalo * D) continue;
            const int64_t pp = p_end - kConvHalo + m;
            if (pp >= pos) {
                const Tin* row = src + ((size_t)(start + (pp - pos)) * H + hh) * D;
                val[u] = rotate ? rope(row, c, pp - pos) : to_f32(row[c]);
            } else if (pp >= 0) {
                val[u] = hist[(((size_t)n * kConvHalo + (size_t)(m + len)) * H + hh) * D + c];
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int idx = tid + u * kCT, m = idx / D, c = idx % D;
            if (idx < kConvHalo * D) hist[(((size_t)n * kConvHalo + m) * H + hh) * D + c] = val[u];
        }
    };
    if (y == 0) {  // gates of the new tokens still waiting to be absorbed
        constexpr int U = 8;
        const int64_t i0 = max((int64_t)0, max(len - W, ns - pos));
        for (int64_t b = i0 * L.Hq + tid; b < len * L.Hq; b += (int64_t)U * kCT) {
            float gv[U], bv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = b + (int64_t)u * kCT;
                if (i < len * L.Hq) {
                    gv[u] = g[(size_t)(start * L.Hq + i)];
                    bv[u] = beta[(size_t)(start * L.Hq + i)];
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = b + (int64_t)u * kCT;
                if (i >= len * L.Hq) continue;
                const int64_t tt = i / L.Hq, p = pos + tt;
                const int h = (int)(i % L.Hq);
                const size_t gs = ((size_t)n * L.Hq + h) * P + (size_t)(p % P);
                s.pend_g[gs] = gv[u];
                s.pend_beta[gs] = bv[u];
            }
        }
        return;
    }
    if (y <= L.Hq) {  // a q-head's conv history
        advance_history(s.conv_q, q, L.Hq, y - 1, true);
        return;
    }
    if (y <= L.Hq + L.Hkv) {  // a kv head's conv histories
        const int kv = y - 1 - L.Hq;
        advance_history(s.conv_k, k, L.Hkv, kv, true);
        advance_history(s.conv_v, v, L.Hkv, kv, false);
        return;
    }
    const int kv = (y - 1 - L.Hq - L.Hkv) / kStGroups, grp = (y - 1 - L.Hq - L.Hkv) % kStGroups;
    Tin* kring = static_cast<Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    Tin* vring = static_cast<Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    // the rows that stay: new sinks [0, i_sink) and the final window [i_win, len); this CTA's share of them
    const int64_t first = max((int64_t)0, min(len, p_end - W - pos));  // index of the first final-window token
    const int64_t i_sink = min(len, max((int64_t)0, ns - pos));
    const int64_t i_win = max(first, i_sink);
    const int64_t n_rows = i_sink + (len - i_win);
    const int64_t per = (n_rows + kStGroups - 1) / kStGroups;
    const int64_t r_lo = min(n_rows, grp * per), r_hi = min(n_rows, r_lo + per);
    auto row_of = [&](int64_t r) { return r < i_sink ? r : i_win + (r - i_sink); };
    const size_t e0 = (size_t)__ldg(ext_cu + n) + (size_t)cont_n_old(pos, ns, W);  // extended row of position pos
    constexpr int U = 4;
    for (int64_t b = r_lo * HALF + tid; b < r_hi * HALF; b += (int64_t)U * kCT) {  // RoPE'd key pairs
        float2 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t idx = b + (int64_t)u * kCT;
            if (idx >= r_hi * HALF) continue;
            const int64_t i = row_of(idx / HALF);
            const int ii = (int)(idx % HALF);
            const Tin* row = k + ((size_t)(start + i) * L.Hkv + kv) * D;
            val[u] = make_float2(rope(row, ii, i), rope(row, ii + HALF, i));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t idx = b + (int64_t)u * kCT;
            if (idx >= r_hi * HALF) continue;
            const int64_t i = row_of(idx / HALF);
            const int ii = (int)(idx % HALF);
            const size_t slot = (size_t)cont_ring_slot(pos + i, ns, W) * D;
            kring[slot + ii] = from_f32<Tin>(val[u].x);
            kring[slot + ii + HALF] = from_f32<Tin>(val[u].y);
        }
    }
    for (int64_t b = r_lo * D + tid; b < r_hi * D; b += (int64_t)U * kCT) {  // values and pending features
        Tin vv[U];
        float pk[U], pv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t idx = b + (int64_t)u * kCT;
            if (idx >= r_hi * D) continue;
            const int64_t i = row_of(idx / D);
            const int c = (int)(idx % D);
            vv[u] = v[((size_t)(start + i) * L.Hkv + kv) * D + c];
            const size_t er = ((e0 + (size_t)i) * L.Hkv + kv) * D + c;
            pk[u] = __half2float(kh[er]);
            pv[u] = __half2float(vh[er]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t idx = b + (int64_t)u * kCT;
            if (idx >= r_hi * D) continue;
            const int64_t i = row_of(idx / D), p = pos + i;
            const int c = (int)(idx % D);
            vring[(size_t)cont_ring_slot(p, ns, W) * D + c] = vv[u];
            if (p >= ns && p >= p_end - W) {
                const size_t ps = (((size_t)n * L.Hkv + kv) * P + (size_t)(p % P)) * D + c;
                s.pend_k[ps] = pk[u];
                s.pend_v[ps] = pv[u];
            }
        }
    }
}

// 8. pos += len, after every launch above has read it
__global__ void cont_tc_advance_kernel(LayerDims L, const int32_t* __restrict__ cu, int64_t* __restrict__ pos) {
    pdl_wait();  // programmatic dependent launch: the launch before this one has completed
    pdl_trigger();
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= L.n_seqs) return;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    if (pos[n] >= 0) pos[n] += len;
}

}  // namespace

cudaError_t launch_continue_table(const LayerDims& L, const int32_t* cu, const hla_state& s, int32_t* ext_cu,
                                  cudaStream_t st) {
    if (L.d != kCD) return cudaErrorInvalidValue;
    LaunchCfg lc(dim3(1), dim3(1024), 0, st, true);
    return cudaLaunchKernelEx(&lc.cfg, cont_ext_table_kernel, L, cu, s, ext_cu);
}

cudaError_t launch_continue_rows(const LayerDims& L, const LayerDims& Lx, const int32_t* cu, const hla_state& s,
                                 const int32_t* ext_cu, __half* qr, __half* kr, __half* qh, __half* kh, __half* vh,
                                 __nv_bfloat16* ev, float* eg, float* eb, float2* ang, const __nv_bfloat16* q,
                                 const __nv_bfloat16* k, const __nv_bfloat16* v, const float* g, const float* beta,
                                 const float* wq, const float* wk, const float* wv, cudaStream_t st) {
    {
        LaunchCfg lc(dim3(1024), dim3(kCT), 0, st, true);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, cont_prep_kernel, L, Lx, cu, s, ext_cu, qr, kr, qh, kh, vh, ev, eg, eb,
                                           g, beta, ang);
        if (e != cudaSuccess) return e;
    }
    {
        LaunchCfg lc(dim3(L.n_sinks + L.window, L.n_seqs), dim3(kCT), 0, st, true);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, cont_gather_kernel, L, s, ext_cu, qr, kr, qh, kh, vh, ev, eg, eb);
        if (e != cudaSuccess) return e;
    }
    if (L.total > 0) {
        static DeviceCache cache;  // CTAs of the feature kernel resident on the device at once
        int resident = 0;
        cudaError_t e = device_cached(cache, &resident, [](int dev, int* val) {
            int n_sm = 0, per_sm = 0;
            cudaError_t r = sm_count(dev, &n_sm);
            if (r == cudaSuccess)
                r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cont_features_kernel, 32 * kFW, kFeatSmem);
            *val = std::max(1, n_sm * std::max(1, per_sm));
            return r;
        });
        if (e != cudaSuccess) return e;
        // the smallest multiple of 8 tokens per span for which the grid (spans x row groups) is one wave
        const int row_groups = (L.Hq + 2 * L.Hkv + kFW - 1) / kFW;
        const int64_t spans = std::max<int64_t>(1, resident / row_groups);
        const int64_t span = std::max<int64_t>(kFB, ((L.total + spans - 1) / spans + kFB - 1) / kFB * kFB);
        const dim3 grid((unsigned)((L.total + span - 1) / span), (unsigned)row_groups);
        LaunchCfg lc(grid, dim3(32 * kFW), kFeatSmem, st, true);
        e = cudaLaunchKernelEx(&lc.cfg, cont_features_kernel, L, q, k, v, wq, wk, wv, cu, s, ext_cu,
                               static_cast<const float2*>(ang), qr, kr, qh, kh, vh, ev, (int)span);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_continue_finish(const LayerDims& L, const int32_t* cu, const hla_state& s, const int32_t* ext_cu,
                                   const __nv_bfloat16* ext_out, __nv_bfloat16* out, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v, const float* g, const float* beta,
                                   const __half* kh, const __half* vh, const float2* ang, cudaStream_t st) {
    if (L.total > 0) {
        LaunchCfg lc(dim3((unsigned)L.total), dim3(kCT), 0, st, true);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, cont_out_kernel, L, cu, s, ext_cu, ext_out, out);
        if (e != cudaSuccess) return e;
    }
    {
        LaunchCfg lc(dim3(L.n_seqs, 1 + L.Hq + L.Hkv * (1 + kStGroups)), dim3(kCT), 0, st, true);
        cudaError_t e = cudaLaunchKernelEx(&lc.cfg, cont_state_kernel<__nv_bfloat16>, L, q, k, v, g, beta, cu, s, ext_cu,
                                           kh, vh, ang);
        if (e != cudaSuccess) return e;
    }
    LaunchCfg lc(dim3((L.n_seqs + 127) / 128), dim3(128), 0, st, true);
    return cudaLaunchKernelEx(&lc.cfg, cont_tc_advance_kernel, L, cu, s.pos);
}

}  // namespace hla
