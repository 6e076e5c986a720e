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
//  1. the extended sequence table (and positions < 0 flagged in the state's error word);
//  2. the prefill's work tables on it; rows past the last sequence (up to the workspace's bound) zeroed;
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
// flagged).  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) cont_ext_table_kernel(LayerDims L, const int32_t* __restrict__ cu, hla_state s,
                                                              int32_t* __restrict__ ext_cu) {
    __shared__ int32_t part[1024];
    const int N = L.n_seqs, tid = threadIdx.x, per = (N + 1023) / 1024;
    const int lo = min(N, tid * per), hi = min(N, lo + per);
    auto rows = [&](int i) -> int32_t {
        int64_t a, len;
        seq_range(cu, i, L.total, &a, &len);
        const int64_t p = s.pos[i];
        return p < 0 ? 0 : (int32_t)(cont_n_old(p, L.n_sinks, L.window) + len);
    };
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

// 2b. rows past the last extended row, up to the workspace's bound: zero.  The tensor-core kernels read
// whole tiles, and a tile that runs past a sequence's end must meet finite rows (masked rows are multiplied
// by zero, and zero times a stale non-finite value would not vanish).
__global__ void __launch_bounds__(kCT)
cont_zero_tail_kernel(LayerDims Lx, const int32_t* __restrict__ ext_cu, __half* __restrict__ qr,
                      __half* __restrict__ kr, __half* __restrict__ qh, __half* __restrict__ kh, __half* __restrict__ vh,
                      __nv_bfloat16* __restrict__ ev, float* __restrict__ eg, float* __restrict__ eb) {
    const int64_t first = __ldg(ext_cu + Lx.n_seqs);
    const int D = kCD;
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
}

// 3. the cached rows: CTA per (cached row i, sequence)
__global__ void __launch_bounds__(kCT)
cont_gather_kernel(LayerDims L, hla_state s, const int32_t* __restrict__ ext_cu, __half* __restrict__ qr,
                   __half* __restrict__ kr, __half* __restrict__ qh, __half* __restrict__ kh, __half* __restrict__ vh,
                   __nv_bfloat16* __restrict__ ev, float* __restrict__ eg, float* __restrict__ eb) {
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

// 4. the new rows: CTA per (block of kTB new tokens, group of 8 feature rows), a warp per feature row
// (q-heads, then k-heads, then v-heads) walking the block's tokens in order with the last 8 conv inputs of
// its lane's channels (l + 32 e; RoPE pairs (l + 32 e, l + 32 e + 64) in the same lane) in registers, fed at
// the block's start from the tokens before it (the state's history before the call)
constexpr int kTB = 32;  // new tokens per CTA
template <typename Tin>
__global__ void __launch_bounds__(kCT)
cont_features_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                     const float* __restrict__ g, const float* __restrict__ beta, const float* __restrict__ wq,
                     const float* __restrict__ wk, const float* __restrict__ wv, const int32_t* __restrict__ cu,
                     hla_state s, const int32_t* __restrict__ ext_cu, __half* __restrict__ qr, __half* __restrict__ kr,
                     __half* __restrict__ qh, __half* __restrict__ kh, __half* __restrict__ vh,
                     __nv_bfloat16* __restrict__ ev, float* __restrict__ eg, float* __restrict__ eb) {
    constexpr int D = kCD, HALF = D / 2, E = D / 32, NP = kTB + kConvHalo;  // positions t0 - 7 .. t0 + kTB - 1
    __shared__ float cs[NP][HALF], sn[NP][HALF];
    __shared__ int64_t tok_pos[kTB];   // true position of each token of the block (-1: not a new token)
    __shared__ int64_t tok_ext[kTB];   // its extended row
    const int64_t t0 = (int64_t)blockIdx.x * kTB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_rows = L.Hq + 2 * L.Hkv;
    // the block's tokens (they may span sequences)
    if (tid < kTB) {
        const int64_t t = t0 + tid;
        int64_t p = -1, e = 0;
        if (t < L.total) {
            const int n = seq_of_token(cu, L.n_seqs, t);
            int64_t start, len;
            seq_range(cu, n, L.total, &start, &len);
            const int64_t pos = s.pos[n];
            if (pos >= 0 && t >= start && t < start + len) {
                p = pos + (t - start);
                e = (int64_t)__ldg(ext_cu + n) + cont_n_old(pos, L.n_sinks, L.window) + (t - start);
            }
        }
        tok_pos[tid] = p;
        tok_ext[tid] = e;
    }
    __syncthreads();
    // angles: slot u < 7 for the positions before the first token, 7 + i for token i (at its position)
    for (int idx = tid; idx < NP * HALF; idx += kCT) {
        const int u = idx / HALF, ii = idx % HALF;
        int64_t pp;
        if (u < kConvHalo) pp = tok_pos[0] < 0 ? -1 : tok_pos[0] - kConvHalo + u;
        else pp = tok_pos[u - kConvHalo];
        float c = 1.f, sv = 0.f;
        if (pp >= 0) rope_cs_exact(pp, L.theta[ii], &c, &sv);
        cs[u][ii] = c;
        sn[u][ii] = sv;
    }
    __syncthreads();
    const int r = blockIdx.y * (kCT / 32) + warp;
    if (r < n_rows) {
        const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
        const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
        const int H = kind == 0 ? L.Hq : L.Hkv;
        const Tin* src = kind == 0 ? q : kind == 1 ? k : v;
        const float* hist = kind == 0 ? s.conv_q : kind == 1 ? s.conv_k : s.conv_v;
        float w[E][kConvWidth];
#pragma unroll
        for (int ee = 0; ee < E; ++ee) {
            const float4* w4 = reinterpret_cast<const float4*>((kind == 0 ? wq : kind == 1 ? wk : wv) +
                                                               ((size_t)hh * D + lane + 32 * ee) * kConvWidth);
            const float4 a4 = w4[0], b4 = w4[1];
            w[ee][0] = a4.x; w[ee][1] = a4.y; w[ee][2] = a4.z; w[ee][3] = a4.w;
            w[ee][4] = b4.x; w[ee][5] = b4.y; w[ee][6] = b4.z; w[ee][7] = b4.w;
        }
        // the conv input of token t (global row) at position p, angle slot u
        auto input = [&](int64_t t, int u, float* x) {
            const Tin* row = src + ((size_t)t * H + hh) * D;
            if (kind == 2) {
#pragma unroll
                for (int ee = 0; ee < E; ++ee) x[ee] = to_f32(row[lane + 32 * ee]);
            } else {
#pragma unroll
                for (int ee = 0; ee < E / 2; ++ee) {
                    const int ii = lane + 32 * ee;
                    const float x1 = to_f32(row[ii]), x2 = to_f32(row[ii + HALF]);
                    x[ee] = x1 * cs[u][ii] - x2 * sn[u][ii];
                    x[ee + E / 2] = x2 * cs[u][ii] + x1 * sn[u][ii];
                }
            }
        };
        float win[kConvWidth][E];  // win[m]: the input at position p - 7 + m
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m)
#pragma unroll
            for (int ee = 0; ee < E; ++ee) win[m][ee] = 0.f;
        int64_t prev_p = -2;  // position of the last token processed (the window follows it)
        for (int i = 0; i < kTB; ++i) {
            const int64_t p = tok_pos[i], t = t0 + i;
            if (p < 0) {
                prev_p = -2;
                continue;
            }
            if (p == prev_p + 1) {  // the next token of the same sequence: shift
#pragma unroll
                for (int m = 0; m + 1 < kConvWidth; ++m)
#pragma unroll
                    for (int ee = 0; ee < E; ++ee) win[m][ee] = win[m + 1][ee];
            } else {  // a block or sequence start: the 7 inputs before p
                const int n = seq_of_token(cu, L.n_seqs, t);
                int64_t start, len;
                seq_range(cu, n, L.total, &start, &len);
                const int64_t pos = s.pos[n];
#pragma unroll
                for (int m = 0; m < kConvHalo; ++m) {
                    const int64_t pp = p - kConvHalo + m;
                    if (pp < 0) {
#pragma unroll
                        for (int ee = 0; ee < E; ++ee) win[m][ee] = 0.f;
                    } else if (pp >= pos) {  // a new token before this block: RoPE at its own position
                        const Tin* row = src + ((size_t)(t - kConvHalo + m) * H + hh) * D;
                        float cv[E / 2], sv[E / 2];
                        if (kind != 2) {
#pragma unroll
                            for (int ee = 0; ee < E / 2; ++ee) rope_cs_exact(pp, L.theta[lane + 32 * ee], &cv[ee], &sv[ee]);
                        }
#pragma unroll
                        for (int ee = 0; ee < E / 2; ++ee) {
                            const int ii = lane + 32 * ee;
                            if (kind == 2) {
                                win[m][ee] = to_f32(row[ii]);
                                win[m][ee + E / 2] = to_f32(row[ii + HALF]);
                            } else {
                                const float x1 = to_f32(row[ii]), x2 = to_f32(row[ii + HALF]);
                                win[m][ee] = x1 * cv[ee] - x2 * sv[ee];
                                win[m][ee + E / 2] = x2 * cv[ee] + x1 * sv[ee];
                            }
                        }
                    } else {  // before the call: the state's history
                        const float* hr = hist + (((size_t)n * kConvHalo + (size_t)(pp - pos + kConvHalo)) * H + hh) * D;
#pragma unroll
                        for (int ee = 0; ee < E; ++ee) win[m][ee] = hr[lane + 32 * ee];
                    }
                }
            }
            input(t, kConvHalo + i, win[kConvWidth - 1]);
            prev_p = p;
            float acc[E];
#pragma unroll
            for (int ee = 0; ee < E; ++ee) {
                acc[ee] = 0.f;
#pragma unroll
                for (int m = 0; m < kConvWidth; ++m) acc[ee] = fmaf(w[ee][m], win[m][ee], acc[ee]);
            }
            const size_t o = ((size_t)tok_ext[i] * H + hh) * D;
            if (kind == 2) {
#pragma unroll
                for (int ee = 0; ee < E; ++ee) {
                    vh[o + lane + 32 * ee] = __float2half_rn(acc[ee]);
                    ev[o + lane + 32 * ee] = __float2bfloat16_rn(win[kConvWidth - 1][ee]);
                }
                continue;
            }
            float ss = 0.f;
#pragma unroll
            for (int ee = 0; ee < E; ++ee) ss = fmaf(acc[ee], acc[ee], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = (kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q)) ? rsqrtf(ss + 1e-6f) : 1.f;
            __half* xr = kind == 0 ? qr : kr;
            __half* xh = kind == 0 ? qh : kh;
#pragma unroll
            for (int ee = 0; ee < E; ++ee) {
                xr[o + lane + 32 * ee] = __float2half_rn(win[kConvWidth - 1][ee]);
                xh[o + lane + 32 * ee] = __float2half_rn(acc[ee] * inv);
            }
        }
    }
    if (blockIdx.y == 0) {  // the gates
        for (int idx = tid; idx < kTB * L.Hq; idx += kCT) {
            const int i = idx / L.Hq, h = idx % L.Hq;
            if (tok_pos[i] < 0) continue;
            const size_t e = (size_t)tok_ext[i];
            eg[e * L.Hq + h] = g[(size_t)(t0 + i) * L.Hq + h];
            eb[e * L.Hq + h] = beta[(size_t)(t0 + i) * L.Hq + h];
        }
    }
}

// 6. the new rows of the extended output into out (16-byte copies)
__global__ void __launch_bounds__(kCT)
cont_out_kernel(LayerDims L, const int32_t* __restrict__ cu, hla_state s, const int32_t* __restrict__ ext_cu,
                const __nv_bfloat16* __restrict__ eo, __nv_bfloat16* __restrict__ out) {
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

// 7. the state after the call: CTA per (sequence, y); y = 0: the pending gates; y = 1 + kv: that kv head's
// ring entries, pending khat / vhat and conv histories; y = 1 + Hkv + h: q-head h's conv history
template <typename Tin>
__global__ void __launch_bounds__(kCT)
cont_state_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta, const int32_t* __restrict__ cu,
                  hla_state s, const int32_t* __restrict__ ext_cu, const __half* __restrict__ kh,
                  const __half* __restrict__ vh) {
    constexpr int D = kCD, HALF = D / 2;
    const int n = blockIdx.x, y = blockIdx.y, tid = threadIdx.x;
    const int ns = L.n_sinks, W = L.window, P = W + 1, R = ns + W;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t pos = s.pos[n];
    if (pos < 0 || len == 0) return;
    const int64_t p_end = pos + len;
    const size_t e0 = (size_t)__ldg(ext_cu + n) + (size_t)cont_n_old(pos, ns, W);  // extended row of position pos
    auto rope = [&](const Tin* row, int c, int64_t p) {
        const int ii = c % HALF;
        float cv, sv;
        rope_cs_exact(p, L.theta[ii], &cv, &sv);
        const float x1 = to_f32(row[ii]), x2 = to_f32(row[ii + HALF]);
        return c < HALF ? x1 * cv - x2 * sv : x2 * cv + x1 * sv;
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
                val[u] = rotate ? rope(row, c, pp) : to_f32(row[c]);
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
        const int64_t i0 = max((int64_t)0, max(len - W, ns - pos));
        for (int64_t i = i0 * L.Hq + tid; i < (int64_t)len * L.Hq; i += kCT) {
            const int64_t tt = i / L.Hq, p = pos + tt;
            const int h = (int)(i % L.Hq);
            const size_t gs = ((size_t)n * L.Hq + h) * P + (size_t)(p % P);
            s.pend_g[gs] = g[(size_t)(start + tt) * L.Hq + h];
            s.pend_beta[gs] = beta[(size_t)(start + tt) * L.Hq + h];
        }
        return;
    }
    if (y > L.Hkv) {  // a q-head's conv history
        advance_history(s.conv_q, q, L.Hq, y - 1 - L.Hkv, true);
        return;
    }
    const int kv = y - 1;
    Tin* kring = static_cast<Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    Tin* vring = static_cast<Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    // the new tokens that stay in the ring (sinks, and the final window) and in the pending ring
    const int64_t first = max((int64_t)0, min(len, p_end - W - pos));  // index of the first final-window token
    // the rows that stay: new sinks [0, i_sink) and the final window [i_win, len), all at once
    const int64_t i_sink = min(len, max((int64_t)0, ns - pos));
    const int64_t i_win = max(first, i_sink);
    const int64_t n_rows = i_sink + (len - i_win);
    auto row_of = [&](int64_t r) { return r < i_sink ? r : i_win + (r - i_sink); };
    for (int64_t idx = tid; idx < n_rows * HALF; idx += kCT) {  // RoPE'd key pairs (ii, ii + d/2): one angle
        const int64_t i = row_of(idx / HALF), p = pos + i;
        const int ii = (int)(idx % HALF);
        const size_t row = ((size_t)(start + i) * L.Hkv + kv) * D, slot = (size_t)cont_ring_slot(p, ns, W) * D;
        float cv, sv;
        rope_cs_exact(p, L.theta[ii], &cv, &sv);
        const float x1 = to_f32(k[row + ii]), x2 = to_f32(k[row + ii + HALF]);
        kring[slot + ii] = from_f32<Tin>(x1 * cv - x2 * sv);
        kring[slot + ii + HALF] = from_f32<Tin>(x2 * cv + x1 * sv);
    }
    for (int64_t idx = tid; idx < n_rows * D; idx += kCT) {
        const int64_t i = row_of(idx / D), p = pos + i;
        const int c = (int)(idx % D);
        const size_t row = ((size_t)(start + i) * L.Hkv + kv) * D, slot = (size_t)cont_ring_slot(p, ns, W) * D;
        vring[slot + c] = v[row + c];
        if (p >= ns && p >= p_end - W) {
            const size_t ps = (((size_t)n * L.Hkv + kv) * P + (size_t)(p % P)) * D + c;
            const size_t er = ((e0 + (size_t)i) * L.Hkv + kv) * D + c;
            s.pend_k[ps] = __half2float(kh[er]);
            s.pend_v[ps] = __half2float(vh[er]);
        }
    }
    advance_history(s.conv_k, k, L.Hkv, kv, true);
    advance_history(s.conv_v, v, L.Hkv, kv, false);
}

// 8. pos += len, after every launch above has read it
__global__ void cont_tc_advance_kernel(LayerDims L, const int32_t* __restrict__ cu, int64_t* __restrict__ pos) {
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
    cont_ext_table_kernel<<<1, 1024, 0, st>>>(L, cu, s, ext_cu);
    return cudaGetLastError();
}

cudaError_t launch_continue_rows(const LayerDims& L, const LayerDims& Lx, const int32_t* cu, const hla_state& s,
                                 const int32_t* ext_cu, __half* qr, __half* kr, __half* qh, __half* kh, __half* vh,
                                 __nv_bfloat16* ev, float* eg, float* eb, const __nv_bfloat16* q,
                                 const __nv_bfloat16* k, const __nv_bfloat16* v, const float* g, const float* beta,
                                 const float* wq, const float* wk, const float* wv, cudaStream_t st) {
    cont_zero_tail_kernel<<<1024, kCT, 0, st>>>(Lx, ext_cu, qr, kr, qh, kh, vh, ev, eg, eb);
    cont_gather_kernel<<<dim3(L.n_sinks + L.window, L.n_seqs), kCT, 0, st>>>(L, s, ext_cu, qr, kr, qh, kh, vh, ev, eg,
                                                                             eb);
    if (L.total > 0) {
        const dim3 grid((unsigned)((L.total + kTB - 1) / kTB), (unsigned)((L.Hq + 2 * L.Hkv + kCT / 32 - 1) / (kCT / 32)));
        cont_features_kernel<__nv_bfloat16><<<grid, kCT, 0, st>>>(L, q, k, v, g, beta, wq, wk, wv, cu, s, ext_cu, qr,
                                                                  kr, qh, kh, vh, ev, eg, eb);
    }
    return cudaGetLastError();
}

cudaError_t launch_continue_finish(const LayerDims& L, const int32_t* cu, const hla_state& s, const int32_t* ext_cu,
                                   const __nv_bfloat16* ext_out, __nv_bfloat16* out, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v, const float* g, const float* beta,
                                   const __half* kh, const __half* vh, cudaStream_t st) {
    if (L.total > 0) cont_out_kernel<<<(unsigned)L.total, kCT, 0, st>>>(L, cu, s, ext_cu, ext_out, out);
    cont_state_kernel<__nv_bfloat16><<<dim3(L.n_seqs, 1 + L.Hkv + L.Hq), kCT, 0, st>>>(L, q, k, v, g, beta, cu, s,
                                                                                       ext_cu, kh, vh);
    cont_tc_advance_kernel<<<(L.n_seqs + 127) / 128, 128, 0, st>>>(L, cu, s.pos);
    return cudaGetLastError();
}

}  // namespace hla
