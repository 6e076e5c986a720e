// Component-usage diagnostics of the hybrid layer (synthetic analysis only):
//   - how much each branch contributes: per (sequence, q-head), the sums over
//     positions of |o_sm|^2 and |lambda_h o_lin|^2 ("Untangling Component
//     Imbalance in Hybrid Linear Attention Conversion", sections 摘要 and
//     方法详解: hybrids come to lean on the window softmax and bypass the
//     linear branch);
//   - how concentrated the keys are: per position p and kv head, with u_i the
//     softmax branch's RoPE'd key i normalised to unit length and m_p the mean
//     of u_0..u_p, the concentration |m_p| and the projection residual
//     |u_p - (mhat_p . u_p) mhat_p| ("迈向线性的关键：分析驱动的 Transformer
//     线性化", sections 从 softmax 到 delta 规则的一阶近似 (Lemma 2: projection
//     onto the orthogonal complement of the mean key) and 填补近似缺口的实用设计:
//     the residual grows where keys do not share one direction).
#include "hla_common.cuh"

namespace hla {

namespace {

constexpr int kSqThreads = 256;
constexpr int kSqUnroll = 8;  // 16-byte loads in flight per thread

// CTA per (q-head, sequence): the sum over the sequence's rows of |out[p][h]|^2 into sq[(n Hq + h) 2 + which].
// The head's rows are read as 16-byte pieces: thread t takes piece t mod (pieces per row) of rows
// t / (pieces per row) + k (256 / pieces per row), kSqUnroll rows in flight; each thread sums its pieces in
// order and the CTA joins the threads in a fixed tree, so the result does not depend on timing.
template <typename T>
__global__ void __launch_bounds__(kSqThreads)
branch_sq_kernel(LayerDims L, const T* __restrict__ out, const int32_t* __restrict__ cu, float* __restrict__ sq,
                 int which) {
    constexpr int EP = 16 / (int)sizeof(T);  // elements per piece
    __shared__ float red[kSqThreads / 32];
    const int h = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int per_row = L.d / EP;  // pieces per row (d is 64 or 128: 4 to 32, a divisor of 256)
    const int rows_per_pass = kSqThreads / per_row;
    const size_t row_stride = (size_t)L.Hq * L.d;
    const T* base = out + ((size_t)start * L.Hq + h) * L.d + (size_t)(tid % per_row) * EP;
    float total = 0.f;
    for (int64_t r0 = tid / per_row; r0 < len; r0 += (int64_t)rows_per_pass * kSqUnroll) {
        uint4 v[kSqUnroll];
#pragma unroll
        for (int u = 0; u < kSqUnroll; ++u) {
            const int64_t r = r0 + (int64_t)u * rows_per_pass;
            v[u] = r < len ? __ldg(reinterpret_cast<const uint4*>(base + (size_t)r * row_stride))
                           : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kSqUnroll; ++u) {
            const T* e = reinterpret_cast<const T*>(&v[u]);
#pragma unroll
            for (int k = 0; k < EP; ++k) {
                const float x = to_f32(e[k]);
                total = fmaf(x, x, total);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    if ((tid & 31) == 0) red[tid >> 5] = total;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < kSqThreads / 32; ++w) t += red[w];
        sq[((size_t)n * L.Hq + h) * 2 + which] = t;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kKsWarps = 32;  // warps of a key-statistics CTA, each over one range of positions

// A key row in a warp, lane l holding dims l, l + 32, ... (zeros past the range: row null)
template <typename Tf, int E>
__device__ __forceinline__ void load_key(const Tf* row, int lane, float* x) {
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = row ? to_f32(row[lane + 32 * e]) : 0.f;
}
// Scaled to unit length (a zero key stays zero)
template <int E>
__device__ __forceinline__ void unit_key(float* u) {
    float nk = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) nk = fmaf(u[e], u[e], nk);
    nk = warp_sum(nk);
    const float inv_k = nk > 0.f ? rsqrtf(nk) : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) u[e] *= inv_k;
}

// CTA per (kv head, sequence): the sequence's positions cut into kKsWarps consecutive ranges, one per warp.
// Each warp sums the unit keys of its range; the sums of the ranges before each one give its starting point
// (summed in range order); then each warp walks its range with the running sum m of the unit keys so far
// and writes, per position p, the concentration |m_p| (m_p the mean of u_0..u_p) and the projection
// residual |u_p - (mhat_p . u_p) mhat_p| into stats[((start + p) Hkv + kv) 2 + {0, 1}] (1 where m_p = 0).
template <typename Tf, int D>
__global__ void __launch_bounds__(32 * kKsWarps)
key_stats_kernel(LayerDims L, const Tf* __restrict__ kr, const int32_t* __restrict__ cu, float* __restrict__ stats) {
    constexpr int E = D / 32;
    __shared__ float part[kKsWarps][D];  // each range's sum, then the sum of the ranges before it
    const int kv = blockIdx.x, n = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t per = (len + kKsWarps - 1) / kKsWarps;
    const int64_t p_lo = min(len, (int64_t)warp * per), p_hi = min(len, p_lo + per);
    const Tf* rows = kr + ((size_t)start * L.Hkv + kv) * D;
    const size_t stride = (size_t)L.Hkv * D;
    float m[E];
#pragma unroll
    for (int e = 0; e < E; ++e) m[e] = 0.f;
    // each walk loads the row after the one it is on, so a load is in flight while a row is reduced
    float nxt[E];
    load_key<Tf, E>(p_lo < p_hi ? rows + (size_t)p_lo * stride : nullptr, lane, nxt);
    for (int64_t p = p_lo; p < p_hi; ++p) {
        float u[E];
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] = nxt[e];
        load_key<Tf, E>(p + 1 < p_hi ? rows + (size_t)(p + 1) * stride : nullptr, lane, nxt);
        unit_key<E>(u);
#pragma unroll
        for (int e = 0; e < E; ++e) m[e] += u[e];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) part[warp][lane + 32 * e] = m[e];
    __syncthreads();
    if (threadIdx.x < D) {  // exclusive prefix over the ranges, dim by dim
        float acc = 0.f;
        for (int w = 0; w < kKsWarps; ++w) {
            const float x = part[w][threadIdx.x];
            part[w][threadIdx.x] = acc;
            acc += x;
        }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) m[e] = part[warp][lane + 32 * e];
    load_key<Tf, E>(p_lo < p_hi ? rows + (size_t)p_lo * stride : nullptr, lane, nxt);
    for (int64_t p = p_lo; p < p_hi; ++p) {
        float u[E];
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] = nxt[e];
        load_key<Tf, E>(p + 1 < p_hi ? rows + (size_t)(p + 1) * stride : nullptr, lane, nxt);
        unit_key<E>(u);
        const float inv_n = 1.f / (float)(p + 1);
        float nm = 0.f, dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            m[e] += u[e];
            const float mc = m[e] * inv_n;
            nm = fmaf(mc, mc, nm);
            dot = fmaf(mc, u[e], dot);
        }
        nm = sqrtf(warp_sum(nm));
        dot = warp_sum(dot);
        float res = 1.f;
        if (nm > 0.f) {
            const float proj = dot / nm, s = inv_n / nm;
            float r = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x = u[e] - proj * m[e] * s;
                r = fmaf(x, x, r);
            }
            res = sqrtf(warp_sum(r));  // (nm is the same in every lane: the warp takes one branch)
        }
        if (lane == 0) {
            float2* o = reinterpret_cast<float2*>(stats + ((size_t)(start + p) * L.Hkv + kv) * 2);
            *o = make_float2(nm, res);
        }
    }
}

}  // namespace

template <typename T>
cudaError_t launch_branch_sq(const LayerDims& L, const T* out, const int32_t* cu, float* sq, int which, cudaStream_t st) {
    branch_sq_kernel<T><<<dim3(L.Hq, L.n_seqs), kSqThreads, 0, st>>>(L, out, cu, sq, which);
    return cudaGetLastError();
}
template cudaError_t launch_branch_sq<float>(const LayerDims&, const float*, const int32_t*, float*, int, cudaStream_t);
template cudaError_t launch_branch_sq<__nv_bfloat16>(const LayerDims&, const __nv_bfloat16*, const int32_t*, float*,
                                                     int, cudaStream_t);

template <typename Tf>
cudaError_t launch_key_stats(const LayerDims& L, const Tf* kr, const int32_t* cu, float* stats, cudaStream_t st) {
    if (L.d == 128)
        key_stats_kernel<Tf, 128><<<dim3(L.Hkv, L.n_seqs), 32 * kKsWarps, 0, st>>>(L, kr, cu, stats);
    else
        key_stats_kernel<Tf, 64><<<dim3(L.Hkv, L.n_seqs), 32 * kKsWarps, 0, st>>>(L, kr, cu, stats);
    return cudaGetLastError();
}
template cudaError_t launch_key_stats<float>(const LayerDims&, const float*, const int32_t*, float*, cudaStream_t);
template cudaError_t launch_key_stats<__half>(const LayerDims&, const __half*, const int32_t*, float*, cudaStream_t);

}  // namespace hla
