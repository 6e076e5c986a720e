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

constexpr int kSqThreads = 128;
constexpr int kSqBlock = 256;  // positions summed in fp32 before joining the running sum

// CTA per (q-head, sequence): the sum over the sequence's rows of |out[p][h]|^2 into sq[(n Hq + h) 2 + which].
template <typename T>
__global__ void __launch_bounds__(kSqThreads)
branch_sq_kernel(LayerDims L, const T* __restrict__ out, const int32_t* __restrict__ cu, float* __restrict__ sq,
                 int which) {
    __shared__ float red[kSqThreads / 32];
    const int h = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    float total = 0.f;
    for (int64_t p0 = 0; p0 < len; p0 += kSqBlock) {
        const int64_t p1 = min(len, p0 + kSqBlock);
        float part = 0.f;
        for (int64_t p = p0; p < p1; ++p) {
            const T* row = out + ((size_t)(start + p) * L.Hq + h) * L.d;
            for (int c = tid; c < L.d; c += kSqThreads) {
                const float x = to_f32(row[c]);
                part = fmaf(x, x, part);
            }
        }
        total += part;
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

// One warp per (kv head, sequence), lane l holding dims l, l + 32, ...: a running sum of the unit keys
// over the positions of the sequence; per position the concentration and the residual into
// stats[((start + p) Hkv + kv) 2 + {0, 1}].
template <typename Tf, int D>
__global__ void __launch_bounds__(32)
key_stats_kernel(LayerDims L, const Tf* __restrict__ kr, const int32_t* __restrict__ cu, float* __restrict__ stats) {
    constexpr int E = D / 32;
    const int kv = blockIdx.x, n = blockIdx.y, lane = threadIdx.x;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    float m[E];
#pragma unroll
    for (int e = 0; e < E; ++e) m[e] = 0.f;
    for (int64_t p = 0; p < len; ++p) {
        const Tf* row = kr + ((size_t)(start + p) * L.Hkv + kv) * D;
        float u[E];
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] = to_f32(row[lane + 32 * e]);
        float nk = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) nk = fmaf(u[e], u[e], nk);
        nk = warp_sum(nk);
        const float inv_k = nk > 0.f ? rsqrtf(nk) : 0.f;
        const float inv_n = 1.f / (float)(p + 1);
        float nm = 0.f, dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            u[e] *= inv_k;
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
        key_stats_kernel<Tf, 128><<<dim3(L.Hkv, L.n_seqs), 32, 0, st>>>(L, kr, cu, stats);
    else
        key_stats_kernel<Tf, 64><<<dim3(L.Hkv, L.n_seqs), 32, 0, st>>>(L, kr, cu, stats);
    return cudaGetLastError();
}
template cudaError_t launch_key_stats<float>(const LayerDims&, const float*, const int32_t*, float*, cudaStream_t);
template cudaError_t launch_key_stats<__half>(const LayerDims&, const __half*, const int32_t*, float*, cudaStream_t);

}  // namespace hla
