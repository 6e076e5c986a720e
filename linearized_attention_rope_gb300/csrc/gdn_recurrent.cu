// Linear branch, token-serial form: the Gated DeltaNet update
//   S <- alpha_j (I - beta_j khat_j khat_j^T) S + beta_j khat_j vhat_j^T
// ("迈向线性的关键：分析驱动的 Transformer 线性化", section 线性注意力替换机制,
// with a scalar gate), applied to token j when it leaves the window, i.e. at
// position j + W (section 填补近似缺口的实用设计: the linear path covers the
// tokens outside the sink + window budget), followed by the read-out
// o_lin[j + W] = S^T qhat[j + W].  With HLA_FLAG_GLA the update is the gated
// linear attention of the same section, S <- alpha_j S + khat_j vhat_j^T.
//
// One CTA per (sequence, query head); four adjacent threads own one column of
// S (the value dim), a quarter of its key rows each, in registers; dot
// products over the key dim finish with two shuffles.  fp32 throughout; this is
// the fp32 layer's path and the cross-check for the chunked kernel.
#include "hla_common.cuh"

namespace hla {

constexpr int kRecTile = 16;  // tokens staged in shared memory per step
constexpr int kRecParts = 4;  // threads sharing one column of S

// Shared-memory row layout: the four row quarters of a key/query vector sit
// 36 floats apart so the four parts of a warp read distinct banks.
template <int D> __device__ __forceinline__ int rec_pad(int c) {
    constexpr int Q = D / kRecParts;
    return (c / Q) * (Q + 4) + c % Q;
}

template <typename Tf, int D>
__global__ void __launch_bounds__(D * kRecParts)
gdn_recurrent_kernel(LayerDims L, const Tf* __restrict__ qhat, const Tf* __restrict__ khat,
                     const Tf* __restrict__ vhat, const float* __restrict__ g,
                     const float* __restrict__ beta, const int32_t* __restrict__ cu,
                     float* __restrict__ o_lin, float* __restrict__ S_out) {
    constexpr int Q = D / kRecParts;           // rows of S per thread
    constexpr int ROW = kRecParts * (Q + 4);   // padded row length
    constexpr int NT = D * kRecParts;
    __shared__ __align__(16) float ks[kRecTile][ROW];
    __shared__ __align__(16) float qs[kRecTile][ROW];
    __shared__ float vs[kRecTile][D];
    __shared__ float as[kRecTile], bs[kRecTile];

    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G;
    const int col = threadIdx.x / kRecParts, part = threadIdx.x % kRecParts;
    const int W = L.window;
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);

    float S[Q];  // S[part*Q + i][col]
#pragma unroll
    for (int i = 0; i < Q; ++i) S[i] = 0.f;

    const int64_t j_end = len - W;  // tokens n_sinks .. j_end-1 get absorbed
    for (int64_t jt = L.n_sinks; jt < j_end; jt += kRecTile) {
        const int cnt = (int)min((int64_t)kRecTile, j_end - jt);
        __syncthreads();
        for (int idx = threadIdx.x; idx < cnt * D; idx += NT) {
            int r = idx / D, c = idx % D;
            size_t t = (size_t)(start + jt + r);
            ks[r][rec_pad<D>(c)] = to_f32(khat[(t * L.Hkv + kv) * D + c]);
            qs[r][rec_pad<D>(c)] = to_f32(qhat[((t + W) * L.Hq + h) * D + c]);
            vs[r][c] = to_f32(vhat[(t * L.Hkv + kv) * D + c]);
        }
        if (threadIdx.x < cnt) {
            size_t t = (size_t)(start + jt + threadIdx.x);
            as[threadIdx.x] = expf(g[t * L.Hq + h]);
            bs[threadIdx.x] = beta[t * L.Hq + h];
        }
        __syncthreads();
        for (int r = 0; r < cnt; ++r) {
            const float alpha = as[r], b = bs[r];
            const float4* k4 = reinterpret_cast<const float4*>(&ks[r][part * (Q + 4)]);
            const float4* q4 = reinterpret_cast<const float4*>(&qs[r][part * (Q + 4)]);
            float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
            for (int i = 0; i < Q / 4; ++i) {
                float4 kk = k4[i];
                x0 = fmaf(kk.x, S[4 * i + 0], x0);
                x1 = fmaf(kk.y, S[4 * i + 1], x1);
                x2 = fmaf(kk.z, S[4 * i + 2], x2);
                x3 = fmaf(kk.w, S[4 * i + 3], x3);
            }
            float x = (x0 + x1) + (x2 + x3);
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);  // (k^T S)[col]
            // delta rule: u = beta (v - alpha k^T S); GLA (no erase): u = v
            const float u = gla ? vs[r][col] : b * (vs[r][col] - alpha * x);
            float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
            for (int i = 0; i < Q / 4; ++i) {
                float4 kk = k4[i];
                float4 qq = q4[i];
                S[4 * i + 0] = fmaf(alpha, S[4 * i + 0], kk.x * u);
                S[4 * i + 1] = fmaf(alpha, S[4 * i + 1], kk.y * u);
                S[4 * i + 2] = fmaf(alpha, S[4 * i + 2], kk.z * u);
                S[4 * i + 3] = fmaf(alpha, S[4 * i + 3], kk.w * u);
                o0 = fmaf(qq.x, S[4 * i + 0], o0);
                o1 = fmaf(qq.y, S[4 * i + 1], o1);
                o2 = fmaf(qq.z, S[4 * i + 2], o2);
                o3 = fmaf(qq.w, S[4 * i + 3], o3);
            }
            float o = (o0 + o1) + (o2 + o3);
            o += __shfl_xor_sync(0xffffffffu, o, 1);
            o += __shfl_xor_sync(0xffffffffu, o, 2);
            if (part == 0) {
                size_t t = (size_t)(start + jt + r + W);
                o_lin[(t * L.Hq + h) * D + col] = o;
            }
        }
    }
    if (S_out) {
        float* dst = S_out + ((size_t)n * L.Hq + h) * D * D;
#pragma unroll
        for (int i = 0; i < Q; ++i) dst[(size_t)(part * Q + i) * D + col] = S[i];
    }
}

template <typename Tf>
cudaError_t launch_gdn_recurrent(const LayerDims& L, const Tf* qhat, const Tf* khat, const Tf* vhat,
                                 const float* g, const float* beta, const int32_t* cu, float* o_lin,
                                 float* S_out, cudaStream_t st) {
    dim3 grid(L.Hq, L.n_seqs);
    if (L.d == 128)
        gdn_recurrent_kernel<Tf, 128><<<grid, 128 * kRecParts, 0, st>>>(L, qhat, khat, vhat, g, beta, cu, o_lin, S_out);
    else
        gdn_recurrent_kernel<Tf, 64><<<grid, 64 * kRecParts, 0, st>>>(L, qhat, khat, vhat, g, beta, cu, o_lin, S_out);
    return cudaGetLastError();
}

template cudaError_t launch_gdn_recurrent<float>(const LayerDims&, const float*, const float*,
                                                 const float*, const float*, const float*,
                                                 const int32_t*, float*, float*, cudaStream_t);
template cudaError_t launch_gdn_recurrent<__half>(const LayerDims&, const __half*, const __half*,
                                                  const __half*, const float*, const float*,
                                                  const int32_t*, float*, float*, cudaStream_t);

}  // namespace hla
