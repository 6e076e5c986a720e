// Feature path of the linear branch: RoPE -> causal depthwise short conv
// (width 8) -> L2 norm, on q and k; short conv alone on v.
// Source: "迈向线性的关键：分析驱动的 Transformer 线性化", section 实践建议,
// item 3 (a kernel-8 short convolution after RoPE and before L2
// normalisation).  The RoPE'd q and k are also written out: the exact
// softmax branch reads them (frozen-backbone attention).
#include "hla_common.cuh"

namespace hla {

// RoPE angles at position p = 64 a + b come from two small tables and the
// angle-addition identities, so the per-token work is fp32 only while every
// table entry is formed and range-reduced in double precision.
__global__ void rope_tables_kernel(LayerDims L, float2* __restrict__ fine,
                                   float2* __restrict__ coarse, int n_coarse) {
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
}

cudaError_t launch_rope_tables(const LayerDims& L, float2* fine, float2* coarse, int n_coarse,
                               cudaStream_t st) {
    int64_t n = (int64_t)(64 + n_coarse) * (L.d / 2);
    int blocks = (int)((n + 255) / 256);
    rope_tables_kernel<<<blocks, 256, 0, st>>>(L, fine, coarse, n_coarse);
    return cudaGetLastError();
}

constexpr int kFeatTokens = 32;    // tokens per CTA
constexpr int kFeatThreads = 128;

// One CTA = 32 tokens x one head (q, k or v head, chosen by blockIdx.y).
template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(kFeatThreads)
features_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                const Tin* __restrict__ v, const float* __restrict__ wq,
                const float* __restrict__ wk, const float* __restrict__ wv,
                const int32_t* __restrict__ cu, const float2* __restrict__ fine,
                const float2* __restrict__ coarse, Tf* __restrict__ qr, Tf* __restrict__ kr,
                Tf* __restrict__ qhat, Tf* __restrict__ khat, Tf* __restrict__ vhat,
                int32_t* __restrict__ err) {
    constexpr int TT = kFeatTokens;
    constexpr int ROWS = TT + kConvHalo;
    constexpr int HALF = D / 2;
    constexpr int RPT = TT * D / kFeatThreads;   // output rows per thread
    constexpr int RSTEP = kFeatThreads / D;      // row stride between them
    constexpr int WPR = D / 32;                  // warps covering one row
    __shared__ float xs[ROWS][D];
    __shared__ int rpos[ROWS];
    __shared__ float red[TT][WPR];

    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * TT;
    int head = blockIdx.y;
    int kind = 0;  // 0 = q, 1 = k, 2 = v
    if (head >= L.Hq + L.Hkv) { kind = 2; head -= L.Hq + L.Hkv; }
    else if (head >= L.Hq) { kind = 1; head -= L.Hq; }
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const Tin* src = kind == 0 ? q : (kind == 1 ? k : v);
    const float* w = kind == 0 ? wq : (kind == 1 ? wk : wv);

    if (tid < ROWS) {
        int64_t t = t0 - kConvHalo + tid;
        int p = -1;
        if (t >= 0 && t < L.total) {
            int s = seq_of_token(cu, L.n_seqs, t);
            int64_t start, len;
            seq_range(cu, s, L.total, &start, &len);
            if (t >= start && t < start + len) p = (int)(t - start);
            else if (err && blockIdx.y == 0) atomicExch(err, kErrSeqlens);
        }
        rpos[tid] = p;
    }
    for (int idx = tid; idx < ROWS * D; idx += kFeatThreads) {
        int r = idx / D, c = idx % D;
        int64_t t = t0 - kConvHalo + r;
        float x = 0.f;
        if (t >= 0 && t < L.total) x = to_f32(src[((size_t)t * H + head) * D + c]);
        xs[r][c] = x;
    }
    __syncthreads();

    if (kind != 2) {
        for (int idx = tid; idx < ROWS * HALF; idx += kFeatThreads) {
            int r = idx / HALF, i = idx % HALF;
            int p = rpos[r];
            if (p < 0) continue;
            float2 f = __ldg(fine + (p & 63) * HALF + i);
            float2 g = __ldg(coarse + (p >> 6) * HALF + i);
            float cs = g.x * f.x - g.y * f.y;
            float sn = g.y * f.x + g.x * f.y;
            float x1 = xs[r][i], x2 = xs[r][i + HALF];
            xs[r][i] = x1 * cs - x2 * sn;
            xs[r][i + HALF] = x2 * cs + x1 * sn;
        }
        __syncthreads();
        Tf* rot = kind == 0 ? qr : kr;
        for (int idx = tid; idx < TT * D; idx += kFeatThreads) {
            int r = idx / D, c = idx % D;
            int64_t t = t0 + r;
            if (t < L.total) rot[((size_t)t * H + head) * D + c] = from_f32<Tf>(xs[r + kConvHalo][c]);
        }
    }

    // causal depthwise conv, zero history before the start of each sequence
    const int c = tid % D;
    const int r0 = tid / D;
    float wr[kConvWidth];
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) wr[m] = __ldg(w + ((size_t)head * D + c) * kConvWidth + m);
    float acc[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        int r = r0 + j * RSTEP;
        int p = rpos[r + kConvHalo];
        float a = 0.f;
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m)
            if (p - kConvHalo + m >= 0) a = fmaf(wr[m], xs[r + m][c], a);
        acc[j] = a;
    }

    Tf* dst = kind == 0 ? qhat : (kind == 1 ? khat : vhat);
    bool norm = kind == 1 || (kind == 0 && (L.flags & HLA_FLAG_L2NORM_Q));
    if (norm) {
        const int lane = tid & 31;
        const int wir = c / 32;  // which warp of the row this thread's channel sits in
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            float ss = acc[j] * acc[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) red[r0 + j * RSTEP][wir] = ss;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            int r = r0 + j * RSTEP;
            float ss = 0.f;
#pragma unroll
            for (int u = 0; u < WPR; ++u) ss += red[r][u];
            acc[j] *= rsqrtf(ss + 1e-6f);
        }
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        int r = r0 + j * RSTEP;
        int64_t t = t0 + r;
        if (t < L.total) dst[((size_t)t * H + head) * D + c] = from_f32<Tf>(acc[j]);
    }
}

template <typename Tin, typename Tf>
cudaError_t launch_features(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                            const float* wq, const float* wk, const float* wv, const int32_t* cu,
                            const float2* fine, const float2* coarse, Tf* qr, Tf* kr, Tf* qhat,
                            Tf* khat, Tf* vhat, int32_t* err, cudaStream_t st) {
    dim3 grid((unsigned)((L.total + kFeatTokens - 1) / kFeatTokens), L.Hq + 2 * L.Hkv);
    if (L.d == 128)
        features_kernel<Tin, Tf, 128><<<grid, kFeatThreads, 0, st>>>(
            L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr, qhat, khat, vhat, err);
    else
        features_kernel<Tin, Tf, 64><<<grid, kFeatThreads, 0, st>>>(
            L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr, qhat, khat, vhat, err);
    return cudaGetLastError();
}

template cudaError_t launch_features<float, float>(const LayerDims&, const float*, const float*,
                                                   const float*, const float*, const float*,
                                                   const float*, const int32_t*, const float2*,
                                                   const float2*, float*, float*, float*, float*,
                                                   float*, int32_t*, cudaStream_t);
template cudaError_t launch_features<__nv_bfloat16, __half>(
    const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*,
    const float*, const float*, const float*, const int32_t*, const float2*, const float2*, __half*,
    __half*, __half*, __half*, __half*, int32_t*, cudaStream_t);

}  // namespace hla
