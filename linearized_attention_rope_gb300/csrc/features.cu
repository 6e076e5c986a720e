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

constexpr int kTT = 32;                   // output tokens per CTA
constexpr int kRowsPerCta = 4;            // feature rows (q, k or v heads) per CTA
constexpr int kStage = kTT + kConvHalo;   // staged tokens: 7 of conv history, then the outputs
constexpr int kFeatThreads = 128;

template <typename T> struct Vec8;  // eight elements as one or two 16-byte words
template <> struct Vec8<__nv_bfloat16> {
    static constexpr int kChunks = 1;
    __device__ static void unpack(const unsigned char* p, float* x) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    }
};
template <> struct Vec8<__half> {
    static constexpr int kChunks = 1;
    __device__ static void unpack(const unsigned char* p, float* x) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    }
    __device__ static void pack(unsigned char* p, const float* x) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec8<float> {
    static constexpr int kChunks = 2;
    __device__ static void unpack(const unsigned char* p, float* x) {
        const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 16);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    __device__ static void pack(unsigned char* p, const float* x) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(p + 16) = make_float4(x[4], x[5], x[6], x[7]);
    }
};

// One CTA = kTT tokens x kRowsPerCta feature rows (q heads, then k heads,
// then v heads, in that order across the grid).  The rows of the kTT tokens
// and their 7 predecessors are staged in shared memory, rotated there in
// place (RoPE on q and k; cos/sin from the fine and coarse tables by angle
// addition, both reduced in double precision) and written out as the RoPE'd
// q and k; then one thread per (token, row, 8 channels) runs the width-8
// causal conv over the staged rows with its 64 weights held in registers,
// and the D / 8 lanes of a row finish the L2 norm with shuffles.  Conv taps
// before a sequence's first token read as zero.
template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(kFeatThreads, 4)
features_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                const Tin* __restrict__ v, const float* __restrict__ wq,
                const float* __restrict__ wk, const float* __restrict__ wv,
                const int32_t* __restrict__ cu, const float2* __restrict__ fine,
                const float2* __restrict__ coarse, Tf* __restrict__ qr, Tf* __restrict__ kr,
                Tf* __restrict__ qhat, Tf* __restrict__ khat, Tf* __restrict__ vhat,
                int32_t* __restrict__ err) {
    static_assert(sizeof(Tin) == sizeof(Tf), "rows are rotated in place");
    constexpr int HALF = D / 2, G8 = D / 8, E = (int)sizeof(Tin);
    constexpr int ROWB = D * E;                                     // bytes per staged row
    constexpr int CH = 16 / E;                                      // elements per 16-byte chunk
    extern __shared__ __align__(16) unsigned char xs[];             // [kStage tokens][kRowsPerCta][D]
    __shared__ int pos_s[kStage];
    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * kTT;
    const int n_rows = L.Hq + 2 * L.Hkv;

    // row j of this CTA: kind (0 q, 1 k, 2 v), head, and whether it exists
    auto row_info = [&](int j, int* kind, int* head) {
        int hr = blockIdx.y * kRowsPerCta + j;
        const bool on = hr < n_rows;
        if (!on) hr = n_rows - 1;
        *kind = 0;
        if (hr >= L.Hq + L.Hkv) { *kind = 2; hr -= L.Hq + L.Hkv; }
        else if (hr >= L.Hq) { *kind = 1; hr -= L.Hq; }
        *head = hr;
        return on;
    };

    // ---- stage the rows (zeros outside the token range)
    for (int idx = tid; idx < kStage * kRowsPerCta * (ROWB / 16); idx += kFeatThreads) {
        const int chunk = idx % (ROWB / 16), rj = idx / (ROWB / 16), j = rj % kRowsPerCta, tk = rj / kRowsPerCta;
        int kind, head;
        const bool on = row_info(j, &kind, &head);
        const int64_t t = t0 - kConvHalo + tk;
        const bool in = on && t >= 0 && t < L.total;
        const Tin* src = kind == 0 ? q : (kind == 1 ? k : v);
        const size_t H = kind == 0 ? L.Hq : L.Hkv;
        const Tin* gp = src + ((size_t)(in ? t : 0) * H + head) * D + chunk * CH;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(xs + (size_t)rj * ROWB + chunk * 16)),
                     "l"(gp), "r"(in ? 16u : 0u)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (tid < kStage) {  // position of each staged token inside its sequence (-1: none)
        const int64_t t = t0 - kConvHalo + tid;
        int p = -1;
        if (t >= 0 && t < L.total) {
            const int s = seq_of_token(cu, L.n_seqs, t);
            int64_t start, len;
            seq_range(cu, s, L.total, &start, &len);
            if (t >= start && t < start + len) p = (int)(t - start);
            else if (err && blockIdx.y == 0) atomicExch(err, kErrSeqlens);
        }
        pos_s[tid] = p;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // ---- RoPE in place on q and k rows (bf16 -> fp16 or fp32 -> fp32), RoPE'd rows out
    for (int idx = tid; idx < kStage * kRowsPerCta * (HALF / 8); idx += kFeatThreads) {
        const int f8 = idx % (HALF / 8), rj = idx / (HALF / 8), j = rj % kRowsPerCta, tk = rj / kRowsPerCta;
        int kind, head;
        const bool on = row_info(j, &kind, &head);
        unsigned char* r = xs + (size_t)rj * ROWB;
        float x1[8], x2[8];
        Vec8<Tin>::unpack(r + f8 * 8 * E, x1);
        Vec8<Tin>::unpack(r + (HALF + f8 * 8) * E, x2);
        const int p = pos_s[tk];
        if (kind != 2 && p >= 0) {
            const float2* fp = fine + (p & 63) * HALF + f8 * 8;
            const float2* gp = coarse + (p >> 6) * HALF + f8 * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 f = __ldg(fp + i), g = __ldg(gp + i);
                const float c = g.x * f.x - g.y * f.y, sn = g.y * f.x + g.x * f.y;
                const float a = x1[i], b = x2[i];
                x1[i] = a * c - b * sn;
                x2[i] = b * c + a * sn;
            }
        }
        Vec8<Tf>::pack(r + f8 * 8 * E, x1);
        Vec8<Tf>::pack(r + (HALF + f8 * 8) * E, x2);
        const int64_t t = t0 - kConvHalo + tk;
        if (on && kind != 2 && tk >= kConvHalo && t < L.total) {
            Tf* dst = (kind == 0 ? qr : kr) + ((size_t)t * (kind == 0 ? L.Hq : L.Hkv) + head) * D;
            Vec8<Tf>::pack(reinterpret_cast<unsigned char*>(dst + f8 * 8), x1);
            Vec8<Tf>::pack(reinterpret_cast<unsigned char*>(dst + HALF + f8 * 8), x2);
        }
    }
    __syncthreads();

    // ---- causal conv (tap m reads token t - 7 + m) and L2 norm; a thread keeps one (row, 8 channels)
    static_assert((kFeatThreads % (kRowsPerCta * G8)) == 0, "a thread keeps its row and channels");
    const int cg = tid % G8, j = (tid / G8) % kRowsPerCta;
    int kind, head;
    const bool on = row_info(j, &kind, &head);
    const bool do_norm = kind == 1 || (kind == 0 && (L.flags & HLA_FLAG_L2NORM_Q));
    float wt[8][kConvWidth];
    {
        const float4* wp = reinterpret_cast<const float4*>((kind == 0 ? wq : (kind == 1 ? wk : wv)) +
                                                           ((size_t)head * D + cg * 8) * kConvWidth);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 a = __ldg(wp + 2 * c), b = __ldg(wp + 2 * c + 1);
            wt[c][0] = a.x; wt[c][1] = a.y; wt[c][2] = a.z; wt[c][3] = a.w;
            wt[c][4] = b.x; wt[c][5] = b.y; wt[c][6] = b.z; wt[c][7] = b.w;
        }
    }
    Tf* hat = (kind == 0 ? qhat : (kind == 1 ? khat : vhat)) + (size_t)head * D + cg * 8;
    const size_t H = kind == 0 ? L.Hq : L.Hkv;
    constexpr int kTokStep = kFeatThreads / (kRowsPerCta * G8);
#pragma unroll 1
    for (int to = tid / (kRowsPerCta * G8); to < kTT; to += kTokStep) {
        const int64_t t = t0 + to;
        const int p = pos_s[to + kConvHalo];
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) {
            if (m < kConvHalo - p) continue;  // before the sequence's first token (p < 0: none)
            float x[8];
            Vec8<Tf>::unpack(xs + ((size_t)(to + m) * kRowsPerCta + j) * ROWB + cg * 8 * E, x);
#pragma unroll
            for (int c = 0; c < 8; ++c) y[c] = fmaf(wt[c][m], x[c], y[c]);
        }
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) ss = fmaf(y[c], y[c], ss);
#pragma unroll
        for (int o = G8 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (do_norm) {
            const float rs = rsqrtf(ss + 1e-6f);
#pragma unroll
            for (int c = 0; c < 8; ++c) y[c] *= rs;
        }
        if (on && t < L.total && p >= 0) Vec8<Tf>::pack(reinterpret_cast<unsigned char*>(hat + (size_t)t * H * D), y);
    }
}

template <typename Tin, typename Tf>
cudaError_t launch_features(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                            const float* wq, const float* wk, const float* wv, const int32_t* cu,
                            const float2* fine, const float2* coarse, Tf* qr, Tf* kr, Tf* qhat,
                            Tf* khat, Tf* vhat, int32_t* err, cudaStream_t st) {
    dim3 grid((unsigned)((L.total + kTT - 1) / kTT), (unsigned)((L.Hq + 2 * L.Hkv + kRowsPerCta - 1) / kRowsPerCta));
    if (L.total <= 0) return cudaSuccess;
    const size_t smem = (size_t)kStage * kRowsPerCta * L.d * sizeof(Tin);
    if (L.d == 128) {
        static bool configured = false;
        if (!configured) {
            cudaError_t e = cudaFuncSetAttribute(features_kernel<Tin, Tf, 128>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            configured = true;
        }
        features_kernel<Tin, Tf, 128><<<grid, kFeatThreads, smem, st>>>(
            L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr, qhat, khat, vhat, err);
    } else {
        features_kernel<Tin, Tf, 64><<<grid, kFeatThreads, smem, st>>>(
            L, q, k, v, wq, wk, wv, cu, fine, coarse, qr, kr, qhat, khat, vhat, err);
    }
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
