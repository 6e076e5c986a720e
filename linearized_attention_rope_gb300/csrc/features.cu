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

constexpr int kRun = 32;          // output tokens per CTA
constexpr int kHist = 8;          // tokens before the run that are read for the conv history (7 used)
constexpr int kReseed = 16;       // cos/sin re-formed from the tables every 16 positions
constexpr int kFeatThreads = 256;

// Eight consecutive raw elements of one row, as loaded (16 B for bf16, 32 B for fp32).
template <typename Tin> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    static constexpr int kWords = 4;
    uint32_t w[4];
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
    __device__ __forceinline__ void unpack(float* x) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    }
};
template <> struct Raw8<float> {
    static constexpr int kWords = 8;
    uint32_t w[8];
    __device__ __forceinline__ void load(const float* p) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        w[0] = __float_as_uint(a.x); w[1] = __float_as_uint(a.y); w[2] = __float_as_uint(a.z); w[3] = __float_as_uint(a.w);
        w[4] = __float_as_uint(b.x); w[5] = __float_as_uint(b.y); w[6] = __float_as_uint(b.z); w[7] = __float_as_uint(b.w);
    }
    __device__ __forceinline__ void unpack(float* x) const {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(w[i]);
    }
};

__device__ __forceinline__ void store8(__half* p, const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
}

// One CTA = kRun tokens x HPC feature rows (q heads, then k heads, then v
// heads).  D / 8 lanes cover one row, 8 channels each, and walk the tokens in
// order in batches of 8 (every batch starts at a multiple of 8): the rotated
// values of the last 8 tokens sit in a register ring indexed by token mod 8,
// which serves as the conv history; RoPE's partner half (channel c +- D/2)
// comes from lane xor D/16, and cos/sin advance by one position with a
// rotation by theta_i, re-formed from the tables (angle addition, both
// reduced in double precision) at every 16th position of a sequence and at
// the CTA's first token.
template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(kFeatThreads, 1)
features_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                const Tin* __restrict__ v, const float* __restrict__ wq,
                const float* __restrict__ wk, const float* __restrict__ wv,
                const int32_t* __restrict__ cu, const float2* __restrict__ fine,
                const float2* __restrict__ coarse, Tf* __restrict__ qr, Tf* __restrict__ kr,
                Tf* __restrict__ qhat, Tf* __restrict__ khat, Tf* __restrict__ vhat,
                int32_t* __restrict__ err) {
    constexpr int G8 = D / 8, HALF = D / 2, RPW = 32 / G8, HPC = (kFeatThreads / 32) * RPW;
    constexpr bool kPrefetch = sizeof(Tin) == 2;  // bf16 rows of a batch are loaded up front
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cg = lane % G8, c0 = 8 * cg;
    const int n_rows = L.Hq + 2 * L.Hkv;
    int head = blockIdx.y * HPC + warp * RPW + lane / G8;
    const bool active = head < n_rows;  // idle lanes still take part in the shuffles
    if (!active) head = n_rows - 1;
    int kind = 0;  // 0 = q, 1 = k, 2 = v
    if (head >= L.Hq + L.Hkv) { kind = 2; head -= L.Hq + L.Hkv; }
    else if (head >= L.Hq) { kind = 1; head -= L.Hq; }
    const size_t row_stride = (size_t)(kind == 0 ? L.Hq : L.Hkv) * D;  // elements between tokens
    const bool do_rot = kind != 2;
    const bool do_norm = kind == 1 || (kind == 0 && (L.flags & HLA_FLAG_L2NORM_Q));
    const float sgn = c0 < HALF ? -1.f : 1.f;  // x1' = x1 c - x2 s,  x2' = x2 c + x1 s
    const int f0 = c0 % HALF;

    float wt[8][kConvWidth];
    {
        const float4* wp = reinterpret_cast<const float4*>((kind == 0 ? wq : (kind == 1 ? wk : wv)) +
                                                           ((size_t)head * D + c0) * kConvWidth);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 a = __ldg(wp + 2 * j), b = __ldg(wp + 2 * j + 1);
            wt[j][0] = a.x; wt[j][1] = a.y; wt[j][2] = a.z; wt[j][3] = a.w;
            wt[j][4] = b.x; wt[j][5] = b.y; wt[j][6] = b.z; wt[j][7] = b.w;
        }
    }
    float2 stp[8];  // (cos, sin) of theta_i
#pragma unroll
    for (int j = 0; j < 8; ++j) stp[j] = __ldg(fine + HALF + f0 + j);

    const int64_t t_out = (int64_t)blockIdx.x * kRun;
    const int64_t t_first = t_out - kHist > 0 ? t_out - kHist : 0;
    const int64_t t_end = t_out + kRun < L.total ? t_out + kRun : L.total;
    int s = seq_of_token(cu, L.n_seqs, t_first);
    int64_t s_start, s_len;
    seq_range(cu, s, L.total, &s_start, &s_len);

    const Tin* src = (kind == 0 ? q : (kind == 1 ? k : v)) + (size_t)head * D + c0;
    Tf* rot_dst = (kind == 0 ? qr : kr) + (size_t)head * D + c0;
    Tf* hat_dst = (kind == 0 ? qhat : (kind == 1 ? khat : vhat)) + (size_t)head * D + c0;

    float ring[8][8];  // rotated rows of tokens t = 8 b + slot
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int j = 0; j < 8; ++j) ring[m][j] = 0.f;
    float cs[8], sn[8];
    bool seeded = false;

#pragma unroll 1
    for (int64_t tb = t_out - kHist; tb < t_end; tb += 8) {
        Raw8<Tin> raw[8];
        if (kPrefetch) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (tb + u >= t_first && tb + u < t_end) raw[u].load(src + (size_t)(tb + u) * row_stride);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t t = tb + u;
            if (t < t_first || t >= t_end) continue;  // same t across the CTA: uniform
            if (!kPrefetch) raw[u].load(src + (size_t)t * row_stride);
            while (t >= s_start + s_len && s + 1 < L.n_seqs) {
                ++s;
                seq_range(cu, s, L.total, &s_start, &s_len);
            }
            const bool in_seq = t >= s_start && t < s_start + s_len;
            if (!in_seq && err && threadIdx.x == 0 && blockIdx.y == 0) atomicExch(err, kErrSeqlens);
            const int pos = in_seq ? (int)(t - s_start) : 0;
            if (pos == 0) {  // a sequence starts: zero conv history
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int j = 0; j < 8; ++j) ring[m][j] = 0.f;
            }
            if (!seeded || (pos & (kReseed - 1)) == 0) {
                const float2* fp = fine + (pos & 63) * HALF + f0;
                const float2* gp = coarse + (pos >> 6) * HALF + f0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 f = __ldg(fp + j), g = __ldg(gp + j);
                    cs[j] = g.x * f.x - g.y * f.y;
                    sn[j] = g.y * f.x + g.x * f.y;
                }
                seeded = true;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float c = cs[j] * stp[j].x - sn[j] * stp[j].y;
                    sn[j] = sn[j] * stp[j].x + cs[j] * stp[j].y;
                    cs[j] = c;
                }
            }
            Raw8<Tin> partner;
#pragma unroll
            for (int i = 0; i < Raw8<Tin>::kWords; ++i) partner.w[i] = __shfl_xor_sync(0xffffffffu, raw[u].w[i], G8 / 2);
            float x[8], xp[8];
            raw[u].unpack(x);
            partner.unpack(xp);
            if (do_rot && in_seq) {
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = fmaf(x[j], cs[j], sgn * xp[j] * sn[j]);
            }
            const bool out_row = t >= t_out && active;
            if (out_row && do_rot) store8(rot_dst + (size_t)t * row_stride, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) ring[u][j] = in_seq ? x[j] : 0.f;
            // causal depthwise conv: tap m multiplies token t - 7 + m, ring slot (u + 1 + m) mod 8
            float y[8];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < kConvWidth; ++m) a = fmaf(wt[j][m], ring[(u + 1 + m) & 7][j], a);
                y[j] = a;
                ss = fmaf(a, a, ss);
            }
#pragma unroll
            for (int o = G8 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (do_norm) {
                const float r = rsqrtf(ss + 1e-6f);
#pragma unroll
                for (int j = 0; j < 8; ++j) y[j] *= r;
            }
            if (out_row) store8(hat_dst + (size_t)t * row_stride, y);
        }
    }
}

template <typename Tin, typename Tf>
cudaError_t launch_features(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                            const float* wq, const float* wk, const float* wv, const int32_t* cu,
                            const float2* fine, const float2* coarse, Tf* qr, Tf* kr, Tf* qhat,
                            Tf* khat, Tf* vhat, int32_t* err, cudaStream_t st) {
    const int hpc = (kFeatThreads / 32) * (32 / (L.d / 8));
    dim3 grid((unsigned)((L.total + kRun - 1) / kRun), (unsigned)((L.Hq + 2 * L.Hkv + hpc - 1) / hpc));
    if (L.total <= 0) return cudaSuccess;
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
