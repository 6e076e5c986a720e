// Exact branch: softmax over the sink tokens plus the sliding window, scale
// 1/sqrt(d), on the RoPE'd q, k and the raw v; then the linear branch,
// weighted by lambda_h, is added in the epilogue:
//   o_t = softmax_{j in sinks U window}(q_t . k_j / sqrt(d)) v_j + lambda_h o_lin_t.
// Sources: "迈向线性的关键：分析驱动的 Transformer 线性化", section
// 填补近似缺口的实用设计 (8 sinks + window keep full attention) and Lemma 1 of
// section 从 softmax 到 delta 规则的一阶近似 (the 1/sqrt(d) scale);
// "Untangling Component Imbalance in Hybrid Linear Attention Conversion",
// section 关键设计 (1) (inference-time weighting of the two branches).
//
// One warp per (token, query head): each lane owns d/32 channels, dot
// products are finished with butterfly shuffles, and four keys are in
// flight per step.  Online softmax in base 2.
#include "hla_common.cuh"

namespace hla {

constexpr int kSmWarps = 8;

template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(kSmWarps * 32)
window_softmax_kernel(LayerDims L, const Tf* __restrict__ qr, const Tf* __restrict__ kr,
                      const Tin* __restrict__ v, const float* __restrict__ o_lin,
                      const float* __restrict__ lambda, const int32_t* __restrict__ cu,
                      Tin* __restrict__ out) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t wid = (int64_t)blockIdx.x * kSmWarps + (threadIdx.x >> 5);
    if (wid >= L.total * L.Hq) return;
    const int64_t t = wid / L.Hq;
    const int h = (int)(wid % L.Hq), kv = h / L.G;
    const int s = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, s, L.total, &start, &len);
    if (t < start || t >= start + len) return;  // malformed cu_seqlens: flagged by the feature pass
    const int64_t p = t - start;
    const int c0 = lane * E;

    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;  // 1/sqrt(d) * log2(e)
    float qv[E];
    load_vec<E>(qr + ((size_t)t * L.Hq + h) * D + c0, qv);
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] *= qscale;

    const int64_t n_sink_keys = p + 1 < L.n_sinks ? p + 1 : L.n_sinks;
    const int64_t w_lo = (p - L.window + 1) > L.n_sinks ? (p - L.window + 1) : L.n_sinks;
    const int64_t n_win = p >= w_lo ? p - w_lo + 1 : 0;
    const int64_t n_keys = n_sink_keys + n_win;

    float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;

    const size_t kv_stride = (size_t)L.Hkv * D;
    const Tf* kbase = kr + (size_t)start * kv_stride + (size_t)kv * D + c0;
    const Tin* vbase = v + (size_t)start * kv_stride + (size_t)kv * D + c0;
    for (int64_t i0 = 0; i0 < n_keys; i0 += 4) {
        float sc[4];
        int64_t jj[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int64_t i = i0 + u;
            jj[u] = i < n_sink_keys ? i : w_lo + (i - n_sink_keys);
            float kx[E];
            float part = 0.f;
            if (i < n_keys) {
                load_vec<E>(kbase + (size_t)jj[u] * kv_stride, kx);
#pragma unroll
                for (int e = 0; e < E; ++e) part = fmaf(qv[e], kx[e], part);
            }
            sc[u] = part;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int u = 0; u < 4; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], o);
        }
        float mx = m;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (i0 + u >= n_keys) sc[u] = -INFINITY;
            mx = fmaxf(mx, sc[u]);
        }
        const float corr = exp2f(m - mx);
        l *= corr;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (i0 + u < n_keys) {
                float pu = exp2f(sc[u] - mx);
                l += pu;
                float vx[E];
                load_vec<E>(vbase + (size_t)jj[u] * kv_stride, vx);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(pu, vx[e], acc[e]);
            }
        }
        m = mx;
    }

    const bool sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF);
    const bool lin_on = !(L.flags & HLA_FLAG_LINEAR_OFF) && (p - L.window >= L.n_sinks);
    float res[E];
    const float inv_l = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) res[e] = sm_on ? acc[e] * inv_l : 0.f;
    if (lin_on) {
        const float lam = __ldg(lambda + h);
        float ol[E];
        load_vec<E>(o_lin + ((size_t)t * L.Hq + h) * D + c0, ol);
#pragma unroll
        for (int e = 0; e < E; ++e) res[e] = fmaf(lam, ol[e], res[e]);
    }
    Tin* dst = out + ((size_t)t * L.Hq + h) * D + c0;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = from_f32<Tin>(res[e]);
}

template <typename Tin, typename Tf>
cudaError_t launch_window_softmax(const LayerDims& L, const Tf* qr, const Tf* kr, const Tin* v,
                                  const float* o_lin, const float* lambda, const int32_t* cu,
                                  Tin* out, cudaStream_t st) {
    int64_t rows = L.total * L.Hq;
    unsigned blocks = (unsigned)((rows + kSmWarps - 1) / kSmWarps);
    if (L.d == 128)
        window_softmax_kernel<Tin, Tf, 128><<<blocks, kSmWarps * 32, 0, st>>>(L, qr, kr, v, o_lin, lambda, cu, out);
    else
        window_softmax_kernel<Tin, Tf, 64><<<blocks, kSmWarps * 32, 0, st>>>(L, qr, kr, v, o_lin, lambda, cu, out);
    return cudaGetLastError();
}

template cudaError_t launch_window_softmax<float, float>(const LayerDims&, const float*, const float*,
                                                         const float*, const float*, const float*,
                                                         const int32_t*, float*, cudaStream_t);
template cudaError_t launch_window_softmax<__nv_bfloat16, __half>(
    const LayerDims&, const __half*, const __half*, const __nv_bfloat16*, const float*, const float*,
    const int32_t*, __nv_bfloat16*, cudaStream_t);

}  // namespace hla
