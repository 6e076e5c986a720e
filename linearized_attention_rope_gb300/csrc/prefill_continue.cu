// Prefill that continues from a decode state: new tokens appended to
// sequences that already hold a context (positions start at the state's pos),
// with the fixed-budget cache of "迈向线性的关键：分析驱动的 Transformer
// 线性化", section 填补近似缺口的实用设计 (sinks + window exact, the GDN
// state of section 线性注意力替换机制 absorbing every non-sink token that
// leaves the window) carried across the boundary: the conv histories, the
// window keys and values in the KV ring, the tokens still waiting to be
// absorbed in the pending ring, and S.  The result is that of decoding the
// new tokens one at a time (or of one prefill over the whole sequence).
//
// Four launches, token-serial inside each sequence (a general path for
// prompts appended to live sequences, not the throughput path of a fresh
// prefill):
//  A. per (kv head, sequence): RoPE'd key, khat and vhat of every new token,
//     the conv histories read from the state and advanced there;
//  B. per (q-head, sequence): per new token, qhat (the head's conv history,
//     advanced in the state), the absorption of token p - W (from the
//     pending ring if it precedes the new tokens, else from launch A's
//     output) into S held in registers, o_lin = S^T qhat, and the softmax
//     over the sinks and the window (keys from the ring before the new
//     tokens, from launch A after); out = o_sm + lambda_h o_lin; then S and
//     the head's pending gates are written back;
//  C. per (kv head, sequence): the new tokens' keys and values into the ring
//     and the pending ring;
//  D. per sequence: pos += the number of new tokens.
// Launch B reads the ring and pending entries that launch C overwrites, and
// every launch reads pos, so the order is A, B, C, D on one stream.
#include "hla_common.cuh"

namespace hla {

namespace {

__device__ __forceinline__ int64_t ring_slot_of(int64_t p, int n_sinks, int window) {
    return p < n_sinks ? p : n_sinks + (p - n_sinks) % window;
}

template <typename Tin>
__device__ __forceinline__ float rope_at(const Tin* __restrict__ x, int c, int D, int64_t p, const LayerDims& L) {
    const int half = D / 2, i = c % half;
    float cs, sn;
    rope_cs_exact(p, L.theta[i], &cs, &sn);
    const float x1 = to_f32(x[i]), x2 = to_f32(x[i + half]);
    return c < half ? x1 * cs - x2 * sn : x2 * cs + x1 * sn;
}

// sum over the CTA's threads (blockDim.x <= 1024) of v, for every thread; red holds 32 floats
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    __syncthreads();
    return t;
}
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int i = 0; i < nw; ++i) t = fmaxf(t, red[i]);
    __syncthreads();
    return t;
}

// ---- A: per (kv head, sequence), thread per channel
template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(D)
cont_kv_features_kernel(LayerDims L, const Tin* __restrict__ k, const Tin* __restrict__ v,
                        const float* __restrict__ wk, const float* __restrict__ wv, const int32_t* __restrict__ cu,
                        hla_state s, Tf* __restrict__ kr_out, Tf* __restrict__ khat_out, Tf* __restrict__ vhat_out) {
    __shared__ float red[32];
    const int kv = blockIdx.x, n = blockIdx.y, c = threadIdx.x;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p0 = s.pos[n];
    if (p0 < 0) {  // flagged by launch B
        return;
    }
    const size_t hist = ((size_t)n * kConvHalo * L.Hkv + kv) * D + c, step = (size_t)L.Hkv * D;
    float hk[kConvHalo], hv[kConvHalo], w_k[kConvWidth], w_v[kConvWidth];
#pragma unroll
    for (int m = 0; m < kConvHalo; ++m) {
        hk[m] = s.conv_k[hist + m * step];
        hv[m] = s.conv_v[hist + m * step];
    }
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) {
        w_k[m] = wk[((size_t)kv * D + c) * kConvWidth + m];
        w_v[m] = wv[((size_t)kv * D + c) * kConvWidth + m];
    }
    for (int64_t t = 0; t < len; ++t) {
        const size_t row = ((size_t)(start + t) * L.Hkv + kv) * D;
        const float xk = rope_at(k + row, c, D, p0 + t, L);
        const float xv = to_f32(v[row + c]);
        float ak = w_k[kConvHalo] * xk, av = w_v[kConvHalo] * xv;
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) {
            ak = fmaf(w_k[m], hk[m], ak);
            av = fmaf(w_v[m], hv[m], av);
        }
#pragma unroll
        for (int m = 0; m + 1 < kConvHalo; ++m) {
            hk[m] = hk[m + 1];
            hv[m] = hv[m + 1];
        }
        hk[kConvHalo - 1] = xk;
        hv[kConvHalo - 1] = xv;
        const float inv = rsqrtf(block_sum(ak * ak, red) + 1e-6f);
        kr_out[row + c] = from_f32<Tf>(xk);
        khat_out[row + c] = from_f32<Tf>(ak * inv);
        vhat_out[row + c] = from_f32<Tf>(av);
    }
#pragma unroll
    for (int m = 0; m < kConvHalo; ++m) {
        s.conv_k[hist + m * step] = hk[m];
        s.conv_v[hist + m * step] = hv[m];
    }
}

// ---- B: per (q-head, sequence), 4 threads per value column of S (the layout of the token-serial GDN
// kernel); softmax keys spread over all threads
constexpr int kParts = 4;

template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(D * kParts)
cont_head_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ v, const float* __restrict__ g,
                 const float* __restrict__ beta, const float* __restrict__ lambda, const float* __restrict__ wq,
                 const int32_t* __restrict__ cu, hla_state s, const Tf* __restrict__ kr_new,
                 const Tf* __restrict__ khat_new, const Tf* __restrict__ vhat_new, Tin* __restrict__ out) {
    constexpr int Q = D / kParts, NT = D * kParts;
    constexpr int kMaxKeys = 1024;  // keys handled per pass of the softmax
    __shared__ __align__(16) float qh_s[D], qr_s[D], kj_s[D], vj_s[D];
    __shared__ float lg_s[kMaxKeys];
    __shared__ float red[32];
    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G, tid = threadIdx.x;
    const int col = tid / kParts, part = tid % kParts;
    const int ns = L.n_sinks, W = L.window, P = W + 1, R = ns + W;
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    const bool lin_on = !(L.flags & HLA_FLAG_LINEAR_OFF), sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p0 = s.pos[n];
    if (p0 < 0) {  // not a position a prefill or a decode step can leave: flag it, touch nothing
        if (tid == 0 && h == 0) atomicExch(s.err, kErrState);
        return;
    }
    const float lam = lambda[h];
    const Tin* kring = static_cast<const Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    const Tin* vring = static_cast<const Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;

    float S[Q];  // S[part * Q + i][col]
    const float* Sg = s.S + ((size_t)n * L.Hq + h) * D * D;
#pragma unroll
    for (int i = 0; i < Q; ++i) S[i] = Sg[(size_t)(part * Q + i) * D + col];
    // q conv history of this head (channel tid < D)
    const size_t qhist = ((size_t)n * kConvHalo * L.Hq + h) * D + tid, qstep = (size_t)L.Hq * D;
    float hq[kConvHalo], w_q[kConvWidth];
    if (tid < D) {
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) hq[m] = s.conv_q[qhist + m * qstep];
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) w_q[m] = wq[((size_t)h * D + tid) * kConvWidth + m];
    }
    const float qscale = rsqrtf((float)D);

    for (int64_t t = 0; t < len; ++t) {
        const int64_t p = p0 + t;
        // ---- qhat and the RoPE'd query of token p
        float aq = 0.f;
        if (tid < D) {
            const float xr = rope_at(q + ((size_t)(start + t) * L.Hq + h) * D, tid, D, p, L);
            aq = w_q[kConvHalo] * xr;
#pragma unroll
            for (int m = 0; m < kConvHalo; ++m) aq = fmaf(w_q[m], hq[m], aq);
#pragma unroll
            for (int m = 0; m + 1 < kConvHalo; ++m) hq[m] = hq[m + 1];
            hq[kConvHalo - 1] = xr;
            qr_s[tid] = xr;
        }
        const float qinv = (L.flags & HLA_FLAG_L2NORM_Q) ? rsqrtf(block_sum(aq * aq, red) + 1e-6f) : 1.f;
        if (tid < D) qh_s[tid] = aq * qinv;

        // ---- absorb token j = p - W (not a sink): its own gate and beta, no decay while it waited
        const int64_t j = p - W;
        if (j >= ns) {
            float alpha, b;
            if (j < p0) {  // still in the pending ring
                const size_t slot = (size_t)(j % P);
                if (tid < D) {
                    const size_t ps = (((size_t)n * L.Hkv + kv) * P + slot) * D + tid;
                    kj_s[tid] = s.pend_k[ps];
                    vj_s[tid] = s.pend_v[ps];
                }
                alpha = expf(s.pend_g[((size_t)n * L.Hq + h) * P + slot]);
                b = s.pend_beta[((size_t)n * L.Hq + h) * P + slot];
            } else {  // one of the new tokens
                const size_t row = (size_t)(start + (j - p0));
                if (tid < D) {
                    kj_s[tid] = to_f32(khat_new[(row * L.Hkv + kv) * D + tid]);
                    vj_s[tid] = to_f32(vhat_new[(row * L.Hkv + kv) * D + tid]);
                }
                alpha = expf(g[row * L.Hq + h]);
                b = beta[row * L.Hq + h];
            }
            __syncthreads();
            float x = 0.f;
#pragma unroll
            for (int i = 0; i < Q; ++i) x = fmaf(kj_s[part * Q + i], S[i], x);
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);  // (k^T S)[col]
            const float u = gla ? vj_s[col] : b * (vj_s[col] - alpha * x);
#pragma unroll
            for (int i = 0; i < Q; ++i) S[i] = fmaf(alpha, S[i], kj_s[part * Q + i] * u);
        }
        __syncthreads();  // qh_s complete
        float ol = 0.f;
#pragma unroll
        for (int i = 0; i < Q; ++i) ol = fmaf(qh_s[part * Q + i], S[i], ol);
        ol += __shfl_xor_sync(0xffffffffu, ol, 1);
        ol += __shfl_xor_sync(0xffffffffu, ol, 2);  // o_lin[col]

        // ---- softmax over the sinks and the window: key index e < n_keys enumerates positions
        const int64_t nsk = min((int64_t)ns, p + 1);
        const int64_t wlo = max((int64_t)ns, p - W + 1);
        const int n_keys = (int)(nsk + max((int64_t)0, p + 1 - wlo));
        auto key_pos = [&](int e) { return e < nsk ? (int64_t)e : wlo + (e - nsk); };
        float m_run = -INFINITY, l_run = 0.f, acc = 0.f;  // acc: channel `col` of P V, by thread part 0
        for (int e0 = 0; e0 < n_keys; e0 += kMaxKeys) {
            const int ne = min(kMaxKeys, n_keys - e0);
            float mloc = -INFINITY;
            for (int e = tid; e < ne; e += NT) {
                const int64_t jp = key_pos(e0 + e);
                float dot = 0.f;
                if (jp < p0) {
                    const Tin* kk = kring + (size_t)ring_slot_of(jp, ns, W) * D;
                    for (int c = 0; c < D; ++c) dot = fmaf(qr_s[c], to_f32(kk[c]), dot);
                } else {
                    const Tf* kk = kr_new + ((size_t)(start + (jp - p0)) * L.Hkv + kv) * D;
                    for (int c = 0; c < D; ++c) dot = fmaf(qr_s[c], to_f32(kk[c]), dot);
                }
                lg_s[e] = dot * qscale;
                mloc = fmaxf(mloc, lg_s[e]);
            }
            const float m_new = fmaxf(m_run, block_max(mloc, red));
            const float corr = m_run == -INFINITY ? 0.f : expf(m_run - m_new);
            float lloc = 0.f;
            for (int e = tid; e < ne; e += NT) {
                lg_s[e] = expf(lg_s[e] - m_new);
                lloc += lg_s[e];
            }
            l_run = l_run * corr + block_sum(lloc, red);  // (its barriers also publish lg_s)
            m_run = m_new;
            // P V for channel col: the part-th quarter of the keys, summed over the four parts
            float pv = 0.f;
            for (int e = part; e < ne; e += kParts) {
                const int64_t jp = key_pos(e0 + e);
                const float vv = jp < p0 ? to_f32(vring[(size_t)ring_slot_of(jp, ns, W) * D + col])
                                         : to_f32(v[((size_t)(start + (jp - p0)) * L.Hkv + kv) * D + col]);
                pv = fmaf(lg_s[e], vv, pv);
            }
            pv += __shfl_xor_sync(0xffffffffu, pv, 1);
            pv += __shfl_xor_sync(0xffffffffu, pv, 2);
            acc = acc * corr + pv;
            __syncthreads();  // lg_s is rewritten by the next pass
        }
        if (part == 0) {
            const float o_sm = sm_on && l_run > 0.f ? acc / l_run : 0.f;
            const float o = lin_on ? fmaf(lam, ol, o_sm) : o_sm;
            out[((size_t)(start + t) * L.Hq + h) * D + col] = from_f32<Tin>(o);
        }
    }
    // ---- write back: S, the q history, the gates of the new tokens still waiting to be absorbed
#pragma unroll
    for (int i = 0; i < Q; ++i) s.S[((size_t)n * L.Hq + h) * D * D + (size_t)(part * Q + i) * D + col] = S[i];
    if (tid < D) {
#pragma unroll
        for (int m = 0; m < kConvHalo; ++m) s.conv_q[qhist + m * qstep] = hq[m];
    }
    const int64_t p_end = p0 + len;
    for (int64_t t = tid; t < len; t += NT) {
        const int64_t p = p0 + t;
        if (p < p_end - W || p < ns) continue;  // absorbed already, or a sink (never absorbed)
        const size_t gs = ((size_t)n * L.Hq + h) * P + (size_t)(p % P);
        s.pend_g[gs] = g[(size_t)(start + t) * L.Hq + h];
        s.pend_beta[gs] = beta[(size_t)(start + t) * L.Hq + h];
    }
}

// ---- C: per (kv head, sequence): ring, pending ring, position
template <typename Tin, typename Tf, int D>
__global__ void __launch_bounds__(D)
cont_kv_state_kernel(LayerDims L, const Tin* __restrict__ v, const int32_t* __restrict__ cu, hla_state s,
                     const Tf* __restrict__ kr_new, const Tf* __restrict__ khat_new, const Tf* __restrict__ vhat_new) {
    const int kv = blockIdx.x, n = blockIdx.y, c = threadIdx.x;
    const int ns = L.n_sinks, W = L.window, P = W + 1, R = ns + W;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p0 = s.pos[n];
    if (p0 < 0) return;
    const int64_t p_end = p0 + len;
    Tin* kring = static_cast<Tin*>(s.k_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    Tin* vring = static_cast<Tin*>(s.v_ring) + ((size_t)n * L.Hkv + kv) * R * D;
    for (int64_t t = 0; t < len; ++t) {
        const int64_t p = p0 + t;
        const size_t row = ((size_t)(start + t) * L.Hkv + kv) * D + c;
        if (p < ns || p >= p_end - W) {  // a sink, or in the final window
            const size_t slot = (size_t)ring_slot_of(p, ns, W) * D + c;
            kring[slot] = from_f32<Tin>(to_f32(kr_new[row]));
            vring[slot] = v[row];
        }
        if (p >= p_end - W && p >= ns) {  // still waiting to be absorbed (sinks never are)
            const size_t ps = (((size_t)n * L.Hkv + kv) * P + (size_t)(p % P)) * D + c;
            s.pend_k[ps] = to_f32(khat_new[row]);
            s.pend_v[ps] = to_f32(vhat_new[row]);
        }
    }
}

// ---- D: pos += the number of new tokens (after every launch above has read it)
__global__ void cont_advance_kernel(LayerDims L, const int32_t* __restrict__ cu, int64_t* __restrict__ pos) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= L.n_seqs) return;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    if (pos[n] >= 0) pos[n] += len;
}

}  // namespace

template <typename Tin, typename Tf>
cudaError_t launch_prefill_continue(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* g,
                                    const float* beta, const float* lambda, const float* wq, const float* wk,
                                    const float* wv, const int32_t* cu, const hla_state& s, Tf* kr, Tf* khat,
                                    Tf* vhat, Tin* out, cudaStream_t st) {
    const dim3 gk(L.Hkv, L.n_seqs), gq(L.Hq, L.n_seqs);
    if (L.d == 128) {
        cont_kv_features_kernel<Tin, Tf, 128><<<gk, 128, 0, st>>>(L, k, v, wk, wv, cu, s, kr, khat, vhat);
        cont_head_kernel<Tin, Tf, 128><<<gq, 128 * kParts, 0, st>>>(L, q, v, g, beta, lambda, wq, cu, s, kr, khat,
                                                                     vhat, out);
        cont_kv_state_kernel<Tin, Tf, 128><<<gk, 128, 0, st>>>(L, v, cu, s, kr, khat, vhat);
    } else {
        cont_kv_features_kernel<Tin, Tf, 64><<<gk, 64, 0, st>>>(L, k, v, wk, wv, cu, s, kr, khat, vhat);
        cont_head_kernel<Tin, Tf, 64><<<gq, 64 * kParts, 0, st>>>(L, q, v, g, beta, lambda, wq, cu, s, kr, khat,
                                                                   vhat, out);
        cont_kv_state_kernel<Tin, Tf, 64><<<gk, 64, 0, st>>>(L, v, cu, s, kr, khat, vhat);
    }
    cont_advance_kernel<<<(L.n_seqs + 127) / 128, 128, 0, st>>>(L, cu, s.pos);
    return cudaGetLastError();
}

template cudaError_t launch_prefill_continue<float, float>(const LayerDims&, const float*, const float*, const float*,
                                                           const float*, const float*, const float*, const float*,
                                                           const float*, const float*, const int32_t*,
                                                           const hla_state&, float*, float*, float*, float*,
                                                           cudaStream_t);
template cudaError_t launch_prefill_continue<__nv_bfloat16, __half>(
    const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, const float*, const float*,
    const float*, const float*, const float*, const float*, const int32_t*, const hla_state&, __half*, __half*, __half*,
    __nv_bfloat16*, cudaStream_t);

}  // namespace hla
