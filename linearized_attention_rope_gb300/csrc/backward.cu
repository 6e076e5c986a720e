// Backward of the hybrid layer: the gradients of L = sum(dO . o) with respect
// to q, k, v, the gates g, beta, the branch weight lambda and the conv
// filters, for the layer of "迈向线性的关键：分析驱动的 Transformer 线性化"
// (RoPE -> short conv -> L2 norm feature path of section 实践建议 item 3, the
// delayed GDN of sections 线性注意力替换机制 and 填补近似缺口的实用设计, the
// sink + window softmax) combined as o = o_sm + lambda_h o_lin ("Untangling
// Component Imbalance in Hybrid Linear Attention Conversion", 关键设计 (1)).
//
// fp32 throughout, on the CUDA cores; every reduction has a fixed order (no
// atomics).  Launches, in order:
//  1. rope: RoPE'd q and k rows (fp32) for every token and head;
//  2. conv: q~, k~ (and their L2-normalised qhat, khat) and vhat = conv(v);
//  3. GDN (per sequence and q-head): a forward pass that stores the state
//     every kCk absorptions (and the lambda gradient's partial sum), then a
//     reverse pass over the positions: segments of kCk absorptions are
//     recomputed from their checkpoint into scratch, and the read-out and
//     absorption steps are differentiated in reverse order (dqhat, and per
//     head dkhat, dvhat, dg, dbeta);
//  4. softmax (per sequence and q-head): per query the max, sum and
//     D = sum_j P dP and dqr; then per key the queries that see it give dkr
//     and dv (per head);
//  5. feature backward of q (L2, conv, RoPE); of k and v after the per-head
//     gradients of each kv group are summed;
//  6. the conv filters' gradients (per token block, then over the blocks);
//  7. lambda's gradient over the sequences.
#include "hla_common.cuh"

namespace hla {

namespace {

constexpr int kCk = 64;     // absorptions between GDN checkpoints
constexpr int kWB = 256;    // tokens per block of the conv-filter reduction

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// sum over the CTA of v, for every thread (red: 32 floats)
__device__ __forceinline__ float cta_sum_f(float v, float* red) {
    v = warp_sum_f(v);
    const int nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    __syncthreads();
    return t;
}
__device__ __forceinline__ float cta_max_f(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int i = 0; i < nw; ++i) t = fmaxf(t, red[i]);
    __syncthreads();
    return t;
}

// ---- 1. RoPE'd rows: row r < Hq is q-head r, else k-head r - Hq; thread per channel
template <typename Tin>
__global__ void bwd_rope_kernel(LayerDims L, const Tin* __restrict__ q, const Tin* __restrict__ k,
                                const int32_t* __restrict__ cu, float* __restrict__ qr, float* __restrict__ kr,
                                int32_t* __restrict__ err) {
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d, half = D / 2;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    // a token outside every sequence: cu_seqlens is not a monotone table from 0 to total
    if ((p < 0 || p >= len) && r == 0 && c == 0) atomicExch(err, kErrSeqlens);
    const bool isq = r < L.Hq;
    const int hh = isq ? r : r - L.Hq, H = isq ? L.Hq : L.Hkv;
    const Tin* x = (isq ? q : k) + ((size_t)t * H + hh) * D;
    const int i = c % half;
    float cs, sn;
    rope_cs_exact(p, L.theta[i], &cs, &sn);
    const float x1 = to_f32(x[i]), x2 = to_f32(x[i + half]);
    (isq ? qr : kr)[((size_t)t * H + hh) * D + c] = c < half ? x1 * cs - x2 * sn : x2 * cs + x1 * sn;
}

// ---- 2. conv (+ L2): rows r < Hq: q-heads, < Hq + Hkv: k-heads, else v-heads; thread per channel
template <typename Tin>
__global__ void bwd_conv_kernel(LayerDims L, const Tin* __restrict__ v, const float* __restrict__ wq,
                                const float* __restrict__ wk, const float* __restrict__ wv,
                                const int32_t* __restrict__ cu, const float* __restrict__ qr,
                                const float* __restrict__ kr, float* __restrict__ qt, float* __restrict__ qh,
                                float* __restrict__ kt, float* __restrict__ kh, float* __restrict__ vh) {
    __shared__ float red[32];
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* w = (kind == 0 ? wq : kind == 1 ? wk : wv) + ((size_t)hh * D + c) * kConvWidth;
    float acc = 0.f;
    for (int m = 0; m < kConvWidth; ++m) {
        const int64_t pp = p - (kConvWidth - 1) + m;
        if (pp < 0) continue;
        const size_t row = ((size_t)(start + pp) * H + hh) * D + c;
        const float x = kind == 0 ? qr[row] : kind == 1 ? kr[row] : to_f32(v[row]);
        acc = fmaf(w[m], x, acc);
    }
    const size_t o = ((size_t)t * H + hh) * D + c;
    if (kind == 2) {
        vh[o] = acc;
        return;
    }
    const bool norm = kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q);
    const float inv = norm ? rsqrtf(cta_sum_f(acc * acc, red) + 1e-6f) : 1.f;
    (kind == 0 ? qt : kt)[o] = acc;
    (kind == 0 ? qh : kh)[o] = acc * inv;
}

// ---- 3. GDN: per (q-head, sequence), 4 threads per value column (thread (col, part) holds rows
// part * Q .. + Q - 1 of column col).  States in checkpoints and scratch use the private layout
// [i][col][part] (a warp's accesses for one i are 128 contiguous bytes).
constexpr int kParts = 4;

template <int D>
__device__ __forceinline__ size_t st_idx(int i, int col, int part) {
    return ((size_t)i * D + col) * kParts + part;
}

// out[row] = sum over the columns of val[i] (row = part * Q + i), for every row; written to out_s (D floats)
template <int D>
__device__ __forceinline__ void row_reduce(const float* val, float* red /*[D/8][D]*/, float* out_s) {
    constexpr int Q = D / kParts;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, part = tid % kParts;
    float x[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        float y = val[i];
        y += __shfl_xor_sync(0xffffffffu, y, 4);
        y += __shfl_xor_sync(0xffffffffu, y, 8);
        y += __shfl_xor_sync(0xffffffffu, y, 16);
        x[i] = y;
    }
    if (lane < kParts) {
#pragma unroll
        for (int i = 0; i < Q; ++i) red[warp * D + part * Q + i] = x[i];
    }
    __syncthreads();
    if (tid < D) {
        float s = 0.f;
        for (int w = 0; w < D / 8; ++w) s += red[w * D + tid];
        out_s[tid] = s;
    }
    __syncthreads();
}

template <typename Tin, int D>
__global__ void __launch_bounds__(D * kParts)
bwd_gdn_kernel(LayerDims L, const float* __restrict__ g, const float* __restrict__ beta,
               const float* __restrict__ lambda, const Tin* __restrict__ dout, const int32_t* __restrict__ cu,
               const float* __restrict__ qh, const float* __restrict__ kh, const float* __restrict__ vh,
               float* __restrict__ ckpt, float* __restrict__ scratch, float* __restrict__ dqh,
               float* __restrict__ dkh_h, float* __restrict__ dvh_h, float* __restrict__ dg,
               float* __restrict__ dbeta, float* __restrict__ dlam_part) {
    constexpr int Q = D / kParts;
    __shared__ __align__(16) float qv_s[D], kv_s[D], vv_s[D], do_s[D], out_s[D];
    __shared__ float red_s[(D / 8) * D];
    __shared__ float red[32];
    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G, tid = threadIdx.x;
    const int col = tid / kParts, part = tid % kParts;
    const int ns = L.n_sinks, W = L.window;
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t n_abs = max((int64_t)0, len - W - ns);
    const float lam = lambda[h];
    const size_t DD = (size_t)D * D;
    const int64_t ck0 = start / kCk + n;  // this sequence's first checkpoint slot
    float* my_scratch = scratch + ((size_t)n * L.Hq + h) * (kCk + 1) * DD;
    auto ck = [&](int64_t s) { return ckpt + ((size_t)(ck0 + s) * L.Hq + h) * DD; };
    auto row_h = [&](const float* base, int64_t t, int heads, int hh) { return base + ((size_t)t * heads + hh) * D; };
    auto out_row = [&](float* base, int64_t t) { return base + ((size_t)t * L.Hq + h) * D; };

    // one absorption of token j into S (registers), as in the forward
    auto absorb = [&](float* S, int64_t j) {
        if (tid < D) {
            kv_s[tid] = row_h(kh, start + j, L.Hkv, kv)[tid];
            vv_s[tid] = row_h(vh, start + j, L.Hkv, kv)[tid];
        }
        __syncthreads();
        const float a = expf(g[(size_t)(start + j) * L.Hq + h]), b = beta[(size_t)(start + j) * L.Hq + h];
        float x = 0.f;
#pragma unroll
        for (int i = 0; i < Q; ++i) x = fmaf(kv_s[part * Q + i], S[i], x);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        const float u = gla ? vv_s[col] : b * (vv_s[col] - a * x);
#pragma unroll
        for (int i = 0; i < Q; ++i) S[i] = fmaf(a, S[i], kv_s[part * Q + i] * u);
        __syncthreads();
    };

    // ---- forward: checkpoints and lambda's partial sum (sum_p dO_p . o_lin,p)
    float S[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) S[i] = 0.f;
    float dl = 0.f;
    int64_t k_abs = 0;
    if (L.flags & HLA_FLAG_LINEAR_OFF) {  // o does not depend on the linear branch
        if (tid == 0) dlam_part[(size_t)n * L.Hq + h] = 0.f;
        return;
    }
#pragma unroll
    for (int i = 0; i < Q; ++i) ck(0)[st_idx<D>(i, col, part)] = 0.f;
    for (int64_t p = 0; p < len; ++p) {
        if (p - W >= ns) {
            absorb(S, p - W);
            ++k_abs;
            if (k_abs % kCk == 0) {
#pragma unroll
                for (int i = 0; i < Q; ++i) ck(k_abs / kCk)[st_idx<D>(i, col, part)] = S[i];
            }
        }
        if (k_abs > 0) {
            if (tid < D) qv_s[tid] = row_h(qh, start + p, L.Hq, h)[tid];
            __syncthreads();
            float o = 0.f;
#pragma unroll
            for (int i = 0; i < Q; ++i) o = fmaf(qv_s[part * Q + i], S[i], o);
            o += __shfl_xor_sync(0xffffffffu, o, 1);
            o += __shfl_xor_sync(0xffffffffu, o, 2);
            if (part == 0) dl = fmaf(to_f32(dout[((size_t)(start + p) * L.Hq + h) * D + col]), o, dl);
            __syncthreads();
        }
    }
    dl = cta_sum_f(dl, red);
    if (tid == 0) dlam_part[(size_t)n * L.Hq + h] = dl;

    // ---- reverse pass
    float dS[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) dS[i] = 0.f;
    int64_t seg = -1;  // segment whose states S_{seg K} .. S_{seg K + K} are in scratch
    auto load_state = [&](int64_t m, float* dst) {
        const float* src = my_scratch + (size_t)(m - seg * kCk) * DD;
#pragma unroll
        for (int i = 0; i < Q; ++i) dst[i] = src[st_idx<D>(i, col, part)];
    };
    for (int64_t p = len - 1; p >= 0; --p) {
        const int64_t kp = min(n_abs, max((int64_t)0, p - W - ns + 1));  // absorptions up to position p
        const bool here = p - W >= ns;                                   // token p - W absorbed at p
        if (kp == 0) continue;  // the read-out sees the empty state: no gradient flows
        const int64_t lowest = here ? kp - 1 : kp;
        const int64_t s = lowest / kCk;
        if (s != seg) {  // recompute S_{s K} .. S_{s K + K} from the checkpoint
            seg = s;
            float R[Q];
#pragma unroll
            for (int i = 0; i < Q; ++i) R[i] = ck(s)[st_idx<D>(i, col, part)];
#pragma unroll
            for (int i = 0; i < Q; ++i) my_scratch[st_idx<D>(i, col, part)] = R[i];
            for (int64_t m = s * kCk; m < min(n_abs, s * kCk + kCk); ++m) {
                absorb(R, ns + m);
#pragma unroll
                for (int i = 0; i < Q; ++i) my_scratch[(size_t)(m + 1 - s * kCk) * DD + st_idx<D>(i, col, part)] = R[i];
            }
            __syncthreads();
        }
        // read-out at p: o_lin = S_kp^T qhat_p
        float Sc[Q];
        load_state(kp, Sc);
        if (tid < D) {
            qv_s[tid] = row_h(qh, start + p, L.Hq, h)[tid];
            do_s[tid] = lam * to_f32(dout[((size_t)(start + p) * L.Hq + h) * D + tid]);
        }
        __syncthreads();
        {
            float val[Q];
#pragma unroll
            for (int i = 0; i < Q; ++i) val[i] = Sc[i] * do_s[col];
            row_reduce<D>(val, red_s, out_s);  // dqhat_p = S_kp dO_lin
            if (tid < D) out_row(dqh, start + p)[tid] = out_s[tid];
#pragma unroll
            for (int i = 0; i < Q; ++i) dS[i] = fmaf(qv_s[part * Q + i], do_s[col], dS[i]);
        }
        __syncthreads();  // qv_s, do_s are rewritten next
        if (!here) continue;
        // absorption of token j = p - W, from S_prev = S_{kp - 1}
        const int64_t j = p - W;
        float Sp[Q];
        load_state(kp - 1, Sp);
        if (tid < D) {
            kv_s[tid] = row_h(kh, start + j, L.Hkv, kv)[tid];
            vv_s[tid] = row_h(vh, start + j, L.Hkv, kv)[tid];
        }
        __syncthreads();
        const float a = expf(g[(size_t)(start + j) * L.Hq + h]), b = beta[(size_t)(start + j) * L.Hq + h];
        float x = 0.f, du = 0.f, gs = 0.f;
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            x = fmaf(kv_s[part * Q + i], Sp[i], x);
            du = fmaf(kv_s[part * Q + i], dS[i], du);
            gs = fmaf(dS[i], Sp[i], gs);
        }
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        du += __shfl_xor_sync(0xffffffffu, du, 1);
        du += __shfl_xor_sync(0xffffffffu, du, 2);
        const float u = gla ? vv_s[col] : b * (vv_s[col] - a * x);
        // dv, dbeta, dalpha
        if (part == 0) out_row(dvh_h, start + j)[col] = gla ? du : b * du;
        const float dbp = part == 0 && !gla ? du * (vv_s[col] - a * x) : 0.f;
        const float dap = gs + (part == 0 && !gla ? -b * du * x : 0.f);
        const float db = cta_sum_f(dbp, red);
        const float da = cta_sum_f(dap, red);
        if (tid == 0) {
            dbeta[(size_t)(start + j) * L.Hq + h] = db;
            dg[(size_t)(start + j) * L.Hq + h] = da * a;
        }
        // dk = dS u - a b S_prev du (GLA: dS v)
        {
            float val[Q];
#pragma unroll
            for (int i = 0; i < Q; ++i) val[i] = gla ? dS[i] * u : fmaf(dS[i], u, -a * b * Sp[i] * du);
            row_reduce<D>(val, red_s, out_s);
            if (tid < D) out_row(dkh_h, start + j)[tid] = out_s[tid];
        }
        // dS_prev = a dS - a b k du^T (GLA: a dS)
#pragma unroll
        for (int i = 0; i < Q; ++i) dS[i] = gla ? a * dS[i] : a * fmaf(-b * kv_s[part * Q + i], du, dS[i]);
        __syncthreads();
    }
}

// ---- 4. softmax backward, per (q-head, sequence)
constexpr int kSmT = 256;

template <typename Tin>
__global__ void __launch_bounds__(kSmT)
bwd_softmax_kernel(LayerDims L, const Tin* __restrict__ v, const Tin* __restrict__ dout,
                   const int32_t* __restrict__ cu, const float* __restrict__ qr, const float* __restrict__ kr,
                   float* __restrict__ stats, float* __restrict__ dqr, float* __restrict__ dkr_h,
                   float* __restrict__ dv_h) {
    __shared__ float red[32];
    __shared__ float ws_s[kSmT], wp_s[kSmT];
    __shared__ int64_t pq_s[kSmT];
    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G, tid = threadIdx.x, D = L.d;
    const int ns = L.n_sinks, W = L.window;
    const float scale = rsqrtf((float)D);
    const bool sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    auto qrow = [&](int64_t p) { return qr + ((size_t)(start + p) * L.Hq + h) * D; };
    auto krow = [&](int64_t j) { return kr + ((size_t)(start + j) * L.Hkv + kv) * D; };
    auto vrow = [&](int64_t j) { return v + ((size_t)(start + j) * L.Hkv + kv) * D; };
    auto drow = [&](int64_t p) { return dout + ((size_t)(start + p) * L.Hq + h) * D; };
    auto logit = [&](int64_t p, int64_t j) {
        const float* a = qrow(p);
        const float* b = krow(j);
        float s = 0.f;
        for (int c = 0; c < D; ++c) s = fmaf(a[c], b[c], s);
        return s * scale;
    };
    auto dpv = [&](int64_t p, int64_t j) {
        const Tin* a = drow(p);
        const Tin* b = vrow(j);
        float s = 0.f;
        for (int c = 0; c < D; ++c) s = fmaf(to_f32(a[c]), to_f32(b[c]), s);
        return s;
    };
    // keys visible from p: e < nsk are sinks 0..nsk-1, then the window from wlo
    auto nsk_of = [&](int64_t p) { return min((int64_t)ns, p + 1); };
    auto wlo_of = [&](int64_t p) { return max((int64_t)ns, p - W + 1); };
    // ---- per query: max, sum, D = sum_j P dP; dqr = scale sum_j P (dP - D) kr_j
    for (int64_t p = 0; p < len; ++p) {
        const int64_t nsk = nsk_of(p), wlo = wlo_of(p);
        const int64_t nk = nsk + max((int64_t)0, p + 1 - wlo);
        auto key = [&](int64_t e) { return e < nsk ? e : wlo + (e - nsk); };
        float mx = -INFINITY;
        for (int64_t e = tid; e < nk; e += kSmT) mx = fmaxf(mx, logit(p, key(e)));
        mx = cta_max_f(mx, red);
        float se = 0.f, sd = 0.f;
        for (int64_t e = tid; e < nk; e += kSmT) {
            const float w = expf(logit(p, key(e)) - mx);
            se += w;
            sd = fmaf(w, dpv(p, key(e)), sd);
        }
        se = cta_sum_f(se, red);
        const float Dp = cta_sum_f(sd, red) / se;
        if (tid == 0) {
            stats[((size_t)(start + p) * L.Hq + h) * 3 + 0] = mx;
            stats[((size_t)(start + p) * L.Hq + h) * 3 + 1] = se;
            stats[((size_t)(start + p) * L.Hq + h) * 3 + 2] = Dp;
        }
        // dqr: channel-parallel over the keys in chunks of kSmT (weights first)
        float acc = 0.f;  // channel tid (tid < D)
        for (int64_t e0 = 0; e0 < nk; e0 += kSmT) {
            const int64_t e = e0 + tid;
            if (e < nk) {
                const int64_t j = key(e);
                const float P = expf(logit(p, j) - mx) / se;
                ws_s[tid] = sm_on ? P * (dpv(p, j) - Dp) : 0.f;
                pq_s[tid] = j;
            }
            __syncthreads();
            const int cnt = (int)min((int64_t)kSmT, nk - e0);
            if (tid < D)
                for (int i = 0; i < cnt; ++i) acc = fmaf(ws_s[i], krow(pq_s[i])[tid], acc);
            __syncthreads();
        }
        if (tid < D) dqr[((size_t)(start + p) * L.Hq + h) * D + tid] = acc * scale;
    }
    __syncthreads();
    // ---- per key j: the queries that see it (all later ones for a sink, else p in [j, j + W - 1])
    for (int64_t j = 0; j < len; ++j) {
        const int64_t q_hi = j < ns ? len : min(len, j + W);
        float akr = 0.f, av = 0.f;  // channel tid
        for (int64_t p0 = j; p0 < q_hi; p0 += kSmT) {
            const int64_t p = p0 + tid;
            if (p < q_hi) {
                const size_t si = ((size_t)(start + p) * L.Hq + h) * 3;
                const float P = expf(logit(p, j) - stats[si]) / stats[si + 1];
                ws_s[tid] = sm_on ? P * (dpv(p, j) - stats[si + 2]) : 0.f;
                wp_s[tid] = sm_on ? P : 0.f;
                pq_s[tid] = p;
            }
            __syncthreads();
            const int cnt = (int)min((int64_t)kSmT, q_hi - p0);
            if (tid < D)
                for (int i = 0; i < cnt; ++i) {
                    akr = fmaf(ws_s[i], qrow(pq_s[i])[tid], akr);
                    av = fmaf(wp_s[i], to_f32(drow(pq_s[i])[tid]), av);
                }
            __syncthreads();
        }
        if (tid < D) {
            dkr_h[((size_t)(start + j) * L.Hq + h) * D + tid] = akr * scale;
            dv_h[((size_t)(start + j) * L.Hq + h) * D + tid] = av;
        }
    }
}

// ---- 5. feature backward: rows r < Hq are q-heads, < Hq + Hkv k-heads, else v-heads; thread per channel.
// First the L2 backward into d(pre-norm) (kind-specific inputs), written over dpre; the conv and RoPE
// backward then run in bwd_feat_out_kernel.
__global__ void bwd_l2_kernel(LayerDims L, const int32_t* __restrict__ cu, const float* __restrict__ qt,
                              const float* __restrict__ kt, const float* __restrict__ dqh,
                              const float* __restrict__ dkh_h, const float* __restrict__ dvh_h,
                              float* __restrict__ dqt, float* __restrict__ dkt, float* __restrict__ dvt) {
    __shared__ float red[32];
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    if (kind == 2) {  // vhat = conv(v): the per-head gradients of the group summed
        float s = 0.f;
        for (int gq = 0; gq < L.G; ++gq) s += dvh_h[((size_t)t * L.Hq + hh * L.G + gq) * D + c];
        dvt[((size_t)t * L.Hkv + hh) * D + c] = s;
        return;
    }
    float dyh;
    const float* pre;
    if (kind == 0) {
        dyh = dqh[((size_t)t * L.Hq + hh) * D + c];
        pre = qt + ((size_t)t * L.Hq + hh) * D;
    } else {
        dyh = 0.f;
        for (int gq = 0; gq < L.G; ++gq) dyh += dkh_h[((size_t)t * L.Hq + hh * L.G + gq) * D + c];
        pre = kt + ((size_t)t * L.Hkv + hh) * D;
    }
    const bool norm = kind == 1 || (L.flags & HLA_FLAG_L2NORM_Q);
    float dx = dyh;
    if (norm) {  // y = x / nrm, nrm = sqrt(|x|^2 + eps): dx = (dy - x (x . dy) / nrm^2) / nrm
        const float x = pre[c];
        const float n2 = cta_sum_f(x * x, red) + 1e-6f;
        const float xd = cta_sum_f(x * dyh, red);
        dx = (dyh - x * xd / n2) * rsqrtf(n2);
    }
    (kind == 0 ? dqt : dkt)[((size_t)t * (kind == 0 ? L.Hq : L.Hkv) + hh) * D + c] = dx;
}

// conv backward (the taps that read position p, from the later positions of the same sequence),
// plus the softmax branch's gradient, then RoPE's transpose; writes dq, dk, dv
__global__ void bwd_feat_out_kernel(LayerDims L, const int32_t* __restrict__ cu, const float* __restrict__ wq,
                                    const float* __restrict__ wk, const float* __restrict__ wv,
                                    const float* __restrict__ dqt, const float* __restrict__ dkt,
                                    const float* __restrict__ dvt, const float* __restrict__ dqr_sm,
                                    const float* __restrict__ dkr_h, const float* __restrict__ dv_h,
                                    float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv) {
    __shared__ float gx[128];
    const int64_t t = blockIdx.x;
    const int r = blockIdx.y, c = threadIdx.x, D = L.d, half = D / 2;
    const int n = seq_of_token(cu, L.n_seqs, t);
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t p = t - start;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* w = (kind == 0 ? wq : kind == 1 ? wk : wv) + ((size_t)hh * D + c) * kConvWidth;
    const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
    // x_p feeds y_{p + 7 - m} through tap m
    float acc = 0.f;
    for (int m = 0; m < kConvWidth; ++m) {
        const int64_t pp = p + (kConvWidth - 1) - m;
        if (pp >= len) continue;
        acc = fmaf(w[m], dy[((size_t)(start + pp) * H + hh) * D + c], acc);
    }
    // the softmax branch's gradient of the RoPE'd row (q, k) or of raw v, summed over the group for k, v
    if (kind == 0) {
        acc += dqr_sm[((size_t)t * L.Hq + hh) * D + c];
    } else {
        for (int gq = 0; gq < L.G; ++gq) acc += (kind == 1 ? dkr_h : dv_h)[((size_t)t * L.Hq + hh * L.G + gq) * D + c];
    }
    if (kind == 2) {
        dv[((size_t)t * L.Hkv + hh) * D + c] = acc;
        return;
    }
    // RoPE's transpose: rotate the pair (i, i + D/2) back by the angle p theta_i
    gx[c] = acc;
    __syncthreads();
    const int i = c % half;
    float cs, sn;
    rope_cs_exact(p, L.theta[i], &cs, &sn);
    const float g1 = gx[i], g2 = gx[i + half];
    (kind == 0 ? dq : dk)[((size_t)t * H + hh) * D + c] = c < half ? g1 * cs + g2 * sn : g2 * cs - g1 * sn;
}

// ---- 6. conv filters: partial sums over a block of kWB tokens, per (row, channel, tap); then the blocks
template <typename Tin>
__global__ void bwd_convw_part_kernel(LayerDims L, const Tin* __restrict__ v, const int32_t* __restrict__ cu,
                                      const float* __restrict__ qr, const float* __restrict__ kr,
                                      const float* __restrict__ dqt, const float* __restrict__ dkt,
                                      const float* __restrict__ dvt, float* __restrict__ part) {
    const int blk = blockIdx.x, r = blockIdx.y, c = threadIdx.x, D = L.d;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    const int H = kind == 0 ? L.Hq : L.Hkv;
    const float* dy = kind == 0 ? dqt : kind == 1 ? dkt : dvt;
    float acc[kConvWidth];
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) acc[m] = 0.f;
    const int64_t t0 = (int64_t)blk * kWB, t1 = min(L.total, t0 + kWB);
    for (int64_t t = t0; t < t1; ++t) {
        const int n = seq_of_token(cu, L.n_seqs, t);
        int64_t start, len;
        seq_range(cu, n, L.total, &start, &len);
        const int64_t p = t - start;
        const float d_y = dy[((size_t)t * H + hh) * D + c];
#pragma unroll
        for (int m = 0; m < kConvWidth; ++m) {
            const int64_t pp = p - (kConvWidth - 1) + m;
            if (pp < 0) continue;
            const size_t row = ((size_t)(start + pp) * H + hh) * D + c;
            const float x = kind == 0 ? qr[row] : kind == 1 ? kr[row] : to_f32(v[row]);
            acc[m] = fmaf(d_y, x, acc[m]);
        }
    }
    const int rows = L.Hq + 2 * L.Hkv;
#pragma unroll
    for (int m = 0; m < kConvWidth; ++m) part[(((size_t)blk * rows + r) * D + c) * kConvWidth + m] = acc[m];
}

__global__ void bwd_convw_sum_kernel(LayerDims L, int n_blocks, const float* __restrict__ part,
                                     float* __restrict__ dwq, float* __restrict__ dwk, float* __restrict__ dwv) {
    const int r = blockIdx.x, c = threadIdx.x, D = L.d, rows = L.Hq + 2 * L.Hkv;
    const int kind = r < L.Hq ? 0 : (r < L.Hq + L.Hkv ? 1 : 2);
    const int hh = kind == 0 ? r : (kind == 1 ? r - L.Hq : r - L.Hq - L.Hkv);
    float* dw = (kind == 0 ? dwq : kind == 1 ? dwk : dwv) + ((size_t)hh * D + c) * kConvWidth;
    for (int m = 0; m < kConvWidth; ++m) {
        float s = 0.f;
        for (int b = 0; b < n_blocks; ++b) s += part[(((size_t)b * rows + r) * D + c) * kConvWidth + m];
        dw[m] = s;
    }
}

// ---- 7. lambda: partial sums over the sequences
__global__ void bwd_lambda_kernel(LayerDims L, const float* __restrict__ part, float* __restrict__ dlam) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= L.Hq) return;
    float s = 0.f;
    for (int n = 0; n < L.n_seqs; ++n) s += part[(size_t)n * L.Hq + h];
    dlam[h] = s;
}

}  // namespace

BwdLayout bwd_layout(const LayerDims& L) {
    BwdLayout b;
    const size_t T = (size_t)L.total, Hq = (size_t)L.Hq, Hkv = (size_t)L.Hkv, D = (size_t)L.d, N = (size_t)L.n_seqs;
    const size_t slots = T / kCk + N + 1, rows = Hq + 2 * Hkv, nblk = (T + kWB - 1) / kWB;
    size_t off = 256;  // bytes 0..15: the device error word
    b.err = 0;
    auto take = [&](size_t floats) {
        const size_t o = off;
        off = (off + floats * sizeof(float) + 255) / 256 * 256;
        return o;
    };
    b.qr = take(T * Hq * D);
    b.kr = take(T * Hkv * D);
    b.qt = take(T * Hq * D);
    b.qh = take(T * Hq * D);
    b.kt = take(T * Hkv * D);
    b.kh = take(T * Hkv * D);
    b.vh = take(T * Hkv * D);
    b.dqh = take(T * Hq * D);
    b.dkh_h = take(T * Hq * D);
    b.dvh_h = take(T * Hq * D);
    b.dqr_sm = take(T * Hq * D);
    b.dkr_h = take(T * Hq * D);
    b.dv_h = take(T * Hq * D);
    b.dqt = take(T * Hq * D);
    b.dkt = take(T * Hkv * D);
    b.dvt = take(T * Hkv * D);
    b.stats = take(T * Hq * 3);
    b.ckpt = take(slots * Hq * D * D);
    b.scratch = take(N * Hq * (kCk + 1) * D * D);
    b.dlam_part = take(N * Hq);
    b.convw_part = take(nblk * rows * D * kConvWidth);
    b.n_blocks = (int)nblk;
    b.total = off;
    return b;
}

template <typename Tin>
cudaError_t launch_backward(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* g,
                            const float* beta, const float* lambda, const float* wq, const float* wk, const float* wv,
                            const int32_t* cu, const Tin* dout, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, float* dlam, float* dwq, float* dwk, float* dwv, char* ws,
                            const BwdLayout& b, cudaStream_t st) {
    auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const size_t T = (size_t)L.total;
    const int D = L.d, rows = L.Hq + 2 * L.Hkv;
    cudaError_t e;
    // tokens that no state absorbs keep zero gradients of g, beta, khat, vhat
    if ((e = cudaMemsetAsync(dg, 0, T * L.Hq * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dbeta, 0, T * L.Hq * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(F(b.dkh_h), 0, T * L.Hq * D * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(F(b.dvh_h), 0, T * L.Hq * D * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(F(b.dqh), 0, T * L.Hq * D * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(ws + b.err, 0, 16, st)) != cudaSuccess) return e;
    bwd_rope_kernel<Tin><<<dim3((unsigned)T, L.Hq + L.Hkv), D, 0, st>>>(L, q, k, cu, F(b.qr), F(b.kr),
                                                                        reinterpret_cast<int32_t*>(ws + b.err));
    bwd_conv_kernel<Tin><<<dim3((unsigned)T, rows), D, 0, st>>>(L, v, wq, wk, wv, cu, F(b.qr), F(b.kr), F(b.qt), F(b.qh),
                                                                F(b.kt), F(b.kh), F(b.vh));
    if (D == 128)
        bwd_gdn_kernel<Tin, 128><<<dim3(L.Hq, L.n_seqs), 128 * kParts, 0, st>>>(
            L, g, beta, lambda, dout, cu, F(b.qh), F(b.kh), F(b.vh), F(b.ckpt), F(b.scratch), F(b.dqh), F(b.dkh_h),
            F(b.dvh_h), dg, dbeta, F(b.dlam_part));
    else
        bwd_gdn_kernel<Tin, 64><<<dim3(L.Hq, L.n_seqs), 64 * kParts, 0, st>>>(
            L, g, beta, lambda, dout, cu, F(b.qh), F(b.kh), F(b.vh), F(b.ckpt), F(b.scratch), F(b.dqh), F(b.dkh_h),
            F(b.dvh_h), dg, dbeta, F(b.dlam_part));
    bwd_softmax_kernel<Tin><<<dim3(L.Hq, L.n_seqs), kSmT, 0, st>>>(L, v, dout, cu, F(b.qr), F(b.kr), F(b.stats),
                                                                    F(b.dqr_sm), F(b.dkr_h), F(b.dv_h));
    bwd_l2_kernel<<<dim3((unsigned)T, rows), D, 0, st>>>(L, cu, F(b.qt), F(b.kt), F(b.dqh), F(b.dkh_h), F(b.dvh_h),
                                                         F(b.dqt), F(b.dkt), F(b.dvt));
    bwd_feat_out_kernel<<<dim3((unsigned)T, rows), D, 0, st>>>(L, cu, wq, wk, wv, F(b.dqt), F(b.dkt), F(b.dvt),
                                                               F(b.dqr_sm), F(b.dkr_h), F(b.dv_h), dq, dk, dv);
    bwd_convw_part_kernel<Tin><<<dim3(b.n_blocks, rows), D, 0, st>>>(L, v, cu, F(b.qr), F(b.kr), F(b.dqt), F(b.dkt),
                                                                      F(b.dvt), F(b.convw_part));
    bwd_convw_sum_kernel<<<rows, D, 0, st>>>(L, b.n_blocks, F(b.convw_part), dwq, dwk, dwv);
    bwd_lambda_kernel<<<(L.Hq + 127) / 128, 128, 0, st>>>(L, F(b.dlam_part), dlam);
    return cudaGetLastError();
}

template cudaError_t launch_backward<float>(const LayerDims&, const float*, const float*, const float*, const float*,
                                            const float*, const float*, const float*, const float*, const float*,
                                            const int32_t*, const float*, float*, float*, float*, float*, float*,
                                            float*, float*, float*, float*, char*, const BwdLayout&, cudaStream_t);
template cudaError_t launch_backward<__nv_bfloat16>(const LayerDims&, const __nv_bfloat16*, const __nv_bfloat16*,
                                                    const __nv_bfloat16*, const float*, const float*, const float*,
                                                    const float*, const float*, const float*, const int32_t*,
                                                    const __nv_bfloat16*, float*, float*, float*, float*, float*,
                                                    float*, float*, float*, float*, char*, const BwdLayout&,
                                                    cudaStream_t);

}  // namespace hla
