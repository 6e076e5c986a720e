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
//
// Context-parallel form (HLA_FLAG_GDN_SCAN): the absorptions of a sequence
// are cut into parts of part_len; the state after a part is an affine map of
// the state before it, S' = P S + R, since every update is.  Three launches:
//   1. per part (all parts at once): R, the part run from S = 0, and P, the
//      part run from S = I with zero values (d x d; the part's state
//      transition);
//   2. per (sequence, q-head, 8 value columns): the scan S_{i+1} = P_i S_i +
//      R_i over the parts, giving every part its start state;
//   3. per part (all at once): the part from its start state, with the
//      read-outs; the sequence's last part writes the final state.
// Three times the work of one pass, on parts-times as many CTAs.
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

constexpr int kRecWhole = 0;  // grid (Hq, n_seqs): whole sequences from S = 0
constexpr int kRecMap = 1;    // grid (Hq, parts, 2): a part's R (z = 0) and P (z = 1) into pr; no read-outs
constexpr int kRecPart = 2;   // grid (Hq, parts): a part from its start state, with the read-outs

template <typename Tf, int D>
__global__ void __launch_bounds__(D * kRecParts)
gdn_recurrent_kernel(LayerDims L, const Tf* __restrict__ qhat, const Tf* __restrict__ khat,
                     const Tf* __restrict__ vhat, const float* __restrict__ g,
                     const float* __restrict__ beta, const int32_t* __restrict__ cu,
                     float* __restrict__ o_lin, float* __restrict__ S_out, int mode, RecScan rs) {
    constexpr int Q = D / kRecParts;           // rows of S per thread
    constexpr int ROW = kRecParts * (Q + 4);   // padded row length
    constexpr int NT = D * kRecParts;
    __shared__ __align__(16) float ks[kRecTile][ROW];
    __shared__ __align__(16) float qs[kRecTile][ROW];
    __shared__ float vs[kRecTile][D];
    __shared__ float as[kRecTile], bs[kRecTile];

    const int h = blockIdx.x, kv = h / L.G;
    const int col = threadIdx.x / kRecParts, part = threadIdx.x % kRecParts;
    const int W = L.window;
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    int n = blockIdx.y, kind = 0;
    int64_t gp = 0, ip = 0;  // global and in-sequence part index
    bool last = true;
    if (mode != kRecWhole) {
        gp = blockIdx.y;
        if (gp >= __ldg(rs.base + L.n_seqs)) return;
        int lo = 0, hi = L.n_seqs - 1;  // the sequence owning part gp
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(rs.base + mid) <= gp) lo = mid; else hi = mid - 1;
        }
        n = lo;
        ip = gp - __ldg(rs.base + n);
        last = ip == (int64_t)__ldg(rs.base + n + 1) - __ldg(rs.base + n) - 1;
        kind = mode == kRecMap ? (int)blockIdx.z : 0;
        if (mode == kRecMap && last) return;  // the scan needs no map of a sequence's last part
    }
    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    // absorbed tokens [j_lo, j_end) of this CTA
    int64_t j_lo = L.n_sinks, j_end = len - W;
    if (mode != kRecWhole) {
        j_lo = L.n_sinks + ip * rs.part_len;
        j_end = min(j_end, j_lo + rs.part_len);
    }
    const bool readout = mode != kRecMap, unit = mode == kRecMap && kind == 1;  // unit: S from I, values 0

    float S[Q];  // S[part*Q + i][col]
#pragma unroll
    for (int i = 0; i < Q; ++i) S[i] = unit && part * Q + i == col ? 1.f : 0.f;
    if (mode == kRecPart && ip > 0) {
        const float* src = rs.s_part + ((size_t)gp * L.Hq + h) * D * D;
#pragma unroll
        for (int i = 0; i < Q; ++i) S[i] = src[(size_t)(part * Q + i) * D + col];
    }

    for (int64_t jt = j_lo; jt < j_end; jt += kRecTile) {
        const int cnt = (int)min((int64_t)kRecTile, j_end - jt);
        __syncthreads();
        for (int idx = threadIdx.x; idx < cnt * D; idx += NT) {
            int r = idx / D, c = idx % D;
            size_t t = (size_t)(start + jt + r);
            ks[r][rec_pad<D>(c)] = to_f32(khat[(t * L.Hkv + kv) * D + c]);
            qs[r][rec_pad<D>(c)] = readout ? to_f32(qhat[((t + W) * L.Hq + h) * D + c]) : 0.f;
            vs[r][c] = unit ? 0.f : to_f32(vhat[(t * L.Hkv + kv) * D + c]);
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
            if (part == 0 && readout) {
                size_t t = (size_t)(start + jt + r + W);
                o_lin[(t * L.Hq + h) * D + col] = o;
            }
        }
    }
    float* dst = nullptr;
    if (mode == kRecMap)
        dst = rs.pr + (((size_t)gp * L.Hq + h) * 2 + kind) * D * D;
    else if (last && S_out)
        dst = S_out + ((size_t)n * L.Hq + h) * D * D;
    if (dst) {
#pragma unroll
        for (int i = 0; i < Q; ++i) dst[(size_t)(part * Q + i) * D + col] = S[i];
    }
}

// The scan over a sequence's parts, for 8 value columns of one q-head: S_0 = 0, S_{i+1} = P_i S_i + R_i
// (fp32, fixed order) into s_part for parts 1 ..; a sequence without parts gets S_out = 0 here.  P_{i+1}
// and the columns of R_{i+1} are copied into shared memory (cp.async) while step i computes.
constexpr int kScanThreads = 256;
template <int D> constexpr size_t scan_smem_bytes() { return (size_t)(2 * D * (D + 4) + 2 * D * 8 + D * 8) * 4; }

__device__ __forceinline__ void scan_cp16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kScanThreads)
gdn_part_scan_kernel(LayerDims L, RecScan rs, float* __restrict__ S_out) {
    constexpr int TPR = kScanThreads / D, CPT = 8 / TPR, LDP = D + 4;  // threads per row, columns per thread
    extern __shared__ __align__(16) float scan_sm[];
    float* Pb = scan_sm;                 // [2][D][LDP]
    float* Rb = Pb + 2 * D * LDP;        // [2][D][8]
    float* Ss = Rb + 2 * D * 8;          // [D][8]
    const int h = blockIdx.x / (D / 8), cg = blockIdx.x % (D / 8), n = blockIdx.y, tid = threadIdx.x;
    const int r = tid / TPR, c0 = (tid % TPR) * CPT;
    const int b0 = __ldg(rs.base + n), np = __ldg(rs.base + n + 1) - b0;
    for (int idx = tid; idx < D * 8; idx += kScanThreads) Ss[idx] = 0.f;
    if (np <= 0) {
        if (S_out) {
            float* dst = S_out + (((size_t)n * L.Hq + h) * D + r) * D + cg * 8 + c0;
#pragma unroll
            for (int c = 0; c < CPT; ++c) dst[c] = 0.f;
        }
        return;
    }
    auto fetch = [&](int i) {  // P_i and R_i's 8 columns into buffer i & 1
        const float* R = rs.pr + (((size_t)(b0 + i) * L.Hq + h) * 2 + 0) * D * D;
        const float* P = rs.pr + (((size_t)(b0 + i) * L.Hq + h) * 2 + 1) * D * D;
        float* pb = Pb + (i & 1) * D * LDP;
        float* rb = Rb + (i & 1) * D * 8;
        for (int idx = tid; idx < D * D / 4; idx += kScanThreads) {
            const int row = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
            scan_cp16(pb + row * LDP + c4, P + (size_t)row * D + c4);
        }
        for (int idx = tid; idx < D * 2; idx += kScanThreads) {
            const int row = idx / 2, c4 = (idx % 2) * 4;
            scan_cp16(rb + row * 8 + c4, R + (size_t)row * D + cg * 8 + c4);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (np > 1) fetch(0);
    for (int i = 0; i + 1 < np; ++i) {
        if (i + 2 < np) {
            fetch(i + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();  // P_i, R_i and the previous step's S are visible
        const float* pr = Pb + (i & 1) * D * LDP + r * LDP;
        const float* rb = Rb + (i & 1) * D * 8 + r * 8;
        float acc[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] = rb[c0 + c];
#pragma unroll 4
        for (int k4 = 0; k4 < D / 4; ++k4) {
            const float4 p = *reinterpret_cast<const float4*>(pr + 4 * k4);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                acc[c] = fmaf(p.x, Ss[(4 * k4 + 0) * 8 + c0 + c], acc[c]);
                acc[c] = fmaf(p.y, Ss[(4 * k4 + 1) * 8 + c0 + c], acc[c]);
                acc[c] = fmaf(p.z, Ss[(4 * k4 + 2) * 8 + c0 + c], acc[c]);
                acc[c] = fmaf(p.w, Ss[(4 * k4 + 3) * 8 + c0 + c], acc[c]);
            }
        }
        __syncthreads();  // every thread has read S_i (and this buffer) before they change
#pragma unroll
        for (int c = 0; c < CPT; ++c) Ss[r * 8 + c0 + c] = acc[c];
        float* dst = rs.s_part + ((size_t)(b0 + i + 1) * L.Hq + h) * D * D + (size_t)r * D + cg * 8 + c0;
#pragma unroll
        for (int c = 0; c < CPT; ++c) dst[c] = acc[c];
    }
}

template <typename Tf>
cudaError_t launch_gdn_recurrent(const LayerDims& L, const Tf* qhat, const Tf* khat, const Tf* vhat,
                                 const float* g, const float* beta, const int32_t* cu, float* o_lin,
                                 float* S_out, const RecScan* rs, cudaStream_t st) {
    const int D = L.d, nt = D * kRecParts;
    auto run = [&](dim3 grid, int mode) {
        const RecScan r = rs ? *rs : RecScan{};
        if (D == 128)
            gdn_recurrent_kernel<Tf, 128><<<grid, nt, 0, st>>>(L, qhat, khat, vhat, g, beta, cu, o_lin, S_out, mode, r);
        else
            gdn_recurrent_kernel<Tf, 64><<<grid, nt, 0, st>>>(L, qhat, khat, vhat, g, beta, cu, o_lin, S_out, mode, r);
    };
    if (!rs) {
        run(dim3(L.Hq, L.n_seqs), kRecWhole);
        return cudaGetLastError();
    }
    if (rs->part_len <= 0 || rs->n_parts <= 0 || rs->n_parts > 65535) return cudaErrorInvalidValue;
    run(dim3(L.Hq, rs->n_parts, 2), kRecMap);
    static DeviceCache cache;  // the scan's shared-memory attribute, per device
    cudaError_t e = device_cached(cache, nullptr, [](int, int*) {
        cudaError_t r = cudaFuncSetAttribute(gdn_part_scan_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)scan_smem_bytes<128>());
        return r == cudaSuccess ? cudaFuncSetAttribute(gdn_part_scan_kernel<64>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)scan_smem_bytes<64>())
                                : r;
    });
    if (e != cudaSuccess) return e;
    if (D == 128)
        gdn_part_scan_kernel<128><<<dim3(L.Hq * 16, L.n_seqs), kScanThreads, scan_smem_bytes<128>(), st>>>(L, *rs, S_out);
    else
        gdn_part_scan_kernel<64><<<dim3(L.Hq * 8, L.n_seqs), kScanThreads, scan_smem_bytes<64>(), st>>>(L, *rs, S_out);
    run(dim3(L.Hq, rs->n_parts), kRecPart);
    return cudaGetLastError();
}

template cudaError_t launch_gdn_recurrent<float>(const LayerDims&, const float*, const float*,
                                                 const float*, const float*, const float*,
                                                 const int32_t*, float*, float*, const RecScan*, cudaStream_t);
template cudaError_t launch_gdn_recurrent<__half>(const LayerDims&, const __half*, const __half*,
                                                  const __half*, const float*, const float*,
                                                  const int32_t*, float*, float*, const RecScan*, cudaStream_t);

}  // namespace hla
