// Exact branch on the tcgen05 tensor cores: softmax over the sink tokens plus
// the sliding window ("迈向线性的关键：分析驱动的 Transformer 线性化", section
// 填补近似缺口的实用设计; scale 1/sqrt(d) from Lemma 1 of section
// 从 softmax 到 delta 规则的一阶近似), with the lambda-weighted linear branch
// added in the epilogue ("Untangling Component Imbalance in Hybrid Linear
// Attention Conversion", section 关键设计 (1)).
//
// One CTA of 256 threads per (kv head, block of QB = 256 / G query positions):
// the G query heads of the kv group are stacked into 256 rows, two M = 128
// halves.  The keys a block can see are gathered as [sinks | window span]
// into groups of 128 key slots; per group:
//   D_S[half] = Q_half K^T            (tcgen05, fp16 operands, fp32 in TMEM)
//   masked softmax, one thread per row, P (fp16) -> shared memory
//   D_O[half] (+)= P_half V           (tcgen05)
// with a running max and sum per row; when a block needs more than one group
// the accumulated output is rescaled in TMEM before the next P V.  For the
// 8 + 56 budget every block's keys fit one group.  A block that straddles a
// sequence boundary is processed one sequence segment at a time.
#include "hla_common.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kD = 128;
constexpr int kRows = 256;
constexpr int kThreads = 256;
constexpr int kKeys = 128;  // key slots per group
constexpr uint32_t kWaitLimit = 1u << 22;

constexpr uint32_t kQ = 0;          // two halves, 128 x 128 fp16 K-major each
constexpr uint32_t kK = 65536;      // 128 keys x 128 fp16 K-major
constexpr uint32_t kV = 98304;      // 128 keys x 128 fp16 MN-major
constexpr uint32_t kP = 131072;     // two halves, 128 rows x 128 keys fp16 K-major
constexpr uint32_t kMisc = 196608;  // mbarrier, TMEM slot
constexpr uint32_t kSmemAlloc = kMisc + 64 + 1024;

constexpr uint32_t kColS = 0, kColO = 256, kTmemCols = 512;

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        o[i] = pack_h2(f.x, f.y);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 16-byte global -> shared copy that bypasses registers; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(unsigned char* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(umma::smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}

// Key position held by key slot i of a segment: the sinks first, then the window span.
__device__ __forceinline__ int64_t key_at(int64_t i, int64_t n_sink, int64_t span_lo, int64_t n_keys) {
    if (i >= n_keys) return -1;
    return i < n_sink ? i : span_lo + (i - n_sink);
}

__global__ void __launch_bounds__(kThreads, 1)
window_softmax_tc_kernel(LayerDims L, const __half* __restrict__ qr, const __half* __restrict__ kr,
                         const __nv_bfloat16* __restrict__ v, const float* __restrict__ o_lin,
                         const float* __restrict__ lambda, const int32_t* __restrict__ cu,
                         __nv_bfloat16* __restrict__ out, int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* mbar_p = reinterpret_cast<uint64_t*>(sm + kMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, half = warp >> 2;
    const int Lr = ((warp & 3) << 5) + lane;
    const int row = half * 128 + Lr;
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    const int G = L.G, QB = kRows / G;
    const int kv = blockIdx.y;
    const int g = row / QB, qi = row % QB, h = kv * G + g;
    const int64_t t0 = (int64_t)blockIdx.x * QB;
    const uint32_t sbase = umma::smem_addr(sm);
    const uint32_t mbar = umma::smem_addr(mbar_p);
    const float qscale = 0.088388347648318447f * 1.4426950408889634f;  // 1/sqrt(128) * log2(e)

    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t srow = tmem + lane_base + kColS + 128 * half;
    const uint32_t orow = tmem + lane_base + kColO + 128 * half;
    uint32_t phase = 0;
    bool ok = true;

    auto wait_mma = [&]() {
        bool done = umma::mbar_wait(mbar, phase, kWaitLimit);
        phase ^= 1u;
        if (!done && err) atomicExch(err, kErrTimeout);
        umma::fence_after_sync();
        return __syncthreads_or(!done) == 0;
    };

    const int64_t t_end = min(t0 + QB, L.total);
    int64_t ta = t0;
    while (ta < t_end && ok) {
        // ---- the part of this block that lies in one sequence
        const int s = seq_of_token(cu, L.n_seqs, ta);
        int64_t start, len;
        seq_range(cu, s, L.total, &start, &len);
        if (ta < start || ta >= start + len) break;  // malformed table: flagged by the feature pass
        const int64_t tb = min(t_end, start + len);
        const int64_t pa = ta - start, pb = tb - start;  // query positions [pa, pb)
        const int64_t n_sink = min((int64_t)L.n_sinks, pb);
        const int64_t span_lo = max((int64_t)L.n_sinks, pa - L.window + 1);
        const int64_t n_span = pb > span_lo ? pb - span_lo : 0;
        const int64_t n_keys = n_sink + n_span;
        const int n_groups = (int)((n_keys + kKeys - 1) / kKeys);

        // this thread's row: query position p (valid when row_on); the key slots
        // it sees form two ranges, [0, hi1) (sinks) and [lo2, hi2) (window)
        const int64_t t_row = t0 + qi;
        const bool row_on = t_row >= ta && t_row < tb;
        const int64_t p = row_on ? t_row - start : -1;
        int hi1 = 0, lo2 = 0, hi2 = 0;
        if (row_on) {
            hi1 = (int)min(n_sink, p + 1);
            lo2 = (int)(n_sink + max((int64_t)0, p - L.window + 1 - span_lo));
            hi2 = (int)(p >= span_lo ? n_sink + (p - span_lo) + 1 : lo2);
        }

        // ---- Q rows of the block (zero outside the segment), streamed with cp.async
#pragma unroll
        for (int u = 0; u < kRows * 16 / kThreads; ++u) {
            const int e = tid + kThreads * u, r = e >> 4, cc = (e & 15) * 8;
            const int rg = r / QB, rq = r % QB;
            const int64_t t = t0 + rq;
            const bool in = t >= ta && t < tb;
            cp_async16(sm + kQ + (r >> 7) * 32768 + umma::sw128_offset(r & 127, cc, 128),
                       qr + ((size_t)(in ? t : ta) * L.Hq + kv * G + rg) * kD + cc, in ? 16u : 0u);
        }

        float m_run = -INFINITY, l_run = 0.f;
        for (int grp = 0; grp < n_groups; ++grp) {
            // ---- K (fp16) and V (bf16 -> fp16) rows of the group's key slots
#pragma unroll
            for (int u = 0; u < kKeys * 16 / kThreads; ++u) {
                const int e = tid + kThreads * u, slot = e >> 4, cc = (e & 15) * 8;
                const int64_t j = key_at((int64_t)grp * kKeys + slot, n_sink, span_lo, n_keys);
                const size_t rowi = ((size_t)(start + (j >= 0 ? j : 0)) * L.Hkv + kv) * kD + cc;
                const uint32_t off = umma::sw128_offset(slot, cc, 128);
                cp_async16(sm + kK + off, kr + rowi, j >= 0 ? 16u : 0u);
                cp_async16(sm + kV + off, v + rowi, j >= 0 ? 16u : 0u);
            }
            cp_async_wait_all();  // (Q rows too, on the first group)
            // values arrive as bf16; the MMA takes fp16 for both operands
#pragma unroll
            for (int u = 0; u < kKeys * 16 / kThreads; ++u) {
                const int e = tid + kThreads * u, slot = e >> 4, cc = (e & 15) * 8;
                uint4* pv = reinterpret_cast<uint4*>(sm + kV + umma::sw128_offset(slot, cc, 128));
                *pv = bf16x8_to_f16x8(*pv);
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            __syncthreads();

            // ---- D_S = Q K^T for both halves
            if (tid == 0) {
                umma::fence_after_sync();
                const uint32_t id = umma::idesc_f16(128, kKeys, false, false, false);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int s16 = 0; s16 < kD / 16; ++s16)
                        umma::mma(tmem + kColS + 128 * hh, umma::kmajor(sbase + kQ + 32768 * hh, 128, s16),
                                  umma::kmajor(sbase + kK, 128, s16), id, s16 > 0);
                umma::commit(mbar);
            }
            if (!(ok = wait_mma())) break;

            // ---- masked softmax of this row (two passes over TMEM, 32 columns at a time)
            float mg = -INFINITY;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float sc[32];
                umma::tmem_ld32(srow + 32 * q4, sc);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int gi = grp * kKeys + 32 * q4 + i;
                    if (gi < hi1 || (gi >= lo2 && gi < hi2)) mg = fmaxf(mg, sc[i] * qscale);
                }
            }
            const float m_new = fmaxf(m_run, mg);
            const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
            float lsum = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float sc[32];
                umma::tmem_ld32(srow + 32 * q4, sc);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int gi = grp * kKeys + 32 * q4 + i;
                    const bool vis = gi < hi1 || (gi >= lo2 && gi < hi2);
                    sc[i] = vis ? exp2f(sc[i] * qscale - m_new) : 0.f;
                    lsum += sc[i];
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const float* x = sc + 8 * c8;
                    const uint4 pk = make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]),
                                                pack_h2(x[6], x[7]));
                    *reinterpret_cast<uint4*>(sm + kP + 32768 * half +
                                              umma::sw128_offset(Lr, 32 * q4 + 8 * c8, 128)) = pk;
                }
            }
            l_run = l_run * corr + lsum;
            m_run = m_new;
            if (grp > 0) {  // rescale the output accumulated over the earlier groups
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float o[32];
                    umma::tmem_ld32(orow + 32 * q4, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= corr;
                    umma::tmem_st32(orow + 32 * q4, o);
                }
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            __syncthreads();

            // ---- D_O (+)= P V for both halves
            if (tid == 0) {
                umma::fence_after_sync();
                const uint32_t id = umma::idesc_f16(128, kD, false, true, false);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int s16 = 0; s16 < kKeys / 16; ++s16)
                        umma::mma(tmem + kColO + 128 * hh, umma::kmajor(sbase + kP + 32768 * hh, 128, s16),
                                  umma::mnmajor(sbase + kV, 16384, s16), id, grp > 0 || s16 > 0);
                umma::commit(mbar);
            }
            if (!(ok = wait_mma())) break;
        }
        if (!ok) break;

        // ---- epilogue: o = o_sm + lambda_h o_lin for the rows of this segment
        {
            const bool sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF);
            const bool lin_on = row_on && !(L.flags & HLA_FLAG_LINEAR_OFF) && (p - L.window >= L.n_sinks);
            const float inv_l = (sm_on && row_on) ? 1.f / l_run : 0.f;
            const float lam = lin_on ? __ldg(lambda + h) : 0.f;
            const size_t base = ((size_t)(row_on ? t_row : 0) * L.Hq + h) * kD;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float o[32];
                umma::tmem_ld32(orow + 32 * q4, o);  // every warp loads; rows outside the segment drop it
                if (!row_on) continue;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float r8[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) r8[x] = o[8 * c8 + x] * inv_l;
                    const int col = 32 * q4 + 8 * c8;
                    if (lin_on) {
                        const float4 a = *reinterpret_cast<const float4*>(o_lin + base + col);
                        const float4 b = *reinterpret_cast<const float4*>(o_lin + base + col + 4);
                        r8[0] = fmaf(lam, a.x, r8[0]); r8[1] = fmaf(lam, a.y, r8[1]);
                        r8[2] = fmaf(lam, a.z, r8[2]); r8[3] = fmaf(lam, a.w, r8[3]);
                        r8[4] = fmaf(lam, b.x, r8[4]); r8[5] = fmaf(lam, b.y, r8[5]);
                        r8[6] = fmaf(lam, b.z, r8[6]); r8[7] = fmaf(lam, b.w, r8[7]);
                    }
                    uint32_t w[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        __nv_bfloat162 bb = __floats2bfloat162_rn(r8[2 * x], r8[2 * x + 1]);
                        w[x] = *reinterpret_cast<uint32_t*>(&bb);
                    }
                    *reinterpret_cast<uint4*>(out + base + col) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        umma::fence_before_sync();
        __syncthreads();  // shared tiles and TMEM are reused by the next segment
        ta = tb;
    }

    if (!ok && tid == 0) umma::mbar_wait(mbar, phase ^ 1u, kWaitLimit);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool window_softmax_tc_supported(const LayerDims& L) {
    return L.d == kD && (L.G == 1 || L.G == 2 || L.G == 4 || L.G == 8);
}

cudaError_t launch_window_softmax_tc(const LayerDims& L, const __half* qr, const __half* kr,
                                     const __nv_bfloat16* v, const float* o_lin, const float* lambda,
                                     const int32_t* cu, __nv_bfloat16* out, int32_t* err, cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(window_softmax_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int QB = kRows / L.G;
    dim3 grid((unsigned)((L.total + QB - 1) / QB), L.Hkv);
    window_softmax_tc_kernel<<<grid, kThreads, kSmemAlloc, st>>>(L, qr, kr, v, o_lin, lambda, cu, out, err);
    return cudaGetLastError();
}

}  // namespace hla
