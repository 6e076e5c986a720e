// Chunk-local part of the chunked GDN form that does not depend on the
// state: for every chunk of 64 absorbed tokens and every query head, with the
// gates cumulated inside the chunk (G_r = sum_{i<=r} g_i, gamma_r = e^{G_r}),
//   A[r,i] = beta_r e^{G_r - G_i} k_r . k_i  (i < r),   T = (I + A)^{-1},
//   P[r,i] = e^{G_r - G_i} q_r . k_i  (i <= r)
// (the UT transform of the GDN update of "迈向线性的关键：分析驱动的
// Transformer 线性化", section 线性注意力替换机制; q_r is qhat at position
// r + W).  All chunks are independent, so this runs fully parallel, ahead of
// the state-carrying kernel.  Per (chunk, q-head) it writes a record:
//   -Wm = -T diag(beta gamma) K             64 x 128 fp16 K-major 128B-swizzled
//                                          image (two 8 KB key-dim halves)
//   T diag(beta), P                        64 x 64 images of the same kind (8 KB each)
//   gamma[64], e^{G_63 - G}[64]            fp32
// which the state kernel copies into shared memory unchanged.
//
// Chunk slots: sequence s owns slots [chunk_base[s], chunk_base[s+1]); its
// chunk c covers absorbed tokens n_sinks + 64 c .. + 63.
//
// With HLA_FLAG_GLA (gated linear attention, S <- alpha S + k v^T, the other
// update of section 线性注意力替换机制) the same record serves the state
// kernel unchanged: A = 0 gives T = I, the write gain is 1 in place of beta,
// and nothing is erased, so -Wm = 0; then U = V, O = diag(gamma) Q S0 + P V
// and S1 = gamma_C S0 + (diag(e^{G_C - G}) K)^T V.
#include <algorithm>

#include "hla_common.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kC = kGdnChunk, kD = 128, kThreads = 128;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kTmemCols = 128;               // Gram (64 columns), then Wm^T (128)
constexpr uint32_t kK = 0;                        // [K ; Q] rows, K-major
constexpr uint32_t kTbg = 8192;                   // T diag(beta gamma) image, over the first query block
constexpr int kSA = 65;                           // row stride of A (odd: row-per-thread writes hit distinct banks)
constexpr uint32_t kA32 = 32768;                  // A fp32 [64][kSA]
constexpr uint32_t kT32 = kA32 + 64 * 68 * 4;     // T fp32 [64][68] (rows 16-byte aligned)
constexpr uint32_t kX32 = kT32 + 64 * 68 * 4;     // [32][36]
constexpr uint32_t kVec = kX32 + 32 * 36 * 4;     // G (log2 units), beta, gamma, 2^-G
constexpr uint32_t kMisc = kVec + 4 * 64 * 4;
constexpr uint32_t kSmemAlloc = kMisc + 64 + 1024;

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Inverse of a 32 x 32 unit lower-triangular diagonal block b of (I + A),
// one warp per block: lane l owns column l of the inverse and runs the
// forward substitution x_r = [r == l] - sum_{m < r} A[r][m] x_m in row order
// (the A entries are shared-memory broadcasts, x stays in registers; four
// partial sums per row keep the dependent chain short).  (The kernel is
// persistent, so this fully unrolled code stays in the instruction cache.)
__device__ __forceinline__ void invert_diag_block32(const float* sA, float* sT, int b, int l) {
    float x[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float* ar = sA + (32 * b + r) * kSA + 32 * b;
        float acc[4] = {r == l ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < r; ++m) acc[m & 3] = fmaf(-ar[m], x[m], acc[m & 3]);
        x[r] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) sT[(32 * b + r) * 68 + 32 * b + l] = x[r];
}

// Launched with programmatic stream serialization, this grid may run beside the one before it in the
// stream (it reads nothing that grid writes); waiting for that grid before leaving keeps "this grid is
// done" implying "the one before it is done" for whatever follows in the stream.  No effect on a plain
// launch.
__device__ __forceinline__ void grid_dependency_wait() { pdl_wait(); }

__global__ void __launch_bounds__(kThreads, 3)
gdn_inverse_kernel(LayerDims L, const __half* __restrict__ qhat, const __half* __restrict__ khat,
                   const float* __restrict__ g,
                   const float* __restrict__ beta, const int32_t* __restrict__ cu,
                   const int32_t* __restrict__ chunk_base, int slot_lo, int slot_hi,
                   int32_t* __restrict__ counter, unsigned char* __restrict__ rec_out, int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    // The state launch that follows with programmatic stream serialization may place its CTAs (each needs
    // an SM to itself) as SMs drain, and set up; it waits for this grid before its first global read.
    pdl_trigger();
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* sA = reinterpret_cast<float*>(sm + kA32);
    float* sT = reinterpret_cast<float*>(sm + kT32);
    float* sX = reinterpret_cast<float*>(sm + kX32);
    float* sG = reinterpret_cast<float*>(sm + kVec);
    float* sBeta = sG + 64;
    float* sGam = sG + 128;
    float* sEg = sG + 192;  // 2^-G_i, the column factor of e^(G_r - G_i) (see the A and P tiles)
    uint64_t* mbar_p = reinterpret_cast<uint64_t*>(sm + kMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc + 8);
    float* carry = reinterpret_cast<float*>(sm + kMisc + 16);
    volatile int* next_s = reinterpret_cast<volatile int*>(sm + kMisc + 24);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t mbar = umma::smem_addr(mbar_p), sbase = umma::smem_addr(sm);
    // GLA (no erase, write gain 1): A = 0, so T = I; beta taken as 1; Wm = 0
    const bool gla = (L.flags & HLA_FLAG_GLA) != 0;
    // items (chunk slot, q-head) of slots [slot_lo, slot_hi), taken one at a time from `counter`
    const int64_t item_lo = (int64_t)slot_lo * L.Hq;
    const int64_t item_hi = (int64_t)min(slot_hi, __ldg(chunk_base + L.n_seqs)) * L.Hq;
    if (item_lo >= item_hi) {  // whole CTA leaves together
        grid_dependency_wait();
        return;
    }

    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
    for (int i = tid; i < 32 * 32; i += kThreads) sT[(i >> 5) * 68 + 32 + (i & 31)] = 0.f;  // T01 = 0
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    uint32_t phase = 0;

    // persistent loop over (chunk slot, q-head) items, fetched dynamically so the CTAs that are
    // resident (possibly beside another kernel) share all of them
    for (;;) {
    if (tid == 0) *next_s = atomicAdd(counter, 1);
    __syncthreads();
    const int64_t item = item_lo + *next_s;
    if (item >= item_hi) break;
    const int slot = (int)(item / L.Hq), h = (int)(item % L.Hq), kv = h / L.G;
    // sequence owning the slot: the last s with chunk_base[s] <= slot
    int lo = 0, hi = L.n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(chunk_base + mid) <= slot) lo = mid; else hi = mid - 1;
    }
    const int s = lo, c = slot - __ldg(chunk_base + s);
    int64_t start, len;
    seq_range(cu, s, L.total, &start, &len);
    const int64_t j0 = L.n_sinks + (int64_t)c * kC;
    const int nv = (int)max((int64_t)0, min((int64_t)kC, len - L.window - j0));

    // ---- K rows into rows 0..63, the shifted queries into rows 64..127 (zero
    //      past the chunk), gates
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int e = tid + kThreads * u, r = e >> 4, c8 = (e & 15) * 8;
        const int rr = r & 63;
        const size_t t = (size_t)(start + j0 + (rr < nv ? rr : 0));
        const void* src = r < 64 ? (const void*)(khat + (t * L.Hkv + kv) * kD + c8)
                                 : (const void*)(qhat + ((t + L.window) * L.Hq + h) * kD + c8);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                         umma::smem_addr(sm + kK + umma::sw128_offset(r, c8, 128))),
                     "l"(src), "r"(rr < nv ? 16u : 0u)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    float gi = 0.f;
    if (tid < kC) {
        const size_t t = (size_t)(start + j0 + tid);
        gi = tid < nv ? g[t * L.Hq + h] * 1.4426950408889634f : 0.f;
        sBeta[tid] = tid < nv ? (gla ? 1.f : beta[t * L.Hq + h]) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, gi, o);
            if (lane >= o) gi += y;
        }
        if (tid == 31) *carry = gi;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    umma::fence_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (tid >= 32 && tid < kC) gi += *carry;
    if (tid < kC) {
        sG[tid] = gi;
        sEg[tid] = exp2f(-gi);
    }

    // ---- Gram: D = [K; Q] K^T
    if (tid == 0) {
        const uint32_t id = umma::idesc_f16(128, kC, false, false, false);
#pragma unroll
        for (int s16 = 0; s16 < kD / 16; ++s16)
            umma::mma(tmem, umma::kmajor(sbase + kK, 128, s16), umma::kmajor(sbase + kK, 128, s16), id, s16 > 0);
        umma::commit(mbar);
    }
    const bool done = __syncthreads_and(umma::mbar_wait(mbar, phase, kWaitLimit));  // also: sG complete
    phase ^= 1u;
    if (!done && err && tid == 0) atomicExch(err, kErrTimeout);
    umma::fence_after_sync();
    unsigned char* rec = rec_out + ((size_t)slot * L.Hq + h) * kRecordBytes;
    // both 32-column halves of this thread's Gram row in flight together, one wait
    uint32_t dg[2][32];
    if (done) {
        umma::tmem_ld32_async(tmem + ((uint32_t)(warp * 32) << 16), dg[0]);
        umma::tmem_ld32_async(tmem + ((uint32_t)(warp * 32) << 16) + 32, dg[1]);
        umma::tmem_wait_ld();
        umma::reg_fence32(dg[0]);
        umma::reg_fence32(dg[1]);
    }
    // e^(G_r - G_i) (i <= r, so at most 1): as 2^G_r 2^-G_i, one exponential per row and per column, while
    // the chunk's gates keep both factors inside fp32 (G_63 >= -100 in log2 units); else per entry.  The
    // choice is uniform over the CTA, so only one of the two forms runs.
    const bool split_exp = sG[kC - 1] >= -100.f;  // G is non-increasing
    // w[ii] = e^(G_r - G_i) for columns i = 32 half + ii
    auto weights = [&](int r, int half, float* w) {
        const float gr = sG[r];
        if (split_exp) {
            const float er = exp2f(gr);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
                const float4 e4 = *reinterpret_cast<const float4*>(sEg + 32 * half + 4 * i4);
                w[4 * i4] = er * e4.x; w[4 * i4 + 1] = er * e4.y; w[4 * i4 + 2] = er * e4.z; w[4 * i4 + 3] = er * e4.w;
            }
        } else {
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
                const float4 g4 = *reinterpret_cast<const float4*>(sG + 32 * half + 4 * i4);
                w[4 * i4] = exp2f(gr - g4.x); w[4 * i4 + 1] = exp2f(gr - g4.y);
                w[4 * i4 + 2] = exp2f(gr - g4.z); w[4 * i4 + 3] = exp2f(gr - g4.w);
            }
        }
    };
    if (warp < 2 && done) {  // rows 0..63: K K^T -> A
        const int r = tid;
        const float br = sBeta[r];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float w[32];
            weights(r, half, w);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const int i = 32 * half + ii;
                sA[r * kSA + i] = (i < r && !gla) ? br * w[ii] * __uint_as_float(dg[half][ii]) : 0.f;
            }
        }
    } else if (done) {  // rows 64..127: Q K^T -> P
        const int r = tid - 64;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float d[32];
            weights(r, half, d);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const int i = 32 * half + ii;
                d[ii] = (i <= r) ? d[ii] * __uint_as_float(dg[half][ii]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float* x = d + 8 * u;
                *reinterpret_cast<uint4*>(rec + kRecP + umma::sw128_offset(r, 32 * half + 8 * u, 64)) =
                    make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
            }
        }
    }
    if (tid < kC) {  // gamma and the key decay over the rest of the chunk
        float* vec = reinterpret_cast<float*>(rec + kRecVec);
        const float gam = exp2f(sG[tid]);
        vec[tid] = gam;
        sGam[tid] = gam;
        vec[kC + tid] = exp2f(sG[kC - 1] - sG[tid]);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (!done) break;

    // ---- T = (I + A)^{-1}: 32 x 32 diagonal blocks, then T10 = -T11 (A10 T00)
    if (warp < 2) invert_diag_block32(sA, sT, warp, lane);
    __syncthreads();
    {
        const int i = tid >> 2, j0c = (tid & 3) * 8;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = j0c; k < 32; ++k) {  // T00 is lower triangular
            const float a = sA[(32 + i) * kSA + k];
            const float4 t0 = *reinterpret_cast<const float4*>(&sT[k * 68 + j0c]);
            const float4 t1 = *reinterpret_cast<const float4*>(&sT[k * 68 + j0c + 4]);
            x[0] = fmaf(a, t0.x, x[0]); x[1] = fmaf(a, t0.y, x[1]); x[2] = fmaf(a, t0.z, x[2]); x[3] = fmaf(a, t0.w, x[3]);
            x[4] = fmaf(a, t1.x, x[4]); x[5] = fmaf(a, t1.y, x[5]); x[6] = fmaf(a, t1.z, x[6]); x[7] = fmaf(a, t1.w, x[7]);
        }
        *reinterpret_cast<float4*>(&sX[i * 36 + j0c]) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(&sX[i * 36 + j0c + 4]) = make_float4(x[4], x[5], x[6], x[7]);
        __syncthreads();
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k <= i; ++k) {  // T11 is lower triangular
            const float t = sT[(32 + i) * 68 + 32 + k];
            const float4 x0 = *reinterpret_cast<const float4*>(&sX[k * 36 + j0c]);
            const float4 x1 = *reinterpret_cast<const float4*>(&sX[k * 36 + j0c + 4]);
            y[0] = fmaf(t, x0.x, y[0]); y[1] = fmaf(t, x0.y, y[1]); y[2] = fmaf(t, x0.z, y[2]); y[3] = fmaf(t, x0.w, y[3]);
            y[4] = fmaf(t, x1.x, y[4]); y[5] = fmaf(t, x1.y, y[5]); y[6] = fmaf(t, x1.z, y[6]); y[7] = fmaf(t, x1.w, y[7]);
        }
        *reinterpret_cast<float4*>(&sT[(32 + i) * 68 + j0c]) = make_float4(-y[0], -y[1], -y[2], -y[3]);
        *reinterpret_cast<float4*>(&sT[(32 + i) * 68 + j0c + 4]) = make_float4(-y[4], -y[5], -y[6], -y[7]);
        __syncthreads();
    }

    // ---- T diag(beta) and T diag(beta gamma) -> fp16 images of swizzled K-major tiles
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = tid + kThreads * u, r = e >> 3, c8 = (e & 7) * 8;
        float tr[8], be[8], ga[8], tb[8], tbg[8];
        // 16-byte reads (rows of sT start on 16-byte boundaries, as do sBeta and sGam)
        *reinterpret_cast<float4*>(tr) = *reinterpret_cast<const float4*>(sT + r * 68 + c8);
        *reinterpret_cast<float4*>(tr + 4) = *reinterpret_cast<const float4*>(sT + r * 68 + c8 + 4);
        *reinterpret_cast<float4*>(be) = *reinterpret_cast<const float4*>(sBeta + c8);
        *reinterpret_cast<float4*>(be + 4) = *reinterpret_cast<const float4*>(sBeta + c8 + 4);
        *reinterpret_cast<float4*>(ga) = *reinterpret_cast<const float4*>(sGam + c8);
        *reinterpret_cast<float4*>(ga + 4) = *reinterpret_cast<const float4*>(sGam + c8 + 4);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            tb[x] = tr[x] * be[x];
            tbg[x] = gla ? 0.f : tb[x] * ga[x];
        }
        const uint32_t off = umma::sw128_offset(r, c8, 64);
        *reinterpret_cast<uint4*>(rec + kRecTb + off) =
            make_uint4(pack_h2(tb[0], tb[1]), pack_h2(tb[2], tb[3]), pack_h2(tb[4], tb[5]), pack_h2(tb[6], tb[7]));
        // T diag(beta gamma) over the query rows of the stack (no longer needed)
        *reinterpret_cast<uint4*>(sm + kTbg + off) = make_uint4(
            pack_h2(tbg[0], tbg[1]), pack_h2(tbg[2], tbg[3]), pack_h2(tbg[4], tbg[5]), pack_h2(tbg[6], tbg[7]));
    }
    umma::fence_async_smem();
    umma::fence_before_sync();
    __syncthreads();

    // ---- Wm = T diag(beta gamma) K: M = 128 (rows 64..127 of A are don't-care),
    //      N = 128 key dims, K = 64 tokens (the key rows of the stack, MN-major)
    if (tid == 0) {
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, kD, false, true, false);
#pragma unroll
        for (int s16 = 0; s16 < kC / 16; ++s16)
            umma::mma(tmem, umma::kmajor(sbase + kTbg, 128, s16), umma::mnmajor(sbase + kK, 16384, s16), id,
                      s16 > 0);
        umma::commit(mbar);
    }
    const bool done_w = __syncthreads_and(umma::mbar_wait(mbar, phase, kWaitLimit));
    phase ^= 1u;
    if (!done_w) {
        if (tid == 0 && err) atomicExch(err, kErrTimeout);
        break;
    }
    umma::fence_after_sync();
    if (warp < 2) {  // -Wm row r -> record image
        const int r = tid;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {  // two 32-column TMEM loads in flight per wait
            uint32_t w2[2][32];
            umma::tmem_ld32_async(tmem + ((uint32_t)(warp * 32) << 16) + 64 * q2, w2[0]);
            umma::tmem_ld32_async(tmem + ((uint32_t)(warp * 32) << 16) + 64 * q2 + 32, w2[1]);
            umma::tmem_wait_ld();
            umma::reg_fence32(w2[0]);
            umma::reg_fence32(w2[1]);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(w2[hh][8 * u + e]);
                    *reinterpret_cast<uint4*>(rec + kRecWm + umma::sw128_offset(r, 64 * q2 + 32 * hh + 8 * u, 64)) =
                        make_uint4(pack_h2(-x[0], -x[1]), pack_h2(-x[2], -x[3]), pack_h2(-x[4], -x[5]),
                                   pack_h2(-x[6], -x[7]));
                }
            }
        }
    }
    umma::fence_before_sync();
    __syncthreads();  // shared tiles and TMEM are reused by the next item
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
    grid_dependency_wait();
}

}  // namespace

size_t gdn_chunk_slots(int64_t total, int n_seqs) { return (size_t)(total / kC) + (size_t)n_seqs + 1; }

cudaError_t launch_gdn_inverse(const LayerDims& L, const __half* qhat, const __half* khat, const float* g,
                               const float* beta, const int32_t* cu, const int32_t* chunk_base, int slot_lo,
                               int slot_hi, int32_t* counter, unsigned char* rec_out, int32_t* err, bool beside_prior,
                               cudaStream_t st) {
    if (slot_hi <= slot_lo) return cudaSuccess;
    static DeviceCache cache;  // the shared-memory attribute and the SM count, per device
    int n_sm = 0;
    cudaError_t e = device_cached(cache, &n_sm, [](int dev, int* v) {
        cudaError_t r = cudaFuncSetAttribute(gdn_inverse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemAlloc);
        return r == cudaSuccess ? sm_count(dev, v) : r;
    });
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)(slot_hi - slot_lo) * L.Hq;
    const unsigned grid = (unsigned)std::min<int64_t>(items, (int64_t)n_sm * 3);
    LaunchCfg lc(dim3(grid), dim3(kThreads), kSmemAlloc, st, beside_prior);
    return cudaLaunchKernelEx(&lc.cfg, gdn_inverse_kernel, L, qhat, khat, g, beta, cu, chunk_base, slot_lo, slot_hi,
                              counter, rec_out, err);
}

}  // namespace hla
