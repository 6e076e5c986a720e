// Linear branch, chunked form on the tcgen05 tensor cores: the state-carrying
// part.
//
// The GDN recurrence of "迈向线性的关键：分析驱动的 Transformer 线性化" (section
// 线性注意力替换机制, scalar gate) with the delayed, fixed-budget routing of
// section 填补近似缺口的实用设计 (token j enters the state at position j + W)
// is evaluated in chunks of C = 64 absorbed tokens.  The parallel chunk kernel
// has already produced, per chunk, -Wm = -T diag(beta gamma) K, T diag(beta)
// (T = (I + A)^{-1}), P, the per-token gamma and key decay, and V^T; with them
//   U  = T diag(beta) V - Wm S0
//   O  = diag(gamma) Q S0 + P U
//   S1 = gamma_C S0 + (diag(e^{G_C - G}) K)^T U
// where the query of token j is qhat at position j + W.
//
// The value columns of S never mix (every product above acts on S from the
// left), so a CTA owns one slice of NS value columns of one (sequence,
// q-head) state: 128 / NS CTAs share a head and the state chain runs on that
// many SMs at once.  With the chunk rows stacked on the 128 TMEM lanes every
// MMA has M = 128 and N = NS:
//   D1[b] = [-Wm ; Q] S0  +  [T diag(beta) ; 0] V      rows 0..63 = U, 64..127 = Q S0
//   D2[b] = [0 ; P] U                                   rows 64..127 = P U
//   DS    = K^T diag(e^{G_C - G}) U                     (key dims on the lanes)
// fp16 operands in shared memory, fp32 accumulators in TMEM; the zero blocks
// pad the 64-row operands to M = 128.  S0 stays in fp32 registers (one key
// row per thread) and is re-rounded to fp16 for the next chunk's MMA.
//
// Roles (256 threads): warps 0-3 run the chain (MMA issue, U and S
// epilogues); warps 4-5 load chunk c+1 into the other buffer (cp.async);
// warps 6-7 turn the double-buffered D1/D2 rows 64..127 into o_lin rows
// (o = gamma Q S0 + P U).  Handoffs use mbarriers: ready[b] (load -> chain),
// free[b] (chain + output -> load), ofull[b] (MMA -> output), ofree[b]
// (output -> chain).  Every wait has an iteration limit; on expiry the kernel
// records a timeout in the error word and all roles stop.
#include "hla_common.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kC = 64;    // chunk length (absorbed tokens)
constexpr int kD = 128;   // head dim
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared-memory plan for value-slice width NS (bytes from a 1024-aligned base)
template <int NS>
struct Plan {
    // one chunk buffer
    static constexpr uint32_t kA1 = 0;              // [-Wm ; Q] 128 x 128, K-major
    static constexpr uint32_t kTZP = 32768;         // [T diag(beta) | 0 | P], three 64 x 64 K-major images
    static constexpr uint32_t kK = 57344;           // K rows 64 x 128 (MN-major A of DS)
    static constexpr uint32_t kVt = 73728;          // V^T slice NS x 64 (K-major B)
    static constexpr uint32_t kVec = kVt + NS * 128;  // gamma[64], key decay[64]
    static constexpr uint32_t kBuf = (kVec + 512 + 1023) / 1024 * 1024;
    // chain operands
    static constexpr uint32_t kS = 2 * kBuf;         // S0 slice, NS x 128 (K-major B)
    static constexpr uint32_t kU = kS + NS * 256;    // U slice, NS x 64 (K-major B)
    static constexpr uint32_t kUk = kU + NS * 128;   // diag(key decay) U slice
    static constexpr uint32_t kBar = kUk + NS * 128;
    static constexpr uint32_t kSmemAlloc = kBar + 128 + 1024;
    // TMEM columns
    static constexpr uint32_t kColD1 = 0, kColD2 = 2 * NS, kColS = 4 * NS;
    static constexpr uint32_t kTmemCols = 5 * NS <= 256 ? 256 : 512;
};

// mbarrier indices
constexpr int kReady = 0, kFree = 2, kMma1 = 4, kMma2 = 5, kOFull = 6, kOFree = 8, kNumBars = 10;

__device__ __forceinline__ void st16(unsigned char* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// 16-byte global -> shared copy that bypasses registers; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(unsigned char* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(umma::smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// barrier among the `count` threads of one role (ids 1-3; 0 is __syncthreads)
__device__ __forceinline__ void group_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// All `count` threads of role `id` vote; true only if every one passes `v`.
__device__ __forceinline__ bool group_all(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// NS fp32 TMEM columns of this thread's lane.
template <int NS>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
#pragma unroll
    for (int q = 0; q < NS / 32; ++q) umma::tmem_ld32(taddr + 32 * q, v + 32 * q);
}

// Writes x[0..NS) of this thread (row k of a K-major image with NS rows,
// element (n, k) = x[n] of thread k) as fp16, pairing with the neighbour lane
// k ^ 1 so every store is 4 bytes: the even lane stores even rows n, the odd
// lane odd rows.  The thread's own values are scaled by own_scale, the
// partner's by partner_scale (per-row factors of the K index).
template <int NS>
__device__ __forceinline__ void store_transposed(unsigned char* img, const float* x, int k, float own_scale,
                                                 float partner_scale) {
    const bool odd = k & 1;
#pragma unroll
    for (int m = 0; m < NS / 2; ++m) {
        const float send = odd ? x[2 * m] : x[2 * m + 1];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        const float own = odd ? x[2 * m + 1] : x[2 * m];
        const float lo = odd ? recv * partner_scale : own * own_scale;
        const float hi = odd ? own * own_scale : recv * partner_scale;
        *reinterpret_cast<uint32_t*>(img + umma::sw128_offset(2 * m + (odd ? 1 : 0), k & ~1, NS)) =
            pack_h2(lo, hi);
    }
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chunked_kernel(LayerDims L, const __half* __restrict__ qhat, const __half* __restrict__ khat,
                   const int32_t* __restrict__ cu, const int32_t* __restrict__ chunk_base,
                   const unsigned char* __restrict__ rec_in, const unsigned char* __restrict__ vt_in,
                   float* __restrict__ o_lin, float* __restrict__ S_out, int32_t* __restrict__ err) {
    using P = Plan<NS>;
    constexpr int kSlices = kD / NS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + P::kBar + 8 * kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + P::kBar + 8 * kNumBars + 4);

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    const int h = blockIdx.x / kSlices, slice = blockIdx.x % kSlices, n = blockIdx.y;
    const int kv = h / L.G, W = L.window;
    const uint32_t sbase = umma::smem_addr(sm);
    const uint32_t bar0 = umma::smem_addr(sm + P::kBar);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t j_end = len - W;
    const int n_chunks = j_end > L.n_sinks ? (int)((j_end - L.n_sinks + kC - 1) / kC) : 0;
    const int slot0 = __ldg(chunk_base + n);

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) umma::mbar_init(bar(i), (i == kFree || i == kFree + 1) ? 2 : 1);
        umma::fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, P::kTmemCols);
    for (int i = tid; i < NS * 256 / 16; i += kThreads) st16(sm + P::kS + 16 * i, make_uint4(0, 0, 0, 0));
    for (int i = tid; i < 2 * 512; i += kThreads)  // the zero blocks of both buffers
        st16(sm + (i >> 9) * P::kBuf + P::kTZP + 8192 + 16 * (i & 511), make_uint4(0, 0, 0, 0));
    umma::fence_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto wait = [&](int i, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        const bool done = umma::mbar_wait(bar(i), parity, kWaitLimit);
        if (!done) {
            *abort_flag = 1;
            if (err) atomicExch(err, kErrTimeout);
        }
        umma::fence_after_sync();
        return done;
    };

    if (warp < 4) {
        // ================= the state chain =================
        float S[NS];  // S0[tid][slice columns]: fp32 master copy
#pragma unroll
        for (int i = 0; i < NS; ++i) S[i] = 0.f;
        const uint32_t id = umma::idesc_f16(128, NS, false, false, false);
        const uint32_t id_amn = umma::idesc_f16(128, NS, true, false, false);
        uint32_t ph1 = 0, ph2 = 0;
        bool ok = true;
        for (int c = 0; c < n_chunks && ok; ++c) {
            const int b = c & 1;
            const uint32_t buf = (uint32_t)b * P::kBuf;
            ok = group_all(1, 128, wait(kReady + b, (uint32_t)((c >> 1) & 1)));
            if (ok && c >= 2) ok = group_all(1, 128, wait(kOFree + b, (uint32_t)(((c - 2) >> 1) & 1)));
            if (!ok) break;

            // D1[b] = [-Wm ; Q] S0 + [T diag(beta) ; 0] V
            if (tid == 0) {
                const uint32_t d1 = tmem + P::kColD1 + NS * b;
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    umma::mma(d1, umma::kmajor(sbase + buf + P::kA1, 128, s), umma::kmajor(sbase + P::kS, NS, s), id,
                              s > 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(d1, umma::kmajor(sbase + buf + P::kTZP, 128, s), umma::kmajor(sbase + buf + P::kVt, NS, s),
                              id, true);
                umma::commit(bar(kMma1));
            }
            ok = group_all(1, 128, wait(kMma1, ph1));
            ph1 ^= 1u;
            if (!ok) break;

            // U (rows 0..63) -> fp16 K-major images U and diag(key decay) U
            if (warp < 2) {
                const float* kdec = reinterpret_cast<const float*>(sm + buf + P::kVec) + kC;
                float u[NS];
                tmem_ld<NS>(tmem + lane_base + P::kColD1 + NS * b, u);
                store_transposed<NS>(sm + P::kU, u, tid, 1.f, 1.f);
                store_transposed<NS>(sm + P::kUk, u, tid, kdec[tid], kdec[tid ^ 1]);
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1, 128);

            // D2[b] = [0 ; P] U;  DS = K^T diag(key decay) U
            if (tid == 0) {
                umma::fence_after_sync();
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + P::kColD2 + NS * b, umma::kmajor(sbase + buf + P::kTZP + 8192, 128, s),
                              umma::kmajor(sbase + P::kU, NS, s), id, s > 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + P::kColS, umma::mnmajor(sbase + buf + P::kK, 8192, s),
                              umma::kmajor(sbase + P::kUk, NS, s), id_amn, s > 0);
                umma::commit(bar(kMma2));
                umma::commit(bar(kOFull + b));
            }
            ok = group_all(1, 128, wait(kMma2, ph2));
            ph2 ^= 1u;
            if (!ok) break;
            const float gC = reinterpret_cast<const float*>(sm + buf + P::kVec)[kC - 1];  // gamma_C
            group_sync(1, 128);
            if (tid == 0) mbar_arrive(bar(kFree + b));  // the chain is done with buffer b

            // S <- gamma_C S + DS; fp16 copy for the next chunk
            {
                float ds[NS];
                tmem_ld<NS>(tmem + lane_base + P::kColS, ds);
#pragma unroll
                for (int i = 0; i < NS; ++i) S[i] = fmaf(gC, S[i], ds[i]);
                store_transposed<NS>(sm + P::kS, S, tid, 1.f, 1.f);
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1, 128);
        }
        if (ok && S_out) {
            float* dst = S_out + (((size_t)n * L.Hq + h) * kD + tid) * kD + slice * NS;
#pragma unroll
            for (int i = 0; i < NS; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
        }
    } else if (warp < 6) {
        // ================= loads, one chunk ahead =================
        const int p = tid - 128;
        for (int c = 0; c < n_chunks; ++c) {
            const int b = c & 1;
            if (c >= 2 && !group_all(2, 64, wait(kFree + b, (uint32_t)(((c - 2) >> 1) & 1)))) break;
            unsigned char* buf = sm + b * P::kBuf;
            const int64_t j0 = L.n_sinks + (int64_t)c * kC;
            const int nv = (int)min((int64_t)kC, j_end - j0);
#pragma unroll 4
            for (int u = 0; u < 16; ++u) {  // query rows (positions j + W) and key rows, zero past the chunk
                const int e = p + 64 * u, r = e >> 4, c8 = (e & 15) * 8;
                const uint32_t nb = r < nv ? 16u : 0u;
                const size_t t = (size_t)(start + j0 + (r < nv ? r : 0));
                cp_async16(buf + P::kA1 + umma::sw128_offset(64 + r, c8, 128), qhat + ((t + W) * L.Hq + h) * kD + c8, nb);
                cp_async16(buf + P::kK + umma::sw128_offset(r, c8, 64), khat + (t * L.Hkv + kv) * kD + c8, nb);
            }
            const unsigned char* rec = rec_in + ((size_t)(slot0 + c) * L.Hq + h) * kRecordBytes;
#pragma unroll 4
            for (int u = 0; u < 8; ++u) {
                const uint32_t o = 16u * (uint32_t)(p + 64 * u);
                cp_async16(buf + P::kA1 + o, rec + kRecWm + o, 16u);                 // -Wm, key dims 0..63
                cp_async16(buf + P::kA1 + 16384 + o, rec + kRecWm + 8192 + o, 16u);  // key dims 64..127
                cp_async16(buf + P::kTZP + o, rec + kRecTb + o, 16u);
                cp_async16(buf + P::kTZP + 16384 + o, rec + kRecP + o, 16u);
            }
            if (p < 32) cp_async16(buf + P::kVec + 16 * p, rec + kRecVec + 16 * p, 16u);
            const unsigned char* vt =
                vt_in + ((size_t)(slot0 + c) * L.Hkv + kv) * kVtBytes + (size_t)slice * NS * 128;
#pragma unroll
            for (int u = 0; u < NS * 128 / 16 / 64; ++u) {
                const uint32_t o = 16u * (uint32_t)(p + 64 * u);
                cp_async16(buf + P::kVt + o, vt + o, 16u);
            }
            cp_async_commit();
            cp_async_wait_all();
            umma::fence_async_smem();
            group_sync(2, 64);
            if (p == 0) mbar_arrive(bar(kReady + b));
        }
    } else {
        // ================= o_lin rows: gamma (Q S0) + P U =================
        const int r = tid - 192;  // chunk row; TMEM lane 64 + r
        for (int c = 0; c < n_chunks; ++c) {
            const int b = c & 1;
            if (!group_all(3, 64, wait(kOFull + b, (uint32_t)((c >> 1) & 1)))) break;
            const float gr = reinterpret_cast<const float*>(sm + b * P::kBuf + P::kVec)[r];
            float d1[NS], d2[NS];
            tmem_ld<NS>(tmem + lane_base + P::kColD1 + NS * b, d1);
            tmem_ld<NS>(tmem + lane_base + P::kColD2 + NS * b, d2);
            umma::fence_before_sync();
            group_sync(3, 64);
            if (r == 0) {
                mbar_arrive(bar(kOFree + b));
                mbar_arrive(bar(kFree + b));
            }
            const int64_t j0 = L.n_sinks + (int64_t)c * kC;
            if (r < j_end - j0) {
                float* orow = o_lin + ((size_t)(start + j0 + r + W) * L.Hq + h) * kD + slice * NS;
#pragma unroll
                for (int i = 0; i < NS; i += 4)
                    *reinterpret_cast<float4*>(orow + i) =
                        make_float4(fmaf(gr, d1[i], d2[i]), fmaf(gr, d1[i + 1], d2[i + 1]),
                                    fmaf(gr, d1[i + 2], d2[i + 2]), fmaf(gr, d1[i + 3], d2[i + 3]));
            }
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, P::kTmemCols);
}

template <int NS>
cudaError_t launch_ns(const LayerDims& L, const __half* qhat, const __half* khat, const int32_t* cu,
                      const int32_t* chunk_base, const unsigned char* rec_in, const unsigned char* vt_in,
                      float* o_lin, float* S_out, int32_t* err, cudaStream_t st) {
    static bool configured = false;  // the attribute is per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gdn_chunked_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Plan<NS>::kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(L.Hq * (kD / NS), L.n_seqs);
    gdn_chunked_kernel<NS><<<grid, kThreads, Plan<NS>::kSmemAlloc, st>>>(L, qhat, khat, cu, chunk_base, rec_in,
                                                                        vt_in, o_lin, S_out, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_chunked(const LayerDims& L, const __half* qhat, const __half* khat, const int32_t* cu,
                               const int32_t* chunk_base, const unsigned char* rec_in,
                               const unsigned char* vt_in, float* o_lin, float* S_out, int32_t* err,
                               cudaStream_t st) {
    static int n_sm = 0;  // per-process device property cache
    if (!n_sm) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
            n_sm = 148;
    }
    // narrow slices while the state chains alone do not fill the SMs
    const int64_t chains = (int64_t)L.n_seqs * L.Hq;
    if (chains * (kD / 32) <= n_sm)
        return launch_ns<32>(L, qhat, khat, cu, chunk_base, rec_in, vt_in, o_lin, S_out, err, st);
    return launch_ns<64>(L, qhat, khat, cu, chunk_base, rec_in, vt_in, o_lin, S_out, err, st);
}

}  // namespace hla
