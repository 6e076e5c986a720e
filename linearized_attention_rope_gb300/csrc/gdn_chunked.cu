// Linear branch, chunked form on the tcgen05 tensor cores: the state-carrying
// part.
//
// The GDN recurrence of "迈向线性的关键：分析驱动的 Transformer 线性化" (section
// 线性注意力替换机制, scalar gate) with the delayed, fixed-budget routing of
// section 填补近似缺口的实用设计 (token j enters the state at position j + W)
// is evaluated in chunks of C = 64 absorbed tokens.  The parallel chunk kernel
// has already produced, per chunk, T diag(beta), T diag(beta gamma) (T = (I +
// A)^{-1}), P and the per-token gamma and key decay; with them
//   U = T diag(beta) V - T diag(beta gamma) K S0
//   O = diag(gamma) Q S0 + P U
//   S1 = gamma_C S0 + (diag(e^{G_C - G}) K)^T U
// where the query of token j is qhat at position j + W.  Every product is a
// tcgen05 MMA with fp16 operands in shared memory and fp32 accumulators in
// tensor memory, laid out with the value dim (or the key dim for Wm) on the
// 128 TMEM lanes so every MMA has M = 128:
//   D_U[b] [dv x tok] = V^T (T diag beta)^T,        then += S0^T (-Wm^T)
//   D_W    [dk x tok] = K^T (T diag(beta gamma))^T    (= Wm^T)
//   D_O[b] [dv x tok] = S0^T (diag(gamma) Q)^T,       then += U^T P^T
//   D_S    [dv x dk]  = (U^T diag(e^{G_C - G})) K     (= ((decayed K)^T U)^T)
//
// One CTA of 256 threads per (sequence, q-head), two warp-specialised groups:
//   prep   (warps 4-7): chunk c+1 -- cp.async loads one chunk ahead, gamma Q in
//          place, D_U and D_W, Wm^T; and the o_lin rows of chunk c-1 from its
//          (double-buffered) output accumulator;
//   serial (warps 0-3): chunk c -- D_U += S0^T(-Wm^T) and D_O, U^T (twice),
//          D_S and D_O += U^T P^T, S <- gamma_C S + dS in fp32 registers.
// Chunk buffers b = c % 2 pass between the groups through the mbarriers
// ready[b] (prep -> serial) and free[b] (serial -> prep).  Every wait has an
// iteration limit; on expiry the kernel records a timeout in the error word
// and both groups stop.
#include "hla_common.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kC = 64;    // chunk length (absorbed tokens)
constexpr int kD = 128;   // head dim
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared-memory plan (bytes from a 1024-aligned base)
constexpr uint32_t kStk0 = 0, kStk1 = 32768;    // [K ; Q] 128 x 128; Q rows scaled by gamma in place
constexpr uint32_t kVt = 65536;                 // V [tok][dv] (MN-major A)
constexpr uint32_t kTb = 81920;                 // T diag(beta) (K-major B), 8 KB
constexpr uint32_t kTbg = 90112;                // T diag(beta gamma) (K-major B), 8 KB
constexpr uint32_t kP0 = 98304, kP1 = 106496;   // P 64 x 64 (K-major B), 8 KB each
constexpr uint32_t kW0 = 114688, kW1 = 131072;  // Wm^T [dk][tok] (MN-major B), 16 KB each
constexpr uint32_t kSt = 147456;                // S0^T [dv][dk] (K-major A), 32 KB
constexpr uint32_t kUt = 180224;                // U^T [dv][tok] (K-major A), 16 KB
constexpr uint32_t kUtk = 196608;               // U^T diag(e^{G_C - G}) (K-major A), 16 KB
constexpr uint32_t kVec0 = 212992, kVec1 = kVec0 + 512;  // gamma[64], key decay[64] per buffer
constexpr uint32_t kBar = kVec1 + 512;
constexpr uint32_t kSmemBytes = kBar + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

// TMEM columns
constexpr uint32_t kColW = 0, kColU0 = 64, kColO0 = 192, kColS = 320, kTmemCols = 512;

__device__ __forceinline__ void st16(unsigned char* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ uint4 ld16(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8(const float* v) {
    return make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
}
__device__ __forceinline__ uint4 scale8(uint4 u, float s) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        v[2 * i] = f.x * s;
        v[2 * i + 1] = f.y * s;
    }
    return pack8(v);
}
// 16-byte global -> shared copy that bypasses registers; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(unsigned char* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(umma::smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// barrier among the 128 threads of one warp group (ids 1 and 2; 0 is __syncthreads)
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// All 128 threads of group `id` vote; true only if every one passes `v`.
__device__ __forceinline__ bool group_all(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, 128, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
gdn_chunked_kernel(LayerDims L, const __half* __restrict__ qhat, const __half* __restrict__ khat,
                   const __half* __restrict__ vhat, const int32_t* __restrict__ cu,
                   const int32_t* __restrict__ chunk_base, const unsigned char* __restrict__ rec_in,
                   float* __restrict__ o_lin, float* __restrict__ S_out, int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);  // mma_prep, mma_serial, ready[2], free[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kBar + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kBar + 68);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Lr = ((warp & 3) << 5) + lane;  // TMEM lane / row owned
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G, W = L.window;
    const uint32_t sbase = umma::smem_addr(sm);
    const uint32_t bar0 = umma::smem_addr(bars);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t j_end = len - W;
    const int n_chunks = j_end > L.n_sinks ? (int)((j_end - L.n_sinks + kC - 1) / kC) : 0;
    const int slot0 = __ldg(chunk_base + n);

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) umma::mbar_init(bar(i), 1);
        umma::fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
    for (int i = tid; i < 32768 / 16; i += kThreads) st16(sm + kSt + 16 * i, make_uint4(0, 0, 0, 0));
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

    // o_lin rows of chunk c (positions j + W), from D_O[c % 2]
    auto store_out = [&](int c) {
        const int64_t j0 = L.n_sinks + (int64_t)c * kC;
        const int nv = (int)min((int64_t)kC, j_end - j0);
        float* orow = o_lin + ((size_t)(start + j0 + W) * L.Hq + h) * kD + Lr;
        const size_t ostride = (size_t)L.Hq * kD;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float o[32];
            umma::tmem_ld32(tmem + lane_base + kColO0 + 64 * (c & 1) + 32 * hf, o);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii)
                if (32 * hf + ii < nv) orow[(size_t)(32 * hf + ii) * ostride] = o[ii];
        }
    };

    if (warp >= 4) {
        // ================= prep group: one chunk ahead of the serial group =================
        const int pt = tid - 128;
        // rows of chunk c -> stack[b], V, records -> (T diag beta, T diag(beta gamma), P[b], vec[b])
        auto load = [&](int c, int b) {
            const int64_t pj0 = L.n_sinks + (int64_t)c * kC;
            const int pnv = (int)min((int64_t)kC, j_end - pj0);
            unsigned char* stk = sm + (b ? kStk1 : kStk0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = pt + 128 * u, r = e >> 4, c8 = (e & 15) * 8;
                const uint32_t nb = r < pnv ? 16u : 0u;
                const size_t t = (size_t)(start + pj0 + (r < pnv ? r : 0));
                cp_async16(stk + umma::sw128_offset(r, c8, 128), khat + (t * L.Hkv + kv) * kD + c8, nb);
                cp_async16(stk + umma::sw128_offset(64 + r, c8, 128), qhat + ((t + W) * L.Hq + h) * kD + c8, nb);
                cp_async16(sm + kVt + umma::sw128_offset(r, c8, 64), vhat + (t * L.Hkv + kv) * kD + c8, nb);
            }
            const unsigned char* rec = rec_in + ((size_t)(slot0 + c) * L.Hq + h) * kRecordBytes;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t o = 16u * (uint32_t)(pt + 128 * u);
                cp_async16(sm + kTb + o, rec + kRecTb + o, 16u);
                cp_async16(sm + kTbg + o, rec + kRecTbg + o, 16u);
                cp_async16(sm + (b ? kP1 : kP0) + o, rec + kRecP + o, 16u);
            }
            if (pt < 32) cp_async16(sm + (b ? kVec1 : kVec0) + 16 * pt, rec + kRecVec + 16 * pt, 16u);
            cp_async_commit();
        };
        if (n_chunks > 0) load(0, 0);
        uint32_t ph = 0;
        bool ok = true;
        for (int c = 0; c < n_chunks && ok; ++c) {
            const int b = c & 1;
            const uint32_t ostk = b ? kStk1 : kStk0;
            const float* gam = reinterpret_cast<const float*>(sm + (b ? kVec1 : kVec0));

            // -- a. chunk c has landed; gamma Q in place
            cp_async_wait_all();
            group_sync(2);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = pt + 128 * u, r = e >> 4, c8 = (e & 15) * 8;
                unsigned char* p = sm + ostk + umma::sw128_offset(64 + r, c8, 128);
                st16(p, scale8(ld16(p), gam[r]));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(2);

            // -- b. D_U[b] = V^T (T diag beta)^T;  D_W = K^T (T diag(beta gamma))^T
            if (pt == 0) {
                umma::fence_after_sync();
                const uint32_t id = umma::idesc_f16(128, kC, true, false, false);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColU0 + 64 * b, umma::mnmajor(sbase + kVt, 8192, s),
                              umma::kmajor(sbase + kTb, 64, s), id, s > 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColW, umma::mnmajor(sbase + ostk, 16384, s), umma::kmajor(sbase + kTbg, 64, s),
                              id, s > 0);
                umma::commit(bar(0));
            }
            ok = group_all(2, wait(0, ph));
            ph ^= 1u;
            if (!ok) break;

            // -- c. Wm^T -> W[b] (MN-major B); chunk c is then ready for the serial group
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float w[32];
                umma::tmem_ld32(tmem + lane_base + kColW + 32 * hf, w);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st16(sm + (b ? kW1 : kW0) + umma::sw128_offset(Lr, 32 * hf + 8 * u, 128), pack8(w + 8 * u));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(2);
            if (pt == 0) mbar_arrive(bar(2 + b));

            // -- d. once the serial group is done with chunk c-1: its o_lin rows, and the
            //       next chunk's loads into the buffer it released
            if (c >= 1) {
                ok = group_all(2, wait(4 + ((c - 1) & 1), (uint32_t)(((c - 1) >> 1) & 1)));
                if (!ok) break;
                store_out(c - 1);
            }
            if (c + 1 < n_chunks) load(c + 1, (c + 1) & 1);

        }
        if (ok && n_chunks > 0) {  // the last chunk's o_lin rows
            const int c = n_chunks - 1;
            if (group_all(2, wait(4 + (c & 1), (uint32_t)((c >> 1) & 1)))) store_out(c);
        }
    } else {
        // ================= serial group: the state chain =================
        float S[kD];  // S0^T[Lr][0 .. 127]: fp32 master copy of the state
#pragma unroll
        for (int i = 0; i < kD; ++i) S[i] = 0.f;
        uint32_t ph = 0;
        bool ok = true;
        for (int c = 0; c < n_chunks && ok; ++c) {
            const int b = c & 1;
            const uint32_t ostk = b ? kStk1 : kStk0;
            ok = group_all(1, wait(2 + b, (uint32_t)((c >> 1) & 1)));
            if (!ok) break;

            // D_U[b] += S0^T (-Wm^T);  D_O[b] = S0^T (gamma Q)^T
            if (tid == 0) {
                const uint32_t id1 = umma::idesc_f16(128, kC, false, true, true);
                const uint32_t id3 = umma::idesc_f16(128, kC, false, false, false);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    umma::mma(tmem + kColU0 + 64 * b, umma::kmajor(sbase + kSt, 128, s),
                              umma::mnmajor(sbase + (b ? kW1 : kW0), 16384, s), id1, true);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    umma::mma(tmem + kColO0 + 64 * b, umma::kmajor(sbase + kSt, 128, s),
                              umma::kmajor(sbase + ostk + 64 * 128, 128, s), id3, s > 0);
                umma::commit(bar(1));
            }
            ok = group_all(1, wait(1, ph));
            ph ^= 1u;
            if (!ok) break;

            // U^T and U^T diag(e^{G_C - G}) -> fp16 K-major tiles
            {
                const float* kdec = reinterpret_cast<const float*>(sm + (b ? kVec1 : kVec0)) + kC;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float u32[32];
                    umma::tmem_ld32(tmem + lane_base + kColU0 + 64 * b + 32 * hf, u32);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        st16(sm + kUt + umma::sw128_offset(Lr, 32 * hf + 8 * u, 128), pack8(u32 + 8 * u));
#pragma unroll
                    for (int i = 0; i < 32; ++i) u32[i] *= kdec[32 * hf + i];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        st16(sm + kUtk + umma::sw128_offset(Lr, 32 * hf + 8 * u, 128), pack8(u32 + 8 * u));
                }
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1);

            // D_S = (U^T diag(e^{G_C - G})) K;  D_O[b] += U^T P^T
            if (tid == 0) {
                umma::fence_after_sync();
                const uint32_t id2 = umma::idesc_f16(128, kD, false, true, false);
                const uint32_t id3 = umma::idesc_f16(128, kC, false, false, false);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColS, umma::kmajor(sbase + kUtk, 128, s), umma::mnmajor(sbase + ostk, 16384, s),
                              id2, s > 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColO0 + 64 * b, umma::kmajor(sbase + kUt, 128, s),
                              umma::kmajor(sbase + (b ? kP1 : kP0), 64, s), id3, true);
                umma::commit(bar(1));
            }
            ok = group_all(1, wait(1, ph));
            ph ^= 1u;
            if (!ok) break;
            const float gC = reinterpret_cast<const float*>(sm + (b ? kVec1 : kVec0))[kC - 1];  // gamma_C
            umma::fence_before_sync();
            group_sync(1);
            if (tid == 0) mbar_arrive(bar(4 + b));  // buffer b may be refilled

            // S <- gamma_C S + dS; fp16 copy for the next chunk
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float ds[32];
                umma::tmem_ld32(tmem + lane_base + kColS + 32 * q4, ds);
#pragma unroll
                for (int i = 0; i < 32; ++i) S[32 * q4 + i] = fmaf(gC, S[32 * q4 + i], ds[i]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st16(sm + kSt + umma::sw128_offset(Lr, 32 * q4 + 8 * u, 128), pack8(S + 32 * q4 + 8 * u));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1);
        }
        if (ok && S_out) {
            float* dst = S_out + ((size_t)n * L.Hq + h) * kD * kD + Lr;
#pragma unroll
            for (int i = 0; i < kD; ++i) dst[(size_t)i * kD] = S[i];
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gdn_chunked(const LayerDims& L, const __half* qhat, const __half* khat, const __half* vhat,
                               const int32_t* cu, const int32_t* chunk_base, const unsigned char* rec_in,
                               float* o_lin, float* S_out, int32_t* err, cudaStream_t st) {
    static bool configured = false;  // the attribute is per function
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gdn_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(L.Hq, L.n_seqs);
    gdn_chunked_kernel<<<grid, kThreads, kSmemAlloc, st>>>(L, qhat, khat, vhat, cu, chunk_base, rec_in, o_lin,
                                                          S_out, err);
    return cudaGetLastError();
}

}  // namespace hla
