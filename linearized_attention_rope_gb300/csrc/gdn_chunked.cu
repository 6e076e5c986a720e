// Linear branch, chunked form on the tcgen05 tensor cores: the state-carrying
// part.
//
// The GDN recurrence of "迈向线性的关键：分析驱动的 Transformer 线性化" (section
// 线性注意力替换机制, scalar gate) with the delayed, fixed-budget routing of
// section 填补近似缺口的实用设计 (token j enters the state at position j + W)
// is evaluated in chunks of C = 64 absorbed tokens.  With the gates cumulated
// inside the chunk, G_r = sum_{i<=r} g_i, gamma_r = e^{G_r}, and T = (I + A)^{-1}
// from the parallel inverse kernel:
//   U~ = T diag(beta) V,    Wm = T diag(beta gamma) K,    U = U~ - Wm S0
//   O  = diag(gamma) Q S0 + P U,   P[r,i] = e^{G_r - G_i} q_r . k_i (i <= r)
//   S1 = gamma_C S0 + Kt^T U,      Kt = diag(e^{G_C - G}) K
// where the query of token j is qhat at position j + W.  Every product is a
// tcgen05 MMA with fp16 operands in shared memory and fp32 accumulators in
// tensor memory, laid out with the value dim (or the key dim for Wm) on the
// 128 TMEM lanes so every MMA has M = 128:
//   D_G  [128 x 64]  = [K; Q] K^T                  (only the Q K^T rows are used)
//   D_U  [dv x tok]  = (diag(beta) V)^T T^T,   then  += S0^T (-Wm^T)
//   D_W  [dk x tok]  = (diag(beta gamma) K)^T T^T   (= Wm^T)
//   D_O  [dv x tok]  = S0^T (diag(gamma) Q)^T, then  += U^T P^T
//   D_S  [dv x dk]   = U^T Kt                       (= (Kt^T U)^T)
//
// One CTA of 256 threads per (sequence, q-head), two warp-specialised groups:
//   prep   (warps 4-7): chunk c+1 -- loads (cp.async, one chunk ahead), gates,
//          D_G -> P, beta V and beta gamma K, D_U and D_W, Wm^T, Kt, gamma Q;
//   serial (warps 0-3): chunk c -- the state chain D_U += S0^T(-Wm^T), D_O,
//          U^T, D_S, D_O += U^T P^T, S <- gamma_C S + dS (fp32 registers),
//          o_lin rows.
// The two groups hand chunk buffers over through mbarriers: ready[b]
// (prep -> serial) and free[b] (serial -> prep), b = chunk parity.  Every wait
// has an iteration limit; on expiry the kernel records a timeout in the error
// word and both groups stop.
#include "hla_common.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kC = 64;    // chunk length (absorbed tokens)
constexpr int kD = 128;   // head dim
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared-memory plan (bytes from a 1024-aligned base)
constexpr uint32_t kStk0 = 0, kStk1 = 32768;    // [K ; Q] 128 x 128, later [Kt ; gamma Q]
constexpr uint32_t kVt = 65536;                 // V [tok][dv] (MN-major A), scaled by beta in place
constexpr uint32_t kKbg = 81920;                // beta gamma K [tok][dk] (MN-major A)
constexpr uint32_t kTt = 98304;                 // T 64 x 64 (K-major B), 8 KB
constexpr uint32_t kP0 = 106496, kP1 = 114688;  // P 64 x 64 (K-major B), 8 KB each
constexpr uint32_t kW0 = 122880, kW1 = 139264;  // Wm^T [dk][tok] (MN-major B), 16 KB each
constexpr uint32_t kSt = 155648;                // S0^T [dv][dk] (K-major A), 32 KB
constexpr uint32_t kUt = 188416;                // U^T [dv][tok] (K-major A), 16 KB
constexpr uint32_t kVec = 204800;               // per buffer: G (log2), beta, gamma, Kt decay
constexpr uint32_t kBar = kVec + 2 * 4 * 64 * 4;
constexpr uint32_t kSmemBytes = kBar + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

// TMEM columns
constexpr uint32_t kColG = 0, kColW = 64, kColU0 = 128, kColO = 256, kColS = 320, kTmemCols = 512;

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
                   const __half* __restrict__ vhat, const float* __restrict__ g,
                   const float* __restrict__ beta, const int32_t* __restrict__ cu,
                   const int32_t* __restrict__ chunk_base, const __half* __restrict__ t_in,
                   float* __restrict__ o_lin, float* __restrict__ S_out, int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* vec = reinterpret_cast<float*>(sm + kVec);  // [buffer][G, beta, gamma, Kt decay][64]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);  // mma_prep, mma_serial, ready[2], free[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kBar + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kBar + 68);
    float* carry = reinterpret_cast<float*>(sm + kBar + 72);

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

    if (warp >= 4) {
        // ================= prep group: chunk-local work, one chunk ahead =================
        const int pt = tid - 128;
        float g_next = 0.f, b_next = 0.f;
        auto load_kq = [&](int c, int b) {
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
            }
        };
        auto load_vt = [&](int c) {
            const int64_t pj0 = L.n_sinks + (int64_t)c * kC;
            const int pnv = (int)min((int64_t)kC, j_end - pj0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = pt + 128 * u, r = e >> 4, c8 = (e & 15) * 8;
                const uint32_t nb = r < pnv ? 16u : 0u;
                const size_t t = (size_t)(start + pj0 + (r < pnv ? r : 0));
                cp_async16(sm + kVt + umma::sw128_offset(r, c8, 64), vhat + (t * L.Hkv + kv) * kD + c8, nb);
            }
            const unsigned char* ti =
                reinterpret_cast<const unsigned char*>(t_in + ((size_t)(slot0 + c) * L.Hq + h) * kC * kC);
#pragma unroll
            for (int u = 0; u < 4; ++u) cp_async16(sm + kTt + 16 * (pt + 128 * u), ti + 16 * (pt + 128 * u), 16u);
            if (pt < kC) {
                const size_t t = (size_t)(start + pj0 + pt);
                g_next = pt < pnv ? g[t * L.Hq + h] * 1.4426950408889634f : 0.f;  // log2 units
                b_next = pt < pnv ? beta[t * L.Hq + h] : 0.f;
            }
        };
        if (n_chunks > 0) {
            load_kq(0, 0);
            load_vt(0);
            cp_async_commit();
        }
        uint32_t ph = 0;
        bool ok = true;
        for (int c = 0; c < n_chunks && ok; ++c) {
            const int b = c & 1;
            const uint32_t ostk = b ? kStk1 : kStk0;
            unsigned char* stk = sm + ostk;
            float* vG = vec + b * 256;
            float* vB = vG + 64;
            float* vGam = vG + 128;
            float* vKd = vG + 192;

            // -- a. this chunk's rows and T have landed; gates -> vec[b]
            cp_async_wait_all();
            float gi = g_next;
            if (pt < kC) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gi, o);
                    if (lane >= o) gi += y;
                }
                if (pt == 31) *carry = gi;
                vB[pt] = b_next;
            }
            group_sync(2);
            if (pt < kC) {
                if (pt >= 32) gi += *carry;
                vG[pt] = gi;
            }
            group_sync(2);
            if (pt < kC) {
                vGam[pt] = exp2f(vG[pt]);
                vKd[pt] = exp2f(vG[kC - 1] - vG[pt]);
            }
            umma::fence_async_smem();
            group_sync(2);

            // -- b. D_G = [K; Q] K^T
            if (pt == 0) {
                umma::fence_after_sync();
                const uint32_t id = umma::idesc_f16(128, kC, false, false, false);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    umma::mma(tmem + kColG, umma::kmajor(sbase + ostk, 128, s), umma::kmajor(sbase + ostk, 128, s), id,
                              s > 0);
                umma::commit(bar(0));
            }
            ok = group_all(2, wait(0, ph));
            ph ^= 1u;
            if (!ok) break;

            // -- c. P rows (TMEM lanes 64..127); beta V in place and beta gamma K (warps 4, 5)
            if (warp >= 6) {
                const int r = Lr - 64;
                const float gr = vG[r];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float d[32];
                    umma::tmem_ld32(tmem + lane_base + kColG + 32 * hf, d);
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii) {
                        const int i = 32 * hf + ii;
                        d[ii] = (i <= r) ? exp2f(gr - vG[i]) * d[ii] : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        st16(sm + (b ? kP1 : kP0) + umma::sw128_offset(r, 32 * hf + 8 * u, 64), pack8(d + 8 * u));
                }
            } else {
#pragma unroll 4
                for (int u = 0; u < 16; ++u) {
                    const int e = pt + 64 * u, r = e >> 4, c8 = (e & 15) * 8;
                    const uint32_t off = umma::sw128_offset(r, c8, 64);
                    st16(sm + kVt + off, scale8(ld16(sm + kVt + off), vB[r]));
                    st16(sm + kKbg + off, scale8(ld16(stk + umma::sw128_offset(r, c8, 128)), vB[r] * vGam[r]));
                }
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(2);

            // -- d. D_U[b] = (beta V)^T T^T;  D_W = (beta gamma K)^T T^T
            if (pt == 0) {
                umma::fence_after_sync();
                const uint32_t id = umma::idesc_f16(128, kC, true, false, false);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColU0 + 64 * b, umma::mnmajor(sbase + kVt, 8192, s),
                              umma::kmajor(sbase + kTt, 64, s), id, s > 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColW, umma::mnmajor(sbase + kKbg, 8192, s), umma::kmajor(sbase + kTt, 64, s), id,
                              s > 0);
                umma::commit(bar(0));
            }
            ok = group_all(2, wait(0, ph));
            ph ^= 1u;
            if (!ok) break;

            // -- e. start the next chunk's loads: V and T now, its stack once the serial
            //       group has released that buffer
            if (c + 1 < n_chunks) {
                bool fr = true;
                if (c + 1 >= 2) fr = wait(4 + ((c + 1) & 1), (uint32_t)(((c - 1) >> 1) & 1));
                ok = group_all(2, fr);
                if (!ok) break;
                load_kq(c + 1, (c + 1) & 1);
                load_vt(c + 1);
                cp_async_commit();
            }

            // -- f. Wm^T -> W[b] (MN-major B); Kt and gamma Q in place in the stack
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float w[32];
                umma::tmem_ld32(tmem + lane_base + kColW + 32 * hf, w);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st16(sm + (b ? kW1 : kW0) + umma::sw128_offset(Lr, 32 * hf + 8 * u, 128), pack8(w + 8 * u));
            }
#pragma unroll 4
            for (int u = 0; u < 16; ++u) {
                const int e = pt + 128 * u, row = e >> 4, c8 = (e & 15) * 8;
                const uint32_t off = umma::sw128_offset(row, c8, 128);
                const float s = row < 64 ? vKd[row] : vGam[row - 64];
                st16(stk + off, scale8(ld16(stk + off), s));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(2);
            if (pt == 0) mbar_arrive(bar(2 + b));
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
            const int64_t j0 = L.n_sinks + (int64_t)c * kC;
            const int nv = (int)min((int64_t)kC, j_end - j0);
            ok = group_all(1, wait(2 + b, (uint32_t)((c >> 1) & 1)));
            if (!ok) break;

            // D_U[b] += S0^T (-Wm^T);  D_O = S0^T (gamma Q)^T
            if (tid == 0) {
                const uint32_t id1 = umma::idesc_f16(128, kC, false, true, true);
                const uint32_t id3 = umma::idesc_f16(128, kC, false, false, false);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    umma::mma(tmem + kColU0 + 64 * b, umma::kmajor(sbase + kSt, 128, s),
                              umma::mnmajor(sbase + (b ? kW1 : kW0), 16384, s), id1, true);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    umma::mma(tmem + kColO, umma::kmajor(sbase + kSt, 128, s),
                              umma::kmajor(sbase + ostk + 64 * 128, 128, s), id3, s > 0);
                umma::commit(bar(1));
            }
            ok = group_all(1, wait(1, ph));
            ph ^= 1u;
            if (!ok) break;

            // U^T -> fp16 K-major tile
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float u32[32];
                umma::tmem_ld32(tmem + lane_base + kColU0 + 64 * b + 32 * hf, u32);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st16(sm + kUt + umma::sw128_offset(Lr, 32 * hf + 8 * u, 128), pack8(u32 + 8 * u));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1);

            // D_S = U^T Kt;  D_O += U^T P^T
            if (tid == 0) {
                umma::fence_after_sync();
                const uint32_t id2 = umma::idesc_f16(128, kD, false, true, false);
                const uint32_t id3 = umma::idesc_f16(128, kC, false, false, false);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColS, umma::kmajor(sbase + kUt, 128, s), umma::mnmajor(sbase + ostk, 16384, s),
                              id2, s > 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s)
                    umma::mma(tmem + kColO, umma::kmajor(sbase + kUt, 128, s),
                              umma::kmajor(sbase + (b ? kP1 : kP0), 64, s), id3, true);
                umma::commit(bar(1));
            }
            ok = group_all(1, wait(1, ph));
            ph ^= 1u;
            if (!ok) break;
            const float gC = vec[b * 256 + 128 + kC - 1];  // gamma over the chunk
            umma::fence_before_sync();
            group_sync(1);
            if (tid == 0) mbar_arrive(bar(4 + b));  // chunk buffers b may be refilled

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
            // o_lin rows of the chunk's queries (positions j + W)
            float* orow = o_lin + ((size_t)(start + j0 + W) * L.Hq + h) * kD + Lr;
            const size_t ostride = (size_t)L.Hq * kD;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float o[32];
                umma::tmem_ld32(tmem + lane_base + kColO + 32 * hf, o);
#pragma unroll
                for (int ii = 0; ii < 32; ++ii)
                    if (32 * hf + ii < nv) orow[(size_t)(32 * hf + ii) * ostride] = o[ii];
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
                               const float* g, const float* beta, const int32_t* cu, const int32_t* chunk_base,
                               const __half* t_in, float* o_lin, float* S_out, int32_t* err, cudaStream_t st) {
    static bool configured = false;  // the attribute is per function
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gdn_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(L.Hq, L.n_seqs);
    gdn_chunked_kernel<<<grid, kThreads, kSmemAlloc, st>>>(L, qhat, khat, vhat, g, beta, cu, chunk_base, t_in,
                                                          o_lin, S_out, err);
    return cudaGetLastError();
}

}  // namespace hla
