// Linear branch, chunked form on the tcgen05 tensor cores.
//
// The GDN recurrence of "迈向线性的关键：分析驱动的 Transformer 线性化" (section
// 线性注意力替换机制, scalar gate) with the delayed, fixed-budget routing of
// section 填补近似缺口的实用设计 (token j enters the state at position j + W)
// is evaluated in chunks of C = 64 absorbed tokens.  With the gates cumulated
// inside the chunk, G_r = sum_{i<=r} g_i, gamma_r = e^{G_r}:
//   A[r,i] = beta_r e^{G_r - G_i} k_r . k_i  (i < r),    T = (I + A)^{-1}
//   U~ = T diag(beta) V,    Wm = T diag(beta gamma) K,   U = U~ - Wm S0
//   O  = diag(gamma) Q S0 + P U,   P[r,i] = e^{G_r - G_i} q_r . k_i (i <= r)
//   S1 = gamma_C S0 + Kt^T U,      Kt = diag(e^{G_C - G}) K
// where the query of token j is qhat at position j + W.  Every product is a
// tcgen05 MMA with fp16 operands in shared memory and fp32 accumulators in
// tensor memory; the state is kept in fp32 registers (its fp16 copy is the
// MMA operand).  All accumulators are laid out with the value dimension (or
// the key dimension for Wm) on the 128 TMEM lanes, so every MMA has M = 128:
//   Gram   D_G[128 x 64]  = [K; Q] K^T
//   D_U    [dv x tok]     = V^T (T diag beta)^T,  then  += S0^T (-Wm^T)
//   D_W    [dk x tok]     = K^T (T diag(beta gamma))^T          (= Wm^T)
//   D_O    [dv x tok]     = S0^T (diag(gamma) Q)^T,  then  += U^T P^T
//   D_S    [dv x dk]      = U^T Kt                             (= (Kt^T U)^T)
// The triangular inverse T is formed on the CUDA cores in fp32 (32 x 32
// diagonal blocks by warp-level forward substitution, then one block merge).
//
// One CTA of 256 threads per (sequence, q-head), head_dim 128.  Thread t owns
// TMEM lane L = 32 (warp % 4) + lane and the column half wg = warp / 4.
#include "hla_common.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kC = 64;          // chunk length (absorbed tokens)
constexpr int kD = 128;         // head dim
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared-memory plan (bytes from a 1024-aligned base)
// The stack and V tiles are double-buffered: chunk c + 1 streams in (cp.async)
// while chunk c is processed.
constexpr uint32_t kStack0 = 0;                // [K ; Q] 128 x 128 fp16, later [Kt ; gamma Q]
constexpr uint32_t kStack1 = 32768;
constexpr uint32_t kVt0 = 65536;               // V (MN-major A), later Wm^T (MN-major B)
constexpr uint32_t kVt1 = 81920;
constexpr uint32_t kP = 98304;                 // P 64 x 64 K-major
constexpr uint32_t kTb = kP + 8192;            // T diag(beta)
constexpr uint32_t kTbg = kTb + 8192;          // T diag(beta gamma)
constexpr uint32_t kSt = kTbg + 8192;          // S0^T 128 x 128 K-major
constexpr uint32_t kUt = kSt + 32768;          // U^T 128 x 64 K-major
constexpr uint32_t kA32 = kUt + 16384;         // A fp32 [64][68]
constexpr uint32_t kT32 = kA32 + 64 * 68 * 4;  // T fp32 [64][68]
constexpr uint32_t kX32 = kT32 + 64 * 68 * 4;  // block product [32][36]
constexpr uint32_t kVec = kX32 + 32 * 36 * 4;  // G (log2 units), beta, gamma, Kt decay: 4 x 64 fp32
constexpr uint32_t kSmemBytes = kVec + 4 * 64 * 4 + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // slack for the 1024-byte alignment

// TMEM columns
constexpr uint32_t kColG = 0, kColW = 64, kColU = 128, kColO = 192, kColS = 256, kTmemCols = 512;

__device__ __forceinline__ void st16(unsigned char* base, uint32_t off, uint4 v) {
    *reinterpret_cast<uint4*>(base + off) = v;
}
__device__ __forceinline__ uint4 ld16(const unsigned char* base, uint32_t off) {
    return *reinterpret_cast<const uint4*>(base + off);
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8(const float* v) {
    return make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
}
__device__ __forceinline__ void unpack8(uint4 u, float* v) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
// 16-byte global -> shared copy that bypasses registers; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(unsigned char* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(umma::smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint4 scale8(uint4 u, float s) {
    float v[8];
    unpack8(u, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= s;
    return pack8(v);
}

// Forward substitution for a 32 x 32 unit lower-triangular diagonal block of
// (I + A): one warp per block, lane l owns row l of the inverse.
__device__ __forceinline__ void invert_diag_block32(const float* sA, float* sT, int b, int l) {
    float a[32], t[32];
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        a[m] = sA[(32 * b + l) * 68 + 32 * b + m];
        t[m] = (m == l) ? 1.f : 0.f;
    }
#pragma unroll
    for (int m = 0; m < 31; ++m) {
        // row m is final once rows 0..m-1 have been folded into it
#pragma unroll
        for (int k = 0; k <= m; ++k) {
            const float tm = __shfl_sync(0xffffffffu, t[k], m);
            if (l > m) t[k] = fmaf(-a[m], tm, t[k]);
        }
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) sT[(32 * b + l) * 68 + 32 * b + m] = t[m];
}

__global__ void __launch_bounds__(kThreads, 1)
gdn_chunked_kernel(LayerDims L, const __half* __restrict__ qhat, const __half* __restrict__ khat,
                   const __half* __restrict__ vhat, const float* __restrict__ g,
                   const float* __restrict__ beta, const int32_t* __restrict__ cu,
                   float* __restrict__ o_lin, float* __restrict__ S_out, int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* sA = reinterpret_cast<float*>(sm + kA32);
    float* sT = reinterpret_cast<float*>(sm + kT32);
    float* sX = reinterpret_cast<float*>(sm + kX32);
    float* sG = reinterpret_cast<float*>(sm + kVec);
    float* sBeta = sG + 64;
    float* sGam = sG + 128;
    float* sKdec = sG + 192;
    uint64_t* mbar_p = reinterpret_cast<uint64_t*>(sm + kVec + 4 * 64 * 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kVec + 4 * 64 * 4 + 8);
    float* scan_carry = reinterpret_cast<float*>(sm + kVec + 4 * 64 * 4 + 16);
    int* abort_flag = reinterpret_cast<int*>(sm + kVec + 4 * 64 * 4 + 20);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
    const int Lr = ((warp & 3) << 5) + lane;            // TMEM lane / row owned
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    const int h = blockIdx.x, n = blockIdx.y, kv = h / L.G, W = L.window;
    const uint32_t sbase = umma::smem_addr(sm);
    const uint32_t mbar = umma::smem_addr(mbar_p);

    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t j_end = len - W;
    const int n_chunks = j_end > L.n_sinks ? (int)((j_end - L.n_sinks + kC - 1) / kC) : 0;

    // ---- set-up: barrier, TMEM, zero state copies
    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
    for (int i = tid; i < 32768 / 16; i += kThreads) st16(sm + kSt, i * 16, make_uint4(0, 0, 0, 0));
    for (int i = tid; i < 64 * 68; i += kThreads) sT[i] = 0.f;
    umma::fence_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    float S[64];  // S0^T[Lr][64 wg .. 64 wg + 63], fp32 master copy
#pragma unroll
    for (int i = 0; i < 64; ++i) S[i] = 0.f;
    uint32_t phase = 0;
    bool ok = true;

    auto wait_mma = [&]() {
        bool done = umma::mbar_wait(mbar, phase, kWaitLimit);
        phase ^= 1u;
        if (!done) {
            *abort_flag = 1;
            if (err) atomicExch(err, kErrTimeout);
        }
        umma::fence_after_sync();
        return __syncthreads_or(!done) == 0;
    };
    auto sync_for_mma = [&]() {  // shared-memory writes -> MMA reads; TMEM reads done
        umma::fence_async_smem();
        umma::fence_before_sync();
        __syncthreads();
    };

    // chunk rows -> (stack, V) buffer `buf` with cp.async; gates -> registers
    float g_next = 0.f, b_next = 0.f;
    auto prefetch = [&](int cc, int buf) {
        const int64_t pj0 = L.n_sinks + (int64_t)cc * kC;
        const int pnv = (int)min((int64_t)kC, j_end - pj0);
        unsigned char* stk = sm + (buf ? kStack1 : kStack0);
        unsigned char* vt = sm + (buf ? kVt1 : kVt0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = tid + kThreads * u, r = e >> 4, c8 = (e & 15) * 8;
            const uint32_t nb = r < pnv ? 16u : 0u;
            const size_t t = (size_t)(start + pj0 + (r < pnv ? r : 0));
            cp_async16(stk + umma::sw128_offset(r, c8, 128), khat + (t * L.Hkv + kv) * kD + c8, nb);
            cp_async16(stk + umma::sw128_offset(64 + r, c8, 128), qhat + ((t + W) * L.Hq + h) * kD + c8, nb);
            cp_async16(vt + umma::sw128_offset(r, c8, 64), vhat + (t * L.Hkv + kv) * kD + c8, nb);
        }
        cp_async_commit();
        if (tid < kC) {
            const size_t t = (size_t)(start + pj0 + tid);
            g_next = tid < pnv ? g[t * L.Hq + h] : 0.f;
            b_next = tid < pnv ? beta[t * L.Hq + h] : 0.f;
        }
    };
    if (n_chunks > 0) prefetch(0, 0);

    for (int c = 0; c < n_chunks && ok; ++c) {
        const int64_t j0 = L.n_sinks + (int64_t)c * kC;
        const int nv = (int)min((int64_t)kC, j_end - j0);
        const uint32_t oStk = (c & 1) ? kStack1 : kStack0;
        const uint32_t oVt = (c & 1) ? kVt1 : kVt0;

        // ---- 1. gates of the chunk: G (inclusive cumsum), beta, gamma, Kt decay
        float gcum = 0.f;
        if (tid < kC) {
            float gi = g_next * 1.4426950408889634f;  // log2 units
            sBeta[tid] = b_next;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float y = __shfl_up_sync(0xffffffffu, gi, o);
                if (lane >= o) gi += y;
            }
            gcum = gi;
            if (tid == 31) *scan_carry = gi;
        }
        __syncthreads();
        if (tid < kC) {
            if (tid >= 32) gcum += *scan_carry;
            sG[tid] = gcum;
        }
        __syncthreads();
        if (tid < kC) {
            sGam[tid] = exp2f(sG[tid]);
            sKdec[tid] = exp2f(sG[kC - 1] - sG[tid]);
        }

        // ---- 2. this chunk's rows have streamed into (stack, V)[c % 2]; start the next
        cp_async_wait_all();
        if (c + 1 < n_chunks) prefetch(c + 1, (c + 1) & 1);
        sync_for_mma();

        // ---- 3. Gram: D_G = [K; Q] K^T
        if (tid == 0) {
            umma::fence_after_sync();
            const uint32_t id = umma::idesc_f16(128, 64, false, false, false);
#pragma unroll
            for (int s = 0; s < kD / 16; ++s)
                umma::mma(tmem + kColG, umma::kmajor(sbase + oStk, 128, s),
                          umma::kmajor(sbase + oStk, 128, s), id, s > 0);
            umma::commit(mbar);
        }
        if (!(ok = wait_mma())) break;

        // ---- 4. A (rows of K K^T) into fp32 smem, P (rows of Q K^T) into its fp16 tile
        {
            float d[32];
            umma::tmem_ld32(tmem + lane_base + kColG + 32 * wg, d);
            if (Lr < 64) {
                const int r = Lr;
                const float br = sBeta[r], gr = sG[r];
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * wg + ii;
                    sA[r * 68 + i] = (i < r) ? br * exp2f(gr - sG[i]) * d[ii] : 0.f;
                }
            } else {
                const int r = Lr - 64;
                const float gr = sG[r];
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * wg + ii;
                    d[ii] = (i <= r) ? exp2f(gr - sG[i]) * d[ii] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st16(sm + kP, umma::sw128_offset(r, 32 * wg + 8 * u, 64), pack8(d + 8 * u));
            }
        }
        umma::fence_before_sync();
        __syncthreads();

        // ---- 5. T = (I + A)^{-1}: two 32 x 32 diagonal blocks by forward
        // substitution, then T10 = -T11 (A10 T00)
        if (warp < 2) invert_diag_block32(sA, sT, warp, lane);
        __syncthreads();
        {
            const int i = tid >> 3, j0c = (tid & 7) * 4;
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = j0c; k < 32; ++k) {  // T00 is lower triangular
                const float a = sA[(32 + i) * 68 + k];
                const float4 t4 = *reinterpret_cast<const float4*>(&sT[k * 68 + j0c]);
                x[0] = fmaf(a, t4.x, x[0]); x[1] = fmaf(a, t4.y, x[1]);
                x[2] = fmaf(a, t4.z, x[2]); x[3] = fmaf(a, t4.w, x[3]);
            }
            *reinterpret_cast<float4*>(&sX[i * 36 + j0c]) = make_float4(x[0], x[1], x[2], x[3]);
            __syncthreads();
            float y[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k <= i; ++k) {  // T11 is lower triangular
                const float t = sT[(32 + i) * 68 + 32 + k];
                const float4 x4 = *reinterpret_cast<const float4*>(&sX[k * 36 + j0c]);
                y[0] = fmaf(t, x4.x, y[0]); y[1] = fmaf(t, x4.y, y[1]);
                y[2] = fmaf(t, x4.z, y[2]); y[3] = fmaf(t, x4.w, y[3]);
            }
            *reinterpret_cast<float4*>(&sT[(32 + i) * 68 + j0c]) = make_float4(-y[0], -y[1], -y[2], -y[3]);
            __syncthreads();
        }

        // ---- 6. T diag(beta) and T diag(beta gamma) as fp16 K-major tiles
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = tid + kThreads * u, r = e >> 3, cc = (e & 7) * 8;
            float tb[8], tbg[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float t = sT[r * 68 + cc + x];
                tb[x] = t * sBeta[cc + x];
                tbg[x] = tb[x] * sGam[cc + x];
            }
            st16(sm + kTb, umma::sw128_offset(r, cc, 64), pack8(tb));
            st16(sm + kTbg, umma::sw128_offset(r, cc, 64), pack8(tbg));
        }
        sync_for_mma();

        // ---- 7. D_U = V^T (T diag beta)^T;  D_W = K^T (T diag(beta gamma))^T
        if (tid == 0) {
            umma::fence_after_sync();
            const uint32_t id = umma::idesc_f16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < kC / 16; ++s)
                umma::mma(tmem + kColU, umma::mnmajor(sbase + oVt, 8192, s), umma::kmajor(sbase + kTb, 64, s), id,
                          s > 0);
#pragma unroll
            for (int s = 0; s < kC / 16; ++s)
                umma::mma(tmem + kColW, umma::mnmajor(sbase + oStk, 16384, s), umma::kmajor(sbase + kTbg, 64, s),
                          id, s > 0);
            umma::commit(mbar);
        }
        if (!(ok = wait_mma())) break;

        // ---- 8. Wm^T -> MN-major tile (over V); K -> Kt and Q -> gamma Q in place
        {
            float w[32];
            umma::tmem_ld32(tmem + lane_base + kColW + 32 * wg, w);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                st16(sm + oVt, umma::sw128_offset(Lr, 32 * wg + 8 * u, 128), pack8(w + 8 * u));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = tid + kThreads * u, row = e >> 4, cc = (e & 15) * 8;
            const uint32_t off = umma::sw128_offset(row, cc, 128);
            const float s = row < 64 ? sKdec[row] : sGam[row - 64];
            st16(sm + oStk, off, scale8(ld16(sm + oStk, off), s));
        }
        sync_for_mma();

        // ---- 9. D_U += S0^T (-Wm^T);  D_O = S0^T (gamma Q)^T
        if (tid == 0) {
            umma::fence_after_sync();
            const uint32_t id1 = umma::idesc_f16(128, 64, false, true, true);
            const uint32_t id3 = umma::idesc_f16(128, 64, false, false, false);
#pragma unroll
            for (int s = 0; s < kD / 16; ++s)
                umma::mma(tmem + kColU, umma::kmajor(sbase + kSt, 128, s), umma::mnmajor(sbase + oVt, 16384, s), id1,
                          true);
#pragma unroll
            for (int s = 0; s < kD / 16; ++s)
                umma::mma(tmem + kColO, umma::kmajor(sbase + kSt, 128, s),
                          umma::kmajor(sbase + oStk + 64 * 128, 128, s), id3, s > 0);
            umma::commit(mbar);
        }
        if (!(ok = wait_mma())) break;

        // ---- 10. U^T -> fp16 K-major tile
        {
            float u32[32];
            umma::tmem_ld32(tmem + lane_base + kColU + 32 * wg, u32);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                st16(sm + kUt, umma::sw128_offset(Lr, 32 * wg + 8 * u, 128), pack8(u32 + 8 * u));
        }
        sync_for_mma();

        // ---- 11. D_S = U^T Kt;  D_O += U^T P^T
        if (tid == 0) {
            umma::fence_after_sync();
            const uint32_t id2 = umma::idesc_f16(128, 128, false, true, false);
            const uint32_t id3 = umma::idesc_f16(128, 64, false, false, false);
#pragma unroll
            for (int s = 0; s < kC / 16; ++s)
                umma::mma(tmem + kColS, umma::kmajor(sbase + kUt, 128, s), umma::mnmajor(sbase + oStk, 16384, s), id2,
                          s > 0);
#pragma unroll
            for (int s = 0; s < kC / 16; ++s)
                umma::mma(tmem + kColO, umma::kmajor(sbase + kUt, 128, s), umma::kmajor(sbase + kP, 64, s), id3, true);
            umma::commit(mbar);
        }
        if (!(ok = wait_mma())) break;

        // ---- 12. S <- gamma_C S + dS (fp32 registers, fp16 copy for the next chunk); o_lin rows
        {
            const float gC = sGam[kC - 1];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float ds[32];
                umma::tmem_ld32(tmem + lane_base + kColS + 64 * wg + 32 * half, ds);
#pragma unroll
                for (int i = 0; i < 32; ++i) S[32 * half + i] = fmaf(gC, S[32 * half + i], ds[i]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st16(sm + kSt, umma::sw128_offset(Lr, 64 * wg + 8 * u, 128), pack8(S + 8 * u));
            float o[32];
            umma::tmem_ld32(tmem + lane_base + kColO + 32 * wg, o);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const int tok = 32 * wg + ii;
                if (tok < nv) o_lin[((size_t)(start + j0 + tok + W) * L.Hq + h) * kD + Lr] = o[ii];
            }
        }
        sync_for_mma();
    }

    if (ok && S_out) {
        float* dst = S_out + ((size_t)n * L.Hq + h) * kD * kD;
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[(size_t)(64 * wg + i) * kD + Lr] = S[i];
    }
    if (!ok && tid == 0) {
        // give in-flight MMAs a bounded chance to drain before TMEM is released
        umma::mbar_wait(mbar, phase ^ 1u, kWaitLimit);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gdn_chunked(const LayerDims& L, const __half* qhat, const __half* khat, const __half* vhat,
                               const float* g, const float* beta, const int32_t* cu, float* o_lin,
                               float* S_out, int32_t* err, cudaStream_t st) {
    static bool configured = false;  // per process; the attribute is per function
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gdn_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemAlloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(L.Hq, L.n_seqs);
    gdn_chunked_kernel<<<grid, kThreads, kSmemAlloc, st>>>(L, qhat, khat, vhat, g, beta, cu, o_lin, S_out, err);
    return cudaGetLastError();
}

namespace {

}  // namespace

}  // namespace hla
