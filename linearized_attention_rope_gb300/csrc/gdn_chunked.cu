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
// left), so a CTA owns one 64-column slice of the value dims of one
// (sequence, q-head) state: two CTAs share a head and the state chains run
// on twice as many SMs.  With the chunk rows stacked on the 128 TMEM lanes
// every MMA has M = 128 and N = 64:
//   D1[b] = [-Wm ; Q] S0  +  [T diag(beta) ; 0] V      rows 0..63 = U, 64..127 = Q S0
//   D2[b] = [0 ; P] U                                   rows 64..127 = P U
//   DS    = K^T diag(e^{G_C - G}) U                     (key dims on the lanes)
// fp16 operands in shared memory, fp32 accumulators in TMEM; the zero blocks
// pad the 64-row operands to M = 128.  S0, V, U are MN-major B operands (one
// 128-byte row per key dim or token), so every epilogue thread writes its
// own row.  S0 stays in fp32 registers (32 columns of a key row per thread) and is
// re-rounded to fp16 for the next chunk's MMA.
//
// Roles (384 threads; the rest of warps 8-9 idle).  One thread of warp 8 loads chunk c+2 into the buffer
// of chunk c (TMA: tensor copies of the query, key and value rows, bulk copies of the record), each of
// three groups as soon as chunk c is done with its region (T diag(beta) and V once its V product
// completed, [-Wm ; Q] once its D1 product completed, P, K and the gate vectors once it was released),
// and queues chunk c+1's S-independent D1 = [T diag(beta) ; 0] V right after chunk c's D1 product, so
// the tensor pipe runs it while the chain forms U.  Warps 0-7 run the chain (warps w and w + 4 on the
// same TMEM lanes, each with half of the slice's columns): D1 += [-Wm ; Q] S0, the U epilogue, DS, the S
// epilogue.  One thread of warp 9 queues D2 behind DS.  Warps 10-11 turn the
// double-buffered D1/D2 rows 64..127 into the layer output of their positions:
// out = o_sm + lambda_h (gamma Q S0 + P U), o_sm being the normalised softmax branch the softmax kernel
// left for these rows.  Handoffs use mbarriers: loadedv[b] and loaded[b] (TMA bytes of the V product's
// operands and of the rest), ready[b] (the V product's commit and the loader's arrival once every byte is
// in -> chain and load), d1done[b] (the chain's D1 MMAs -> load), dsqueued[b] (chain -> D2 issue),
// free[b] (chain + output -> load), ofull[b] (D2 -> output).  Token rows past a chunk's end hold
// whatever follows (zeros past the tensor): they meet zero rows of -Wm, T diag(beta) and U, or produce
// output rows that are not stored.  Every wait has an iteration limit; on expiry the kernel records a
// timeout in the error word and all roles stop.  Loops stay rolled where registers allow: the whole
// kernel is executed once per chunk by every role, and compact code keeps it resident in the instruction
// cache.
#include "hla_common.cuh"
#include "tma.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kC = kGdnChunk;  // chunk length (absorbed tokens)
constexpr int kD = 128;   // head dim
constexpr int kNS = 64;   // value columns per CTA
constexpr int kSlices = kD / kNS;
constexpr int kThreads = 384;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared-memory plan (bytes from a 1024-aligned base); one chunk buffer:
constexpr uint32_t kA1 = 0;         // [-Wm ; Q] 128 x 128, K-major
constexpr uint32_t kTZP = 32768;    // [T diag(beta) | 0 | P], three 64 x 64 K-major images
constexpr uint32_t kK = 57344;      // K rows 64 x 128 (MN-major A of DS)
constexpr uint32_t kV = 73728;      // V slice rows 64 x 64 (MN-major B)
constexpr uint32_t kVec = 81920;    // gamma[64], key decay[64]
constexpr uint32_t kBuf = 82944;
// chain operands
constexpr uint32_t kS = 2 * kBuf;   // S0 slice rows 128 x 64 (MN-major B)
constexpr uint32_t kU = kS + 16384;     // U slice rows 64 x 64 (MN-major B), one per buffer
constexpr uint32_t kUk = kU + 2 * 8192;  // diag(key decay) U
constexpr uint32_t kBar = kUk + 8192;
constexpr uint32_t kSmemAlloc = kBar + 256 + 1024;
// TMEM columns
constexpr uint32_t kColD1 = 0, kColD2 = 128, kColS = 256, kTmemCols = 512;

// mbarrier indices
constexpr int kReady = 0, kFree = 2, kMma1 = 4, kMma2 = 5, kOFull = 6, kLoaded = 8, kD1Done = 10, kLoadedV = 12,
              kDsQueued = 14, kNumBars = 16;
static_assert(8 * kNumBars + 8 + 32 + 4 <= 256,
              "barrier area: mbarriers, TMEM base, abort flag, 2 slots x 4 ids, the CTA's sequence");
constexpr int kMaxRankedSeqs = 64;  // up to this many sequences, the grid takes them longest first
constexpr uint32_t kLoadBytes = kRecordBytes + 5 * 8192;  // record + query, key rows (2 boxes each) + value slice
constexpr uint32_t kLoadVBytes = 2 * 8192;                // T diag(beta) + value slice (the V product's operands)

__device__ __forceinline__ void st16(unsigned char* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8(const float* v, float s) {
    return make_uint4(pack_h2(v[0] * s, v[1] * s), pack_h2(v[2] * s, v[3] * s), pack_h2(v[4] * s, v[5] * s),
                      pack_h2(v[6] * s, v[7] * s));
}
// barrier among the `count` threads of one role (ids 1-3; 0 is __syncthreads)
__device__ __forceinline__ void group_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}

// Descriptor offsets (address field, 16-byte units) of K step s: a 128-row
// K-major tile advances 32 B inside a 64-column block and 16 KB per block;
// an MN-major tile advances 16 rows = 2 KB.
__device__ __forceinline__ uint64_t kstep128(int s) { return (uint64_t)((s >> 2) * 1024 + (s & 3) * 2); }
__device__ __forceinline__ uint64_t mnstep(int s) { return (uint64_t)(s * 128); }

__global__ void __launch_bounds__(kThreads, 1)
gdn_chunked_kernel(LayerDims L, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const int32_t* __restrict__ cu,
                   const int32_t* __restrict__ chunk_base, int slot_lo, int slot_hi,
                   const unsigned char* __restrict__ rec_in, const __half* __restrict__ o_sm,
                   const float* __restrict__ lambda, __nv_bfloat16* __restrict__ out,
                   const float* __restrict__ S_in, const float* __restrict__ S_init, float* __restrict__ S_out,
                   int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    // A launch that follows this one with programmatic stream serialization (the next part's chunk-local
    // kernel) may start as soon as every CTA of this grid has reached this point, i.e. is resident, even
    // before the wait below: it reads only what the features and table launches wrote, which completed
    // before the chunk-local launch this one waits for started.  No effect on a plain launch.
    pdl_trigger();
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kBar + 8 * kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kBar + 8 * kNumBars + 4);
    volatile int* decision = reinterpret_cast<volatile int*>(sm + kBar + 8 * kNumBars + 8);  // [role id][2]
    volatile int* seq_slot = reinterpret_cast<volatile int*>(sm + kBar + 8 * kNumBars + 40);

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    const int h = blockIdx.x / kSlices, slice = blockIdx.x % kSlices;
    // The CTA's sequence: row y of the grid takes the sequence of rank y by length, longest first (ties in
    // index order), so that with sequences of mixed lengths the longest chains start in the first wave of
    // CTAs (the rows are placed in order) rather than behind shorter ones.  The ranking reads only
    // cu_seqlens, an input of the call, so it runs before the wait for the launch before this one.
    if (L.n_seqs <= kMaxRankedSeqs) {
        for (int q = tid; q < L.n_seqs; q += kThreads) {
            int64_t qs, ql;
            seq_range(cu, q, L.total, &qs, &ql);
            int rank = 0;
            for (int o = 0; o < L.n_seqs; ++o) {
                int64_t os, ol;
                seq_range(cu, o, L.total, &os, &ol);
                rank += (ol > ql || (ol == ql && o < q)) ? 1 : 0;
            }
            if (rank == (int)blockIdx.y) *seq_slot = q;  // exactly one sequence has each rank
        }
    } else if (tid == 0) {
        *seq_slot = blockIdx.y;
    }
    const int kv = h / L.G, W = L.window;
    const uint32_t sbase = umma::smem_addr(sm);
    const uint32_t bar0 = umma::smem_addr(sm + kBar);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i)
            umma::mbar_init(bar(i), (i == kFree || i == kFree + 1 || i == kReady || i == kReady + 1) ? 2 : 1);
        umma::fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
#pragma unroll 1
    for (int i = tid; i < 16384 / 16; i += kThreads) st16(sm + kS + 16 * i, make_uint4(0, 0, 0, 0));
#pragma unroll 1
    for (int i = tid; i < 2 * 512; i += kThreads)  // the zero blocks of both buffers
        st16(sm + (i >> 9) * kBuf + kTZP + 8192 + 16 * (i & 511), make_uint4(0, 0, 0, 0));
    umma::fence_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int n = *seq_slot;
    // Launched with programmatic stream serialization, the CTAs get here while the launch before this
    // one (the chunk-local kernel) may still run: wait for it to complete, and its writes (and those of
    // every launch before it) to be visible, before the first global read.  No effect on a plain launch.
    pdl_wait();

    int64_t start, len;
    seq_range(cu, n, L.total, &start, &len);
    const int64_t j_end = len - W;
    const int seq_chunks = j_end > L.n_sinks ? (int)((j_end - L.n_sinks + kC - 1) / kC) : 0;
    const int slot0 = __ldg(chunk_base + n);
    // this launch: the sequence's chunks c_lo .. c_lo + n_chunks - 1 (those in slots [slot_lo, slot_hi)),
    // loop index c = chunk - c_lo
    const int c_lo = min(max(slot_lo - slot0, 0), seq_chunks);
    const int n_chunks = min(max(slot_hi - slot0, 0), seq_chunks) - c_lo;
    // continue from the state the previous launch left, or (a sequence's first chunks) from S_init
    const float* S_src = c_lo > 0 ? S_in : S_init;
    const bool resume = S_src != nullptr;

    // The stall test hook: the loader issues nothing, so every wait below runs out (after a millisecond
    // instead of the usual two seconds) and the kernel reports a timeout without any copy or MMA in flight.
    const bool stall = (L.flags & HLA_FLAG_TEST_STALL) != 0;
    const uint64_t wait_ns = stall ? 1000000ull : 2000000000ull;

    // One leader per role polls the mbarrier (an inline try first, the bounded
    // loop only if the phase is still open) and posts the outcome in a shared
    // slot; the role (`count` threads on named barrier `id`; 0 for a one-thread
    // role) then meets on the barrier and every thread reads the same outcome,
    // so all take the same branch, and fences before touching the results.  The
    // two slots of a role alternate (counter k), so a slot is rewritten only
    // after the whole role has passed the barrier in between.
    auto role_wait = [&](int i, uint32_t parity, int id, int count, bool leader, int& k) -> bool {
        bool w = true;
        if (leader) {
            w = !*abort_flag &&
                (umma::mbar_try_wait(bar(i), parity) || umma::mbar_wait(bar(i), parity, kWaitLimit, wait_ns));
            if (!w) {
                *abort_flag = 1;
                if (err) atomicExch(err, kErrTimeout);
            }
            if (count) decision[2 * id + (k & 1)] = w;
        }
        if (count) {
            group_sync(id, count);
            w = decision[2 * id + (k & 1)] != 0;
            ++k;
        }
        umma::fence_after_sync();
        return w;
    };

    if (warp < 8) {
        // ================= the state chain =================
        // key row `row` (the thread's TMEM lane), value columns col0 .. col0 + 31 of the slice: warps w and
        // w + 4 share a lane quarter and split its columns
        const int row = tid & 127, col0 = 32 * (warp >> 2);
        float S[32];  // S0[row][col0 ..]: fp32 master copy
#pragma unroll
        for (int i = 0; i < 32; ++i) S[i] = 0.f;
        if (resume) {  // the saved state and its fp16 image (the zero image above is overwritten)
            const float* src = S_src + (((size_t)n * L.Hq + h) * kD + row) * kD + slice * kNS + col0;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + i);
                S[i] = x.x; S[i + 1] = x.y; S[i + 2] = x.z; S[i + 3] = x.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st16(sm + kS + umma::sw128_offset(row, col0 + 8 * j, 128), pack8(S + 8 * j, 1.f));
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1, 256);
        }
        const uint32_t id_b = umma::idesc_f16(128, kNS, false, true, false);
        const uint32_t id_ab = umma::idesc_f16(128, kNS, true, true, false);
        uint32_t ph1 = 0, ph2 = 0;
        int kr = 0;
        bool ok = true;
#pragma unroll 1
        for (int c = 0; c < n_chunks && ok; ++c) {
            const int b = c & 1;
            const uint32_t buf = (uint32_t)b * kBuf;
            // ready[b]: the chunk is loaded and D1[b] holds [T diag(beta) ; 0] V; the
            // loader waited for free[b], so the output rows of chunk c - 2 are out of D1/D2[b]
            if (!(ok = role_wait(kReady + b, (uint32_t)((c >> 1) & 1), 1, 256, tid == 0, kr))) break;
            const uint32_t ub = kU + (uint32_t)b * 8192u;  // this chunk's U image

            // D1[b] += [-Wm ; Q] S0
            if (tid == 0) {
                const uint32_t d1 = tmem + kColD1 + kNS * b;
                const uint64_t a1 = umma::kmajor(sbase + buf + kA1, 128, 0), bs = umma::mnmajor(sbase + kS, 8192u, 0);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) umma::mma(d1, a1 + kstep128(s), bs + mnstep(s), id_b, true);
                umma::commit(bar(kMma1));
                umma::commit(bar(kD1Done + b));
            }
            if (!(ok = role_wait(kMma1, ph1, 1, 256, tid == 0, kr))) break;
            ph1 ^= 1u;

            // U (rows 0..63) -> fp16 rows of U and diag(key decay) U
            if (row < kC) {
                const float kd = reinterpret_cast<const float*>(sm + buf + kVec)[kC + row];
                uint32_t u[32];
                umma::tmem_ld32_async(tmem + lane_base + kColD1 + kNS * b + col0, u);
                umma::tmem_wait_ld();
                umma::reg_fence32(u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(u[8 * j + e]);
                    const uint32_t off = umma::sw128_offset(row, col0 + 8 * j, 64);
                    st16(sm + ub + off, pack8(x, 1.f));
                    st16(sm + kUk + off, pack8(x, kd));
                }
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            group_sync(1, 256);

            // DS = K^T diag(key decay) U, which the chain waits for; the output role queues D2[b] = [0 ; P] U
            // behind it
            if (tid == 0) {
                umma::fence_after_sync();
                const uint64_t ak = umma::mnmajor(sbase + buf + kK, 8192u, 0), buk = umma::mnmajor(sbase + kUk, 8192u, 0);
#pragma unroll
                for (int s = 0; s < kC / 16; ++s) umma::mma(tmem + kColS, ak + mnstep(s), buk + mnstep(s), id_ab, s > 0);
                umma::commit(bar(kMma2));
                mbar_arrive(bar(kDsQueued + b));
            }
            const float gC = reinterpret_cast<const float*>(sm + buf + kVec)[kC - 1];  // gamma_C
            if (!(ok = role_wait(kMma2, ph2, 1, 256, tid == 0, kr))) break;
            ph2 ^= 1u;
            // the chain is done with buffer b (every thread read gamma_C before the wait's barrier; D2's reads
            // of the buffer end before the output role arrives)
            if (tid == 0) mbar_arrive(bar(kFree + b));

            // S <- gamma_C S + DS; fp16 row for the next chunk
            {
                uint32_t ds[32];
                umma::tmem_ld32_async(tmem + lane_base + kColS + col0, ds);
                umma::tmem_wait_ld();
                umma::reg_fence32(ds);
#pragma unroll
                for (int i = 0; i < 32; ++i) S[i] = fmaf(gC, S[i], __uint_as_float(ds[i]));
#pragma unroll
                for (int j = 0; j < 4; ++j) st16(sm + kS + umma::sw128_offset(row, col0 + 8 * j, 128), pack8(S + 8 * j, 1.f));
            }
            // the barrier of the next chunk's ready wait orders these rows before its D1 MMAs
            umma::fence_async_smem();
            umma::fence_before_sync();
        }
        if (ok && S_out) {
            float* dst = S_out + (((size_t)n * L.Hq + h) * kD + row) * kD + slice * kNS + col0;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
        }
    } else if (tid == 256) {
        // ================= loads, one chunk ahead of the V products (one thread) =================
        // Iteration c: chunk c's T diag(beta) and V (once chunk c - 2's V product completed) and [-Wm ; Q]
        // (once its D1 product completed); chunk c - 1's V product, after chunk c - 2's D1 product so that
        // it runs while the chain forms U; chunk c - 1 released to the chain once all its bytes are in
        // (ready[b] takes the V product's commit and that arrival); then chunk c's P, gate vectors and key
        // rows once chunk c - 2 was released by the chain and the output role (which also frees D1/D2 of
        // the buffer in TMEM).
        const uint32_t id_b = umma::idesc_f16(128, kNS, false, true, false);
        int kl = 0;  // (unused by one-thread waits)
        auto loads_early = [&](int c) -> bool {
            const int b = c & 1;
            const uint32_t buf = sbase + (uint32_t)b * kBuf, ld = bar(kLoaded + b), ldv = bar(kLoadedV + b);
            const uint32_t prev = (uint32_t)(((c - 2) >> 1) & 1);  // phase of chunk c - 2 (same buffer)
            const int tok = (int)(start + L.n_sinks + (int64_t)(c_lo + c) * kC);  // first absorbed token
            const unsigned char* rec = rec_in + ((size_t)(slot0 + c_lo + c) * L.Hq + h) * kRecordBytes;
            if (c >= 2 && !role_wait(kReady + b, prev, 0, 0, true, kl)) return false;
            tma::expect_tx(ldv, kLoadVBytes);
            tma::bulk_load(buf + kTZP, rec + kRecTb, 8192, ldv);
            tma::tensor_load_3d(buf + kV, &map_v, slice * kNS, kv, tok, ldv);
            if (c >= 2 && !role_wait(kD1Done + b, prev, 0, 0, true, kl)) return false;
            tma::expect_tx(ld, kLoadBytes - kLoadVBytes);
            tma::bulk_load(buf + kA1, rec + kRecWm, 8192, ld);                   // -Wm, key dims 0..63
            tma::bulk_load(buf + kA1 + 16384, rec + kRecWm + 8192, 8192, ld);    // key dims 64..127
            tma::tensor_load_3d(buf + kA1 + 8192, &map_q, 0, h, tok + W, ld);    // query rows (positions j + W)
            tma::tensor_load_3d(buf + kA1 + 16384 + 8192, &map_q, 64, h, tok + W, ld);
            return true;
        };
        auto loads_late = [&](int c) -> bool {
            const int b = c & 1;
            const uint32_t buf = sbase + (uint32_t)b * kBuf, ld = bar(kLoaded + b);
            const int tok = (int)(start + L.n_sinks + (int64_t)(c_lo + c) * kC);
            const unsigned char* rec = rec_in + ((size_t)(slot0 + c_lo + c) * L.Hq + h) * kRecordBytes;
            if (c >= 2 && !role_wait(kFree + b, (uint32_t)(((c - 2) >> 1) & 1), 0, 0, true, kl)) return false;
            tma::bulk_load(buf + kTZP + 16384, rec + kRecP, 8192, ld);
            tma::bulk_load(buf + kVec, rec + kRecVec, kRecordBytes - kRecVec, ld);
            tma::tensor_load_3d(buf + kK, &map_k, 0, kv, tok, ld);
            tma::tensor_load_3d(buf + kK + 8192, &map_k, 64, kv, tok, ld);
            return true;
        };
        // D1[b] = [T diag(beta) ; 0] V, committed to ready[b]; then, once every byte of the chunk is in,
        // ready[b]'s other arrival
        auto start_chunk = [&](int c) -> bool {
            const int b = c & 1;
            const uint32_t buf = sbase + (uint32_t)b * kBuf, par = (uint32_t)((c >> 1) & 1);
            if (!role_wait(kLoadedV + b, par, 0, 0, true, kl)) return false;
            if (c >= 1 && !role_wait(kD1Done + (b ^ 1), (uint32_t)(((c - 1) >> 1) & 1), 0, 0, true, kl)) return false;
            const uint64_t tb = umma::kmajor(buf + kTZP, 128, 0), bv = umma::mnmajor(buf + kV, 8192u, 0);
#pragma unroll
            for (int s = 0; s < kC / 16; ++s) umma::mma(tmem + kColD1 + kNS * b, tb + kstep128(s), bv + mnstep(s), id_b, s > 0);
            umma::commit(bar(kReady + b));
            if (!role_wait(kLoaded + b, par, 0, 0, true, kl)) return false;
            mbar_arrive(bar(kReady + b));
            return true;
        };
        const int n_load = stall ? 0 : n_chunks;
#pragma unroll 1
        for (int c = 0; c <= n_load; ++c) {
            if (c < n_load && !loads_early(c)) break;
            if (c >= 1 && !start_chunk(c - 1)) break;
            if (c < n_load && !loads_late(c)) break;
        }
    } else if (tid == 288) {
        // ================= D2[b] = [0 ; P] U (one thread) =================
        // queued once the chain has queued its DS, so it runs behind DS, beside the S epilogue.  D2[b] in TMEM
        // was read out for chunk c - 2 and U[b] is rewritten for chunk c + 2 only: the chain starts a chunk
        // once its last load group is in, which waits for the output role to release the chunk two back.
        const uint32_t id_b = umma::idesc_f16(128, kNS, false, true, false);
        int kq = 0;  // (unused by one-thread waits)
#pragma unroll 1
        for (int c = 0; c < n_chunks; ++c) {
            const int b = c & 1;
            if (!role_wait(kDsQueued + b, (uint32_t)((c >> 1) & 1), 0, 0, true, kq)) break;
            const uint64_t zp = umma::kmajor(sbase + (uint32_t)b * kBuf + kTZP + 8192, 128, 0);
            const uint64_t bu = umma::mnmajor(sbase + kU + (uint32_t)b * 8192u, 8192u, 0);
#pragma unroll
            for (int s = 0; s < kC / 16; ++s) umma::mma(tmem + kColD2 + kNS * b, zp + kstep128(s), bu + mnstep(s), id_b, s > 0);
            umma::commit(bar(kOFull + b));
        }
    } else if (warp >= 10) {
        // ================= output rows: o_sm + lambda_h (gamma (Q S0) + P U) =================
        const int r = tid - 320;  // chunk row; TMEM lane 64 + r
        const bool emit = out && !(L.flags & HLA_FLAG_LINEAR_OFF);
        const float lam = __ldg(lambda + h);
        int ko = 0;
#pragma unroll 1
        for (int c = 0; c < n_chunks; ++c) {
            const int b = c & 1;
            if (!role_wait(kOFull + b, (uint32_t)((c >> 1) & 1), 3, 64, r == 0, ko)) break;
            const float gr = reinterpret_cast<const float*>(sm + b * kBuf + kVec)[r] * lam;
            // lambda o_lin of this row into registers, then release the chunk buffer and D1/D2[b]
            float o[kNS];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float d1[32], d2[32];
                umma::tmem_ld32(tmem + lane_base + kColD1 + kNS * b + 32 * q, d1);
                umma::tmem_ld32(tmem + lane_base + kColD2 + kNS * b + 32 * q, d2);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[32 * q + i] = fmaf(gr, d1[i], lam * d2[i]);
            }
            umma::fence_before_sync();
            group_sync(3, 64);
            if (r == 0) mbar_arrive(bar(kFree + b));
            const int64_t j0 = L.n_sinks + (int64_t)(c_lo + c) * kC;
            if (emit && r < j_end - j0) {
                const size_t base = ((size_t)(start + j0 + r + W) * L.Hq + h) * kD + slice * kNS;
#pragma unroll
                for (int i = 0; i < kNS; i += 8) {
                    const uint4 sv = *reinterpret_cast<const uint4*>(o_sm + base + i);
                    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
                    uint32_t ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&sw[e]));
                        const __nv_bfloat162 o2 = __floats2bfloat162_rn(f.x + o[i + 2 * e], f.y + o[i + 2 * e + 1]);
                        ow[e] = *reinterpret_cast<const uint32_t*>(&o2);
                    }
                    *reinterpret_cast<uint4*>(out + base + i) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                }
            }
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gdn_chunked(const LayerDims& L, const __half* qhat, const __half* khat, const __half* vhat,
                               const int32_t* cu, const int32_t* chunk_base, int slot_lo, int slot_hi,
                               const unsigned char* rec_in, const __half* o_sm, const float* lambda,
                               __nv_bfloat16* out, const float* S_in, const float* S_init, float* S_out, int32_t* err,
                               bool beside_prior, cudaStream_t st) {
    static DeviceCache cache;  // the shared-memory attribute, per device
    cudaError_t e = device_cached(cache, nullptr, [](int, int*) {
        return cudaFuncSetAttribute(gdn_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    });
    if (e != cudaSuccess) return e;
    if (L.total <= 0)  // no token anywhere: the final states are zero
        return S_out ? cudaMemsetAsync(S_out, 0, (size_t)L.n_seqs * L.Hq * kD * kD * sizeof(float), st) : cudaSuccess;
    CUtensorMap mq, mk, mv;
    if (!tma::make_map_f16_3d(&mq, qhat, kD, (uint64_t)L.Hq, (uint64_t)L.total) ||
        !tma::make_map_f16_3d(&mk, khat, kD, (uint64_t)L.Hkv, (uint64_t)L.total) ||
        !tma::make_map_f16_3d(&mv, vhat, kD, (uint64_t)L.Hkv, (uint64_t)L.total))
        return cudaErrorInvalidValue;
    LaunchCfg lc(dim3(L.Hq * kSlices, L.n_seqs), dim3(kThreads), kSmemAlloc, st, beside_prior);
    return cudaLaunchKernelEx(&lc.cfg, gdn_chunked_kernel, L, mq, mk, mv, cu, chunk_base, slot_lo, slot_hi, rec_in, o_sm,
                              lambda, out, S_in, S_init, S_out, err);
}

}  // namespace hla
