// Exact branch on the tcgen05 tensor cores: softmax over the sink tokens plus
// the sliding window ("迈向线性的关键：分析驱动的 Transformer 线性化", section
// 填补近似缺口的实用设计; scale 1/sqrt(d) from Lemma 1 of section
// 从 softmax 到 delta 规则的一阶近似).  The lambda-weighted linear branch
// ("Untangling Component Imbalance in Hybrid Linear Attention Conversion",
// section 关键设计 (1)) is added afterwards by the GDN state kernel: rows that
// have a linear term (position >= n_sinks + W) leave here as the normalised
// softmax output in fp16 (o_sm); every other row is final and goes to `out`.
//
// Work item = (kv head, block of QB = 128 / G query positions inside one
// sequence); the G query heads of the kv group and the QB positions form the
// 128 rows of one M = 128 tile (row = position * G + head, the order a TMA box
// (64, G, QB) of the [tokens][heads][128] feature tensor lands in).  The keys
// the block can see are gathered as key slots [sinks (padded to 8) | window
// span] in TMA boxes (64 rows for aligned runs of window slots, else 8) and
// processed in groups of up to 128 slots:
//   D_S = Q K^T                       (fp16 operands, fp32 in TMEM)
//   online softmax, two threads per row (one per half of the group's slots),
//   P (bf16) over the key tile, which the MMA above has finished with
//   D_O (+)= P V                      (bf16 operands; V straight from the input)
// with the running max and sum per row, rescaling D_O in TMEM between groups.
// Slots past the visible keys hold whatever rows follow (zeros past the
// tensor's end) and are masked.  Persistent CTAs (two per SM: 96 KB of shared
// memory, 256 TMEM columns each) walk the items; every wait is bounded and
// reports a timeout in the error word.
#include <algorithm>

#include "hla_common.cuh"
#include "tma.cuh"
#include "umma.cuh"

namespace hla {

namespace {

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kGroup = 128;  // key slots per group
constexpr uint32_t kWaitLimit = 1u << 22;

constexpr uint32_t kQ = 0;        // 128 rows x 128 fp16, K-major (two 16 KB column blocks)
constexpr uint32_t kK = 32768;    // group keys kGroup x 128 fp16 K-major; then P, 128 rows x kGroup bf16 K-major
constexpr uint32_t kV = 65536;    // group values kGroup x 128 bf16 (MN-major B)
constexpr uint32_t kRed = 98304;  // per-row partial max / sum of the two column halves: [2][2][128] fp32
constexpr uint32_t kBar = kRed + 2048;
constexpr uint32_t kSmemAlloc = kBar + 64 + 1024;
constexpr uint32_t kColS = 0, kColO = 128, kTmemCols = 256;

// 2^x by the PTX approximate base-2 exponential (one special-function-unit op; flush-to-zero; 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 2)
window_softmax_tc_kernel(LayerDims L, const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_k64, const __grid_constant__ CUtensorMap map_v64,
                         const int32_t* __restrict__ cu, const int32_t* __restrict__ blk_base,
                         __half* __restrict__ o_sm, __nv_bfloat16* __restrict__ out, int32_t* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* red = reinterpret_cast<float*>(sm + kRed);  // [0: max | 1: sum][column half][row]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kBar + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = ((warp & 3) << 5) + lane, chalf = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    const int G = L.G, QB = kD / G;
    const int qi = row / G, gq = row % G;
    const uint32_t sbase = umma::smem_addr(sm);
    const uint32_t bar_ld = umma::smem_addr(sm + kBar), bar_mma = bar_ld + 8, bar_q = bar_ld + 24;
    const float qscale = 0.088388347648318447f * 1.4426950408889634f;  // 1/sqrt(128) * log2(e)
    if (tid == 0) {
        umma::mbar_init(bar_ld, 1);
        umma::mbar_init(bar_mma, 1);
        umma::mbar_init(bar_q, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Launched with programmatic stream serialization, the CTAs get here while the features launch may
    // still run: wait for it (and everything before it) before the first global read.  Only then may a
    // launch that follows this one with programmatic stream serialization start (the chunk-local GDN,
    // which reads the features without a wait of its own); its CTAs take the room these leave free.
    pdl_wait();
    pdl_trigger();
    const int64_t n_blocks = __ldg(blk_base + L.n_seqs);
    const int64_t n_items = n_blocks * L.Hkv;
    if ((int64_t)blockIdx.x >= n_items) {  // whole CTA leaves together
        umma::fence_before_sync();
        __syncthreads();
        if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
        return;
    }
    uint32_t ph_ld = 0, ph_mma = 0, ph_q = 0;

    // tid 0 waits with a bound; the CTA then agrees on the outcome
    auto cta_wait = [&](uint32_t mbar, uint32_t& ph) -> bool {
        bool w = true;
        if (tid == 0) {
            w = umma::mbar_try_wait(mbar, ph) || umma::mbar_wait(mbar, ph, kWaitLimit);
            if (!w && err) atomicExch(err, kErrTimeout);
        }
        ph ^= 1u;
        const bool ok = __syncthreads_and(w);
        umma::fence_after_sync();
        return ok;
    };

    // an item's block of query positions and its key slots [sinks (padded to 8) | window span]
    struct Item {
        int kv, sink_pad, n_slots, n_groups;
        int64_t start, pa, pb, n_sink, span_lo;
    };
    auto describe = [&](int64_t item) {
        Item it;
        it.kv = (int)(item / n_blocks);
        const int blk = (int)(item % n_blocks);
        int lo = 0, hi = L.n_seqs - 1;  // sequence owning the block
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(blk_base + mid) <= blk) lo = mid; else hi = mid - 1;
        }
        int64_t len;
        seq_range(cu, lo, L.total, &it.start, &len);
        it.pa = (int64_t)(blk - __ldg(blk_base + lo)) * QB;
        it.pb = min(len, it.pa + QB);
        it.n_sink = min((int64_t)L.n_sinks, it.pb);
        it.sink_pad = (int)((it.n_sink + 7) & ~7);
        it.span_lo = max((int64_t)L.n_sinks, it.pa - L.window + 1);
        const int64_t n_span = it.pb > it.span_lo ? it.pb - it.span_lo : 0;
        it.n_slots = (int)((it.sink_pad + n_span + 15) & ~15);
        it.n_groups = (it.n_slots + kGroup - 1) / kGroup;
        return it;
    };
    // the query tile (thread 0)
    auto issue_q = [&](const Item& it) {
        if (tid == 0) {
            tma::expect_tx(bar_q, 32768u);
            const int tq = (int)(it.start + it.pa);
            tma::tensor_load_3d(sbase + kQ, &map_q, 0, it.kv * G, tq, bar_q);
            tma::tensor_load_3d(sbase + kQ + 16384, &map_q, 64, it.kv * G, tq, bar_q);
        }
    };
    // one group's keys and values (every thread): thread 0 posts the byte count; box b goes to lane b / 8
    // of warp b % 8, so the copies are issued by all warps at once (copies issued back to back by one
    // thread serialise; an early complete_tx just leaves the count below zero until the post); boxes of
    // 8 slots, a 64-slot run of window rows at a 64-aligned offset is one box
    auto issue_kv = [&](const Item& it, int grp) {
        const int g0 = grp * kGroup, n = min(kGroup, it.n_slots - g0);
        if (tid == 0) tma::expect_tx(bar_ld, (uint32_t)n * 2u * 2u * 128u);
        for (int j = 8 * (warp + 8 * lane); j < n; j += 8 * kThreads) {
            const int slot = g0 + j;
            const bool wide = slot >= it.sink_pad && (j & 63) == 0 && j + 64 <= n;
            const bool covered = slot >= it.sink_pad && (j & 63) != 0 && (j & ~63) + 64 <= n &&
                                 g0 + (j & ~63) >= it.sink_pad;  // inside a wide box issued by another lane
            if (covered) continue;
            const int tk = (int)(it.start + (slot < it.sink_pad ? slot : it.span_lo + (slot - it.sink_pad)));
            const uint32_t off = (uint32_t)j * 128u;
            const CUtensorMap* mk = wide ? &map_k64 : &map_k;
            const CUtensorMap* mv = wide ? &map_v64 : &map_v;
            tma::tensor_load_3d(sbase + kK + off, mk, 0, it.kv, tk, bar_ld);
            tma::tensor_load_3d(sbase + kK + 16384 + off, mk, 64, it.kv, tk, bar_ld);
            tma::tensor_load_3d(sbase + kV + off, mv, 0, it.kv, tk, bar_ld);
            tma::tensor_load_3d(sbase + kV + 16384 + off, mv, 64, it.kv, tk, bar_ld);
        }
    };

    const bool sm_on = !(L.flags & HLA_FLAG_SOFTMAX_OFF), lin_off = (L.flags & HLA_FLAG_LINEAR_OFF) != 0;
    bool ok = true;
    // The next item's loads are issued while this one finishes: its query tile once this item's last
    // Q K^T has completed (the query region is free), its first keys and values once this item's last
    // P V has completed (the key / P and value regions are free), so they land during the epilogue.
    Item it = describe(blockIdx.x);
    if (it.n_groups > 0) {
        issue_q(it);
        issue_kv(it, 0);
    }
#pragma unroll 1
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int64_t next = item + gridDim.x;
        const bool has_next = next < n_items;
        const Item nx = has_next ? describe(next) : it;
        const bool pref = has_next && nx.n_groups > 0;
        const int kv = it.kv;
        const int64_t start = it.start, pa = it.pa, pb = it.pb, n_sink = it.n_sink, span_lo = it.span_lo;
        const int sink_pad = it.sink_pad, n_slots = it.n_slots, n_groups = it.n_groups;

        // this row's query position and its visible key slots [0, hi1) and [lo2, hi2)
        const int64_t p = pa + qi;
        const bool row_on = p < pb;
        int hi1 = 0, lo2 = 0, hi2 = 0;
        if (row_on) {
            hi1 = (int)min(n_sink, p + 1);
            lo2 = sink_pad + (int)max((int64_t)0, p - L.window + 1 - span_lo);
            hi2 = p >= span_lo ? sink_pad + (int)(p - span_lo) + 1 : lo2;
        }

        float m_run = -INFINITY, l_run = 0.f;
        for (int grp = 0; grp < n_groups && ok; ++grp) {
            const int g0 = grp * kGroup, n = min(kGroup, n_slots - g0);  // a multiple of 16
            if (grp > 0) issue_kv(it, grp);
            if (grp == 0 && !(ok = cta_wait(bar_q, ph_q))) break;
            if (!(ok = cta_wait(bar_ld, ph_ld))) break;

            // ---- D_S = Q K^T (N = n)
            if (tid == 0) {
                const uint32_t id = umma::idesc_f16(128, n, false, false, false);
                const uint64_t a0 = umma::kmajor(sbase + kQ, 128, 0), b0 = umma::kmajor(sbase + kK, kGroup, 0);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint64_t ks = (uint64_t)((s >> 2) * 1024 + (s & 3) * 2);  // 16 KB per block, 32 B per step
                    umma::mma(tmem + kColS, a0 + ks, b0 + ks, id, s > 0);
                }
                umma::commit(bar_mma);
            }
            if (!(ok = cta_wait(bar_mma, ph_mma))) break;
            if (grp == n_groups - 1 && pref) issue_q(nx);
            // ---- online softmax: this thread covers slots [c_lo, c_hi) of the group (16-slot chunks,
            //      split evenly between the two threads of the row), read from TMEM once: 64 columns
            //      from c_lo (inside the 128 allocated), the ones at or past c_hi masked
            const int n16 = n >> 4, c_lo = chalf ? ((n16 + 1) >> 1) * 16 : 0, c_hi = chalf ? n : ((n16 + 1) >> 1) * 16;
            float sc[64];
            {
                uint32_t r0[32], r1[32];
                umma::tmem_ld32_async(tmem + lane_base + kColS + c_lo, r0);
                umma::tmem_ld32_async(tmem + lane_base + kColS + c_lo + 32, r1);
                umma::tmem_wait_ld();
                umma::reg_fence32(r0);
                umma::reg_fence32(r1);
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    sc[x] = __uint_as_float(r0[x]);
                    sc[32 + x] = __uint_as_float(r1[x]);
                }
            }
            float mg = -INFINITY;  // raw scores: the scale is positive
#pragma unroll
            for (int x = 0; x < 64; ++x) {
                const int gi = g0 + c_lo + x;
                const bool vis = c_lo + x < c_hi && (gi < hi1 || (gi >= lo2 && gi < hi2));
                sc[x] = vis ? sc[x] : -INFINITY;
                mg = fmaxf(mg, sc[x]);
            }
            red[chalf * 128 + row] = mg * qscale;
            __syncthreads();
            const float m_new = fmaxf(m_run, fmaxf(red[row], red[128 + row]));
            const float corr = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
            float lsum = 0.f;
#pragma unroll
            for (int x = 0; x < 64; ++x) {
                sc[x] = sc[x] == -INFINITY ? 0.f : ex2_approx(fmaf(sc[x], qscale, -m_new));
                lsum += sc[x];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // P over the key tile: K-major, slots = K (this thread's chunks only)
                if (c_lo + 8 * j < c_hi) {
                    const float* x = sc + 8 * j;
                    *reinterpret_cast<uint4*>(sm + kK + umma::sw128_offset(row, c_lo + 8 * j, 128)) =
                        make_uint4(pack_bf2(x[0], x[1]), pack_bf2(x[2], x[3]), pack_bf2(x[4], x[5]),
                                   pack_bf2(x[6], x[7]));
                }
            }
            red[256 + chalf * 128 + row] = lsum;
            if (grp > 0) {  // rescale this thread's half of the accumulated output (warp-uniform: TMEM access is collective)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float o[32];
                    const uint32_t ta = tmem + lane_base + kColO + chalf * 64 + 32 * q;
                    umma::tmem_ld32(ta, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= corr;
                    umma::tmem_st32(ta, o);
                }
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            __syncthreads();
            l_run = l_run * corr + red[256 + row] + red[256 + 128 + row];
            m_run = m_new;

            // ---- D_O (+)= P V (K = n)
            if (tid == 0) {
                umma::fence_after_sync();
                const uint32_t id = umma::idesc_bf16(128, kD, false, true);
                const uint64_t a0 = umma::kmajor(sbase + kK, 128, 0), b0 = umma::mnmajor(sbase + kV, 16384u, 0);
                for (int s = 0; s < n / 16; ++s)
                    umma::mma(tmem + kColO, a0 + (uint64_t)((s >> 2) * 1024 + (s & 3) * 2), b0 + (uint64_t)(s * 128),
                              id, grp > 0 || s > 0);
                umma::commit(bar_mma);
            }
            if (!(ok = cta_wait(bar_mma, ph_mma))) break;
        }
        if (!ok) break;
        if (pref) issue_kv(nx, 0);

        // ---- epilogue: this thread's 64 output columns of its row
        {
            const float inv_l = (sm_on && row_on && l_run > 0.f) ? 1.f / l_run : 0.f;
            const bool lin_row = !lin_off && p >= (int64_t)L.n_sinks + L.window;
            const size_t base = ((size_t)(start + (row_on ? p : 0)) * L.Hq + kv * G + gq) * kD + chalf * 64;
            uint32_t oa[32], ob[32];  // both halves in flight together, one wait
            umma::tmem_ld32_async(tmem + lane_base + kColO + chalf * 64, oa);
            umma::tmem_ld32_async(tmem + lane_base + kColO + chalf * 64 + 32, ob);
            umma::tmem_wait_ld();
            umma::reg_fence32(oa);
            umma::reg_fence32(ob);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float o[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) o[x] = __uint_as_float(q ? ob[x] : oa[x]);
                if (!row_on) continue;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    const float* x = o + 8 * c8;
                    const int col = 32 * q + 8 * c8;
                    if (lin_row)
                        *reinterpret_cast<uint4*>(o_sm + base + col) =
                            make_uint4(pack_h2(x[0] * inv_l, x[1] * inv_l), pack_h2(x[2] * inv_l, x[3] * inv_l),
                                       pack_h2(x[4] * inv_l, x[5] * inv_l), pack_h2(x[6] * inv_l, x[7] * inv_l));
                    else
                        *reinterpret_cast<uint4*>(out + base + col) =
                            make_uint4(pack_bf2(x[0] * inv_l, x[1] * inv_l), pack_bf2(x[2] * inv_l, x[3] * inv_l),
                                       pack_bf2(x[4] * inv_l, x[5] * inv_l), pack_bf2(x[6] * inv_l, x[7] * inv_l));
                }
            }
        }
        umma::fence_before_sync();
        __syncthreads();  // shared tiles and TMEM are reused by the next item
        it = nx;
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool window_softmax_tc_supported(const LayerDims& L) {
    return L.d == kD && (L.G == 1 || L.G == 2 || L.G == 4 || L.G == 8);
}

cudaError_t launch_window_softmax_tc(const LayerDims& L, const __half* qr, const __half* kr, const __nv_bfloat16* v,
                                     const int32_t* cu, int32_t* blk_base, __half* o_sm, __nv_bfloat16* out,
                                     int32_t* err, bool after_prior, cudaStream_t st) {
    static DeviceCache cache;  // the shared-memory attribute and the SM count, per device
    int n_sm = 0;
    cudaError_t e = device_cached(cache, &n_sm, [](int dev, int* v) {
        cudaError_t r = cudaFuncSetAttribute(window_softmax_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemAlloc);
        return r == cudaSuccess ? sm_count(dev, v) : r;
    });
    if (e != cudaSuccess) return e;
    if (L.total <= 0) return cudaSuccess;
    const int QB = kD / L.G;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mv, mk64, mv64;
    if (!tma::make_map_3d(&mq, qr, false, kD, (uint64_t)L.Hq, (uint64_t)L.total, 64, (uint32_t)L.G, (uint32_t)QB) ||
        !tma::make_map_3d(&mk, kr, false, kD, (uint64_t)L.Hkv, (uint64_t)L.total, 64, 1, 8) ||
        !tma::make_map_3d(&mv, v, true, kD, (uint64_t)L.Hkv, (uint64_t)L.total, 64, 1, 8) ||
        !tma::make_map_3d(&mk64, kr, false, kD, (uint64_t)L.Hkv, (uint64_t)L.total, 64, 1, 64) ||
        !tma::make_map_3d(&mv64, v, true, kD, (uint64_t)L.Hkv, (uint64_t)L.total, 64, 1, 64))
        return cudaErrorInvalidValue;
    const int64_t items_max = (L.total / QB + L.n_seqs + 1) * (int64_t)L.Hkv;
    const unsigned grid = (unsigned)std::min<int64_t>(items_max, (int64_t)n_sm * 2);
    LaunchCfg lc(dim3(grid), dim3(kThreads), kSmemAlloc, st, after_prior);
    return cudaLaunchKernelEx(&lc.cfg, window_softmax_tc_kernel, L, mq, mk, mv, mk64, mv64, cu, blk_base, o_sm, out,
                              err);
}

}  // namespace hla
