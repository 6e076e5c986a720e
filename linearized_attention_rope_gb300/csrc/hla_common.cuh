// Shared device-side definitions of libhla (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/hla.h"

namespace hla {

constexpr int kConvWidth = 8;
constexpr int kConvHalo = kConvWidth - 1;  // rows of history the conv needs
constexpr int kMaxHalfDim = 64;            // head_dim <= 128

// device error word codes (written with atomicExch / plain stores)
constexpr int kErrSeqlens = 1;   // cu_seqlens not monotone / not ending at total
constexpr int kErrTimeout = 2;   // a bounded wait ran out
constexpr int kErrState = 3;     // decode position inconsistent with the state

// Per-launch constants, passed by value.  theta[i] = base^(-2i/d) computed on
// the host in double precision.
struct LayerDims {
    int Hq, Hkv, d, G;  // G = Hq / Hkv
    int n_sinks, window;
    int n_seqs;
    int64_t total;
    unsigned flags;
    double theta[kMaxHalfDim];
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// Packed fp32 FMA (fma.rn.f32x2): d = a * b + c on both lanes, each rounded
// as fmaf, in one instruction.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// Loads E (2 or 4) consecutive elements starting at an E-aligned index as fp32.
template <int E> __device__ __forceinline__ void load_vec(const float* p, float* o) {
    if constexpr (E == 4) { float4 x = *reinterpret_cast<const float4*>(p); o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; }
    else { float2 x = *reinterpret_cast<const float2*>(p); o[0] = x.x; o[1] = x.y; }
}
template <int E> __device__ __forceinline__ void load_vec(const __half* p, float* o) {
    if constexpr (E == 4) {
        uint2 x = *reinterpret_cast<const uint2*>(p);
        float2 a = __half22float2(*reinterpret_cast<__half2*>(&x.x));
        float2 b = __half22float2(*reinterpret_cast<__half2*>(&x.y));
        o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    } else {
        unsigned x = *reinterpret_cast<const unsigned*>(p);
        float2 a = __half22float2(*reinterpret_cast<__half2*>(&x));
        o[0] = a.x; o[1] = a.y;
    }
}
template <int E> __device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float* o) {
    if constexpr (E == 4) {
        uint2 x = *reinterpret_cast<const uint2*>(p);
        float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x.x));
        float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x.y));
        o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    } else {
        unsigned x = *reinterpret_cast<const unsigned*>(p);
        float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x));
        o[0] = a.x; o[1] = a.y;
    }
}

// Sequence that owns global token t: largest s with cu[s] <= t (cu clamped to
// [0, total] so a malformed table can never send an access out of range).
__device__ __forceinline__ int seq_of_token(const int32_t* __restrict__ cu, int n_seqs, int64_t t) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int64_t clamp_i64(int64_t x, int64_t lo, int64_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

// (start, length) of sequence s, clamped into [0, total].
__device__ __forceinline__ void seq_range(const int32_t* __restrict__ cu, int s, int64_t total,
                                          int64_t* start, int64_t* len) {
    int64_t a = clamp_i64(__ldg(cu + s), 0, total);
    int64_t b = clamp_i64(__ldg(cu + s + 1), a, total);
    *start = a;
    *len = b - a;
}

// cos/sin of p * theta with the angle formed and reduced to [-pi, pi] in
// double precision, then evaluated in fp32 (used where few angles are needed).
__device__ __forceinline__ void rope_cs_exact(int64_t p, double theta, float* c, float* s) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    double a = (double)p * theta;
    a -= two_pi * rint(a * inv_two_pi);  // any integer near a / 2 pi leaves |a| within pi and a rounding
    sincosf((float)a, s, c);
}

// ---- per-device set-up ------------------------------------------------------

constexpr int kMaxDevices = 64;

// Host-side values a launcher needs once per device (a kernel attribute set,
// an SM or occupancy count).  One instance per launcher (per kernel
// instantiation); safe to share between threads and devices.
struct DeviceCache {
    std::mutex m;
    bool ready[kMaxDevices] = {};
    int value[kMaxDevices] = {};
};

// With the current device dev: the first call runs setup(dev, &v) under the
// cache's lock and keeps v (a failed setup is retried by the next call);
// every call stores the device's value in *value (may be null).
template <class F>
cudaError_t device_cached(DeviceCache& c, int* value, F setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(c.m);
    if (!c.ready[dev]) {
        int v = 0;
        e = setup(dev, &v);
        if (e != cudaSuccess) return e;
        c.value[dev] = v;
        c.ready[dev] = true;
    }
    if (value) *value = c.value[dev];
    return cudaSuccess;
}

// Streaming multiprocessors of device dev.
inline cudaError_t sm_count(int dev, int* n) {
    cudaError_t e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
    return e == cudaSuccess && *n <= 0 ? cudaErrorInvalidValue : e;
}

// ---- kernel launchers (each returns the cudaError_t of its launch) --------

// Launch configuration for cudaLaunchKernelEx; with after_prior, programmatic
// stream serialization: the kernel's CTAs may start once every CTA of the
// launch before it in the stream has executed griddepcontrol.launch_dependents
// (or exited), and the kernel orders itself after that launch with
// griddepcontrol.wait.  Used in place (cfg points at attr).
struct LaunchCfg {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool after_prior) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = after_prior ? 1 : 0;
    }
    LaunchCfg(const LaunchCfg&) = delete;
    LaunchCfg& operator=(const LaunchCfg&) = delete;
};
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// What the first launch of a prefill writes besides the RoPE tables (device
// pointers; a null table is skipped): err[0..3] = 0, counters[0..n_counters)
// = 0 (n_counters <= 32), st_err[0] = kErrState if some st_pos[n] != 0, and
// per-sequence work tables blk_base / chunk_base / part_base
// (n_seqs + 1 int32 each): base[s] = the items of sequences before s, where
// a sequence of len rows has ceil(len / blk_rows) softmax row blocks,
// ceil((len - n_sinks - W) / chunk_rows) GDN chunks and
// ceil((len - n_sinks - W) / part_rows) GDN parts (none if not positive).
struct PrefillTables {
    const int32_t* cu;
    int32_t* err;
    int32_t* counters;
    int n_counters;
    int32_t* blk_base;
    int blk_rows;
    int32_t* chunk_base;
    int chunk_rows;
    // decode state to fill (may be null): a position that is not 0 marks a
    // state that was not freshly initialised; st_err[0] = kErrState then
    const int64_t* st_pos;
    int32_t* st_err;
    int32_t* part_base;  // parts of the context-parallel token-serial GDN (part_rows absorptions each)
    int part_rows;
};
// RoPE tables: fine[b][i] = (cos, sin)(b * theta_i), b < 64;
// coarse[a][i] = (cos, sin)(64 a * theta_i), a < n_coarse; plus the tables
// above.  One launch.
cudaError_t launch_prefill_tables(const LayerDims& L, float2* fine, float2* coarse, int n_coarse,
                                  const PrefillTables& t, cudaStream_t st);

// Feature path for every (token, head): RoPE'd q/k, and qhat, khat, vhat.
// Tf = float (fp32 layer) or __half (bf16 layer).
// With after_prior, launched with programmatic stream serialization after the
// table launch (its CTAs wait for it before their first read).
template <typename Tin, typename Tf>
cudaError_t launch_features(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                            const float* wq, const float* wk, const float* wv, const int32_t* cu,
                            const float2* fine, const float2* coarse, Tf* qr, Tf* kr, Tf* qhat,
                            Tf* khat, Tf* vhat, int32_t* err, bool after_prior, cudaStream_t st);

constexpr int kMaxGdnParts = 4;  // parts of the chunk slots the chunked GDN may run in

// Context-parallel form of the token-serial GDN: part table base [n_seqs + 1] (parts of part_len
// absorptions per sequence; n_parts bounds base[n_seqs]), the parts' maps pr [n_parts][Hq][2][d][d]
// (R, then P) and start states s_part [n_parts][Hq][d][d], fp32.
struct RecScan {
    const int32_t* base;
    int part_len;
    int n_parts;
    float* pr;
    float* s_part;
};
// Token-serial fp32 GDN with delayed absorption: o_lin [total, Hq, d] fp32
// for positions p >= n_sinks + window; final S into S_out (may be null).
// rs != null: the context-parallel form (three launches).
template <typename Tf>
cudaError_t launch_gdn_recurrent(const LayerDims& L, const Tf* qhat, const Tf* khat, const Tf* vhat,
                                 const float* g, const float* beta, const int32_t* cu, float* o_lin,
                                 float* S_out, const RecScan* rs, cudaStream_t st);

// Chunked (C = 64) GDN with delayed absorption on tcgen05 tensor cores,
// head_dim 128, fp16 features: same outputs as launch_gdn_recurrent.
// Step 1 (parallel over chunks): chunk table (n_seqs + 1 entries) and, per
// chunk and q-head, a record of kRecordBytes: -Wm = -T diag(beta gamma) K
// (64 x 128), T diag(beta) and P (64 x 64) as fp16 swizzled K-major tile
// images, then gamma and the key decay (fp32, 64 each).
// Step 2: the state-carrying kernel.
constexpr int kGdnChunk = 64;  // C, rows of a chunk
constexpr uint32_t kRecWm = 0, kRecTb = 16384, kRecP = 24576, kRecVec = 32768, kRecordBytes = 33280;
// The chunk table (n_seqs + 1 entries, on the device; chunk_rows = 64) and
// zeroed item counters come from launch_prefill_tables; each
// launch_gdn_inverse covers the chunk slots [slot_lo, slot_hi) (clipped to
// the table's total), its CTAs taking items from its own counter.  With
// beside_prior it is launched with programmatic stream serialization: its
// CTAs are placed once every CTA of the launch before it in the stream (a
// softmax or state launch, which signal this at entry) is resident, and it
// completes only after that launch has.
size_t gdn_chunk_slots(int64_t total, int n_seqs);
cudaError_t launch_gdn_inverse(const LayerDims& L, const __half* qhat, const __half* khat, const float* g,
                               const float* beta, const int32_t* cu, const int32_t* chunk_base, int slot_lo,
                               int slot_hi, int32_t* counter, unsigned char* rec_out, int32_t* err, bool beside_prior,
                               cudaStream_t st);
// The chunks of slots [slot_lo, slot_hi) of every sequence, continuing from
// S_in (fp32 [n_seqs][Hq][d][d]; read only for sequences with chunks before
// slot_lo; may be null if none has), a sequence's first chunks from S_init
// (same layout; null: the zero state).  out rows of
// positions >= n_sinks + W of those chunks: bf16(o_sm + lambda_h o_lin) (none
// if out is null or the linear branch is switched off); the state after the
// last chunk in range into S_out (may be null).  With beside_prior it is
// launched with programmatic stream serialization: its CTAs may be placed and
// set up while the launch before it (which signals this at entry) still
// runs, and wait for that launch to complete before their first global read.
cudaError_t launch_gdn_chunked(const LayerDims& L, const __half* qhat, const __half* khat, const __half* vhat,
                               const int32_t* cu, const int32_t* chunk_base, int slot_lo, int slot_hi,
                               const unsigned char* rec_in, const __half* o_sm, const float* lambda,
                               __nv_bfloat16* out, const float* S_in, const float* S_init, float* S_out, int32_t* err,
                               bool beside_prior, cudaStream_t st);

// Tensor-core continuation (bf16, head_dim 128): the extended sequence table ext_cu [n_seqs + 1] from
// the state's positions; the extended rows (cached rows from the state, new rows from the inputs) of the
// RoPE'd q, k, qhat, khat, vhat (fp16), v (bf16), g, beta (fp32); then the new output rows into out and
// the state (ring, pending ring, conv histories, pos).  L: the call's own dims (total = new tokens).
cudaError_t launch_continue_table(const LayerDims& L, const int32_t* cu, const hla_state& s, int32_t* ext_cu,
                                  cudaStream_t st);
cudaError_t launch_continue_rows(const LayerDims& L, const LayerDims& Lx, const int32_t* cu, const hla_state& s,
                                 const int32_t* ext_cu, __half* qr, __half* kr, __half* qh, __half* kh, __half* vh,
                                 __nv_bfloat16* ev, float* eg, float* eb, float2* ang, const __nv_bfloat16* q,
                                 const __nv_bfloat16* k, const __nv_bfloat16* v, const float* g, const float* beta,
                                 const float* wq, const float* wk, const float* wv, cudaStream_t st);
cudaError_t launch_continue_finish(const LayerDims& L, const int32_t* cu, const hla_state& s, const int32_t* ext_cu,
                                   const __nv_bfloat16* ext_out, __nv_bfloat16* out, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v, const float* g, const float* beta,
                                   const __half* kh, const __half* vh, const float2* ang, cudaStream_t st);

// Sink + window softmax with the lambda-weighted linear branch added.
template <typename Tin, typename Tf>
cudaError_t launch_window_softmax(const LayerDims& L, const Tf* qr, const Tf* kr, const Tin* v,
                                  const float* o_lin, const float* lambda, const int32_t* cu,
                                  Tin* out, cudaStream_t st);

// Sink + window softmax on tcgen05 (bf16 layer, head_dim 128, G in {1,2,4,8}).
// Tensor-core sink + window softmax (head_dim 128, G in {1, 2, 4, 8}; bf16
// values).  Rows of positions >= n_sinks + W (unless the linear branch is
// off) get the normalised softmax output in o_sm (fp16) for the GDN kernel to
// finish; all other rows are written to out.  blk_base: the per-sequence
// block table from launch_prefill_tables with blk_rows = 128 / G.
bool window_softmax_tc_supported(const LayerDims& L);
inline int window_softmax_tc_rows(const LayerDims& L) { return 128 / L.G; }
// With after_prior, launched with programmatic stream serialization after the
// features launch: CTAs set up beside it, then wait for it.
cudaError_t launch_window_softmax_tc(const LayerDims& L, const __half* qr, const __half* kr, const __nv_bfloat16* v,
                                     const int32_t* cu, int32_t* blk_base, __half* o_sm, __nv_bfloat16* out,
                                     int32_t* err, bool after_prior, cudaStream_t st);

// Diagnostics: sq[(n Hq + h) 2 + which] = sum over the rows of sequence n of |out[p][h]|^2; and per
// position p and kv head the key concentration and projection residual of the RoPE'd keys kr
// (stats[(p Hkv + kv) 2 + {0, 1}]).
template <typename T>
cudaError_t launch_branch_sq(const LayerDims& L, const T* out, const int32_t* cu, float* sq, int which, cudaStream_t st);
template <typename Tf>
cudaError_t launch_key_stats(const LayerDims& L, const Tf* kr, const int32_t* cu, float* stats, cudaStream_t st);

// Prefill that continues every sequence from its decode state (positions from pos[n]); kr, khat,
// vhat: [total, Hkv, d] scratch in the feature type.  Four launches on st; pos advances last.
template <typename Tin, typename Tf>
cudaError_t launch_prefill_continue(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* g,
                                    const float* beta, const float* lambda, const float* wq, const float* wk,
                                    const float* wv, const int32_t* cu, const hla_state& s, Tf* kr, Tf* khat,
                                    Tf* vhat, Tin* out, cudaStream_t st);

// Backward of the layer (fp32): workspace layout (byte offsets) and launches.  Gradients of
// sum(dout . o): dq [total, Hq, d], dk, dv [total, Hkv, d], dg, dbeta [total, Hq], dlam [Hq],
// dwq [Hq, d, 8], dwk, dwv [Hkv, d, 8], all fp32.
struct BwdLayout {
    size_t err, qr, kr, qt, qh, kt, kh, vh, dqh, dkh_h, dvh_h, dqr_sm, dkr_h, dv_h, dqt, dkt, dvt, stats, alpha,
        ckpt, sub, dlam_part, convw_part, sm_base, sink_k, sink_v, total;
    int n_blocks, n_sm_blocks;
};
BwdLayout bwd_layout(const LayerDims& L);
template <typename Tin>
cudaError_t launch_backward(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v, const float* g,
                            const float* beta, const float* lambda, const float* wq, const float* wk, const float* wv,
                            const int32_t* cu, const Tin* dout, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, float* dlam, float* dwq, float* dwk, float* dwv, char* ws,
                            const BwdLayout& b, const cudaEvent_t* marks, int n_marks, cudaStream_t st);

// Prefill -> decode state hand-off.
template <typename Tin, typename Tf>
cudaError_t launch_state_fill(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                              const float* g, const float* beta, const Tf* khat, const Tf* vhat,
                              const int32_t* cu, const hla_state& s, cudaStream_t st);

// One decode step for all sequences, then pos += 1.  At most kMaxDecodeGroup
// query heads per kv head.  A negative position is flagged in the state's
// error word (kErrState) and that sequence is left as it is.
constexpr int kMaxDecodeGroup = 8;
// Bytes of the per-step decode scratch (hla_state.scratch).
size_t decode_scratch_bytes(int n_seqs, int Hq, int D, int n_sinks, int window);
template <typename Tin>
cudaError_t launch_decode_step(const LayerDims& L, const Tin* q, const Tin* k, const Tin* v,
                               const float* g, const float* beta, const float* lambda,
                               const float* wq, const float* wk, const float* wv,
                               const hla_state& s, Tin* out, cudaStream_t st);

}  // namespace hla
