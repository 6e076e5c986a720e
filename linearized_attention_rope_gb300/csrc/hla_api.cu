// Host side of the libhla C ABI: argument checks, workspace layout, launch
// order.  Declarations and contracts: include/hla.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <type_traits>

#include "hla_common.cuh"

using namespace hla;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_params(const hla_params* prm) {
    if (!prm) return HLA_ERR_INVALID_ARG;
    if (prm->n_q_heads <= 0 || prm->n_kv_heads <= 0 || prm->n_q_heads % prm->n_kv_heads != 0)
        return HLA_ERR_INVALID_ARG;
    if (prm->n_sinks < 0 || prm->window < 1 || !(prm->rope_base > 1.0f)) return HLA_ERR_INVALID_ARG;
    if (prm->conv_width != kConvWidth) return HLA_ERR_UNSUPPORTED;
    if (prm->head_dim != 64 && prm->head_dim != 128) return HLA_ERR_UNSUPPORTED;
    if (prm->dtype != HLA_DTYPE_F32 && prm->dtype != HLA_DTYPE_BF16) return HLA_ERR_UNSUPPORTED;
    const unsigned known = HLA_FLAG_L2NORM_Q | HLA_FLAG_SOFTMAX_OFF | HLA_FLAG_LINEAR_OFF |
                           HLA_FLAG_GDN_RECURRENT | HLA_FLAG_GLA | HLA_FLAG_TEST_STALL | HLA_FLAG_GDN_SCAN;
    if (prm->flags & ~known) return HLA_ERR_INVALID_ARG;
    return HLA_OK;
}

LayerDims make_dims(const hla_params* prm, int n_seqs, int64_t total) {
    LayerDims L;
    std::memset(&L, 0, sizeof(L));
    L.Hq = prm->n_q_heads;
    L.Hkv = prm->n_kv_heads;
    L.d = prm->head_dim;
    L.G = prm->n_q_heads / prm->n_kv_heads;
    L.n_sinks = prm->n_sinks;
    L.window = prm->window;
    L.n_seqs = n_seqs;
    L.total = total;
    L.flags = prm->flags;
    for (int i = 0; i < prm->head_dim / 2; ++i)
        L.theta[i] = std::pow((double)prm->rope_base, -2.0 * i / (double)prm->head_dim);
    return L;
}

size_t dtype_bytes(int dtype) { return dtype == HLA_DTYPE_F32 ? 4 : 2; }
// feature (MMA operand) element size: fp32 layer keeps fp32, bf16 layer uses fp16
size_t feat_bytes(int dtype) { return dtype == HLA_DTYPE_F32 ? 4 : 2; }

// Workspace layout of one prefill.
struct WsLayout {
    size_t err, fine, coarse, qr, kr, qhat, khat, vhat, olin, osm, blk_base, chunk_base, counters, tinv, smid,
        part_base, pr, s_part, total;
    int n_coarse, part_len, n_parts;
};

// The tensor-core path (chunked GDN + tensor-core softmax) serves bf16 layers
// with head_dim 128 and 1, 2, 4 or 8 query heads per kv head.
bool uses_chunked_gdn(const hla_params* prm) {
    const int G = prm->n_kv_heads > 0 ? prm->n_q_heads / prm->n_kv_heads : 0;
    return prm->dtype == HLA_DTYPE_BF16 && prm->head_dim == 128 && !(prm->flags & HLA_FLAG_GDN_RECURRENT) &&
           (G == 1 || G == 2 || G == 4 || G == 8);
}

// Absorptions per part of the context-parallel token-serial GDN (0: not used): enough parts for about
// 256 (sequence, head, part) CTAs, at least 64 absorptions each, at most 65535 parts in all.
int scan_part_len(const hla_params* prm, int64_t total, int n_seqs) {
    if (!(prm->flags & HLA_FLAG_GDN_SCAN) || uses_chunked_gdn(prm) || n_seqs <= 0 || n_seqs >= 65535) return 0;
    const int64_t units = (int64_t)prm->n_q_heads * n_seqs;
    const int64_t parts = std::max<int64_t>(1, (256 + units - 1) / units);
    const int64_t avg = std::max<int64_t>(1, total / n_seqs - prm->window - prm->n_sinks);
    int64_t pl = std::max<int64_t>(64, ((avg + parts - 1) / parts + 63) / 64 * 64);
    pl = std::max<int64_t>(pl, (total + (65535 - n_seqs) - 1) / (65535 - n_seqs));
    return (int)std::min<int64_t>(pl, INT32_MAX);
}

WsLayout ws_layout(const hla_params* prm, int64_t total, int n_seqs) {
    WsLayout w;
    const size_t fb = feat_bytes(prm->dtype), d = (size_t)prm->head_dim, half = d / 2;
    const size_t Hq = (size_t)prm->n_q_heads, Hkv = (size_t)prm->n_kv_heads, T = (size_t)total;
    w.n_coarse = (int)(total / 64 + 1);
    size_t off = 0;
    w.err = off;    off = align_up(off + 16);
    w.fine = off;   off = align_up(off + 64 * half * sizeof(float2));
    w.coarse = off; off = align_up(off + (size_t)w.n_coarse * half * sizeof(float2));
    w.qr = off;     off = align_up(off + T * Hq * d * fb);
    w.kr = off;     off = align_up(off + T * Hkv * d * fb);
    w.qhat = off;   off = align_up(off + T * Hq * d * fb);
    w.khat = off;   off = align_up(off + T * Hkv * d * fb);
    w.vhat = off;   off = align_up(off + T * Hkv * d * fb);
    const bool chunked = uses_chunked_gdn(prm);
    // token-serial path: fp32 o_lin; chunked path: fp16 softmax rows for the GDN kernel to finish
    w.olin = off;   off = align_up(off + (chunked ? 0 : T * Hq * d * sizeof(float)));
    w.osm = off;    off = align_up(off + (chunked ? T * Hq * d * sizeof(__half) : 0));
    w.blk_base = off; off = align_up(off + (chunked ? ((size_t)n_seqs + 1) * sizeof(int32_t) : 0));
    w.chunk_base = off; off = align_up(off + (chunked ? ((size_t)n_seqs + 1) * sizeof(int32_t) : 0));
    w.counters = off; off = align_up(off + (chunked ? kMaxGdnParts * sizeof(int32_t) : 0));
    w.tinv = off;   off = align_up(off + (chunked ? gdn_chunk_slots(total, n_seqs) * Hq * kRecordBytes : 0));
    // the state between the two halves of the chunked GDN (fp32, per sequence and q-head)
    w.smid = off;   off = align_up(off + (chunked ? (size_t)n_seqs * Hq * d * d * sizeof(float) : 0));
    // context-parallel token-serial GDN: part table, the parts' maps (R, P) and start states
    w.part_len = scan_part_len(prm, total, n_seqs);
    w.n_parts = w.part_len ? (int)(total / w.part_len + n_seqs) : 0;
    const size_t np = (size_t)w.n_parts;
    w.part_base = off; off = align_up(off + (w.part_len ? ((size_t)n_seqs + 1) * sizeof(int32_t) : 0));
    w.pr = off;     off = align_up(off + np * Hq * 2 * d * d * sizeof(float));
    w.s_part = off; off = align_up(off + np * Hq * d * d * sizeof(float));
    w.total = off;
    return w;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? HLA_OK : HLA_ERR_CUDA; }

// Workspace of a continuation on the tensor-core path: the prefill layout for the extended rows
// (every sequence's cached sinks and window in front of its new tokens; this bounds them), then the
// extended sequence table and the extended v, g, beta and output.
struct ContLayout {
    WsLayout w;
    int64_t ext_bound;
    size_t ext_cu, ev, eg, eb, eo, ang, total;
};
bool continue_on_tensor_cores(const hla_params* prm) { return uses_chunked_gdn(prm); }
ContLayout cont_layout(const hla_params* prm, int64_t total, int n_seqs) {
    ContLayout c;
    c.ext_bound = total + (int64_t)n_seqs * (prm->n_sinks + prm->window);
    c.w = ws_layout(prm, c.ext_bound, n_seqs);
    const size_t X = (size_t)c.ext_bound, Hq = (size_t)prm->n_q_heads, Hkv = (size_t)prm->n_kv_heads;
    const size_t d = (size_t)prm->head_dim;
    size_t off = c.w.total;
    c.ext_cu = off; off = align_up(off + ((size_t)n_seqs + 1) * sizeof(int32_t));
    c.ev = off;     off = align_up(off + X * Hkv * d * sizeof(__nv_bfloat16));
    c.eg = off;     off = align_up(off + X * Hq * sizeof(float));
    c.eb = off;     off = align_up(off + X * Hq * sizeof(float));
    c.eo = off;     off = align_up(off + X * Hq * d * sizeof(__nv_bfloat16));
    c.ang = off;    off = align_up(off + ((size_t)total + 1) * (d / 2) * sizeof(float2));
    c.total = off;
    return c;
}
size_t continue_workspace_bytes(const hla_params* prm, int64_t total, int n_seqs) {
    return continue_on_tensor_cores(prm) ? cont_layout(prm, total, n_seqs).total : ws_layout(prm, total, n_seqs).total;
}

// Parts of the chunk slots the chunked GDN runs in (1 .. kMaxGdnParts).
constexpr int kGdnParts = 2;
static_assert(kGdnParts >= 1 && kGdnParts <= kMaxGdnParts, "GDN parts");

// Measurement hook: events recorded between the stages of hla_prefill on the
// calling thread (see hla_prefill_stage_events).
thread_local cudaEvent_t* t_stage_events = nullptr;
thread_local int t_n_stage_events = 0;

cudaError_t mark_stage(int i, cudaStream_t s) {
    if (i < t_n_stage_events && t_stage_events[i]) return cudaEventRecord(t_stage_events[i], s);
    return cudaSuccess;
}


#define HLA_TRY(...)                                           \
    do {                                                       \
        cudaError_t e_ = (__VA_ARGS__);                             \
        if (e_ != cudaSuccess) return HLA_ERR_CUDA;            \
    } while (0)

template <typename Tin, typename Tf>
int run_prefill(const hla_params* prm, const LayerDims& L, const void* q, const void* k,
                const void* v, const float* g, const float* beta, const float* lambda,
                const float* wq, const float* wk, const float* wv, const int32_t* cu, void* out,
                const hla_state* st, char* ws, const WsLayout& w, cudaStream_t stream) {
    int32_t* err = reinterpret_cast<int32_t*>(ws + w.err);
    float2* fine = reinterpret_cast<float2*>(ws + w.fine);
    float2* coarse = reinterpret_cast<float2*>(ws + w.coarse);
    Tf* qr = reinterpret_cast<Tf*>(ws + w.qr);
    Tf* kr = reinterpret_cast<Tf*>(ws + w.kr);
    Tf* qh = reinterpret_cast<Tf*>(ws + w.qhat);
    Tf* kh = reinterpret_cast<Tf*>(ws + w.khat);
    Tf* vh = reinterpret_cast<Tf*>(ws + w.vhat);
    float* olin = reinterpret_cast<float*>(ws + w.olin);
    const Tin* qi = static_cast<const Tin*>(q);
    const Tin* ki = static_cast<const Tin*>(k);
    const Tin* vi = static_cast<const Tin*>(v);

    float* S_out = st ? st->S : nullptr;
    bool chunked = false;
    if constexpr (std::is_same<Tf, __half>::value) chunked = uses_chunked_gdn(prm);
    PrefillTables tabs = {cu, err, nullptr, 0, nullptr, 0, nullptr, 0, st ? st->pos : nullptr, st ? st->err : nullptr};
    RecScan scan = {};
    if (w.part_len) {
        tabs.part_base = reinterpret_cast<int32_t*>(ws + w.part_base);
        tabs.part_rows = w.part_len;
        scan = RecScan{tabs.part_base, w.part_len, w.n_parts, reinterpret_cast<float*>(ws + w.pr),
                       reinterpret_cast<float*>(ws + w.s_part)};
    }
    if (chunked) {
        tabs.counters = reinterpret_cast<int32_t*>(ws + w.counters);
        tabs.n_counters = kGdnParts;
        tabs.blk_base = reinterpret_cast<int32_t*>(ws + w.blk_base);
        tabs.blk_rows = window_softmax_tc_rows(L);
        tabs.chunk_base = reinterpret_cast<int32_t*>(ws + w.chunk_base);
        tabs.chunk_rows = kGdnChunk;
    }
    HLA_TRY(mark_stage(0, stream));
    HLA_TRY(launch_prefill_tables(L, fine, coarse, w.n_coarse, tabs, stream));
    // The GDN launches run with programmatic stream serialization (their CTAs set up while the launch
    // before them drains), unless the stage hook wants each launch timed alone; the features and softmax
    // launches are plain (CTAs waiting beside the kernel before them slowed it by more than the launch
    // latency they hid).  The order stays transitive: a kernel that reads data without waiting for its
    // predecessor (the chunk-local GDN) starts only after a trigger that its predecessor gives once its
    // own wait has returned, and every kernel waits for its predecessor before it completes, so a
    // completed launch implies that all launches before it completed.
    const bool overlap = t_n_stage_events == 0;
    HLA_TRY(launch_features<Tin, Tf>(L, qi, ki, vi, wq, wk, wv, cu, fine, coarse, qr, kr, qh, kh, vh,
                                     err, false, stream));
    HLA_TRY(mark_stage(1, stream));
    if (chunked) {
        // features -> softmax (final rows, fp16 rows to finish) -> per part: chunk-local GDN (beside
        // the launch before it) -> GDN state + combine
        if constexpr (std::is_same<Tf, __half>::value) {
            __half* osm = reinterpret_cast<__half*>(ws + w.osm);
            int32_t* blk_base = reinterpret_cast<int32_t*>(ws + w.blk_base);
            int32_t* chunk_base = reinterpret_cast<int32_t*>(ws + w.chunk_base);
            int32_t* counters = reinterpret_cast<int32_t*>(ws + w.counters);
            unsigned char* rec = reinterpret_cast<unsigned char*>(ws + w.tinv);
            float* smid = reinterpret_cast<float*>(ws + w.smid);
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
            // The GDN runs in kGdnParts parts of the chunk slots, all on the caller's stream, every launch
            // after the softmax with programmatic stream serialization.  A chunk-local launch follows the
            // softmax or the previous part's state launch: its CTAs are placed once every CTA of that
            // launch is resident and take the SMs it leaves free (a state CTA, of 227 KB, needs an SM to
            // itself), and it completes only after that launch has.  A state launch follows its part's
            // chunk-local launch: its CTAs are placed as SMs drain and set up, then wait for that launch
            // to complete.  Each state launch continues from the state the previous one saved.  With the
            // stage hook on, the launches run one after another so that each can be timed alone.
            const int n_slots = (int)gdn_chunk_slots(L.total, L.n_seqs);
            int bound[kGdnParts + 1];
            for (int p = 0; p <= kGdnParts; ++p) bound[p] = (int)((int64_t)n_slots * p / kGdnParts);
            HLA_TRY(launch_window_softmax_tc(L, qr, kr, vi, cu, blk_base, osm, o, err, false, stream));
            HLA_TRY(mark_stage(2, stream));
            HLA_TRY(mark_stage(3, stream));
            HLA_TRY(mark_stage(4, stream));
            for (int p = 0; p < kGdnParts; ++p) {
                HLA_TRY(mark_stage(7 + 4 * p, stream));
                HLA_TRY(launch_gdn_inverse(L, qh, kh, g, beta, cu, chunk_base, bound[p], bound[p + 1], counters + p,
                                           rec, err, overlap, stream));
                HLA_TRY(mark_stage(8 + 4 * p, stream));
                HLA_TRY(mark_stage(9 + 4 * p, stream));
                HLA_TRY(launch_gdn_chunked(L, qh, kh, vh, cu, chunk_base, bound[p], bound[p + 1], rec, osm, lambda, o,
                                           p > 0 ? smid : nullptr, nullptr, p + 1 < kGdnParts ? smid : S_out, err,
                                           overlap, stream));
                HLA_TRY(mark_stage(10 + 4 * p, stream));
            }
            for (int p = kGdnParts; p < kMaxGdnParts; ++p)  // absent parts: zero-length marks
                for (int m = 7; m <= 10; ++m) HLA_TRY(mark_stage(m + 4 * p, stream));
        }
    } else {
        // features -> GDN (fp32 o_lin) -> softmax + combine
        HLA_TRY(mark_stage(2, stream));
        HLA_TRY(mark_stage(3, stream));
        HLA_TRY(launch_gdn_recurrent<Tf>(L, qh, kh, vh, g, beta, cu, olin, S_out, w.part_len ? &scan : nullptr,
                                         stream));
        HLA_TRY(mark_stage(4, stream));
        HLA_TRY(launch_window_softmax<Tin, Tf>(L, qr, kr, vi, olin, lambda, cu, static_cast<Tin*>(out),
                                               stream));
    }
    HLA_TRY(mark_stage(5, stream));
    if (st) HLA_TRY(launch_state_fill<Tin, Tf>(L, qi, ki, vi, g, beta, kh, vh, cu, *st, stream));
    HLA_TRY(mark_stage(6, stream));
    return HLA_OK;
}

// Continuation on the tensor-core path: the prefill's kernels on the extended rows (see continue_tc.cu).
int run_continue_tc(const hla_params* prm, const LayerDims& L, const void* q, const void* k, const void* v,
                    const float* g, const float* beta, const float* lambda, const float* wq, const float* wk,
                    const float* wv, const int32_t* cu, void* out, const hla_state* st, char* ws, const ContLayout& c,
                    cudaStream_t stream) {
    const WsLayout& w = c.w;
    const LayerDims Lx = make_dims(prm, L.n_seqs, c.ext_bound);
    int32_t* err = reinterpret_cast<int32_t*>(ws + w.err);
    int32_t* ext_cu = reinterpret_cast<int32_t*>(ws + c.ext_cu);
    __half* qr = reinterpret_cast<__half*>(ws + w.qr);
    __half* kr = reinterpret_cast<__half*>(ws + w.kr);
    __half* qh = reinterpret_cast<__half*>(ws + w.qhat);
    __half* kh = reinterpret_cast<__half*>(ws + w.khat);
    __half* vh = reinterpret_cast<__half*>(ws + w.vhat);
    __nv_bfloat16* ev = reinterpret_cast<__nv_bfloat16*>(ws + c.ev);
    float* eg = reinterpret_cast<float*>(ws + c.eg);
    float* eb = reinterpret_cast<float*>(ws + c.eb);
    __nv_bfloat16* eo = reinterpret_cast<__nv_bfloat16*>(ws + c.eo);
    __half* osm = reinterpret_cast<__half*>(ws + w.osm);
    int32_t* blk_base = reinterpret_cast<int32_t*>(ws + w.blk_base);
    int32_t* chunk_base = reinterpret_cast<int32_t*>(ws + w.chunk_base);
    int32_t* counters = reinterpret_cast<int32_t*>(ws + w.counters);
    unsigned char* rec = reinterpret_cast<unsigned char*>(ws + w.tinv);
    float* smid = reinterpret_cast<float*>(ws + w.smid);
    const __nv_bfloat16* qi = static_cast<const __nv_bfloat16*>(q);
    const __nv_bfloat16* ki = static_cast<const __nv_bfloat16*>(k);
    const __nv_bfloat16* vi = static_cast<const __nv_bfloat16*>(v);
    HLA_TRY(launch_continue_table(L, cu, *st, ext_cu, stream));
    PrefillTables tabs = {ext_cu, err, counters, kGdnParts, blk_base, window_softmax_tc_rows(Lx), chunk_base,
                          kGdnChunk, nullptr, nullptr};
    HLA_TRY(launch_prefill_tables(Lx, reinterpret_cast<float2*>(ws + w.fine), reinterpret_cast<float2*>(ws + w.coarse),
                                  w.n_coarse, tabs, stream));
    HLA_TRY(launch_continue_rows(L, Lx, cu, *st, ext_cu, qr, kr, qh, kh, vh, ev, eg, eb,
                                 reinterpret_cast<float2*>(ws + c.ang), qi, ki, vi, g, beta, wq, wk, wv, stream));
    HLA_TRY(launch_window_softmax_tc(Lx, qr, kr, ev, ext_cu, blk_base, osm, eo, err, true, stream));
    const int n_slots = (int)gdn_chunk_slots(Lx.total, Lx.n_seqs);
    int bound[kGdnParts + 1];
    for (int p = 0; p <= kGdnParts; ++p) bound[p] = (int)((int64_t)n_slots * p / kGdnParts);
    for (int p = 0; p < kGdnParts; ++p) {
        HLA_TRY(launch_gdn_inverse(Lx, qh, kh, eg, eb, ext_cu, chunk_base, bound[p], bound[p + 1], counters + p, rec,
                                   err, true, stream));
        HLA_TRY(launch_gdn_chunked(Lx, qh, kh, vh, ext_cu, chunk_base, bound[p], bound[p + 1], rec, osm, lambda, eo,
                                   p > 0 ? smid : nullptr, st->S, p + 1 < kGdnParts ? smid : st->S, err, true,
                                   stream));
    }
    HLA_TRY(launch_continue_finish(L, cu, *st, ext_cu, eo, static_cast<__nv_bfloat16*>(out), qi, ki, vi, g, beta, kh,
                                   vh, reinterpret_cast<const float2*>(ws + c.ang), stream));
    return HLA_OK;
}

bool state_ok(const hla_state* st) {
    if (!st) return false;
    const void* ptrs[] = {st->S, st->k_ring, st->v_ring, st->pend_k, st->pend_v, st->pend_g,
                          st->pend_beta, st->conv_q, st->conv_k, st->conv_v, st->pos, st->err, st->scratch};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return false;
    return true;
}

int read_error_word(int32_t* dev, cudaStream_t stream, int32_t* code) {
    int32_t h[4] = {0, 0, 0, 0};
    HLA_TRY(cudaStreamSynchronize(stream));
    HLA_TRY(cudaMemcpy(h, dev, sizeof(h), cudaMemcpyDeviceToHost));
    HLA_TRY(cudaMemset(dev, 0, sizeof(h)));
    if (code) *code = h[0];
    if (h[0] == 0) return HLA_OK;
    if (h[0] == kErrTimeout) return HLA_ERR_TIMEOUT;
    return HLA_ERR_STATE;
}

}  // namespace

extern "C" {

HLA_API const char* hla_status_string(int status) {
    switch (status) {
        case HLA_OK: return "ok";
        case HLA_ERR_INVALID_ARG: return "invalid argument";
        case HLA_ERR_UNSUPPORTED: return "unsupported configuration";
        case HLA_ERR_STATE: return "inconsistent state or sequence table";
        case HLA_ERR_CUDA: return "CUDA error";
        case HLA_ERR_TIMEOUT: return "device-side wait timed out";
        case HLA_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

HLA_API int hla_state_bytes(const hla_params* prm, int n_seqs, hla_state_sizes* out) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (n_seqs < 0 || !out) return HLA_ERR_INVALID_ARG;
    const size_t N = (size_t)n_seqs, Hq = (size_t)prm->n_q_heads, Hkv = (size_t)prm->n_kv_heads;
    const size_t d = (size_t)prm->head_dim, R = (size_t)(prm->n_sinks + prm->window);
    const size_t P = (size_t)prm->window + 1, eb = dtype_bytes(prm->dtype);
    out->S = N * Hq * d * d * 4;
    out->k_ring = N * Hkv * R * d * eb;
    out->v_ring = out->k_ring;
    out->pend_k = N * Hkv * P * d * 4;
    out->pend_v = out->pend_k;
    out->pend_g = N * Hq * P * 4;
    out->pend_beta = out->pend_g;
    out->conv_q = N * kConvHalo * Hq * d * 4;
    out->conv_k = N * kConvHalo * Hkv * d * 4;
    out->conv_v = out->conv_k;
    out->pos = N * 8;
    out->err = 16;
    out->scratch = decode_scratch_bytes(n_seqs, prm->n_q_heads, prm->head_dim, prm->n_sinks, prm->window);
    return HLA_OK;
}

HLA_API int hla_prefill_workspace_bytes(const hla_params* prm, int64_t total_tokens, int n_seqs,
                                        size_t* bytes) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (total_tokens < 0 || n_seqs < 0 || !bytes) return HLA_ERR_INVALID_ARG;
    *bytes = ws_layout(prm, total_tokens, n_seqs).total;
    return HLA_OK;
}

HLA_API int hla_state_init(const hla_params* prm, int n_seqs, const hla_state* st, void* stream) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (n_seqs < 0 || !state_ok(st)) return HLA_ERR_INVALID_ARG;
    hla_state_sizes sz;
    hla_state_bytes(prm, n_seqs, &sz);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ptrs[] = {st->S, st->k_ring, st->v_ring, st->pend_k, st->pend_v, st->pend_g,
                    st->pend_beta, st->conv_q, st->conv_k, st->conv_v, st->pos, st->err, st->scratch};
    size_t sizes[] = {sz.S, sz.k_ring, sz.v_ring, sz.pend_k, sz.pend_v, sz.pend_g,
                      sz.pend_beta, sz.conv_q, sz.conv_k, sz.conv_v, sz.pos, sz.err, sz.scratch};
    for (int i = 0; i < 13; ++i)
        if (sizes[i]) HLA_TRY(cudaMemsetAsync(ptrs[i], 0, sizes[i], s));
    return HLA_OK;
}

HLA_API int hla_prefill(const hla_params* prm, const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* lambda,
                        const float* conv_wq, const float* conv_wk, const float* conv_wv,
                        const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, void* out,
                        const hla_state* st, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (n_seqs < 1 || total_tokens < 0 || total_tokens > (int64_t)INT32_MAX) return HLA_ERR_INVALID_ARG;
    // with no tokens, the per-token tensors may be empty (null)
    const void* ptrs[] = {cu_seqlens, ws, lambda, conv_wq, conv_wk, conv_wv, q, k, v, g, beta, out};
    const int n_required = total_tokens > 0 ? 12 : 2;
    for (int i = 0; i < 12; ++i) {
        if (!ptrs[i] && i >= n_required) continue;
        if (!ptrs[i] || !aligned16(ptrs[i])) return HLA_ERR_INVALID_ARG;
    }
    if (st && !state_ok(st)) return HLA_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(prm, total_tokens, n_seqs);
    if (ws_bytes < w.total) return HLA_ERR_WORKSPACE;
    const LayerDims L = make_dims(prm, n_seqs, total_tokens);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* wsb = static_cast<char*>(ws);
    if (total_tokens == 0) {
        // nothing to compute; a given state keeps its freshly initialised contents
        HLA_TRY(cudaMemsetAsync(wsb + w.err, 0, 16, s));
        return HLA_OK;
    }
    if (prm->dtype == HLA_DTYPE_F32)
        return run_prefill<float, float>(prm, L, q, k, v, g, beta, lambda, conv_wq, conv_wk, conv_wv,
                                         cu_seqlens, out, st, wsb, w, s);
    return run_prefill<__nv_bfloat16, __half>(prm, L, q, k, v, g, beta, lambda, conv_wq, conv_wk,
                                              conv_wv, cu_seqlens, out, st, wsb, w, s);
}

HLA_API int hla_decode_step(const hla_params* prm, int n_seqs, const void* q, const void* k,
                            const void* v, const float* g, const float* beta, const float* lambda,
                            const float* conv_wq, const float* conv_wk, const float* conv_wv,
                            const hla_state* st, void* out, void* stream) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (n_seqs < 0) return HLA_ERR_INVALID_ARG;
    if (prm->n_q_heads / prm->n_kv_heads > kMaxDecodeGroup) return HLA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, g, beta, lambda, conv_wq, conv_wk, conv_wv, out};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return HLA_ERR_INVALID_ARG;
    if (!state_ok(st)) return HLA_ERR_INVALID_ARG;
    if (n_seqs == 0) return HLA_OK;
    const LayerDims L = make_dims(prm, n_seqs, 0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (prm->dtype == HLA_DTYPE_F32)
        return cuda_status(launch_decode_step<float>(
            L, static_cast<const float*>(q), static_cast<const float*>(k),
            static_cast<const float*>(v), g, beta, lambda, conv_wq, conv_wk, conv_wv, *st,
            static_cast<float*>(out), s));
    return cuda_status(launch_decode_step<__nv_bfloat16>(
        L, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), g, beta, lambda, conv_wq, conv_wk, conv_wv, *st,
        static_cast<__nv_bfloat16*>(out), s));
}

HLA_API int hla_check_device_error(const hla_state* st, void* stream, int32_t* code) {
    if (!st || !st->err) return HLA_ERR_INVALID_ARG;
    return read_error_word(st->err, static_cast<cudaStream_t>(stream), code);
}

HLA_API int hla_prefill_stage_events(void** events, int n_events) {
    if (n_events < 0 || (n_events > 0 && !events)) return HLA_ERR_INVALID_ARG;
    t_stage_events = reinterpret_cast<cudaEvent_t*>(events);
    t_n_stage_events = n_events;
    return HLA_OK;
}

HLA_API int hla_prefill_launch_count(const hla_params* prm, int with_state, int* out) {
    const int rc = check_params(prm);
    if (rc != HLA_OK) return rc;
    if (!out) return HLA_ERR_INVALID_ARG;
    // rope tables, features; tensor-core path: softmax block table + softmax, chunk table, one
    // chunk-local and one state launch per part; token-serial path: GDN, softmax
    // (the context-parallel token-serial GDN: three launches in place of one)
    const bool scan = (prm->flags & HLA_FLAG_GDN_SCAN) && !uses_chunked_gdn(prm);
    *out = (uses_chunked_gdn(prm) ? 3 + 2 * kGdnParts : scan ? 6 : 4) + (with_state ? 1 : 0);
    return HLA_OK;
}

HLA_API int hla_prefill_continue(const hla_params* prm, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const float* lambda,
                                 const float* conv_wq, const float* conv_wk, const float* conv_wv,
                                 const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, void* out,
                                 const hla_state* st, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (n_seqs < 1 || total_tokens < 0 || total_tokens > (int64_t)INT32_MAX) return HLA_ERR_INVALID_ARG;
    const void* ptrs[] = {cu_seqlens, ws, lambda, conv_wq, conv_wk, conv_wv, q, k, v, g, beta, out};
    const int n_required = total_tokens > 0 ? 12 : 2;
    for (int i = 0; i < 12; ++i) {
        if (!ptrs[i] && i >= n_required) continue;
        if (!ptrs[i] || !aligned16(ptrs[i])) return HLA_ERR_INVALID_ARG;
    }
    if (!state_ok(st)) return HLA_ERR_INVALID_ARG;
    if (ws_bytes < continue_workspace_bytes(prm, total_tokens, n_seqs)) return HLA_ERR_WORKSPACE;
    const WsLayout w = ws_layout(prm, total_tokens, n_seqs);
    if (total_tokens == 0) return HLA_OK;  // nothing appended; the state is unchanged
    const LayerDims L = make_dims(prm, n_seqs, total_tokens);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* wsb = static_cast<char*>(ws);
    if (continue_on_tensor_cores(prm)) {
        const ContLayout c = cont_layout(prm, total_tokens, n_seqs);
        if (c.ext_bound > (int64_t)INT32_MAX) return HLA_ERR_UNSUPPORTED;
        HLA_TRY(cudaMemsetAsync(wsb + w.err, 0, 16, s));
        return run_continue_tc(prm, L, q, k, v, g, beta, lambda, conv_wq, conv_wk, conv_wv, cu_seqlens, out, st, wsb,
                               c, s);
    }
    if (prm->dtype == HLA_DTYPE_F32)
        return cuda_status(launch_prefill_continue<float, float>(
            L, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), g, beta,
            lambda, conv_wq, conv_wk, conv_wv, cu_seqlens, *st, reinterpret_cast<float*>(wsb + w.kr),
            reinterpret_cast<float*>(wsb + w.khat), reinterpret_cast<float*>(wsb + w.vhat), static_cast<float*>(out),
            s));
    return cuda_status(launch_prefill_continue<__nv_bfloat16, __half>(
        L, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), g, beta, lambda, conv_wq, conv_wk, conv_wv, cu_seqlens, *st,
        reinterpret_cast<__half*>(wsb + w.kr), reinterpret_cast<__half*>(wsb + w.khat),
        reinterpret_cast<__half*>(wsb + w.vhat), static_cast<__nv_bfloat16*>(out), s));
}

HLA_API int hla_prefill_continue_workspace_bytes(const hla_params* prm, int64_t total_tokens, int n_seqs,
                                                 size_t* bytes) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (total_tokens < 0 || n_seqs < 0 || !bytes) return HLA_ERR_INVALID_ARG;
    *bytes = continue_workspace_bytes(prm, total_tokens, n_seqs);
    return HLA_OK;
}

HLA_API int hla_prefill_diagnostics(const hla_params* prm, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const float* lambda,
                                    const float* conv_wq, const float* conv_wk, const float* conv_wv,
                                    const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, void* out,
                                    float* branch_sq, float* key_stats, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (!branch_sq || !key_stats || !aligned16(branch_sq) || !aligned16(key_stats)) return HLA_ERR_INVALID_ARG;
    // the two branches alone, each through the whole prefill path (argument checks included)
    hla_params run = *prm;
    run.flags = (prm->flags & ~(unsigned)HLA_FLAG_SOFTMAX_OFF) | HLA_FLAG_LINEAR_OFF;
    rc = hla_prefill(&run, q, k, v, g, beta, lambda, conv_wq, conv_wk, conv_wv, cu_seqlens, n_seqs, total_tokens,
                     out, nullptr, ws, ws_bytes, stream);
    if (rc) return rc;
    const LayerDims L = make_dims(prm, n_seqs, total_tokens);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool f32 = prm->dtype == HLA_DTYPE_F32;
    if (total_tokens == 0)  // no rows: every sum is zero
        return cuda_status(cudaMemsetAsync(branch_sq, 0, (size_t)n_seqs * prm->n_q_heads * 2 * sizeof(float), s));
    HLA_TRY(f32 ? launch_branch_sq(L, static_cast<const float*>(out), cu_seqlens, branch_sq, 0, s)
                : launch_branch_sq(L, static_cast<const __nv_bfloat16*>(out), cu_seqlens, branch_sq, 0, s));
    run.flags = (prm->flags & ~(unsigned)HLA_FLAG_LINEAR_OFF) | HLA_FLAG_SOFTMAX_OFF;
    rc = hla_prefill(&run, q, k, v, g, beta, lambda, conv_wq, conv_wk, conv_wv, cu_seqlens, n_seqs, total_tokens,
                     out, nullptr, ws, ws_bytes, stream);
    if (rc) return rc;
    HLA_TRY(f32 ? launch_branch_sq(L, static_cast<const float*>(out), cu_seqlens, branch_sq, 1, s)
                : launch_branch_sq(L, static_cast<const __nv_bfloat16*>(out), cu_seqlens, branch_sq, 1, s));
    // the RoPE'd keys the feature path left in the workspace
    const WsLayout w = ws_layout(prm, total_tokens, n_seqs);
    const char* wsb = static_cast<const char*>(ws);
    HLA_TRY(f32 ? launch_key_stats(L, reinterpret_cast<const float*>(wsb + w.kr), cu_seqlens, key_stats, s)
                : launch_key_stats(L, reinterpret_cast<const __half*>(wsb + w.kr), cu_seqlens, key_stats, s));
    return HLA_OK;
}

HLA_API int hla_backward_workspace_bytes(const hla_params* prm, int64_t total_tokens, int n_seqs, size_t* bytes) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (total_tokens < 0 || total_tokens > (int64_t)INT32_MAX || n_seqs < 0 || !bytes) return HLA_ERR_INVALID_ARG;
    *bytes = bwd_layout(make_dims(prm, n_seqs, total_tokens)).total;
    return HLA_OK;
}

HLA_API int hla_backward(const hla_params* prm, const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* lambda, const float* conv_wq, const float* conv_wk,
                         const float* conv_wv, const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens,
                         const void* dout, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlambda,
                         float* dconv_wq, float* dconv_wk, float* dconv_wv, void* ws, size_t ws_bytes,
                         void* stream) {
    int rc = check_params(prm);
    if (rc) return rc;
    if (prm->flags & HLA_FLAG_TEST_STALL) return HLA_ERR_INVALID_ARG;
    if (n_seqs < 1 || total_tokens < 0 || total_tokens > (int64_t)INT32_MAX) return HLA_ERR_INVALID_ARG;
    const void* ptrs[] = {cu_seqlens, ws, lambda, conv_wq, conv_wk, conv_wv, dlambda, dconv_wq, dconv_wk, dconv_wv,
                          q, k, v, g, beta, dout, dq, dk, dv, dg, dbeta};
    const int n_ptrs = (int)(sizeof(ptrs) / sizeof(ptrs[0])), n_required = total_tokens > 0 ? n_ptrs : 10;
    for (int i = 0; i < n_ptrs; ++i) {
        if (!ptrs[i] && i >= n_required) continue;
        if (!ptrs[i] || !aligned16(ptrs[i])) return HLA_ERR_INVALID_ARG;
    }
    const LayerDims L = make_dims(prm, n_seqs, total_tokens);
    const BwdLayout b = bwd_layout(L);
    if (ws_bytes < b.total) return HLA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* wsb = static_cast<char*>(ws);
    if (total_tokens == 0) {  // no tokens: the output, and every gradient, is empty or zero
        const size_t Hq = (size_t)prm->n_q_heads, Hkv = (size_t)prm->n_kv_heads, d = (size_t)prm->head_dim;
        HLA_TRY(cudaMemsetAsync(wsb + b.err, 0, 16, s));
        HLA_TRY(cudaMemsetAsync(dlambda, 0, Hq * sizeof(float), s));
        HLA_TRY(cudaMemsetAsync(dconv_wq, 0, Hq * d * kConvWidth * sizeof(float), s));
        HLA_TRY(cudaMemsetAsync(dconv_wk, 0, Hkv * d * kConvWidth * sizeof(float), s));
        HLA_TRY(cudaMemsetAsync(dconv_wv, 0, Hkv * d * kConvWidth * sizeof(float), s));
        return HLA_OK;
    }
    if (prm->dtype == HLA_DTYPE_F32)
        return cuda_status(launch_backward<float>(
            L, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), g, beta,
            lambda, conv_wq, conv_wk, conv_wv, cu_seqlens, static_cast<const float*>(dout), dq, dk, dv, dg, dbeta,
            dlambda, dconv_wq, dconv_wk, dconv_wv, wsb, b, t_stage_events, t_n_stage_events, s));
    return cuda_status(launch_backward<__nv_bfloat16>(
        L, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), g, beta, lambda, conv_wq, conv_wk, conv_wv, cu_seqlens,
        static_cast<const __nv_bfloat16*>(dout), dq, dk, dv, dg, dbeta, dlambda, dconv_wq, dconv_wk, dconv_wv, wsb, b,
        t_stage_events, t_n_stage_events, s));
}

HLA_API int hla_check_workspace_error(void* ws, void* stream, int32_t* code) {
    if (!ws || !aligned16(ws)) return HLA_ERR_INVALID_ARG;
    return read_error_word(static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream), code);
}

}  // extern "C"
