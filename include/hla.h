/*
 * hla.h — C ABI of libhla, the GB300 (sm_103a) hybrid linear-attention layer.
 *
 * The layer replaces softmax attention in a frozen LLaMA/Qwen backbone, as in
 * "The Key to Going Linear: Analysis-Driven Transformer Linearization"
 * (summary page "迈向线性的关键：分析驱动的 Transformer 线性化"):
 *   - exact softmax over a fixed cache budget of n_sinks sink tokens plus a
 *     sliding window (section 填补近似缺口的实用设计);
 *   - a Gated DeltaNet state S (d x d, fp32, one per query head) that absorbs
 *     every non-sink token when it leaves the window (GDN equation, section
 *     线性注意力替换机制, with a scalar gate alpha = exp(g));
 *   - keys and queries of the linear branch go RoPE -> causal depthwise
 *     short conv (width 8) -> L2 norm (section 实践建议, item 3);
 *   - o_t = softmax_{j in sinks U window}(q_t k_j / sqrt(d)) V
 *           + lambda_h * qhat_t^T S_t,
 *     the inference-time weighting of the two branches of "Untangling
 *     Component Imbalance in Hybrid Linear Attention Conversion", section
 *     关键设计 (1).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless marked "host".  The
 *     caller owns every buffer; the library allocates no device memory and
 *     never synchronises the stream, except hla_check_device_error.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Every kernel of a call runs on it, some with programmatic dependent
 *     launch; the library creates no stream or event of its own.
 *   - Argument errors are detected on the host, before any launch, and return
 *     HLA_ERR_INVALID_ARG / HLA_ERR_UNSUPPORTED without touching the GPU.
 *   - A failed launch returns HLA_ERR_CUDA (the CUDA error is consumed).
 *   - Problems found on the device (malformed cu_seqlens, a bounded wait that
 *     ran out) are recorded in a device error word and read back with
 *     hla_check_device_error / hla_check_workspace_error.
 *   - Results are deterministic: fixed reduction order, no atomics in the
 *     numeric path.
 *   - Tensors are dense and row-major; every pointer must be 16-byte aligned.
 *   - Positions restart at 0 at the start of every sequence.
 */
#ifndef HLA_H
#define HLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HLA_API __attribute__((visibility("default")))

/* status codes */
#define HLA_OK 0
#define HLA_ERR_INVALID_ARG 1 /* bad pointer, size, alignment or parameter */
#define HLA_ERR_UNSUPPORTED 2 /* valid but not implemented (e.g. head_dim 96) */
#define HLA_ERR_STATE 3       /* decode state inconsistent (device error word) */
#define HLA_ERR_CUDA 4        /* a CUDA call or launch failed */
#define HLA_ERR_TIMEOUT 5     /* a bounded device-side wait ran out */
#define HLA_ERR_WORKSPACE 6   /* workspace smaller than hla_prefill_workspace_bytes */

/* element type of q, k, v, out and of the KV ring */
#define HLA_DTYPE_F32 0
#define HLA_DTYPE_BF16 1

/* flags */
#define HLA_FLAG_L2NORM_Q 0x1u       /* qhat = L2(conv(RoPE q)); set by default */
#define HLA_FLAG_SOFTMAX_OFF 0x2u    /* test hook: drop the softmax branch */
#define HLA_FLAG_LINEAR_OFF 0x4u     /* test hook: drop the linear branch */
#define HLA_FLAG_GDN_RECURRENT 0x8u  /* use the token-serial fp32 GDN kernel in
                                        place of the chunked tensor-core one */
#define HLA_FLAG_GLA 0x10u           /* gated linear attention in place of the
                                        delta rule: S <- alpha S + khat vhat^T
                                        (no erase term, beta unused), the other
                                        update of section 线性注意力替换机制 */
#define HLA_FLAG_GDN_SCAN 0x40u      /* token-serial GDN path (fp32 layers, head
                                        dim 64, or with HLA_FLAG_GDN_RECURRENT)
                                        in its context-parallel form: each
                                        sequence's absorptions are cut into
                                        parts; every part's state map
                                        S -> P S + R is formed at once, a scan
                                        over the parts gives their start
                                        states, then all parts run at once.
                                        Three times the work on many more
                                        SMs: for long sequences with few
                                        (sequence, head) units.  No effect on
                                        the tensor-core path. */
#define HLA_FLAG_TEST_STALL 0x20u    /* test hook (tensor-core path): the GDN
                                        state kernel loads nothing, so its
                                        bounded waits run out after about a
                                        millisecond; the call completes and the
                                        workspace error word reads back
                                        HLA_ERR_TIMEOUT.  Outputs are then
                                        undefined. */

/* Layer shape.  n_q_heads must be a multiple of n_kv_heads (grouped-query
 * attention: q-head h reads kv-head h / (n_q_heads / n_kv_heads)).
 * head_dim: 64 or 128.  n_sinks >= 0, window >= 1 (the window includes the
 * current token).  conv_width: 8.  rope_base: RoPE base (rotate-half pairs
 * (i, i + d/2), angle p * base^(-2i/d)).  flags: HLA_FLAG_*. */
typedef struct hla_params {
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int n_sinks;
    int window;
    int conv_width;
    float rope_base;
    int dtype;
    unsigned flags;
} hla_params;

/* Decode state of n_seqs sequences: caller-owned device buffers.
 *   S         fp32  [N, Hq, d, d]     GDN state, S[n][h][i][j], i = key dim
 *   k_ring    dtype [N, Hkv, n_sinks + window, d]  RoPE'd keys: slot p for a
 *             sink p < n_sinks, slot n_sinks + (p - n_sinks) % window otherwise
 *   v_ring    dtype [N, Hkv, n_sinks + window, d]  raw values, same slots
 *   pend_k    fp32  [N, Hkv, window + 1, d]  khat of tokens still in the window,
 *             slot p % (window + 1)
 *   pend_v    fp32  [N, Hkv, window + 1, d]  vhat, same slots
 *   pend_g    fp32  [N, Hq, window + 1]      log-gate g of those tokens
 *   pend_beta fp32  [N, Hq, window + 1]      beta of those tokens
 *   conv_q    fp32  [N, 7, Hq, d]   RoPE'd q of positions p-7 .. p-1
 *   conv_k    fp32  [N, 7, Hkv, d]  RoPE'd k of positions p-7 .. p-1
 *   conv_v    fp32  [N, 7, Hkv, d]  raw v of positions p-7 .. p-1
 *   pos       int64 [N]  next position of each sequence
 *   err       int32 [4]  device error word (0 = fine)
 *   scratch   per-step temporaries of hla_decode_step (size from
 *             hla_state_bytes); dead between calls, not part of the state
 * Every buffer but scratch is the resumable state: copying them out and back
 * in resumes decoding exactly. */
typedef struct hla_state {
    float* S;
    void* k_ring;
    void* v_ring;
    float* pend_k;
    float* pend_v;
    float* pend_g;
    float* pend_beta;
    float* conv_q;
    float* conv_k;
    float* conv_v;
    int64_t* pos;
    int32_t* err;
    void* scratch;
} hla_state;

/* byte sizes of the hla_state buffers, in struct order */
typedef struct hla_state_sizes {
    size_t S, k_ring, v_ring, pend_k, pend_v, pend_g, pend_beta, conv_q, conv_k, conv_v, pos, err, scratch;
} hla_state_sizes;

/* Human-readable name of a status code (static string). */
HLA_API const char* hla_status_string(int status);

/* Sizes of the decode-state buffers for n_seqs sequences (host only). */
HLA_API int hla_state_bytes(const hla_params* params, int n_seqs, hla_state_sizes* out);

/* Workspace bytes hla_prefill needs for total_tokens tokens in n_seqs
 * sequences (host only).  The workspace holds the feature-path outputs and
 * the linear-branch output between kernels. */
HLA_API int hla_prefill_workspace_bytes(const hla_params* params, int64_t total_tokens, int n_seqs,
                                        size_t* bytes);

/* Zeroes every buffer of `st` (positions 0, empty state, empty caches).
 * Asynchronous on `stream`. */
HLA_API int hla_state_init(const hla_params* params, int n_seqs, const hla_state* st, void* stream);

/* Prefill: runs the layer over n_seqs packed sequences.
 *   q [total, Hq, d], k, v [total, Hkv, d]  pre-RoPE, in params->dtype
 *   g, beta [total, Hq] fp32      log alpha (<= 0) and beta in (0, 1), per
 *                                 token and query head
 *   lambda [Hq] fp32              weight of the linear branch per query head
 *   conv_wq [Hq*d, 8], conv_wk [Hkv*d, 8], conv_wv [Hkv*d, 8] fp32  depthwise
 *                                 filters, tap 7 on the current token
 *   cu_seqlens int32 [n_seqs + 1] (device) sequence offsets: 0 = c_0 <= c_1
 *                                 <= ... <= c_n = total_tokens
 *   out [total, Hq, d]            params->dtype
 *   st                            NULL, or a state freshly set up by
 *                                 hla_state_init for n_seqs sequences: it
 *                                 receives everything decoding needs.  A
 *                                 state with a position other than 0 is
 *                                 not fresh: the first kernel flags it in
 *                                 the state's error word (then
 *                                 hla_check_device_error returns
 *                                 HLA_ERR_STATE) and its contents are
 *                                 undefined; `out` is unaffected
 *   ws, ws_bytes                  workspace of at least
 *                                 hla_prefill_workspace_bytes bytes
 * With total_tokens == 0 the per-token pointers may be NULL.
 * Asynchronous; no allocation, no synchronisation.  Malformed cu_seqlens are
 * clamped on the device (no out-of-range access) and flagged in the workspace
 * error word. */
HLA_API int hla_prefill(const hla_params* params, const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* lambda,
                        const float* conv_wq, const float* conv_wk, const float* conv_wv,
                        const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, void* out,
                        const hla_state* st, void* ws, size_t ws_bytes, void* stream);

/* hla_prefill without a caller-supplied workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc, for instance a plugin inside a host framework that owns every
 * byte of device memory through its own pool and gives the plugin no
 * allocator, or a latency-critical caller that cannot afford the implicit
 * device-wide synchronisation of cudaMalloc/cudaFree.
 * Arguments and results are those of hla_prefill; the scratch memory comes
 * from a 64 MiB buffer inside the library.  That buffer is device memory of
 * every process that loads libhla.so, on every GPU where the library's
 * device code gets loaded (at context creation under eager module loading;
 * under lazy loading, the CUDA default, once this entry point first runs on
 * that GPU), whether or not the process ever calls hla_prefill_noalloc, and
 * it is held until the process exits.  Prefills whose
 * hla_prefill_workspace_bytes exceeds 64 MiB (about 1,300 tokens of a
 * 32 q / 8 kv head, head_dim 128 bf16 layer) return HLA_ERR_WORKSPACE before
 * any GPU work.
 * The first call on each device (and the first after that device's context
 * was reset) looks up the buffer's device address, a host-side set-up step;
 * make that first call before any stream capture.
 * It allocates nothing: no cudaMalloc, no cudaFree.
 * All calls share the one buffer and each overwrites what the last left in
 * it: calls that overlap on the GPU (other streams, other threads) race, so
 * order them on one stream.  Problems found on the device (malformed
 * cu_seqlens, a bounded wait that ran out) land in the buffer's error word:
 * read it with hla_prefill_noalloc_check_error. */
HLA_API int hla_prefill_noalloc(const hla_params* params, const void* q, const void* k,
                                const void* v, const float* g, const float* beta,
                                const float* lambda, const float* conv_wq, const float* conv_wk,
                                const float* conv_wv, const int32_t* cu_seqlens, int n_seqs,
                                int64_t total_tokens, void* out, const hla_state* st, void* stream);

/* The device error word of hla_prefill_noalloc's buffer on the current
 * device, as hla_check_workspace_error reads a workspace's: synchronises
 * `stream`, stores the word in *code (may be NULL), clears it, and returns
 * HLA_OK if it was zero, else the matching HLA_ERR_* status.  Allocates
 * nothing. */
HLA_API int hla_prefill_noalloc_check_error(void* stream, int32_t* code);

/* One decode step for every sequence of `st`: token pos[n] of sequence n.
 *   q [N, Hq, d], k, v [N, Hkv, d]  (params->dtype), g, beta [N, Hq] fp32,
 *   lambda and conv filters as for hla_prefill, out [N, Hq, d].
 * The token leaving the window (position pos - window, if not a sink) is
 * absorbed into S first; then the new token's output is formed; pos += 1.
 * At most 8 query heads per kv head (else HLA_ERR_UNSUPPORTED).  A sequence
 * whose pos is negative (no prefill or decode step leaves one) is left as it
 * is, its output row is undefined, and the state's error word reports
 * HLA_ERR_STATE.  Asynchronous. */
HLA_API int hla_decode_step(const hla_params* params, int n_seqs, const void* q, const void* k,
                            const void* v, const float* g, const float* beta, const float* lambda,
                            const float* conv_wq, const float* conv_wk, const float* conv_wv,
                            const hla_state* st, void* out, void* stream);

/* Prefill that continues from a decode state: appends the tokens of each
 * sequence to the context st already holds (after hla_prefill with a state,
 * hla_decode_step, or an earlier call of this one), the first at position
 * st->pos[n].  Arguments as for hla_prefill, except that st is required and
 * is read and advanced: the conv histories, the window keys and values, the
 * tokens still waiting to be absorbed and S carry across the boundary, and
 * pos[n] grows by the sequence's token count.  The outputs and the state
 * afterwards are those of one prefill over the whole sequence (equivalently,
 * of decoding the new tokens one at a time).  A state that never passed
 * through hla_state_init starts from whatever its buffers hold; pos < 0 is
 * flagged in the state's error word (HLA_ERR_STATE) and that sequence is left
 * as it is (its output rows are undefined).  ws, ws_bytes: a workspace of at
 * least hla_prefill_continue_workspace_bytes bytes (its error word as for
 * hla_prefill).  On the tensor-core path (bf16, head_dim 128, 1, 2, 4 or 8
 * query heads per kv head) each sequence's cached sinks and window are laid
 * in front of its new tokens, the positions between them left out, and the
 * prefill's softmax and chunked GDN kernels run on these rows from the cached
 * S; the other layers take a token-serial path (one CTA per query head).
 * There, a sequence table whose sequences overlap (cu_seqlens decreasing once
 * clamped to [0, total_tokens]) is flagged in the state's error word (the
 * sequence-table code, 1) and the outputs and the state are undefined; every
 * write still stays inside ws, out and the state.
 * Asynchronous; no allocation. */
HLA_API int hla_prefill_continue(const hla_params* params, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const float* lambda,
                                 const float* conv_wq, const float* conv_wk, const float* conv_wv,
                                 const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, void* out,
                                 const hla_state* st, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes hla_prefill_continue needs for total_tokens new tokens in
 * n_seqs sequences (host only): on the tensor-core path the prefill's
 * workspace for the new tokens plus every sequence's n_sinks + window cached
 * rows, and the extended rows' v, g, beta and output. */
HLA_API int hla_prefill_continue_workspace_bytes(const hla_params* params, int64_t total_tokens, int n_seqs,
                                                 size_t* bytes);

/* Component-usage diagnostics of a prefill (synthetic analysis; not part of
 * the layer's output path).  Arguments as for hla_prefill, without a decode
 * state, plus:
 *   out [total, Hq, d]      params->dtype, scratch for the branch outputs:
 *                           afterwards it holds lambda_h o_lin (the linear
 *                           branch alone)
 *   branch_sq [n_seqs, Hq, 2] fp32: per sequence and q-head, the sums over
 *                           its positions of |o_sm|^2 (index 0) and of
 *                           |lambda_h o_lin|^2 (index 1), from the rounded
 *                           branch outputs: how much each branch carries
 *                           ("Untangling Component Imbalance in Hybrid Linear
 *                           Attention Conversion", sections 摘要, 方法详解)
 *   key_stats [total, Hkv, 2] fp32: per position p and kv head, with u_i the
 *                           RoPE'd key i scaled to unit length and m_p the mean
 *                           of u_0..u_p within the sequence: the key
 *                           concentration |m_p| (index 0) and the projection
 *                           residual |u_p - (mhat_p . u_p) mhat_p| (index 1;
 *                           1 where m_p = 0), the quantities of the analysis in
 *                           "迈向线性的关键：分析驱动的 Transformer 线性化",
 *                           sections 从 softmax 到 delta 规则的一阶近似 (Lemma 2)
 *                           and 填补近似缺口的实用设计
 *   ws, ws_bytes            as for hla_prefill
 * Runs the prefill twice (each branch alone; HLA_FLAG_SOFTMAX_OFF and
 * HLA_FLAG_LINEAR_OFF in params are overridden) and three reduction kernels.
 * Asynchronous; no allocation. */
HLA_API int hla_prefill_diagnostics(const hla_params* params, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const float* lambda,
                                    const float* conv_wq, const float* conv_wk, const float* conv_wv,
                                    const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, void* out,
                                    float* branch_sq, float* key_stats, void* ws, size_t ws_bytes,
                                    void* stream);

/* Workspace bytes hla_backward needs for total_tokens tokens in n_seqs
 * sequences (host only).  fp32 throughout: the recomputed features and the
 * per-head gradients before the kv-group sums (about 10 T Hq d + 6 T Hkv d
 * floats for T tokens), the softmax rows' max, sum and D (3 T Hq), the GDN
 * state every 64 absorptions ((T / 64 + n_seqs + 1) Hq d^2), the states of
 * one 64-absorption block per sequence and q-head (n_seqs Hq 8 d^2 for d 128,
 * 4 d^2 for d 64), and the sink keys' partial sums per 64-query block
 * (2 (T / 64 + n_seqs) Hq n_sinks d). */
HLA_API int hla_backward_workspace_bytes(const hla_params* params, int64_t total_tokens, int n_seqs,
                                         size_t* bytes);

/* Backward of the layer: the gradients of sum(dout . o) with respect to every
 * input of hla_prefill, for the training of the layer's new parameters (the
 * gates, beta, lambda and the conv filters) on a frozen backbone ("迈向线性的
 * 关键：分析驱动的 Transformer 线性化", section 实践建议).  Arguments q .. n_seqs,
 * total_tokens as for hla_prefill, plus:
 *   dout [total, Hq, d]        params->dtype, the gradient of the output
 *   dq [total, Hq, d], dk, dv [total, Hkv, d]   fp32 (a kv head's gradient
 *                              sums over the q-heads that read it)
 *   dg, dbeta [total, Hq]      fp32 (zero for tokens no state absorbs: the
 *                              sinks and the last `window` positions)
 *   dlambda [Hq]               fp32
 *   dconv_wq [Hq*d, 8], dconv_wk, dconv_wv [Hkv*d, 8]   fp32
 *   ws, ws_bytes               workspace of at least
 *                              hla_backward_workspace_bytes bytes
 * Every output is overwritten.  The forward is recomputed inside (the
 * features, the softmax row statistics, the GDN states), in fp32 from the
 * stored inputs, whatever the forward path (the tensor-core prefill's bf16 and
 * fp16 operands are not reproduced).  GDN: per sequence and q-head a cluster
 * of 8 CTAs, each with d / 8 value columns of S; a forward pass stores the
 * state every 64 absorptions, then per 64-absorption block (last first) the
 * states every 8 (d 128) or 16 (d 64) absorptions are recomputed, and per such
 * stage its states are held in registers while the read-out and absorption
 * steps run backwards.  Softmax: 64 x 64 fp32 tiles, per query block then per
 * key block.  HLA_FLAG_GLA differentiates the GLA update;
 * HLA_FLAG_SOFTMAX_OFF / HLA_FLAG_LINEAR_OFF the layer without that branch;
 * HLA_FLAG_GDN_RECURRENT and HLA_FLAG_GDN_SCAN have no effect; HLA_FLAG_TEST_STALL is rejected
 * (HLA_ERR_INVALID_ARG).  Deterministic (fixed reduction order, no atomics).
 * Malformed cu_seqlens are clamped on the device and flagged in the
 * workspace's error word (hla_check_workspace_error).  With total_tokens == 0
 * the per-token pointers may be NULL and the parameter gradients are zeroed.
 * Asynchronous; no allocation. */
HLA_API int hla_backward(const hla_params* params, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lambda,
                         const float* conv_wq, const float* conv_wk, const float* conv_wv,
                         const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens, const void* dout,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlambda,
                         float* dconv_wq, float* dconv_wk, float* dconv_wv, void* ws, size_t ws_bytes,
                         void* stream);

/* Synchronises `stream`, reads the state's device error word into *code
 * (may be NULL), clears it, and returns HLA_OK if it was zero, else the
 * matching HLA_ERR_* status. */
HLA_API int hla_check_device_error(const hla_state* st, void* stream, int32_t* code);

/* Same for the error word at the head of a prefill workspace. */
HLA_API int hla_check_workspace_error(void* ws, void* stream, int32_t* code);

/* Measurement hook (not part of the layer): for the calling thread, makes
 * hla_prefill record events[i] (cudaEvent_t handles owned by the caller) on
 * its stream at stage boundaries.  Tensor-core path (bf16, head_dim 128):
 * 0 before the first kernel, 1 after the feature path, 2 after the softmax
 * branch, 6 after the decode-state hand-off.  The linear branch runs in up to
 * four parts of the chunk slots, each a chunk-local launch and a state launch
 * (which also combines the two branches), all on the caller's stream: for
 * part p, 7 + 4p before and 8 + 4p after its chunk-local launch, 9 + 4p
 * before and 10 + 4p after its state launch.  Without the hook each
 * chunk-local launch runs beside the launch before it (the softmax, or the
 * previous part's state launch); with the hook on, every launch runs alone,
 * so each interval times one launch.  3 = 4 = 2; marks of parts not run are
 * recorded together after the last state launch, 5 after it.
 * Token-serial path: 0, 1 as above, 2 = 3 = 1, 4 after the GDN kernel, 5
 * after the softmax + combine, 6 after the hand-off (7 to 22 not recorded).
 * hla_backward, with the hook on, records 0 before its first kernel and
 * i = 1 .. 8 after its i-th stage (RoPE rows, conv and L2 features, GDN
 * backward, softmax backward, L2 backward, conv and RoPE backward, filter
 * partial sums + their reduction as one, lambda reduction); the L2, conv and
 * RoPE backward are one launch, so 5 = 4; its launches run one after another
 * either way.
 * Entries beyond n_events, or NULL entries, are skipped; n_events = 0
 * switches the hook off.  The array must stay valid while the hook is on. */
HLA_API int hla_prefill_stage_events(void** events, int n_events);

/* Measurement hook (not part of the layer): *out = the number of kernels one
 * hla_prefill call with these params launches (with_state != 0: with a
 * decode state to fill).  Memsets and event records are not counted.  Returns
 * the params check's status. */
HLA_API int hla_prefill_launch_count(const hla_params* params, int with_state, int* out);

#ifdef __cplusplus
}
#endif

#endif /* HLA_H */
