// hla_prefill_noalloc: hla_prefill with its scratch memory taken from a
// fixed-size buffer that lives inside this library, for callers that cannot
// allocate device memory themselves (see include/hla.h for who and why).
//
// The buffer is a file-scope __device__ array: every GPU where the library's
// device code is loaded holds it until the process exits.  Host code cannot
// use the array's name as a device address (on the host it is only a
// stand-in), so the device address is looked up with cudaGetSymbolAddress,
// with that device current, the first time a device is used, and again
// whenever the device's context has changed since (after a cudaDeviceReset
// the module is loaded afresh and the array may sit elsewhere).
#include <cudaTypedefs.h>

#include <mutex>

#include "hla_common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

struct ScratchSlot {
    unsigned long long ctx_id;
    void* addr;
};

std::mutex g_scratch_mutex;
ScratchSlot g_scratch[hla::kMaxDevices] = {};

// Identifier of the current context (driver entry points, looked up once).
bool current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool tried = false;
    if (!tried) {  // under g_scratch_mutex
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    }
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the static scratch on the current device.  Set-up (the
// symbol lookup) runs on the first call per device and after a context change.
int static_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HLA_ERR_CUDA;
    if (dev < 0 || dev >= hla::kMaxDevices) return HLA_ERR_UNSUPPORTED;
    // makes the device's primary context current (created if needed), so it can be identified
    if (cudaSetDevice(dev) != cudaSuccess) return HLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) return HLA_ERR_CUDA;
    ScratchSlot& slot = g_scratch[dev];
    if (!slot.addr || slot.ctx_id != ctx) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            slot.addr = nullptr;
            return HLA_ERR_CUDA;
        }
        slot.addr = p;
        slot.ctx_id = ctx;
    }
    *out = slot.addr;
    return HLA_OK;
}

}  // namespace

extern "C" HLA_API int hla_prefill_noalloc(const hla_params* params, const void* q, const void* k,
                                           const void* v, const float* g, const float* beta,
                                           const float* lambda, const float* conv_wq,
                                           const float* conv_wk, const float* conv_wv,
                                           const int32_t* cu_seqlens, int n_seqs,
                                           int64_t total_tokens, void* out, const hla_state* st,
                                           void* stream) {
    size_t need = 0;
    int rc = hla_prefill_workspace_bytes(params, total_tokens, n_seqs, &need);
    if (rc != HLA_OK) return rc;
    if (need > kStaticScratchBytes) return HLA_ERR_WORKSPACE;  // before any GPU call
    void* ws = nullptr;
    rc = static_scratch(&ws);
    if (rc != HLA_OK) return rc;
    return hla_prefill(params, q, k, v, g, beta, lambda, conv_wq, conv_wk, conv_wv, cu_seqlens,
                       n_seqs, total_tokens, out, st, ws, kStaticScratchBytes, stream);
}

extern "C" HLA_API int hla_prefill_noalloc_check_error(void* stream, int32_t* code) {
    void* ws = nullptr;
    const int rc = static_scratch(&ws);
    if (rc != HLA_OK) return rc;
    return hla_check_workspace_error(ws, stream, code);  // the error word heads the scratch
}
