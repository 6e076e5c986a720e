// hla_prefill_noalloc: hla_prefill with its scratch memory taken from a
// fixed-size buffer that lives inside this library, for callers that cannot
// allocate device memory themselves (see include/hla.h for who and why).
//
// The buffer is a file-scope __device__ array: every GPU that loads the
// library holds it until the process exits.  Host code cannot use the
// array's name as a device address (on the host it is only a stand-in), so
// the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and cached.
#include <mutex>

#include "hla_common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (set-up on the
// first call per device).
int static_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HLA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return HLA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
