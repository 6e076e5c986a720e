// The side stream of hla_common.cuh: one per host thread and device.
#include "hla_common.cuh"

namespace hla {

constexpr int kMaxDevices = 64;
thread_local SideStream t_side[kMaxDevices];

cudaError_t side_stream(SideStream** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    SideStream& ss = t_side[dev];
    if (!ss.s) {
        if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (cudaEvent_t* ev : {&ss.fork, &ss.join})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &ss;
    return cudaSuccess;
}

}  // namespace hla
