// Host side of tma.cuh: tensor-map encoding through the driver entry point.
#include <cudaTypedefs.h>

#include "tma.cuh"

namespace hla {
namespace tma {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

bool make_map_3d(CUtensorMap* map, const void* base, bool bf16, uint64_t n0, uint64_t n1, uint64_t n2, uint32_t b0,
                 uint32_t b1, uint32_t b2) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || !base || n0 == 0 || n1 == 0 || n2 == 0 || b0 * 2 > 128) return false;
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
              dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tma
}  // namespace hla
