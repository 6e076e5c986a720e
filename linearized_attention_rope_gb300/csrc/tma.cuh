// Tensor Memory Accelerator (TMA) helpers: tensor maps built on the host
// through the driver entry point (no link against libcuda), and the
// device-side bulk copies that complete on an mbarrier's transaction count.
//
// A feature tensor [tokens, heads, 128] fp16 is described as a 3-D map
// (dims fastest first: 128, heads, tokens); a box of 64 x 1 x 64 lands as 64
// token rows of 128 bytes in the 128-byte-swizzled layout of umma.cuh, so the
// destination must be 1024-byte aligned.  Coordinates past the tensor's end
// read as zeros; the innermost coordinate is always a multiple of 64
// elements (128 bytes).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hla {
namespace tma {

// Host: a 3-D 16-bit map (fp16, or bf16 if `bf16`) over [n2][n1][n0] with
// box (b0, b1, b2), b0 * 2 <= 128 bytes, and 128-byte swizzle.  Returns false
// if the driver rejects it.
bool make_map_3d(CUtensorMap* map, const void* base, bool bf16, uint64_t n0, uint64_t n1, uint64_t n2, uint32_t b0,
                 uint32_t b1, uint32_t b2);
// The (64, 1, 64) fp16 box used for chunks of 64 token rows.
inline bool make_map_f16_3d(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1, uint64_t n2) {
    return make_map_3d(map, base, false, n0, n1, n2, 64, 1, 64);
}

__device__ __forceinline__ void expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}

// Contiguous global -> shared copy; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// Box (x, y, z) of a 3-D map into shared memory at dst.
__device__ __forceinline__ void tensor_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                               uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

}  // namespace tma
}  // namespace hla
