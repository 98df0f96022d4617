// Host-side creation of TMA tensor maps (cuTensorMapEncodeTiled through the
// runtime's driver entry point, so the library needs no link to libcuda) and
// the device-side tensor copy.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace impfp4 {

// A 2-D uint8 tensor map: `rows` x `row_bytes`, row pitch `pitch` bytes,
// box of `box_rows` x `box_bytes`, 128-byte swizzle, out-of-range reads
// return zero.  Returns false if the driver rejects the map.
bool make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t row_bytes,
                     uint64_t pitch, uint32_t box_rows, uint32_t box_bytes, bool swizzle128);

// 2-D tensor load of one box into shared memory; completion is counted on
// `bar` (transaction bytes = the whole box, zero-filled parts included).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch one box of a 2-D tensor into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// Prefetch `bytes` (a multiple of 16) at 16-byte aligned `src` into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace impfp4
