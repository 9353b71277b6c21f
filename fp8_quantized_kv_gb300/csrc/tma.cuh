// tma.cuh -- TMA (cp.async.bulk) wrappers: tensor-map tile loads and 1-D
// bulk copies into shared memory, completing on an mbarrier transaction
// count.  Every copy here is issued by one thread.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "umma.cuh"

namespace fp8kv {
namespace tma {

// Arrive on `bar` once and add `bytes` to its expected transaction count.
__device__ __forceinline__ void arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}\n" ::"r"(
          umma::smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// 2-D tile load: box at coordinates (x = inner element index, y = row).
__device__ __forceinline__ void load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];\n" ::"r"(umma::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(umma::smem_u32(bar))
      : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned).
__device__ __forceinline__ void load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          umma::smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(umma::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace tma
}  // namespace fp8kv
