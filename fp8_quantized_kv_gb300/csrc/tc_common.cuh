// tc_common.cuh -- helpers shared by the tensor-core (tcgen05) kernels:
// operand layout offsets, E4M3 and exponent helpers, bounded waits, named
// barriers of the softmax warpgroups, and TMA tensor-map encoding on the host.
#pragma once

#include "common.cuh"
#include "tma.cuh"
#include "umma.cuh"

namespace fp8kv {

// Byte offset of (row r, byte column c) in a `rows`-row operand stored in the
// 128-byte-swizzled UMMA layout: 128-byte column blocks are separate
// [rows][128 B] regions; inside a block, the 16-byte chunk index is XOR-ed
// with (row % 8).
__device__ __forceinline__ int sw128_off(int r, int byte_col, int rows) {
  const int blk = byte_col >> 7, within = byte_col & 127;
  return blk * rows * 128 + r * 128 + ((((within >> 4) ^ (r & 7))) << 4) + (within & 15);
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturating); element 0
// in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}
__device__ __forceinline__ uint8_t e4m3_rn(float x) { return (uint8_t)(e4m3x2_rn(x, 0.f) & 0xFF); }
__device__ __forceinline__ float e4m3_val(uint8_t c) {
  float f[4];
  e4m3x4_to_f32_scaled((uint32_t)c, f);
  return f[0] * kTwoPow120;
}
// 2^e for e in the normal exponent range, by building the bits.
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// 2^x with results below 2^-126 flushed to zero.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// log2(x) by the hardware approximation (absolute error ~2^-22); -inf for 0.
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float warp_max_redux(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(x));
  return r;
}
// The same maximum as a pure function, so that several independent ones
// can be scheduled back to back.
__device__ __forceinline__ float warp_max_f32(float x) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(x));
  return r;
}
// Maxima (or sums) of N = 8 or 16 values over the 32 lanes of a warp,
// transposed: lane L returns the maximum (sum) over all lanes of v[idx], idx
// = (L >> (5 - log2 N)) & (N - 1).  Each butterfly step sends half of the values still held, so the
// whole reduction takes N shuffles (16 for 16 values) instead of one
// reduction per value.
template <int N, bool SUM = false>
__device__ __forceinline__ float warp_reduce_transposed(const float (&v)[N], int lane) {
  static_assert(N == 8 || N == 16, "8 or 16 values");
  auto op = [](float x, float y) { return SUM ? x + y : fmaxf(x, y); };
  float a[8];
  if constexpr (N == 16) {
    const bool hi = lane & 16;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float send = hi ? v[j] : v[j + 8], keep = hi ? v[j + 8] : v[j];
      a[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = v[j];
  }
  constexpr int S0 = N == 16 ? 8 : 16;            // lane bit of the next step
  float b[4];
  {
    const bool hi = lane & S0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = hi ? a[j] : a[j + 4], keep = hi ? a[j + 4] : a[j];
      b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, S0));
    }
  }
  float c[2];
  {
    const bool hi = lane & (S0 >> 1);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = hi ? b[j] : b[j + 2], keep = hi ? b[j + 2] : b[j];
      c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, S0 >> 1));
    }
  }
  float d;
  {
    const bool hi = lane & (S0 >> 2);
    const float send = hi ? c[0] : c[1], keep = hi ? c[1] : c[0];
    d = op(keep, __shfl_xor_sync(0xffffffffu, send, S0 >> 2));
  }
#pragma unroll
  for (int o = S0 >> 3; o > 0; o >>= 1) d = op(d, __shfl_xor_sync(0xffffffffu, d, o));
  return d;
}

template <int N>
__device__ __forceinline__ float warp_max_transposed(const float (&v)[N], int lane) {
  return warp_reduce_transposed<N, false>(v, lane);
}
template <int N>
__device__ __forceinline__ float warp_sum_transposed(const float (&v)[N], int lane) {
  return warp_reduce_transposed<N, true>(v, lane);
}

// 2^e for an integer e <= 127, with results below 2^-126 flushed to zero
// (built from the bits: e + 127 <= 0 gives the pattern of +0).
__device__ __forceinline__ float pow2_ftz(int e) { return __int_as_float(max(e + 127, 0) << 23); }

// 2^(d + e) for an integer-valued d <= 0 (a difference of two anchors, or
// -inf / NaN when an anchor is missing) and a small integer e <= 111; results
// below 2^-126 (d = -inf, NaN included) give 0.  Floating-point and integer
// pipes only: d + e + 127 + 2^23 puts the biased exponent in the low
// mantissa bits, which then move to the exponent field.
__device__ __forceinline__ float pow2_diff(float d, int e) {
  const float x = fmaxf(d + (float)e, -127.f) + 8388735.f;    // 2^23 + 127
  return __int_as_float((__float_as_int(x) & 0xFF) << 23);
}

// Exponent e with amax * 2^-e <= 448 (e = 0 for amax = 0).
__device__ __forceinline__ int e4m3_row_exp(float amax) {
  int e = 0;
  (void)frexpf(amax * (1.0f / 448.0f), &e);
  return e;
}

// Bounded wait shared by all roles of a CTA: gives up after ~2 s (SM clock
// cycles, checked every 64 polls) or as soon as another role has given up
// (abort flag).
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (umma::mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (umma::mbar_try(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        *abort = 1;
        return false;
      }
    }
  }
}

// As wait_or_abort, but each poll resumes as soon as the phase completes
// (no suspend-time hint): for hand-offs on the critical path of a pipeline.
__device__ __forceinline__ bool wait_fast(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (umma::mbar_test(bar, parity)) return true;         // completed: no blocking poll
  if (umma::mbar_try_wake(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (umma::mbar_try_wake(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        *abort = 1;
        return false;
      }
    }
  }
}

// OR of `pred` over the 128 threads of softmax warpgroup `wg` (named barrier
// 1 + wg), and a plain barrier over the same threads.
__device__ __forceinline__ bool group_any(int wg, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(1 + wg)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_sync(int wg) { asm volatile("bar.sync %0, 128;\n" ::"r"(1 + wg) : "memory"); }

// ------------------------------------------------------------- clusters --
// Cluster-wide barrier, split into arrive and wait (acquire).  Arrive is
// relaxed: used after fence.mbarrier_init, when the only thing to publish is
// the initialisation of barriers that other CTAs will signal.  A thread that
// arrives once and never again need not wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;\n" ::: "memory"); }
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(saddr), "r"(rank));
  return ra;
}
// 16-byte store into another CTA's shared memory; completes 16 bytes of the
// transaction count of the mbarrier `rbar` in that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];\n"
               ::"r"(raddr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
               : "memory");
}
// Bounded wait (as wait_fast) with cluster-scope acquire: for data that other
// CTAs of the cluster delivered with st.async.
__device__ __forceinline__ bool mbar_try_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(umma::smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_cluster(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Two E4M3 codes (low byte element 0) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(codes));
  return r;
}

// ------------------------------------------------------------ host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  // looked up once per process (thread-safe initialisation of a static)
  static const EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    (void)cudaGetLastError();
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// Tensor map of a K or V store viewed as [rows][128 elements], boxes of
// `box_rows` rows by 128 bytes, 128-byte swizzle.
inline bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(bf16 ? 256 : 128)};
  const cuuint32_t box[2] = {(cuuint32_t)(bf16 ? 64 : 128), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fp8kv
