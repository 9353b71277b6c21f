// common.cuh -- device helpers shared by the FP8-KV kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fp8kv.h"

namespace fp8kv {

constexpr int kTileTokens = 64;       // KV tile (tokens) of every attention kernel
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwoPow120 = 1.329227995784916e36f;   // 2^120, exact in fp32

// Cache element kinds, resolved at compile time per kernel instance.
// ELEM_MX: e4m3 codes with one E8M0 (power-of-two) scale per 32-element
// block of the row, the block scales of a row packed into its 4-byte scale
// slot (byte b = block b); K side only.
enum : int { ELEM_E4M3 = 0, ELEM_BF16 = 1, ELEM_MX = 2 };

// Plain-data view of a cache, passed by value to kernels.
struct CacheView {
  const uint8_t* k;
  const uint8_t* v;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const float* k_bias;             // pre-bias residual keys: [kv_heads][head_dim], or null
  const float* rope_cos;           // rotated bias: [positions][head_dim / 2], or null
  const float* rope_sin;
  int batch, kv_heads, head_dim;
  int max_tokens;                  // contiguous capacity
  int page_size, page_shift, num_pages, max_pages_per_seq;
  int paged;
};

// Rotated key bias (R_t b)_d of KV head h at position t ("rotate half":
// dims i and i + D/2 form pair i), in fp32 with each product with sin
// rounded first: fma(b_d, cos, -(b_{d+D/2} sin)) or fma(b_d, cos, b_{d-D/2} sin).
__device__ __forceinline__ float rope_bias(const CacheView& c, int h, int t, int d) {
  const int H = c.head_dim >> 1;
  const int p = d < H ? d : d - H;
  const float cs = c.rope_cos[(int64_t)t * H + p], sn = c.rope_sin[(int64_t)t * H + p];
  const float* b = c.k_bias + (int64_t)h * c.head_dim;
  return d < H ? fmaf(b[d], cs, -__fmul_rn(b[d + H], sn)) : fmaf(b[d], cs, __fmul_rn(b[d - H], sn));
}

__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- e4m3 ----
// E4M3 -> fp32 by moving bits: sign to bit 31, the 7 exponent+mantissa bits
// to bits 20..26.  The result is the code's value times 2^-120 (fp32 bias 127
// vs E4M3 bias 7), exact for every finite code, subnormals included (they
// land on fp32 subnormals, which the FMA pipe keeps since nothing here is
// compiled with flush-to-zero).  Callers multiply the 2^120 back in once per
// dot product or output row.  Byte i of the word is element i.
__device__ __forceinline__ void e4m3x4_to_f32_scaled(uint32_t w, float (&f)[4]) {
  f[0] = __int_as_float(((int)(w << 24) >> 4) & 0x87F00000);
  f[1] = __int_as_float(((int)(w << 16) >> 4) & 0x87F00000);
  f[2] = __int_as_float(((int)(w << 8) >> 4) & 0x87F00000);
  f[3] = __int_as_float(((int)w >> 4) & 0x87F00000);
}

// bf16 pair (one 32-bit word, element 0 in the low half) -> two exact fp32.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float (&f)[2]) {
  f[0] = __uint_as_float(w << 16);
  f[1] = __uint_as_float(w & 0xFFFF0000u);
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// ------------------------------------------------------------ cp.async ----
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem_src));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ------------------------------------------------------------- swizzle ----
// 16-byte chunk permutation inside a shared-memory row of `cpr` chunks, so
// that threads reading the same logical chunk of consecutive rows hit
// different bank groups.  Rows of >= 8 chunks XOR the low 3 bits with the row
// index; 4-chunk rows (two per 128-byte bank line) XOR with row/2.
__device__ __forceinline__ int swz_chunk(int chunk, int row, int cpr) {
  return cpr >= 8 ? (chunk ^ (row & 7)) : (chunk ^ ((row >> 1) & 3));
}

// ----------------------------------------------------------- reductions ---
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ----------------------------------------------------------------- MXFP8 --
// Block scale of an MXFP8 block ("FP8 KV attention: hardware paths and tile
// preparation", section "Measure block-scaled QK": one E8M0 scale per 32
// elements): X = 2^E with E the smallest integer such that amax <= 448 * 2^E,
// clamped to [-127, 127], so no element saturates.  With amax = m * 2^e,
// m in [0.5, 1): 448 * 2^(e-9) = 0.875 * 2^e, hence E = e - 9 if m <= 0.875,
// else e - 8.  An all-zero block takes E = -127.
__device__ __forceinline__ int mx_block_exp(float amax) {
  if (amax == 0.f) return -127;
  int e = 0;
  const float m = frexpf(amax, &e);
  const int E = m <= 0.875f ? e - 9 : e - 8;
  return max(-127, min(127, E));
}

// Power of two 2^k for k in [-149, 127], exact.
__device__ __forceinline__ float pow2_exact(int k) {
  return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// Location of cache row (sequence b, KV head h, token t) in elements of
// head_dim; returns -1 (and raises an error bit) for an invalid page.
__device__ __forceinline__ int64_t cache_row(const CacheView& c, int b, int h, int t,
                                             unsigned int* err) {
  if (c.paged) {
    int pi = t >> c.page_shift;
    if (pi >= c.max_pages_per_seq) { raise_error(err, FP8KV_DEVERR_SEQ_TOO_LONG); return -1; }
    int page = c.page_table[(int64_t)b * c.max_pages_per_seq + pi];
    if (page < 0 || page >= c.num_pages) { raise_error(err, FP8KV_DEVERR_BAD_PAGE); return -1; }
    return ((int64_t)page * c.kv_heads + h) * c.page_size + (t & (c.page_size - 1));
  }
  if (t >= c.max_tokens) { raise_error(err, FP8KV_DEVERR_SEQ_TOO_LONG); return -1; }
  return ((int64_t)b * c.kv_heads + h) * c.max_tokens + t;
}

__device__ __forceinline__ int cache_capacity(const CacheView& c) {
  return c.paged ? c.max_pages_per_seq * c.page_size : c.max_tokens;
}

// Host-side caches of the launch code (kernel attributes, occupancy) are
// shared by every host thread that calls the library: one lock guards them.
inline std::mutex& host_cache_lock() {
  static std::mutex m;
  return m;
}

// Opt a kernel into `bytes` of dynamic shared memory, once per (kernel,
// device).  A failure is read and cleared before it is returned, so that it
// does not stay pending on the stream.
inline cudaError_t ensure_smem_optin(const void* func, int bytes) {
  constexpr int kMaxDev = 64, kMaxFn = 128;
  static const void* done_fn[kMaxDev][kMaxFn];
  static int done_n[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { (void)cudaGetLastError(); return e; }
  if (dev < 0 || dev >= kMaxDev) dev = 0;
  std::lock_guard<std::mutex> lock(host_cache_lock());
  for (int i = 0; i < done_n[dev]; ++i)
    if (done_fn[dev][i] == func) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) { (void)cudaGetLastError(); return e; }
  if (done_n[dev] < kMaxFn) done_fn[dev][done_n[dev]++] = func;
  return cudaSuccess;
}

}  // namespace fp8kv
