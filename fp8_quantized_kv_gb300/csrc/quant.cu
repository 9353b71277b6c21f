// quant.cu -- quantise bf16 K/V rows into E4M3 codes + one fp32 scale per
// (token, KV head), and append them to a contiguous or paged cache.
//
// "FP8 KV cache (fp8_kv, opt-in)", bullet "Storage": K and V in e4m3 with one
// fp32 scale per (token, KV head), scale = amax(|row|)/448 over the head
// dimension, written once when the token is appended and never re-quantised.
//
// One warp per row: each lane loads its slice of the row with one 4- or
// 8-byte load, the row amax is a warp-shuffle max, the scale is one IEEE fp32
// division (amax/448), and every element is encoded from the IEEE fp32
// quotient x/scale by the hardware round-to-nearest-even, saturating
// conversion (cvt.rn.satfinite.e4m3x2.f32).  An all-zero row gets scale 0 and
// codes 0x00 (the pages are silent there).  Memory-bound streaming: 2*D bytes
// in, D + 4 bytes out per row.
#include "params.cuh"

namespace fp8kv {

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise one row of D bf16 values held by a warp (EPL elements per lane,
// lane l owning elements [l*EPL, l*EPL+EPL)).  Writes EPL codes per lane.
template <int EPL>
__device__ __forceinline__ void quantize_warp_row(const float (&x)[EPL], uint8_t* codes_row,
                                                  float* scale_out, int lane) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = warp_max(amax);
  const float scale = __fdiv_rn(amax, 448.0f);
  uint32_t packed = 0;
  if (amax != 0.f) {
#pragma unroll
    for (int i = 0; i < EPL; i += 2) {
      float y0 = __fdiv_rn(x[i], scale);
      float y1 = __fdiv_rn(x[i + 1], scale);
      packed |= (uint32_t)cvt_e4m3x2(y0, y1) << (8 * i);
    }
  }
  if (EPL == 4)
    *reinterpret_cast<uint32_t*>(codes_row + lane * 4) = packed;
  else
    *reinterpret_cast<uint16_t*>(codes_row + lane * 2) = (uint16_t)packed;
  if (lane == 0) *scale_out = scale;
}

// MXFP8 row held by a warp (EPL elements per lane): block b is lanes
// [b*32/EPL, (b+1)*32/EPL).  The block amax is a shuffle max over its lanes;
// each element is encoded from the fp32 product x * 2^-E (exact unless the
// product is below the fp32 normal range); the first lane of each block
// writes its E8M0 byte E + 127 to scale_row[b].
template <int EPL>
__device__ __forceinline__ void mx_quantize_warp_row(const float (&x)[EPL], uint8_t* codes_row,
                                                     uint8_t* scale_row, int lane) {
  constexpr int LPB = 32 / EPL;                 // lanes per 32-element block
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < LPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int E = mx_block_exp(amax);
  const float inv = pow2_exact(-E);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < EPL; i += 2) packed |= (uint32_t)cvt_e4m3x2(x[i] * inv, x[i + 1] * inv) << (8 * i);
  if (EPL == 4)
    *reinterpret_cast<uint32_t*>(codes_row + lane * 4) = packed;
  else
    *reinterpret_cast<uint16_t*>(codes_row + lane * 2) = (uint16_t)packed;
  if (lane % LPB == 0) scale_row[lane / LPB] = (uint8_t)(E + 127);
}

template <int EPL>
__device__ __forceinline__ void load_bf16_slice(const __nv_bfloat16* row, int lane, float (&x)[EPL]) {
  if (EPL == 4) {
    uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
    float a[2], b[2];
    bf16x2_to_f32(u.x, a);
    bf16x2_to_f32(u.y, b);
    x[0] = a[0]; x[1] = a[1]; x[2] = b[0]; x[3] = b[1];
  } else {
    uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
    float a[2];
    bf16x2_to_f32(u, a);
    x[0] = a[0]; x[1] = a[1];
  }
}

// Standalone quantiser: rows of D = 32*EPL values.
template <int EPL>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                            int64_t rows, uint8_t* __restrict__ codes,
                                                            float* __restrict__ scales) {
  constexpr int D = 32 * EPL;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float v[EPL];
  load_bf16_slice<EPL>(x + row * D, lane, v);
  quantize_warp_row<EPL>(v, codes + row * D, scales + row, lane);
}

// Standalone MXFP8 quantiser: rows of D = 32*EPL values -> codes and D/32
// E8M0 bytes per row.
template <int EPL>
__global__ void __launch_bounds__(256) quantize_mx_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                               int64_t rows, uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ scales) {
  constexpr int D = 32 * EPL;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float v[EPL];
  load_bf16_slice<EPL>(x + row * D, lane, v);
  mx_quantize_warp_row<EPL>(v, codes + row * D, scales + row * (D / 32), lane);
}

// Append: warp per (token, KV head, K-or-V) row.  KE/VE: element kind of the
// K and V sides of the cache (E4M3 codes or bf16 copies).
template <int EPL, int KE, int VE>
__global__ void __launch_bounds__(256) append_kernel(CacheView c, const __nv_bfloat16* __restrict__ k_new,
                                                     const __nv_bfloat16* __restrict__ v_new,
                                                     const int32_t* __restrict__ seq_idx,
                                                     const int32_t* __restrict__ pos, int64_t n_tokens,
                                                     unsigned int* err) {
  constexpr int D = 32 * EPL;
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t rows = n_tokens * c.kv_heads;
  if (w >= 2 * rows) return;
  const bool is_v = w >= rows;
  const int64_t r = is_v ? w - rows : w;
  const int64_t tok = r / c.kv_heads;
  const int h = (int)(r - tok * c.kv_heads);
  const int b = seq_idx[tok];
  const int t = pos[tok];
  if (b < 0 || b >= c.batch || t < 0) {
    if (lane == 0) raise_error(err, FP8KV_DEVERR_SEQ_TOO_LONG);
    return;
  }
  const int64_t dst = cache_row(c, b, h, t, lane == 0 ? err : nullptr);
  if (dst < 0) return;
  const __nv_bfloat16* src = (is_v ? v_new : k_new) + r * D;
  const int kind = is_v ? VE : KE;
  if (kind == ELEM_BF16) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(const_cast<uint8_t*>(is_v ? c.v : c.k)) + dst * D;
    if (EPL == 4)
      reinterpret_cast<uint2*>(out)[lane] = reinterpret_cast<const uint2*>(src)[lane];
    else
      reinterpret_cast<uint32_t*>(out)[lane] = reinterpret_cast<const uint32_t*>(src)[lane];
    return;
  }
  float v[EPL];
  load_bf16_slice<EPL>(src, lane, v);
  if (!is_v && c.k_bias != nullptr) {            // pre-bias residual: fp32(k) - b, or - R_t b
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      v[i] -= c.rope_cos != nullptr ? rope_bias(c, h, t, lane * EPL + i) : c.k_bias[h * D + lane * EPL + i];
  }
  uint8_t* codes = const_cast<uint8_t*>(is_v ? c.v : c.k) + dst * D;
  float* scale = const_cast<float*>(is_v ? c.v_scale : c.k_scale) + dst;
  if (kind == ELEM_MX)
    mx_quantize_warp_row<EPL>(v, codes, reinterpret_cast<uint8_t*>(scale), lane);
  else
    quantize_warp_row<EPL>(v, codes, scale, lane);
}

// Decode-step append: the new token of sequence b goes to position
// seq_lens[b] - 1 (the length already counts it).  k_new, v_new: [B][Hkv][D].
template <int EPL, int KE, int VE>
__global__ void __launch_bounds__(256) append_step_kernel(CacheView c, const __nv_bfloat16* __restrict__ k_new,
                                                          const __nv_bfloat16* __restrict__ v_new,
                                                          const int32_t* __restrict__ seq_lens, unsigned int* err) {
  constexpr int D = 32 * EPL;
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t rows = (int64_t)c.batch * c.kv_heads;
  if (w >= 2 * rows) return;
  const bool is_v = w >= rows;
  const int64_t r = is_v ? w - rows : w;
  const int b = (int)(r / c.kv_heads), h = (int)(r - (int64_t)b * c.kv_heads);
  const int t = seq_lens[b] - 1;
  if (t < 0) return;                                   // an empty sequence appends nothing
  const int64_t dst = cache_row(c, b, h, t, lane == 0 ? err : nullptr);
  if (dst < 0) return;
  const __nv_bfloat16* src = (is_v ? v_new : k_new) + r * D;
  const int kind = is_v ? VE : KE;
  if (kind == ELEM_BF16) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(const_cast<uint8_t*>(is_v ? c.v : c.k)) + dst * D;
    if (EPL == 4)
      reinterpret_cast<uint2*>(out)[lane] = reinterpret_cast<const uint2*>(src)[lane];
    else
      reinterpret_cast<uint32_t*>(out)[lane] = reinterpret_cast<const uint32_t*>(src)[lane];
    return;
  }
  float v[EPL];
  load_bf16_slice<EPL>(src, lane, v);
  if (!is_v && c.k_bias != nullptr) {            // pre-bias residual: fp32(k) - b, or - R_t b
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      v[i] -= c.rope_cos != nullptr ? rope_bias(c, h, t, lane * EPL + i) : c.k_bias[h * D + lane * EPL + i];
  }
  uint8_t* codes = const_cast<uint8_t*>(is_v ? c.v : c.k) + dst * D;
  float* scale = const_cast<float*>(is_v ? c.v_scale : c.k_scale) + dst;
  if (kind == ELEM_MX)
    mx_quantize_warp_row<EPL>(v, codes, reinterpret_cast<uint8_t*>(scale), lane);
  else
    quantize_warp_row<EPL>(v, codes, scale, lane);
}

// ------------------------------------------------------------ launchers ---
cudaError_t launch_quantize(const void* x, int64_t rows, int head_dim, uint8_t* codes, float* scales,
                            cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int warps = 8;
  const unsigned grid = (unsigned)((rows + warps - 1) / warps);
  if (head_dim == 128)
    quantize_rows_kernel<4><<<grid, 32 * warps, 0, s>>>((const __nv_bfloat16*)x, rows, codes, scales);
  else
    quantize_rows_kernel<2><<<grid, 32 * warps, 0, s>>>((const __nv_bfloat16*)x, rows, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mx(const void* x, int64_t rows, int head_dim, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int warps = 8;
  const unsigned grid = (unsigned)((rows + warps - 1) / warps);
  if (head_dim == 128)
    quantize_mx_rows_kernel<4><<<grid, 32 * warps, 0, s>>>((const __nv_bfloat16*)x, rows, codes, scales);
  else
    quantize_mx_rows_kernel<2><<<grid, 32 * warps, 0, s>>>((const __nv_bfloat16*)x, rows, codes, scales);
  return cudaGetLastError();
}

template <int EPL>
static void append_dispatch(int dtype, unsigned grid, cudaStream_t s, const CacheView& c,
                            const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* si,
                            const int32_t* ps, int64_t n, unsigned int* err) {
  if (dtype == FP8KV_K8V8)
    append_kernel<EPL, ELEM_E4M3, ELEM_E4M3><<<grid, 256, 0, s>>>(c, k, v, si, ps, n, err);
  else if (dtype == FP8KV_K16V8)
    append_kernel<EPL, ELEM_BF16, ELEM_E4M3><<<grid, 256, 0, s>>>(c, k, v, si, ps, n, err);
  else if (dtype == FP8KV_K8V16)
    append_kernel<EPL, ELEM_E4M3, ELEM_BF16><<<grid, 256, 0, s>>>(c, k, v, si, ps, n, err);
  else if (dtype == FP8KV_MXK8V8)
    append_kernel<EPL, ELEM_MX, ELEM_E4M3><<<grid, 256, 0, s>>>(c, k, v, si, ps, n, err);
  else
    append_kernel<EPL, ELEM_BF16, ELEM_BF16><<<grid, 256, 0, s>>>(c, k, v, si, ps, n, err);
}

cudaError_t launch_append(const CacheView& c, int dtype, const void* k_new, const void* v_new,
                          const int32_t* seq_idx, const int32_t* pos, int64_t n_tokens,
                          unsigned int* err, cudaStream_t s) {
  if (n_tokens == 0) return cudaSuccess;
  const int64_t warps_needed = 2 * n_tokens * c.kv_heads;
  const unsigned grid = (unsigned)((warps_needed + 7) / 8);
  const auto* k = (const __nv_bfloat16*)k_new;
  const auto* v = (const __nv_bfloat16*)v_new;
  if (c.head_dim == 128)
    append_dispatch<4>(dtype, grid, s, c, k, v, seq_idx, pos, n_tokens, err);
  else
    append_dispatch<2>(dtype, grid, s, c, k, v, seq_idx, pos, n_tokens, err);
  return cudaGetLastError();
}

template <int EPL>
static void append_step_dispatch(int dtype, unsigned grid, cudaStream_t s, const CacheView& c,
                                 const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* lens,
                                 unsigned int* err) {
  if (dtype == FP8KV_K8V8)
    append_step_kernel<EPL, ELEM_E4M3, ELEM_E4M3><<<grid, 256, 0, s>>>(c, k, v, lens, err);
  else if (dtype == FP8KV_K16V8)
    append_step_kernel<EPL, ELEM_BF16, ELEM_E4M3><<<grid, 256, 0, s>>>(c, k, v, lens, err);
  else if (dtype == FP8KV_K8V16)
    append_step_kernel<EPL, ELEM_E4M3, ELEM_BF16><<<grid, 256, 0, s>>>(c, k, v, lens, err);
  else if (dtype == FP8KV_MXK8V8)
    append_step_kernel<EPL, ELEM_MX, ELEM_E4M3><<<grid, 256, 0, s>>>(c, k, v, lens, err);
  else
    append_step_kernel<EPL, ELEM_BF16, ELEM_BF16><<<grid, 256, 0, s>>>(c, k, v, lens, err);
}

cudaError_t launch_append_step(const CacheView& c, int dtype, const void* k_new, const void* v_new,
                               const int32_t* seq_lens, unsigned int* err, cudaStream_t s) {
  const int64_t warps_needed = 2 * (int64_t)c.batch * c.kv_heads;
  if (warps_needed == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((warps_needed + 7) / 8);
  const auto* k = (const __nv_bfloat16*)k_new;
  const auto* v = (const __nv_bfloat16*)v_new;
  if (c.head_dim == 128)
    append_step_dispatch<4>(dtype, grid, s, c, k, v, seq_lens, err);
  else
    append_step_dispatch<2>(dtype, grid, s, c, k, v, seq_lens, err);
  return cudaGetLastError();
}

}  // namespace fp8kv
