// params.cuh -- kernel parameter blocks and launcher declarations shared by
// the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include "common.cuh"

namespace fp8kv {

struct DecodeParams {
  CacheView c;
  const __nv_bfloat16* q;    // [B][Hq][D]
  const int32_t* seq_lens;   // [B]
  float* part_o;             // [B][Hq][S][D]  unnormalised O of each split
  float* part_m;             // [B][Hq][S]     running max, log2 domain
  float* part_l;             // [B][Hq][S]     running sum
  unsigned int* err;         // device error word
  int q_heads, group, num_splits, chunk_tiles;
  float scale_log2;          // sm_scale * log2(e)
  // Fused decode step (tensor-core kernel only; zero/null otherwise):
  const __nv_bfloat16* k_new;  // [B][Hkv][D] new token of each sequence, appended at seq_lens[b]-1
  const __nv_bfloat16* v_new;
  int* counters;             // [B][Hkv] arrivals of finished splits (zero between calls)
  void* out;                 // [B][Hq][D] merged output (bf16 or fp32)
  int out_f32;
  int fused;
  int cluster;               // fused step launched with the splits of a (sequence, KV head) as one cluster
  int pdl;                   // fused step launched as a programmatic dependent of the previous kernel
  int k_f16;                 // tensor-core kernel on the transform path (K converted to f16 on chip):
                             // 0 no, 1 by the softmax warpgroups, 2 by the producer warp
  int hpc, hpc_shift;        // tensor-core kernel: KV heads per CTA (a power of two; a tile is
                             // 128 rows = hpc heads x 128/hpc tokens)
};

// KV heads one tensor-core decode CTA takes (1, 2, 4 or 8): on a paged cache
// with fewer than 8 query heads per KV head, neighbouring KV heads' rows of
// a page are contiguous in the pool, so a CTA taking 8 / G of them fetches
// each page side with one larger copy (the paged decode is bound by the
// number of copies); everything else takes one KV head.
inline int decode_heads_per_cta(int paged, int kv_heads, int group, int page_size) {
  if (!paged || group < 1 || group >= 8 || 8 % group != 0) return 1;
  int hpc = 8 / group;
  while (hpc > 1 && (kv_heads % hpc != 0 || hpc * page_size > 128)) hpc /= 2;
  return hpc;
}

struct PrefillParams {
  CacheView c;
  const __nv_bfloat16* q;    // [B][n_q][Hq][D]
  const int32_t* q_pos0;     // [B]
  void* out;                 // [B][n_q][Hq][D]
  unsigned int* err;
  int n_q, q_heads, group, out_f32;
  float scale_log2;
};

cudaError_t launch_quantize(const void* x, int64_t rows, int head_dim, uint8_t* codes, float* scales,
                            cudaStream_t s);
cudaError_t launch_quantize_mx(const void* x, int64_t rows, int head_dim, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s);
cudaError_t launch_append(const CacheView& c, int dtype, const void* k_new, const void* v_new,
                          const int32_t* seq_idx, const int32_t* pos, int64_t n_tokens,
                          unsigned int* err, cudaStream_t s);
cudaError_t launch_append_step(const CacheView& c, int dtype, const void* k_new, const void* v_new,
                               const int32_t* seq_lens, unsigned int* err, cudaStream_t s);
cudaError_t launch_decode_fma(const DecodeParams& p, int dtype, int batch, cudaStream_t st);
cudaError_t launch_decode_mma(const DecodeParams& p, int dtype, int batch, cudaStream_t st);
cudaError_t launch_decode_merge(const float* part_o, const float* part_m, const float* part_l, int S,
                                int64_t rows, int head_dim, void* out, int out_f32, cudaStream_t st);
cudaError_t launch_prefill_fma(const PrefillParams& p, int dtype, int batch, cudaStream_t st);
cudaError_t launch_prefill_tc(const PrefillParams& p, int batch, cudaStream_t st);

}  // namespace fp8kv
