/*
 * fp8kv.h -- C ABI of the GB300 (sm_103a) FP8-KV attention library.
 *
 * Fused attention over a quantised KV cache.  K and V live in HBM as FP8 E4M3
 * codes with one fp32 scale per (token, KV head), scale = amax(|row|)/448 over
 * the head dimension, written once when the token is appended ("FP8 KV cache
 * (fp8_kv, opt-in)", bullet "Storage").  K may instead be kept in bf16
 * ("K16/V8", "Fused KV-cache quantization", section "FlashInfer K16/V8"), and a
 * bf16/bf16 cache is provided as the control ("FP8 KV attention: hardware
 * paths and tile preparation", section "Collect the profiler evidence", the
 * four dtype controls).  Attention folds the K scale into the scores and the V
 * scale into P, with P rounded to bf16 before P.V ("FP8 KV cache", bullet
 * "Math"), and advances an online softmax tile by tile ("03 · 8n — FA-style
 * tiled prefill attention", section 2.1).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no memory.  Scratch space for decode is sized by
 *    fp8kv_decode_workspace_bytes() and passed in.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and returns a status; no C++ exception crosses the ABI.
 *  - A CUDA launch error is read and cleared (cudaGetLastError) before
 *    FP8KV_ERR_CUDA is returned, so it does not poison later work on the
 *    stream ("03 · 8n", section 3.3, the shared-memory opt-in pitfall).
 *  - Data-dependent faults found on the device (a sequence longer than the
 *    cache, a page id out of range, a bounded wait that ran out) never fault
 *    the GPU: the kernel skips the access and raises a bit in a device error
 *    word, read with fp8kv_get_device_error().
 *  - bf16 means IEEE binary32 truncated to its upper 16 bits (torch.bfloat16);
 *    codes are OCP E4M3 bytes (torch.float8_e4m3fn).
 *  - Supported shapes: head_dim 64 or 128; q_heads a multiple of kv_heads with
 *    group size q_heads/kv_heads from 1 to 8 for decode and from 1 to 16 for
 *    prefill; page_size 16, 32 or 64; contiguous capacity max_tokens a
 *    multiple of 16; at most 2^31 - 1 cache rows (batch x kv_heads x
 *    max_tokens, or num_pages x kv_heads x page_size).  Anything else
 *    returns FP8KV_ERR_UNSUPPORTED.
 *  - Calls may come from several host threads.  Per-device values (the
 *    device addresses of the library's error word and of the array of
 *    fp8kv_decode_attention_static, kernel attributes) are looked up on the
 *    first call on each device and kept for the life of the process:
 *    resetting a device (cudaDeviceReset) after the library has run on it is
 *    not supported.
 */
#ifndef FP8KV_H
#define FP8KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define FP8KV_API __attribute__((visibility("default")))
#else
#define FP8KV_API
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA. */
typedef struct CUstream_st *fp8kv_stream_t;

typedef enum {
  FP8KV_OK = 0,
  FP8KV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum */
  FP8KV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, group, page size */
  FP8KV_ERR_WORKSPACE = 3,     /* workspace pointer null or too small */
  FP8KV_ERR_CUDA = 4,          /* a CUDA runtime call failed (error cleared) */
  FP8KV_ERR_TIMEOUT = 5,       /* a bounded device wait ran out */
  FP8KV_ERR_DEVICE_CHECK = 6   /* the device error word is non-zero */
} fp8kv_status;

/* Cache element types: which of K and V are E4M3 codes and which are bf16. */
typedef enum {
  FP8KV_K8V8 = 0,    /* K codes, V codes (symmetric FP8)            */
  FP8KV_K16V8 = 1,   /* K bf16, V codes (no K transform)           */
  FP8KV_K16V16 = 2,  /* K bf16, V bf16 (the bf16-cache control)     */
  FP8KV_K8V16 = 3,   /* K codes, V bf16 (the remaining control)     */
  /* K as MXFP8: e4m3 codes with one E8M0 (power-of-two) scale per 32-dim
   * block, the four block bytes of a row in its 4-byte k_scale slot (byte b
   * = dims 32b..32b+31), as fp8kv_quantize_mx writes them; V codes with an
   * fp32 scale per row.  head_dim 128 only.  Every kernel weights each
   * block's partial dot product by its scale: the decode on both kernels
   * and the CUDA-core prefill; the transform paths and the tensor-core
   * prefill return FP8KV_ERR_UNSUPPORTED ("FP8 KV attention: hardware paths
   * and tile preparation", section "Measure block-scaled QK"). */
  FP8KV_MXK8V8 = 4
} fp8kv_kv_dtype;

typedef enum {
  FP8KV_LAYOUT_CONTIGUOUS = 0,  /* k, v: [batch][kv_heads][max_tokens][head_dim]
                                   scales: [batch][kv_heads][max_tokens]       */
  FP8KV_LAYOUT_PAGED = 1        /* k, v: [num_pages][kv_heads][page_size][head_dim]
                                   scales: [num_pages][kv_heads][page_size]
                                   token t of sequence b sits in page
                                   page_table[b][t / page_size], slot t % page_size */
} fp8kv_layout;

typedef enum { FP8KV_OUT_BF16 = 0, FP8KV_OUT_F32 = 1 } fp8kv_out_dtype;

/* Which split kernel a decode call runs.  AUTO picks the tensor cores
 * wherever that kernel is built (head_dim 128, 1 to 8 query heads per KV
 * head: it was measured faster at every group size), the CUDA cores
 * otherwise.  The tensor-core kernel (tcgen05) walks 128-token tiles; the
 * CUDA-core kernel walks 64-token tiles. */
typedef enum {
  FP8KV_KERNEL_AUTO = 0,
  FP8KV_KERNEL_CUDA_CORES = 1,
  FP8KV_KERNEL_TENSOR_CORES = 2,
  /* Decode only, K8V8 at head_dim 128: the tensor-core kernel on the
   * transform path.  Each landed e4m3 K tile is converted to f16 in shared
   * memory and QK runs as a 16-bit MMA on an f16 query, in place of the
   * native e4m3 QK; V, P and the merge are unchanged.  _K_F16: the softmax
   * warpgroup that owns the tile converts it; _K_F16_PRODUCER: the TMA
   * producer warp does.  Comparison points for where the K preparation runs
   * ("FP8 KV attention: hardware paths and tile preparation", sections
   * "Measure the BF16-Q/FP8-KV transform path" and "Pipeline the existing
   * transform"); AUTO never picks them.  Rejected (FP8KV_ERR_UNSUPPORTED)
   * for other dtypes and head dims, and by the prefill
   * (FP8KV_ERR_INVALID_ARG). */
  FP8KV_KERNEL_TENSOR_CORES_K_F16 = 3,
  FP8KV_KERNEL_TENSOR_CORES_K_F16_PRODUCER = 4
} fp8kv_decode_kernel;

/* Device error word bits (fp8kv_get_device_error). */
#define FP8KV_DEVERR_SEQ_TOO_LONG 0x1u   /* a length/position exceeds the cache */
#define FP8KV_DEVERR_BAD_PAGE 0x2u       /* a page id outside [0, num_pages)    */
#define FP8KV_DEVERR_TIMEOUT 0x4u        /* a bounded mbarrier wait ran out    */

/* A KV cache.  The struct is read on the host at every call (pass it by
 * pointer; it may live on the stack).  All pointers are device pointers owned
 * by the caller and 16-byte aligned.  For a bf16 side the scale pointer must
 * be NULL. */
typedef struct {
  int32_t dtype;              /* fp8kv_kv_dtype                                */
  int32_t layout;             /* fp8kv_layout                                  */
  int32_t batch;              /* sequences (rows of page_table)                */
  int32_t kv_heads;
  int32_t head_dim;           /* 64 or 128                                     */
  int32_t max_tokens;         /* contiguous: capacity per sequence (mult. of 16) */
  int32_t page_size;          /* paged: tokens per page (16, 32 or 64)         */
  int32_t num_pages;          /* paged: pages in the pool                      */
  int32_t max_pages_per_seq;  /* paged: columns of page_table                  */
  int32_t rope_positions;     /* rotated bias: rows of rope_cos / rope_sin    */
  void *k;                    /* e4m3 codes (uint8) or bf16, layout above      */
  void *v;
  float *k_scale;             /* fp32 per (token, KV head); NULL if K is bf16;
                                 FP8KV_MXK8V8: the row's four E8M0 bytes      */
  float *v_scale;             /* NULL if V is bf16                             */
  const int32_t *page_table;  /* paged: [batch][max_pages_per_seq]; else NULL  */
  /* Pre-bias residual keys ("Fused KV-cache quantization", section
   * "Bias-aware symmetric FP8"): NULL, or [kv_heads][head_dim] fp32, a fixed
   * key bias b kept exact.  Appends then quantise each K row's residual
   * fp32(k) - b with the per-row rule, so a large bias no longer sets the
   * row's scale.  Only for FP8KV_K8V8 and FP8KV_K8V16 (else
   * FP8KV_ERR_INVALID_ARG).  Attention reads the residual codes as the keys:
   * the dropped score term q.b is the same for every key a query row sees,
   * so it cancels in the softmax.  b is one vector per KV head for all
   * positions, unless rope_cos and rope_sin are set (below). */
  const float *k_bias;
  /* Rotated pre-bias residual keys (same sections; the pages' post-rotary
   * residual layout): NULL, or both set, with k_bias.  The cache then holds
   * rotated keys and b is a bias added before the rotary embedding, so the
   * key at position t carries R_t b.  Appends quantise fp32(k) - R_t b, and
   * attention reads dequant(r) + R_t b.  R_t is the "rotate half" layout:
   * dims i and i + head_dim/2 form pair i at angle theta_{t,i}, with
   *   (R_t b)_i           = fma(b_i, cos, -(b_{i+head_dim/2} * sin))
   *   (R_t b)_{i+head_dim/2} = fma(b_{i+head_dim/2}, cos, b_i * sin)
   * in fp32 (each product with sin rounded first), cos = rope_cos[t][i],
   * sin = rope_sin[t][i]: [rope_positions][head_dim/2] fp32 device arrays,
   * 16-byte aligned, rope_positions at least the cache's capacity (else
   * FP8KV_ERR_INVALID_ARG).  Built on the CUDA-core kernels: the decode
   * (AUTO picks it) and the prefill; the tensor-core kernels return
   * FP8KV_ERR_UNSUPPORTED. */
  const float *rope_cos;
  const float *rope_sin;
} fp8kv_cache;

/* Quantise `rows` rows of `head_dim` bf16 values into E4M3 codes and one fp32
 * scale per row ("FP8 KV cache (fp8_kv, opt-in)", bullet "Storage",
 * quantize_fp8_kv): scale = amax(|row|)/448 (IEEE fp32 division), code =
 * round-to-nearest-even, saturating encode of the IEEE fp32 quotient x/scale;
 * an all-zero row gets scale 0 and codes 0x00.
 *   x:      [rows][head_dim] bf16      codes: [rows][head_dim] uint8
 *   scales: [rows] fp32 */
FP8KV_API fp8kv_status fp8kv_quantize(const void *x, int64_t rows, int32_t head_dim,
                            uint8_t *codes, float *scales,
                            fp8kv_stream_t stream);

/* Quantise `rows` rows of `head_dim` bf16 values into MXFP8: E4M3 codes and
 * one E8M0 byte per 32-element block ("FP8 KV attention: hardware paths and
 * tile preparation", section "Measure block-scaled QK").  Block scale
 * X = 2^E, E the smallest integer with amax(|block|) <= 448 * 2^E, clamped
 * to [-127, 127] (no element saturates; an all-zero block gets E = -127);
 * byte = E + 127; code = round-to-nearest-even encode of the fp32 product
 * x * 2^-E (the sign of a zero is kept).
 *   x:      [rows][head_dim] bf16      codes: [rows][head_dim] uint8
 *   scales: [rows][head_dim / 32] uint8 (E8M0)
 * head_dim 64 or 128 (else FP8KV_ERR_UNSUPPORTED). */
FP8KV_API fp8kv_status fp8kv_quantize_mx(const void *x, int64_t rows, int32_t head_dim,
                               uint8_t *codes, uint8_t *scales,
                               fp8kv_stream_t stream);

/* Append new tokens to the cache: each (token, KV head) row of K and of V is
 * quantised as in fp8kv_quantize (or copied, for a bf16 side) and written
 * once into its slot ("FP8 KV cache", bullet "Storage", Fp8KVCache.append).
 *   k_new, v_new: [n_tokens][kv_heads][head_dim] bf16
 *   seq_idx, pos: [n_tokens] int32 device arrays; token i goes to sequence
 *                 seq_idx[i] at position pos[i].
 * Rows whose position is outside the cache, or whose page id is out of range,
 * are skipped and raise a device error bit. */
FP8KV_API fp8kv_status fp8kv_append(const fp8kv_cache *cache, const void *k_new,
                          const void *v_new, const int32_t *seq_idx,
                          const int32_t *pos, int64_t n_tokens,
                          fp8kv_stream_t stream);

/* The flash-decoding split count a decode call will use for `num_splits`
 * (0 = automatic: about four CTAs per SM, "FP8 KV cache", bullet "Speed").
 * Returns 0 on invalid arguments. */
FP8KV_API int32_t fp8kv_decode_num_splits(const fp8kv_cache *cache, int32_t q_heads,
                                int32_t num_splits, int32_t kernel);

/* Bytes of workspace fp8kv_decode_attention needs for these arguments: the
 * fp32 partials (O, m, l) of every (sequence, query head, split). */
FP8KV_API size_t fp8kv_decode_workspace_bytes(const fp8kv_cache *cache, int32_t q_heads,
                                    int32_t num_splits, int32_t kernel);

/* Decode attention: one query token per sequence, grouped-query heads, per-
 * sequence lengths ("FP8 KV cache", bullet "Math", fp8_kv_attention).  Kernel
 * 1 splits each sequence's cache over CTAs (flash-decoding, bullet "Speed")
 * and writes fp32 partials; kernel 2 merges them.
 *   q:        [batch][q_heads][head_dim] bf16; query head h reads KV head
 *             h / (q_heads / kv_heads)
 *   seq_lens: [batch] int32 device array; sequence b attends its tokens
 *             0..seq_lens[b]-1; a length of 0 gives a zero output row
 *   sm_scale: softmax scale (1/sqrt(head_dim) in the usual case)
 *   kernel:   fp8kv_decode_kernel
 *   out:      [batch][q_heads][head_dim], bf16 or fp32 per out_dtype
 * Split boundaries are multiples of the kernel's tile (64 or 128 tokens), so
 * results for different num_splits differ only by fp32 re-association. */
FP8KV_API fp8kv_status fp8kv_decode_attention(const void *q, const fp8kv_cache *cache,
                                    const int32_t *seq_lens, int32_t q_heads,
                                    float sm_scale, int32_t num_splits, int32_t kernel,
                                    void *workspace, size_t workspace_bytes,
                                    void *out, int32_t out_dtype,
                                    fp8kv_stream_t stream);

/* The two kernels of fp8kv_decode_attention as separate calls (same
 * arguments, same results).  fp8kv_decode_split runs the flash-decoding split
 * kernel and leaves the fp32 partials in `workspace`; fp8kv_decode_merge
 * reduces them into `out`.  Both must be given the same cache, q_heads,
 * num_splits and kernel, and the merge must follow the split on the same
 * stream (or be ordered after it). */
FP8KV_API fp8kv_status fp8kv_decode_split(const void *q, const fp8kv_cache *cache,
                                          const int32_t *seq_lens, int32_t q_heads,
                                          float sm_scale, int32_t num_splits, int32_t kernel,
                                          void *workspace, size_t workspace_bytes,
                                          fp8kv_stream_t stream);
FP8KV_API fp8kv_status fp8kv_decode_merge(const fp8kv_cache *cache, int32_t q_heads,
                                          int32_t num_splits, int32_t kernel,
                                          const void *workspace,
                                          size_t workspace_bytes, void *out,
                                          int32_t out_dtype, fp8kv_stream_t stream);

/* One decode step in one call: append the new token of every sequence to
 * the cache (as fp8kv_append, at position seq_lens[b] - 1: the lengths
 * already count the new token), then decode attention over seq_lens[b]
 * tokens, as fp8kv_decode_attention.  On the tensor-core kernel all of it
 * is one launch: the CTA that owns the new token's tile writes it before
 * loading that tile, and the last split of each (sequence, KV head) to
 * finish merges the partials, so no separate append or merge kernel runs.
 *   k_new, v_new: [batch][kv_heads][head_dim] bf16
 *   workspace:    fp8kv_decode_step_workspace_bytes() bytes; it also holds
 *                 one arrival counter per (sequence, KV head), which must be
 *                 zero before the first call (allocate it zero-filled).
 *                 Every call that returns FP8KV_OK and whose device error
 *                 word stays clear leaves the counters zero again; after a
 *                 timeout, zero the workspace before reusing it.
 *   flags:        0, or FP8KV_STEP_EARLY_CACHE_READ (below).
 * q, k_new, v_new, seq_lens and out may also point to page-locked host
 * memory (cudaHostAlloc / cudaMallocHost), which the device addresses at
 * the same pointer under unified addressing: the kernels then read the
 * step's inputs and write its output across the host link themselves, with
 * no copy calls (on GB300 the link is the coherent chip-to-chip one).
 * Other arguments as in fp8kv_decode_attention. */
FP8KV_API size_t fp8kv_decode_step_workspace_bytes(const fp8kv_cache *cache, int32_t q_heads,
                                                   int32_t num_splits, int32_t kernel);
FP8KV_API fp8kv_status fp8kv_decode_step(const void *q, const void *k_new, const void *v_new,
                                         const fp8kv_cache *cache, const int32_t *seq_lens,
                                         int32_t q_heads, float sm_scale, int32_t num_splits,
                                         int32_t kernel, void *workspace, size_t workspace_bytes,
                                         void *out, int32_t out_dtype, uint32_t flags,
                                         fp8kv_stream_t stream);

/* Flag of fp8kv_decode_step (tensor-core kernel; ignored by the CUDA-core
 * kernel): the step may start before the kernel issued just before it on
 * the stream has finished (programmatic dependent launch).  It then reads
 * seq_lens and starts streaming the cache rows already appended before this
 * call while that kernel runs, and waits for it before it reads q, k_new or
 * v_new and before it writes anything (the new rows, the workspace, out).
 * Set it only when the kernel issued just before on the stream writes
 * neither this cache nor seq_lens -- as in a model, where the step follows
 * the query/key/value projection and every layer has its own cache. */
#define FP8KV_STEP_EARLY_CACHE_READ 1u

/* Decode attention that allocates nothing (a convenience of this library;
 * the source pages have no such call).  Same arguments and results as
 * fp8kv_decode_attention without the workspace: the fp32 partials go to a
 * fixed array of fp8kv_decode_static_scratch_bytes() bytes (16 MiB) compiled
 * into the library, which every GPU that loads the library keeps until the
 * process exits.  The kernel is chosen as with FP8KV_KERNEL_AUTO.  It is
 * for callers that cannot call cudaMalloc -- for
 * example a runtime whose memory pool owns the device and forbids
 * allocation on its serving path, or a plugin given only its input and
 * output tensors.  The call makes no cudaMalloc, cudaFree or allocating
 * library call.
 *  - With num_splits 0 the split count is the automatic one, lowered to the
 *    largest count whose partials fit when they would not.  A call whose
 *    partials cannot fit (an explicit num_splits too large, or not even one
 *    split fitting) returns FP8KV_ERR_WORKSPACE and launches nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents; nothing in it needs to start at zero.  Calls that overlap on
 *    the GPU (other streams, or other host threads) race on it: order them. */
FP8KV_API fp8kv_status fp8kv_decode_attention_static(const void *q, const fp8kv_cache *cache,
                                                     const int32_t *seq_lens, int32_t q_heads,
                                                     float sm_scale, int32_t num_splits,
                                                     void *out, int32_t out_dtype,
                                                     fp8kv_stream_t stream);

/* Size in bytes of the fixed array used by fp8kv_decode_attention_static. */
FP8KV_API size_t fp8kv_decode_static_scratch_bytes(void);

/* Causal prefill attention over the cache ("03 · 8n — FA-style tiled prefill
 * attention", sections 2-3): query tiles, online softmax over 64-token KV
 * tiles.  Query i of sequence b sits at absolute position q_pos0[b] + i and
 * attends cache tokens 0..q_pos0[b]+i (the cache must already hold them:
 * append first).
 *   q:      [batch][n_q][q_heads][head_dim] bf16
 *   q_pos0: [batch] int32 device array
 *   kernel: FP8KV_KERNEL_* -- TENSOR_CORES (128-query tiles on tcgen05, K8V8
 *           with head_dim 128 only, else FP8KV_ERR_UNSUPPORTED),
 *           CUDA_CORES (64-query tiles, every dtype, MXFP8 keys included),
 *           AUTO (tensor cores where built)
 *   out:    [batch][n_q][q_heads][head_dim], bf16 or fp32 per out_dtype */
FP8KV_API fp8kv_status fp8kv_prefill_attention(const void *q, const fp8kv_cache *cache,
                                     const int32_t *q_pos0, int32_t n_q,
                                     int32_t q_heads, float sm_scale, int32_t kernel,
                                     void *out, int32_t out_dtype, fp8kv_stream_t stream);

/* Read (and, if `clear` is non-zero, reset) the device error word of the
 * current device.  Synchronous: waits for all work on the device. */
FP8KV_API fp8kv_status fp8kv_get_device_error(uint32_t *bits, int32_t clear);

/* Human-readable name of a status. */
FP8KV_API const char *fp8kv_status_string(fp8kv_status status);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H */
