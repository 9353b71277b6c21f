// api.cu -- the extern "C" boundary: argument checks, launch configuration,
// status codes.  Every entry point validates on the host, launches on the
// caller's stream and returns; nothing here allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "params.cuh"

namespace fp8kv {

// Device error word (one per device that loads the library).  Kernels get
// its address as an argument.
__device__ unsigned int g_device_error;

// Per-device values looked up on first use and kept; atomics, so host
// threads making their first call at once (each looking the value up and
// storing the same result) do not race.
static unsigned int* device_error_ptr() {
  constexpr int kMaxDev = 64;
  static std::atomic<unsigned int*> ptrs[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return nullptr; }
  if (dev < 0 || dev >= kMaxDev) return nullptr;
  unsigned int* p = ptrs[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_device_error) != cudaSuccess) { (void)cudaGetLastError(); return nullptr; }
    p = static_cast<unsigned int*>(a);
    ptrs[dev].store(p, std::memory_order_release);
  }
  return p;
}

static int sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> counts[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return 148; }
  if (dev < 0 || dev >= kMaxDev) return 148;
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = 148;
    }
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

static fp8kv_status check_cache(const fp8kv_cache* c, CacheView* view) {
  if (c == nullptr) return FP8KV_ERR_INVALID_ARG;
  if (c->dtype < FP8KV_K8V8 || c->dtype > FP8KV_MXK8V8) return FP8KV_ERR_INVALID_ARG;
  if (c->layout != FP8KV_LAYOUT_CONTIGUOUS && c->layout != FP8KV_LAYOUT_PAGED) return FP8KV_ERR_INVALID_ARG;
  if (c->batch < 0 || c->kv_heads <= 0 || c->head_dim <= 0) return FP8KV_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return FP8KV_ERR_UNSUPPORTED;
  if (c->dtype == FP8KV_MXK8V8 && c->head_dim != 128) return FP8KV_ERR_UNSUPPORTED;
  if (c->k == nullptr || c->v == nullptr) return FP8KV_ERR_INVALID_ARG;
  const bool k8 = c->dtype == FP8KV_K8V8 || c->dtype == FP8KV_K8V16 || c->dtype == FP8KV_MXK8V8;
  const bool v8 = c->dtype == FP8KV_K8V8 || c->dtype == FP8KV_K16V8 || c->dtype == FP8KV_MXK8V8;
  if (k8 != (c->k_scale != nullptr) || v8 != (c->v_scale != nullptr)) return FP8KV_ERR_INVALID_ARG;
  if (c->k_bias != nullptr && c->dtype != FP8KV_K8V8 && c->dtype != FP8KV_K8V16) return FP8KV_ERR_INVALID_ARG;
  // rotated bias: both tables, with a bias
  if ((c->rope_cos == nullptr) != (c->rope_sin == nullptr)) return FP8KV_ERR_INVALID_ARG;
  if (c->rope_cos != nullptr && c->k_bias == nullptr) return FP8KV_ERR_INVALID_ARG;
  // 16-byte vector copies read the cache: every base pointer must be aligned
  const uintptr_t align = (uintptr_t)c->k | (uintptr_t)c->v | (uintptr_t)c->k_scale |
                          (uintptr_t)c->v_scale | (uintptr_t)c->page_table | (uintptr_t)c->k_bias |
                          (uintptr_t)c->rope_cos | (uintptr_t)c->rope_sin;
  if (align & 15) return FP8KV_ERR_INVALID_ARG;
  std::memset(view, 0, sizeof(*view));
  if (c->layout == FP8KV_LAYOUT_CONTIGUOUS) {
    if (c->max_tokens < 0) return FP8KV_ERR_INVALID_ARG;
    if (c->max_tokens % 16 != 0) return FP8KV_ERR_UNSUPPORTED;
  } else {
    if (c->page_table == nullptr || c->num_pages <= 0 || c->max_pages_per_seq <= 0)
      return FP8KV_ERR_INVALID_ARG;
    if (!is_pow2(c->page_size) || c->page_size < 16 || c->page_size > 64) return FP8KV_ERR_UNSUPPORTED;
    view->page_size = c->page_size;
    int sh = 0;
    while ((1 << sh) < c->page_size) ++sh;
    view->page_shift = sh;
    view->num_pages = c->num_pages;
    view->max_pages_per_seq = c->max_pages_per_seq;
    view->page_table = c->page_table;
    view->paged = 1;
  }
  // cache rows are addressed with 32-bit signed row coordinates
  const int64_t rows = c->layout == FP8KV_LAYOUT_CONTIGUOUS
                           ? (int64_t)c->batch * c->kv_heads * c->max_tokens
                           : (int64_t)c->num_pages * c->kv_heads * c->page_size;
  if (rows > INT32_MAX) return FP8KV_ERR_UNSUPPORTED;
  if (c->rope_cos != nullptr) {               // every position the cache can hold has a table row
    const int64_t cap = c->layout == FP8KV_LAYOUT_PAGED ? (int64_t)c->max_pages_per_seq * c->page_size
                                                       : (int64_t)c->max_tokens;
    if (c->rope_positions < cap) return FP8KV_ERR_INVALID_ARG;
  }
  view->k = static_cast<const uint8_t*>(c->k);
  view->v = static_cast<const uint8_t*>(c->v);
  view->k_scale = c->k_scale;
  view->v_scale = c->v_scale;
  view->k_bias = c->k_bias;
  view->rope_cos = c->rope_cos;
  view->rope_sin = c->rope_sin;
  view->batch = c->batch;
  view->kv_heads = c->kv_heads;
  view->head_dim = c->head_dim;
  view->max_tokens = c->layout == FP8KV_LAYOUT_CONTIGUOUS ? c->max_tokens : 0;
  return FP8KV_OK;
}

static int capacity_of(const fp8kv_cache* c) {
  return c->layout == FP8KV_LAYOUT_PAGED ? c->max_pages_per_seq * c->page_size : c->max_tokens;
}

// Split plan: split boundaries are multiples of the kernel's tile anchored
// at token 0.  Automatic: enough CTAs for about `ctas_per_sm` per SM over the
// (sequence, KV head) units, each split at least kMinSplitTiles tiles.
constexpr int kMinSplitTiles = 2;
constexpr int kTcWaveChunk = 56;

struct SplitPlan { int splits, chunk_tiles, tile, kernel; };

// The kernel a decode call runs (FP8KV_KERNEL_CUDA_CORES or _TENSOR_CORES),
// or 0 if the requested kernel does not support the shape.
static int resolve_kernel(const fp8kv_cache* c, int q_heads, int requested) {
  const int G = q_heads / c->kv_heads;
  const bool mma_ok = c->head_dim == 128 && G >= 1 && G <= 8;
  // rotated-bias residual keys: the CUDA-core kernel only (it adds each
  // key's rotated bias to its score)
  if (c->rope_cos != nullptr)
    return requested == FP8KV_KERNEL_AUTO || requested == FP8KV_KERNEL_CUDA_CORES ? FP8KV_KERNEL_CUDA_CORES : 0;
  // MXFP8 keys: both kernels apply each 32-dim block's scale to its partial
  // dot product; the transform paths (f16 K tiles) are not built for them
  if (c->dtype == FP8KV_MXK8V8) {
    if (requested == FP8KV_KERNEL_CUDA_CORES) return FP8KV_KERNEL_CUDA_CORES;
    if (requested == FP8KV_KERNEL_TENSOR_CORES) return mma_ok ? FP8KV_KERNEL_TENSOR_CORES : 0;
    if (requested == FP8KV_KERNEL_AUTO) return mma_ok ? FP8KV_KERNEL_TENSOR_CORES : FP8KV_KERNEL_CUDA_CORES;
    return 0;
  }
  if (requested == FP8KV_KERNEL_TENSOR_CORES) return mma_ok ? FP8KV_KERNEL_TENSOR_CORES : 0;
  if (requested == FP8KV_KERNEL_TENSOR_CORES_K_F16 || requested == FP8KV_KERNEL_TENSOR_CORES_K_F16_PRODUCER)
    return mma_ok && c->dtype == FP8KV_K8V8 ? requested : 0;
  if (requested == FP8KV_KERNEL_CUDA_CORES) return FP8KV_KERNEL_CUDA_CORES;
  if (requested != FP8KV_KERNEL_AUTO) return 0;
  // measured on the B16 decode (G 1, 2, 4, 8) and the paged B64 decode
  // (G 4): the tensor-core kernel is 1.8-2.8x faster at every group size
  return mma_ok ? FP8KV_KERNEL_TENSOR_CORES : FP8KV_KERNEL_CUDA_CORES;
}

// KV heads per tensor-core CTA for this cache and kernel (1 elsewhere).
static int heads_per_cta(const fp8kv_cache* c, int q_heads, int kernel) {
  if (kernel != FP8KV_KERNEL_TENSOR_CORES) return 1;
  return decode_heads_per_cta(c->layout == FP8KV_LAYOUT_PAGED, c->kv_heads, q_heads / c->kv_heads, c->page_size);
}

static SplitPlan plan_splits(const fp8kv_cache* c, int requested, int kernel, int hpc) {
  const bool tc = kernel >= FP8KV_KERNEL_TENSOR_CORES;
  const int tile = tc ? 128 / hpc : kTileTokens;          // tokens per KV head in a tile
  const int max_tiles = (capacity_of(c) + tile - 1) / tile;
  if (max_tiles <= 0) return {1, 1, tile, kernel};
  int want = requested;
  if (want <= 0) {
    const long units = (long)c->batch * (c->kv_heads / hpc);
    // tensor cores: one CTA per SM, and no partial second wave; CUDA cores:
    // about four CTAs per SM
    const long target = (long)(tc ? 1 : 4) * sm_count();
    if (units <= 0) want = 1;
    else want = tc ? (int)(target / units) : (int)((target + units - 1) / units);
    // tensor cores with more units than SMs: several waves in any case;
    // chunks of about kTcWaveChunk tiles let the waves balance when the
    // sequences' lengths differ (measured on the paged batch-64 decode,
    // 64-token tiles up to 16K tokens: 5 splits against 4 or 6, 2-3% faster
    // than 6 for e4m3 keys, every dtype at or near its best)
    if (tc && units >= sm_count()) want = (max_tiles + kTcWaveChunk - 1) / kTcWaveChunk;
    const int cap_by_min = (max_tiles + kMinSplitTiles - 1) / kMinSplitTiles;
    if (want > cap_by_min) want = cap_by_min;
  }
  if (want < 1) want = 1;
  if (want > max_tiles) want = max_tiles;
  const int chunk = (max_tiles + want - 1) / want;
  const int splits = (max_tiles + chunk - 1) / chunk;
  return {splits, chunk, tile, kernel};
}

}  // namespace fp8kv

using namespace fp8kv;

static fp8kv_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FP8KV_OK;
  (void)cudaGetLastError();
  return FP8KV_ERR_CUDA;
}

extern "C" {

const char* fp8kv_status_string(fp8kv_status s) {
  switch (s) {
    case FP8KV_OK: return "ok";
    case FP8KV_ERR_INVALID_ARG: return "invalid argument";
    case FP8KV_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case FP8KV_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8KV_ERR_CUDA: return "CUDA runtime error";
    case FP8KV_ERR_TIMEOUT: return "bounded device wait ran out";
    case FP8KV_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

fp8kv_status fp8kv_quantize(const void* x, int64_t rows, int32_t head_dim, uint8_t* codes, float* scales,
                            fp8kv_stream_t stream) {
  if (rows < 0) return FP8KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FP8KV_ERR_UNSUPPORTED;
  if (rows > 0 && (x == nullptr || codes == nullptr || scales == nullptr)) return FP8KV_ERR_INVALID_ARG;
  return cuda_status(launch_quantize(x, rows, head_dim, codes, scales, (cudaStream_t)stream));
}

fp8kv_status fp8kv_quantize_mx(const void* x, int64_t rows, int32_t head_dim, uint8_t* codes, uint8_t* scales,
                               fp8kv_stream_t stream) {
  if (rows < 0) return FP8KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FP8KV_ERR_UNSUPPORTED;
  if (rows > 0 && (x == nullptr || codes == nullptr || scales == nullptr)) return FP8KV_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_mx(x, rows, head_dim, codes, scales, (cudaStream_t)stream));
}

fp8kv_status fp8kv_append(const fp8kv_cache* cache, const void* k_new, const void* v_new,
                          const int32_t* seq_idx, const int32_t* pos, int64_t n_tokens,
                          fp8kv_stream_t stream) {
  CacheView view;
  fp8kv_status st = check_cache(cache, &view);
  if (st != FP8KV_OK) return st;
  if (n_tokens < 0) return FP8KV_ERR_INVALID_ARG;
  if (n_tokens == 0) return FP8KV_OK;
  if (!k_new || !v_new || !seq_idx || !pos) return FP8KV_ERR_INVALID_ARG;
  unsigned int* err = device_error_ptr();
  if (!err) return FP8KV_ERR_CUDA;
  return cuda_status(launch_append(view, cache->dtype, k_new, v_new, seq_idx, pos, n_tokens, err,
                                   (cudaStream_t)stream));
}

int32_t fp8kv_decode_num_splits(const fp8kv_cache* cache, int32_t q_heads, int32_t num_splits,
                                int32_t kernel) {
  CacheView view;
  if (check_cache(cache, &view) != FP8KV_OK) return 0;
  if (q_heads <= 0 || q_heads % cache->kv_heads != 0 || num_splits < 0) return 0;
  const int k = resolve_kernel(cache, q_heads, kernel);
  if (k == 0) return 0;
  return plan_splits(cache, num_splits, k, heads_per_cta(cache, q_heads, k)).splits;
}

size_t fp8kv_decode_workspace_bytes(const fp8kv_cache* cache, int32_t q_heads, int32_t num_splits,
                                    int32_t kernel) {
  const int S = fp8kv_decode_num_splits(cache, q_heads, num_splits, kernel);
  if (S <= 0) return 0;
  const size_t rows = (size_t)cache->batch * q_heads * S;
  return rows * ((size_t)cache->head_dim + 2) * sizeof(float);
}

}  // extern "C"

namespace {

// Checks shared by the decode calls; fills the parameter block and the plan.
fp8kv_status prepare_decode(const void* q, const fp8kv_cache* cache, const int32_t* seq_lens,
                            int32_t q_heads, float sm_scale, int32_t num_splits, int32_t kernel,
                            const void* workspace, size_t workspace_bytes, bool need_q, DecodeParams* p,
                            int* resolved) {
  CacheView view;
  fp8kv_status st = check_cache(cache, &view);
  if (st != FP8KV_OK) return st;
  if (q_heads <= 0 || q_heads % cache->kv_heads != 0 || num_splits < 0) return FP8KV_ERR_INVALID_ARG;
  if (kernel < FP8KV_KERNEL_AUTO || kernel > FP8KV_KERNEL_TENSOR_CORES_K_F16_PRODUCER) return FP8KV_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return FP8KV_ERR_INVALID_ARG;
  const int G = q_heads / cache->kv_heads;
  if (G > 8) return FP8KV_ERR_UNSUPPORTED;
  const int k = resolve_kernel(cache, q_heads, kernel);
  if (k == 0) return FP8KV_ERR_UNSUPPORTED;
  if (need_q && cache->batch > 0 && (!q || !seq_lens)) return FP8KV_ERR_INVALID_ARG;
  const int hpc = heads_per_cta(cache, q_heads, k);
  const SplitPlan plan = plan_splits(cache, num_splits, k, hpc);
  const size_t need = fp8kv_decode_workspace_bytes(cache, q_heads, num_splits, kernel);
  if (cache->batch > 0 && (workspace == nullptr || workspace_bytes < need)) return FP8KV_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 15) != 0) return FP8KV_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)cache->batch * q_heads;
  p->c = view;
  p->q = static_cast<const __nv_bfloat16*>(q);
  p->seq_lens = seq_lens;
  p->part_o = static_cast<float*>(const_cast<void*>(workspace));
  p->part_m = p->part_o + rows * plan.splits * cache->head_dim;
  p->part_l = p->part_m + rows * plan.splits;
  p->err = nullptr;
  p->q_heads = q_heads;
  p->group = G;
  p->num_splits = plan.splits;
  p->chunk_tiles = plan.chunk_tiles;
  p->scale_log2 = sm_scale * kLog2e;
  p->k_new = nullptr;
  p->v_new = nullptr;
  p->counters = nullptr;
  p->out = nullptr;
  p->out_f32 = 0;
  p->fused = 0;
  p->cluster = 0;
  p->pdl = 0;
  p->k_f16 = k == FP8KV_KERNEL_TENSOR_CORES_K_F16 ? 1 : k == FP8KV_KERNEL_TENSOR_CORES_K_F16_PRODUCER ? 2 : 0;
  p->hpc = hpc;
  p->hpc_shift = hpc == 8 ? 3 : hpc == 4 ? 2 : hpc == 2 ? 1 : 0;
  *resolved = k >= FP8KV_KERNEL_TENSOR_CORES ? FP8KV_KERNEL_TENSOR_CORES : k;
  return FP8KV_OK;
}

}  // namespace

extern "C" {

fp8kv_status fp8kv_decode_split(const void* q, const fp8kv_cache* cache, const int32_t* seq_lens,
                                int32_t q_heads, float sm_scale, int32_t num_splits, int32_t kernel,
                                void* workspace, size_t workspace_bytes, fp8kv_stream_t stream) {
  DecodeParams p;
  int k = 0;
  fp8kv_status st = prepare_decode(q, cache, seq_lens, q_heads, sm_scale, num_splits, kernel, workspace,
                                   workspace_bytes, true, &p, &k);
  if (st != FP8KV_OK || cache->batch == 0) return st;
  p.err = device_error_ptr();
  if (!p.err) return FP8KV_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(k == FP8KV_KERNEL_TENSOR_CORES ? launch_decode_mma(p, cache->dtype, cache->batch, s)
                                                    : launch_decode_fma(p, cache->dtype, cache->batch, s));
}

fp8kv_status fp8kv_decode_merge(const fp8kv_cache* cache, int32_t q_heads, int32_t num_splits,
                                int32_t kernel, const void* workspace, size_t workspace_bytes, void* out,
                                int32_t out_dtype, fp8kv_stream_t stream) {
  if (out_dtype != FP8KV_OUT_BF16 && out_dtype != FP8KV_OUT_F32) return FP8KV_ERR_INVALID_ARG;
  DecodeParams p;
  int k = 0;
  fp8kv_status st = prepare_decode(nullptr, cache, nullptr, q_heads, 1.0f, num_splits, kernel, workspace,
                                   workspace_bytes, false, &p, &k);
  if (st != FP8KV_OK || cache->batch == 0) return st;
  if (!out) return FP8KV_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)cache->batch * q_heads;
  return cuda_status(launch_decode_merge(p.part_o, p.part_m, p.part_l, p.num_splits, rows,
                                         cache->head_dim, out, out_dtype == FP8KV_OUT_F32,
                                         (cudaStream_t)stream));
}

fp8kv_status fp8kv_decode_attention(const void* q, const fp8kv_cache* cache, const int32_t* seq_lens,
                                    int32_t q_heads, float sm_scale, int32_t num_splits, int32_t kernel,
                                    void* workspace, size_t workspace_bytes, void* out, int32_t out_dtype,
                                    fp8kv_stream_t stream) {
  if (out_dtype != FP8KV_OUT_BF16 && out_dtype != FP8KV_OUT_F32) return FP8KV_ERR_INVALID_ARG;
  if (cache != nullptr && cache->batch > 0 && out == nullptr) return FP8KV_ERR_INVALID_ARG;
  fp8kv_status st = fp8kv_decode_split(q, cache, seq_lens, q_heads, sm_scale, num_splits, kernel,
                                       workspace, workspace_bytes, stream);
  if (st != FP8KV_OK) return st;
  return fp8kv_decode_merge(cache, q_heads, num_splits, kernel, workspace, workspace_bytes, out,
                            out_dtype, stream);
}

size_t fp8kv_decode_step_workspace_bytes(const fp8kv_cache* cache, int32_t q_heads, int32_t num_splits,
                                         int32_t kernel) {
  const size_t part = fp8kv_decode_workspace_bytes(cache, q_heads, num_splits, kernel);
  if (part == 0) return 0;
  const size_t ctr = ((size_t)cache->batch * cache->kv_heads * sizeof(int) + 15) & ~(size_t)15;
  return ((part + 15) & ~(size_t)15) + ctr;
}

fp8kv_status fp8kv_decode_step(const void* q, const void* k_new, const void* v_new, const fp8kv_cache* cache,
                               const int32_t* seq_lens, int32_t q_heads, float sm_scale, int32_t num_splits,
                               int32_t kernel, void* workspace, size_t workspace_bytes, void* out,
                               int32_t out_dtype, uint32_t flags, fp8kv_stream_t stream) {
  if (out_dtype != FP8KV_OUT_BF16 && out_dtype != FP8KV_OUT_F32) return FP8KV_ERR_INVALID_ARG;
  if (flags & ~FP8KV_STEP_EARLY_CACHE_READ) return FP8KV_ERR_INVALID_ARG;
  DecodeParams p;
  int k = 0;
  fp8kv_status st = prepare_decode(q, cache, seq_lens, q_heads, sm_scale, num_splits, kernel, workspace,
                                   workspace_bytes, true, &p, &k);
  if (st != FP8KV_OK || cache->batch == 0) return st;
  if (!out || !k_new || !v_new) return FP8KV_ERR_INVALID_ARG;
  const size_t need = fp8kv_decode_step_workspace_bytes(cache, q_heads, num_splits, kernel);
  if (workspace_bytes < need) return FP8KV_ERR_WORKSPACE;
  p.err = device_error_ptr();
  if (!p.err) return FP8KV_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (k == FP8KV_KERNEL_TENSOR_CORES) {
    const size_t part = fp8kv_decode_workspace_bytes(cache, q_heads, num_splits, kernel);
    p.k_new = static_cast<const __nv_bfloat16*>(k_new);
    p.v_new = static_cast<const __nv_bfloat16*>(v_new);
    p.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + ((part + 15) & ~(size_t)15));
    p.out = out;
    p.out_f32 = out_dtype == FP8KV_OUT_F32;
    p.fused = 1;
    p.pdl = (flags & FP8KV_STEP_EARLY_CACHE_READ) ? 1 : 0;
    return cuda_status(launch_decode_mma(p, cache->dtype, cache->batch, s));
  }
  cudaError_t e = launch_append_step(p.c, cache->dtype, k_new, v_new, seq_lens, p.err, s);
  if (e == cudaSuccess) e = launch_decode_fma(p, cache->dtype, cache->batch, s);
  if (e == cudaSuccess)
    e = launch_decode_merge(p.part_o, p.part_m, p.part_l, p.num_splits, (int64_t)cache->batch * q_heads,
                            cache->head_dim, out, out_dtype == FP8KV_OUT_F32, s);
  return cuda_status(e);
}

fp8kv_status fp8kv_prefill_attention(const void* q, const fp8kv_cache* cache, const int32_t* q_pos0,
                                     int32_t n_q, int32_t q_heads, float sm_scale, int32_t kernel,
                                     void* out, int32_t out_dtype, fp8kv_stream_t stream) {
  CacheView view;
  fp8kv_status st = check_cache(cache, &view);
  if (st != FP8KV_OK) return st;
  if (n_q < 0 || q_heads <= 0 || q_heads % cache->kv_heads != 0) return FP8KV_ERR_INVALID_ARG;
  if (out_dtype != FP8KV_OUT_BF16 && out_dtype != FP8KV_OUT_F32) return FP8KV_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return FP8KV_ERR_INVALID_ARG;
  if (q_heads / cache->kv_heads > 16) return FP8KV_ERR_UNSUPPORTED;
  if (kernel < FP8KV_KERNEL_AUTO || kernel > FP8KV_KERNEL_TENSOR_CORES) return FP8KV_ERR_INVALID_ARG;
  const bool tc_built = cache->dtype == FP8KV_K8V8 && cache->head_dim == 128 && cache->rope_cos == nullptr;
  if (kernel == FP8KV_KERNEL_TENSOR_CORES && !tc_built) return FP8KV_ERR_UNSUPPORTED;
  const bool use_tc = kernel == FP8KV_KERNEL_TENSOR_CORES || (kernel == FP8KV_KERNEL_AUTO && tc_built);
  if (cache->batch == 0 || n_q == 0) return FP8KV_OK;
  if (!q || !q_pos0 || !out) return FP8KV_ERR_INVALID_ARG;
  if (n_q > capacity_of(cache)) return FP8KV_ERR_INVALID_ARG;
  unsigned int* err = device_error_ptr();
  if (!err) return FP8KV_ERR_CUDA;
  PrefillParams p;
  p.c = view;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.q_pos0 = q_pos0;
  p.out = out;
  p.err = err;
  p.n_q = n_q;
  p.q_heads = q_heads;
  p.group = q_heads / cache->kv_heads;
  p.out_f32 = out_dtype == FP8KV_OUT_F32;
  p.scale_log2 = sm_scale * kLog2e;
  if (use_tc) return cuda_status(launch_prefill_tc(p, cache->batch, (cudaStream_t)stream));
  return cuda_status(launch_prefill_fma(p, cache->dtype, cache->batch, (cudaStream_t)stream));
}

fp8kv_status fp8kv_get_device_error(uint32_t* bits, int32_t clear) {
  if (bits == nullptr) return FP8KV_ERR_INVALID_ARG;
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
  }
  if (e != cudaSuccess) return cuda_status(e);
  *bits = v;
  if (v & FP8KV_DEVERR_TIMEOUT) return FP8KV_ERR_TIMEOUT;
  return v ? FP8KV_ERR_DEVICE_CHECK : FP8KV_OK;
}

}  // extern "C"
