// decode_static.cu -- decode attention for callers that cannot allocate
// device memory.
//
// fp8kv_decode_attention needs a workspace for the fp32 partials of the
// flash-decoding split, which the caller normally allocates.  Some callers
// cannot: a runtime that hands all device memory to its own pool and forbids
// cudaMalloc on its serving path (cudaMalloc may synchronise the device and
// fails while a stream is being captured), or a host that owns no allocator
// at all, such as a plugin given only the tensors it reads and writes.  This
// entry point keeps the partials in a fixed array compiled into the library
// instead, so it calls no cudaMalloc, cudaFree or allocating library routine.
//
// The array lives in every GPU that loads the library, until the process
// exits.  Its address is a device address; the host-side name of a
// __device__ array is only a stand-in, so the address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and passed to the
// kernels.
#include <atomic>

#include "params.cuh"

namespace fp8kv {

constexpr size_t kStaticScratchBytes = 16u << 20;   // 16 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device, looked up on the
// first use per device and kept (atomically: host threads making their first
// call at once each look it up and store the same value).  Returns nullptr
// if the lookup fails.
static void* static_scratch_ptr(cudaError_t* err) {
  constexpr int kMaxDev = 64;
  static std::atomic<void*> ptrs[kMaxDev];
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) { (void)cudaGetLastError(); return nullptr; }
  if (dev < 0 || dev >= kMaxDev) { *err = cudaErrorInvalidDevice; return nullptr; }
  void* p = ptrs[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*err != cudaSuccess) { (void)cudaGetLastError(); return nullptr; }
    ptrs[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace fp8kv

extern "C" {

fp8kv_status fp8kv_decode_attention_static(const void* q, const fp8kv_cache* cache,
                                           const int32_t* seq_lens, int32_t q_heads, float sm_scale,
                                           int32_t num_splits, void* out, int32_t out_dtype,
                                           fp8kv_stream_t stream) {
  // Invalid arguments give need == 0 here and are reported by the checks of
  // fp8kv_decode_attention below.
  size_t need = fp8kv_decode_workspace_bytes(cache, q_heads, num_splits, FP8KV_KERNEL_AUTO);
  if (need > fp8kv::kStaticScratchBytes && num_splits == 0) {
    // The automatic split count needs more partials than the array holds:
    // take the largest count that fits (fewer splits, fewer partials).
    for (int s = fp8kv_decode_num_splits(cache, q_heads, 0, FP8KV_KERNEL_AUTO) - 1; s >= 1; --s) {
      need = fp8kv_decode_workspace_bytes(cache, q_heads, s, FP8KV_KERNEL_AUTO);
      if (need <= fp8kv::kStaticScratchBytes) {
        num_splits = s;
        break;
      }
    }
  }
  if (need > fp8kv::kStaticScratchBytes) return FP8KV_ERR_WORKSPACE;
  cudaError_t e = cudaSuccess;
  void* scratch = fp8kv::static_scratch_ptr(&e);
  if (scratch == nullptr) return FP8KV_ERR_CUDA;
  // Every split writes all of its partials (empty splits write m = -inf,
  // l = 0, O = 0) before the merge reads them, so nothing needs clearing.
  return fp8kv_decode_attention(q, cache, seq_lens, q_heads, sm_scale, num_splits, FP8KV_KERNEL_AUTO, scratch,
                                fp8kv::kStaticScratchBytes, out, out_dtype, stream);
}

size_t fp8kv_decode_static_scratch_bytes(void) { return fp8kv::kStaticScratchBytes; }

}  // extern "C"
