// decode_mma.cu -- flash-decoding split kernel on the tcgen05 tensor cores,
// warp-specialised and software-pipelined.
//
// Same computation and partials as decode_fma.cu ("FP8 KV cache (fp8_kv,
// opt-in)", bullets "Math" and "Speed"), for head_dim 128 and up to 8 query
// heads per KV head.  A CTA owns one (split, KV head, sequence) and walks its
// 128-token tiles:
//
//   S^T[128 tokens x 16] = K_tile[128 x 128] . Q^T         tcgen05.mma -> TMEM
//   per token (one thread each): s = S * k_scale * sm_scale (log2 units),
//     per warp (32 tokens): anchor U = ceil(max of s + log2 v_scale),
//     p = 2^(s - U), P' = bf16_rn(p * v_scale)               (CUDA cores)
//   O^T[128 dims x 16]   = V_tile^T[128 x 128] . P'^T        tcgen05.mma -> TMEM
//   per dim (one thread each): O = O * 2^(m-m') + sum over the four warps w
//     of 2^(U_w-m') * O_tile,w  (each warp's tokens are one PV k-step)
//
// The e4m3 cache tiles are MMA operands as they land in shared memory
// (kind::f8f6f4; K tile K-major, V tile MN-major): no per-element K or V
// preparation runs on the CUDA cores ("FP8 KV attention: hardware paths and
// tile preparation", sections "Measure the K8/V8 break-even" and "NVIDIA
// Blackwell": the prepare-K and prepare-V stages of the tile interval vanish).
// The other operand of each MMA must then be e4m3 too, so the bf16 query row
// and the bf16-rounded P' row are each written as the sum of two e4m3 numbers
// (hi = e4m3(x), lo = e4m3(x - hi)); hi and lo occupy the 16 columns of the N
// dimension that 8 query heads leave free, and are summed after the MMA.  The
// query row is first scaled by a power of two; P' needs no per-row scaling:
// its anchor puts the warp's largest P' in (1/2, 1], so 2^8 P' lies in
// (128, 256].  For every component within 2^-11 of that maximum the pair is
// exact; smaller components carry an absolute error below 2^-19 of it -- and
// since the anchor follows p * v_scale, not p, a token whose V scale is far
// below its neighbours' still sets the scale when its weight dominates.
// A bf16 K (K16/V8) or V (K16/V16) side uses kind::f16 with exact operands.
//
// Anchors are integer-valued and depend on the tile alone: split and unsplit
// runs round P' alike, and every fold factor is an exact power of two.
//
// Warp roles ("FP8 KV attention: hardware paths and tile preparation",
// section "Operating model": producer and consumer warps interleave the
// stages across adjacent tiles):
//   warp 0     TMA producer: 128-byte-swizzled tensor loads of the K and V
//              tiles straight into the UMMA operand layout, a ring of NST
//              stages (full/empty mbarriers).  Native-QK kernels with an
//              even ring: warps 0 and 11 issue alternate tiles.  Contiguous
//              cache: scale rows by 1-D bulk copy.  Paged cache: one page per
//              lane (its K and V boxes and, by cp.async, its scale rows),
//              page ids four tiles ahead by cp.async.
//   warp 1     TMEM owner and QK issuer (one thread).
//   warp 10    PV issuer (one thread).  Issuing a few tcgen05.mma costs the
//              issuing thread a fraction of a microsecond; one thread issuing
//              both QK and PV set the tile interval, two run side by side.
//   warps 2-9  two softmax warpgroups on alternate tiles: the O fold of the
//              group's tile before last, then the softmax of the next tile
//              (thread = TMEM lane = token for S, = head dim for O); merged
//              at the end like two splits.  The four warps of a group share
//              no barrier inside the loop: each publishes its tile anchors
//              in shared memory before its P-ready arrival, and the O fold
//              reads them after that phase completed.  Warp maxima come from
//              redux.sync, so every lane holds all heads' anchors.
// S, O (TMEM) and P (shared memory) are double-buffered per group, so the
// QKs and PVs of neighbouring tiles overlap the softmax.  A QK chains its
// k-steps into one accumulator (it runs far enough ahead of the softmax that
// their latency is hidden; MXFP8 keys keep one accumulator per 32-dim block
// for the block scales).  A PV keeps one accumulator per k-step, the token
// slice of one softmax warp with its own anchor, combined by the O fold.
// Every wait is bounded; a wait that runs out
// raises FP8KV_DEVERR_TIMEOUT, the CTA writes an empty partial and leaves.
// V rows past the sequence end are zeroed before PV (0 * NaN would poison
// the product).
//
// The fused decode step (append + split + merge in one launch) merges the
// splits of a (sequence, KV head) in one of two ways.  With 2..8 splits whose
// clusters all fit on the GPU at once, the splits run as one thread-block
// cluster and exchange their partials through distributed shared memory
// (cluster_exchange: each rank merges a slice of the head dimension).
// Otherwise every split writes its partial to global memory and the last
// one to finish, found with an atomic counter, merges them all.
#include <cuda_fp16.h>

#include "params.cuh"
#include "tc_common.cuh"

namespace fp8kv {

constexpr int kMmaTile = 128;
// Split partials the global merge stages in the (idle) ring at a time.
constexpr int kMergeChunk = 44;
// warp 0 TMA producer, warp 1 QK issuer and TMEM owner, warps 2-9 softmax,
// warp 10 PV issuer; where TcCfg::NPW is 2 a twelfth warp is a second
// producer (warps 0 and 11 issue the even and the odd tiles).
constexpr int kTcThreads = 352;

// XK: where K is prepared (an ablation).  XK_NATIVE: QK is the native e4m3
// MMA on the query's e4m3 hi/lo pair.  On the transform path each landed
// e4m3 K tile is converted to f16 in shared memory and QK runs as kind::f16
// on an f16 query, the conversion done by the producer warp (XK_PRODUCER)
// or by the softmax warpgroup that owns the tile (XK_CONSUMER).  The K scale
// stays in score space on every path.
enum : int { XK_NATIVE = 0, XK_PRODUCER = 1, XK_CONSUMER = 2 };

template <int KE, int VE, int XK = XK_NATIVE>
struct TcCfg {
  static constexpr int D = 128;
  static constexpr bool K8 = KE != ELEM_BF16;                       // K as 8-bit codes (e4m3 or MXFP8)
  static constexpr bool KMX = KE == ELEM_MX;                         // per-32-dim block scales on K
  static constexpr bool QHL = K8 && XK == XK_NATIVE;                 // query as an e4m3 hi/lo pair
  static constexpr int KB = K8 ? 1 : 2, VB = VE == ELEM_E4M3 ? 1 : 2;
  static constexpr int K_TILE = kMmaTile * D * KB;
  static constexpr int V_TILE = kMmaTile * D * VB;
  // K tile, V tile, then the K and V scale rows of an 8-bit side
  static constexpr int STAGE = ((K_TILE + V_TILE + (K8 || VE == ELEM_E4M3 ? 2 * kMmaTile * 4 : 0)) + 1023) / 1024 * 1024;
  static constexpr int NST = XK != XK_NATIVE ? 4 : (K8 && VE == ELEM_E4M3) ? 6 : (K8 == (VE == ELEM_E4M3) ? 3 : 4);
  // Producer warps.  One warp's chain of dependent instructions per tile
  // (on a paged cache: a page lookup, addresses and a copy per page and
  // side) fell behind the softmax's pace, so the native-QK kernels run two
  // that issue alternate tiles.  Tile i's ring slot is i % NST with NST
  // even, so each producer's tiles keep to their own slots.
  static constexpr int NPW = XK == XK_NATIVE && NST % 2 == 0 ? 2 : 1;
  static constexpr int THREADS = kTcThreads + (NPW - 1) * 32;
  static constexpr int KCV = XK != XK_NATIVE ? 2 * kMmaTile * D * 2 : 0;   // two converted f16 K tiles
  static constexpr int QOP = QHL ? 16 * 128 : 2 * 16 * 128;
  static constexpr int POP = VE == ELEM_E4M3 ? 16 * 128 : 2 * 16 * 128;   // [128 tokens][16 or 32 B]
  static constexpr int XO = 8 * 128 * 4;    // group 1's O handed to group 0
  static constexpr int MISC = 8192;         // barriers, small tables, cluster receive buffers, page-id ring
  static constexpr int BYTES = NST * STAGE + KCV + QOP + 4 * POP + XO + MISC + 1024;
  static_assert(BYTES <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
  static_assert(NST * STAGE + KCV >= (8 * kMergeChunk * D + 2 * 8 * kMergeChunk) * 4,
                "ring too small to stage a chunk of partials for the merge");
  static_assert(XK == XK_NATIVE || KE == ELEM_E4M3, "the K transform converts e4m3 codes");
};

struct DecodeTmaParams {
  CUtensorMap tmk;
  CUtensorMap tmv;
  DecodeParams p;
};

// Per-warpgroup barrier set (S, P and O double buffers).
struct WgBars {
  uint64_t s_full[2], s_empty[2], p_full[2], o_full[2], o_empty[2];
};

#ifdef FP8KV_TRACE
// Per-tile clock64 stamps of CTA (0, 0, 0), read by fp8kv_trace_read():
// slot 8*i + {0: producer issue, 1: QK issue, 2: PV issue, 3: softmax start,
// 4: P ready (first warp), 5: O folded, 6: P ready (last warp)}; 1010..1014:
// teardown steps; 1020/1021: kernel begin/end.
__device__ unsigned long long g_trace[1024];
// %globaltimer at entry and exit of every CTA (first 4096 CTAs).
__device__ unsigned long long g_cta_time[4096][8];   // start, end, published, last-flag seen, table, loads, stored
#define TRACE(slot)                                                          \
  do {                                                                       \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (slot) < 1024) \
      g_trace[(slot)] = clock64();                                           \
  } while (0)
#define TRACE_MAX(slot)                                                      \
  do {                                                                       \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (slot) < 1024) \
      atomicMax(&g_trace[(slot)], (unsigned long long)clock64());            \
  } while (0)
// fine stamps inside one tile's softmax (tile 8, thread 0 of its group)
#define TRACE_SUB(tile, k)                                                   \
  do {                                                                       \
    if ((tile) == 8 && (t) == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) \
      g_trace[900 + (k)] = clock64();                                        \
  } while (0)
#else
#define TRACE_SUB(tile, k) \
  do {                     \
  } while (0)
#define TRACE(slot) \
  do {              \
  } while (0)
#define TRACE_MAX(slot) \
  do {                  \
  } while (0)
#endif

// Programmatic dependent launch: wait for the kernel issued before this one
// on the stream (its writes visible), and let the next one be scheduled.
// Both are no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Merge of the fused step when the splits of one (sequence, KV head) run as
// one thread-block cluster (split = cluster rank, S <= 8).  Rank r owns the
// four-dim groups [g4_lo(r), g4_lo(r+1)) of the head dimension, all 8 heads.
// Each rank stages its split's O as [head][dim] in shared memory and pushes
// every (head, four-dim group) as one 16-byte st.async into the owning
// rank's receive buffer ([sender][head][group]); thread t < S pushes the
// split's (m, l) to rank t.  Every st.async counts down the receiver's
// mbarrier, whose transaction count was armed at setup with all the bytes
// it will get.  Each rank then waits for its slice and merges it from local
// shared memory, one (head, four-dim group) output per thread: one one-way
// trip over the cluster network, no cluster-wide barrier.  Called by the 128
// merging threads (warps 2-5, thread t = dim t of the partial) of every CTA;
// `stage` is [8][128] floats of this CTA's shared memory that is idle now.
__device__ __forceinline__ int g4_lo(int r, int S) { return (32 * r) / S; }
// Owner rank of four-dim group q: the largest r with g4_lo(r, S) <= q, i.e.
// floor(32 r / S) <= q  <=>  r < (q + 1) S / 32.
__device__ __forceinline__ int g4_owner(int q, int S) { return ((q + 1) * S - 1) >> 5; }

__device__ __forceinline__ void cluster_exchange(const DecodeParams& p, float* rx_ml, float* rx_o, uint64_t* rx_bar,
                                              const int* slice, float* stage, const float (&Og)[8],
                                              const float (&Mg)[8], const float (&Lg)[8], int64_t hq0, int QH,
                                              int t, volatile int* abort) {
  constexpr int D = 128;
  const int S = p.num_splits;
  const int k = (int)cluster_rank();
  if (t == 0) TRACE(1002);
#pragma unroll
  for (int g = 0; g < 8; ++g) stage[g * D + t] = Og[g];
  group_sync(0);
  // (the caller passed the cluster barrier after setup: every rank's receive
  // barrier is initialised and armed)
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int c = t + 128 * j, g = c >> 5, q = c & 31;   // head g, four-dim group q
    const int r = g4_owner(q, S);
    const int lo = slice[r], n4 = slice[r + 1] - lo;
    const float4 v = *reinterpret_cast<const float4*>(stage + g * D + 4 * q);
    st_async_v4(mapa_u32(umma::smem_u32(rx_o + 4 * ((k * 8 + g) * n4 + (q - lo))), (uint32_t)r), v,
                mapa_u32(umma::smem_u32(rx_bar), (uint32_t)r));
  }
  if (t < S) {
    const uint32_t bar_t = mapa_u32(umma::smem_u32(rx_bar), (uint32_t)t);
    const uint32_t dml = mapa_u32(umma::smem_u32(rx_ml + k * 16), (uint32_t)t);
    st_async_v4(dml, make_float4(Mg[0], Mg[1], Mg[2], Mg[3]), bar_t);
    st_async_v4(dml + 16, make_float4(Mg[4], Mg[5], Mg[6], Mg[7]), bar_t);
    st_async_v4(dml + 32, make_float4(Lg[0], Lg[1], Lg[2], Lg[3]), bar_t);
    st_async_v4(dml + 48, make_float4(Lg[4], Lg[5], Lg[6], Lg[7]), bar_t);
  }
  if (t == 0) TRACE(1003);
  const bool ok = wait_cluster(rx_bar, 0, abort);
  if (t == 0) TRACE(1004);
  if (!ok) {
    if (t == 0) raise_error(p.err, FP8KV_DEVERR_TIMEOUT);
    return;
  }
  const int mlo = slice[k], m4 = slice[k + 1] - mlo;
  if (t < 8 * m4) {
    int g = 0;          // t / m4 without a division: m4 <= 16, t < 128
#pragma unroll
    for (int u = 1; u < 8; ++u) g += t >= u * m4;
    const int j = t - g * m4;
    // (S <= 8: unrolled, every load independent; anchors are integer-valued,
    // so the weights are exact powers of two)
    float mk[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mk[kk] = kk < S ? rx_ml[kk * 16 + g] : -INFINITY;
    float M = mk[0];
#pragma unroll
    for (int kk = 1; kk < 8; ++kk) M = fmaxf(M, mk[kk]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (kk < S) {
        const float w = pow2_diff(mk[kk] - M, 0);
        const float4 v = *reinterpret_cast<const float4*>(rx_o + 4 * ((kk * 8 + g) * m4 + j));
        L += w * rx_ml[kk * 16 + 8 + g];
        o.x += w * v.x; o.y += w * v.y; o.z += w * v.z; o.w += w * v.w;
      }
    }
    if (g < QH) {
      const float inv = L > 0.f ? __frcp_rn(L) : 0.f;
      const int64_t oi = (hq0 + g) * D + 4 * (mlo + j);
      const float r4[4] = {o.x * inv, o.y * inv, o.z * inv, o.w * inv};
      if ((reinterpret_cast<uintptr_t>(p.out) & 15) != 0) {   // caller's buffer not 16-byte aligned
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (p.out_f32) reinterpret_cast<float*>(p.out)[oi + e] = r4[e];
          else reinterpret_cast<__nv_bfloat16*>(p.out)[oi + e] = __float2bfloat16_rn(r4[e]);
        }
      } else if (p.out_f32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + oi) = make_float4(r4[0], r4[1], r4[2], r4[3]);
      } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(r4[0], r4[1]);
        const __nv_bfloat162 c = __floats2bfloat162_rn(r4[2], r4[3]);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + oi) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&c));
      }
    }
  }
  if (t == 0) TRACE(1005);
}

// Bytes a rank receives in the cluster merge: S senders x (8 heads x its
// four-dim groups x 16 bytes + 16 (m, l) floats).
__device__ __forceinline__ uint32_t cluster_rx_bytes(int rank, int S) {
  return (uint32_t)(S * (128 * (g4_lo(rank + 1, S) - g4_lo(rank, S)) + 64));
}

// One e4m3 K tile (K-major, 128-byte swizzle: row r = token, 16-byte chunk
// c = dims 16c..16c+15 at chunk position c ^ (r & 7)) -> the f16 K operand:
// two 64-dim atoms of the same swizzle (atom a holds dims 64a..64a+63, one
// 128-byte row per token).  Every e4m3 value is exact in f16.  Called by the
// NT threads (32: one warp, 128: a warpgroup), idx = 0..NT-1: thread = (row,
// chunk), so each group of eight consecutive threads reads one whole 128-byte
// row.  Eight rows' loads are issued before any store (the compiler cannot
// move a load above a store to the same shared memory), so their latencies
// overlap.
template <int NT>
__device__ __forceinline__ void k_tile_to_f16(const uint8_t* src, uint8_t* dst, int idx) {
  constexpr int RP = NT / 8;                      // rows per pass
  const int c = idx & 7, a = c >> 2, c0 = 2 * (c & 3);
#pragma unroll 1
  for (int r0 = idx >> 3; r0 < kMmaTile; r0 += 8 * RP) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = r0 + RP * j;
      v[j] = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = r0 + RP * j;
      uint8_t* row = dst + a * (kMmaTile * 128) + r * 128;
      *reinterpret_cast<uint4*>(row + ((c0 ^ (r & 7)) << 4)) =
          make_uint4(e4m3x2_to_f16x2((uint16_t)v[j].x), e4m3x2_to_f16x2((uint16_t)(v[j].x >> 16)),
                     e4m3x2_to_f16x2((uint16_t)v[j].y), e4m3x2_to_f16x2((uint16_t)(v[j].y >> 16)));
      *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) =
          make_uint4(e4m3x2_to_f16x2((uint16_t)v[j].z), e4m3x2_to_f16x2((uint16_t)(v[j].z >> 16)),
                     e4m3x2_to_f16x2((uint16_t)v[j].w), e4m3x2_to_f16x2((uint16_t)(v[j].w >> 16)));
    }
  }
}

// PG: the instantiation for paged caches whose scale rows the softmax threads
// load themselves (the native-QK kernels); other paged launches use PG = false.
template <int KE, int VE, int XK, bool PG>
__global__ void __launch_bounds__(TcCfg<KE, VE, XK>::THREADS, 1)
    decode_split_tc(const __grid_constant__ DecodeTmaParams tp) {
  using C = TcCfg<KE, VE, XK>;
  constexpr int NPW = C::NPW;
  static_assert(NPW == 1 || C::NST % 2 == 0, "two producers need an even ring");
  constexpr int D = 128;
  const DecodeParams& p = tp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kcv = smem + C::NST * C::STAGE;                  // [2] f16 K tiles (transform path)
  uint8_t* qop = kcv + C::KCV;
  uint8_t* pop0 = qop + C::QOP;                            // [wg][buffer] P operands
  float* xo = reinterpret_cast<float*>(pop0 + 4 * C::POP);   // [8][128]
  uint8_t* misc = pop0 + 4 * C::POP + C::XO;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);     // [8]
  uint64_t* empty = full + 8;                              // [8]
  WgBars* wb = reinterpret_cast<WgBars*>(empty + 8);       // [2]
  uint64_t* appended = reinterpret_cast<uint64_t*>(wb + 2);   // new token written (fused step)
  uint64_t* rx_bar = appended + 1;                         // cluster merge: this rank's slice received
  uint32_t* tslot = reinterpret_cast<uint32_t*>(rx_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tslot + 2);
  uint64_t* kc_full = reinterpret_cast<uint64_t*>(misc + 320);   // [2] transform path: f16 K tile ready
  uint64_t* kc_empty = kc_full + 2;                              // [2] its QK completed
  float* qscale = reinterpret_cast<float*>(misc + 512);    // [8] query scale x softmax scale (log2 units)
  float* wscr = reinterpret_cast<float*>(misc + 6656);     // [softmax warp][40]: fold factors
  float* lred = reinterpret_cast<float*>(misc + 1120);     // [wg][4][8]
  float* xml = lred + 64;                                  // [16]: m and l of warpgroup 1
  int* slice_tab = reinterpret_cast<int*>(misc + 1472);    // [9] first four-dim group of each rank
  float* rx_ml = reinterpret_cast<float*>(misc + 1536);    // [sender][m 8 | l 8]
  float* rx_o = reinterpret_cast<float*>(misc + 2048);     // [sender][dim of this rank's slice][8 heads]
  float* anc0 = reinterpret_cast<float*>(misc + 544);      // [4 slots][4 warps][8 heads]: group 0's anchors
  int* pg_ring = reinterpret_cast<int*>(misc + 7936);      // [8 tiles][8 pages]: the producer's page ids

  const int split = blockIdx.x, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // KV heads hkv0 .. hkv0 + HPC - 1 and their QH = HPC G query heads; a tile
  // holds TT tokens of each (HPC > 1 only on a paged cache: rows ordered by
  // page, then head, then token within the page)
  const int HPC = p.hpc, hs = p.hpc_shift;
  const int hkv0 = blockIdx.y << hs;
  if (tid == 0) {                                 // the TMA unit fetches the maps while the CTA sets up
    tma::prefetch_map(&tp.tmk);
    tma::prefetch_map(&tp.tmv);
  }
  const CacheView& c = p.c;
  const int G = p.group, S = p.num_splits;
  const int QH = G << hs, TT = kMmaTile >> hs;
  const int64_t hq_row0 = (int64_t)b * p.q_heads + (int64_t)hkv0 * G;   // (sequence, first query head) row

  int T = p.seq_lens[b];
  const int cap = cache_capacity(c);
  if (T < 0 || T > cap) {
    if (tid == 0) raise_error(p.err, FP8KV_DEVERR_SEQ_TOO_LONG);
    T = 0;
  }
  const int tiles = (T + TT - 1) / TT;
  const int t_begin = split * p.chunk_tiles;
  const int t_end = min(t_begin + p.chunk_tiles, tiles);
  const int64_t part0 = hq_row0 * S + split;
  if (t_begin >= t_end) {
    if (p.pdl) grid_dep_wait();                   // writes below
    if (p.cluster) {
      // no tiles: an empty partial (m = -inf, l = 0) in the cluster merge
      if (tid == 0) {
        *abort_flag = 0;
        umma::mbar_init(rx_bar, 1);
        tma::arrive_expect_tx(rx_bar, cluster_rx_bytes((int)cluster_rank(), S));
        umma::mbar_fence_init();
        for (int r = 0; r <= S; ++r) slice_tab[r] = g4_lo(r, S);
      }
      __syncthreads();
      cluster_arrive_relaxed();
      if (tid >= 64 && tid < 192) {
        cluster_wait();
        float Og[8], Mg[8], Lg[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) { Og[g] = 0.f; Mg[g] = -INFINITY; Lg[g] = 0.f; }
        cluster_exchange(p, rx_ml, rx_o, rx_bar, slice_tab, xo, Og, Mg, Lg, hq_row0, QH, tid - 64, abort_flag);
      }
      return;
    }
    if (p.fused) {
      // No partial: splits without work take no part in the merge.  A
      // sequence with no tokens gets its zero output from split 0.
      if (tiles == 0 && split == 0)
        for (int i = tid; i < QH * D; i += blockDim.x) {
          const int64_t o = (hq_row0 + i / D) * D + (i % D);
          if (p.out_f32) reinterpret_cast<float*>(p.out)[o] = 0.f;
          else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
        }
      return;
    }
    for (int i = tid; i < QH * D; i += blockDim.x)
      p.part_o[(part0 + (int64_t)(i / D) * S) * D + (i % D)] = 0.f;
    if (tid < QH) {
      p.part_m[part0 + (int64_t)tid * S] = -INFINITY;
      p.part_l[part0 + (int64_t)tid * S] = 0.f;
    }
    return;
  }
  const int n_tiles = t_end - t_begin;
  // Fused step: the CTA whose range holds position T-1 writes the new token
  // before its producer loads that tile.
  const int tile_new = T > 0 ? (T - 1) / TT : -1;
  const bool appender = p.fused && p.k_new != nullptr && tile_new >= t_begin && tile_new < t_end;
  const int i_new = appender ? tile_new - t_begin : n_tiles;
  if (tid == 0) TRACE(1020);
#ifdef FP8KV_TRACE
  const int cta_lin = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  if (tid == 0 && cta_lin < 4096) g_cta_time[cta_lin][0] = umma::globaltimer_ns();
#endif

  // ---------------------------------------------------------------- setup
  // Overlapped before the one CTA-wide barrier: thread 0 initialises the
  // barriers and issues the first tiles' loads, warp 1 allocates TMEM, warps
  // 2-5 write the query operand.
  const int64_t cont_row0 = ((int64_t)b * c.kv_heads + hkv0) * c.max_tokens;
  // Issue the TMA copies of tile i into its stage.  Called by all 32 lanes
  // of warp 0.  Contiguous layout: lane 0 issues the tile's few copies.
  // Paged layout: lane j issues page j's copies (K and V boxes of the HPC
  // heads' rows, which are contiguous in the pool, and their scale rows),
  // lane 0 arms the stage's barrier (the transaction count is signed, so a
  // copy may land first).  Each lane's page ids come kPageAhead tiles ahead
  // by a 4-byte cp.async into a ring in shared memory (one commit group per
  // tile), so no register ever holds a pending table load: page ids kept in
  // registers and shifted down one register per tile made every tile wait
  // for the previous tile's lookup (a register move waits for its load),
  // and that latency set the paged decode's pace.
  constexpr int kPageAhead = 4;
  // Paged layout: the producer's per-tile address arithmetic reduced to
  // shifts and adds on per-CTA constants (pages are a power of two long and
  // divide the tile's token stretch TT): the producer issues one tile after
  // another, so its chain of dependent instructions per tile sets the pace.
  const int pshift = c.page_shift;
  const int ppt = TT >> pshift;                      // pages of a full tile
  const int PR = 1 << (pshift + hs);                 // rows of one page (HPC heads x P tokens)
  const uint32_t per_page = PR * 128 * (C::KB + C::VB);
  const int pool_rpp = c.kv_heads << pshift;         // pool rows per page, all KV heads
  const int row_h0 = hkv0 << pshift;                 // row of head hkv0 within its page
  const int* pt_cta = c.paged ? c.page_table + (int64_t)b * c.max_pages_per_seq + ((t_begin * TT) >> pshift) : nullptr;
  auto pages_of = [&](int i) -> int {                // pages holding tile i's tokens
    const int rem = T - (t_begin + i) * TT;
    return rem >= TT ? ppt : (rem + (1 << pshift) - 1) >> pshift;
  };
  // (each producer fetches, and waits for, its own tiles' ids: cp.async
  // groups are per thread)
  auto fetch_page = [&](int i) {   // tile i's page ids -> ring slot i & 7; one group
    if (i < n_tiles && lane < pages_of(i))
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(umma::smem_u32(pg_ring + (i & 7) * 8 + lane)),
                   "l"(pt_cta + i * ppt + lane)
                   : "memory");
    cp_async_commit();
  };
  auto produce = [&](int i) {
    const int s = i % C::NST;
    uint8_t* st = smem + s * C::STAGE;
    float* kss = reinterpret_cast<float*>(st + C::K_TILE + C::V_TILE);
    float* vss = kss + kMmaTile;
    if (!c.paged) {
      if (lane == 0) {
        const int t0 = (t_begin + i) * TT;
        const int valid = min(TT, T - t0);
        const int nsc = min(kMmaTile, (valid + 15) & ~15);
        const uint32_t bytes = C::K_TILE + C::V_TILE + (C::K8 ? nsc * 4 : 0) +
                               (VE == ELEM_E4M3 ? nsc * 4 : 0);
        tma::arrive_expect_tx(&full[s], bytes);
        const int row = (int)(cont_row0 + t0);
        tma::load_2d(st, &tp.tmk, 0, row, &full[s]);
        if (!C::K8) tma::load_2d(st + kMmaTile * 128, &tp.tmk, 64, row, &full[s]);
        tma::load_2d(st + C::K_TILE, &tp.tmv, 0, row, &full[s]);
        if (VE != ELEM_E4M3) tma::load_2d(st + C::K_TILE + kMmaTile * 128, &tp.tmv, 64, row, &full[s]);
        if (C::K8) tma::load_1d(kss, c.k_scale + cont_row0 + t0, nsc * 4, &full[s]);
        if (VE == ELEM_E4M3) tma::load_1d(vss, c.v_scale + cont_row0 + t0, nsc * 4, &full[s]);
      }
    } else {
      // The K and V boxes come by TMA (counted in the transaction bytes).
      // The scale rows come by cp.async, each lane's page rows, and each
      // lane's cp.async.mbarrier.arrive adds one pending arrival to the stage
      // barrier that completes when the lane's copies land (before lane 0's
      // arrival, the barrier's only expected one, so the phase cannot
      // complete without the scale rows).  The next page ids are fetched
      // after that arrival, so the stage does not wait for them as well.
      const int np = pages_of(i);
      cp_async_wait<kPageAhead / NPW - 1>();       // tile i's group has landed
      int page = lane < np ? pg_ring[(i & 7) * 8 + lane] : 0;
      if (lane < np && (unsigned)page >= (unsigned)c.num_pages) {
        raise_error(p.err, FP8KV_DEVERR_BAD_PAGE);
        page = 0;      // read a valid page; the result is flagged as wrong
      }
      const int row = page * pool_rpp + row_h0;
      if (lane < np && (C::K8 || VE == ELEM_E4M3)) {
        for (int q = 0; q < PR / 4; ++q) {
          if (C::K8) cp_async16(kss + lane * PR + 4 * q, c.k_scale + row + 4 * q);
          if (VE == ELEM_E4M3) cp_async16(vss + lane * PR + 4 * q, c.v_scale + row + 4 * q);
        }
        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];\n" ::"r"(umma::smem_u32(&full[s]))
                     : "memory");
      }
      fetch_page(i + kPageAhead);
      __syncwarp();
      if (lane == 0) tma::arrive_expect_tx(&full[s], per_page * np);
      if (lane < np) {
        const int off = lane * PR * 128;
        tma::load_2d(st + off, &tp.tmk, 0, row, &full[s]);
        if (!C::K8) tma::load_2d(st + kMmaTile * 128 + off, &tp.tmk, 64, row, &full[s]);
        tma::load_2d(st + C::K_TILE + off, &tp.tmv, 0, row, &full[s]);
        if (VE != ELEM_E4M3)
          tma::load_2d(st + C::K_TILE + kMmaTile * 128 + off, &tp.tmv, 64, row, &full[s]);
      }
    }
    if (lane == 0) TRACE(8 * i + 0);
  };
  const int n_first = min(min(n_tiles, C::NST), i_new);
  if (tid == 0) {
    // the ring's barriers first, so the first loads go out as early as possible
    for (int i = 0; i < C::NST; ++i) {
      umma::mbar_init(&full[i], 1);
      umma::mbar_init(&empty[i], 1 + 4);     // PV commit + the four warps of the owning group
    }
    *abort_flag = 0;
    *last_flag = 0;
    umma::mbar_fence_init();
  }
  if (warp == 0 || (NPW == 2 && warp == 11)) {
    const int pw = warp == 0 ? 0 : 1;
    if (NPW == 2) {
      // the second producer starts once the ring's barriers exist
      if (warp == 0) {
        __syncwarp();
        asm volatile("bar.arrive 4, 64;\n" ::: "memory");
      } else {
        asm volatile("bar.sync 4, 64;\n" ::: "memory");
      }
    } else {
      __syncwarp();
    }
    if (c.paged)
      for (int k = pw; k < kPageAhead; k += NPW) fetch_page(k);
    for (int i = pw; i < n_first; i += NPW) produce(i);
  }
  if (tid == 0) {
    for (int w = 0; w < 2; ++w)
      for (int i = 0; i < 2; ++i) {
        umma::mbar_init(&wb[w].s_full[i], 1);
        umma::mbar_init(&wb[w].s_empty[i], 4);
        umma::mbar_init(&wb[w].p_full[i], 4);
        umma::mbar_init(&wb[w].o_full[i], 1);
        umma::mbar_init(&wb[w].o_empty[i], 4);
      }
    umma::mbar_init(appended, 1);
    if (XK != XK_NATIVE)
      for (int i = 0; i < 2; ++i) {
        umma::mbar_init(&kc_full[i], XK == XK_CONSUMER ? 4 : 1);   // the owning group's four warps
        umma::mbar_init(&kc_empty[i], 1);
      }
    if (p.cluster) {
      umma::mbar_init(rx_bar, 1);
      tma::arrive_expect_tx(rx_bar, cluster_rx_bytes(split, S));
      for (int r = 0; r <= S; ++r) slice_tab[r] = g4_lo(r, S);
    }
    umma::mbar_fence_init();
  }
  if (warp == 1) {
    umma::tmem_alloc(tslot, 512);
    umma::tmem_relinquish();
  }
  if (p.pdl) {
    // the first cache tiles are in flight; q, k_new and v_new, and every
    // write, wait for the previous kernel on the stream
    grid_dep_wait();
    if (tid == 0) grid_dep_launch();
  }
  if (warp >= 2 && warp < 6) {   // zero the operand buffers (group 0 only, then its own barrier)
    for (int i = tid - 64; i < (C::QOP + 4 * C::POP) / 16; i += 128)
      reinterpret_cast<uint4*>(qop)[i] = make_uint4(0, 0, 0, 0);
    group_sync(0);
  }
  if (warp >= 2 && warp < 6) {   // query rows -> B operand of QK (e4m3 hi/lo pairs, or bf16)
    for (int g = warp - 2; g < 8; g += 4) {
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (g < QH) {
        const __nv_bfloat16* qr = p.q + (hq_row0 + g) * D + lane * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = __bfloat162float(qr[e]);
      }
      if constexpr (XK != XK_NATIVE) {
        // f16 query for the f16 QK: each head's row scaled by a power of two
        // so its largest magnitude lies in [2^14, 2^15) (bf16 -> f16 exact)
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        amax = warp_max_redux(amax);
        int e = 0;
        (void)frexpf(amax, &e);
        const int ex = e - 15;
        if (lane == 0) qscale[g] = ldexpf(1.0f, ex) * p.scale_log2;
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
          *reinterpret_cast<__half*>(qop + sw128_off(g, (lane * 4 + e4) * 2, 16)) = __float2half_rn(ldexpf(x[e4], -ex));
      } else if constexpr (C::K8) {
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        amax = warp_max_redux(amax);
        const int ex = e4m3_row_exp(amax);
        if (lane == 0) qscale[g] = ldexpf(1.0f, ex) * p.scale_log2;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float xs = ldexpf(x[e], -ex);
          const uint8_t hi = e4m3_rn(xs);
          const uint8_t lo = e4m3_rn(xs - e4m3_val(hi));
          qop[sw128_off(g, lane * 4 + e, 16)] = hi;
          qop[sw128_off(g + 8, lane * 4 + e, 16)] = lo;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<__nv_bfloat16*>(qop + sw128_off(g, (lane * 4 + e) * 2, 16)) = __float2bfloat16_rn(x[e]);
        if (lane == 0) qscale[g] = p.scale_log2;
      }
    }
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  if (p.cluster) {
    // every rank's receive barrier initialised: the merging warps wait for
    // that here, while the first tiles are still in flight
    cluster_arrive_relaxed();
    if (warp >= 2 && warp < 6) cluster_wait();
  }

  if (appender && warp == 0) {
    // Quantise and write the new token's K and V rows (the arithmetic of
    // fp8kv_append: amax/448 with IEEE division, RNE saturating encode),
    // then publish them to the TMA loads of the producer.  The producer warp
    // does it: its first loads are in flight and no ring slot frees up for
    // a few microseconds, while the softmax warps start on the first tiles.
    for (int hh = 0; hh < HPC; ++hh) {          // the CTA's KV heads
      const int hk = hkv0 + hh;
      const int tpos = T - 1;
      const int64_t row = cache_row(c, b, hk, tpos, lane == 0 ? p.err : nullptr);
      if (row >= 0) {
#pragma unroll
        for (int side = 0; side < 2; ++side) {
          const __nv_bfloat16* src = (side == 0 ? p.k_new : p.v_new) + ((int64_t)b * c.kv_heads + hk) * D + lane * 4;
          const uint2 raw = *reinterpret_cast<const uint2*>(src);
          const bool fp8 = side == 0 ? C::K8 : VE == ELEM_E4M3;
          uint8_t* dst = const_cast<uint8_t*>(side == 0 ? c.k : c.v);
          if (!fp8) {
            *reinterpret_cast<uint2*>(dst + (row * D + lane * 4) * 2) = raw;
          } else {
            float x[4], t2[2];
            bf16x2_to_f32(raw.x, t2); x[0] = t2[0]; x[1] = t2[1];
            bf16x2_to_f32(raw.y, t2); x[2] = t2[0]; x[3] = t2[1];
            if (side == 0 && c.k_bias != nullptr) {      // pre-bias residual key
#pragma unroll
              for (int e = 0; e < 4; ++e) x[e] -= c.k_bias[hk * D + lane * 4 + e];
            }
            float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
            if (C::KMX && side == 0) {
              // MXFP8 key: the arithmetic of fp8kv_quantize_mx, block = 8 lanes
#pragma unroll
              for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
              const int E = mx_block_exp(amax);
              const float inv = pow2_exact(-E);
              *reinterpret_cast<uint32_t*>(dst + row * D + lane * 4) =
                  e4m3x2_rn(x[0] * inv, x[1] * inv) | (e4m3x2_rn(x[2] * inv, x[3] * inv) << 16);
              if ((lane & 7) == 0)
                reinterpret_cast<uint8_t*>(const_cast<float*>(c.k_scale) + row)[lane >> 3] = (uint8_t)(E + 127);
            } else {
              amax = warp_max(amax);
              const float scale = __fdiv_rn(amax, 448.0f);
              uint32_t packed = 0;
              if (amax != 0.f)
                packed = e4m3x2_rn(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)) |
                         (e4m3x2_rn(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)) << 16);
              *reinterpret_cast<uint32_t*>(dst + row * D + lane * 4) = packed;
              if (lane == 0) const_cast<float*>(side == 0 ? c.k_scale : c.v_scale)[row] = scale;
            }
          }
        }
      }
    }
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
    __syncwarp();
    if (lane == 0) umma::mbar_arrive(appended);
  }

  if (warp == 0 || (NPW == 2 && warp == 11)) {
    // ----------------------------------------------------------- producers
    // (the whole warp: lane 0 waits for each stage and the others follow it;
    // producer pw issues tiles pw, pw + NPW, ...)
    const int pw = warp == 0 ? 0 : 1;
    int issued = n_first;
    if constexpr (XK != XK_PRODUCER) {
      int i = pw;
      for (; i < n_tiles; i += NPW) {
        if (i < n_first) continue;
        const int s = i % C::NST, u = i / C::NST;
        bool ok = true;
        if (lane == 0) {
          if (i < 100) TRACE(500 + i);
          ok = u == 0 || wait_fast(&empty[s], (u - 1) & 1, abort_flag);
          ok = ok && (i != i_new || wait_or_abort(appended, 0, abort_flag));
          if (i < 100) TRACE(400 + i);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        produce(i);
      }
      issued = max(i, n_first);   // this producer's tiles below it are issued
    } else {
      // Transform path: issue tiles as stages free up and convert each
      // landed K tile into the free f16 buffer, whichever is ready first.
      int nc = 0;
      long long t_prog = clock64();
      uint32_t idle = 0;
      while (nc < n_tiles) {
        bool prog = false;
        if (issued < n_tiles) {
          const int i = issued, s = i % C::NST, u = i / C::NST;
          int ready = 0;
          if (lane == 0)
            ready = (u == 0 || umma::mbar_test(&empty[s], (u - 1) & 1)) &&
                    (i != i_new || umma::mbar_test(appended, 0));
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            produce(i);
            ++issued;
            prog = true;
          }
        }
        if (nc < issued) {
          const int s = nc % C::NST, u = nc / C::NST, kb = nc & 1, ku = nc >> 1;
          int ready = 0;
          if (lane == 0)
            ready = umma::mbar_test(&full[s], u & 1) && (ku == 0 || umma::mbar_test(&kc_empty[kb], (ku - 1) & 1));
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            k_tile_to_f16<32>(smem + s * C::STAGE, kcv + kb * (kMmaTile * D * 2), lane);
            umma::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              umma::mbar_arrive(&kc_full[kb]);
              TRACE(8 * nc + 7);
            }
            ++nc;
            prog = true;
          }
        }
        if (prog) {
          idle = 0;
          continue;
        }
        __nanosleep(20);
        if ((++idle & 63) == 0) {
          if (idle == 64) t_prog = clock64();
          if (*abort_flag) break;
          if (clock64() - t_prog > kWaitLimitCycles) {
            *abort_flag = 1;
            break;
          }
        }
      }
    }
    // Before leaving, let every copy this warp issued land (only an aborted
    // run has copies that nobody waited for).
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    if (lane == 0) {
      for (int i = max(0, issued - C::NST); i < issued; ++i)
        if (i % NPW == pw) (void)umma::mbar_wait(&full[i % C::NST], (i / C::NST) & 1, 100000000ull);
      TRACE(1013);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- QK issuer
    // One thread issues every QK; the PV issuer is warp 10.  An issue of a
    // few tcgen05.mma takes a fraction of a microsecond of the issuing
    // thread, so QK and PV each get their own thread and run side by side.
    if (lane == 0) {
      constexpr uint32_t ID_QK = C::K8
          ? umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_K, umma::MAJOR_K, 128, 16)
          : umma::idesc(umma::FMT_BF16, umma::FMT_BF16, umma::MAJOR_K, umma::MAJOR_K, 128, 16);
      const uint32_t qa = umma::smem_u32(qop);
      for (int nq = 0; nq < n_tiles; ++nq) {
        const int s = nq % C::NST, u = nq / C::NST, w = nq & 1, li = nq >> 1, bb = li & 1, ub = li >> 1;
        bool ok = XK != XK_NATIVE ? wait_fast(&kc_full[nq & 1], (nq >> 1) & 1, abort_flag)
                                  : wait_fast(&full[s], u & 1, abort_flag);
        ok = ok && (ub == 0 || wait_fast(&wb[w].s_empty[bb], (ub - 1) & 1, abort_flag));
        if (!ok) break;
        umma::fence_after_sync();
        const uint32_t ka =
            umma::smem_u32(XK != XK_NATIVE ? kcv + (nq & 1) * (kMmaTile * D * 2) : smem + s * C::STAGE);
        // One accumulator for the whole dot product (QK runs far enough
        // ahead of the softmax that the chained k-steps' latency is hidden,
        // and the softmax then reads 16 columns instead of summing four
        // accumulators).  MXFP8 keys: one accumulator per 32-dim block, each
        // scaled by its block's E8M0 byte in the softmax.
        const uint32_t d = tmem + 256 * w + 64 * bb;
        if constexpr (XK != XK_NATIVE) {
          constexpr uint32_t ID_F16 =
              umma::idesc(umma::FMT_F16, umma::FMT_F16, umma::MAJOR_K, umma::MAJOR_K, 128, 16);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma::mma_f16_ss(d,
                             umma::sdesc(ka + (k >> 2) * (kMmaTile * 128) + (k & 3) * 32, 16, 1024,
                                         umma::SWIZZLE_128B),
                             umma::sdesc(qa + (k >> 2) * (16 * 128) + (k & 3) * 32, 16, 1024, umma::SWIZZLE_128B),
                             ID_F16, k > 0);
        } else if constexpr (C::K8) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma::mma_f8_ss(C::KMX ? d + 16 * k : d, umma::sdesc(ka + k * 32, 16, 1024, umma::SWIZZLE_128B),
                            umma::sdesc(qa + k * 32, 16, 1024, umma::SWIZZLE_128B), ID_QK, !C::KMX && k > 0);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma::mma_f16_ss(d,
                             umma::sdesc(ka + (k >> 2) * (kMmaTile * 128) + (k & 3) * 32, 16, 1024,
                                         umma::SWIZZLE_128B),
                             umma::sdesc(qa + (k >> 2) * (16 * 128) + (k & 3) * 32, 16, 1024, umma::SWIZZLE_128B),
                             ID_QK, k > 0);
        }
        umma::mma_commit(&wb[w].s_full[bb]);
        if (XK == XK_PRODUCER) umma::mma_commit(&kc_empty[nq & 1]);
        TRACE(8 * nq + 1);
      }
    }
  } else if (warp == 10) {
    // -------------------------------------------------------- PV issuer
    if (lane == 0) {
      constexpr uint32_t ID_PV = VE == ELEM_E4M3
          ? umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_MN, umma::MAJOR_MN, 128, 16)
          : umma::idesc(umma::FMT_BF16, umma::FMT_BF16, umma::MAJOR_MN, umma::MAJOR_MN, 128, 16);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % C::NST, w = j & 1, lj = j >> 1, bb = lj & 1, ub = lj >> 1;
        // P ready implies S ready, which implies the tile landed; the
        // transform path's QK did not read the stage itself, so wait for it
        bool ok = wait_fast(&wb[w].p_full[bb], ub & 1, abort_flag);
        ok = ok && (ub == 0 || wait_fast(&wb[w].o_empty[bb], (ub - 1) & 1, abort_flag));
        ok = ok && (XK == XK_NATIVE || wait_fast(&full[s], (j / C::NST) & 1, abort_flag));
        if (!ok) break;
        if (XK == XK_NATIVE) TRACE(8 * j + 7);
        umma::fence_after_sync();
        const uint32_t va = umma::smem_u32(smem + s * C::STAGE + C::K_TILE);
        const uint32_t pa = umma::smem_u32(pop0 + (2 * w + bb) * C::POP);
        const uint32_t d = tmem + 256 * w + 128 + 64 * bb;
        if constexpr (VE == ELEM_E4M3) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma::mma_f8_ss(d + 16 * k, umma::sdesc(va + k * 4 * 1024, 1024, 1024, umma::SWIZZLE_128B),
                            umma::sdesc(pa + k * 512, 128, 128, umma::SWIZZLE_NONE), ID_PV, 0);
        } else {
          // 16-token k-steps: accumulator j takes k-steps 2j and 2j+1, the
          // 32 tokens of softmax warp j (each warp's tokens carry their own
          // anchor); the second of each pair is issued after the four firsts
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int k = 2 * (kk & 3) + (kk >> 2);
            umma::mma_f16_ss(d + 16 * (k >> 1), umma::sdesc(va + k * 2 * 1024, kMmaTile * 128, 1024, umma::SWIZZLE_128B),
                             umma::sdesc(pa + k * 512, 256, 128, umma::SWIZZLE_NONE), ID_PV, kk >= 4);
          }
        }
        umma::mma_commit(&wb[w].o_full[bb]);
        umma::mma_commit(&empty[s]);
        TRACE(8 * j + 2);
      }
      TRACE(1014);
    }
  } else {
    // ------------------------------------- softmax and O update (2 groups)
    const int wg = (warp - 2) >> 2;                 // warpgroup: even or odd tiles
    const int t = 32 * (warp & 3) + lane;           // TMEM lane of this thread
    const int sw = warp & 3;                        // lane quarter
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t s_col = 256 * wg, o_col = 256 * wg + 128;
    WgBars& B = wb[wg];
    // row t of every tile: token tok of the tile's stretch of KV head hkv0 +
    // hh, whose query heads are the score columns in cmask
    int tok = t, hh = 0;
    uint32_t cmask = 0xFFu;
    if (HPC > 1) {
      const int ps = c.page_shift;
      hh = (t >> ps) & (HPC - 1);
      tok = ((t >> (ps + hs)) << ps) | (t & (c.page_size - 1));
      cmask = ((1u << G) - 1u) << (hh * G);
    }
    // Anchors.  The tokens one warp holds of a tile are referenced to the
    // integer-valued U = ceil(max of s + log2(v_scale)) over them (log2
    // units; for a bf16 V side, of s): p = 2^(s - U), and P' = bf16(p *
    // v_scale) then lies in [0, 1] with its largest entry above 1/2, so the
    // e4m3 P' column is exact to bf16 precision after the constant scaling
    // by 2^8, whatever the spread of the V scales.  (log2(v_scale) is
    // clamped at -100 so that p stays finite for a token whose V row is zero
    // or nearly so.)  U depends on the tile alone, so split and unsplit runs
    // round P' alike, and every fold factor is an exact power of two.
    //   m_w: this warp's running anchor per head (reference of its threads'
    //        partial sums l_thr);
    //   m_o: the group's running anchor over its four warps (reference of
    //        O).
    // Every lane keeps m_w for all eight heads (the warp maxima come from
    // redux.sync); m_o of head g is tracked by the lanes that fold it.
    // No barrier across the group's warps inside the loop: each warp's P'
    // columns feed their own PV k-step accumulator (tokens 32w..32w+31),
    // and the O fold weights accumulator w with warp w's published anchor.
    constexpr int kPShift = VE == ELEM_E4M3 ? 8 : 0;  // e4m3 P' columns hold 2^8 P'
    float l_thr[8], o_run[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) { l_thr[g] = 0.f; o_run[g] = 0.f; }
    float m_w[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) m_w[g] = -INFINITY;
    float m_ol = -INFINITY;                          // m_o of head lane & 7
    float* wsc = wscr + (warp - 2) * 40;
    // published anchors, [4 slots][4 warps][8 heads]; group 1's table shares
    // the buffer that hands its O to group 0 once its loop is over
    float* ancA = wg == 0 ? anc0 : xo;
    bool failed = false;
    const int nl = (n_tiles - wg + 1) / 2;          // tiles of this group
    // iteration li: the O fold of the group's tile li-2 (its PV finished
    // long ago), then the softmax of tile li
    for (int li = 0; li < nl + 2; ++li) {
      if (li >= 2) {
        const int lj = li - 2, bb = lj & 1, ub = lj >> 1;
        TRACE_SUB(2 * li + wg, 0);
        bool ok = wait_fast(&B.o_full[bb], ub & 1, abort_flag);
        // p_full of tile lj completed before its PV: the four warps'
        // anchors of that tile were written before their arrivals
        ok = ok && wait_fast(&B.p_full[bb], ub & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        TRACE_SUB(2 * li + wg, 1);
        umma::fence_after_sync();
        uint32_t r[4][16];
#pragma unroll
        for (int k = 0; k < 4; ++k) umma::tmem_ld16_nowait(tmem + o_col + 64 * bb + 16 * k + lane_off, r[k]);
        // fold factors, one (warp k, head g) per lane: the head's new anchor
        // is the maximum of the four warps' anchors and its running m_o;
        // accumulator k gets 2^(U_k - kPShift - m_o'), the old O 2^(m_o - m_o')
        {
          const float Aq = ancA[(lj & 3) * 32 + lane];
          float am = fmaxf(Aq, __shfl_xor_sync(0xffffffffu, Aq, 8));
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 16));
          const float mn = fmaxf(m_ol, am);
          wsc[lane] = pow2_diff(Aq - mn, -kPShift);
          if (lane < 8) wsc[32 + lane] = pow2_diff(m_ol - mn, 0);
          m_ol = mn;
        }
        __syncwarp();
        float fk[4][8], fa[8];
        {
          const float4* w4 = reinterpret_cast<const float4*>(wsc);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 x = w4[2 * k], y = w4[2 * k + 1];
            fk[k][0] = x.x; fk[k][1] = x.y; fk[k][2] = x.z; fk[k][3] = x.w;
            fk[k][4] = y.x; fk[k][5] = y.y; fk[k][6] = y.z; fk[k][7] = y.w;
          }
          const float4 x = w4[8], y = w4[9];
          fa[0] = x.x; fa[1] = x.y; fa[2] = x.z; fa[3] = x.w;
          fa[4] = y.x; fa[5] = y.y; fa[6] = y.z; fa[7] = y.w;
        }
        TRACE_SUB(2 * li + wg, 2);
        umma::tmem_wait_ld();
        TRACE_SUB(2 * li + wg, 3);
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) umma::mbar_arrive(&B.o_empty[bb]);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          float o = o_run[g] * fa[g];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float ot = VE == ELEM_E4M3 ? __uint_as_float(r[k][g]) + __uint_as_float(r[k][g + 8])
                                             : __uint_as_float(r[k][g]);
            o = fmaf(ot, fk[k][g], o);
          }
          o_run[g] = o;
        }
        TRACE_SUB(2 * li + wg, 4);
        if (t == 0) TRACE(8 * (2 * lj + wg) + 5);
      }
      if (li < nl) {
        const int i = 2 * li + wg;
        const int s = i % C::NST, u = i / C::NST, bb = li & 1, ub = li >> 1;
        if constexpr (XK == XK_CONSUMER) {
          // convert this tile's K into the group's own f16 buffer (free: the
          // group consumed the S of its previous tile, so that QK is done)
          const bool landed = wait_or_abort(&full[s], u & 1, abort_flag);
          if (!__all_sync(0xffffffffu, landed)) { failed = true; break; }
          k_tile_to_f16<128>(smem + s * C::STAGE, kcv + wg * (kMmaTile * D * 2), t);
          umma::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) umma::mbar_arrive(&kc_full[wg]);
        }
        // hand-offs on the critical path: poll without a suspend-time hint
        bool ok = wait_fast(&B.s_full[bb], ub & 1, abort_flag);
        ok = ok && wait_fast(&full[s], u & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
        if (t == 0) TRACE(8 * i + 3);
        TRACE_SUB(i, 5);
        umma::fence_after_sync();
        uint8_t* st = smem + s * C::STAGE;
        const float* kss = reinterpret_cast<const float*>(st + C::K_TILE + C::V_TILE);
        const float* vss = kss + kMmaTile;
        const int t0 = (t_begin + i) * TT;
        const int valid = min(TT, T - t0);
        const bool tok_ok = tok < valid;
        const float kf = KE == ELEM_E4M3 ? kss[t] : 1.f;   // (MXFP8: below)
        const float vsc = VE == ELEM_E4M3 ? (tok_ok ? vss[t] : 0.f) : 1.f;
        float sc[16];
        {
          constexpr int NACC = C::KMX ? 4 : 1;
          uint32_t r[NACC][16];
#pragma unroll
          for (int k = 0; k < NACC; ++k) umma::tmem_ld16_nowait(tmem + s_col + 64 * bb + 16 * k + lane_off, r[k]);
          umma::tmem_wait_ld();
          TRACE_SUB(i, 6);
          if constexpr (C::KMX) {
            // MXFP8 keys: accumulator k holds dims 32k..32k+31 of the dot
            // product, so the key's E8M0 block scale k applies to it here
            // (the block-scaled product, summed over the four blocks)
            const uint32_t e8 = reinterpret_cast<const uint32_t*>(st + C::K_TILE + C::V_TILE)[t];
            float w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = pow2_exact((int)((e8 >> (8 * k)) & 0xFF) - 127);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              sc[j] = (w[0] * __uint_as_float(r[0][j]) + w[1] * __uint_as_float(r[1][j])) +
                      (w[2] * __uint_as_float(r[2][j]) + w[3] * __uint_as_float(r[3][j]));
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) sc[j] = __uint_as_float(r[0][j]);
          }
        }
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) umma::mbar_arrive(&B.s_empty[bb]);
        // scores (log2 units) and s + log2(v_scale)
        const float lvs = VE == ELEM_E4M3 ? fmaxf(lg2_approx(vsc), -100.f) : 0.f;
        float qsc[8];                      // (re-read each tile: registers are scarce)
        {
          const float4 x = reinterpret_cast<const float4*>(qscale)[0], y = reinterpret_cast<const float4*>(qscale)[1];
          qsc[0] = x.x; qsc[1] = x.y; qsc[2] = x.z; qsc[3] = x.w;
          qsc[4] = y.x; qsc[5] = y.y; qsc[6] = y.z; qsc[7] = y.w;
        }
        float sg[8], uu[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float raw = C::QHL ? (sc[g] + sc[g + 8]) : sc[g];
          sg[g] = tok_ok && ((cmask >> g) & 1u) ? raw * (qsc[g] * kf) : -INFINITY;
          uu[g] = sg[g] + lvs;
        }
        TRACE_SUB(i, 7);
        // per head: the anchor U (the warp maximum, in every lane), and the
        // factors that bring the threads' l sums to the new running anchor
        float Uh[8], f1[8], f2[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) Uh[g] = ceilf(warp_max_f32(uu[g]));
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          // one of the two factors is 1, the other 2^-|U - m_w| (both 0 or
          // 1 when neither anchor exists yet: l is still 0 then)
          const bool up = Uh[g] > m_w[g];
          const float e = pow2_diff(-fabsf(Uh[g] - m_w[g]), 0);
          f1[g] = up ? e : 1.f;
          f2[g] = up ? 1.f : e;
          m_w[g] = fmaxf(m_w[g], Uh[g]);
        }
        TRACE_SUB(i, 8);
        if (!tok_ok) {      // V rows past the sequence end: zero them for PV
          uint4* vrow = reinterpret_cast<uint4*>(st + C::K_TILE);
#pragma unroll
          for (int blk = 0; blk < C::VB; ++blk)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              vrow[(blk * kMmaTile * 128 + t * 128 + ch * 16) / 16] = make_uint4(0, 0, 0, 0);
        }
        // p (unrounded, into l) and P' = bf16(p * v_scale), head pairs
        uint32_t pw[4];
#pragma unroll
        for (int g = 0; g < 8; g += 2) {
          // (a warp without valid tokens has U = -inf and all scores -inf)
          const float p0 = ex2(sg[g] - (Uh[g] > -INFINITY ? Uh[g] : 0.f));
          const float p1 = ex2(sg[g + 1] - (Uh[g + 1] > -INFINITY ? Uh[g + 1] : 0.f));
          l_thr[g] = l_thr[g] * f1[g] + p0 * f2[g];
          l_thr[g + 1] = l_thr[g + 1] * f1[g + 1] + p1 * f2[g + 1];
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0 * vsc, p1 * vsc);
          pw[g >> 1] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        TRACE_SUB(i, 9);
        uint8_t* pop = pop0 + (2 * wg + bb) * C::POP;
        // P^T operand, MN-major without swizzle: token t's 16 bytes (e4m3:
        // hi of heads 0..7 then lo; bf16: heads 0..7) in one 16-byte store.
        if constexpr (VE == ELEM_E4M3) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // 2^8 P' (exact), written as hi + lo e4m3
            const float x0 = __uint_as_float(pw[j] << 16) * 256.f;
            const float x1 = __uint_as_float(pw[j] & 0xFFFF0000u) * 256.f;
            const uint32_t hi = e4m3x2_rn(x0, x1);
            float hv[4];
            e4m3x4_to_f32_scaled(hi, hv);
            hw[j] = hi;
            lw[j] = e4m3x2_rn(x0 - hv[0] * kTwoPow120, x1 - hv[1] * kTwoPow120);
          }
          *reinterpret_cast<uint4*>(pop + t * 16) =
              make_uint4(hw[0] | (hw[1] << 16), hw[2] | (hw[3] << 16), lw[0] | (lw[1] << 16), lw[2] | (lw[3] << 16));
        } else {
          *reinterpret_cast<uint4*>(pop + (t >> 3) * 256 + (t & 7) * 16) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
        TRACE_SUB(i, 10);
        umma::fence_proxy_async_smem();
        __syncwarp();
        TRACE_SUB(i, 11);
        if (lane == 0) {
          float4* da = reinterpret_cast<float4*>(ancA + ((li & 3) * 4 + sw) * 8);
          da[0] = make_float4(Uh[0], Uh[1], Uh[2], Uh[3]);
          da[1] = make_float4(Uh[4], Uh[5], Uh[6], Uh[7]);
          umma::mbar_arrive(&B.p_full[bb]);
          umma::mbar_arrive(&empty[s]);
        }
        if (t == 0) TRACE(8 * i + 4);
        TRACE_SUB(i, 12);
        if (lane == 0) TRACE_MAX(8 * i + 6);
      }
    }
    // a warp that gave up left the loop early; the group's result is empty
    // if any of its warps did
    failed = group_any(wg, failed);
    float m_run[8];                                 // m_o of every head
#pragma unroll
    for (int g = 0; g < 8; ++g) m_run[g] = __shfl_sync(0xffffffffu, m_ol, g);
    if (failed) {
      if (t == 0) raise_error(p.err, FP8KV_DEVERR_TIMEOUT);
#pragma unroll
      for (int g = 0; g < 8; ++g) { m_run[g] = -INFINITY; o_run[g] = 0.f; }
    }
    // l: each warp's sums (reference m_w) by a transposed butterfly, one
    // head per four lanes, brought to the group's m_o: lred[wg][warp][head]
    {
      // (each thread's sums brought to m_o first: an exact power-of-two
      // scaling, so the order does not change the result)
#pragma unroll
      for (int g = 0; g < 8; ++g) l_thr[g] *= pow2_diff(m_w[g] - m_run[g], 0);
      const float ws = warp_sum_transposed<8>(l_thr, lane);           // head (lane >> 2) & 7
      if ((lane & 3) == 0) lred[(wg * 4 + sw) * 8 + (lane >> 2)] = failed ? 0.f : ws;
    }
    if (t == 0 && wg == 0) TRACE(1010);
    // The two groups' running states are merged like two splits: group 1
    // hands its m and O to group 0 through shared memory (both groups' l
    // sums are in lred).
    if (t == 0 && wg == 1) TRACE(1000);
    if (wg == 1) {
#pragma unroll
      for (int g = 0; g < 8; ++g) xo[g * D + t] = o_run[g];
      if (t < 8) xml[t] = failed ? -INFINITY : m_ol;      // lane t holds m_o of head t
    }
    asm volatile("bar.sync 3, 256;\n" ::: "memory");
    if (t == 0 && wg == 0) TRACE(1011);
    if (wg == 0) {
      float Mg[8], Lg[8], Og[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float m1 = xml[g];
        const float M = fmaxf(m_run[g], m1);
        const float f0 = pow2_diff(m_run[g] - M, 0), f1 = pow2_diff(m1 - M, 0);
        const float l0 = (lred[g] + lred[8 + g]) + (lred[16 + g] + lred[24 + g]);
        const float l1 = (lred[32 + g] + lred[40 + g]) + (lred[48 + g] + lred[56 + g]);
        Og[g] = o_run[g] * f0 + xo[g * D + t] * f1;
        Mg[g] = M;
        Lg[g] = l0 * f0 + l1 * f1;
      }
      if (t == 0) TRACE(1001);
      // splits with work (only the global-memory merge needs it)
      const int n_busy = p.cluster ? 0 : (tiles + p.chunk_tiles - 1) / p.chunk_tiles;
      if (p.cluster) {
        cluster_exchange(p, rx_ml, rx_o, rx_bar, slice_tab, xo, Og, Mg, Lg, hq_row0, QH, t, abort_flag);
      } else if (p.fused && n_busy == 1) {
        // the only split of this sequence: normalise and write the output
#pragma unroll
        for (int g = 0; g < 8; ++g)
          if (g < QH) {
            const float r = Lg[g] > 0.f ? Og[g] / Lg[g] : 0.f;
            const int64_t o = (hq_row0 + g) * D + t;
            if (p.out_f32) reinterpret_cast<float*>(p.out)[o] = r;
            else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(r);
          }
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          if (g < QH) p.part_o[(part0 + (int64_t)g * S) * D + t] = Og[g];
          if (t == g && g < QH) {
            p.part_m[part0 + (int64_t)g * S] = Mg[g];
            p.part_l[part0 + (int64_t)g * S] = Lg[g];
          }
        }
        if (p.fused) {
          // The last split of this (sequence, KV head) to finish merges all
          // of them: publish the partials, count the arrival, and let the
          // last arrival read every split's partials back (from L2).
          __threadfence();
          group_sync(0);
#ifdef FP8KV_TRACE
          if (t == 0 && cta_lin < 4096) g_cta_time[cta_lin][2] = umma::globaltimer_ns();
#endif
          if (t == 0) {
            int* ctr = p.counters + (int64_t)b * c.kv_heads + hkv0;
            const int old = atomicAdd(ctr, 1);
            const int last = old == n_busy - 1;
            if (last) *ctr = 0;                 // ready for the next call
            *last_flag = last;
          }
          group_sync(0);
#ifdef FP8KV_TRACE
          if (t == 0 && cta_lin < 4096) g_cta_time[cta_lin][3] = *last_flag ? umma::globaltimer_ns() : 0;
#endif
          if (*last_flag) {
            __threadfence();
            // Stage every split's partials into the stage ring (idle now: all
            // tiles are consumed and all MMAs done) with cp.async, so all the
            // L2 reads are in flight at once, then reduce from shared memory.
            float* po_sh = reinterpret_cast<float*>(smem);              // [8 heads][nb][D]
            float* pm_sh = po_sh + 8 * kMergeChunk * D;                          // [8][kMergeChunk]
            float* pl_sh = pm_sh + 8 * kMergeChunk;                              // [8][kMergeChunk]
            for (int k0 = 0; k0 < n_busy; k0 += kMergeChunk) {
              const int nb = min(kMergeChunk, n_busy - k0);
              const int chunks = QH * nb * (D / 4);                     // 16-byte chunks of O
              for (int i = t; i < chunks; i += 128) {
                const int g = i / (nb * (D / 4)), rem = i % (nb * (D / 4)), k = rem / (D / 4), c4 = rem % (D / 4);
                const int64_t pr = (hq_row0 + g) * S + k0 + k;
                cp_async16(po_sh + (g * kMergeChunk + k) * D + c4 * 4, p.part_o + pr * D + c4 * 4);
              }
              for (int i = t; i < QH * nb; i += 128) {      // (up to 8 x kMergeChunk entries)
                const int g = i / nb, k = i % nb;
                const int64_t pr = (hq_row0 + g) * S + k0 + k;
                pm_sh[g * kMergeChunk + k] = __ldcg(p.part_m + pr);
                pl_sh[g * kMergeChunk + k] = __ldcg(p.part_l + pr);
              }
              cp_async_commit();
              cp_async_wait<0>();
              group_sync(0);
#ifdef FP8KV_TRACE
              if (t == 0 && cta_lin < 4096) g_cta_time[cta_lin][4] = umma::globaltimer_ns();
#endif
#ifdef FP8KV_TRACE
              const long long cc0 = clock64();
#endif
              if (k0 == 0 && nb <= 4) {
                // common case, fully unrolled: every load independent
                float mv[8][4], lv[8][4], oo[8][4];
#pragma unroll
                for (int g = 0; g < 8; ++g)
#pragma unroll
                  for (int u = 0; u < 4; ++u) {
                    const bool in = g < QH && u < nb;
                    mv[g][u] = in ? pm_sh[g * kMergeChunk + u] : -INFINITY;
                    lv[g][u] = in ? pl_sh[g * kMergeChunk + u] : 0.f;
                    oo[g][u] = in ? po_sh[(g * kMergeChunk + u) * D + t] : 0.f;
                  }
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  const float M = fmaxf(fmaxf(mv[g][0], mv[g][1]), fmaxf(mv[g][2], mv[g][3]));
                  float w[4];
#pragma unroll
                  for (int u = 0; u < 4; ++u) w[u] = pow2_diff(mv[g][u] - M, 0);
                  Mg[g] = M;
                  Lg[g] = (w[0] * lv[g][0] + w[1] * lv[g][1]) + (w[2] * lv[g][2] + w[3] * lv[g][3]);
                  Og[g] = (w[0] * oo[g][0] + w[1] * oo[g][1]) + (w[2] * oo[g][2] + w[3] * oo[g][3]);
                }
              } else {
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                if (g < QH) {
                  // up to four splits at a time, their loads independent
                  float M = k0 == 0 ? -INFINITY : Mg[g];
                  for (int k4 = 0; k4 < nb; k4 += 4) {
                    float mk[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) mk[u] = k4 + u < nb ? pm_sh[g * kMergeChunk + k4 + u] : -INFINITY;
                    M = fmaxf(M, fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3])));
                  }
                  const float resc = k0 == 0 ? 0.f : pow2_diff(Mg[g] - M, 0);
                  float L = k0 == 0 ? 0.f : Lg[g] * resc, o = k0 == 0 ? 0.f : Og[g] * resc;
                  for (int k4 = 0; k4 < nb; k4 += 4) {
                    float w[4], lv[4], ovv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                      const bool in = k4 + u < nb;
                      const float mk = in ? pm_sh[g * kMergeChunk + k4 + u] : -INFINITY;
                      w[u] = pow2_diff(mk - M, 0);
                      lv[u] = in ? pl_sh[g * kMergeChunk + k4 + u] : 0.f;
                      ovv[u] = in ? po_sh[(g * kMergeChunk + k4 + u) * D + t] : 0.f;
                    }
                    L += (w[0] * lv[0] + w[1] * lv[1]) + (w[2] * lv[2] + w[3] * lv[3]);
                    o += (w[0] * ovv[0] + w[1] * ovv[1]) + (w[2] * ovv[2] + w[3] * ovv[3]);
                  }
                  Mg[g] = M; Lg[g] = L; Og[g] = o;
                }
              }
              }
#ifdef FP8KV_TRACE
              const long long cc1 = clock64();
              if (t == 0 && cta_lin < 4096) g_cta_time[cta_lin][7] = (unsigned long long)(cc1 - cc0) + (Og[0] == 1234.5f);
#endif
              group_sync(0);
            }
#ifdef FP8KV_TRACE
            if (t == 0 && cta_lin < 4096) g_cta_time[cta_lin][5] = umma::globaltimer_ns();
#endif
#pragma unroll
            for (int g = 0; g < 8; ++g)
              if (g < QH) {
                const float r = Lg[g] > 0.f ? Og[g] / Lg[g] : 0.f;
                const int64_t oi = (hq_row0 + g) * D + t;
                if (p.out_f32) reinterpret_cast<float*>(p.out)[oi] = r;
                else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(r);
              }
#ifdef FP8KV_TRACE
            if (t == 0 && cta_lin < 4096) g_cta_time[cta_lin][6] = umma::globaltimer_ns();
#endif
          }
        }
      }
      if (t == 0) TRACE(1012);
    }
  }
  // (threads other than the merging ones arrived at the cluster barrier at
  // setup and never wait on it: they arrive only once)
  umma::fence_before_sync();
  if (lane == 0) TRACE_MAX(1015);          // last warp at the final barrier
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 1) umma::tmem_dealloc(tmem, 512);
  if (tid == 0) TRACE(1021);
#ifdef FP8KV_TRACE
  if (tid == 0 && cta_lin < 4096) g_cta_time[cta_lin][1] = umma::globaltimer_ns();
#endif
}

// ------------------------------------------------------------ host side --

// True when every cluster of grid.x CTAs (one per (sequence, KV head)) can
// be resident at once, so the cluster launch runs in a single wave like the
// plain launch.  Cached per device, kernel and grid shape.
static bool cluster_fits(const void* fn, dim3 grid, int smem, int threads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return false; }
  struct Key { int dev; const void* fn; unsigned x; };
  static Key keys[16];
  static int vals[16];
  static int n = 0;
  std::lock_guard<std::mutex> lock(host_cache_lock());
  int max_clusters = -1;
  for (int i = 0; i < n; ++i)
    if (keys[i].dev == dev && keys[i].fn == fn && keys[i].x == grid.x) max_clusters = vals[i];
  if (max_clusters < 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      max_clusters = 0;
    }
    if (n < 16) { keys[n] = Key{dev, fn, grid.x}; vals[n] = max_clusters; ++n; }
  }
  return (long long)max_clusters >= (long long)grid.y * grid.z;
}

template <int KE, int VE, int XK = XK_NATIVE, bool PG = false>
static cudaError_t launch_tc_t(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = TcCfg<KE, VE, XK>::BYTES;
  cudaError_t e = ensure_smem_optin((const void*)decode_split_tc<KE, VE, XK, PG>, smem);
  if (e != cudaSuccess) return e;
  DecodeTmaParams tp;
  const CacheView& c = p.c;
  const int64_t rows = c.paged ? (int64_t)c.num_pages * c.kv_heads * c.page_size
                               : (int64_t)c.batch * c.kv_heads * c.max_tokens;
  const int box_rows = c.paged ? c.page_size * p.hpc : kMmaTile;
  if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (!make_map(&tp.tmk, c.k, KE == ELEM_BF16, rows, box_rows) ||
      !make_map(&tp.tmv, c.v, VE != ELEM_E4M3, rows, box_rows))
    return cudaErrorInvalidValue;
  tp.p = p;
  tp.p.cluster = 0;
  const void* fn = (const void*)decode_split_tc<KE, VE, XK, PG>;
  cudaLaunchConfig_t cfg = {};
  constexpr int threads = TcCfg<KE, VE, XK>::THREADS;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (p.fused && p.num_splits >= 2 && p.num_splits <= 8 && cluster_fits(fn, grid, smem, threads)) {
    tp.p.cluster = 1;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = grid.x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (p.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e2 = cudaLaunchKernelEx(&cfg, decode_split_tc<KE, VE, XK, PG>, tp);
  if (e2 != cudaSuccess) (void)cudaGetLastError();
  return e2;
}

#ifdef FP8KV_TRACE
// Zero the per-tile stamps (the TRACE_MAX slots keep a maximum across launches).
extern "C" __attribute__((visibility("default"))) int fp8kv_trace_clear() {
  static const unsigned long long zeros[1024] = {};
  return cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int fp8kv_trace_read(unsigned long long* out, int n) {
  if (n > 1024) n = 1024;
  return cudaMemcpyFromSymbol(out, g_trace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int fp8kv_trace_read_cta(unsigned long long* out, int n) {
  if (n > 4096) n = 4096;
  return cudaMemcpyFromSymbol(out, g_cta_time, n * 8 * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_decode_mma(const DecodeParams& p, int dtype, int batch, cudaStream_t st) {
  dim3 grid(p.num_splits, p.c.kv_heads / p.hpc, batch);
  const bool pg = p.c.paged != 0;
  if (dtype == FP8KV_K8V8) {
    if (p.k_f16 == 1) return launch_tc_t<ELEM_E4M3, ELEM_E4M3, XK_CONSUMER>(p, grid, st);
    if (p.k_f16 == 2) return launch_tc_t<ELEM_E4M3, ELEM_E4M3, XK_PRODUCER>(p, grid, st);
    return pg ? launch_tc_t<ELEM_E4M3, ELEM_E4M3, XK_NATIVE, true>(p, grid, st)
              : launch_tc_t<ELEM_E4M3, ELEM_E4M3>(p, grid, st);
  }
  if (dtype == FP8KV_K16V8)
    return pg ? launch_tc_t<ELEM_BF16, ELEM_E4M3, XK_NATIVE, true>(p, grid, st) : launch_tc_t<ELEM_BF16, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K8V16)
    return pg ? launch_tc_t<ELEM_E4M3, ELEM_BF16, XK_NATIVE, true>(p, grid, st) : launch_tc_t<ELEM_E4M3, ELEM_BF16>(p, grid, st);
  if (dtype == FP8KV_MXK8V8)
    return pg ? launch_tc_t<ELEM_MX, ELEM_E4M3, XK_NATIVE, true>(p, grid, st) : launch_tc_t<ELEM_MX, ELEM_E4M3>(p, grid, st);
  return launch_tc_t<ELEM_BF16, ELEM_BF16>(p, grid, st);
}

}  // namespace fp8kv
