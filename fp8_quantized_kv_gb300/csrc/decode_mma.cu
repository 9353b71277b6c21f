// decode_mma.cu -- flash-decoding split kernel on the tcgen05 tensor cores,
// warp-specialised and software-pipelined.
//
// Same computation and partials as decode_fma.cu ("FP8 KV cache (fp8_kv,
// opt-in)", bullets "Math" and "Speed"), for head_dim 128 and up to 8 query
// heads per KV head.  A CTA owns one (split, KV head, sequence) and walks its
// 128-token tiles:
//
//   S^T[128 tokens x 16] = K_tile[128 x 128] . Q^T         tcgen05.mma -> TMEM
//   per token (one thread each): s = S * k_scale * sm_scale, tile max, p,
//     P' = bf16_rn(p * v_scale)                              (CUDA cores)
//   O^T[128 dims x 16]   = V_tile^T[128 x 128] . P'^T        tcgen05.mma -> TMEM
//   per dim (one thread each): O = O * e^(m-m') + e^(m_t-m') * O_tile
//
// The e4m3 cache tiles are MMA operands as they land in shared memory
// (kind::f8f6f4; K tile K-major, V tile MN-major): no per-element K or V
// preparation runs on the CUDA cores ("FP8 KV attention: hardware paths and
// tile preparation", sections "Measure the K8/V8 break-even" and "NVIDIA
// Blackwell": the prepare-K and prepare-V stages of the tile interval vanish).
// The other operand of each MMA must then be e4m3 too, so the bf16 query row
// and the bf16-rounded P row are each written as the sum of two e4m3 numbers
// (hi = e4m3(x), lo = e4m3(x - hi)) after an exact power-of-two scaling of
// the row; hi and lo occupy the 16 columns of the N dimension that 8 query
// heads leave free, and are summed after the MMA.  For every component
// within 2^-11 of its row's largest magnitude the pair is exact; smaller
// components carry an absolute error below 2^-19 of the row maximum.
// A bf16 K (K16/V8) or V (K16/V16) side uses kind::f16 with exact operands.
//
// Warp roles ("FP8 KV attention: hardware paths and tile preparation",
// section "Operating model": producer and consumer warps interleave the
// stages across adjacent tiles):
//   warp 0     TMA producer: 128-byte-swizzled tensor loads of the K and V
//              tiles straight into the UMMA operand layout, 1-D bulk copies
//              of the scale rows; a ring of NST stages (full/empty mbarriers).
//   warp 1     TMEM owner and MMA issuer (one thread): QK of tile i, then
//              PV of tile i-1.
//   warps 2-5  softmax of tile i, then the O update of tile i-1 (thread =
//              TMEM lane = token for S, = head dim for O).
// S, O (TMEM) and P (shared memory) are double-buffered, so QK(i+1), PV(i)
// and the softmax of tile i+1 overlap.  Every wait is bounded; a wait that
// runs out raises FP8KV_DEVERR_TIMEOUT, the CTA writes an empty partial and
// leaves.  V rows past the sequence end are zeroed before PV (0 * NaN would
// poison the product).
#include "params.cuh"
#include "tma.cuh"
#include "umma.cuh"

namespace fp8kv {

constexpr int kMmaTile = 128;

template <int KE, int VE>
struct TcCfg {
  static constexpr int D = 128;
  static constexpr int KB = KE == ELEM_E4M3 ? 1 : 2, VB = VE == ELEM_E4M3 ? 1 : 2;
  static constexpr int K_TILE = kMmaTile * D * KB;
  static constexpr int V_TILE = kMmaTile * D * VB;
  static constexpr int STAGE = ((K_TILE + V_TILE + 2 * kMmaTile * 4) + 1023) / 1024 * 1024;
  static constexpr int NST = (KE == ELEM_E4M3 && VE == ELEM_E4M3) ? 6 : (VE == ELEM_E4M3 ? 4 : 3);
  static constexpr int QOP = KE == ELEM_E4M3 ? 16 * 128 : 2 * 16 * 128;
  static constexpr int POP = VE == ELEM_E4M3 ? 16 * 128 : 2 * 16 * 128;
  static constexpr int XO = 8 * 128 * 4;    // group 1's O handed to group 0
  static constexpr int MISC = 2048;
  static constexpr int BYTES = NST * STAGE + QOP + 4 * POP + XO + MISC + 1024;
  static_assert(BYTES <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

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
__device__ __forceinline__ float warp_max_redux(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(x));
  return r;
}
// Exponent e with amax * 2^-e <= 448 (e = 0 for amax = 0).
__device__ __forceinline__ int e4m3_row_exp(float amax) {
  int e = 0;
  (void)frexpf(amax * (1.0f / 448.0f), &e);
  return e;
}

// Bounded wait shared by all roles of a CTA: gives up after 2 s of wall time
// or as soon as another role has given up (abort flag).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  constexpr uint64_t kLimitNs = 2000000000ull;
  if (umma::mbar_try(bar, parity)) return true;
  const uint64_t t0 = umma::globaltimer_ns();
  while (true) {
    if (umma::mbar_try(bar, parity)) return true;
    if (*abort) return false;
    if (umma::globaltimer_ns() - t0 > kLimitNs) {
      *abort = 1;
      return false;
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

struct DecodeTmaParams {
  CUtensorMap tmk;
  CUtensorMap tmv;
  DecodeParams p;
};

// Per-warpgroup barrier set (S, P and O double buffers).
struct WgBars {
  uint64_t s_full[2], s_empty[2], p_full[2], o_full[2], o_empty[2];
};

template <int KE, int VE>
__global__ void __launch_bounds__(320, 1) decode_split_tc(const __grid_constant__ DecodeTmaParams tp) {
  using C = TcCfg<KE, VE>;
  constexpr int D = 128;
  const DecodeParams& p = tp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qop = smem + C::NST * C::STAGE;
  uint8_t* pop0 = qop + C::QOP;                            // [wg][buffer] P operands
  float* xo = reinterpret_cast<float*>(pop0 + 4 * C::POP);   // [8][128]
  uint8_t* misc = pop0 + 4 * C::POP + C::XO;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);     // [8]
  uint64_t* empty = full + 8;                              // [8]
  WgBars* wb = reinterpret_cast<WgBars*>(empty + 8);       // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(wb + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* qscale = reinterpret_cast<float*>(misc + 512);    // [8]
  float* red = qscale + 8;                                 // [wg][2][4][9]
  float* lred = red + 144;                                 // [wg][4][8]
  float* xml = lred + 64;                                  // [16]: m and l of warpgroup 1

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const CacheView& c = p.c;
  const int G = p.group, S = p.num_splits;

  int T = p.seq_lens[b];
  const int cap = cache_capacity(c);
  if (T < 0 || T > cap) {
    if (tid == 0) raise_error(p.err, FP8KV_DEVERR_SEQ_TOO_LONG);
    T = 0;
  }
  const int tiles = (T + kMmaTile - 1) / kMmaTile;
  const int t_begin = split * p.chunk_tiles;
  const int t_end = min(t_begin + p.chunk_tiles, tiles);
  const int64_t part0 = ((int64_t)b * p.q_heads + (int64_t)h * G) * S + split;
  if (t_begin >= t_end) {
    for (int i = tid; i < G * D; i += blockDim.x)
      p.part_o[(part0 + (int64_t)(i / D) * S) * D + (i % D)] = 0.f;
    if (tid < G) {
      p.part_m[part0 + (int64_t)tid * S] = -INFINITY;
      p.part_l[part0 + (int64_t)tid * S] = 0.f;
    }
    return;
  }
  const int n_tiles = t_end - t_begin;

  // ---------------------------------------------------------------- setup
  for (int i = tid; i < (C::QOP + 4 * C::POP) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(qop)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 1) {
    umma::tmem_alloc(tslot, 128);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < C::NST; ++i) {
      umma::mbar_init(&full[i], 1);
      umma::mbar_init(&empty[i], 1 + 4);     // PV commit + the four warps of the owning group
    }
    for (int w = 0; w < 2; ++w)
      for (int i = 0; i < 2; ++i) {
        umma::mbar_init(&wb[w].s_full[i], 1);
        umma::mbar_init(&wb[w].s_empty[i], 4);
        umma::mbar_init(&wb[w].p_full[i], 4);
        umma::mbar_init(&wb[w].o_full[i], 1);
        umma::mbar_init(&wb[w].o_empty[i], 4);
      }
    *abort_flag = 0;
    umma::mbar_fence_init();
  }
  if (tid == 32) {
    tma::prefetch_map(&tp.tmk);
    tma::prefetch_map(&tp.tmv);
  }
  __syncthreads();
  if (warp >= 2 && warp < 6) {   // the B operand of QK: query rows (e4m3 hi/lo pairs, or bf16)
    for (int g = warp - 2; g < 8; g += 4) {
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (g < G) {
        const __nv_bfloat16* qr = p.q + ((int64_t)b * p.q_heads + (int64_t)h * G + g) * D + lane * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = __bfloat162float(qr[e]);
      }
      if constexpr (KE == ELEM_E4M3) {
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        amax = warp_max_redux(amax);
        const int ex = e4m3_row_exp(amax);
        if (lane == 0) qscale[g] = ldexpf(1.0f, ex);
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
        if (lane == 0) qscale[g] = 1.f;
      }
    }
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int64_t cont_row0 = ((int64_t)b * c.kv_heads + h) * c.max_tokens;
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % C::NST, u = i / C::NST;
        if (u > 0 && !wait_or_abort(&empty[s], (u - 1) & 1, abort_flag)) break;
        uint8_t* st = smem + s * C::STAGE;
        float* kss = reinterpret_cast<float*>(st + C::K_TILE + C::V_TILE);
        float* vss = kss + kMmaTile;
        const int t0 = (t_begin + i) * kMmaTile;
        const int valid = min(kMmaTile, T - t0);
        if (!c.paged) {
          const int nsc = min(kMmaTile, (valid + 15) & ~15);
          const uint32_t bytes = C::K_TILE + C::V_TILE + (KE == ELEM_E4M3 ? nsc * 4 : 0) +
                                 (VE == ELEM_E4M3 ? nsc * 4 : 0);
          tma::arrive_expect_tx(&full[s], bytes);
          const int row = (int)(cont_row0 + t0);
          tma::load_2d(st, &tp.tmk, 0, row, &full[s]);
          if (KE != ELEM_E4M3) tma::load_2d(st + kMmaTile * 128, &tp.tmk, 64, row, &full[s]);
          tma::load_2d(st + C::K_TILE, &tp.tmv, 0, row, &full[s]);
          if (VE != ELEM_E4M3) tma::load_2d(st + C::K_TILE + kMmaTile * 128, &tp.tmv, 64, row, &full[s]);
          if (KE == ELEM_E4M3) tma::load_1d(kss, c.k_scale + cont_row0 + t0, nsc * 4, &full[s]);
          if (VE == ELEM_E4M3) tma::load_1d(vss, c.v_scale + cont_row0 + t0, nsc * 4, &full[s]);
        } else {
          const int P = c.page_size;
          const int np = (valid + P - 1) / P;
          const uint32_t per_page = P * 128 * (C::KB + C::VB) + P * 4 * ((KE == ELEM_E4M3) + (VE == ELEM_E4M3));
          tma::arrive_expect_tx(&full[s], per_page * np);
          for (int j = 0; j < np; ++j) {
            int page = c.page_table[(int64_t)b * c.max_pages_per_seq + ((t0 >> c.page_shift) + j)];
            if (page < 0 || page >= c.num_pages) {
              raise_error(p.err, FP8KV_DEVERR_BAD_PAGE);
              page = 0;      // read a valid page; the result is flagged as wrong
            }
            const int64_t row = ((int64_t)page * c.kv_heads + h) * P;
            const int off = j * P * 128;
            tma::load_2d(st + off, &tp.tmk, 0, (int)row, &full[s]);
            if (KE != ELEM_E4M3) tma::load_2d(st + kMmaTile * 128 + off, &tp.tmk, 64, (int)row, &full[s]);
            tma::load_2d(st + C::K_TILE + off, &tp.tmv, 0, (int)row, &full[s]);
            if (VE != ELEM_E4M3)
              tma::load_2d(st + C::K_TILE + kMmaTile * 128 + off, &tp.tmv, 64, (int)row, &full[s]);
            if (KE == ELEM_E4M3) tma::load_1d(kss + j * P, c.k_scale + row, P * 4, &full[s]);
            if (VE == ELEM_E4M3) tma::load_1d(vss + j * P, c.v_scale + row, P * 4, &full[s]);
          }
        }
        ++issued;
      }
      // Before leaving, let every copy this thread issued land (only an
      // aborted run has copies that nobody waited for).
      for (int i = max(0, issued - C::NST); i < issued; ++i)
        (void)umma::mbar_wait(&full[i % C::NST], (i / C::NST) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t ID_QK = KE == ELEM_E4M3
          ? umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_K, umma::MAJOR_K, 128, 16)
          : umma::idesc(umma::FMT_BF16, umma::FMT_BF16, umma::MAJOR_K, umma::MAJOR_K, 128, 16);
      constexpr uint32_t ID_PV = VE == ELEM_E4M3
          ? umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_MN, umma::MAJOR_K, 128, 16)
          : umma::idesc(umma::FMT_BF16, umma::FMT_BF16, umma::MAJOR_MN, umma::MAJOR_K, 128, 16);
      const uint32_t qa = umma::smem_u32(qop);
      for (int i = 0; i <= n_tiles; ++i) {
        if (i < n_tiles) {
          const int s = i % C::NST, u = i / C::NST, w = i & 1, li = i >> 1, bb = li & 1, ub = li >> 1;
          if (!wait_or_abort(&full[s], u & 1, abort_flag)) break;
          if (ub > 0 && !wait_or_abort(&wb[w].s_empty[bb], (ub - 1) & 1, abort_flag)) break;
          umma::fence_after_sync();
          const uint32_t ka = umma::smem_u32(smem + s * C::STAGE);
          const uint32_t d = tmem + 64 * w + 16 * bb;
          if constexpr (KE == ELEM_E4M3) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma::mma_f8_ss(d, umma::sdesc(ka + k * 32, 16, 1024, umma::SWIZZLE_128B),
                              umma::sdesc(qa + k * 32, 16, 1024, umma::SWIZZLE_128B), ID_QK, k > 0);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              umma::mma_f16_ss(d,
                               umma::sdesc(ka + (k >> 2) * (kMmaTile * 128) + (k & 3) * 32, 16, 1024,
                                           umma::SWIZZLE_128B),
                               umma::sdesc(qa + (k >> 2) * (16 * 128) + (k & 3) * 32, 16, 1024,
                                           umma::SWIZZLE_128B),
                               ID_QK, k > 0);
          }
          umma::mma_commit(&wb[w].s_full[bb]);
        }
        if (i >= 1) {
          const int j = i - 1, s = j % C::NST, w = j & 1, lj = j >> 1, bb = lj & 1, ub = lj >> 1;
          if (!wait_or_abort(&wb[w].p_full[bb], ub & 1, abort_flag)) break;
          if (ub > 0 && !wait_or_abort(&wb[w].o_empty[bb], (ub - 1) & 1, abort_flag)) break;
          umma::fence_after_sync();
          const uint32_t va = umma::smem_u32(smem + s * C::STAGE + C::K_TILE);
          const uint32_t pa = umma::smem_u32(pop0 + (2 * w + bb) * C::POP);
          const uint32_t d = tmem + 64 * w + 32 + 16 * bb;
          if constexpr (VE == ELEM_E4M3) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma::mma_f8_ss(d, umma::sdesc(va + k * 4 * 1024, 1024, 1024, umma::SWIZZLE_128B),
                              umma::sdesc(pa + k * 32, 16, 1024, umma::SWIZZLE_128B), ID_PV, k > 0);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              umma::mma_f16_ss(d, umma::sdesc(va + k * 2 * 1024, kMmaTile * 128, 1024, umma::SWIZZLE_128B),
                               umma::sdesc(pa + (k >> 2) * (16 * 128) + (k & 3) * 32, 16, 1024,
                                           umma::SWIZZLE_128B),
                               ID_PV, k > 0);
          }
          umma::mma_commit(&wb[w].o_full[bb]);
          umma::mma_commit(&empty[s]);
        }
      }
    }
  } else {
    // ------------------------------------- softmax and O update (2 groups)
    const int wg = (warp - 2) >> 2;                 // warpgroup: even or odd tiles
    const int t = 32 * (warp & 3) + lane;           // TMEM lane of this thread
    const int sw = warp & 3;                        // lane quarter
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t s_col = 64 * wg, o_col = 64 * wg + 32;
    WgBars& B = wb[wg];
    float qs[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) qs[g] = qscale[g] * p.scale_log2;
    float m_run[8], l_thr[8], o_run[8], a_prev[8], b_prev[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      m_run[g] = -INFINITY; l_thr[g] = 0.f; o_run[g] = 0.f; a_prev[g] = 0.f; b_prev[g] = 0.f;
    }
    float pf_prev = 1.f;
    bool failed = false;
    const int nl = (n_tiles - wg + 1) / 2;          // tiles of this group
    for (int li = 0; li <= nl && !failed; ++li) {
      float a_cur[8], b_cur[8];
      float pf_cur = 1.f;
      if (li < nl) {
        const int i = 2 * li + wg;
        const int s = i % C::NST, u = i / C::NST, bb = li & 1, ub = li >> 1;
        bool ok = wait_or_abort(&B.s_full[bb], ub & 1, abort_flag);
        ok = ok && wait_or_abort(&full[s], u & 1, abort_flag);
        if (group_any(wg, !ok)) { failed = true; break; }
        umma::fence_after_sync();
        float sc[16];
        umma::tmem_ld16(tmem + s_col + 16 * bb + lane_off, sc);
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) umma::mbar_arrive(&B.s_empty[bb]);

        uint8_t* st = smem + s * C::STAGE;
        const float* kss = reinterpret_cast<const float*>(st + C::K_TILE + C::V_TILE);
        const float* vss = kss + kMmaTile;
        const int t0 = (t_begin + i) * kMmaTile;
        const int valid = min(kMmaTile, T - t0);
        const bool tok_ok = t < valid;
        const float kf = KE == ELEM_E4M3 ? kss[t] : 1.f;
        const float vsc = VE == ELEM_E4M3 ? (tok_ok ? vss[t] : 0.f) : 1.f;
        float sg[8];
        float* rb = red + (wg * 2 + (li & 1)) * 36;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float raw = KE == ELEM_E4M3 ? (sc[g] + sc[g + 8]) : sc[g];
          sg[g] = tok_ok ? raw * (qs[g] * kf) : -INFINITY;
          const float wm = warp_max_redux(sg[g]);
          if (lane == 0) rb[sw * 9 + g] = wm;
        }
        if (VE == ELEM_E4M3) {
          const float vm = warp_max_redux(vsc);
          if (lane == 0) rb[sw * 9 + 8] = vm;
        }
        if (!tok_ok) {      // V rows past the sequence end: zero them for PV
          uint4* vrow = reinterpret_cast<uint4*>(st + C::K_TILE);
#pragma unroll
          for (int blk = 0; blk < C::VB; ++blk)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              vrow[(blk * kMmaTile * 128 + t * 128 + ch * 16) / 16] = make_uint4(0, 0, 0, 0);
        }
        group_sync(wg);
        int pex = 0;
        if (VE == ELEM_E4M3) {
          const float vmax = fmaxf(fmaxf(rb[8], rb[17]), fmaxf(rb[26], rb[35]));
          pex = e4m3_row_exp(vmax);
          pf_cur = pow2i(pex);
        }
        const float pinv = pow2i(-pex);
        uint8_t* pop = pop0 + (2 * wg + bb) * C::POP;
        float pb[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float mt = fmaxf(fmaxf(rb[g], rb[9 + g]), fmaxf(rb[18 + g], rb[27 + g]));
          const float mn = fmaxf(m_run[g], mt);
          a_cur[g] = ex2(m_run[g] - mn);
          b_cur[g] = ex2(mt - mn);
          m_run[g] = mn;
          const float pj = ex2(sg[g] - mt);
          l_thr[g] = l_thr[g] * a_cur[g] + pj * b_cur[g];
          pb[g] = bf16_round(pj * vsc);
        }
        if constexpr (VE == ELEM_E4M3) {
#pragma unroll
          for (int g = 0; g < 8; g += 2) {
            const float p0 = pb[g] * pinv, p1 = pb[g + 1] * pinv;
            const uint32_t hi = e4m3x2_rn(p0, p1);
            float hv[4];
            e4m3x4_to_f32_scaled(hi, hv);
            const uint32_t lo = e4m3x2_rn(p0 - hv[0] * kTwoPow120, p1 - hv[1] * kTwoPow120);
            pop[sw128_off(g, t, 16)] = (uint8_t)(hi & 0xFF);
            pop[sw128_off(g + 1, t, 16)] = (uint8_t)(hi >> 8);
            pop[sw128_off(g + 8, t, 16)] = (uint8_t)(lo & 0xFF);
            pop[sw128_off(g + 9, t, 16)] = (uint8_t)(lo >> 8);
          }
        } else {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *reinterpret_cast<__nv_bfloat16*>(pop + sw128_off(g, t * 2, 16)) = __float2bfloat16_rn(pb[g]);
        }
        umma::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          umma::mbar_arrive(&B.p_full[bb]);
          umma::mbar_arrive(&empty[s]);
        }
      }
      if (li >= 1) {
        const int lj = li - 1, bb = lj & 1, ub = lj >> 1;
        const bool ok = wait_or_abort(&B.o_full[bb], ub & 1, abort_flag);
        if (group_any(wg, !ok)) { failed = true; break; }
        umma::fence_after_sync();
        float ov[16];
        umma::tmem_ld16(tmem + o_col + 16 * bb + lane_off, ov);
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) umma::mbar_arrive(&B.o_empty[bb]);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float ot = VE == ELEM_E4M3 ? (ov[g] + ov[g + 8]) * pf_prev : ov[g];
          o_run[g] = o_run[g] * a_prev[g] + ot * b_prev[g];
        }
      }
      if (li < nl) {
#pragma unroll
        for (int g = 0; g < 8; ++g) { a_prev[g] = a_cur[g]; b_prev[g] = b_cur[g]; }
        pf_prev = pf_cur;
      }
    }
    if (failed) {
      if (t == 0) raise_error(p.err, FP8KV_DEVERR_TIMEOUT);
#pragma unroll
      for (int g = 0; g < 8; ++g) { m_run[g] = -INFINITY; l_thr[g] = 0.f; o_run[g] = 0.f; }
    }
    // l: per-thread partial sums -> one total per head and group
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float ws = warp_sum(l_thr[g]);
      if (lane == 0) lred[(wg * 4 + sw) * 8 + g] = ws;
    }
    group_sync(wg);
    float l_tot[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float* lr = lred + wg * 32;
      l_tot[g] = (lr[g] + lr[8 + g]) + (lr[16 + g] + lr[24 + g]);
    }
    // The two groups' running states are merged like two splits: group 1
    // hands its (m, l, O) to group 0 through shared memory.
    if (wg == 1) {
#pragma unroll
      for (int g = 0; g < 8; ++g) xo[g * D + t] = o_run[g];
      if (t == 0) {
#pragma unroll
        for (int g = 0; g < 8; ++g) { xml[g] = m_run[g]; xml[8 + g] = l_tot[g]; }
      }
    }
    asm volatile("bar.sync 3, 256;\n" ::: "memory");
    if (wg == 0) {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float m1 = xml[g], l1 = xml[8 + g];
        const float M = fmaxf(m_run[g], m1);
        const float f0 = m_run[g] == -INFINITY ? 0.f : ex2(m_run[g] - M);
        const float f1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
        const float o = o_run[g] * f0 + xo[g * D + t] * f1;
        if (g < G) p.part_o[(part0 + (int64_t)g * S) * D + t] = o;
        if (t == g && g < G) {
          p.part_m[part0 + (int64_t)g * S] = M;
          p.part_l[part0 + (int64_t)g * S] = l_tot[g] * f0 + l1 * f1;
        }
      }
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 1) umma::tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------ host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

// Tensor map of a K or V store viewed as [rows][128 elements], boxes of
// `box_rows` rows by 128 bytes, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t rows, int box_rows) {
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

template <int KE, int VE>
static cudaError_t launch_tc_t(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = TcCfg<KE, VE>::BYTES;
  cudaError_t e = ensure_smem_optin((const void*)decode_split_tc<KE, VE>, smem);
  if (e != cudaSuccess) return e;
  DecodeTmaParams tp;
  const CacheView& c = p.c;
  const int64_t rows = c.paged ? (int64_t)c.num_pages * c.kv_heads * c.page_size
                               : (int64_t)c.batch * c.kv_heads * c.max_tokens;
  const int box_rows = c.paged ? c.page_size : kMmaTile;
  if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (!make_map(&tp.tmk, c.k, KE != ELEM_E4M3, rows, box_rows) ||
      !make_map(&tp.tmv, c.v, VE != ELEM_E4M3, rows, box_rows))
    return cudaErrorInvalidValue;
  tp.p = p;
  decode_split_tc<KE, VE><<<grid, 320, smem, st>>>(tp);
  return cudaGetLastError();
}

cudaError_t launch_decode_mma(const DecodeParams& p, int dtype, int batch, cudaStream_t st) {
  dim3 grid(p.num_splits, p.c.kv_heads, batch);
  if (dtype == FP8KV_K8V8) return launch_tc_t<ELEM_E4M3, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K16V8) return launch_tc_t<ELEM_BF16, ELEM_E4M3>(p, grid, st);
  return launch_tc_t<ELEM_BF16, ELEM_BF16>(p, grid, st);
}

}  // namespace fp8kv
