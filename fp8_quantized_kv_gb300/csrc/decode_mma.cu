// decode_mma.cu -- flash-decoding split kernel on the tcgen05 tensor cores.
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
// The e4m3 cache tiles are MMA operands as they sit in shared memory
// (kind::f8f6f4, K tile K-major, V tile MN-major): no per-element K or V
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
// A bf16 K (K16/V8) or V (K16/V16) side uses kind::f16 with the bf16 operands
// exact.
//
// Tiles are staged by 16-byte cp.async into a multi-stage ring laid out in the
// UMMA canonical 128-byte-swizzled form; rows past the sequence end are
// zero-filled in the V tile (0 * NaN would poison P.V).  TMEM: 32 columns
// (S at 0..15, the tile's O at 16..31).  One thread issues the MMAs; waits
// on their completion are bounded (timeout -> device error bit, zero partial).
#include "params.cuh"
#include "umma.cuh"

namespace fp8kv {

constexpr int kMmaTile = 128;

template <int KE, int VE>
struct MmaCfg {
  static constexpr int D = 128;
  static constexpr int K_TILE = kMmaTile * D * (KE == ELEM_E4M3 ? 1 : 2);
  static constexpr int V_TILE = kMmaTile * D * (VE == ELEM_E4M3 ? 1 : 2);
  static constexpr int SCALES = 2 * kMmaTile * 4;
  static constexpr int STAGE = ((K_TILE + V_TILE + SCALES) + 1023) / 1024 * 1024;
  static constexpr int NSTAGE = (KE == ELEM_E4M3 && VE == ELEM_E4M3) ? 3 : (VE == ELEM_E4M3 ? 2 : 3);
  static constexpr int QOP = KE == ELEM_E4M3 ? 16 * 128 : 2 * 16 * 128;     // B operand of QK
  static constexpr int POP = VE == ELEM_E4M3 ? 16 * 128 : 2 * 16 * 128;     // B operand of PV
  static constexpr int MISC = 1024;
  static constexpr int BYTES = NSTAGE * STAGE + QOP + POP + MISC + 1024;    // + alignment slack
};

template <int KE, int VE>
constexpr int mma_smem_bytes() { return MmaCfg<KE, VE>::BYTES; }

// Byte offset of element (row r, column c) of a 128-row tile whose rows are
// `row_bytes` long, in the 128-byte-swizzled UMMA layout: 128-byte column
// blocks are separate [128 rows][128 B] regions; inside, chunk ^= row % 8.
__device__ __forceinline__ int sw128_off(int r, int byte_col, int rows) {
  const int blk = byte_col >> 7, within = byte_col & 127;
  return blk * rows * 128 + r * 128 + ((((within >> 4) ^ (r & 7))) << 4) + (within & 15);
}

__device__ __forceinline__ uint8_t e4m3_rn(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(0.f), "f"(x));
  return (uint8_t)(r & 0xFF);
}
__device__ __forceinline__ float e4m3_val(uint8_t c) {
  float f[4];
  e4m3x4_to_f32_scaled((uint32_t)c, f);
  return f[0] * kTwoPow120;
}

template <int KE, int VE>
__global__ void __launch_bounds__(128) decode_split_mma(DecodeParams p) {
  using C = MmaCfg<KE, VE>;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qop = smem + C::NSTAGE * C::STAGE;
  uint8_t* pop = qop + C::QOP;
  uint8_t* misc = pop + C::POP;
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(misc);
  uint64_t* bar_o = bar_s + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + 16);
  float* qscale = reinterpret_cast<float*>(misc + 32);        // [8]
  float* red_max = qscale + 8;                                // [4][8]
  float* red_sum = red_max + 32;                              // [4][8]
  float* red_v = red_sum + 32;                                // [4]
  int* flag = reinterpret_cast<int*>(red_v + 4);

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
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
  const int t_begin = s * p.chunk_tiles;
  const int t_end = min(t_begin + p.chunk_tiles, tiles);
  const int64_t part0 = ((int64_t)b * p.q_heads + (int64_t)h * G) * S + s;
  if (t_begin >= t_end) {
    for (int i = tid; i < G * D; i += blockDim.x)
      p.part_o[(part0 + (int64_t)(i / D) * S) * D + (i % D)] = 0.f;
    if (tid < G) {
      p.part_m[part0 + (int64_t)tid * S] = -INFINITY;
      p.part_l[part0 + (int64_t)tid * S] = 0.f;
    }
    return;
  }

  // ---- B operand of QK: the query rows (e4m3 hi/lo pairs, or bf16)
  if (tid == 0) *flag = 0;
  for (int i = tid; i < (C::QOP + C::POP) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(qop)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int g = warp; g < 8; g += 4) {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (g < G) {
      const __nv_bfloat16* qr = p.q + ((int64_t)b * p.q_heads + (int64_t)h * G + g) * D + lane * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = __bfloat162float(qr[e]);
    }
    if constexpr (KE == ELEM_E4M3) {
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
      amax = warp_max(amax);
      int ex = 0;
      (void)frexpf(amax * (1.0f / 448.0f), &ex);      // amax * 2^-ex <= 448
      if (lane == 0) qscale[g] = ldexpf(1.0f, ex);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float xs = ldexpf(x[e], -ex);
        const uint8_t hi = e4m3_rn(xs);
        const uint8_t lo = e4m3_rn(xs - e4m3_val(hi));
        const int d = lane * 4 + e;
        qop[sw128_off(g, d, 16)] = hi;
        qop[sw128_off(g + 8, d, 16)] = lo;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<__nv_bfloat16*>(qop + sw128_off(g, (lane * 4 + e) * 2, 16)) = __float2bfloat16_rn(x[e]);
      if (lane == 0) qscale[g] = 1.f;
    }
  }

  // ---- TMEM and barriers
  if (warp == 0) {
    umma::tmem_alloc(tslot, 32);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(bar_s, 1);
    umma::mbar_init(bar_o, 1);
    umma::mbar_fence_init();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 16;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  const int64_t cont_base = ((int64_t)b * c.kv_heads + h) * c.max_tokens;
  auto row_of = [&](int t) -> int64_t {
    if (!c.paged) return cont_base + t;
    const int page = c.page_table[(int64_t)b * c.max_pages_per_seq + (t >> c.page_shift)];
    if (page < 0 || page >= c.num_pages) { raise_error(p.err, FP8KV_DEVERR_BAD_PAGE); return -1; }
    return ((int64_t)page * c.kv_heads + h) * c.page_size + (t & (c.page_size - 1));
  };
  // Stage one tile: K and V rows in the swizzled operand layout, their scales;
  // V rows past T are zero-filled.
  auto issue = [&](int tile, int stage) {
    uint8_t* st = smem + stage * C::STAGE;
    uint8_t* ks = st;
    uint8_t* vs = st + C::K_TILE;
    float* kss = reinterpret_cast<float*>(st + C::K_TILE + C::V_TILE);
    float* vss = kss + kMmaTile;
    const int t0 = tile * kMmaTile;
    const int valid = min(kMmaTile, T - t0);
    const int nrows = min(kMmaTile, (valid + 15) & ~15);
    constexpr int KCPR = KE == ELEM_E4M3 ? 8 : 16, VCPR = VE == ELEM_E4M3 ? 8 : 16;
    constexpr int KRB = KCPR * 16, VRB = VCPR * 16;
    for (int i = tid; i < nrows * KCPR; i += blockDim.x) {
      const int r = i / KCPR, ch = i % KCPR;
      const int64_t row = row_of(t0 + r);
      if (row >= 0) cp_async16(ks + sw128_off(r, ch * 16, kMmaTile), c.k + row * KRB + ch * 16);
    }
    for (int i = tid; i < kMmaTile * VCPR; i += blockDim.x) {
      const int r = i / VCPR, ch = i % VCPR;
      uint8_t* dst = vs + sw128_off(r, ch * 16, kMmaTile);
      if (r < valid) {
        const int64_t row = row_of(t0 + r);
        if (row >= 0) cp_async16(dst, c.v + row * VRB + ch * 16);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    const int nsc = nrows / 4;
    for (int i = tid; i < 2 * nsc; i += blockDim.x) {
      const bool is_v = i >= nsc;
      const int r = (is_v ? i - nsc : i) * 4;
      const float* src = is_v ? c.v_scale : c.k_scale;
      if (src == nullptr) continue;
      const int64_t row = row_of(t0 + r);
      if (row >= 0) cp_async16((is_v ? vss : kss) + r, src + row);
    }
  };

  const int n_tiles = t_end - t_begin;
#pragma unroll 1
  for (int i = 0; i < C::NSTAGE - 1; ++i) {
    if (i < n_tiles) issue(t_begin + i, i);
    cp_async_commit();
  }

  constexpr uint32_t ID_QK = KE == ELEM_E4M3
      ? umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_K, umma::MAJOR_K, 128, 16)
      : umma::idesc(umma::FMT_BF16, umma::FMT_BF16, umma::MAJOR_K, umma::MAJOR_K, 128, 16);
  constexpr uint32_t ID_PV = VE == ELEM_E4M3
      ? umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_MN, umma::MAJOR_K, 128, 16)
      : umma::idesc(umma::FMT_BF16, umma::FMT_BF16, umma::MAJOR_MN, umma::MAJOR_K, 128, 16);
  constexpr uint32_t kWaitLimit = 1u << 22;

  float m_run[8], l_run[8], o_run[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) { m_run[g] = -INFINITY; l_run[g] = 0.f; o_run[g] = 0.f; }
  float qs[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) qs[g] = qscale[g] * p.scale_log2;

  bool failed = false;
#pragma unroll 1
  for (int it = 0; it < n_tiles; ++it) {
    {
      const int nt = it + C::NSTAGE - 1;
      if (nt < n_tiles) issue(t_begin + nt, nt % C::NSTAGE);
      cp_async_commit();
    }
    cp_async_wait<C::NSTAGE - 1>();
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    uint8_t* st = smem + (it % C::NSTAGE) * C::STAGE;
    const float* kss = reinterpret_cast<const float*>(st + C::K_TILE + C::V_TILE);
    const float* vss = kss + kMmaTile;
    const int t0 = (t_begin + it) * kMmaTile;
    const int valid = min(kMmaTile, T - t0);

    // ---- S^T = K . Q^T
    if (tid == 0) {
      const uint32_t ka = umma::smem_u32(st), qa = umma::smem_u32(qop);
      if constexpr (KE == ELEM_E4M3) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma::mma_f8_ss(tmem_s, umma::sdesc(ka + k * 32, 16, 1024, umma::SWIZZLE_128B),
                          umma::sdesc(qa + k * 32, 16, 1024, umma::SWIZZLE_128B), ID_QK, k > 0);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma::mma_f16_ss(tmem_s,
                           umma::sdesc(ka + (k >> 2) * (kMmaTile * 128) + (k & 3) * 32, 16, 1024, umma::SWIZZLE_128B),
                           umma::sdesc(qa + (k >> 2) * (16 * 128) + (k & 3) * 32, 16, 1024, umma::SWIZZLE_128B),
                           ID_QK, k > 0);
      }
      umma::mma_commit(bar_s);
    }
    bool ok = umma::mbar_wait(bar_s, it & 1, kWaitLimit);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    umma::fence_after_sync();

    // ---- scores of token t = tid, tile max, P
    float sc[16];
    umma::tmem_ld16(tmem_s + lane_base, sc);
    const bool tok_ok = tid < valid;
    const float kf = KE == ELEM_E4M3 ? kss[tid] : 1.f;
    float sg[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float raw = KE == ELEM_E4M3 ? (sc[g] + sc[g + 8]) : sc[g];
      sg[g] = tok_ok ? raw * (qs[g] * kf) : -INFINITY;
      const float wm = warp_max(sg[g]);
      if (lane == 0) red_max[warp * 8 + g] = wm;
    }
    const float vsc = VE == ELEM_E4M3 ? (tok_ok ? vss[tid] : 0.f) : 1.f;
    if (VE == ELEM_E4M3) {
      const float vm = warp_max(vsc);
      if (lane == 0) red_v[warp] = vm;
    }
    __syncthreads();
    float alpha[8], beta[8];
    int pex = 0;
    if (VE == ELEM_E4M3) {
      const float vmax = fmaxf(fmaxf(red_v[0], red_v[1]), fmaxf(red_v[2], red_v[3]));
      (void)frexpf(vmax * (1.0f / 448.0f), &pex);
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float mt = fmaxf(fmaxf(red_max[g], red_max[8 + g]), fmaxf(red_max[16 + g], red_max[24 + g]));
      const float mn = fmaxf(m_run[g], mt);
      alpha[g] = exp2f(m_run[g] - mn);
      beta[g] = exp2f(mt - mn);
      m_run[g] = mn;
      const float pj = exp2f(sg[g] - mt);
      const float pb = bf16_round(pj * vsc);
      if constexpr (VE == ELEM_E4M3) {
        const float ps = ldexpf(pb, -pex);
        const uint8_t hi = e4m3_rn(ps);
        const uint8_t lo = e4m3_rn(ps - e4m3_val(hi));
        pop[sw128_off(g, tid, 16)] = hi;
        pop[sw128_off(g + 8, tid, 16)] = lo;
      } else {
        *reinterpret_cast<__nv_bfloat16*>(pop + sw128_off(g, tid * 2, 16)) = __float2bfloat16_rn(pb);
      }
      const float ws = warp_sum(pj);
      if (lane == 0) red_sum[warp * 8 + g] = ws;
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    // ---- O_tile^T = V^T . P'^T
    if (tid == 0) {
      const uint32_t va = umma::smem_u32(st + C::K_TILE), pa = umma::smem_u32(pop);
      if constexpr (VE == ELEM_E4M3) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma::mma_f8_ss(tmem_o, umma::sdesc(va + k * 4 * 1024, 1024, 1024, umma::SWIZZLE_128B),
                          umma::sdesc(pa + k * 32, 16, 1024, umma::SWIZZLE_128B), ID_PV, k > 0);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma::mma_f16_ss(tmem_o, umma::sdesc(va + k * 2 * 1024, kMmaTile * 128, 1024, umma::SWIZZLE_128B),
                           umma::sdesc(pa + (k >> 2) * (16 * 128) + (k & 3) * 32, 16, 1024, umma::SWIZZLE_128B),
                           ID_PV, k > 0);
      }
      umma::mma_commit(bar_o);
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float lt = (red_sum[g] + red_sum[8 + g]) + (red_sum[16 + g] + red_sum[24 + g]);
      l_run[g] = l_run[g] * alpha[g] + lt * beta[g];
    }
    ok = umma::mbar_wait(bar_o, it & 1, kWaitLimit);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    umma::fence_after_sync();

    // ---- fold the tile's O into the running O (thread tid owns dim tid)
    float ov[16];
    umma::tmem_ld16(tmem_o + lane_base, ov);
    const float pf = VE == ELEM_E4M3 ? ldexpf(1.0f, pex) : 1.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float ot = VE == ELEM_E4M3 ? (ov[g] + ov[g + 8]) * pf : ov[g];
      o_run[g] = o_run[g] * alpha[g] + ot * beta[g];
    }
    umma::fence_before_sync();
  }
  cp_async_wait<0>();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();

  if (failed) {
    if (tid == 0) raise_error(p.err, FP8KV_DEVERR_TIMEOUT);
#pragma unroll
    for (int g = 0; g < 8; ++g) { m_run[g] = -INFINITY; l_run[g] = 0.f; o_run[g] = 0.f; }
  }
#pragma unroll
  for (int g = 0; g < 8; ++g)
    if (g < G) p.part_o[(part0 + (int64_t)g * S) * D + tid] = o_run[g];
  if (tid < G) {
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (g == tid) {
        p.part_m[part0 + (int64_t)g * S] = m_run[g];
        p.part_l[part0 + (int64_t)g * S] = l_run[g];
      }
  }
  if (warp == 0) umma::tmem_dealloc(tmem, 32);
}

template <int KE, int VE>
static cudaError_t launch_mma_t(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = mma_smem_bytes<KE, VE>();
  cudaError_t e = ensure_smem_optin((const void*)decode_split_mma<KE, VE>, smem);
  if (e != cudaSuccess) return e;
  decode_split_mma<KE, VE><<<grid, 128, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_mma(const DecodeParams& p, int dtype, int batch, cudaStream_t st) {
  dim3 grid(p.num_splits, p.c.kv_heads, batch);
  if (dtype == FP8KV_K8V8) return launch_mma_t<ELEM_E4M3, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K16V8) return launch_mma_t<ELEM_BF16, ELEM_E4M3>(p, grid, st);
  return launch_mma_t<ELEM_BF16, ELEM_BF16>(p, grid, st);
}

}  // namespace fp8kv
