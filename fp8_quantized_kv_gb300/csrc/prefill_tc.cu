// prefill_tc.cu -- causal prefill attention over an e4m3 K/V cache on the
// tcgen05 tensor cores.
//
// "03 · 8n — FA-style tiled prefill attention", sections 2.1 and 3.1: query
// tiles against 64-token KV tiles up to the causal limit, online softmax with
// running max m, sum l and an O accumulator; a key is valid for the query at
// position qp iff key <= qp.  FP8 numerics of "FP8 KV cache (fp8_kv, opt-in)",
// bullet "Math": the K scale folds into the scores and the V scale into P,
// which is rounded to a 16-bit operand before P.V.
//
// A CTA owns 128 query rows (two 64-token query tiles: the full-rate tcgen05
// shape is M = 128) of one query head, and walks the KV tiles of that head's
// KV head:
//   S[128 x 64]    = (Q_hi + Q_lo) . K^T  tcgen05.mma kind::f8f6f4 -> TMEM
//   per row (one thread each, whole row thread-local): s = S * k_scale *
//     sm_scale, causal mask (diagonal tiles only), running max with lazy
//     rescale, p = 2^(s - m), l += p, P' = p * v_scale
//   O[128 x 128]  += P' . V                kind::f16 -> TMEM (lane = query row)
// Two softmax warpgroups take alternate KV tiles (even, odd), each with its
// own running (m, l) and its own O accumulator, so the softmax of two tiles
// runs at once; the two states are combined per row in the epilogue, as two
// flash-decoding splits are.  The warps of a group share no barrier inside
// the loop: each query row is one thread and one TMEM lane, so every
// decision (the lazy rescale, a wait that gave up) is a warp vote.
// QK runs on the e4m3 K tile as it lands in shared memory ("FP8 KV
// attention: hardware paths and tile preparation", section "Use a native
// narrow QK path": no K preparation), with each bf16 query row, after a
// power-of-two scaling that puts its largest magnitude at most 448, written
// as two e4m3 terms (hi = e4m3(x), lo = e4m3(x - hi)).  P.V is kind::f16:
// the e4m3 V codes convert to f16 exactly (cvt.rn.f16x2.e4m3x2).  P' is
// rounded once, to the 16-bit operand of the P.V product, as f16 (11-bit
// significand, 8x finer than bf16; the page's own prefill keeps its
// probabilities in f16, section 2.4) after a power-of-two scaling 2^-kp of
// the row: kp follows the largest V scale of the tiles the row has seen (it
// is only ever raised, and O is rescaled with it), so P' stays inside f16's
// range, and it folds into the exponential's argument.  All those scalings
// are undone in fp32.  The per-element fp32 arithmetic runs two-wide.
//
// Warp roles:
//   warp 0      TMA producer: e4m3 code tiles (64 keys x 128 B, 128-byte
//               swizzle) and 1-D bulk copies of the scale rows into a ring.
//   warp 1      TMEM owner and QK issuer (one thread).
//   warp 14     PV issuer (one thread): QK and PV each wait only for their
//               own operands.
//   warps 2-5   softmax of the even tiles, warps 6-9 of the odd tiles (one
//               query row per thread); then the output epilogue.
//   warps 10-13 preparation, warp 10 + w of tiles w, w + 4, ...: V codes ->
//               f16 operand tiles (MN-major), per-key scales and the tile's
//               largest V scale; V rows past the causal end zeroed (0 * NaN
//               would poison P.V).
//   warp 15     idle.
// TMEM: S of each group double-buffered (4 x 64 columns), one O per group
// (2 x 128).  O is rescaled in TMEM only when a row's maximum grows by more
// than 2^8 (then P stays <= 2^8 relative to the stale maximum) or its kp
// rises.  Every wait is bounded; a timeout raises FP8KV_DEVERR_TIMEOUT.
#include "params.cuh"
#include "tc_common.cuh"

namespace fp8kv {

constexpr int kPfRows = 128;   // query rows per CTA
constexpr int kPfKeys = 64;    // keys per KV tile
constexpr int kPfThreads = 512;

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

struct PfTcCfg {
  static constexpr int D = 128;
  static constexpr int QOP = 2 * kPfRows * D;                 // [hi, lo][128 rows][128 B] e4m3
  static constexpr int CODES = kPfKeys * D;                    // e4m3 tile [64][128]
  static constexpr int STAGE = ((2 * CODES + 2 * kPfKeys * 4) + 1023) / 1024 * 1024;
  static constexpr int NS = 4;                                 // e4m3 code stages
  static constexpr int NOP = 4;                                // f16 V operand buffers
  static constexpr int OPT = kPfKeys * D * 2;                 // f16 V tile [2 atoms][64][128 B]
  static constexpr int POP = kPfRows * kPfKeys * 2;           // f16 P [128 rows][128 B], one per group
  static constexpr int CST = 2 * kPfKeys + 4;                   // floats per buffer: k, v column scales, v max
  static constexpr int NCOL = 8;                                // column-scale buffers (tile j: j % 8)
  static constexpr int COLS = CST * 4;
  static constexpr int MISC = 4096;
  static constexpr int BYTES = QOP + NS * STAGE + NOP * OPT + 2 * POP + NCOL * COLS + MISC + 1024;
  static_assert(BYTES <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

#ifdef FP8KV_TRACE
// Per-tile clock64 stamps of CTA (0, 0, 0) (the longest query tile):
// slot 8*j + {0: TMA issue, 1: QK issue, 2: PV issue, 3: operands ready,
// 4: softmax has S, 5: P ready}; 1010: epilogue start; 1020/1021: begin/end.
__device__ unsigned long long g_pf_trace[1024];
// per CTA (launch order): start, epilogue start, end (globaltimer ns), SM id
__device__ unsigned long long g_pf_cta[2048][4];
#define PF_CTA(k, v)                                                                              \
  do {                                                                                            \
    const int cl_ = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;              \
    if (cl_ < 2048) g_pf_cta[cl_][(k)] = (v);                                                     \
  } while (0)
#define PF_TRACE(slot)                                                               \
  do {                                                                               \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (slot) < 1024)      \
      g_pf_trace[(slot)] = clock64();                                                \
  } while (0)
// sub-steps of the softmax of tile 10 (row 0): slots 900 + k
#define PF_SUB(j, k)                                  \
  do {                                                \
    if ((j) == 10 && r == 0) PF_TRACE(900 + (k));     \
  } while (0)
#else
#define PF_TRACE(slot) \
  do {                 \
  } while (0)
#define PF_SUB(j, k) \
  do {               \
  } while (0)
#define PF_CTA(k, v) \
  do {               \
  } while (0)
#endif

struct PrefillTmaParams {
  CUtensorMap tmk;
  CUtensorMap tmv;
  PrefillParams p;
};

// OR of `pred` over the 256 softmax threads (named barrier 3).
__device__ __forceinline__ bool pair_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 3, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_tc(const __grid_constant__ PrefillTmaParams tp) {
  using C = PfTcCfg;
  constexpr int D = 128;
  const PrefillParams& p = tp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qop = smem;
  uint8_t* ring = qop + C::QOP;
  uint8_t* vf = ring + C::NS * C::STAGE;          // [NOP] f16 V operand
  uint8_t* pop = vf + C::NOP * C::OPT;            // [group] f16 P operand
  float* cols = reinterpret_cast<float*>(pop + 2 * C::POP);   // [NCOL][k 64 | v 64 | v max]
  uint8_t* misc = reinterpret_cast<uint8_t*>(cols + C::NCOL * C::CST);
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);        // [NS] codes landed
  uint64_t* empty = full + C::NS;                             // [NS] K read by QK, V converted by the prep warps
  uint64_t* op_full = empty + C::NS;                          // [NOP] f16 V operand + scales ready
  uint64_t* op_free = op_full + C::NOP;                       // [NOP] PV of the buffer's tile finished
  uint64_t* s_full = op_free + C::NOP;                        // [group][2]
  uint64_t* s_free = s_full + 4;                              // [group][2]
  uint64_t* p_full = s_free + 4;                              // [group]
  uint64_t* pv_done = p_full + 2;                             // [group] PV of the group's last tile finished
  uint64_t* drained = pv_done + 2;                            // [2] final commits of the two MMA issuers
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drained + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* m_sh = reinterpret_cast<float*>(misc + 1280);        // [group][128] final reference maxima
  float* l_sh = reinterpret_cast<float*>(misc + 2304);        // [group][128] final row sums
  int* kp_sh = reinterpret_cast<int*>(misc + 256);           // [group][128] final P' exponents
  uint64_t* cols_full = reinterpret_cast<uint64_t*>(misc + 3328);   // [NCOL] column scales of a tile written

  // grid (query head, sequence, query tile), the tile index slowest and
  // reversed: the CTAs with the longest causal ranges launch first
  const int hq = blockIdx.x, b = blockIdx.y, qt = gridDim.z - 1 - blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {                                 // the TMA unit fetches the maps while the CTA sets up
    tma::prefetch_map(&tp.tmk);
    tma::prefetch_map(&tp.tmv);
  }
  const CacheView& c = p.c;
  const int hk = hq / p.group;
  const int pos0 = p.q_pos0[b];
  const int i0 = qt * kPfRows;
  const int last_i = min(p.n_q, i0 + kPfRows) - 1;
  const int kv_end = pos0 + last_i + 1;
  if (pos0 < 0 || kv_end > cache_capacity(c)) {
    if (tid == 0) raise_error(p.err, FP8KV_DEVERR_SEQ_TOO_LONG);
    return;
  }
  const int nkv = (kv_end + kPfKeys - 1) / kPfKeys;
  const int64_t cont_row0 = ((int64_t)b * c.kv_heads + hk) * c.max_tokens;

  auto produce = [&](int j) {
    PF_TRACE(8 * j + 0);
    const int s = j % C::NS;
    uint8_t* st = ring + s * C::STAGE;
    float* kss = reinterpret_cast<float*>(st + 2 * C::CODES);
    float* vss = kss + kPfKeys;
    const int t0 = j * kPfKeys;
    const int valid = min(kPfKeys, kv_end - t0);
    if (!c.paged) {
      const int nsc = min(kPfKeys, (valid + 15) & ~15);
      tma::arrive_expect_tx(&full[s], 2 * C::CODES + 2 * nsc * 4);
      const int row = (int)(cont_row0 + t0);
      tma::load_2d(st, &tp.tmk, 0, row, &full[s]);
      tma::load_2d(st + C::CODES, &tp.tmv, 0, row, &full[s]);
      tma::load_1d(kss, c.k_scale + cont_row0 + t0, nsc * 4, &full[s]);
      tma::load_1d(vss, c.v_scale + cont_row0 + t0, nsc * 4, &full[s]);
    } else {
      const int P = c.page_size;
      const int np = (valid + P - 1) / P;
      tma::arrive_expect_tx(&full[s], np * (2 * P * 128 + 2 * P * 4));
      for (int k = 0; k < np; ++k) {
        int page = c.page_table[(int64_t)b * c.max_pages_per_seq + ((t0 >> c.page_shift) + k)];
        if (page < 0 || page >= c.num_pages) {
          raise_error(p.err, FP8KV_DEVERR_BAD_PAGE);
          page = 0;
        }
        const int64_t row = ((int64_t)page * c.kv_heads + hk) * P;
        tma::load_2d(st + k * P * 128, &tp.tmk, 0, (int)row, &full[s]);
        tma::load_2d(st + C::CODES + k * P * 128, &tp.tmv, 0, (int)row, &full[s]);
        tma::load_1d(kss + k * P, c.k_scale + row, P * 4, &full[s]);
        tma::load_1d(vss + k * P, c.v_scale + row, P * 4, &full[s]);
      }
    }
  };

  // ---------------------------------------------------------------- setup
  const int n_first = min(nkv, C::NS);
  if (tid == 0) PF_TRACE(1020);
#ifdef FP8KV_TRACE
  if (tid == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    PF_CTA(0, umma::globaltimer_ns());
    PF_CTA(3, smid);
  }
#endif
  if (tid == 0) {
    for (int i = 0; i < C::NS; ++i) {
      umma::mbar_init(&full[i], 1);
      umma::mbar_init(&empty[i], 1 + 1);       // QK commit + the prep warp of the tile
    }
    *abort_flag = 0;
    umma::mbar_fence_init();
    for (int j = 0; j < n_first; ++j) produce(j);
    for (int i = 0; i < C::NOP; ++i) {
      umma::mbar_init(&op_full[i], 1);
      umma::mbar_init(&op_free[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      umma::mbar_init(&s_full[i], 1);
      umma::mbar_init(&s_free[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      umma::mbar_init(&p_full[i], 4);
      umma::mbar_init(&pv_done[i], 1);
    }
    umma::mbar_init(&drained[0], 1);
    umma::mbar_init(&drained[1], 1);
    for (int i = 0; i < C::NCOL; ++i) umma::mbar_init(&cols_full[i], 1);
    umma::mbar_fence_init();
  }
  if (warp == 1) {
    umma::tmem_alloc(tslot, 512);
    umma::tmem_relinquish();
  }
  // softmax warps: this thread's query row -> the QK A operand as two e4m3
  // terms (hi = e4m3(x), lo = e4m3(x - hi)) after scaling the row by 2^-kq so
  // its largest magnitude is at most 448; both groups compute the row's
  // scale, each writes 64 of the 128 dims of both terms
  const int r = 32 * (warp & 3) + lane;           // query row (softmax warps) / TMEM lane
  const int wg = (warp - 2) >> 2;                 // softmax group: tiles j with j % 2 == wg
  const int qi = i0 + r;
  const int qpos = qi < p.n_q ? pos0 + qi : -1;
  int kq = 0;
  if (warp >= 2 && warp < 10) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (((int64_t)b * p.n_q + (qi < p.n_q ? qi : 0)) * p.q_heads + hq) * D);
    uint4 mine[8];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 w = qi < p.n_q ? src[k] : make_uint4(0, 0, 0, 0);
      const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f2[2];
        bf16x2_to_f32(w4[u], f2);
        amax = fmaxf(amax, fmaxf(fabsf(f2[0]), fabsf(f2[1])));
      }
      if ((k >> 3) == wg) mine[k & 7] = w;
    }
    kq = max(-100, min(100, e4m3_row_exp(amax)));
    const float qsc = pow2i(-kq);
#pragma unroll
    for (int c16 = 0; c16 < 4; ++c16) {            // 16 dims (one 16-byte e4m3 chunk) each
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {                // 4 dims at a time
        const uint4 w = mine[2 * c16 + (u >> 1)];
        const uint32_t wa = (u & 1) ? w.z : w.x, wb = (u & 1) ? w.w : w.y;
        float f2[2], g2[2];
        bf16x2_to_f32(wa, f2);
        bf16x2_to_f32(wb, g2);
        const float x0 = f2[0] * qsc, x1 = f2[1] * qsc, x2 = g2[0] * qsc, x3 = g2[1] * qsc;
        const uint32_t h = e4m3x2_rn(x0, x1) | (e4m3x2_rn(x2, x3) << 16);
        float hv[4];
        e4m3x4_to_f32_scaled(h, hv);
        hi[u] = h;
        lo[u] = e4m3x2_rn(x0 - hv[0] * kTwoPow120, x1 - hv[1] * kTwoPow120) |
                (e4m3x2_rn(x2 - hv[2] * kTwoPow120, x3 - hv[3] * kTwoPow120) << 16);
      }
      const int ch = 4 * wg + c16;
      const int off = r * 128 + ((ch ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(qop + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(qop + kPfRows * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
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
      int issued = n_first;
      for (int j = n_first; j < nkv; ++j) {
        const int s = j % C::NS, u = j / C::NS;
        if (!wait_fast(&empty[s], (u - 1) & 1, abort_flag)) break;
        produce(j);
        ++issued;
      }
      for (int j = max(0, issued - C::NS); j < issued; ++j)
        (void)umma::mbar_wait(&full[j % C::NS], (j / C::NS) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t ID_QK = umma::idesc(umma::FMT_E4M3, umma::FMT_E4M3, umma::MAJOR_K, umma::MAJOR_K, 128, 64);
      const uint32_t qa = umma::smem_u32(qop);
      // QK issuer.  Tile j: group w = j % 2, its local index lj = j / 2, S
      // buffer lj % 2.  The PVs are issued by another warp (warp 14), so a
      // QK waiting for its K tile never holds up a PV and vice versa.
      for (int j = 0; j < nkv; ++j) {
        const int w = j & 1, lj = j >> 1, bb = lj & 1, ub = lj >> 1, s = j % C::NS, u = j / C::NS;
        if (!wait_fast(&full[s], u & 1, abort_flag)) break;
        if (ub > 0 && !wait_fast(&s_free[2 * w + bb], (ub - 1) & 1, abort_flag)) break;
        umma::fence_after_sync();
        PF_TRACE(8 * j + 1);
        // S = (Q_hi + Q_lo) . K: the e4m3 K codes are the B operand as they
        // landed (K-major, 128-byte swizzle), 32 dims per MMA
        const uint32_t ka = umma::smem_u32(ring + s * C::STAGE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_f8_ss(tmem + 64 * (2 * w + bb),
                          umma::sdesc(qa + (kk >> 2) * (kPfRows * 128) + (kk & 3) * 32, 16, 1024, umma::SWIZZLE_128B),
                          umma::sdesc(ka + (kk & 3) * 32, 16, 1024, umma::SWIZZLE_128B), ID_QK, kk > 0);
        umma::mma_commit(&s_full[2 * w + bb]);
        umma::mma_commit(&empty[s]);
      }
      // all issued MMAs complete before TMEM is released (matters only when
      // a wait above gave up)
      umma::mma_commit(&drained[0]);
      (void)umma::mbar_wait(&drained[0], 0, 100000000ull);
    }
  } else if (warp == 14) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t ID_PV = umma::idesc(umma::FMT_F16, umma::FMT_F16, umma::MAJOR_K, umma::MAJOR_MN, 128, 128);
      for (int j = 0; j < nkv; ++j) {
        const int w = j & 1, lj = j >> 1, ob = j % C::NOP, ou = j / C::NOP;
        if (!wait_fast(&p_full[w], lj & 1, abort_flag)) break;
        if (!wait_fast(&op_full[ob], ou & 1, abort_flag)) break;
        umma::fence_after_sync();
        PF_TRACE(8 * j + 2);
        const uint32_t va = umma::smem_u32(vf + ob * C::OPT);
        const uint32_t pa = umma::smem_u32(pop + w * C::POP);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_f16_ss(tmem + 256 + 128 * w, umma::sdesc(pa + kk * 32, 16, 1024, umma::SWIZZLE_128B),
                           umma::sdesc(va + kk * 2048, kPfKeys * 128, 1024, umma::SWIZZLE_128B), ID_PV,
                           (lj > 0 || kk > 0) ? 1u : 0u);
        umma::mma_commit(&pv_done[w]);
        umma::mma_commit(&op_free[ob]);
      }
      // this thread's MMAs complete before TMEM is released
      umma::mma_commit(&drained[1]);
      (void)umma::mbar_wait(&drained[1], 0, 100000000ull);
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------- softmax
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float qsr = pow2i(kq);
    const int qpos_min = pos0 + i0;                 // smallest position among this CTA's queries
    const int my_tiles = (nkv - wg + 1) >> 1;       // tiles j = 2 lj + wg < nkv
    const uint32_t s_base = tmem + 64 * (2 * wg), o_base = tmem + 256 + 128 * wg;
    uint8_t* my_p = pop + wg * C::POP;
    float m_used = -INFINITY, l = 0.f;
    int kp_row = -1000;                             // this row's P' exponent (none yet)
    bool failed = false;
    for (int lj = 0; lj < my_tiles; ++lj) {
      const int j = 2 * lj + wg, bb = lj & 1, ub = lj >> 1, cb = j % C::NCOL;
      PF_SUB(j, 0);
      bool ok = wait_fast(&s_full[2 * wg + bb], ub & 1, abort_flag);
      ok = ok && wait_fast(&cols_full[cb], (j / C::NCOL) & 1, abort_flag);
      ok = ok && !*abort_flag;
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      umma::fence_after_sync();
      if (r == 0) PF_TRACE(8 * j + 4);
      PF_SUB(j, 1);
      // the row's 64 scores as pairs (packed two-wide fp32 arithmetic below)
      float2 sv[32];
      {
        uint32_t rr[4][16];
#pragma unroll
        for (int k = 0; k < 4; ++k) umma::tmem_ld16_nowait(s_base + 64 * bb + 16 * k + lane_off, rr[k]);
        umma::tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int u = 0; u < 8; ++u) sv[8 * k + u] = make_float2(__uint_as_float(rr[k][2 * u]), __uint_as_float(rr[k][2 * u + 1]));
      }
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&s_free[2 * wg + bb]);
      PF_SUB(j, 2);
      // t = S * k_scale * sm_scale * log2(e); the row's 2^kq comes in below
      const float4* kc4 = reinterpret_cast<const float4*>(cols + cb * C::CST);
      const float4* vc4 = kc4 + kPfKeys / 4;
      const float vmt = cols[cb * C::CST + 2 * kPfKeys];   // largest V scale of the tile
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 kc = kc4[c4];
        sv[2 * c4] = __fmul2_rn(sv[2 * c4], make_float2(kc.x, kc.y));
        sv[2 * c4 + 1] = __fmul2_rn(sv[2 * c4 + 1], make_float2(kc.z, kc.w));
      }
      const int t0 = j * kPfKeys;
      if (t0 + kPfKeys - 1 > qpos_min) {             // causal edge: keys past this row's position drop out
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) {
          sv[cc].x = t0 + 2 * cc <= qpos ? sv[cc].x : -INFINITY;
          sv[cc].y = t0 + 2 * cc + 1 <= qpos ? sv[cc].y : -INFINITY;
        }
      }
      PF_SUB(j, 3);
      // the row's maximum by three-input max: 36 instructions for 64 scores
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        m8[k] = fmax3f(fmax3f(sv[k].x, sv[k].y, sv[k + 8].x), fmax3f(sv[k + 8].y, sv[k + 16].x, sv[k + 16].y),
                       fmaxf(sv[k + 24].x, sv[k + 24].y));
      const float mt = fmax3f(fmax3f(m8[0], m8[1], m8[2]), fmax3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * qsr;
      // lazy rescale: move the row's reference maximum only when it grows by
      // more than 2^8 (or on the first tile with a valid key)
      float alpha = 1.f;
      if (mt != -INFINITY && (m_used == -INFINITY || mt > m_used + 8.f)) {
        alpha = m_used == -INFINITY ? 0.f : ex2(m_used - mt);
        m_used = mt;
      }
      // P' = p * v_scale * 2^-kp_row with p <= 2^8: kp_row (this row's, only
      // ever raised, O rescaled with it) keeps P' below 2^15, inside f16
      float alpha_o = alpha;                        // O's factor: the max move and the exponent move
      if (vmt > 0.f) {
        const int need = max(-100, min(120, ((__float_as_int(vmt) >> 23) & 0xFF) - 127 - 6));   // vmt 2^-need < 128
        if (need > kp_row) {
          if (kp_row > -1000) alpha_o *= pow2_diff((float)(kp_row - need), 0);
          kp_row = need;
        }
      }
      PF_SUB(j, 4);
      const int kpr = kp_row > -1000 ? kp_row : 0;
      const float neg_m = (m_used == -INFINITY ? 0.f : -m_used) - (float)kpr;
      const float2 qsr2 = make_float2(qsr, qsr), nm2 = make_float2(neg_m, neg_m);
      float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
      uint32_t ph[32];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 vc = vc4[c4];
        const float2 a01 = __ffma2_rn(sv[2 * c4], qsr2, nm2), a23 = __ffma2_rn(sv[2 * c4 + 1], qsr2, nm2);
        const float2 p01 = make_float2(ex2_ftz(a01.x), ex2_ftz(a01.y));
        const float2 p23 = make_float2(ex2_ftz(a23.x), ex2_ftz(a23.y));
        la = __fadd2_rn(la, p01);
        lb = __fadd2_rn(lb, p23);
        // (p here is p * 2^-kp_row) P' = p * v_scale * 2^-kp_row, rounded
        // once to the f16 operand
        const float2 q01 = __fmul2_rn(p01, make_float2(vc.x, vc.y)), q23 = __fmul2_rn(p23, make_float2(vc.z, vc.w));
        const __half2 h01 = __floats2half2_rn(q01.x, q01.y);
        const __half2 h23 = __floats2half2_rn(q23.x, q23.y);
        ph[2 * c4] = *reinterpret_cast<const uint32_t*>(&h01);
        ph[2 * c4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
      }
      const float l4[4] = {la.x, la.y, lb.x, lb.y};
      l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3])) * pow2i(kpr);
      PF_SUB(j, 5);
      // this group's previous P.V (tile j-2) must be done before its O is
      // rescaled and before its P buffer is overwritten
      if (lj > 0) {
        const bool done = wait_fast(&pv_done[wg], (lj - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, done)) { failed = true; break; }
      }
      PF_SUB(j, 6);
      if (__any_sync(0xffffffffu, alpha_o != 1.f && lj > 0)) {
        // O rows whose reference moved are rescaled in TMEM: lane = query
        // row, so each thread scales its own row (alpha 1 elsewhere in the warp)
        umma::fence_after_sync();
#pragma unroll 1
        for (int k = 0; k < 8; ++k) {             // 8 chunks of 16 columns (head dims)
          uint32_t rr[16];
          umma::tmem_ld16_nowait(o_base + 16 * k + lane_off, rr);
          umma::tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 16; ++u) rr[u] = __float_as_uint(__uint_as_float(rr[u]) * alpha_o);
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
              "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(o_base + 16 * k + lane_off),
              "r"(rr[0]), "r"(rr[1]), "r"(rr[2]), "r"(rr[3]), "r"(rr[4]), "r"(rr[5]), "r"(rr[6]), "r"(rr[7]),
              "r"(rr[8]), "r"(rr[9]), "r"(rr[10]), "r"(rr[11]), "r"(rr[12]), "r"(rr[13]), "r"(rr[14]), "r"(rr[15]));
        }
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      }
      PF_SUB(j, 7);
      uint8_t* prow = my_p + r * 128;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8)
        *reinterpret_cast<uint4*>(prow + ((c8 ^ (r & 7)) << 4)) =
            make_uint4(ph[4 * c8], ph[4 * c8 + 1], ph[4 * c8 + 2], ph[4 * c8 + 3]);
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&p_full[wg]);
      if (r == 0) PF_TRACE(8 * j + 5);
      PF_SUB(j, 8);
    }
    m_sh[wg * kPfRows + r] = failed ? -INFINITY : m_used;
    kp_sh[wg * kPfRows + r] = kp_row > -1000 ? kp_row : 0;
    l_sh[wg * kPfRows + r] = failed ? 0.f : l;
    // ------------------------------------------------------------ epilogue
    // both groups' states are visible after this barrier; a failure in
    // either group skips the epilogue in both
    bool any_fail = pair_any(failed);
    if (r == 0 && wg == 0) PF_TRACE(1010);
#ifdef FP8KV_TRACE
    if (r == 0 && wg == 0) PF_CTA(1, umma::globaltimer_ns());
#endif
    const int n0 = (nkv + 1) >> 1, n1 = nkv >> 1;   // tiles of each group
    if (!any_fail) {
      bool ok = n0 == 0 || wait_or_abort(&pv_done[0], (n0 - 1) & 1, abort_flag);
      ok = ok && (n1 == 0 || wait_or_abort(&pv_done[1], (n1 - 1) & 1, abort_flag));
      any_fail = pair_any(!ok);
    }
    if (!any_fail) {
      // lane = query row r: combine the two groups' O rows (one flash-decoding
      // style merge per row); group wg writes head dims 64 wg .. 64 wg + 63
      umma::fence_after_sync();
      const float ma = m_sh[r], mb = m_sh[kPfRows + r];
      const float M = fmaxf(ma, mb);
      const float fa = (n0 == 0 || ma == -INFINITY) ? 0.f : ex2(ma - M);
      const float fb = (n1 == 0 || mb == -INFINITY) ? 0.f : ex2(mb - M);
      const float L = l_sh[r] * fa + l_sh[kPfRows + r] * fb;
      const float ofac = L > 0.f ? 1.f / L : 0.f;
      // each group's O holds P' = p * v_scale * 2^-kp of its own row exponent
      const float fa_o = fa * pow2i(kp_sh[r]), fb_o = fb * pow2i(kp_sh[kPfRows + r]);
      const int64_t ob0 = (((int64_t)b * p.n_q + (qi < p.n_q ? qi : 0)) * p.q_heads + hq) * D + 64 * wg;
#pragma unroll 1
      for (int k = 4 * wg; k < 4 * wg + 4; ++k) {   // 16 head dims per chunk
        uint32_t r0[16], r1[16];
        if (n0 > 0) umma::tmem_ld16_nowait(tmem + 256 + 16 * k + lane_off, r0);
        if (n1 > 0) umma::tmem_ld16_nowait(tmem + 384 + 16 * k + lane_off, r1);
        umma::tmem_wait_ld();
        float o[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float x = 0.f;
          if (n0 > 0 && fa != 0.f) x += __uint_as_float(r0[u]) * fa_o;
          if (n1 > 0 && fb != 0.f) x += __uint_as_float(r1[u]) * fb_o;
          o[u] = x * ofac;
        }
        const int64_t oi = ob0 + 16 * (k - 4 * wg);
        if (qi >= p.n_q) continue;                  // (the TMEM loads above are warp-wide)
        if ((reinterpret_cast<uintptr_t>(p.out) & 15) != 0) {   // caller's buffer not 16-byte aligned
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            if (p.out_f32) reinterpret_cast<float*>(p.out)[oi + u] = o[u];
            else reinterpret_cast<__nv_bfloat16*>(p.out)[oi + u] = __float2bfloat16_rn(o[u]);
          }
        } else if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + oi);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
        } else {
          uint32_t w8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[2 * u], o[2 * u + 1]);
            w8[u] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + oi);
          dst[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
          dst[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
        }
      }
    }
    if (any_fail && r == 0 && wg == 0) raise_error(p.err, FP8KV_DEVERR_TIMEOUT);
  } else if (warp >= 10 && warp < 14) {
    // --------------------------------------------------------- preparation
    // Warp 10 + w prepares tiles j = w, w + 4, ... (f16 operand buffer w):
    // four tiles in flight, no barrier between the warps.  The tile's V codes
    // and scales are read into registers first: the column scales go out at
    // once (the softmax waits only for them) and the ring slot is released
    // (the next K tile's load waits only for that); the f16 operand is then
    // written once the buffer's previous P.V has finished.  Column-scale
    // buffer j % 8 is rewritten for tile j + 8 only after this warp saw the
    // P.V of tile j finish (its wait for tile j + 4's buffer), so the softmax
    // of tile j has read it by then.
    static_assert(C::NOP == 4, "one operand buffer per preparation warp");
    const int pw = warp - 10;
    bool failed = false;
    for (int j = pw; j < nkv && !failed; j += 4) {
      const int s = j % C::NS, u = j / C::NS, ob = j % C::NOP, ou = j / C::NOP, cb = j % C::NCOL;
      bool ok = wait_fast(&full[s], u & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      const uint8_t* st = ring + s * C::STAGE;
      const uint8_t* codes = st + C::CODES;
      const float* kss = reinterpret_cast<const float*>(st + 2 * C::CODES);
      const float* vss = kss + kPfKeys;
      const int t0 = j * kPfKeys;
      // 64 key rows x 8 chunks of 16 codes: lane takes chunk ch = lane & 7 of
      // rows 4 it + lane / 8
      uint4 w[16];
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int kr = 4 * it + (lane >> 3), ch = lane & 7;
        w[it] = *reinterpret_cast<const uint4*>(codes + kr * 128 + ((ch ^ (kr & 7)) << 4));
      }
      {
        const float k0 = kss[lane], k1 = kss[lane + 32], v0 = vss[lane], v1 = vss[lane + 32];
        float* cc2 = cols + cb * C::CST;
        const bool ok0 = t0 + lane < kv_end, ok1 = t0 + lane + 32 < kv_end;
        const float va = ok0 ? v0 : 0.f, vb = ok1 ? v1 : 0.f;
        cc2[lane] = ok0 ? k0 * p.scale_log2 : 0.f;
        cc2[lane + 32] = ok1 ? k1 * p.scale_log2 : 0.f;
        cc2[kPfKeys + lane] = va;
        cc2[kPfKeys + lane + 32] = vb;
        const float vm = warp_max(fmaxf(va, vb));
        if (lane == 0) cc2[2 * kPfKeys] = vm;     // the tile's largest V scale
      }
      __syncwarp();
      if (lane == 0) {
        umma::mbar_arrive(&cols_full[cb]);
        umma::mbar_arrive(&empty[s]);
      }
      if (ou > 0) {
        ok = wait_fast(&op_free[ob], (ou - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      }
      uint8_t* dstb = vf + ob * C::OPT;
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int kr = 4 * it + (lane >> 3), ch = lane & 7;
        const bool key_ok = t0 + kr < kv_end;
        uint32_t h[8];
        const uint32_t ww[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          h[2 * u4] = key_ok ? e4m3x2_to_f16x2((uint16_t)(ww[u4] & 0xFFFF)) : 0u;
          h[2 * u4 + 1] = key_ok ? e4m3x2_to_f16x2((uint16_t)(ww[u4] >> 16)) : 0u;
        }
        // dims 16 ch .. 16 ch + 15: atom ch / 4, f16 chunks 2 (ch % 4) and +1
        uint8_t* dst = dstb + (ch >> 2) * (kPfKeys * 128) + kr * 128;
        const int c0 = 2 * (ch & 3), c1 = c0 + 1;
        *reinterpret_cast<uint4*>(dst + ((c0 ^ (kr & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + ((c1 ^ (kr & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      umma::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        PF_TRACE(8 * j + 3);
        umma::mbar_arrive(&op_full[ob]);
      }
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (warp == 1) umma::tmem_dealloc(tmem, 512);
  if (tid == 0) PF_TRACE(1021);
#ifdef FP8KV_TRACE
  if (tid == 0) PF_CTA(2, umma::globaltimer_ns());
#endif
}

#ifdef FP8KV_TRACE
extern "C" __attribute__((visibility("default"))) int fp8kv_trace_clear_prefill() {
  static unsigned long long zero[1024];
  return cudaMemcpyToSymbol(g_pf_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int fp8kv_trace_read_prefill(unsigned long long* out, int n) {
  if (n > 1024) n = 1024;
  return cudaMemcpyFromSymbol(out, g_pf_trace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int fp8kv_trace_read_prefill_cta(unsigned long long* out, int n) {
  if (n > 2048) n = 2048;
  return cudaMemcpyFromSymbol(out, g_pf_cta, n * 4 * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_prefill_tc(const PrefillParams& p, int batch, cudaStream_t st) {
  constexpr int smem = PfTcCfg::BYTES;
  cudaError_t e = ensure_smem_optin((const void*)prefill_tc, smem);
  if (e != cudaSuccess) return e;
  PrefillTmaParams tp;
  const CacheView& c = p.c;
  const int64_t rows = c.paged ? (int64_t)c.num_pages * c.kv_heads * c.page_size
                               : (int64_t)c.batch * c.kv_heads * c.max_tokens;
  const int box_rows = c.paged ? c.page_size : kPfKeys;
  if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (!make_map(&tp.tmk, c.k, false, rows, box_rows) || !make_map(&tp.tmv, c.v, false, rows, box_rows))
    return cudaErrorInvalidValue;
  tp.p = p;
  const int n_qt = (p.n_q + kPfRows - 1) / kPfRows;
  if (n_qt > 65535) return cudaErrorInvalidValue;
  dim3 grid(p.q_heads, batch, n_qt);
  prefill_tc<<<grid, kPfThreads, smem, st>>>(tp);
  return cudaGetLastError();
}

}  // namespace fp8kv
