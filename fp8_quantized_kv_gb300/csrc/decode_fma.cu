// decode_fma.cu -- flash-decoding split kernel on the CUDA cores, plus the
// merge kernel shared by every decode path.
//
// What is computed ("FP8 KV cache (fp8_kv, opt-in)", bullets "Math" and
// "Speed"): for each sequence b and query head h (KV head h/G), attention of
// one bf16 query over the cached tokens 0..T_b-1.  The cache is split over
// CTAs (flash-decoding); each CTA walks its 64-token tiles with an online
// softmax and writes fp32 partials (O, m, l); a second kernel merges them.
//
// Per tile ("FP8 KV attention: hardware paths and tile preparation", section
// "Operating model": K load -> K prep -> QK -> softmax; V load -> V prep -> PV):
//   s_j   = (q . kcode_j) * k_scale_j * sm_scale          (K scale folded into s;
//           MXFP8 keys: each 32-dim block's partial dot times its E8M0 scale;
//           rotated-bias residual keys: plus q . R_t b, the key's rotated
//           bias, as sum_i A_i cos theta_{t,i} + B_i sin theta_{t,i} with
//           A_i = q_i b_i + q_{i+D/2} b_{i+D/2}, B_i = q_{i+D/2} b_i - q_i b_{i+D/2})
//   m_t   = max_j s_j over the tile,   p_j = exp(s_j - m_t)
//   p'_j  = bf16_rn(p_j * v_scale_j)                        (V scale folded into P)
//   O     = O * e^(m - m') + e^(m_t - m') * sum_j p'_j vcode_j,   l likewise with p_j
// P is referenced to its own tile's maximum before the bf16 rounding, so a
// tile contributes the same rounded P whichever split it falls in; split
// boundaries are multiples of 64 tokens anchored at token 0.  Different split
// counts then differ only by fp32 re-association.
//
// Exponentials are base 2 with log2(e) folded into the score scale.
//
// Thread mapping (128 threads, 4 warps, G <= GP query heads of one KV head):
//   QK: thread -> (token j = tid/2, half of head_dim); Q lives in shared
//       memory as fp32 and is read by broadcast; the two halves combine with
//       one shuffle.
//   PV: lane -> head_dim/32 consecutive dims, warp -> every 4th token; each
//       warp keeps a partial O for its tokens, summed once per split.
// Loads: every tile (K codes, V codes, both scale rows) is staged into a
// 3-deep shared-memory ring by 16-byte cp.async copies issued two tiles ahead.
// Shared-memory rows are chunk-swizzled (swz_chunk) so the QK row reads are
// conflict-free.
#include "params.cuh"

namespace fp8kv {

template <int D, int KE, int VE>
struct FmaCfg {
  static constexpr int KB = KE == ELEM_BF16 ? 2 : 1;
  static constexpr int VB = VE == ELEM_E4M3 ? 1 : 2;
  static constexpr int K_ROW = D * KB, V_ROW = D * VB;     // bytes per row
  static constexpr int K_CPR = K_ROW / 16, V_CPR = V_ROW / 16;
  static constexpr int K_TILE = kTileTokens * K_ROW, V_TILE = kTileTokens * V_ROW;
  static constexpr int STAGE = K_TILE + V_TILE + 2 * kTileTokens * 4;
  static constexpr int NSTAGE = 3;
  static constexpr int QS = D + 8;          // q row stride (floats); half 1 shifted by 4
  static constexpr int EPL = D / 32;        // PV dims per lane
};

template <int D, int GP, int KE, int VE>
constexpr int fma_smem_bytes() {
  using C = FmaCfg<D, KE, VE>;
  return C::NSTAGE * C::STAGE + GP * C::QS * 4 + kTileTokens * GP * 4 + 2 * 4 * GP * 4;
}
// rotated-bias residual keys: the per-head A and B of the score term, after the rest
template <int D, int GP>
constexpr int fma_rope_smem_bytes() { return GP * D * 4; }

__device__ __forceinline__ int q_off(int d, int D) { return d + (d >= D / 2 ? 4 : 0); }

// RP: the instantiation for caches with rotated-bias residual keys (rotary
// tables set); the others carry none of its code or registers.
template <int D, int GP, int KE, int VE, bool RP>
__global__ void __launch_bounds__(128) decode_split_fma(DecodeParams p) {
  using C = FmaCfg<D, KE, VE>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem + C::NSTAGE * C::STAGE);
  float* p_s = q_s + GP * C::QS;                 // [64][GP]
  float* red_max = p_s + kTileTokens * GP;        // [4][GP]
  float* red_sum = red_max + 4 * GP;              // [4][GP]
  float* ab_s = red_sum + 4 * GP;                 // [GP][D]: A_i (i < D/2), B_i (rotated bias only)

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
  const int tiles = (T + kTileTokens - 1) / kTileTokens;
  const int t_begin = s * p.chunk_tiles;
  const int t_end = min(t_begin + p.chunk_tiles, tiles);
  const int64_t part0 = ((int64_t)b * p.q_heads + (int64_t)h * G) * S + s;   // + g*S

  if (t_begin >= t_end) {   // nothing of this sequence falls in this split
    for (int i = tid; i < G * D; i += blockDim.x)
      p.part_o[(part0 + (int64_t)(i / D) * S) * D + (i % D)] = 0.f;
    if (tid < G) {
      p.part_m[part0 + (int64_t)tid * S] = -INFINITY;
      p.part_l[part0 + (int64_t)tid * S] = 0.f;
    }
    return;
  }

  // ---- Q (bf16 -> fp32) into shared memory, heads >= G zeroed
  for (int i = tid; i < GP * D; i += blockDim.x) {
    const int g = i / D, d = i % D;
    float v = 0.f;
    if (g < G) v = __bfloat162float(p.q[((int64_t)b * p.q_heads + (int64_t)h * G + g) * D + d]);
    q_s[g * C::QS + q_off(d, D)] = v;
  }

  constexpr bool rope = RP;
  constexpr int H = D / 2;
  if constexpr (rope) {
    __syncthreads();                               // q_s written
    const float* kb = c.k_bias + (int64_t)h * D;
    for (int i = tid; i < GP * H; i += blockDim.x) {
      const int g = i / H, pi = i % H;
      const float q0 = q_s[g * C::QS + q_off(pi, D)], q1 = q_s[g * C::QS + q_off(pi + H, D)];
      const float b0 = kb[pi], b1 = kb[pi + H];
      ab_s[g * D + pi] = fmaf(q0, b0, q1 * b1);
      ab_s[g * D + H + pi] = fmaf(q1, b0, -(q0 * b1));
    }
  }
  const int64_t cont_base = ((int64_t)b * c.kv_heads + h) * c.max_tokens;   // contiguous rows
  // Issue the cp.async copies of one tile into a ring stage.  Rows up to the
  // next multiple of 16 past T are copied (still inside the cache capacity or
  // the page); rows past T are masked in the math.
  auto issue = [&](int tile, int stage) {
    uint8_t* st = smem + stage * C::STAGE;
    uint8_t* ks = st;
    uint8_t* vs = st + C::K_TILE;
    float* kss = reinterpret_cast<float*>(st + C::K_TILE + C::V_TILE);
    float* vss = kss + kTileTokens;
    const int t0 = tile * kTileTokens;
    const int nrows = min(kTileTokens, ((T - t0) + 15) & ~15);
    auto row_of = [&](int r) -> int64_t {     // cache row index of tile row r
      const int t = t0 + r;
      if (!c.paged) return cont_base + t;
      const int page = c.page_table[(int64_t)b * c.max_pages_per_seq + (t >> c.page_shift)];
      if (page < 0 || page >= c.num_pages) { raise_error(p.err, FP8KV_DEVERR_BAD_PAGE); return -1; }
      return ((int64_t)page * c.kv_heads + h) * c.page_size + (t & (c.page_size - 1));
    };
    for (int i = tid; i < nrows * C::K_CPR; i += blockDim.x) {
      const int r = i / C::K_CPR, ch = i % C::K_CPR;
      const int64_t row = row_of(r);
      if (row >= 0) cp_async16(ks + r * C::K_ROW + swz_chunk(ch, r, C::K_CPR) * 16,
                               c.k + row * C::K_ROW + ch * 16);
    }
    for (int i = tid; i < nrows * C::V_CPR; i += blockDim.x) {
      const int r = i / C::V_CPR, ch = i % C::V_CPR;
      const int64_t row = row_of(r);
      if (row >= 0) cp_async16(vs + r * C::V_ROW + swz_chunk(ch, r, C::V_CPR) * 16,
                               c.v + row * C::V_ROW + ch * 16);
    }
    // scales: 4 consecutive rows per 16-byte copy (pages hold >= 16 rows)
    const int nsc = nrows / 4;
    for (int i = tid; i < 2 * nsc; i += blockDim.x) {
      const bool is_v = i >= nsc;
      const int r = (is_v ? i - nsc : i) * 4;
      const float* src = is_v ? c.v_scale : c.k_scale;
      if (src == nullptr) continue;
      const int64_t row = row_of(r);
      if (row >= 0) cp_async16((is_v ? vss : kss) + r, src + row);
    }
  };

  const int n_tiles = t_end - t_begin;
#pragma unroll 1
  for (int i = 0; i < C::NSTAGE - 1; ++i) {
    if (i < n_tiles) issue(t_begin + i, i);
    cp_async_commit();
  }

  float m_run[GP], l_run[GP], acc[GP][C::EPL];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.f;
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) acc[g][e] = 0.f;
  }

  const int j = tid >> 1, hf = tid & 1;

#pragma unroll 1
  for (int it = 0; it < n_tiles; ++it) {
    {
      const int nt = it + C::NSTAGE - 1;
      if (nt < n_tiles) issue(t_begin + nt, nt % C::NSTAGE);
      cp_async_commit();
    }
    cp_async_wait<C::NSTAGE - 1>();
    __syncthreads();

    const uint8_t* st = smem + (it % C::NSTAGE) * C::STAGE;
    const uint8_t* ks = st;
    const uint8_t* vs = st + C::K_TILE;
    const float* kss = reinterpret_cast<const float*>(st + C::K_TILE + C::V_TILE);
    const float* vss = kss + kTileTokens;
    const int t0 = (t_begin + it) * kTileTokens;
    const int nvalid = min(kTileTokens, T - t0);

    // ---- QK on the CUDA cores: thread (j, hf) covers half of token j's row
    float dot[GP];
    constexpr int HCH = C::K_CPR / 2;                    // 16-byte chunks per half row
    constexpr int NBL = KE == ELEM_MX ? HCH / 2 : 1;     // MXFP8: 32-dim blocks per half row
    float dotb[GP][NBL];
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int lb = 0; lb < NBL; ++lb) dotb[g][lb] = 0.f;
    {
      const uint8_t* krow = ks + j * C::K_ROW;
#pragma unroll
      for (int cc = 0; cc < HCH; ++cc) {
        const int ch = hf * HCH + cc;
        const uint4 w = *reinterpret_cast<const uint4*>(krow + swz_chunk(ch, j, C::K_CPR) * 16);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        constexpr int EPW = KE == ELEM_BF16 ? 2 : 4;      // elements per 32-bit word
        const int lb = KE == ELEM_MX ? cc >> 1 : 0;       // two chunks per MXFP8 block
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          float f[4];
          if constexpr (KE != ELEM_BF16) {
            e4m3x4_to_f32_scaled(wv[wi], f);
          } else {
            float f2[2];
            bf16x2_to_f32(wv[wi], f2);
            f[0] = f2[0]; f[1] = f2[1]; f[2] = 0.f; f[3] = 0.f;
          }
          const int d0 = ch * (16 / C::KB) + wi * EPW;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float* qg = q_s + g * C::QS + q_off(d0, D);
            float& dg = dotb[g][lb];
            if constexpr (EPW == 4) {
              const float4 qv = *reinterpret_cast<const float4*>(qg);
              dg = fmaf(qv.x, f[0], dg);
              dg = fmaf(qv.y, f[1], dg);
              dg = fmaf(qv.z, f[2], dg);
              dg = fmaf(qv.w, f[3], dg);
            } else {
              const float2 qv = *reinterpret_cast<const float2*>(qg);
              dg = fmaf(qv.x, f[0], dg);
              dg = fmaf(qv.y, f[1], dg);
            }
          }
        }
      }
    }
    if constexpr (KE == ELEM_MX) {
      // the row's E8M0 bytes (block k in byte k): this half's blocks weighted
      const uint32_t e8 = reinterpret_cast<const uint32_t*>(kss)[j];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float d = 0.f;
#pragma unroll
        for (int lb = 0; lb < NBL; ++lb)
          d = fmaf(dotb[g][lb], pow2_exact((int)((e8 >> (8 * (hf * NBL + lb))) & 0xFF) - 127), d);
        dot[g] = d;
      }
    } else {
#pragma unroll
      for (int g = 0; g < GP; ++g) dot[g] = dotb[g][0];
    }
    const bool valid = j < nvalid;
    const float kfac = (KE == ELEM_E4M3 ? kss[j] : 1.f) * p.scale_log2;
    // rotated-bias residual keys: this thread's half of the pairs of q . R_t b
    float corr[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) corr[g] = 0.f;
    if (rope && valid) {
      const int t = t0 + j;
      const float4* cs4 = reinterpret_cast<const float4*>(c.rope_cos + (int64_t)t * H + hf * (H / 2));
      const float4* sn4 = reinterpret_cast<const float4*>(c.rope_sin + (int64_t)t * H + hf * (H / 2));
#pragma unroll 2
      for (int u = 0; u < H / 8; ++u) {
        const float4 cv = __ldg(cs4 + u), sv = __ldg(sn4 + u);
        const int pi = hf * (H / 2) + 4 * u;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float4 a = *reinterpret_cast<const float4*>(ab_s + g * D + pi);
          const float4 bq = *reinterpret_cast<const float4*>(ab_s + g * D + H + pi);
          float x = corr[g];
          x = fmaf(a.x, cv.x, x); x = fmaf(bq.x, sv.x, x);
          x = fmaf(a.y, cv.y, x); x = fmaf(bq.y, sv.y, x);
          x = fmaf(a.z, cv.z, x); x = fmaf(bq.z, sv.z, x);
          x = fmaf(a.w, cv.w, x); x = fmaf(bq.w, sv.w, x);
          corr[g] = x;
        }
      }
    }
    float sc[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      float d2 = dot[g] + __shfl_xor_sync(0xffffffffu, dot[g], 1);
      if (KE != ELEM_BF16) d2 *= kTwoPow120;
      if constexpr (rope) {
        const float ct = corr[g] + __shfl_xor_sync(0xffffffffu, corr[g], 1);
        sc[g] = valid ? fmaf(d2, KE == ELEM_E4M3 ? kss[j] : 1.f, ct) * p.scale_log2 : -INFINITY;
      } else {
        sc[g] = valid ? d2 * kfac : -INFINITY;
      }
      const float wm = warp_max(sc[g]);
      if (lane == 0) red_max[warp * GP + g] = wm;
    }
    __syncthreads();

    // ---- tile max, P (bf16, V scale folded), tile sums
    float alpha[GP], beta[GP];
    const float vsc = VE == ELEM_E4M3 ? vss[j] : 1.f;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float mt = fmaxf(fmaxf(red_max[g], red_max[GP + g]), fmaxf(red_max[2 * GP + g], red_max[3 * GP + g]));
      const float mn = fmaxf(m_run[g], mt);                 // finite: tile has >= 1 valid token
      alpha[g] = exp2f(m_run[g] - mn);                      // 0 on the first tile
      beta[g] = exp2f(mt - mn);
      const float pj = exp2f(sc[g] - mt);                   // 0 for masked tokens
      const float pv = bf16_round(pj * vsc) * beta[g];
      if ((g & 1) == hf) p_s[j * GP + g] = pv;
      const float ws = warp_sum(hf == 0 ? pj : 0.f);
      if (lane == 0) red_sum[warp * GP + g] = ws;
      m_run[g] = mn;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float lt = (red_sum[g] + red_sum[GP + g]) + (red_sum[2 * GP + g] + red_sum[3 * GP + g]);
      l_run[g] = l_run[g] * alpha[g] + lt * beta[g];
#pragma unroll
      for (int e = 0; e < C::EPL; ++e) acc[g][e] *= alpha[g];
    }

    // ---- PV on the CUDA cores: lane owns EPL dims, warp every 4th token
#pragma unroll 4
    for (int jj = warp; jj < nvalid; jj += 4) {
      const uint8_t* vrow = vs + jj * C::V_ROW;
      float f[C::EPL];
      constexpr int LB = C::EPL * C::VB;                   // bytes per lane
      const int off = lane * LB;
      const uint8_t* src = vrow + swz_chunk(off >> 4, jj, C::V_CPR) * 16 + (off & 15);
      if constexpr (VE == ELEM_E4M3) {
        float t4[4];
        if constexpr (C::EPL == 4)
          e4m3x4_to_f32_scaled(*reinterpret_cast<const uint32_t*>(src), t4);
        else
          e4m3x4_to_f32_scaled((uint32_t)*reinterpret_cast<const uint16_t*>(src), t4);
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) f[e] = t4[e];
      } else if constexpr (C::EPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        float a[2], bb[2];
        bf16x2_to_f32(u.x, a);
        bf16x2_to_f32(u.y, bb);
        f[0] = a[0]; f[1] = a[1]; f[2] = bb[0]; f[3] = bb[1];
      } else {
        float a[2];
        bf16x2_to_f32(*reinterpret_cast<const uint32_t*>(src), a);
        f[0] = a[0]; f[1] = a[1];
      }
      const float* prow = p_s + jj * GP;
#pragma unroll
      for (int g4 = 0; g4 < GP; g4 += 4) {
        float pv[4];
        if constexpr (GP >= 4) {
          const float4 t = *reinterpret_cast<const float4*>(prow + g4);
          pv[0] = t.x; pv[1] = t.y; pv[2] = t.z; pv[3] = t.w;
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) pv[u] = u < GP ? prow[u] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4 && g4 + u < GP; ++u)
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) acc[g4 + u][e] = fmaf(pv[u], f[e], acc[g4 + u][e]);
      }
    }
    __syncthreads();   // the stage and p_s are rewritten next iteration
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- combine the four warps' partial O and write the split's partials
  float* o_red = reinterpret_cast<float*>(smem);   // [4][GP][D], aliases the ring
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) o_red[(warp * GP + g) * D + lane * C::EPL + e] = acc[g][e];
  __syncthreads();
  const float ofac = VE == ELEM_E4M3 ? kTwoPow120 : 1.f;
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int g = i / D, d = i % D;
    const float o = (o_red[(0 * GP + g) * D + d] + o_red[(1 * GP + g) * D + d]) +
                    (o_red[(2 * GP + g) * D + d] + o_red[(3 * GP + g) * D + d]);
    p.part_o[(part0 + (int64_t)g * S) * D + d] = o * ofac;
  }
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < GP; ++g)
      if (g < G) {
        p.part_m[part0 + (int64_t)g * S] = m_run[g];
        p.part_l[part0 + (int64_t)g * S] = l_run[g];
      }
  }
}

// ------------------------------------------------------------------ merge --
// out[b,h] = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, M = max_s m_s;
// a row with no valid split (length 0) is written as zeros.  One CTA per
// (sequence, query head): warp 0 turns the split maxima into weights in
// shared memory, then every thread sums its dim over the splits with
// independent loads.
constexpr int kMergeMaxS = 1024;

template <int D>
__global__ void __launch_bounds__(D) decode_merge(const float* __restrict__ part_o,
                                                  const float* __restrict__ part_m,
                                                  const float* __restrict__ part_l, int S, void* out,
                                                  int out_f32) {
  __shared__ float wsh[kMergeMaxS];
  __shared__ float inv_sh;
  const int64_t bh = blockIdx.x;
  const int d = threadIdx.x;
  const float* pm = part_m + bh * S;
  const float* pl = part_l + bh * S;
  const int Sw = min(S, kMergeMaxS);
  if (d < 32) {
    float M = -INFINITY;
    for (int s = d; s < S; s += 32) M = fmaxf(M, pm[s]);
    M = warp_max(M);
    float L = 0.f;
    for (int s = d; s < S; s += 32) {
      const float ms = pm[s];
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      if (s < Sw) wsh[s] = w;
      L = fmaf(w, pl[s], L);
    }
    L = warp_sum(L);
    if (d == 0) inv_sh = L > 0.f ? 1.0f / L : 0.f;
  }
  __syncthreads();
  const float* po = part_o + bh * S * D + d;
  // loads of 8 splits issued together per round
  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  for (int s0 = 0; s0 < Sw; s0 += 8) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = s0 + k < Sw ? po[(int64_t)(s0 + k) * D] : 0.f;
#pragma unroll
    for (int k = 0; k < 8; k += 4) {
      if (s0 + k < Sw) o0 = fmaf(wsh[s0 + k], v[k], o0);
      if (s0 + k + 1 < Sw) o1 = fmaf(wsh[s0 + k + 1], v[k + 1], o1);
      if (s0 + k + 2 < Sw) o2 = fmaf(wsh[s0 + k + 2], v[k + 2], o2);
      if (s0 + k + 3 < Sw) o3 = fmaf(wsh[s0 + k + 3], v[k + 3], o3);
    }
  }
  if (S > kMergeMaxS) {      // rare: more splits than the weight table holds
    float M = -INFINITY;
    for (int k = 0; k < S; ++k) M = fmaxf(M, pm[k]);
    for (int k = kMergeMaxS; k < S; ++k) {
      const float ms = pm[k];
      if (ms != -INFINITY) o1 = fmaf(exp2f(ms - M), po[(int64_t)k * D], o1);
    }
  }
  const float r = ((o0 + o1) + (o2 + o3)) * inv_sh;
  if (out_f32)
    reinterpret_cast<float*>(out)[bh * D + d] = r;
  else
    reinterpret_cast<__nv_bfloat16*>(out)[bh * D + d] = __float2bfloat16_rn(r);
}

// ------------------------------------------------------------ launchers ---
template <int D, int GP, int KE, int VE, bool RP>
static cudaError_t launch_fma_r(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = fma_smem_bytes<D, GP, KE, VE>() + (RP ? fma_rope_smem_bytes<D, GP>() : 0);
  cudaError_t e = ensure_smem_optin((const void*)decode_split_fma<D, GP, KE, VE, RP>, smem);
  if (e != cudaSuccess) return e;
  decode_split_fma<D, GP, KE, VE, RP><<<grid, 128, smem, st>>>(p);
  return cudaGetLastError();
}

template <int D, int GP, int KE, int VE>
static cudaError_t launch_fma_t(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  if (p.c.rope_cos == nullptr) return launch_fma_r<D, GP, KE, VE, false>(p, grid, st);
  // (rotary tables come only with a key bias, on e4m3 per-row keys)
  if constexpr (KE == ELEM_E4M3) return launch_fma_r<D, GP, KE, VE, true>(p, grid, st);
  return cudaErrorInvalidValue;
}

template <int D, int KE, int VE>
static cudaError_t launch_fma_g(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  const int G = p.group;
  if (G <= 1) return launch_fma_t<D, 1, KE, VE>(p, grid, st);
  if (G <= 2) return launch_fma_t<D, 2, KE, VE>(p, grid, st);
  if (G <= 4) return launch_fma_t<D, 4, KE, VE>(p, grid, st);
  return launch_fma_t<D, 8, KE, VE>(p, grid, st);
}

template <int D>
static cudaError_t launch_fma_d(const DecodeParams& p, int dtype, dim3 grid, cudaStream_t st) {
  if constexpr (D == 128)     // (MXFP8 keys are built for head_dim 128)
    if (dtype == FP8KV_MXK8V8) return launch_fma_g<D, ELEM_MX, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K8V8) return launch_fma_g<D, ELEM_E4M3, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K16V8) return launch_fma_g<D, ELEM_BF16, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K8V16) return launch_fma_g<D, ELEM_E4M3, ELEM_BF16>(p, grid, st);
  return launch_fma_g<D, ELEM_BF16, ELEM_BF16>(p, grid, st);
}

cudaError_t launch_decode_fma(const DecodeParams& p, int dtype, int batch, cudaStream_t st) {
  dim3 grid(p.num_splits, p.c.kv_heads, batch);
  return p.c.head_dim == 128 ? launch_fma_d<128>(p, dtype, grid, st)
                             : launch_fma_d<64>(p, dtype, grid, st);
}

cudaError_t launch_decode_merge(const float* part_o, const float* part_m, const float* part_l, int S,
                                int64_t rows, int head_dim, void* out, int out_f32, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (head_dim == 128)
    decode_merge<128><<<(unsigned)rows, 128, 0, st>>>(part_o, part_m, part_l, S, out, out_f32);
  else
    decode_merge<64><<<(unsigned)rows, 64, 0, st>>>(part_o, part_m, part_l, S, out, out_f32);
  return cudaGetLastError();
}

}  // namespace fp8kv
