// prefill_fma.cu -- causal prefill attention over the FP8 cache on the CUDA
// cores: the simple tiled kernel that the tensor-core kernel is checked and
// timed against, and the path for shapes the tensor-core kernel does not take.
//
// "03 · 8n — FA-style tiled prefill attention", sections 2.1 and 3.1: one CTA
// per (64-query tile, query head), KV consumed in 64-token tiles up to the
// causal limit of the tile's last query, online softmax with running max m,
// sum l and an fp32 O held in registers; a key j is valid for query position
// qp iff j <= qp; a tile with no valid key leaves the state unchanged.  The
// FP8 numerics are those of "FP8 KV cache (fp8_kv, opt-in)", bullet "Math":
// K scale folded into the scores, V scale into P, P rounded to bf16, P
// referenced to the tile's own row maximum (the same convention as decode).
//
// 256 threads: thread t owns query row r = t/4 and a quarter (t%4) of the
// tile's columns for QK and softmax, and the dims d = (t%4) + 4i for PV.
// K and V codes are converted on the fly into fp32 shared-memory tiles (code
// values, the per-token scales applied as above; MXFP8 keys with their block
// scales applied at the conversion; rotated-bias residual keys reconstructed
// there in full, dequant(r) + R_t b).
#include "params.cuh"

namespace fp8kv {

template <int D>
struct PfCfg {
  static constexpr int QS = D + 1;          // fp32 row strides (padded)
  static constexpr int KS = D + 1;
  static constexpr int VS = D;
  static constexpr int SS = kTileTokens + 1;
  static constexpr int BYTES = 4 * (kTileTokens * QS + kTileTokens * KS + kTileTokens * VS +
                                    kTileTokens * SS + 2 * kTileTokens);
};

template <int D, int KE, int VE>
__global__ void __launch_bounds__(256) prefill_fma(PrefillParams p) {
  using C = PfCfg<D>;
  extern __shared__ __align__(16) float fsm[];
  float* Qs = fsm;                              // [64][QS] q (fp32)
  float* Ks = Qs + kTileTokens * C::QS;         // [64][KS] K code values (x 2^-120 for e4m3)
  float* Vs = Ks + kTileTokens * C::KS;         // [64][VS] V code values (x 2^-120 for e4m3)
  float* Ps = Vs + kTileTokens * C::VS;         // [64][SS] P' per (row, key)
  float* kss = Ps + kTileTokens * C::SS;        // [64] K scales
  float* vss = kss + kTileTokens;               // [64] V scales

  const int qt = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int r = tid >> 2, qd = tid & 3;
  const int hk = hq / p.group;
  const CacheView& c = p.c;
  const bool rope = c.rope_cos != nullptr;       // rotated-bias residual keys
  const int pos0 = p.q_pos0[b];
  const int i0 = qt * kTileTokens;
  const int last_i = min(p.n_q, i0 + kTileTokens) - 1;
  const int kv_end = pos0 + last_i + 1;           // keys 0..kv_end-1 may be needed
  if (pos0 < 0 || kv_end > cache_capacity(c)) {
    if (tid == 0) raise_error(p.err, FP8KV_DEVERR_SEQ_TOO_LONG);
    return;
  }

  for (int i = tid; i < kTileTokens * D; i += 256) {
    const int rr = i / D, d = i % D;
    const int qi = i0 + rr;
    Qs[rr * C::QS + d] = qi < p.n_q
        ? __bfloat162float(p.q[(((int64_t)b * p.n_q + qi) * p.q_heads + hq) * D + d]) : 0.f;
  }
  const int qi = i0 + r;
  const int qpos = qi < p.n_q ? pos0 + qi : -1;    // rows past n_q see no key

  float acc[D / 4];
#pragma unroll
  for (int e = 0; e < D / 4; ++e) acc[e] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  const int n_tiles = (kv_end + kTileTokens - 1) / kTileTokens;
#pragma unroll 1
  for (int kt = 0; kt < n_tiles; ++kt) {
    const int t0 = kt * kTileTokens;
    const int nrows = min(kTileTokens, kv_end - t0);
    __syncthreads();     // previous tile fully consumed
    for (int i = tid; i < kTileTokens * D; i += 256) {
      const int rr = i / D, d = i % D;
      float kvv = 0.f, vvv = 0.f;
      if (rr < nrows) {
        const int64_t row = cache_row(c, b, hk, t0 + rr, p.err);
        if (row >= 0) {
          if constexpr (KE == ELEM_E4M3) {
            float f[4];
            e4m3x4_to_f32_scaled((uint32_t)c.k[row * D + d], f);
            kvv = f[0];
            if (rope)     // rotated-bias residual key: dequant(r) + R_t b, in full
              kvv = fmaf(f[0] * kTwoPow120, c.k_scale[row], rope_bias(c, hk, t0 + rr, d));
          } else if constexpr (KE == ELEM_MX) {
            // MXFP8 key: the code's value times its 32-dim block's E8M0
            // scale (byte d / 32 of the row's scale word), exact in fp32
            float f[4];
            e4m3x4_to_f32_scaled((uint32_t)c.k[row * D + d], f);
            const uint32_t e8 = reinterpret_cast<const uint32_t*>(c.k_scale)[row];
            kvv = (f[0] * kTwoPow120) * pow2_exact((int)((e8 >> (8 * (d >> 5))) & 0xFF) - 127);
          } else {
            kvv = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(c.k)[row * D + d]);
          }
          if constexpr (VE == ELEM_E4M3) {
            float f[4];
            e4m3x4_to_f32_scaled((uint32_t)c.v[row * D + d], f);
            vvv = f[0];
          } else {
            vvv = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(c.v)[row * D + d]);
          }
          if (d == 0) {
            kss[rr] = KE == ELEM_E4M3 && !rope ? c.k_scale[row] : 1.f;
            vss[rr] = VE == ELEM_E4M3 ? c.v_scale[row] : 1.f;
          }
        }
      }
      Ks[rr * C::KS + d] = kvv;
      Vs[rr * C::VS + d] = vvv;
    }
    __syncthreads();

    // QK: thread (r, qd) computes columns qd + 4u, u = 0..15
    float s[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) s[u] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      const float qv = Qs[r * C::QS + d];
#pragma unroll
      for (int u = 0; u < 16; ++u) s[u] = fmaf(qv, Ks[(qd + 4 * u) * C::KS + d], s[u]);
    }
    float mt = -INFINITY;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int col = qd + 4 * u;
      const int key = t0 + col;
      const bool ok = col < nrows && key <= qpos;
      float v = s[u];
      if (KE == ELEM_E4M3 && !rope) v *= kTwoPow120;
      s[u] = ok ? v * (kss[col] * p.scale_log2) : -INFINITY;
      mt = fmaxf(mt, s[u]);
    }
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    // A row with no valid key in this tile (mt = -inf) keeps its state and
    // writes zero probabilities.  The shuffles stay outside any branch.
    const bool any = mt != -INFINITY;
    const float mn = any ? fmaxf(m_run, mt) : m_run;
    const float alpha = any ? exp2f(m_run - mn) : 1.f;
    const float beta = any ? exp2f(mt - mn) : 0.f;
    float lt = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int col = qd + 4 * u;
      const float pj = any ? exp2f(s[u] - mt) : 0.f;
      lt += pj;
      Ps[r * C::SS + col] = bf16_round(pj * vss[col]) * beta;
    }
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    if (any) {
      l_run = l_run * alpha + lt * beta;
      m_run = mn;
    }
    __syncthreads();
    // PV: dims d = qd + 4e
#pragma unroll
    for (int e = 0; e < D / 4; ++e) acc[e] *= alpha;
#pragma unroll 2
    for (int col = 0; col < nrows; ++col) {
      const float pv = Ps[r * C::SS + col];
#pragma unroll
      for (int e = 0; e < D / 4; ++e) acc[e] = fmaf(pv, Vs[col * C::VS + qd + 4 * e], acc[e]);
    }
  }

  if (qi < p.n_q) {
    const float ofac = VE == ELEM_E4M3 ? kTwoPow120 : 1.f;
    const float inv = l_run > 0.f ? ofac / l_run : 0.f;
    const int64_t base = (((int64_t)b * p.n_q + qi) * p.q_heads + hq) * D;
#pragma unroll
    for (int e = 0; e < D / 4; ++e) {
      const float o = acc[e] * inv;
      if (p.out_f32)
        reinterpret_cast<float*>(p.out)[base + qd + 4 * e] = o;
      else
        reinterpret_cast<__nv_bfloat16*>(p.out)[base + qd + 4 * e] = __float2bfloat16_rn(o);
    }
  }
}

template <int D, int KE, int VE>
static cudaError_t launch_pf(const PrefillParams& p, dim3 grid, cudaStream_t st) {
  cudaError_t e = ensure_smem_optin((const void*)prefill_fma<D, KE, VE>, PfCfg<D>::BYTES);
  if (e != cudaSuccess) return e;
  prefill_fma<D, KE, VE><<<grid, 256, PfCfg<D>::BYTES, st>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_pf_d(const PrefillParams& p, int dtype, dim3 grid, cudaStream_t st) {
  if constexpr (D == 128)     // (MXFP8 keys are built for head_dim 128)
    if (dtype == FP8KV_MXK8V8) return launch_pf<D, ELEM_MX, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K8V8) return launch_pf<D, ELEM_E4M3, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K16V8) return launch_pf<D, ELEM_BF16, ELEM_E4M3>(p, grid, st);
  if (dtype == FP8KV_K8V16) return launch_pf<D, ELEM_E4M3, ELEM_BF16>(p, grid, st);
  return launch_pf<D, ELEM_BF16, ELEM_BF16>(p, grid, st);
}

cudaError_t launch_prefill_fma(const PrefillParams& p, int dtype, int batch, cudaStream_t st) {
  if (p.n_q == 0 || batch == 0) return cudaSuccess;
  dim3 grid((p.n_q + kTileTokens - 1) / kTileTokens, p.q_heads, batch);
  return p.c.head_dim == 128 ? launch_pf_d<128>(p, dtype, grid, st)
                             : launch_pf_d<64>(p, dtype, grid, st);
}

}  // namespace fp8kv
