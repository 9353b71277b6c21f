/*
 * fp8kv_oracle.c -- the ORACLE for the FP8-KV attention library.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded CPU
 * statement of what the GPU path computes.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant with the CUDA library and never includes a CUDA
 * header.  Build flags: no fast-math, no FP contraction (see oracle/build.py).
 *
 * What it computes, and where the pages define it:
 *
 *  - E4M3 codes.  "FP8 KV cache (fp8_kv, opt-in)", bullet "Storage": K and V
 *    are stored as e4m3 codes.  The code table is the OCP 8-bit E4M3 format:
 *    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 *    S.1111.111 is NaN, largest finite magnitude 448 (the "448" of the scale
 *    rule on that page).  Rounding is round-to-nearest-even with saturation of
 *    finite values to +-448; the sign of a value that rounds to zero is kept.
 *
 *  - Per-(token, KV head) scale.  Same page, bullet "Storage": one fp32 scale
 *    per (token, KV head), scale = amax(|row|) / 448 over the head dimension,
 *    written once at append.  Computed here as one IEEE fp32 division; each
 *    element is encoded from the IEEE fp32 quotient x / scale.  The page is
 *    silent on an all-zero row: scale 0 and all codes 0x00 is taken.
 *
 *  - Dequantisation: value = decode(code) * scale, in fp64.
 *
 *  - Attention.  Same page, bullet "Math": the method is exact softmax
 *    attention over the dequantised cache, with grouped-query heads (query
 *    head h reads KV head h / (Hq/Hkv), as in "03 · 8n — FA-style tiled
 *    prefill attention", section 3.1 "GQA slicing") and per-sequence lengths.
 *    The oracle states the plain definition in fp64:
 *        s_j = sm_scale * sum_d q_d k_{j,d},   o = sum_j e^{s_j - M} v_j / sum_j e^{s_j - M}
 *    with M = max_j s_j.  The pages' K-scale / V-scale folds, bf16 rounding
 *    of P and tile-by-tile online softmax are how the GPU reaches this result;
 *    they are not restated here.
 *
 *  - Causal prefill ("03 · 8n", section 3.1, masked positions): query i at
 *    absolute position pos0 + i attends keys j <= pos0 + i.
 *
 *  - MXFP8 block scales ("FP8 KV attention: hardware paths and tile
 *    preparation", section "Measure block-scaled QK": D = C + (SFA*A)@(SFB*B)
 *    with one E8M0 scale per 32-element block).  The page does not say how a
 *    block's scale is chosen; the reading taken is the per-token rule of the
 *    fp8_kv page (the scale maps amax to 448) restricted to the powers of two
 *    an E8M0 byte can hold: X = 2^E with E the smallest integer such that
 *    amax <= 448 * 2^E, clamped to [-127, 127], so no element saturates.
 *    Each element is encoded from the fp32 product x * 2^-E.  The byte is
 *    E + 127 (an all-zero block gets E = -127, byte 0).  Dequantisation:
 *    decode(code) * 2^E.
 *
 *  - Pre-bias residual keys ("Fused KV-cache quantization", section
 *    "Bias-aware symmetric FP8"; "FP8 KV attention: hardware paths and tile
 *    preparation", section "Treat numerical safety and kernel speed as
 *    separate gates"): the cache quantises the residual r = k - b of each key
 *    row against a fixed per-KV-head bias b kept exact in fp32, with the
 *    per-row rule above applied to the fp32 residual (r = fp32(k) - b, one
 *    IEEE fp32 subtraction per element).  The key the cache represents is
 *    dequant(r) + b, reconstructed here in fp64.
 *
 *  - Rotated pre-bias residual keys (the same sections; the pages list
 *    post-rotary residual layouts, where the cache holds rotated keys and a
 *    bias added before the rotary embedding turns with the key's position):
 *    the residual of the key at position t is r = fp32(k) - R_t b, with R_t
 *    the rotary rotation in the "rotate half" layout (dims i and i + d/2 form
 *    pair i at angle theta_{t,i}; cos and sin come from the caller's tables):
 *      (R_t b)_i       = b_i cos - b_{i+d/2} sin
 *      (R_t b)_{i+d/2} = b_{i+d/2} cos + b_i sin
 *    each evaluated in fp32 as one fused multiply-add on the product with sin
 *    rounded to fp32 first (fmaf(b_own, cos, -+ (float)(b_other * sin))).
 *    The key the cache represents is dequant(r) + R_t b, in fp64.
 *
 *  - Paged addressing: token t of sequence b lives in page
 *    page_table[b][t / page_size] at offset t % page_size ("FP8 KV attention:
 *    hardware paths and tile preparation", section "Collect the profiler
 *    evidence", which sweeps the page size of a paged cache).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 bits -> float: the bf16 pattern is the upper half of an fp32. */
static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

void fp8kv_oracle_bf16_to_double(const uint16_t *x, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (double)bf16_bits_to_float(x[i]);
}

/* ---------------------------------------------------------------- e4m3 -- */

/* Decode one E4M3 code from the format definition. */
double fp8kv_oracle_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;              /* S.1111.111 */
  if (e == 0)
    mag = ldexp((double)m, -9);                   /* subnormal: m/8 * 2^-6 */
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);    /* normal: 1.m * 2^(e-7) */
  return sign ? -mag : mag;
}

/* Encode one fp32 value: round to nearest, ties to even mantissa, saturate
 * finite magnitudes above 448 to 448, keep the sign of zero results. */
uint8_t fp8kv_oracle_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (isnan(v)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);  /* satfinite */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: quantum 2^-9; a result of 8 quanta is the smallest
     * normal 2^-6, whose code (exponent 1, mantissa 0) is also 8. */
    double q = nearbyint(ldexp(a, 9));            /* exact scaling; RNE */
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e2;
  (void)frexp(a, &e2);                            /* a = f * 2^e2, f in [0.5,1) */
  int e = e2 - 1;                                 /* a in [2^e, 2^(e+1)) */
  double q = nearbyint(ldexp(a, 3 - e));          /* mantissa in eighths: 8..16 */
  int qi = (int)q;
  if (qi == 16) { qi = 8; e += 1; }               /* carried into the exponent */
  int ef = e + 7;                                 /* biased exponent, 1..15 */
  int code = (ef << 3) | (qi - 8);
  if (code > 0x7E) code = 0x7E;                   /* never the NaN pattern */
  return (uint8_t)(sign | code);
}

/* Array forms of the two functions above (one call per element). */
void fp8kv_oracle_e4m3_decode_n(const uint8_t *codes, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp8kv_oracle_e4m3_decode(codes[i]);
}

void fp8kv_oracle_e4m3_encode_n(const float *v, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp8kv_oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------- quantise -- */

/* rows x d bf16 -> rows x d codes and rows scales (amax/448 per row). */
void fp8kv_oracle_quantize(const uint16_t *x, int64_t rows, int d,
                           uint8_t *codes, float *scales) {
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t *xr = x + r * d;
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
      float a = fabsf(bf16_bits_to_float(xr[i]));
      if (a > amax) amax = a;
    }
    float scale = amax / 448.0f;
    scales[r] = scale;
    for (int i = 0; i < d; ++i) {
      if (amax == 0.0f) {
        codes[r * d + i] = 0x00;
      } else {
        float y = bf16_bits_to_float(xr[i]) / scale;
        codes[r * d + i] = fp8kv_oracle_e4m3_encode(y);
      }
    }
  }
}

/* Residual rows: r = fp32(x) - bias (bias: d fp32 values shared by the rows
 * of one KV head; row r uses bias + ((r / rows_per_head) % heads) * d, i.e.
 * rows ordered [..][heads][rows_per_head]), then the per-row rule of
 * fp8kv_oracle_quantize on the fp32 residual. */
void fp8kv_oracle_quantize_residual(const uint16_t *x, const float *bias, int64_t rows, int heads,
                                    int64_t rows_per_head, int d, uint8_t *codes, float *scales) {
  for (int64_t r = 0; r < rows; ++r) {
    const float *br = bias + ((r / rows_per_head) % heads) * d;
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
      const float a = fabsf(bf16_bits_to_float(x[r * d + i]) - br[i]);
      if (a > amax) amax = a;
    }
    const float scale = amax / 448.0f;
    scales[r] = scale;
    for (int i = 0; i < d; ++i) {
      if (amax == 0.0f) {
        codes[r * d + i] = 0x00;
      } else {
        const float y = (bf16_bits_to_float(x[r * d + i]) - br[i]) / scale;
        codes[r * d + i] = fp8kv_oracle_e4m3_encode(y);
      }
    }
  }
}

/* (R_t b)_e for element e of a row of width d (see the header). */
static float rope_bias_elem(const float *b, const float *cs, const float *sn, int d, int e) {
  const int h = d / 2;
  if (e < h) {
    const float p = b[e + h] * sn[e];
    return fmaf(b[e], cs[e], -p);
  }
  const float p = b[e - h] * sn[e - h];
  return fmaf(b[e], cs[e - h], p);
}

/* The rotated bias of every (head, token): bias [heads][d], cos and sin
 * [positions][d/2], the tokens' positions pos[T] -> out [heads][T][d]. */
void fp8kv_oracle_rope_bias(const float *bias, const float *cos_t, const float *sin_t, const int32_t *pos,
                            int heads, int64_t T, int d, float *out) {
  const int h2 = d / 2;
  for (int hd = 0; hd < heads; ++hd)
    for (int64_t t = 0; t < T; ++t)
      for (int e = 0; e < d; ++e)
        out[(hd * T + t) * d + e] = rope_bias_elem(bias + hd * d, cos_t + (int64_t)pos[t] * h2,
                                                   sin_t + (int64_t)pos[t] * h2, d, e);
}

/* Key rows x [heads][T][d] (bf16 bits) at positions pos[T]: the per-row rule
 * on the fp32 residual fp32(k) - R_t b. */
void fp8kv_oracle_quantize_residual_rope(const uint16_t *x, const float *bias, const float *cos_t,
                                         const float *sin_t, const int32_t *pos, int heads, int64_t T, int d,
                                         uint8_t *codes, float *scales) {
  const int h2 = d / 2;
  float y[512];
  for (int hd = 0; hd < heads; ++hd)
    for (int64_t t = 0; t < T; ++t) {
      const int64_t r = hd * T + t;
      float amax = 0.0f;
      for (int e = 0; e < d; ++e) {
        const float rb = rope_bias_elem(bias + hd * d, cos_t + (int64_t)pos[t] * h2, sin_t + (int64_t)pos[t] * h2,
                                        d, e);
        y[e] = bf16_bits_to_float(x[r * d + e]) - rb;
        if (fabsf(y[e]) > amax) amax = fabsf(y[e]);
      }
      const float scale = amax / 448.0f;
      scales[r] = scale;
      for (int e = 0; e < d; ++e)
        codes[r * d + e] = amax == 0.0f ? 0x00 : fp8kv_oracle_e4m3_encode(y[e] / scale);
    }
}

/* codes x scale -> fp64 values. */
void fp8kv_oracle_dequantize(const uint8_t *codes, const float *scales,
                             int64_t rows, int d, double *out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int i = 0; i < d; ++i)
      out[r * d + i] = fp8kv_oracle_e4m3_decode(codes[r * d + i]) * (double)scales[r];
}

/* ------------------------------------------------------------- MXFP8 -- */

/* Exponent E of a block's E8M0 scale: the smallest integer with
 * amax <= 448 * 2^E, clamped to [-127, 127].  With amax = m * 2^e,
 * m in [0.5, 1) (frexp): 448 * 2^(e-9) = 0.875 * 2^e, so E = e - 9 when
 * m <= 0.875 and E = e - 8 otherwise. */
static int mx_block_exponent(float amax) {
  if (amax == 0.0f) return -127;
  int e = 0;
  const float m = frexpf(amax, &e);
  int E = m <= 0.875f ? e - 9 : e - 8;
  if (E < -127) E = -127;
  if (E > 127) E = 127;
  return E;
}

/* Rows of d bf16 values (d a multiple of 32) -> e4m3 codes and one E8M0
 * byte per 32-element block: scales[r * (d / 32) + blk]. */
void fp8kv_oracle_mx_quantize(const uint16_t *x, int64_t rows, int d,
                              uint8_t *codes, uint8_t *scales) {
  const int nb = d / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int blk = 0; blk < nb; ++blk) {
      const uint16_t *xb = x + r * d + blk * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        const float a = fabsf(bf16_bits_to_float(xb[i]));
        if (a > amax) amax = a;
      }
      const int E = mx_block_exponent(amax);
      scales[r * nb + blk] = (uint8_t)(E + 127);
      const float inv = ldexpf(1.0f, -E);      /* exact: a power of two */
      for (int i = 0; i < 32; ++i)
        codes[r * d + blk * 32 + i] = fp8kv_oracle_e4m3_encode(bf16_bits_to_float(xb[i]) * inv);
    }
}

/* codes x 2^(byte - 127) per 32-element block -> fp64 values. */
void fp8kv_oracle_mx_dequantize(const uint8_t *codes, const uint8_t *scales,
                                int64_t rows, int d, double *out) {
  const int nb = d / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int i = 0; i < d; ++i)
      out[r * d + i] = fp8kv_oracle_e4m3_decode(codes[r * d + i]) *
                       ldexp(1.0, (int)scales[r * nb + i / 32] - 127);
}

/* ---------------------------------------------------------- paged cache -- */

/* Gather sequence b of a paged pool into token order.
 * pool: [num_pages][heads][page_size][row_bytes] bytes;
 * out:  [heads][n_tokens][row_bytes]. Returns -1 on an out-of-range page. */
int fp8kv_oracle_gather_paged(const uint8_t *pool, int num_pages, int heads,
                              int page_size, int row_bytes,
                              const int32_t *page_table, int max_pages_per_seq,
                              int b, int n_tokens, uint8_t *out) {
  for (int h = 0; h < heads; ++h)
    for (int t = 0; t < n_tokens; ++t) {
      int32_t page = page_table[(int64_t)b * max_pages_per_seq + t / page_size];
      int off = t % page_size;
      if (page < 0 || page >= num_pages) return -1;
      const uint8_t *src =
          pool + (((int64_t)page * heads + h) * page_size + off) * row_bytes;
      memcpy(out + ((int64_t)h * n_tokens + t) * row_bytes, src, (size_t)row_bytes);
    }
  return 0;
}

/* ------------------------------------------------------------ attention -- */

/* One query vector against n keys: the plain softmax-attention definition. */
static void attend_one(const double *q, const double *k, const double *v,
                       int64_t k_stride, int n, int d, double sm_scale,
                       double *out) {
  int i, j;
  for (i = 0; i < d; ++i) out[i] = 0.0;
  if (n <= 0) return;
  double m = -INFINITY;
  for (j = 0; j < n; ++j) {
    double s = 0.0;
    for (i = 0; i < d; ++i) s += q[i] * k[j * k_stride + i];
    s *= sm_scale;
    if (s > m) m = s;
  }
  double denom = 0.0;
  for (j = 0; j < n; ++j) {
    double s = 0.0;
    for (i = 0; i < d; ++i) s += q[i] * k[j * k_stride + i];
    double w = exp(s * sm_scale - m);
    denom += w;
    for (i = 0; i < d; ++i) out[i] += w * v[j * k_stride + i];
  }
  for (i = 0; i < d; ++i) out[i] /= denom;
}

/* Decode: one query token per sequence.
 * q [B][Hq][D]; k, v [B][Hkv][Tmax][D]; out [B][Hq][D]. */
void fp8kv_oracle_decode(const double *q, const double *k, const double *v,
                         const int32_t *seq_lens, int B, int Hq, int Hkv,
                         int Tmax, int D, double sm_scale, double *out) {
  int G = Hq / Hkv;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      int g = h / G;
      const double *kb = k + ((int64_t)b * Hkv + g) * Tmax * D;
      const double *vb = v + ((int64_t)b * Hkv + g) * Tmax * D;
      attend_one(q + ((int64_t)b * Hq + h) * D, kb, vb, D, seq_lens[b], D,
                 sm_scale, out + ((int64_t)b * Hq + h) * D);
    }
}

/* Causal prefill of one sequence: query i sits at absolute position pos0 + i
 * and attends keys 0..pos0+i.  q, out [n_q][Hq][D]; k, v [Hkv][Tk][D]. */
void fp8kv_oracle_prefill(const double *q, const double *k, const double *v,
                          int n_q, int pos0, int Hq, int Hkv, int Tk, int D,
                          double sm_scale, double *out) {
  int G = Hq / Hkv;
  for (int i = 0; i < n_q; ++i)
    for (int h = 0; h < Hq; ++h) {
      int g = h / G;
      int n = pos0 + i + 1;
      if (n > Tk) n = Tk;
      attend_one(q + ((int64_t)i * Hq + h) * D, k + (int64_t)g * Tk * D,
                 v + (int64_t)g * Tk * D, D, n, D, sm_scale,
                 out + ((int64_t)i * Hq + h) * D);
    }
}
