/*
 * w4a16_oracle.c -- the CPU oracle for the INT4 weight-only (W4A16) GEMV, its
 * layer epilogues and the fp16-KV decode attention next to it.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, single-threaded
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check in __graft_entry__ and the cpu_baseline / reference leg of bench.py may
 * load it.  It shares no code, header, table or helper with the CUDA library in
 * int4_weight_only_gemv_gb300/, and the CUDA library never calls it.
 *
 * What it follows.  The format is the one of the page "Costruire un runtime di
 * inference LLM da zero" (datastack.it, summary of "How To Build Your Own LLM
 * Runtime From Scratch"), section "Tre bug che insegnano":
 *   - last paragraph: INT4 weights, symmetric, group-wise with group 128, on
 *     the seven per-layer projections (embedding, rms_norm, lm_head stay FP16);
 *   - third bug: the gate/up/down GEMVs unpack the INT4 nibbles inside the
 *     kernel and multiply FP16 activations.
 * The pages print no packing layout, no scale formula and no rounding rule.
 * The numeric details used here are the workload definition's: per-group
 * scale = max|w| / 7 stored as fp16, q = clamp(round(w / s), -8, 7), and eight
 * nibbles per uint32, little-endian.  Where that is silent too, the readings
 * are: nibble i (bits 4i..4i+3) of word j of row n holds k = 8j + i; scales
 * are fp16[N][K/G] row-major; max|w| / 7 is divided in fp32 and rounded to
 * fp16 to nearest-even; round() is half away from zero on the exact quotient
 * w / s (computed in double, which decides every case exactly, see
 * orc_quantize); a group whose max|w| is 0 gets s = 0 and q = 0.
 *
 * Every floating-point result that has a plain definition is that definition:
 * the GEMV is y[m][n] = sum_k x[m][k] * (q[n][k] * s[n][k/G]) accumulated in
 * FP64 in ascending k (each product is exact in FP64: 11 + 4 + 11 significand
 * bits), and the dequant is fp16_RN(q * s) (q * s is exact, so this is one
 * rounding).
 *
 * binary16 conversions are written from the IEEE 754 definition of the format
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits, subnormals with
 * exponent 2^-14, round to nearest with ties to even); they do not use any
 * compiler or library half-precision type.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (see build.py).
 * -ffp-contract=off keeps every a*b+c as two roundings on both x86-64 and
 * aarch64, so the oracle gives the same bits on both hosts.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_SHAPE 1
#define ORC_ERR_NONFINITE 2
#define ORC_ERR_SCALE_OVERFLOW 3

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16
 * ------------------------------------------------------------------------- */

/* Value of a binary16 bit pattern, exactly, as a double. */
double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* Round a non-negative double that is exact (an integer plus a fraction
 * representable in double) to the nearest integer, ties to even. */
static double round_half_even(double r) {
  double fl = floor(r);
  double d = r - fl; /* exact: r < 2^53 in every caller */
  if (d > 0.5) return fl + 1.0;
  if (d < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary16 nearest to v, ties to even; overflow goes to infinity. */
uint16_t orc_double_to_half(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  if (isnan(v)) return (uint16_t)(sign | 0x7e00);
  double a = fabs(v);
  /* Largest finite is 65504 = 2047 * 2^5; the next step would be 65536, so
   * the midpoint 65520 and everything above rounds to infinity (65520 is a
   * tie between 65504 (odd fraction 1023) and 65536 (even): goes to 65536). */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: multiples of 2^-24 */
    double m = round_half_even(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)m); /* m == 1024 is the smallest normal */
  }
  int E;
  frexp(a, &E);      /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1;     /* a in [2^e, 2^(e+1)), e in [-14, 15] */
  double m = round_half_even(ldexp(a, 10 - e)); /* in [1024, 2048] */
  if (m == 2048.0) {
    m = 1024.0;
    e += 1;
  }
  if (e > 15) return (uint16_t)(sign | 0x7c00);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(m - 1024.0));
}

/* float -> binary16: float -> double is exact, so this is a single rounding. */
uint16_t orc_float_to_half(float v) { return orc_double_to_half((double)v); }

void orc_double_to_half_array(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_double_to_half(v[i]);
}

void orc_half_to_double_array(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_half_to_double(h[i]);
}

/* ---------------------------------------------------------------------------
 * The INT4 group-wise format
 * ------------------------------------------------------------------------- */

/* Signed value of one 4-bit two's-complement nibble. */
static int nibble_value(uint32_t nib) {
  int v = (int)(nib & 0xf);
  if (v >= 8) v -= 16;
  return v;
}

static int shape_ok(int64_t N, int64_t K, int64_t G) {
  return N >= 0 && K > 0 && G > 0 && G % 8 == 0 && K % G == 0;
}

/*
 * Quantise fp32 W[N][K] into qweight uint32[N][K/8] and scales fp16[N][K/G].
 * Per (row n, group g):
 *   s = fp16_RN( float( max_{k in g} |w[n][k]| / 7 ) )   -- fp32 division
 *   q = clamp( round_half_away( w / s ), -8, 7 )          -- s == 0 -> q = 0
 * The quotient is taken in double.  w has 24 significand bits and s 11, so a
 * non-tie quotient w / s differs from every half-integer by far more than
 * double's 2^-53 relative spacing: the double division therefore makes the
 * same rounding decision as the exact real quotient.
 * Nibble i of word j of row n holds k = 8j + i, as q & 0xF.
 * Returns ORC_OK, ORC_ERR_SHAPE, ORC_ERR_NONFINITE or ORC_ERR_SCALE_OVERFLOW.
 */
int orc_quantize(const float* w, int64_t N, int64_t K, int64_t G, uint32_t* qweight,
                 uint16_t* scales) {
  if (!shape_ok(N, K, G)) return ORC_ERR_SHAPE;
  for (int64_t i = 0; i < N * K; ++i)
    if (!isfinite(w[i])) return ORC_ERR_NONFINITE;
  memset(qweight, 0, (size_t)(N * (K / 8)) * sizeof(uint32_t));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < K / G; ++g) {
      const float* wg = w + n * K + g * G;
      float amax = 0.0f;
      for (int64_t k = 0; k < G; ++k) {
        float a = fabsf(wg[k]);
        if (a > amax) amax = a;
      }
      float d = amax / 7.0f;
      uint16_t sbits = orc_float_to_half(d);
      if ((sbits & 0x7c00) == 0x7c00) return ORC_ERR_SCALE_OVERFLOW;
      scales[n * (K / G) + g] = sbits;
      double s = orc_half_to_double(sbits);
      for (int64_t k = 0; k < G; ++k) {
        int q = 0;
        if (s != 0.0) {
          double r = round((double)wg[k] / s); /* C round(): half away from zero */
          if (r > 7.0) r = 7.0;
          if (r < -8.0) r = -8.0;
          q = (int)r;
        }
        int64_t kk = g * G + k;
        qweight[n * (K / 8) + kk / 8] |= ((uint32_t)q & 0xfu) << (4 * (kk % 8));
      }
    }
  }
  return ORC_OK;
}

/* q[n][k] in [-8, 7] from the packed words. */
int orc_unpack(const uint32_t* qweight, int64_t N, int64_t K, int8_t* q) {
  if (N < 0 || K <= 0 || K % 8 != 0) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      uint32_t word = qweight[n * (K / 8) + k / 8];
      q[n * K + k] = (int8_t)nibble_value(word >> (4 * (k % 8)));
    }
  return ORC_OK;
}

/* w_hat[n][k] = q[n][k] * s[n][k/G], exact, as a double. */
static double w_hat(const uint32_t* qweight, const uint16_t* scales, int64_t K, int64_t G,
                    int64_t n, int64_t k) {
  uint32_t word = qweight[n * (K / 8) + k / 8];
  int q = nibble_value(word >> (4 * (k % 8)));
  double s = orc_half_to_double(scales[n * (K / G) + k / G]);
  return (double)q * s;
}

/* Debug dequantisation: w_out fp16[N][K] = fp16_RN(q * s). */
int orc_dequant(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K,
                int64_t G, uint16_t* w_out) {
  if (!shape_ok(N, K, G)) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      w_out[n * K + k] = orc_double_to_half(w_hat(qweight, scales, K, G, n, k));
  return ORC_OK;
}

/* Exact dequantised weights as doubles (used for row norms in the tolerance). */
int orc_dequant_f64(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K,
                    int64_t G, double* w_out) {
  if (!shape_ok(N, K, G)) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) w_out[n * K + k] = w_hat(qweight, scales, K, G, n, k);
  return ORC_OK;
}

/* y[m][i] = sum_k x[m][k] * w_hat[rows[i]][k], FP64, ascending k.
 * x is fp16 [M][K] (bit patterns); y is double [M][nrows]. */
int orc_gemv_rows(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                  int64_t M, int64_t N, int64_t K, int64_t G, const int64_t* rows,
                  int64_t nrows, double* y) {
  if (!shape_ok(N, K, G) || M < 0) return ORC_ERR_SHAPE;
  for (int64_t i = 0; i < nrows; ++i)
    if (rows[i] < 0 || rows[i] >= N) return ORC_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t n = rows[i];
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += orc_half_to_double(x[m * K + k]) * w_hat(qweight, scales, K, G, n, k);
      y[m * nrows + i] = acc;
    }
  }
  return ORC_OK;
}

/* The whole GEMV: y double [M][N]. */
int orc_gemv(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x, int64_t M,
             int64_t N, int64_t K, int64_t G, double* y) {
  if (!shape_ok(N, K, G) || M < 0) return ORC_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += orc_half_to_double(x[m * K + k]) * w_hat(qweight, scales, K, G, n, k);
      y[m * N + n] = acc;
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Layer epilogues around the GEMV (the page on hipfire, "Overview of
 * hipfire-arch-qwen2", "Key Technical Specifications": a SwiGLU feed-forward
 * and attention_bias on the Q, K and V projections).  A bias is added to the
 * GEMV's unrounded FP64 sum by the caller; SwiGLU is defined here.
 * ------------------------------------------------------------------------- */

/* silu(v) = v * sigmoid(v) = v / (1 + e^-v), in double. */
double orc_silu(double v) { return v / (1.0 + exp(-v)); }

/* h[i] = fp16_RN(silu(g[i]) * u[i]) from fp16 g and u, in double with one
 * rounding to fp16 at the end. */
void orc_swiglu(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h) {
  for (int64_t i = 0; i < n; ++i)
    h[i] = orc_double_to_half(orc_silu(orc_half_to_double(g[i])) * orc_half_to_double(u[i]));
}

/* ---------------------------------------------------------------------------
 * Decode attention over an fp16 KV cache (the page "LLM170", README of the
 * LLM170 engine: the paragraph on its HIP attention path, whose decode kernel
 * reads an f16 copy of the KV cache, and the long-context benchmark paragraph,
 * where that decode attention is bandwidth-bound on the f16 KV).  The pages
 * print no formula; this is the standard scaled dot-product attention of one
 * query token with grouped-query heads, the model shape of the page "Costruire
 * un runtime di inference LLM da zero", last paragraph of "Tre bug che
 * insegnano" (28 query heads sharing 4 KV heads, head dimension 128).
 *
 * Query head h (of n_heads) reads KV head g = h / (n_heads / n_kv_heads):
 *   s_t = (q_h . k_{g,t}) / sqrt(D)                     for t = 0 .. T-1
 *   p_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
 *   o_h = sum_t p_t v_{g,t}
 * in double from the fp16 inputs, sums in ascending t (and d).  Layout:
 * q [n_heads][D], k and v [n_kv_heads][t_stride][D] (keys t < T used),
 * o [n_heads][D] as double.
 * ------------------------------------------------------------------------- */
int orc_attn_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t n_heads,
                    int64_t n_kv_heads, int64_t D, int64_t T, int64_t t_stride, double* o) {
  if (n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 || D <= 0 || T <= 0 ||
      t_stride < T)
    return ORC_ERR_SHAPE;
  const int64_t group = n_heads / n_kv_heads;
  double* s = (double*)malloc(sizeof(double) * (size_t)T);
  if (s == NULL) return ORC_ERR_SHAPE;
  const double scale = 1.0 / sqrt((double)D);
  for (int64_t h = 0; h < n_heads; ++h) {
    const int64_t g = h / group;
    double smax = -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d)
        dot += orc_half_to_double(q[h * D + d]) * orc_half_to_double(k[(g * t_stride + t) * D + d]);
      s[t] = dot * scale;
      if (s[t] > smax) smax = s[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      s[t] = exp(s[t] - smax);
      sum += s[t];
    }
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += s[t] * orc_half_to_double(v[(g * t_stride + t) * D + d]);
      o[h * D + d] = acc / sum;
    }
  }
  free(s);
  return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * W4A8: the INT8-activation variant that the page "Costruire un runtime di
 * inference LLM da zero", "Tre bug che insegnano" (third bug) describes
 * trying with dp4a against the FP16-activation GEMV.  The page gives no
 * activation format; the reading here is symmetric int8 per block of 64
 * consecutive k of one activation row (half a weight group):
 *   amax_b = max_{k in b} |x[k]|                  (exact, from fp16 values)
 *   s_b    = amax_b / 127,  inv_b = 127 / amax_b  (each one FP32 division)
 *   xq[k]  = round_half_even(x[k] * inv_b)       (FP32 product; |xq| <= 127)
 * with s_b = inv_b = 0 and xq = 0 for an all-zero block.  These steps are in
 * FP32 because they decide integers: the GPU takes the same decisions in the
 * same precision.  Ties go to even, IEEE's default rounding (the page states
 * no rule).  No clamp is needed: |x| <= amax gives |x inv| <= 127 (1 + 2^-23),
 * which rounds to at most 127.  The GEMV is then
 *   y[m][n] = sum_b s_w[n][b / 2] s_b sum_{k in b} q[n][k] xq[k]
 * with exact integer inner sums, in FP64.
 * ------------------------------------------------------------------------- */
#define ORC_A8_BLOCK 64

/* Quantise one activation row x[K] (K a multiple of 64): xq[K], s[K / 64]. */
int orc_quantize_act_a8(const uint16_t* x, int64_t K, int8_t* xq, float* s) {
  if (K <= 0 || K % ORC_A8_BLOCK != 0) return ORC_ERR_SHAPE;
  for (int64_t b = 0; b < K / ORC_A8_BLOCK; ++b) {
    float amax = 0.0f;
    for (int64_t k = b * ORC_A8_BLOCK; k < (b + 1) * ORC_A8_BLOCK; ++k) {
      const float v = fabsf((float)orc_half_to_double(x[k]));
      if (!(v <= 3.0e38f)) return ORC_ERR_NONFINITE;
      if (v > amax) amax = v;
    }
    const float sb = amax > 0.0f ? amax / 127.0f : 0.0f;
    const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
    s[b] = sb;
    for (int64_t k = b * ORC_A8_BLOCK; k < (b + 1) * ORC_A8_BLOCK; ++k) {
      const float p = (float)orc_half_to_double(x[k]) * inv;
      const float r = nearbyintf(p); /* the default mode: to nearest, ties to even */
      if (r > 127.0f || r < -127.0f) return ORC_ERR_SHAPE; /* cannot happen, see above */
      xq[k] = (int8_t)r;
    }
  }
  return ORC_OK;
}

/* y[M][N] (double) of the W4A8 GEMV above, x fp16 [M][K]. */
int orc_gemv_w4a8(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x, int64_t M,
                  int64_t N, int64_t K, int64_t G, double* y) {
  if (M <= 0 || !shape_ok(N, K, G) || G % ORC_A8_BLOCK != 0) return ORC_ERR_SHAPE;
  int8_t* xq = (int8_t*)malloc((size_t)K);
  float* sx = (float*)malloc(sizeof(float) * (size_t)(K / ORC_A8_BLOCK));
  if (xq == NULL || sx == NULL) {
    free(xq);
    free(sx);
    return ORC_ERR_SHAPE;
  }
  int rc = ORC_OK;
  for (int64_t m = 0; m < M && rc == ORC_OK; ++m) {
    rc = orc_quantize_act_a8(x + m * K, K, xq, sx);
    for (int64_t n = 0; n < N && rc == ORC_OK; ++n) {
      double acc = 0.0;
      for (int64_t b = 0; b < K / ORC_A8_BLOCK; ++b) {
        int64_t isum = 0;
        for (int64_t k = b * ORC_A8_BLOCK; k < (b + 1) * ORC_A8_BLOCK; ++k) {
          const uint32_t word = qweight[n * (K / 8) + k / 8];
          isum += (int64_t)nibble_value(word >> (4 * (k % 8))) * (int64_t)xq[k];
        }
        acc += (double)isum * orc_half_to_double(scales[n * (K / G) + (b * ORC_A8_BLOCK) / G]) * (double)sx[b];
      }
      y[m * N + n] = acc;
    }
  }
  free(xq);
  free(sx);
  return rc;
}

/* ---------------------------------------------------------------------------
 * GGUF Q4_K super-blocks (the page "VTE" (page 1), dequantisation of Q4_K /
 * Q6_K / Q8_0 byte for byte in llama.cpp's reference layout, checked layer
 * by layer against NumPy; the hipEngine page serves GGUF Q4_K_M files).  The
 * pages print no layout; this is the GGUF Q4_K block as published with that
 * format.  A row of K weights (K a multiple of 256) is K / 256 blocks of 144
 * bytes:
 *   bytes 0-1   d     (fp16)   scale of the sub-block scales
 *   bytes 2-3   dmin  (fp16)   scale of the sub-block minima
 *   bytes 4-15  eight 6-bit scales sc_j and eight 6-bit minima m_j:
 *               j < 4:  sc_j = b[j] & 63,  m_j = b[j + 4] & 63
 *               j >= 4: sc_j = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4)
 *                       m_j  = (b[j + 4] >> 4) | ((b[j] >> 6) << 4)
 *               (b = bytes 4-15)
 *   bytes 16-143  256 unsigned 4-bit codes q: weight e of the block, with
 *               c = e / 64 and i = e % 64, is the low nibble of byte
 *               16 + 32 c + i for i < 32 (sub-block j = 2 c) and the high
 *               nibble of byte 16 + 32 c + i - 32 for i >= 32 (j = 2 c + 1).
 * The weight is w = d sc_j q - dmin m_j.  The reference dequantisation works
 * in FP32 as d1 = d sc_j, m1 = dmin m_j, w = d1 q - m1 (three roundings,
 * no fused multiply-add); the GEMV uses the exact value (every product fits
 * FP64 exactly: 11 + 6 + 4 significand bits) in an FP64 sum.
 * ------------------------------------------------------------------------- */
#define ORC_QK 256
#define ORC_QK_BYTES 144

static void q4k_scale_min(int j, const uint8_t* b, int* sc, int* m) {
  if (j < 4) {
    *sc = b[j] & 63;
    *m = b[j + 4] & 63;
  } else {
    *sc = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4);
    *m = (b[j + 4] >> 4) | ((b[j] >> 6) << 4);
  }
}

/* Code, sub-block of weight e (0..255) of one block. */
static int q4k_code(const uint8_t* blk, int e, int* j) {
  const int c = e / 64, i = e % 64;
  if (i < 32) {
    *j = 2 * c;
    return blk[16 + 32 * c + i] & 15;
  }
  *j = 2 * c + 1;
  return blk[16 + 32 * c + i - 32] >> 4;
}

static uint16_t rd_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* w[N][K] as float (the FP32 reference dequantisation above). */
int orc_q4k_dequant(const uint8_t* blocks, int64_t N, int64_t K, float* w) {
  if (N < 0 || K <= 0 || K % ORC_QK != 0) return ORC_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t s = 0; s < K / ORC_QK; ++s) {
      const uint8_t* blk = blocks + (n * (K / ORC_QK) + s) * ORC_QK_BYTES;
      const float d = (float)orc_half_to_double(rd_u16(blk));
      const float dmin = (float)orc_half_to_double(rd_u16(blk + 2));
      for (int e = 0; e < ORC_QK; ++e) {
        int j, sc, m;
        const int q = q4k_code(blk, e, &j);
        q4k_scale_min(j, blk + 4, &sc, &m);
        const float d1 = d * (float)sc;
        const float m1 = dmin * (float)m;
        const float dq = d1 * (float)q;
        w[n * K + s * ORC_QK + e] = dq - m1;
      }
    }
  return ORC_OK;
}

/* y[M][N] = x[M][K] . w^T with the exact weights, in FP64 (ascending k). */
int orc_q4k_gemv(const uint8_t* blocks, const uint16_t* x, int64_t M, int64_t N, int64_t K, double* y) {
  if (M <= 0 || N < 0 || K <= 0 || K % ORC_QK != 0) return ORC_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t* blk = blocks + (n * (K / ORC_QK) + k / ORC_QK) * ORC_QK_BYTES;
        int j, sc, mn;
        const int q = q4k_code(blk, (int)(k % ORC_QK), &j);
        q4k_scale_min(j, blk + 4, &sc, &mn);
        const double wv = orc_half_to_double(rd_u16(blk)) * sc * q - orc_half_to_double(rd_u16(blk + 2)) * mn;
        acc += orc_half_to_double(x[m * K + k]) * wv;
      }
      y[m * N + n] = acc;
    }
  return ORC_OK;
}
