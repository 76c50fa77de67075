/*
 * Oracle: a plain, slow CPU statement of what the int8 MQA decode path
 * computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark use it; the product path never does.
 * It shares no code with the CUDA library.
 *
 * Sources (page titles and sections):
 *  - "Character.AI: inference optimization", 05 Quantization and cost: the
 *    attention KV cache is stored as int8.  The pages fix no granularity or
 *    rounding; the reading here is symmetric per-token absmax with an fp32
 *    scale, s = absmax / 127, code = round-half-even(x / s) clamped to
 *    [-127, 127], all in IEEE fp32.
 *  - "Como funciona a inferencia de IA, explicando claramente", "Por que o
 *    cache KV existe": the new token's query is compared with the key of
 *    every token so far and the values are summed with those weights
 *    (softmax attention).
 *  - "Character.AI: inference optimization", 03 Model architecture, technique
 *    table: Multi-Query Attention, all query heads read one K/V head.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * Floating-point contraction is off so that the fp32 quantizer is exactly
 * the IEEE sequence written below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* Quantize one token's vector x[d] (fp32) to int8 codes and one fp32 scale.
 * A scale of 0 -- amax == 0, or amax so small (below 127 times the smallest
 * subnormal) that amax / 127 rounds to 0 -- gives all codes 0: every code then
 * dequantizes to 0 anyway, and x / 0 has no integer value. */
void oracle_quantize_token(const float* x, int32_t d, int8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int32_t i = 0; i < d; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 127.0f;
  *scale = s;
  for (int32_t i = 0; i < d; ++i) {
    if (s == 0.0f) {
      codes[i] = 0;
      continue;
    }
    float r = nearbyintf(x[i] / s); /* default rounding mode: to nearest, ties to even */
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    codes[i] = (int8_t)r;
  }
}

/* Quantize n tokens (rows of x[n][d]). */
void oracle_quantize_rows(const float* x, int64_t n, int32_t d, int8_t* codes, float* scales) {
  for (int64_t t = 0; t < n; ++t) oracle_quantize_token(x + t * d, d, codes + t * d, scales + t);
}

/* Dequantize codes[T][d] with per-token scales into float64 (exact). */
void oracle_dequantize(const int8_t* codes, const float* scales, int64_t T, int32_t d, double* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int32_t i = 0; i < d; ++i) out[t * d + i] = (double)scales[t] * (double)codes[t * d + i];
}

/* Multi-query softmax attention in float64.
 *   q[Hq][d]  : query of each head
 *   k[T][d], v[T][d] : the single shared K/V head over the attended tokens
 *   out[Hq][d], lse[Hq] : softmax-weighted sum of v, and log sum exp of the logits
 * Logit z_t = c * <q_h, k_t>.  Weights exp(z_t - max z) / sum.  T == 0 gives
 * out = 0, lse = -inf.  Returns 0, or -1 if scratch could not be allocated. */
int oracle_attend(const double* q, int32_t Hq, int32_t d, const double* k, const double* v, int64_t T, double c,
                  double* out, double* lse) {
  double* z = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  if (!z) return -1;
  for (int32_t h = 0; h < Hq; ++h) {
    const double* qh = q + (int64_t)h * d;
    double* oh = out + (int64_t)h * d;
    for (int32_t i = 0; i < d; ++i) oh[i] = 0.0;
    if (T == 0) {
      lse[h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
      double dot = 0.0;
      for (int32_t i = 0; i < d; ++i) dot += qh[i] * k[t * d + i];
      z[t] = c * dot;
      if (z[t] > m) m = z[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      double w = exp(z[t] - m);
      sum += w;
      for (int32_t i = 0; i < d; ++i) oh[i] += w * v[t * d + i];
    }
    for (int32_t i = 0; i < d; ++i) oh[i] /= sum;
    lse[h] = m + log(sum);
  }
  free(z);
  return 0;
}
