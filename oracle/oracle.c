/*
 * oracle.c -- CPU oracle of the decode step (TEST INFRASTRUCTURE; see
 * oracle.h). Holds the precision-independent pieces (bf16 conversion, int8
 * quantisation, argmax, the RoPE frequency table) and instantiates
 * oracle_impl.h once in float and once in double.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * -ffp-contract=off keeps every a*b+c as a rounded multiply then a rounded
 * add, so the arithmetic is exactly what the loops say.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* nanoinfer "Weights": bf16 is the top half of an fp32 word; widening
 * appends 16 zero bits, which is exact for every value. */
float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Narrowing rounds to nearest, ties to even: add 0x7FFF plus the lowest kept
 * bit, then drop the low 16 bits. NaN maps to the canonical quiet NaN. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return 0x7FC0;
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

void orc_bf16_to_f32_n(const uint16_t* b, float* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(b[i]);
}

void orc_f32_to_bf16_n(const float* f, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(f[i]);
}

/* nanoinfer "Quantization": symmetric, range [-127, 127], rounding half away
 * from zero (C's roundf). One scale per vector: s = amax / 127. */
float orc_quantize_row_f32(const float* v, int n, int8_t* q) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 127.0f;
  for (int i = 0; i < n; ++i) {
    if (s == 0.0f) {
      q[i] = 0;
      continue;
    }
    float r = roundf(v[i] / s);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = (int8_t)r;
  }
  return s;
}

/* Per output channel: each row of the bf16 matrix gets its own scale. */
void orc_quantize_weight_f32(const uint16_t* w, int n, int k, int8_t* q, float* scale) {
  float* row = (float*)malloc(sizeof(float) * (size_t)k);
  for (int j = 0; j < n; ++j) {
    for (int i = 0; i < k; ++i) row[i] = orc_bf16_to_f32(w[(long)j * k + i]);
    scale[j] = orc_quantize_row_f32(row, k, q + (long)j * k);
  }
  free(row);
}

int orc_matvec_i8(const int8_t* w, int n, int k, const int8_t* x, int32_t* acc) {
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int j = 0; j < n; ++j) {
    int64_t s = 0;
    for (int i = 0; i < k; ++i) s += (int64_t)w[(long)j * k + i] * (int64_t)x[i];
    if (s > INT32_MAX || s < INT32_MIN) bad = 1;
    acc[j] = (int32_t)s;
  }
  return bad ? -1 : 0;
}

/* Greedy decoding is the argmax (nanoinfer "Sampling": temperature 0);
 * ties go to the lowest index. */
int orc_argmax_f32(const float* v, int n) {
  int best = 0;
  for (int i = 0; i < n; ++i) {
    if (isnan(v[i])) return -1;
    if (v[i] > v[best]) best = i;
  }
  return best;
}

int orc_argmax_f64(const double* v, int n) {
  int best = 0;
  for (int i = 0; i < n; ++i) {
    if (isnan(v[i])) return -1;
    if (v[i] > v[best]) best = i;
  }
  return best;
}

void orc_rope_inv_freq(double theta, int d, float* inv_freq) {
  for (int i = 0; i < d / 2; ++i) inv_freq[i] = (float)(1.0 / pow(theta, (2.0 * i) / d));
}

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

#define REAL float
#define SFX f32
#include "oracle_impl.h"
#undef REAL
#undef SFX

#define REAL double
#define SFX f64
#include "oracle_impl.h"
#undef REAL
#undef SFX
