/*
 * syngen: seeded, counter-based synthetic inputs for the MoE verify-round layer.
 *
 * This module is the ONLY code shared by the CPU oracle side and the GPU side:
 * it produces unpacked tensors (int4 codes as int8, fp16 scale bits, fp32
 * router weights, bf16 activation rows) and holds none of the layer's
 * arithmetic.  Every value is a pure function of (seed, layer, tensor, index),
 * so any slice of any tensor can be generated on its own, in any order, on any
 * number of threads.
 *
 * Random bits: splitmix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Draw i of a stream with key
 * K is the splitmix64 output function applied to K + (i+1)*GAMMA.
 * Stream key: K = mix(mix(mix(seed + G) + (layer+1) G) + (tensor+1) G).
 *
 * Distributions (the workload recipe of the layer's configurations):
 *   int4 code q : uniform over the integers [-8, 7]; 16 codes per 64-bit draw,
 *                 code i uses bits [4*(i%16), 4*(i%16)+4) of draw i/16, minus 8.
 *   N(0,1)      : Box-Muller on one 64-bit draw d: u1 = ((d>>32)+1)/2^32 in
 *                 (0,1], u2 = (d & 0xffffffff)/2^32 in [0,1),
 *                 z = sqrt(-2 ln u1) cos(2 pi u2), evaluated in double.
 *   fp16 scale  : round-to-nearest-even fp16 of |sigma * z|.
 *   fp32 router : (float)(sigma * z).
 *   bf16 rows   : row r, element h: t = x0[h] + (float)sigma * n_r[h] in fp32
 *                 (x0, n_r independent N(0,1) rounded to fp32; multiply then
 *                 add, no contraction), then round-to-nearest-even bf16.
 *
 * Build: plain C99, -O2 -ffp-contract=off, no fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SG_GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t sg_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t sg_stream_key(uint64_t seed, uint32_t layer, uint32_t tensor) {
  uint64_t k = sg_mix(seed + SG_GAMMA);
  k = sg_mix(k + ((uint64_t)layer + 1u) * SG_GAMMA);
  k = sg_mix(k + ((uint64_t)tensor + 1u) * SG_GAMMA);
  return k;
}

uint64_t sg_draw(uint64_t key, uint64_t i) { return sg_mix(key + (i + 1u) * SG_GAMMA); }

static double sg_normal_from_draw(uint64_t d) {
  const double two_m32 = 2.3283064365386963e-10; /* 2^-32 */
  double u1 = ((double)(d >> 32) + 1.0) * two_m32;
  double u2 = (double)(d & 0xffffffffULL) * two_m32;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* ---- IEEE conversions (round to nearest, ties to even) ------------------ */

uint16_t sg_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

uint16_t sg_f64_to_f16(double d) {
  uint16_t sign = (uint16_t)(signbit(d) ? 0x8000u : 0u);
  double a = fabs(d);
  if (isnan(d)) return (uint16_t)(sign | 0x7e00u);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* rounds to infinity */
  if (a < 6.103515625e-05) {                            /* below 2^-14: subnormal */
    double m = nearbyint(a * 16777216.0);               /* units of 2^-24, RNE */
    return (uint16_t)(sign | (uint16_t)m);              /* m == 1024 is the smallest normal */
  }
  int e;
  double fr = frexp(a, &e);          /* a = fr * 2^e, fr in [0.5, 1) */
  double m = nearbyint(fr * 2048.0); /* 11 significant bits, RNE */
  if (m == 2048.0) { m = 1024.0; e += 1; }
  /* a ~ (m/1024) * 2^(e-1); biased exponent = e - 1 + 15 */
  return (uint16_t)(sign | (uint16_t)((e + 14) << 10) | (uint16_t)((int)m - 1024));
}

/* ---- tensor generators --------------------------------------------------- */

void sg_q4(uint64_t seed, uint32_t layer, uint32_t tensor, uint64_t start, uint64_t count,
           int8_t* out) {
  uint64_t key = sg_stream_key(seed, layer, tensor);
  uint64_t i = start, end = start + count;
  while (i < end) {
    uint64_t d = sg_draw(key, i >> 4);
    unsigned sh = (unsigned)(i & 15u);
    for (; sh < 16u && i < end; ++sh, ++i) *out++ = (int8_t)((int)((d >> (4u * sh)) & 15u) - 8);
  }
}

void sg_normal_f32(uint64_t seed, uint32_t layer, uint32_t tensor, uint64_t start,
                   uint64_t count, double sigma, float* out) {
  uint64_t key = sg_stream_key(seed, layer, tensor);
  for (uint64_t i = 0; i < count; ++i) out[i] = (float)(sigma * sg_normal_from_draw(sg_draw(key, start + i)));
}

void sg_absnormal_f16(uint64_t seed, uint32_t layer, uint32_t tensor, uint64_t start,
                      uint64_t count, double sigma, uint16_t* out) {
  uint64_t key = sg_stream_key(seed, layer, tensor);
  for (uint64_t i = 0; i < count; ++i)
    out[i] = sg_f64_to_f16(fabs(sigma * sg_normal_from_draw(sg_draw(key, start + i))));
}

/* Rows of one layer: out[r*H + h].  x0 uses tensor id t_x0, noise uses t_noise
 * with index r*H + h. */
void sg_rows_bf16(uint64_t seed, uint32_t layer, uint32_t t_x0, uint32_t t_noise, int32_t rows,
                  int32_t hidden, double sigma, uint16_t* out) {
  uint64_t k0 = sg_stream_key(seed, layer, t_x0);
  uint64_t kn = sg_stream_key(seed, layer, t_noise);
  float fs = (float)sigma;
  for (int32_t r = 0; r < rows; ++r) {
    for (int32_t h = 0; h < hidden; ++h) {
      float x0 = (float)sg_normal_from_draw(sg_draw(k0, (uint64_t)h));
      float n = (float)sg_normal_from_draw(sg_draw(kn, (uint64_t)r * (uint64_t)hidden + (uint64_t)h));
      float prod = fs * n;
      float t = x0 + prod;
      out[(size_t)r * (size_t)hidden + (size_t)h] = sg_f32_to_bf16(t);
    }
  }
}
