/*
 * Element-level definitions of the synthetic input generator, shared by its host
 * implementation (synth.c) and its device implementation (synth_gpu.cu) so both
 * draw bit-identical tensors: Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11), the Irwin-Hall(8)
 * normal deviate, round-to-nearest-even to bf16, and the E2M1 / E4M3 rounding
 * used to encode synthetic NVFP4 weights.  Input preparation only.
 * Compile without fused multiply-add (-ffp-contract=off / -fmad=false).
 */
#ifndef SYNTH_DEFS_H
#define SYNTH_DEFS_H
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define SYNTH_FN static __host__ __device__ inline
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_PHILOX_M0 0xD2511F53u
#define SYNTH_PHILOX_M1 0xCD9E8D57u
#define SYNTH_PHILOX_W0 0x9E3779B9u
#define SYNTH_PHILOX_W1 0xBB67AE85u

/* four 32-bit words for (key = seed, counter = {block, stream}) */
SYNTH_FN void synth_draw(uint64_t seed, uint64_t stream, uint64_t block, uint32_t out[4]) {
  uint32_t c0 = (uint32_t)block, c1 = (uint32_t)(block >> 32), c2 = (uint32_t)stream, c3 = (uint32_t)(stream >> 32);
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)SYNTH_PHILOX_M0 * c0;
    uint64_t p1 = (uint64_t)SYNTH_PHILOX_M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += SYNTH_PHILOX_W0; k1 += SYNTH_PHILOX_W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* unit-variance Irwin-Hall(8) deviate: eight 16-bit uniforms (j + 1/2) / 65536,
   centred and scaled by sqrt(12/8); integer arithmetic and one multiply */
SYNTH_FN double synth_unit_normal(uint64_t seed, uint64_t stream, uint64_t i) {
  uint32_t w[4];
  synth_draw(seed, stream, i, w);
  int64_t s = 0;
  for (int j = 0; j < 4; ++j) s += (int64_t)(w[j] & 0xFFFFu) + (int64_t)(w[j] >> 16);
  int64_t centred2 = 2 * s + 8 - 8 * 65536; /* 2 * 65536 * (sum - 4) */
  const double k = 1.2247448713915890 / 131072.0;
  return (double)centred2 * k;
}

SYNTH_FN double synth_value(uint64_t seed, uint64_t stream, uint64_t i, double mean, double std) {
  return mean + std * synth_unit_normal(seed, stream, i);
}

/* round-to-nearest-even of a double to bf16 bits, directly (no fp32 step) */
SYNTH_FN uint16_t synth_bf16_rne(double x) {
  uint16_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x8000u : 0u;
  double a = fabs(x);
  if (a != a) return 0x7FC0u;
  if (a == 0.0) return sign;
  int e;
  double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
  double q;
  if (e - 1 < -126) {
    q = ldexp(nearbyint(ldexp(a, 133)), -133);
  } else {
    q = ldexp(nearbyint(ldexp(m, 8)), e - 8);
  }
  if (q > 3.3895313892515355e38) return sign | 0x7F80u;
  float f = (float)q; /* exact */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return sign | (uint16_t)((bits >> 16) & 0x7FFFu);
}

/* E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6: nearest, ties to the even code, saturating */
SYNTH_FN uint8_t synth_e2m1_rne(float v) {
  const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  uint8_t sign = signbit(v) ? 8u : 0u;
  float a = fabsf(v);
  if (!(a < 6.0f)) return sign | 7u;
  int lo = 0;
  for (int c = 7; c >= 0; --c)
    if (grid[c] <= a) { lo = c; break; }
  if (lo == 7) return sign | 7u;
  float dl = a - grid[lo], dh = grid[lo + 1] - a;
  int c = (dl < dh) ? lo : (dh < dl) ? lo + 1 : ((lo % 2 == 0) ? lo : lo + 1);
  return sign | (uint8_t)c;
}

/* E4M3 ("FN": bias 7, no infinities, max 448, subnormal step 2^-9) value of a code */
SYNTH_FN float synth_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return s ? -v : v;
}

/* nearest non-negative E4M3 code, ties to even, saturating at 448 */
SYNTH_FN uint8_t synth_e4m3_rne(float v) {
  if (!(v > 0.0f)) return 0;
  if (v >= 448.0f) return 0x7E;
  if (v < 0.015625f) return (uint8_t)nearbyintf(ldexpf(v, 9)); /* subnormal; 8 = smallest normal */
  int e;
  float f = frexpf(v, &e); /* v = f 2^e, f in [0.5, 1) */
  int E = e - 1;
  float r = nearbyintf(ldexpf(f, 4));
  if (r == 16.0f) { r = 8.0f; E += 1; }
  int code = ((E + 7) << 3) | ((int)r - 8);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)code;
}

#endif
