/*
 * Seeded synthetic inputs for the speculative-decoding verify step.
 *
 * This module draws the inputs both the CUDA path and the CPU oracle consume:
 * bf16 activations / weights / KV history, NVFP4-encoded expert weights, draft
 * trees (parent arrays) and router hot sets.  It holds none of the verify step's
 * arithmetic: no attention, no norm, no GEMM, no routing.
 *
 * Random numbers come from Philox4x32-10, the counter-based generator defined in
 * Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 * (SC'11): a 64-bit key (the seed) and a 128-bit counter (element index in the
 * low 64 bits, a tensor-stream id in the high 64 bits) map to four 32-bit words.
 * Any element of any tensor can therefore be produced on demand, in any order,
 * on any machine, with bit-identical results.
 *
 * Normal deviates use the Irwin-Hall construction: the sum of eight 16-bit
 * uniforms, centred and scaled to unit variance.  It needs integer arithmetic
 * and one multiply only, so every platform draws the same bits (no libm).  Its
 * support is [-4.9, 4.9] sigma; that is the only departure from a true normal.
 *
 * Build with -ffp-contract=off so no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox4x32_10(uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += PHILOX_W0; k1 += PHILOX_W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Four 32-bit words for (seed, stream, block). */
static void draw_block(uint64_t seed, uint64_t stream, uint64_t block, uint32_t out[4]) {
  uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)stream,
                     (uint32_t)(stream >> 32)};
  philox4x32_10(ctr, (uint32_t)seed, (uint32_t)(seed >> 32), out);
}

/* Public: raw words, for tests of the generator itself. */
void synth_philox(uint64_t seed, uint64_t stream, uint64_t block, uint32_t* out4) {
  draw_block(seed, stream, block, out4);
}

/* Stream id for a tensor: kind (16 bits) | layer (16 bits) | expert (16 bits) | part (16 bits). */
uint64_t synth_stream(int kind, int layer, int expert, int part) {
  return ((uint64_t)(uint16_t)kind << 48) | ((uint64_t)(uint16_t)layer << 32) |
         ((uint64_t)(uint16_t)expert << 16) | (uint64_t)(uint16_t)part;
}

/* Unit-variance Irwin-Hall(8) deviate for element i of the stream. */
static double unit_normal(uint64_t seed, uint64_t stream, uint64_t i) {
  uint32_t w[4];
  draw_block(seed, stream, i, w);
  int64_t s = 0;
  for (int j = 0; j < 4; ++j) s += (int64_t)(w[j] & 0xFFFFu) + (int64_t)(w[j] >> 16);
  /* uniforms u = (j + 1/2) / 65536; sum of eight has mean 4 and variance 8/12 */
  int64_t centred2 = 2 * s + 8 - 8 * 65536; /* = 2 * 65536 * (sum - 4) */
  const double k = 1.2247448713915890 / 131072.0; /* sqrt(12/8) / (2 * 65536) */
  return (double)centred2 * k;
}

/* Round-to-nearest-even of a double to bf16 bits (no double rounding via fp32). */
static uint16_t bf16_bits_rne(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (isnan(x)) return 0x7FC0u;
  if (a == 0.0) return sign;
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  double q;
  if (e - 1 < -126) {
    /* subnormal bf16: quantum 2^-133 */
    q = nearbyint(ldexp(a, 133));
    q = ldexp(q, -133);
  } else {
    double r = nearbyint(ldexp(m, 8)); /* 8 significant bits */
    q = ldexp(r, e - 8);
  }
  if (q > 3.3895313892515355e38) return sign | 0x7F80u; /* overflow to inf */
  float f = (float)q; /* exact */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return sign | (uint16_t)((bits >> 16) & 0x7FFFu);
}

void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                      double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = mean + std * unit_normal(seed, stream, (uint64_t)i);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                      float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = (float)(mean + std * unit_normal(seed, stream, (uint64_t)i));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                       uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = bf16_bits_rne(mean + std * unit_normal(seed, stream, (uint64_t)i));
}

/* ---- NVFP4 encoding of synthetic weights (input preparation) ----------------
 * E2M1 magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7, bit 3 = sign).
 * E4M3 (OCP "FN" variant): bias 7, no infinities, max 448, subnormal step 2^-9.
 * Encoding recipe for one matrix [rows][cols], blocks of 16 along cols:
 *   tensor scale ts = amax / (6 * 448)                          (fp32)
 *   block scale  s  = E4M3_rne(amax_block / (6 * ts))           (fp32 in)
 *   code         c  = E2M1_rne(x / (decode(s) * ts)), 0 if s == 0
 */
static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

static uint8_t e2m1_rne(float v) {
  uint8_t sign = signbit(v) ? 8u : 0u;
  float a = fabsf(v);
  if (!(a < 6.0f)) return sign | 7u; /* saturate (and NaN -> max, never occurs) */
  /* find the bracketing grid points and round to nearest, ties to even code */
  int lo = 0;
  for (int c = 7; c >= 0; --c)
    if (kE2M1[c] <= a) { lo = c; break; }
  if (lo == 7) return sign | 7u;
  float dl = a - kE2M1[lo], dh = kE2M1[lo + 1] - a;
  int c;
  if (dl < dh) c = lo;
  else if (dh < dl) c = lo + 1;
  else c = (lo % 2 == 0) ? lo : lo + 1;
  return sign | (uint8_t)c;
}

static float e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  float v;
  if (e == 0) v = ldexpf((float)m, -9);
  else v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return s ? -v : v;
}

static uint8_t e4m3_rne_nonneg(float v) {
  if (!(v > 0.0f)) return 0;
  if (v >= 448.0f) return 0x7E; /* satfinite */
  if (v < 0.015625f) {        /* below 2^-6: subnormal, step 2^-9 */
    float m = nearbyintf(ldexpf(v, 9));
    return (uint8_t)m;           /* m == 8 is exactly the smallest normal's code */
  }
  int e;
  float f = frexpf(v, &e);        /* v = f * 2^e, f in [0.5, 1) */
  int E = e - 1;                  /* v = 1.xxx * 2^E */
  float r = nearbyintf(ldexpf(f, 4)); /* 16 * f in [8, 16] */
  if (r == 16.0f) { r = 8.0f; E += 1; }
  int code = ((E + 7) << 3) | ((int)r - 8);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)code;
}

/* Encode rows x cols fp32 values (cols % 16 == 0). codes: rows*cols/2 bytes, low
 * nibble = even column.  sf: rows*cols/16 E4M3 bytes.  Returns the tensor scale. */
float synth_nvfp4_encode(const float* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf) {
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * cols; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float ts = amax / (6.0f * 448.0f);
  int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* xb = x + r * cols + b * 16;
      float bmax = 0.0f;
      for (int j = 0; j < 16; ++j) {
        float a = fabsf(xb[j]);
        if (a > bmax) bmax = a;
      }
      uint8_t s = (ts > 0.0f) ? e4m3_rne_nonneg(bmax / (6.0f * ts)) : 0;
      sf[r * nb + b] = s;
      float denom = e4m3_value(s) * ts;
      for (int j = 0; j < 16; j += 2) {
        uint8_t c0 = 0, c1 = 0;
        if (s != 0) {
          c0 = e2m1_rne(xb[j] / denom);
          c1 = e2m1_rne(xb[j + 1] / denom);
        }
        codes[(r * cols + b * 16 + j) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
  return ts;
}

/* Draw an N(0, std^2) matrix as fp32 and encode it (scratch: rows*cols floats). */
float synth_nvfp4_matrix(uint64_t seed, uint64_t stream, int64_t rows, int64_t cols, double std,
                         uint8_t* codes, uint8_t* sf, float* scratch) {
  synth_normal_f32(seed, stream, (uint64_t)(rows * cols), 0.0, std, scratch);
  return synth_nvfp4_encode(scratch, rows, cols, codes, sf);
}

/* Uniform integer in [0, n) for element i of a stream (n < 2^32; multiply-shift). */
static uint32_t uniform_below(uint64_t seed, uint64_t stream, uint64_t i, uint32_t n) {
  uint32_t w[4];
  draw_block(seed, stream, i, w);
  return (uint32_t)(((uint64_t)w[0] * n) >> 32);
}

/* Draft tree of n nodes: parent[0] = -1, parent[i] uniform in [0, i). */
void synth_parent(uint64_t seed, uint64_t stream, int n, int32_t* parent) {
  parent[0] = -1;
  for (int i = 1; i < n; ++i) parent[i] = (int32_t)uniform_below(seed, stream, (uint64_t)i, (uint32_t)i);
}

/* m distinct values from [0, n), in the order drawn (partial Fisher-Yates). */
void synth_subset(uint64_t seed, uint64_t stream, int n, int m, int32_t* out) {
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  for (int i = 0; i < n; ++i) perm[i] = i;
  for (int i = 0; i < m; ++i) {
    int j = i + (int)uniform_below(seed, stream, (uint64_t)i, (uint32_t)(n - i));
    int32_t t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
    out[i] = perm[i];
  }
  free(perm);
}

/* Bernoulli(p) draws, p given as a 32-bit threshold fraction. */
void synth_bernoulli(uint64_t seed, uint64_t stream, uint64_t n, double p, uint8_t* out) {
  uint64_t thr = (uint64_t)(p * 4294967296.0);
  for (uint64_t i = 0; i < n; ++i) {
    uint32_t w[4];
    draw_block(seed, stream, i, w);
    out[i] = ((uint64_t)w[0] < thr) ? 1 : 0;
  }
}

uint16_t synth_bf16_from_double(double x) { return bf16_bits_rne(x); }
