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

#include "synth_defs.h"

static void draw_block(uint64_t seed, uint64_t stream, uint64_t block, uint32_t out[4]) {
  synth_draw(seed, stream, block, out);
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

static uint16_t bf16_bits_rne(double x) { return synth_bf16_rne(x); }

void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                      double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = synth_value(seed, stream, (uint64_t)i, mean, std);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                      float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = (float)synth_value(seed, stream, (uint64_t)i, mean, std);
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                       uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = bf16_bits_rne(synth_value(seed, stream, (uint64_t)i, mean, std));
}

/* ---- NVFP4 encoding of synthetic weights (input preparation) ----------------
 * E2M1 magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7, bit 3 = sign).
 * E4M3 (OCP "FN" variant): bias 7, no infinities, max 448, subnormal step 2^-9.
 * Encoding recipe for one matrix [rows][cols], blocks of 16 along cols:
 *   tensor scale ts = amax / (6 * 448)                          (fp32)
 *   block scale  s  = E4M3_rne(amax_block / (6 * ts))           (fp32 in)
 *   code         c  = E2M1_rne(x / (decode(s) * ts)), 0 if s == 0
 */
#define e2m1_rne synth_e2m1_rne
#define e4m3_value synth_e4m3_value
#define e4m3_rne_nonneg synth_e4m3_rne

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
