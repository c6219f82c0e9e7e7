/*
 * CPU oracle for the verify step — TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Plain loops in fp64.  Parallel loops (OpenMP) only split independent outputs;
 * no blocking, fusion or reordering of any single output's arithmetic beyond
 * what the definition states.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bf16: 1 sign, 8 exponent, 7 stored mantissa bits (fp32's upper half).     */
/* Rounding is to nearest, ties to even, directly from fp64.                 */
/* ------------------------------------------------------------------------ */
double or_bf16_round(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x);
  int e;
  double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
  double r;
  if (e - 1 < -126) {
    r = ldexp(nearbyint(ldexp(a, 133)), -133); /* bf16 subnormal quantum 2^-133 */
  } else {
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8);  /* 8 significant bits */
  }
  if (r > 3.3895313892515355e38) r = INFINITY;
  return x < 0 ? -r : r;
}

double or_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t or_bf16_bits(double x) {
  float f = (float)or_bf16_round(x); /* exact */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 = E2M1 elements, one E4M3 scale per 16 consecutive elements, and one */
/* fp32 tensor scale (orcarouter.ai page, § "where the kernel boundary sits": */
/* experts stored in 4-bit NVFP4).                                           */
/* ------------------------------------------------------------------------ */
double or_e2m1_value(uint8_t nib) {
  /* sign bit 3; exponent bits 2..1 (bias 1); mantissa bit 0; e=0 is subnormal */
  int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

double or_e4m3_value(uint8_t c) {
  /* sign bit 7; exponent bits 6..3 (bias 7); mantissa bits 2..0; no infinities;
     S.1111.111 is NaN; e=0 is subnormal with step 2^-9 */
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest representable value, ties to the even code, saturating at +-6. */
uint8_t or_e2m1_encode(float v) {
  uint8_t sign = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(or_e2m1_value((uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
  }
  if (a >= 6.0) best = 7;
  return sign | (uint8_t)best;
}

/* Nearest non-negative E4M3 value, ties to the even code, saturating at 448. */
uint8_t or_e4m3_encode(float v) {
  double a = (double)v;
  if (!(a > 0.0)) return 0;
  if (a >= 448.0) return 0x7E;
  int best = 0;
  double bd = a;
  for (int c = 1; c <= 0x7E; ++c) {
    double d = fabs(or_e4m3_value((uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
  }
  return (uint8_t)best;
}

/* Smallest power of two >= x (0 for x <= 0). */
static float pow2_ceil(float x) {
  if (!(x > 0.0f)) return 0.0f;
  int e;
  float m = frexpf(x, &e); /* x = m 2^e, m in [0.5, 1) */
  return (m == 0.5f) ? x : ldexpf(1.0f, e);
}

/* Quantise one row of n fp32 values (n % 16 == 0) to NVFP4.  The per-row fp32
 * scale is amax / (6 * 448) rounded up to a power of two, so that every block
 * scale fits E4M3 and a tiny change of the row's largest element cannot move
 * the scale of every block; every decision below is taken in fp32. */
float or_nvfp4_quantize(const float* x, int n, uint8_t* codes, uint8_t* sf) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  volatile float ts = pow2_ceil(amax / 2688.0f); /* 6 * 448 */
  for (int b = 0; b < n / 16; ++b) {
    float bmax = 0.0f;
    for (int j = 0; j < 16; ++j) {
      float a = fabsf(x[b * 16 + j]);
      if (a > bmax) bmax = a;
    }
    uint8_t s = 0;
    if (ts > 0.0f) {
      volatile float six_ts = 6.0f * ts;
      s = or_e4m3_encode(bmax / six_ts);
    }
    sf[b] = s;
    volatile float denom = (float)or_e4m3_value(s) * ts;
    for (int j = 0; j < 16; j += 2) {
      uint8_t c0 = 0, c1 = 0;
      if (s != 0) {
        c0 = or_e2m1_encode(x[b * 16 + j] / denom);
        c1 = or_e2m1_encode(x[b * 16 + j + 1] / denom);
      }
      codes[(b * 16 + j) / 2] = (uint8_t)(c0 | (c1 << 4));
    }
  }
  return ts;
}

/* Decoded values of every E2M1 nibble and E4M3 byte, filled from the two
 * definitions above on first use (lookups only; no other arithmetic). */
static double g_e2m1_tab[16], g_e4m3_tab[256];
static int g_tabs_ready = 0;
static void fill_tables(void) {
  if (g_tabs_ready) return;
#pragma omp critical(or_tables)
  {
    if (!g_tabs_ready) {
      for (int i = 0; i < 16; ++i) g_e2m1_tab[i] = or_e2m1_value((uint8_t)i);
      for (int i = 0; i < 256; ++i) g_e4m3_tab[i] = or_e4m3_value((uint8_t)i);
      g_tabs_ready = 1;
    }
  }
}

void or_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, float ts, int n, double* out) {
  fill_tables();
  for (int i = 0; i < n; ++i) {
    uint8_t byte = codes[i / 2];
    uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);
    out[i] = g_e2m1_tab[nib] * g_e4m3_tab[sf[i / 16]] * (double)ts;
  }
}

/* ------------------------------------------------------------------------ */
/* Verification tree (alphasignal.ai page, § "Draft and verify share one      */
/* graph": the target checks a 16-token tree proposed by the draft; the      */
/* orcarouter.ai page, § draft model: a candidate tree, not a linear chain).  */
/* Token i may attend to tree token j iff j is i or an ancestor of i.  The   */
/* root has parent -1 and every other node a parent with a smaller index.    */
/* ------------------------------------------------------------------------ */
int or_tree_mask(const int32_t* parent, int n, uint32_t* anc, int32_t* depth) {
  if (n < 1 || n > 32 || parent[0] != -1) return -1;
  for (int i = 1; i < n; ++i)
    if (parent[i] < 0 || parent[i] >= i) return -1;
  for (int i = 0; i < n; ++i) {
    uint32_t m = 0;
    int dpt = 0;
    for (int j = i; j != -1; j = parent[j]) { /* explicit walk to the root */
      m |= 1u << j;
      if (j != i) ++dpt;
    }
    anc[i] = m;
    depth[i] = dpt;
  }
  return 0;
}

/* y = bf16( x / sqrt(mean(x^2) + eps) * gain ) */
void or_rmsnorm(const double* x, const uint16_t* gain, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = or_bf16_round(x[i] * inv * or_bf16_value(gain[i]));
}

/* Rotary embedding, rotate-half pairing (i, i + D/2), angle pos * theta^(-2i/D). */
void or_rope(double* v, int hd, double pos, double theta) {
  int h = hd / 2;
  for (int i = 0; i < h; ++i) {
    double ang = pos * pow(theta, -2.0 * i / hd);
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + h];
    v[i] = a * c - b * s;
    v[i + h] = b * c + a * s;
  }
}

/* Top-k by value, larger first, equal values to the lower index; weights are
 * the softmax over the k selected logits. */
void or_topk(const float* logits, int n, int k, int32_t* idx, double* w) {
  unsigned char* used = (unsigned char*)calloc((size_t)n, 1);
  for (int c = 0; c < k; ++c) {
    int best = -1;
    for (int e = 0; e < n; ++e) {
      if (used[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e;
    }
    used[best] = 1;
    idx[c] = best;
  }
  free(used);
  double mx = logits[idx[0]], sum = 0.0;
  for (int c = 0; c < k; ++c) sum += exp((double)logits[idx[c]] - mx);
  for (int c = 0; c < k; ++c) w[c] = exp((double)logits[idx[c]] - mx) / sum;
}

/* Attention of one query row over n_keys rows with an explicit 0/1 mask. */
void or_attention_masked(int hd, int n_keys, const double* q, const double* keys,
                         const double* vals, const uint8_t* mask, double* out) {
  double scale = 1.0 / sqrt((double)hd);
  double mx = -INFINITY;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  for (int j = 0; j < n_keys; ++j) {
    s[j] = -INFINITY;
    if (!mask[j]) continue;
    double acc = 0.0;
    for (int t = 0; t < hd; ++t) acc += q[t] * keys[(size_t)j * hd + t];
    s[j] = acc * scale;
    if (s[j] > mx) mx = s[j];
  }
  double den = 0.0;
  for (int t = 0; t < hd; ++t) out[t] = 0.0;
  for (int j = 0; j < n_keys; ++j) {
    if (!mask[j]) continue;
    double p = exp(s[j] - mx);
    den += p;
    for (int t = 0; t < hd; ++t) out[t] += p * vals[(size_t)j * hd + t];
  }
  for (int t = 0; t < hd; ++t) out[t] = den > 0.0 ? out[t] / den : 0.0;
  free(s);
}

/* Tree attention (orcarouter.ai page, § "where the kernel boundary sits": 46
 * layers attend over the most recent 2,048 tokens, 16 globally).  Query i of
 * head h (kv head h / (Hq/Hkv)) sees history row r < pos0 when the layer is
 * global or tpos[i] - r < window, and tree row pos0 + j when j is i or one of
 * its ancestors.  q: [16][Hq][D]; out: [16][Hq*D] (not rounded here). */
void or_attention(const or_dims* dm, int window, const double* q, const uint16_t* k_cache,
                  const uint16_t* v_cache, const uint32_t* anc, const int32_t* tpos, int32_t pos0,
                  double* out) {
  const int D = dm->hd, group = dm->hq / dm->hkv;
  const double scale = 1.0 / sqrt((double)D);
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int i = 0; i < OR_T; ++i) {
    for (int h = 0; h < dm->hq; ++h) {
      const int hk = h / group;
      const double* qv = q + ((size_t)i * dm->hq + h) * D;
      const uint16_t* K = k_cache + (size_t)hk * dm->max_ctx * D;
      const uint16_t* V = v_cache + (size_t)hk * dm->max_ctx * D;
      int n_rows = pos0 + OR_T;
      double* s = (double*)malloc(sizeof(double) * (size_t)n_rows);
      double mx = -INFINITY;
      for (int r = 0; r < n_rows; ++r) {
        int visible;
        if (r < pos0) visible = (window <= 0) || (tpos[i] - r < window);
        else visible = (anc[i] >> (r - pos0)) & 1u;
        s[r] = -INFINITY;
        if (!visible) continue;
        double acc = 0.0;
        for (int t = 0; t < D; ++t) acc += qv[t] * or_bf16_value(K[(size_t)r * D + t]);
        s[r] = acc * scale;
        if (s[r] > mx) mx = s[r];
      }
      double den = 0.0;
      double* o = out + (size_t)i * dm->hq * D + (size_t)h * D;
      for (int t = 0; t < D; ++t) o[t] = 0.0;
      for (int r = 0; r < n_rows; ++r) {
        if (s[r] == -INFINITY) continue;
        double p = exp(s[r] - mx);
        den += p;
        for (int t = 0; t < D; ++t) o[t] += p * or_bf16_value(V[(size_t)r * D + t]);
      }
      for (int t = 0; t < D; ++t) o[t] /= den;
      free(s);
    }
  }
}

/* out[t][n] = sum_k x[t][k] * W[n][k] for the 16 tokens; W bf16 [N][K]. */
static void matmul_bf16(const double* x, const uint16_t* W, int N, int K, double* out) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    const uint16_t* wr = W + (size_t)n * K;
    for (int t = 0; t < OR_T; ++t) {
      double acc = 0.0;
      const double* xr = x + (size_t)t * K;
      for (int k = 0; k < K; ++k) acc += xr[k] * or_bf16_value(wr[k]);
      out[(size_t)t * N + n] = acc;
    }
  }
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------ */
/* One decoder layer, h_in -> h_out, with the bf16 materialisation points:   */
/*   xn  = bf16(RMSNorm(h; g_attn))                                          */
/*   q,k,v = bf16(RoPE(xn W_qkv^T))   (RoPE on q and k at tree positions)    */
/*   K/V rows of tree token i -> cache row pos0 + i                          */
/*   O   = bf16(tree attention)                                              */
/*   h1  = bf16(h + bf16(O W_o^T))                                           */
/*   u   = bf16(bf16(RMSNorm(h1; g_moe)) W_pool^T)                           */
/*   logits = fp32(u W_r^T + b); top-k; w = softmax over the selected k      */
/*   per slot: [g | v] = u W1_e^T (bf16 u, NVFP4 weights); a = silu(g) v;   */
/*             a_q = NVFP4(fp32(a)); y = bf16(a_q W2_e^T)                    */
/*   z   = bf16(sum_slots w y)                                               */
/*   h2  = bf16(h1 + bf16(z W_unp^T))                                        */
/* Pages: the orcarouter.ai page, § "where the kernel boundary sits" (router  */
/* top-8 of 256, pooler before the experts, unpooler after, NVFP4 experts);  */
/* the alphasignal.ai page, § "Launch boundaries leave hardware idle" (the    */
/* chain attention -> ... -> next layer's QKV projection and KV write).       */
/* Precision of the expert GEMMs (same orcarouter.ai section): what leaves   */
/* the first expert GEMM is exchanged as fp4 and what leaves the second as   */
/* bf16.  Read plainly: GEMM1 takes the pooler's bf16 output as it is, its   */
/* SwiGLU result is quantised to NVFP4 before GEMM2, and GEMM2's output is   */
/* bf16.  Nothing on the pages quantises the pooled vector itself.           */
/* ------------------------------------------------------------------------ */
int or_layer(const or_dims* dm, const or_layer_weights* w, int is_global, const uint16_t* h_in,
             uint16_t* h_out, const int32_t* parent, int32_t pos0, uint16_t* k_cache,
             uint16_t* v_cache, or_layer_trace* tr) {
  const int d = dm->d, Hq = dm->hq, Hkv = dm->hkv, D = dm->hd, P = dm->p, F = dm->f,
            E = dm->e, K = dm->k;
  const int NQ = Hq * D, NKV = Hkv * D, NQKV = NQ + 2 * NKV;
  if (pos0 < 0 || pos0 + OR_T > dm->max_ctx || Hq % Hkv != 0 || P % 16 || F % 16) return -1;
  uint32_t anc[OR_T];
  int32_t depth[OR_T], tpos[OR_T];
  if (or_tree_mask(parent, OR_T, anc, depth) != 0) return -1;
  for (int i = 0; i < OR_T; ++i) tpos[i] = pos0 + depth[i];

  double* h = (double*)malloc(sizeof(double) * OR_T * d);
  double* xn = (double*)malloc(sizeof(double) * OR_T * d);
  double* qkv = (double*)malloc(sizeof(double) * OR_T * NQKV);
  double* q = (double*)malloc(sizeof(double) * OR_T * NQ);
  double* att = (double*)malloc(sizeof(double) * OR_T * NQ);
  double* tmp = (double*)malloc(sizeof(double) * OR_T * (d > P ? d : P));
  double* h1 = (double*)malloc(sizeof(double) * OR_T * d);
  double* u = (double*)malloc(sizeof(double) * OR_T * P);
  double* z = (double*)calloc((size_t)OR_T * P, sizeof(double));

  for (int i = 0; i < OR_T * d; ++i) h[i] = or_bf16_value(h_in[i]);

  /* attention half */
  for (int t = 0; t < OR_T; ++t) or_rmsnorm(h + t * d, w->norm_attn, d, dm->rms_eps, xn + t * d);
  matmul_bf16(xn, w->w_qkv, NQKV, d, qkv);
  for (int t = 0; t < OR_T; ++t) {
    double* row = qkv + (size_t)t * NQKV;
    for (int hh = 0; hh < Hq; ++hh) or_rope(row + hh * D, D, (double)tpos[t], dm->rope_theta);
    for (int hh = 0; hh < Hkv; ++hh) or_rope(row + NQ + hh * D, D, (double)tpos[t], dm->rope_theta);
    for (int c = 0; c < NQKV; ++c) row[c] = or_bf16_round(row[c]);
    for (int c = 0; c < NQ; ++c) q[(size_t)t * NQ + c] = row[c];
    for (int hh = 0; hh < Hkv; ++hh)
      for (int c = 0; c < D; ++c) {
        size_t dst = ((size_t)hh * dm->max_ctx + pos0 + t) * D + c;
        k_cache[dst] = or_bf16_bits(row[NQ + hh * D + c]);
        v_cache[dst] = or_bf16_bits(row[NQ + NKV + hh * D + c]);
      }
  }
  or_attention(dm, is_global ? 0 : dm->window, q, k_cache, v_cache, anc, tpos, pos0, att);
  for (int i = 0; i < OR_T * NQ; ++i) att[i] = or_bf16_round(att[i]);
  matmul_bf16(att, w->w_o, d, NQ, tmp);
  for (int i = 0; i < OR_T * d; ++i) h1[i] = or_bf16_round(h[i] + or_bf16_round(tmp[i]));

  /* MoE half */
  for (int t = 0; t < OR_T; ++t) or_rmsnorm(h1 + t * d, w->norm_moe, d, dm->rms_eps, xn + t * d);
  matmul_bf16(xn, w->w_pool, P, d, u);
  for (int i = 0; i < OR_T * P; ++i) u[i] = or_bf16_round(u[i]);

  double* lg = (double*)malloc(sizeof(double) * OR_T * E);
  matmul_bf16(u, w->w_router, E, P, lg);
  float* lgf = (float*)malloc(sizeof(float) * OR_T * E);
  for (int t = 0; t < OR_T; ++t)
    for (int e = 0; e < E; ++e) lgf[t * E + e] = (float)(lg[t * E + e] + (double)w->b_router[e]);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * OR_T * K);
  double* wt = (double*)malloc(sizeof(double) * OR_T * K);
  for (int t = 0; t < OR_T; ++t) or_topk(lgf + t * E, E, K, idx + t * K, wt + t * K);

  /* experts: every (token, slot) pair independently */
  fill_tables();
  double* y = (double*)malloc(sizeof(double) * OR_T * K * P);
#pragma omp parallel for schedule(dynamic)
  for (int ts = 0; ts < OR_T * K; ++ts) {
    const int t = ts / K, e = idx[ts];
    const uint8_t* c1 = w->w1_codes + (size_t)e * 2 * F * P / 2;
    const uint8_t* s1 = w->w1_sf + (size_t)e * 2 * F * P / 16;
    const uint8_t* c2 = w->w2_codes + (size_t)e * P * F / 2;
    const uint8_t* s2 = w->w2_sf + (size_t)e * P * F / 16;
    double* wrow = (double*)malloc(sizeof(double) * (P > F ? P : F));
    double* gv = (double*)malloc(sizeof(double) * 2 * F);
    float* a = (float*)malloc(sizeof(float) * F);
    uint8_t* aq_c = (uint8_t*)malloc((size_t)F / 2);
    uint8_t* aq_s = (uint8_t*)malloc((size_t)F / 16);
    double* adq = (double*)malloc(sizeof(double) * F);
    for (int r = 0; r < 2 * F; ++r) {
      or_nvfp4_dequant(c1 + (size_t)r * P / 2, s1 + (size_t)r * P / 16, w->w1_gs[e], P, wrow);
      double acc = 0.0;
      for (int c = 0; c < P; ++c) acc += u[(size_t)t * P + c] * wrow[c];
      gv[r] = acc;
    }
    for (int j = 0; j < F; ++j) a[j] = (float)(silu(gv[j]) * gv[F + j]);
    float ats = or_nvfp4_quantize(a, F, aq_c, aq_s);
    or_nvfp4_dequant(aq_c, aq_s, ats, F, adq);
    for (int r = 0; r < P; ++r) {
      or_nvfp4_dequant(c2 + (size_t)r * F / 2, s2 + (size_t)r * F / 16, w->w2_gs[e], F, wrow);
      double acc = 0.0;
      for (int c = 0; c < F; ++c) acc += adq[c] * wrow[c];
      y[(size_t)ts * P + r] = or_bf16_round(acc);
    }
    free(wrow); free(gv); free(a); free(aq_c); free(aq_s); free(adq);
  }
  for (int t = 0; t < OR_T; ++t)
    for (int r = 0; r < P; ++r) {
      double acc = 0.0;
      for (int c = 0; c < K; ++c) acc += wt[t * K + c] * y[((size_t)t * K + c) * P + r];
      z[(size_t)t * P + r] = or_bf16_round(acc);
    }
  matmul_bf16(z, w->w_unpool, d, P, tmp);
  for (int i = 0; i < OR_T * d; ++i) h_out[i] = or_bf16_bits(h1[i] + or_bf16_round(tmp[i]));

  if (tr) {
    if (tr->topk_idx) memcpy(tr->topk_idx, idx, sizeof(int32_t) * OR_T * K);
    if (tr->topk_w)
      for (int i = 0; i < OR_T * K; ++i) tr->topk_w[i] = (float)wt[i];
    if (tr->router_logits) memcpy(tr->router_logits, lgf, sizeof(float) * OR_T * E);
    if (tr->attn_out)
      for (int i = 0; i < OR_T * NQ; ++i) tr->attn_out[i] = or_bf16_bits(att[i]);
    if (tr->h_mid)
      for (int i = 0; i < OR_T * d; ++i) tr->h_mid[i] = or_bf16_bits(h1[i]);
    if (tr->pooled)
      for (int i = 0; i < OR_T * P; ++i) tr->pooled[i] = or_bf16_bits(u[i]);
    if (tr->q_out)
      for (int i = 0; i < OR_T * NQ; ++i) tr->q_out[i] = or_bf16_bits(q[i]);
    if (tr->moe_z)
      for (int i = 0; i < OR_T * P; ++i) tr->moe_z[i] = or_bf16_bits(z[i]);
  }
  free(h); free(xn); free(qkv); free(q); free(att); free(tmp); free(h1); free(u); free(z);
  free(lg); free(lgf); free(idx); free(wt);
  free(y);
  return 0;
}

/* logits = fp32( bf16(RMSNorm(h; g_final)) W_lm^T ) */
void or_lm_head(const or_dims* dm, const uint16_t* norm_final, const uint16_t* w_lm, int vocab,
                const uint16_t* h, float* logits) {
  const int d = dm->d;
  double* x = (double*)malloc(sizeof(double) * OR_T * d);
  double* xn = (double*)malloc(sizeof(double) * OR_T * d);
  double* out = (double*)malloc(sizeof(double) * (size_t)OR_T * vocab);
  for (int i = 0; i < OR_T * d; ++i) x[i] = or_bf16_value(h[i]);
  for (int t = 0; t < OR_T; ++t) or_rmsnorm(x + t * d, norm_final, d, dm->rms_eps, xn + t * d);
  matmul_bf16(xn, w_lm, vocab, d, out);
  for (size_t i = 0; i < (size_t)OR_T * vocab; ++i) logits[i] = (float)out[i];
  free(x); free(xn); free(out);
}
