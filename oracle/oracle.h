/*
 * CPU oracle for one speculative-decoding verify step of a batch-1 MoE decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this code: only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition of the layer the pages describe
 * (orcarouter.ai, "Muse Spark Open: 1,109 tokens/s is a kernel-level change", §
 * "where the kernel boundary sits" and § "three bills"; alphasignal.ai, "LMSYS
 * Doubles Muse Spark Open Speed to 1,109 Tokens per Second", § "Draft and verify
 * share one graph"): a 16-token draft tree is verified in one pass through every
 * decoder layer (tree-masked attention over the KV history, sliding-window or
 * global), output projection, pooler, router top-k, two NVFP4 expert GEMMs with
 * SwiGLU, combine, unpooler; then the final norm and LM head.
 *
 * Arithmetic: fp64 throughout, rounded to bf16 exactly at the materialisation
 * points listed in or_layer(); the first expert GEMM reads the bf16 pooled
 * vector as it is; the NVFP4 quantiser of the SwiGLU output (the second expert
 * GEMM's input) takes its decisions in fp32 (the precision the GPU path uses)
 * with a per-row scale of amax / (6 * 448) rounded up to a power of two; router
 * logits are rounded to fp32 before the top-k decision.
 *
 * Layouts (all row-major, bf16 stored as uint16 bit patterns):
 *   w_qkv   [(Hq + 2 Hkv) * D][d]   rows: q heads, then k heads, then v heads
 *   w_o     [d][Hq * D]
 *   w_pool  [P][d]
 *   w_router[E][P], b_router fp32 [E]
 *   w_unpool[d][P]
 *   norm_*  [d]
 *   w1      NVFP4 [E][2F][P]: codes [E][2F][P/2] (low nibble = even column),
 *           scales E4M3 [E][2F][P/16], per-expert fp32 tensor scale [E];
 *           rows [0, F) are the SwiGLU gate, rows [F, 2F) the up projection
 *   w2      NVFP4 [E][P][F] likewise
 *   KV cache per layer: [Hkv][max_ctx][D]; tree token i is stored at row pos0+i
 */
#ifndef MSM_ORACLE_H
#define MSM_ORACLE_H
#include <stdint.h>

#define OR_T 16 /* tokens in the verification tree */

typedef struct {
  int d, hq, hkv, hd, p, f, e, k;
  int window;   /* sliding window W for SWA layers */
  int max_ctx;  /* KV rows per layer */
  double rms_eps, rope_theta;
} or_dims;

typedef struct {
  const uint16_t *w_qkv, *w_o, *w_pool, *w_router, *w_unpool, *norm_attn, *norm_moe;
  const float* b_router;
  const uint8_t *w1_codes, *w1_sf, *w2_codes, *w2_sf;
  const float *w1_gs, *w2_gs;
} or_layer_weights;

/* Optional per-layer observables for tests (any pointer may be NULL). */
typedef struct {
  int32_t* topk_idx;   /* [16][k] */
  float* topk_w;       /* [16][k] */
  float* router_logits;/* [16][E] (fp32-rounded) */
  uint16_t* attn_out;  /* [16][Hq*D] bf16 */
  uint16_t* h_mid;     /* [16][d]  bf16 residual after attention */
  uint16_t* pooled;    /* [16][P]  bf16 */
  uint16_t* q_out;     /* [16][Hq*D] bf16 (post-RoPE) */
  uint16_t* moe_z;     /* [16][P]  bf16 combined expert output (before the unpooler) */
} or_layer_trace;

#ifdef __cplusplus
extern "C" {
#endif

/* number formats */
double or_bf16_round(double x);
double or_bf16_value(uint16_t bits);
uint16_t or_bf16_bits(double x);
double or_e2m1_value(uint8_t nibble);
double or_e4m3_value(uint8_t code);
uint8_t or_e2m1_encode(float v);
uint8_t or_e4m3_encode(float v);
float or_nvfp4_quantize(const float* x, int n, uint8_t* codes, uint8_t* sf);
void or_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, float ts, int n, double* out);

/* the tree: ancestor-or-self bitmask and depth; returns 0, or -1 if parent is invalid */
int or_tree_mask(const int32_t* parent, int n, uint32_t* anc, int32_t* depth);

/* building blocks */
void or_rmsnorm(const double* x, const uint16_t* gain, int n, double eps, double* y);
void or_rope(double* v, int hd, double pos, double theta);
void or_topk(const float* logits, int n, int k, int32_t* idx, double* w);
void or_attention(const or_dims* dm, int window, const double* q, const uint16_t* k_cache,
                  const uint16_t* v_cache, const uint32_t* anc, const int32_t* tpos, int32_t pos0,
                  double* out);
void or_attention_masked(int hd, int n_keys, const double* q, const double* keys,
                         const double* vals, const uint8_t* mask, double* out);

/* one decoder layer; returns 0 or -1 on invalid arguments */
int or_layer(const or_dims* dm, const or_layer_weights* w, int is_global, const uint16_t* h_in,
             uint16_t* h_out, const int32_t* parent, int32_t pos0, uint16_t* k_cache,
             uint16_t* v_cache, or_layer_trace* trace);

/* final RMSNorm + LM head: logits fp32 [16][vocab] */
void or_lm_head(const or_dims* dm, const uint16_t* norm_final, const uint16_t* w_lm, int vocab,
                const uint16_t* h, float* logits);

int or_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
