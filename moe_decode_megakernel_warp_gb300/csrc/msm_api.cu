// Host runtime and C ABI of libmsm (declared in include/msm.h).
//
// A model packs the caller's weights once, owns the exchange buffers the layer
// launches hand data through, and enqueues one persistent kernel launch per
// decoder layer for every verify step (alphasignal.ai, "LMSYS Doubles Muse
// Spark Open Speed to 1,109 Tokens per Second": each layer runs as one kernel,
// § "Launch boundaries leave hardware idle").
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "msm.h"
#include "msm_internal.h"

namespace msm {
cudaError_t launch_pack_dense(const void* W, void* out, int N, int K, int kind, int hd, int hq, int hkv,
                              cudaStream_t s);
cudaError_t launch_pack_nvfp4(const void* codes, const void* sf, void* out, int E, int rows, int K, int swiglu,
                              int F, cudaStream_t s);
cudaError_t launch_fill_u32(void* p, uint64_t n, uint32_t v, cudaStream_t s);
}  // namespace msm

using namespace msm;

namespace {
thread_local std::string g_err;

msm_status fail(msm_status st, const std::string& msg) {
  g_err = msg;
  return st;
}
msm_status cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorString(e);
  return e == cudaErrorMemoryAllocation ? MSM_ERR_OOM : MSM_ERR_CUDA;
}
#define CK(call)                                   \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

struct LayerPack {
  uint8_t *qkv = nullptr, *o = nullptr, *pool = nullptr, *router = nullptr, *unpool = nullptr, *w1 = nullptr,
          *w2 = nullptr;
  uint8_t *up = nullptr, *down = nullptr;  // draft models: FFN gate+up (paired rows) and down
  float *b = nullptr, *w1gs = nullptr, *w2gs = nullptr;
  uint16_t *g_attn = nullptr, *g_moe = nullptr;
};
}  // namespace

struct msm_model {
  int device = 0;
  msm_config cfg{};
  Dims dm{};
  std::vector<uint8_t> global;
  int G = 0, ring_bytes = 0, act_bytes = 0, smem_bytes = 0;
  int g1_b_off = 0, g2_off = 0, ring_ext = 0, unpool_act_off = 0, unpool_ext = 0, sfb_ext = 0, attn_act_off = 0, kv_ext = 0;
  std::vector<LayerPack> L;
  uint8_t* lm = nullptr;
  uint16_t* g_final = nullptr;
  std::vector<void*> allocs;
  uint8_t* x[2] = {nullptr, nullptr};
  uint8_t* sbuf = nullptr;
  XOffsets xo{};
  SOffsets so{};
  uint16_t* in_q[2] = {nullptr, nullptr};
  uint16_t* in_h[2] = {nullptr, nullptr};
  float* rope = nullptr;
  double* inv_freq = nullptr;
  int32_t* routing_idx = nullptr;
  float* routing_w = nullptr;
  uint32_t* hist = nullptr;
  uint32_t* tree_dbg = nullptr;
  uint64_t* timing = nullptr;
  DevStatus* status = nullptr;
  uint64_t packed_bytes = 0;
  uint64_t launch_count = 0, step_count = 0;
  std::vector<CUtensorMap> tmk, tmv;
  std::vector<const void*> tmk_ptr, tmv_ptr;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  cudaStream_t aux = nullptr;
  uint16_t* io_in = nullptr;      // device staging of msm_verify_step_host
  uint16_t* io_hidden = nullptr;
  float* io_logits = nullptr;
  CUtensorMap tma_act[2][5];  // dense activations of each exchange parity (ActMap order)
  int act_box[5] = {0, 0, 0, 0, 0};
  bool act_tma = false;
  // msm_verify_step_noalloc: device address of the static scratch array (looked up at
  // creation, which also loads the module that holds it), the bytes one step needs
  // there, and the activation tensor maps of its two exchange parities
  unsigned char* noalloc = nullptr;
  uint64_t noalloc_need = 0;
  CUtensorMap tma_act_na[2][5];
  bool act_tma_na = false;
  uint64_t launches_run = 0;   // launches enqueued by every verify entry point
  uint8_t* last_x = nullptr;   // exchange buffer of the last launch enqueued
  uint64_t* accept_part = nullptr;  // msm_accept: argmax partial keys [16][G], then
  int32_t* accept_choice = nullptr; // the 16 greedy choices [16] and
  uint32_t* accept_ticket = nullptr;  // the last-block ticket (zero between calls)

  template <class Tp>
  cudaError_t alloc(Tp** p, uint64_t bytes) {
    void* v = nullptr;
    cudaError_t e = cudaMalloc(&v, bytes ? bytes : 256);
    if (e == cudaSuccess) allocs.push_back(v);
    *p = static_cast<Tp*>(v);
    return e;
  }
};

namespace {

// a draft model (MSM_FLAG_DRAFT): dense SwiGLU FFN layers, full attention
msm_status validate_draft_config(const msm_config* c) {
  if (c->d_model <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->ffn_dim <= 0 ||
      c->n_layers <= 0 || c->max_ctx < T || c->vocab <= 0)
    return fail(MSM_ERR_INVALID_ARG, "draft config: non-positive size (vocab is required)");
  if (c->pool_dim != 0 || c->n_experts != 0 || c->top_k != 0)
    return fail(MSM_ERR_INVALID_ARG, "draft config: pool_dim, n_experts and top_k must be 0");
  if (c->n_q_heads % c->n_kv_heads) return fail(MSM_ERR_INVALID_ARG, "config: n_q_heads % n_kv_heads != 0");
  const int group = c->n_q_heads / c->n_kv_heads;
  if (c->head_dim != 64 && c->head_dim != 128) return fail(MSM_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (group != 1 && group != 2 && group != 4 && group != 8)
    return fail(MSM_ERR_UNSUPPORTED, "n_q_heads / n_kv_heads must be 1, 2, 4 or 8");
  if (c->d_model % 64 || (c->n_q_heads * c->head_dim) % 64)
    return fail(MSM_ERR_UNSUPPORTED, "d_model and n_q_heads*head_dim must be multiples of 64");
  if (c->ffn_dim % 128) return fail(MSM_ERR_UNSUPPORTED, "draft ffn_dim must be a multiple of 128 (two staged K halves)");
  // each K half's weight tiles must start on a packed 1024-column tile (or lie in one)
  if (c->ffn_dim > 1024 && c->ffn_dim % 2048)
    return fail(MSM_ERR_UNSUPPORTED, "draft ffn_dim above 1024 must be a multiple of 2048");
  if (c->vocab % 16) return fail(MSM_ERR_UNSUPPORTED, "vocab must be a multiple of 16");
  if (c->grid_blocks < 0 || c->attn_splits < 0) return fail(MSM_ERR_INVALID_ARG, "config: negative grid_blocks / attn_splits");
  if (c->flags & (MSM_FLAG_EXPERT_PREFETCH | MSM_FLAG_KV_PREFETCH))
    return fail(MSM_ERR_INVALID_ARG, "draft config: the expert and KV prefetch flags do not apply");
  return MSM_OK;
}

msm_status validate_config(const msm_config* c) {
  if (!c) return fail(MSM_ERR_INVALID_ARG, "config is NULL");
  if (c->flags & MSM_FLAG_DRAFT) return validate_draft_config(c);
  if (c->d_model <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->pool_dim <= 0 ||
      c->ffn_dim <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->n_layers <= 0 || c->max_ctx < T ||
      c->vocab < 0 || c->window <= 0 || !c->layer_is_global)
    return fail(MSM_ERR_INVALID_ARG, "config: non-positive size or missing layer_is_global");
  if (c->top_k > c->n_experts) return fail(MSM_ERR_INVALID_ARG, "config: top_k > n_experts");
  if (c->n_q_heads % c->n_kv_heads) return fail(MSM_ERR_INVALID_ARG, "config: n_q_heads % n_kv_heads != 0");
  const int group = c->n_q_heads / c->n_kv_heads;
  if (c->head_dim != 64 && c->head_dim != 128) return fail(MSM_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (group != 1 && group != 2 && group != 4 && group != 8)
    return fail(MSM_ERR_UNSUPPORTED, "n_q_heads / n_kv_heads must be 1, 2, 4 or 8");
  if (c->d_model % 64 || c->pool_dim % 64 || c->ffn_dim % 64 || (c->n_q_heads * c->head_dim) % 64)
    return fail(MSM_ERR_UNSUPPORTED, "d_model, pool_dim, ffn_dim, n_q_heads*head_dim must be multiples of 64");
  if (c->pool_dim % kExpBlockK || c->ffn_dim % kExpBlockK)
    return fail(MSM_ERR_UNSUPPORTED, "pool_dim and ffn_dim must be multiples of 256 (expert tensor-core tiles)");
  if (c->ffn_dim > 1024) return fail(MSM_ERR_UNSUPPORTED, "ffn_dim > 1024 (activation scales in tensor memory)");
  if (c->pool_dim > 2048) return fail(MSM_ERR_UNSUPPORTED, "pool_dim > 2048 (activation scales in tensor memory)");
  if (c->top_k > kMaxTopK) return fail(MSM_ERR_UNSUPPORTED, "top_k > 8");
  if (c->n_experts > kMaxExperts || c->n_experts % 16) return fail(MSM_ERR_UNSUPPORTED, "n_experts must be <= 256 and a multiple of 16");
  if (c->vocab % 16) return fail(MSM_ERR_UNSUPPORTED, "vocab must be a multiple of 16");
  if (c->l2_runahead_kb < 0 || c->l2_runahead_kb > (1 << 20))
    return fail(MSM_ERR_INVALID_ARG, "config: l2_runahead_kb outside [0, 1 GiB]");
  if (c->grid_blocks < 0 || c->attn_splits < 0 || c->prefetch_experts < 0)
    return fail(MSM_ERR_INVALID_ARG, "config: negative grid_blocks / attn_splits / prefetch_experts");
  return MSM_OK;
}

bool parent_valid(const int32_t* parent) {
  if (!parent || parent[0] != -1) return false;
  for (int i = 1; i < T; ++i)
    if (parent[i] < 0 || parent[i] >= i) return false;
  return true;
}

msm_status encode_kv_map(msm_model* m, CUtensorMap* map, const void* ptr) {
  const Dims& dm = m->dm;
  cuuint64_t dims[3] = {(cuuint64_t)dm.hd, (cuuint64_t)dm.max_ctx, (cuuint64_t)dm.hkv};
  cuuint64_t strides[2] = {(cuuint64_t)dm.hd * 2, (cuuint64_t)dm.max_ctx * dm.hd * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)dm.kv_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = m->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MSM_ERR_CUDA, "cuTensorMapEncodeTiled failed for a KV cache");
  return MSM_OK;
}

// sentinels (bf16 0xFFFF, fp32 -0.0) in one exchange buffer, its counters zeroed
msm_status arm_exchange(uint8_t* x, const XOffsets& o, cudaStream_t s) {
  CK(launch_fill_u32(x, o.logits / 4, 0xFFFFFFFFu, s));                       // o, h1, u
  CK(launch_fill_u32(x + o.logits, (o.z - o.logits) / 4, 0x80000000u, s));    // logits, a
  CK(launch_fill_u32(x + o.z, (o.cnt - o.z) / 4, 0xFFFFFFFFu, s));            // z, h2, q0, tkv0
  CK(launch_fill_u32(x + o.cnt, (o.b1 - o.cnt) / 4, 0u, s));                  // counters
  return MSM_OK;
}

// tensor maps of the five dense activations of one exchange buffer (ActMap order);
// false if the driver rejects one (the kernel then stages with plain loads)
bool encode_act_maps(msm_model* m, uint8_t* x, CUtensorMap* maps) {
  const Dims& dm = m->dm;
  const XOffsets& xo = m->xo;
  // (a draft model: the two K halves of its FFN activation, [2][16][f/2], in place of u, z)
  const uint64_t zh = (uint64_t)T * (dm.f / 2) * 2;
  const uint64_t offs[5] = {xo.o, xo.h1, dm.draft ? xo.z : xo.u, dm.draft ? xo.z + zh : xo.z, xo.h2};
  const int kz = dm.draft ? dm.f / 2 : dm.p;
  const int ks[5] = {dm.hq * dm.hd, dm.d, kz, kz, dm.d};
  if (!m->encode) return false;
  for (int i = 0; i < 5; ++i) {
    const int nblk = ks[i] / 64;
    int nb = 8;
    while (nblk % nb) nb >>= 1;
    m->act_box[i] = nb;
    cuuint64_t dims[3] = {64, (cuuint64_t)T, (cuuint64_t)nblk};
    cuuint64_t strides[2] = {(cuuint64_t)ks[i] * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)T, (cuuint32_t)nb};
    cuuint32_t es[3] = {1, 1, 1};
    if (m->encode(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x + offs[i], dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// device address of the static scratch array on the current device (defined with the
// array, at the end of this file)
msm_status noalloc_lookup(unsigned char** base);

msm_status rearm_all(msm_model* m, cudaStream_t s) {
  for (int c = 0; c < 2; ++c) {
    msm_status st = arm_exchange(m->x[c], m->xo, s);
    if (st != MSM_OK) return st;
  }
  CK(launch_fill_u32(m->sbuf, m->so.y / 4, 0x80000000u, s));                    // part, ml
  CK(launch_fill_u32(m->sbuf + m->so.y, (m->so.total - m->so.y) / 4, 0xFFFFFFFFu, s));  // y
  return MSM_OK;
}

}  // namespace

extern "C" {

const char* msm_last_error(void) { return g_err.c_str(); }

msm_status msm_model_create(const msm_config* config, const msm_weights* w, int device, msm_model** out) {
  if (!out) return fail(MSM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  msm_status st = validate_config(config);
  if (st != MSM_OK) return st;
  if (!w) return fail(MSM_ERR_INVALID_ARG, "weights is NULL");
  const msm_config& c = *config;
  const bool draft = (c.flags & MSM_FLAG_DRAFT) != 0;
  if (draft) {
    if (!w->w_qkv || !w->w_o || !w->norm_attn || !w->norm_moe || !w->w_gate || !w->w_up || !w->w_down)
      return fail(MSM_ERR_INVALID_ARG, "draft weights: a per-layer pointer array is NULL");
    for (int l = 0; l < c.n_layers; ++l)
      if (!w->w_qkv[l] || !w->w_o[l] || !w->norm_attn[l] || !w->norm_moe[l] || !w->w_gate[l] || !w->w_up[l] || !w->w_down[l])
        return fail(MSM_ERR_INVALID_ARG, "draft weights: NULL pointer for layer " + std::to_string(l));
  } else {
    if (!w->w_qkv || !w->w_o || !w->w_pool || !w->w_router || !w->b_router || !w->w_unpool || !w->norm_attn ||
        !w->norm_moe || !w->w1_codes || !w->w1_scales || !w->w1_tensor_scale || !w->w2_codes || !w->w2_scales ||
        !w->w2_tensor_scale)
      return fail(MSM_ERR_INVALID_ARG, "weights: a per-layer pointer array is NULL");
    for (int l = 0; l < c.n_layers; ++l)
      if (!w->w_qkv[l] || !w->w_o[l] || !w->w_pool[l] || !w->w_router[l] || !w->b_router[l] || !w->w_unpool[l] ||
          !w->norm_attn[l] || !w->norm_moe[l] || !w->w1_codes[l] || !w->w1_scales[l] || !w->w1_tensor_scale[l] ||
          !w->w2_codes[l] || !w->w2_scales[l] || !w->w2_tensor_scale[l])
        return fail(MSM_ERR_INVALID_ARG, "weights: NULL pointer for layer " + std::to_string(l));
    for (int l = 0; l < c.n_layers; ++l)
      if ((reinterpret_cast<uintptr_t>(w->w1_codes[l]) | reinterpret_cast<uintptr_t>(w->w1_scales[l]) |
           reinterpret_cast<uintptr_t>(w->w2_codes[l]) | reinterpret_cast<uintptr_t>(w->w2_scales[l])) & 15)
        return fail(MSM_ERR_INVALID_ARG, "weights: NVFP4 codes and scales must be 16-byte aligned (layer " + std::to_string(l) + ")");
  }
  if (c.vocab > 0 && (!w->norm_final || !w->w_lm)) return fail(MSM_ERR_INVALID_ARG, "vocab > 0 needs norm_final and w_lm");

  int ndev = 0;
  CK(cudaGetDeviceCount(&ndev));
  if (device < 0 || device >= ndev) return fail(MSM_ERR_INVALID_ARG, "no such device");
  CK(cudaSetDevice(device));
  int sms = 0, smem_optin = 0, cc_major = 0, cc_minor = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
  CK(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device));
  CK(cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, device));
  CK(cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, device));
  if (cc_major != 10 || cc_minor != 3) return fail(MSM_ERR_UNSUPPORTED, "libmsm is built for sm_103a (GB300) only");

  msm_model* m = new msm_model();
  m->device = device;
  m->cfg = c;
  if (draft) m->global.assign(c.n_layers, 1);  // the draft attends to its whole history
  else m->global.assign(c.layer_is_global, c.layer_is_global + c.n_layers);
  m->cfg.layer_is_global = nullptr;
  Dims& dm = m->dm;
  dm.d = c.d_model; dm.hq = c.n_q_heads; dm.hkv = c.n_kv_heads; dm.hd = c.head_dim; dm.p = c.pool_dim;
  dm.f = c.ffn_dim; dm.e = c.n_experts; dm.k = c.top_k; dm.vocab = c.vocab; dm.max_ctx = c.max_ctx;
  dm.window = draft ? c.max_ctx : c.window; dm.n_layers = c.n_layers;
  dm.draft = draft ? 1 : 0;
  dm.nqkv = (dm.hq + 2 * dm.hkv) * dm.hd;
  dm.group = dm.hq / dm.hkv;
  dm.attn_rows = dm.hd == 128 ? 32 : 64;
  // two attention tiles per KV ring tile: half the loader's and the barriers' work per byte
  dm.kv_rows = dm.max_ctx >= 2 * dm.attn_rows ? 2 * dm.attn_rows : dm.attn_rows;
  if (draft) {
    // the draft kernel's attention: the 8 / group warps of a head take alternate KV tiles
    dm.attn_nk = dm.attn_rows;
    dm.attn_wph = std::max(1, 8 / dm.group);
  } else {
    dm.attn_nk = std::max(16, dm.attn_rows * dm.group / 8);
    dm.attn_wph = dm.attn_rows / dm.attn_nk;
  }
  dm.rms_eps = c.rms_eps;
  m->G = c.grid_blocks > 0 ? std::min(c.grid_blocks, sms) : sms;
  {
    // the kernel splits work units over the grid in 32-bit arithmetic
    const uint64_t units = std::max({(uint64_t)dm.vocab / 16, (uint64_t)dm.nqkv / 16, (uint64_t)dm.d / 16,
                                     (uint64_t)std::min(dm.e, T * dm.k) * std::max(w1_units(dm.f), w2_units(dm.p))});
    if (units * (uint64_t)(m->G + 1) >= (1ull << 32)) {
      delete m;
      return fail(MSM_ERR_UNSUPPORTED, "too many work units per phase for the grid split");
    }
  }
  dm.splits = c.attn_splits > 0 ? c.attn_splits : std::max(1, m->G / dm.hkv);
  if (dm.hkv * dm.splits > m->G) {
    delete m;
    return fail(MSM_ERR_INVALID_ARG, "attn_splits * n_kv_heads exceeds the grid");
  }
  // shared memory: ring | act | small
  const int D = dm.hd;
  const uint64_t attn_need = (uint64_t)dm.group * (D / 16) * kKStepBytes + 2ull * 16 * D * 2 +
                             (uint64_t)dm.group * dm.attn_wph * 32 * (4 + D / 2) * 4;
  // (a draft model stages its FFN activation in two K halves)
  const uint64_t kmax = (uint64_t)std::max(std::max(dm.d, dm.hq * dm.hd), draft ? dm.f / 2 : dm.p);
  // GEMM1: operand B, the split pooled vectors with their scale groups; GEMM2: two
  // experts' NVFP4 rows (E2M1 + scales) + one fp32 row per warp (both at the top of the
  // buffer; the router stages the bf16 pooled vectors at its bottom, dead once the
  // router phase has split them, before operand B is copied in)
  const uint64_t g1_need = draft ? 0 : b1_bytes(dm.p);
  const uint64_t g2_need = draft ? 0 : ((18ull * dm.f + 1023) & ~1023ull) + (uint64_t)kComputeWarps * dm.f * 4;
  uint64_t act = std::max(std::max(kmax * 32, g1_need), std::max(g2_need, attn_need));
  act = (act + 1023) & ~uint64_t(1023);
  const uint64_t expert_top = (std::max(g1_need, g2_need) + 1023) & ~uint64_t(1023);
  const int smem_cap = std::min(kMaxSmem, smem_optin);
  long long ring = (long long)smem_cap - (long long)act - kSmallBytes;
  ring &= ~1023ll;
  const uint64_t exp_tile = draft ? 0 : (uint64_t)std::max(exp_tile_bytes(dm.p), exp_tile_bytes(dm.f));
  const uint64_t max_tile = std::max(std::max((uint64_t)kDenseTileSteps * kKStepBytes, exp_tile), (uint64_t)dm.kv_rows * D * 4);
  if (ring < (long long)(2 * max_tile)) {
    delete m;
    return fail(MSM_ERR_UNSUPPORTED, "widths too large for the shared-memory budget");
  }
  m->act_bytes = (int)act;
  m->ring_bytes = (int)ring;
  // attention stages Q, the tree rows and its merge scratch at the top of the activation
  // buffer; the KV tiles of a launch after the first may use the rest as ring space
  m->attn_act_off = (int)(act - ((attn_need + 1023) & ~uint64_t(1023)));
  m->kv_ext = m->attn_act_off & ~1023;
  m->g1_b_off = (int)(act - ((g1_need + 1023) & ~uint64_t(1023)));
  m->g2_off = (int)(act - ((g2_need + 1023) & ~uint64_t(1023)));
  m->ring_ext = (int)((act - expert_top) & ~uint64_t(1023));
  // the unpooler stages its [16][pool_dim] input at the top; its tiles may use the rest
  // of the bottom, up to the expert phases' extension (so that no tile ever lands on
  // GEMM1's operand, which a block may still read while its loader is past GEMM2)
  m->unpool_act_off = (int)(act - (((uint64_t)dm.p * 32 + 1023) & ~uint64_t(1023)));
  m->unpool_ext = std::min(m->ring_ext, m->unpool_act_off);
  // GEMM1's operand-B scales are the bottom of its operand: when the operand is what sets
  // the top of the expert phases, the ring may grow over them once they are copied
  m->sfb_ext = (m->g1_b_off == m->ring_ext) ? (int)b1_sfb_bytes(dm.p) : 0;
  if (draft) m->ring_ext = m->unpool_ext = m->sfb_ext = 0;  // (no expert or unpooler tiles)
  m->smem_bytes = (int)(ring + act + kSmallBytes);

  auto bail = [&](msm_status s2) {
    msm_model_destroy(m);
    return s2;
  };
#define CKM(call)                                          \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return bail(cuda_fail(e_, #call)); \
  } while (0)

  CKM(cudaStreamCreateWithFlags(&m->aux, cudaStreamNonBlocking));
  for (int t = 0; t < 2; ++t)
    CKM(cudaFuncSetAttribute(layer_kernel(t != 0, draft), cudaFuncAttributeMaxDynamicSharedMemorySize, m->smem_bytes));
  int occ = 0;
  CKM(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, layer_kernel(false, draft), kThreads, m->smem_bytes));
  if (occ < 1) return bail(fail(MSM_ERR_UNSUPPORTED, "the layer kernel does not fit on an SM"));
  // the blocks of a launch wait on each other (phase counters, handoff slots), so all of
  // them must be resident at once: one block per SM, at most one per SM of the device
  if ((long long)m->G > (long long)sms * occ)
    return bail(fail(MSM_ERR_UNSUPPORTED, "grid larger than the blocks the device holds at once"));

  cudaDriverEntryPointQueryResult qr;
  void* fn = nullptr;
  CKM(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr));
  if (!fn || qr != cudaDriverEntryPointSuccess) return bail(fail(MSM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable"));
  m->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);

  // ---- pack weights ----
  cudaStream_t s = m->aux;
  m->L.resize(c.n_layers);
  const int u1pe = w1_units(dm.f), u2pe = w2_units(dm.p);
  if (draft) {
    // the FFN's gate and up projections go through one [2F][d] staging copy, packed with
    // gate row j and up row j in the same 16-row unit (rows 0-7 / 8-15) for the SwiGLU epilogue
    uint8_t* gu = nullptr;
    const uint64_t b_gu = 2ull * dm.f * dm.d * 2;
    CKM(cudaMalloc(&gu, b_gu));
    for (int l = 0; l < c.n_layers; ++l) {
      LayerPack& lp = m->L[l];
      const uint64_t b_qkv = (dm.nqkv / 16) * dense_unit_bytes(dm.d), b_o = (dm.d / 16) * dense_unit_bytes(dm.hq * dm.hd),
                     b_up = (2ull * dm.f / 16) * dense_unit_bytes(dm.d), b_down = (dm.d / 16) * dense_unit_bytes(dm.f);
      CKM(m->alloc(&lp.qkv, b_qkv));
      CKM(m->alloc(&lp.o, b_o));
      CKM(m->alloc(&lp.up, b_up));
      CKM(m->alloc(&lp.down, b_down));
      CKM(m->alloc(&lp.g_attn, dm.d * 2));
      CKM(m->alloc(&lp.g_moe, dm.d * 2));
      m->packed_bytes += b_qkv + b_o + b_up + b_down;
      CKM(launch_pack_dense(w->w_qkv[l], lp.qkv, dm.nqkv, dm.d, 1, dm.hd, dm.hq, dm.hkv, s));
      CKM(launch_pack_dense(w->w_o[l], lp.o, dm.d, dm.hq * dm.hd, 0, dm.hd, dm.hq, dm.hkv, s));
      CKM(cudaMemcpyAsync(gu, w->w_gate[l], b_gu / 2, cudaMemcpyDeviceToDevice, s));
      CKM(cudaMemcpyAsync(gu + b_gu / 2, w->w_up[l], b_gu / 2, cudaMemcpyDeviceToDevice, s));
      CKM(launch_pack_dense(gu, lp.up, 2 * dm.f, dm.d, 2, dm.hd, dm.hq, dm.hkv, s));
      CKM(launch_pack_dense(w->w_down[l], lp.down, dm.d, dm.f, 0, dm.hd, dm.hq, dm.hkv, s));
      CKM(cudaMemcpyAsync(lp.g_attn, w->norm_attn[l], dm.d * 2, cudaMemcpyDeviceToDevice, s));
      CKM(cudaMemcpyAsync(lp.g_moe, w->norm_moe[l], dm.d * 2, cudaMemcpyDeviceToDevice, s));
    }
    CKM(cudaStreamSynchronize(s));
    CKM(cudaFree(gu));
  }
  for (int l = 0; l < c.n_layers && !draft; ++l) {
    LayerPack& lp = m->L[l];
    const uint64_t b_qkv = (dm.nqkv / 16) * dense_unit_bytes(dm.d), b_o = (dm.d / 16) * dense_unit_bytes(dm.hq * dm.hd),
                   b_pool = (dm.p / 16) * dense_unit_bytes(dm.d), b_r = (dm.e / 16) * dense_unit_bytes(dm.p),
                   b_unp = (dm.d / 16) * dense_unit_bytes(dm.p),
                   b_w1 = (uint64_t)dm.e * u1pe * exp_unit_bytes(dm.p),
                   b_w2 = (uint64_t)dm.e * u2pe * exp_unit_bytes(dm.f);
    CKM(m->alloc(&lp.qkv, b_qkv));
    CKM(m->alloc(&lp.o, b_o));
    CKM(m->alloc(&lp.pool, b_pool));
    CKM(m->alloc(&lp.router, b_r));
    CKM(m->alloc(&lp.unpool, b_unp));
    CKM(m->alloc(&lp.w1, b_w1));
    CKM(m->alloc(&lp.w2, b_w2));
    CKM(m->alloc(&lp.b, dm.e * 4));
    CKM(m->alloc(&lp.w1gs, dm.e * 4));
    CKM(m->alloc(&lp.w2gs, dm.e * 4));
    CKM(m->alloc(&lp.g_attn, dm.d * 2));
    CKM(m->alloc(&lp.g_moe, dm.d * 2));
    m->packed_bytes += b_qkv + b_o + b_pool + b_r + b_unp + b_w1 + b_w2;
    CKM(launch_pack_dense(w->w_qkv[l], lp.qkv, dm.nqkv, dm.d, 1, dm.hd, dm.hq, dm.hkv, s));
    CKM(launch_pack_dense(w->w_o[l], lp.o, dm.d, dm.hq * dm.hd, 0, dm.hd, dm.hq, dm.hkv, s));
    CKM(launch_pack_dense(w->w_pool[l], lp.pool, dm.p, dm.d, 0, dm.hd, dm.hq, dm.hkv, s));
    CKM(launch_pack_dense(w->w_router[l], lp.router, dm.e, dm.p, 0, dm.hd, dm.hq, dm.hkv, s));
    CKM(launch_pack_dense(w->w_unpool[l], lp.unpool, dm.d, dm.p, 0, dm.hd, dm.hq, dm.hkv, s));
    CKM(launch_pack_nvfp4(w->w1_codes[l], w->w1_scales[l], lp.w1, dm.e, 2 * dm.f, dm.p, 1, dm.f, s));
    CKM(launch_pack_nvfp4(w->w2_codes[l], w->w2_scales[l], lp.w2, dm.e, dm.p, dm.f, 0, dm.f, s));
    CKM(cudaMemcpyAsync(lp.b, w->b_router[l], dm.e * 4, cudaMemcpyDeviceToDevice, s));
    CKM(cudaMemcpyAsync(lp.w1gs, w->w1_tensor_scale[l], dm.e * 4, cudaMemcpyDeviceToDevice, s));
    CKM(cudaMemcpyAsync(lp.w2gs, w->w2_tensor_scale[l], dm.e * 4, cudaMemcpyDeviceToDevice, s));
    CKM(cudaMemcpyAsync(lp.g_attn, w->norm_attn[l], dm.d * 2, cudaMemcpyDeviceToDevice, s));
    CKM(cudaMemcpyAsync(lp.g_moe, w->norm_moe[l], dm.d * 2, cudaMemcpyDeviceToDevice, s));
  }
  if (dm.vocab > 0) {
    const uint64_t b_lm = (dm.vocab / 16) * dense_unit_bytes(dm.d);
    CKM(m->alloc(&m->lm, b_lm));
    CKM(m->alloc(&m->g_final, dm.d * 2));
    m->packed_bytes += b_lm;
    CKM(launch_pack_dense(w->w_lm, m->lm, dm.vocab, dm.d, 0, dm.hd, dm.hq, dm.hkv, s));
    CKM(cudaMemcpyAsync(m->g_final, w->norm_final, dm.d * 2, cudaMemcpyDeviceToDevice, s));
  }

  // ---- exchange buffers ----
  XOffsets& xo = m->xo;
  uint64_t o = 0;
  xo.o = o; o += align256((uint64_t)T * dm.hq * dm.hd * 2);
  xo.h1 = o; o += align256((uint64_t)T * dm.d * 2);
  xo.u = o; o += align256((uint64_t)T * dm.p * 2);
  xo.logits = o; o += align256((uint64_t)T * dm.e * 4);
  xo.a = o; o += align256((uint64_t)T * dm.k * dm.f * 4);
  xo.z = o; o += align256((uint64_t)T * (draft ? dm.f : dm.p) * 2);  // (a draft's FFN activation)
  xo.h2 = o; o += align256((uint64_t)T * dm.d * 2);
  xo.q0 = o; o += align256((uint64_t)T * dm.hq * dm.hd * 2);
  xo.tkv0 = o; o += align256(2ull * dm.hkv * T * dm.hd * 2);
  xo.cnt = o; o += kCounterBytes;
  xo.b1 = o; o += align256(b1_bytes(dm.p));
  xo.total = o;
  SOffsets& so = m->so;
  o = 0;
  // (attention partials; a draft's first-half FFN-down partial sums reuse the space)
  so.part = o; o += align256(std::max((uint64_t)dm.hkv * dm.splits * T * dm.group * dm.hd * 4, (uint64_t)T * dm.d * 4));
  so.ml = o; o += align256((uint64_t)dm.hkv * dm.splits * T * dm.group * 2 * 4);
  so.y = o; o += align256((uint64_t)T * dm.k * dm.p * 2);
  so.total = o;
  CKM(m->alloc(&m->x[0], xo.total));
  CKM(m->alloc(&m->x[1], xo.total));
  CKM(m->alloc(&m->sbuf, so.total));
  for (int i = 0; i < 2; ++i) {
    CKM(m->alloc(&m->in_q[i], (uint64_t)T * dm.hq * dm.hd * 2));
    CKM(m->alloc(&m->in_h[i], (uint64_t)T * dm.d * 2));
  }
  // tensor maps of the dense activations for staging by tensor copies; if the driver
  // rejects one, every phase stages with plain loads instead
  m->act_tma = encode_act_maps(m, m->x[0], m->tma_act[0]) && encode_act_maps(m, m->x[1], m->tma_act[1]);
  {
    // the static scratch of msm_verify_step_noalloc: its address is looked up now, so
    // that loading the module holding it (and with it the array's device memory)
    // happens here and never inside a no-allocation call
    const uint64_t q_bytes = align256((uint64_t)T * dm.hq * dm.hd * 2), h_bytes = align256((uint64_t)T * dm.d * 2);
    m->noalloc_need = 2 * xo.total + so.total + 2 * q_bytes + 2 * h_bytes;
    st = noalloc_lookup(&m->noalloc);
    if (st != MSM_OK) return bail(st);
    if (m->noalloc_need <= (uint64_t)MSM_NOALLOC_SCRATCH_BYTES)
      m->act_tma_na = encode_act_maps(m, m->noalloc, m->tma_act_na[0]) &&
                      encode_act_maps(m, m->noalloc + xo.total, m->tma_act_na[1]);
  }
  CKM(m->alloc(&m->rope, (uint64_t)T * (dm.hd / 2) * 2 * 4));
  CKM(m->alloc(&m->inv_freq, (uint64_t)(dm.hd / 2) * 8));
  {
    std::vector<double> inv(dm.hd / 2);
    for (int i = 0; i < dm.hd / 2; ++i) inv[i] = std::pow((double)c.rope_theta, -2.0 * i / dm.hd);
    CKM(cudaMemcpyAsync(m->inv_freq, inv.data(), inv.size() * 8, cudaMemcpyHostToDevice, s));
    CKM(cudaStreamSynchronize(s));
  }
  CKM(m->alloc(&m->routing_idx, (uint64_t)c.n_layers * T * dm.k * 4));
  CKM(m->alloc(&m->routing_w, (uint64_t)c.n_layers * T * dm.k * 4));
  CKM(m->alloc(&m->hist, 2ull * c.n_layers * dm.e * 4));
  CKM(m->alloc(&m->tree_dbg, 32 * 4));
  CKM(m->alloc(&m->timing, (uint64_t)c.n_layers * m->G * kTimingEvents * 8));
  CKM(m->alloc(&m->status, sizeof(DevStatus)));
  CKM(m->alloc(&m->io_in, (uint64_t)T * dm.d * 2));
  CKM(m->alloc(&m->io_hidden, (uint64_t)T * dm.d * 2));
  if (dm.vocab > 0) CKM(m->alloc(&m->io_logits, (uint64_t)T * dm.vocab * 4));
  if (dm.vocab > 0) {
    CKM(m->alloc(&m->accept_part, (uint64_t)T * m->G * 8 + T * 4 + 16));
    m->accept_choice = reinterpret_cast<int32_t*>(m->accept_part + (size_t)T * m->G);
    m->accept_ticket = reinterpret_cast<uint32_t*>(m->accept_choice + T);
    CKM(cudaMemsetAsync(m->accept_ticket, 0, 4, s));
  }
  CKM(cudaMemsetAsync(m->hist, 0, 2ull * c.n_layers * dm.e * 4, s));
  CKM(cudaMemsetAsync(m->status, 0, sizeof(DevStatus), s));
  CKM(cudaMemsetAsync(m->timing, 0, (uint64_t)c.n_layers * m->G * kTimingEvents * 8, s));
  st = rearm_all(m, s);
  if (st != MSM_OK) return bail(st);
  CKM(cudaStreamSynchronize(s));
  m->tmk.resize(c.n_layers);
  m->tmv.resize(c.n_layers);
  m->tmk_ptr.assign(c.n_layers, nullptr);
  m->tmv_ptr.assign(c.n_layers, nullptr);
#undef CKM
  *out = m;
  return MSM_OK;
}

void msm_model_destroy(msm_model* m) {
  if (!m) return;
  cudaSetDevice(m->device);
  cudaDeviceSynchronize();
  for (void* p : m->allocs) cudaFree(p);
  if (m->aux) cudaStreamDestroy(m->aux);
  delete m;
}

}  // extern "C"

namespace {
// The per-step buffers a verify step hands data through: the model's own (their two
// exchange parities alternate launch by launch across steps, each launch re-arming the
// other one) or the static scratch of msm_verify_step_noalloc (both parities armed by
// the call, launch l uses parity l & 1).
struct StepBuffers {
  uint8_t* x[2];
  uint8_t* sbuf;
  uint16_t* in_q[2];
  uint16_t* in_h[2];
  const CUtensorMap (*tma_act)[5];  // [2][5], or null: plain-load staging
  bool model_owned;
};

StepBuffers own_buffers(msm_model* m) {
  StepBuffers b;
  for (int c = 0; c < 2; ++c) {
    b.x[c] = m->x[c];
    b.in_q[c] = m->in_q[c];
    b.in_h[c] = m->in_h[c];
  }
  b.sbuf = m->sbuf;
  b.tma_act = m->act_tma ? m->tma_act : nullptr;
  b.model_owned = true;
  return b;
}

// host-detectable errors of a verify step, found before anything is enqueued
msm_status validate_step(msm_model* m, const void* hidden_in, const int32_t* parent, int32_t pos0,
                         const int32_t* state, void* const* k_cache, void* const* v_cache, float* logits_out,
                         void* hidden_out) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  const Dims& dm = m->dm;
  if (!hidden_in || !k_cache || !v_cache) return fail(MSM_ERR_INVALID_ARG, "NULL hidden_in or cache array");
  if (!state) {
    if (!parent_valid(parent))
      return fail(MSM_ERR_INVALID_ARG, "parent must satisfy parent[0] == -1, 0 <= parent[i] < i");
    if (pos0 < 0 || (int64_t)pos0 + T > dm.max_ctx) return fail(MSM_ERR_INVALID_ARG, "pos0 out of range");
  } else if (reinterpret_cast<uintptr_t>(state) & 3) {
    return fail(MSM_ERR_INVALID_ARG, "state must be 4-byte aligned");
  }
  if (dm.vocab > 0 && !logits_out) return fail(MSM_ERR_INVALID_ARG, "logits_out is NULL but vocab > 0");
  if (dm.vocab == 0 && !hidden_out) return fail(MSM_ERR_INVALID_ARG, "hidden_out is NULL but vocab == 0");
  if ((reinterpret_cast<uintptr_t>(hidden_in) & 15) || (reinterpret_cast<uintptr_t>(hidden_out) & 15) ||
      (reinterpret_cast<uintptr_t>(logits_out) & 15))
    return fail(MSM_ERR_INVALID_ARG, "hidden / logits buffers must be 16-byte aligned");
  for (int l = 0; l < dm.n_layers; ++l) {
    if (!k_cache[l] || !v_cache[l]) return fail(MSM_ERR_INVALID_ARG, "NULL KV cache pointer");
    if ((reinterpret_cast<uintptr_t>(k_cache[l]) & 15) || (reinterpret_cast<uintptr_t>(v_cache[l]) & 15))
      return fail(MSM_ERR_INVALID_ARG, "KV caches must be 16-byte aligned");
  }
  return MSM_OK;
}

// the verify step with the tree and pos0 from the host (state == nullptr) or from a
// device-resident step state that the kernels validate
msm_status enqueue_verify(msm_model* m, const StepBuffers& B, const void* hidden_in, const int32_t* parent,
                          int32_t pos0, const int32_t* state, void* const* k_cache, void* const* v_cache,
                          float* logits_out, void* hidden_out, void* stream, bool draft_call = false) {
  msm_status vst = validate_step(m, hidden_in, parent, pos0, state, k_cache, v_cache, logits_out, hidden_out);
  if (vst != MSM_OK) return vst;
  if ((m->dm.draft != 0) != draft_call)
    return fail(MSM_ERR_INVALID_ARG, draft_call ? "msm_draft_step needs a model created with MSM_FLAG_DRAFT"
                                                : "a draft model (MSM_FLAG_DRAFT) runs with msm_draft_step only");
  const Dims& dm = m->dm;
  CK(cudaSetDevice(m->device));
  for (int l = 0; l < dm.n_layers; ++l) {
    if (m->tmk_ptr[l] != k_cache[l]) {
      msm_status st = encode_kv_map(m, &m->tmk[l], k_cache[l]);
      if (st != MSM_OK) return st;
      m->tmk_ptr[l] = k_cache[l];
    }
    if (m->tmv_ptr[l] != v_cache[l]) {
      msm_status st = encode_kv_map(m, &m->tmv[l], v_cache[l]);
      if (st != MSM_OK) return st;
      m->tmv_ptr[l] = v_cache[l];
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t tmo = (uint64_t)(m->cfg.timeout_us ? m->cfg.timeout_us : 200000u) * 1000ull;
  const int sp = (int)(m->step_count & 1);
  LaunchParams P;
  std::memset(&P, 0, sizeof(P));
  P.dm = dm;
  P.xo = m->xo;
  P.so = m->so;
  P.s_buf = B.sbuf;
  P.rope = m->rope;
  P.inv_freq = m->inv_freq;
  P.tree_dbg = m->tree_dbg;
  P.status = m->status;
  P.pos0 = pos0;
  P.ring_bytes = m->ring_bytes;
  P.act_bytes = m->act_bytes;
  P.g1_b_off = m->g1_b_off;
  P.g2_off = m->g2_off;
  P.ring_ext = m->ring_ext;
  P.sfb_ext = m->sfb_ext;
  P.unpool_act_off = m->unpool_act_off;
  P.attn_act_off = m->attn_act_off;
  P.kv_ext = m->kv_ext;
  P.unpool_ext = m->unpool_ext;
  P.flags = m->cfg.flags;
  P.timeout_ns_lo = (uint32_t)tmo;
  P.timeout_ns_hi = (uint32_t)(tmo >> 32);
  P.prefetch_experts = m->cfg.prefetch_experts > 0 ? m->cfg.prefetch_experts : 14;
  P.runahead_bytes = m->cfg.l2_runahead_kb > 0 ? (uint32_t)m->cfg.l2_runahead_kb * 1024u : 0u;
  P.phase_rot = 13;
  if (state) {
    P.state = state;
    P.pos0 = 0;
  } else {
    std::memcpy(P.parent, parent, sizeof(int32_t) * T);
  }
  P.hidden_in = static_cast<const uint16_t*>(hidden_in);
  P.logits = logits_out;
  const bool timing = (m->cfg.flags & MSM_FLAG_SELF_TIMING) != 0;
  const bool pdl = (m->cfg.flags & MSM_FLAG_PDL) != 0;
  for (int l = 0; l < dm.n_layers; ++l) {
    const LayerPack& lp = m->L[l];
    const bool first = l == 0, last = l == dm.n_layers - 1;
    const int c = B.model_owned ? (int)(m->launch_count & 1) : (l & 1);
    P.layer = l;
    P.first = first;
    P.last = last;
    P.is_global = m->global[l] != 0;
    P.next_global = last ? 0 : (m->global[l + 1] != 0);
    P.w_qkv_pro = first ? lp.qkv : nullptr;
    P.g_attn_pro = first ? lp.g_attn : nullptr;
    P.w_o = lp.o;
    P.w_pool = lp.pool;
    P.w_router = lp.router;
    P.b_router = lp.b;
    P.w_unpool = lp.unpool;
    P.g_moe = lp.g_moe;
    P.w1 = lp.w1;
    P.w2 = lp.w2;
    P.w1_gs = lp.w1gs;
    P.w2_gs = lp.w2gs;
    P.w_up = lp.up;
    P.w_down = lp.down;
    P.w_tail = last ? m->lm : m->L[l + 1].qkv;
    P.g_tail = last ? m->g_final : m->L[l + 1].g_attn;
    P.hidden_out = last ? static_cast<uint16_t*>(hidden_out) : nullptr;
    P.kc = static_cast<uint16_t*>(k_cache[l]);
    P.vc = static_cast<uint16_t*>(v_cache[l]);
    P.kc_next = last ? nullptr : static_cast<uint16_t*>(k_cache[l + 1]);
    P.vc_next = last ? nullptr : static_cast<uint16_t*>(v_cache[l + 1]);
    P.kc_pf = P.kc_next;
    P.vc_pf = P.vc_next;
    P.x_cur = B.x[c];
    P.x_next = B.x[c ^ 1];
    P.act_tma = B.tma_act ? 1 : 0;
    for (int i = 0; i < 5; ++i) {
      if (B.tma_act) P.tmap_act[i] = B.tma_act[c][i];
      P.act_box[i] = m->act_box[i];
    }
    P.in_q = B.in_q[c];
    P.in_h = B.in_h[c];
    P.out_q = B.in_q[c ^ 1];
    P.out_h = B.in_h[c ^ 1];
    P.routing_idx = m->routing_idx + (size_t)l * T * dm.k;
    P.routing_w = m->routing_w + (size_t)l * T * dm.k;
    P.hist_cur = m->hist + ((size_t)sp * dm.n_layers + l) * dm.e;
    P.hist_prev = m->step_count > 0 ? m->hist + ((size_t)(sp ^ 1) * dm.n_layers + l) * dm.e : nullptr;
    P.timing = m->timing + (size_t)l * m->G * kTimingEvents;
    P.tmap_k = m->tmk[l];
    P.tmap_v = m->tmv[l];

    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof(lc));
    lc.gridDim = dim3(m->G);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = m->smem_bytes;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl && !first) {
      attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[na].val.programmaticStreamSerializationAllowed = 1;
      ++na;
    }
    lc.attrs = na ? attr : nullptr;
    lc.numAttrs = na;
    void* args[] = {&P};
    cudaError_t e = cudaLaunchKernelExC(&lc, layer_kernel(timing, dm.draft != 0), args);
    if (e != cudaSuccess) return cuda_fail(e, "layer kernel launch");
    if (B.model_owned) ++m->launch_count;
    ++m->launches_run;
    m->last_x = B.x[c];
  }
  ++m->step_count;
  return MSM_OK;
}
}  // namespace

extern "C" {

msm_status msm_verify_step(msm_model* m, const void* hidden_in, const int32_t* parent, int32_t pos0,
                           void* const* k_cache, void* const* v_cache, float* logits_out, void* hidden_out,
                           void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  return enqueue_verify(m, own_buffers(m), hidden_in, parent, pos0, nullptr, k_cache, v_cache, logits_out, hidden_out,
                        stream);
}

msm_status msm_verify_step_dev(msm_model* m, const void* hidden_in, const int32_t* state, void* const* k_cache,
                               void* const* v_cache, float* logits_out, void* hidden_out, void* stream) {
  if (!state) return fail(MSM_ERR_INVALID_ARG, "state is NULL");
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  return enqueue_verify(m, own_buffers(m), hidden_in, nullptr, 0, state, k_cache, v_cache, logits_out, hidden_out,
                        stream);
}

msm_status msm_sync(msm_model* m, void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  CK(cudaSetDevice(m->device));
  CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  DevStatus ds;
  CK(cudaMemcpy(&ds, m->status, sizeof(ds), cudaMemcpyDeviceToHost));
  if (ds.code == 0) return MSM_OK;
  char buf[160];
  std::snprintf(buf, sizeof(buf), "device wait timed out (layer %d, phase %d, block %d)", ds.layer, ds.phase, ds.block);
  msm_status st = (ds.code == MSM_ERR_DEVICE_TIMEOUT) ? MSM_ERR_DEVICE_TIMEOUT
                  : (ds.code == MSM_ERR_INVALID_ARG) ? MSM_ERR_INVALID_ARG : MSM_ERR_CUDA;
  if (ds.code == MSM_ERR_INVALID_ARG)
    std::snprintf(buf, sizeof(buf), "device-resident step state invalid (pos0, parent or token ids)");
  else if (ds.code != MSM_ERR_DEVICE_TIMEOUT)
    std::snprintf(buf, sizeof(buf), "device error %d (phase %d)", ds.code, ds.phase);
  // re-arm every exchange buffer and clear the status for the next step
  msm_status r = rearm_all(m, m->aux);
  if (r != MSM_OK) return r;
  CK(cudaMemsetAsync(m->status, 0, sizeof(DevStatus), m->aux));
  CK(cudaStreamSynchronize(m->aux));
  return fail(st, buf);
}

msm_status msm_verify_step_host(msm_model* m, const void* hidden_in_host, const int32_t* parent, int32_t pos0,
                                void* const* k_cache, void* const* v_cache, float* logits_host,
                                void* hidden_out_host, void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  const Dims& dm = m->dm;
  if (!hidden_in_host) return fail(MSM_ERR_INVALID_ARG, "hidden_in_host is NULL");
  if (dm.vocab > 0 && !logits_host) return fail(MSM_ERR_INVALID_ARG, "logits_host is NULL but vocab > 0");
  if (dm.vocab == 0 && !hidden_out_host) return fail(MSM_ERR_INVALID_ARG, "hidden_out_host is NULL but vocab == 0");
  CK(cudaSetDevice(m->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t h_bytes = (size_t)T * dm.d * 2, l_bytes = (size_t)T * dm.vocab * 4;
  CK(cudaMemcpyAsync(m->io_in, hidden_in_host, h_bytes, cudaMemcpyHostToDevice, s));
  msm_status st = msm_verify_step(m, m->io_in, parent, pos0, k_cache, v_cache, dm.vocab > 0 ? m->io_logits : nullptr,
                                  hidden_out_host ? m->io_hidden : nullptr, stream);
  if (st != MSM_OK) return st;
  if (dm.vocab > 0) CK(cudaMemcpyAsync(logits_host, m->io_logits, l_bytes, cudaMemcpyDeviceToHost, s));
  if (hidden_out_host) CK(cudaMemcpyAsync(hidden_out_host, m->io_hidden, h_bytes, cudaMemcpyDeviceToHost, s));
  return msm_sync(m, stream);
}

msm_status msm_get_routing(msm_model* m, int32_t* idx, float* w) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  CK(cudaSetDevice(m->device));
  CK(cudaDeviceSynchronize());
  const size_t n = (size_t)m->dm.n_layers * T * m->dm.k;
  if (idx) CK(cudaMemcpy(idx, m->routing_idx, n * 4, cudaMemcpyDeviceToHost));
  if (w) CK(cudaMemcpy(w, m->routing_w, n * 4, cudaMemcpyDeviceToHost));
  return MSM_OK;
}

msm_status msm_get_tree(msm_model* m, uint32_t* anc, int32_t* tpos) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  CK(cudaSetDevice(m->device));
  CK(cudaDeviceSynchronize());
  uint32_t buf[32];
  CK(cudaMemcpy(buf, m->tree_dbg, sizeof(buf), cudaMemcpyDeviceToHost));
  if (anc) std::memcpy(anc, buf, 16 * 4);
  if (tpos) std::memcpy(tpos, buf + 16, 16 * 4);
  return MSM_OK;
}

msm_status msm_get_timing(msm_model* m, uint64_t* buf, size_t n) {
  if (!m || !buf) return fail(MSM_ERR_INVALID_ARG, "model or buffer is NULL");
  const size_t need = (size_t)m->dm.n_layers * m->G * kTimingEvents;
  if (n < need) return fail(MSM_ERR_INVALID_ARG, "timing buffer too small");
  CK(cudaSetDevice(m->device));
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(buf, m->timing, need * 8, cudaMemcpyDeviceToHost));
  return MSM_OK;
}

msm_status msm_get_stats(const msm_model* m, msm_stats* out) {
  if (!m || !out) return fail(MSM_ERR_INVALID_ARG, "model or out is NULL");
  out->grid_blocks = m->G;
  out->threads_per_block = kThreads;
  out->smem_bytes = m->smem_bytes;
  out->attn_splits = m->dm.splits;
  out->launches_per_step = m->dm.n_layers;
  out->cooperative = 0;
  out->packed_weight_bytes = m->packed_bytes;
  out->exchange_bytes = 2 * m->xo.total + m->so.total;
  out->tma_act_staging = m->act_tma ? 1 : 0;
  out->launches_run = m->launches_run;
  out->noalloc_scratch_bytes = m->noalloc_need;
  return MSM_OK;
}

msm_status msm_get_exchange(msm_model* m, const char* name, void* host, size_t bytes) {
  if (!m || !name || !host) return fail(MSM_ERR_INVALID_ARG, "model, name or buffer is NULL");
  if (m->last_x == nullptr) return fail(MSM_ERR_INVALID_ARG, "no step has run");
  const XOffsets& o = m->xo;
  struct { const char* n; uint64_t off, len; } tab[] = {
      {"o", o.o, (uint64_t)T * m->dm.hq * m->dm.hd * 2}, {"h1", o.h1, (uint64_t)T * m->dm.d * 2},
      {"u", o.u, (uint64_t)T * m->dm.p * 2},            {"logits", o.logits, (uint64_t)T * m->dm.e * 4},
      {"a", o.a, (uint64_t)T * m->dm.k * m->dm.f * 4},  {"z", o.z, (uint64_t)T * m->dm.p * 2},
      {"h2", o.h2, (uint64_t)T * m->dm.d * 2}};
  for (auto& e : tab) {
    if (std::strcmp(e.n, name) != 0) continue;
    if (bytes < e.len) return fail(MSM_ERR_INVALID_ARG, "buffer too small");
    CK(cudaSetDevice(m->device));
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(host, m->last_x + e.off, e.len, cudaMemcpyDeviceToHost));
    return MSM_OK;
  }
  return fail(MSM_ERR_INVALID_ARG, std::string("unknown exchange buffer ") + name);
}

}  // extern "C"

namespace {
// the draft step: the n_layers layer launches (the block a chain at pos0, or at the
// state's pos0), the argmax of each slot, and either tokens_out (slot 0 = -1) or the
// proposal written into the state (the chain and tokens 1..15)
msm_status enqueue_draft(msm_model* m, const void* hidden_in, int32_t pos0, int32_t* state, void* const* k_cache,
                         void* const* v_cache, float* logits_out, int32_t* tokens_out, void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  if (!logits_out || (!state && !tokens_out))
    return fail(MSM_ERR_INVALID_ARG, "logits_out and tokens_out (or a state) are required");
  if ((reinterpret_cast<uintptr_t>(tokens_out) & 3) || (reinterpret_cast<uintptr_t>(state) & 3))
    return fail(MSM_ERR_INVALID_ARG, "tokens_out and state must be 4-byte aligned");
  // the slots form a chain (slot i at pos0 + i); the kernels give every slot the whole
  // block, so the chain only fixes the positions
  int32_t chain[T];
  for (int i = 0; i < T; ++i) chain[i] = i - 1;
  msm_status st = enqueue_verify(m, own_buffers(m), hidden_in, chain, pos0, state, k_cache, v_cache, logits_out,
                                 nullptr, stream, true);
  if (st != MSM_OK) return st;
  // each slot's argmax (the smallest index among equal maxima)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (state) {
    CK(launch_accept_argmax(logits_out, m->dm.vocab, m->accept_part, m->G, m->accept_ticket, m->accept_choice, s));
    CK(launch_draft_propose(m->accept_choice, state, s));
  } else {
    CK(launch_accept_argmax(logits_out, m->dm.vocab, m->accept_part, m->G, m->accept_ticket, tokens_out, s));
    CK(cudaMemsetAsync(tokens_out, 0xFF, sizeof(int32_t), s));
  }
  return MSM_OK;
}

msm_status enqueue_embed(msm_model* m, const void* table, const int32_t* state, void* hidden_out, void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  if (!table || !state || !hidden_out) return fail(MSM_ERR_INVALID_ARG, "NULL table, state or hidden_out");
  if (m->dm.vocab <= 0) return fail(MSM_ERR_UNSUPPORTED, "the embedding needs vocab > 0");
  if ((reinterpret_cast<uintptr_t>(table) & 15) || (reinterpret_cast<uintptr_t>(hidden_out) & 15) ||
      (reinterpret_cast<uintptr_t>(state) & 3))
    return fail(MSM_ERR_INVALID_ARG, "table and hidden_out must be 16-byte and state 4-byte aligned");
  CK(cudaSetDevice(m->device));
  CK(launch_embed(table, m->dm.vocab, m->dm.d, state, hidden_out, m->status, static_cast<cudaStream_t>(stream)));
  return MSM_OK;
}

msm_status enqueue_accept(msm_model* m, const float* logits, const int32_t* tokens, const int32_t* parent,
                          int32_t pos0, const int32_t* state, void* const* k_cache, void* const* v_cache,
                          int32_t* result, void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  const Dims& dm = m->dm;
  if (dm.vocab <= 0) return fail(MSM_ERR_UNSUPPORTED, "accept needs the LM head (vocab > 0)");
  if (dm.draft) return fail(MSM_ERR_INVALID_ARG, "a draft model (MSM_FLAG_DRAFT) runs with msm_draft_step only");
  if (!logits || !result || !k_cache || !v_cache)
    return fail(MSM_ERR_INVALID_ARG, "NULL logits, result or cache array");
  if (!state) {
    if (!tokens) return fail(MSM_ERR_INVALID_ARG, "tokens is NULL");
    if (!parent_valid(parent))
      return fail(MSM_ERR_INVALID_ARG, "parent must satisfy parent[0] == -1, 0 <= parent[i] < i");
    for (int i = 0; i < T; ++i)
      if (tokens[i] < 0 || tokens[i] >= dm.vocab) return fail(MSM_ERR_INVALID_ARG, "token id out of [0, vocab)");
    if (pos0 < 0 || (int64_t)pos0 + T > dm.max_ctx) return fail(MSM_ERR_INVALID_ARG, "pos0 out of range");
  } else if (reinterpret_cast<uintptr_t>(state) & 3) {
    return fail(MSM_ERR_INVALID_ARG, "state must be 4-byte aligned");
  }
  if ((reinterpret_cast<uintptr_t>(logits) & 15) || (reinterpret_cast<uintptr_t>(result) & 3))
    return fail(MSM_ERR_INVALID_ARG, "logits must be 16-byte and result 4-byte aligned");
  for (int l = 0; l < dm.n_layers; ++l) {
    if (!k_cache[l] || !v_cache[l]) return fail(MSM_ERR_INVALID_ARG, "NULL KV cache pointer");
    if ((reinterpret_cast<uintptr_t>(k_cache[l]) & 15) || (reinterpret_cast<uintptr_t>(v_cache[l]) & 15))
      return fail(MSM_ERR_INVALID_ARG, "KV caches must be 16-byte aligned");
  }
  CK(cudaSetDevice(m->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CK(launch_accept_argmax(logits, dm.vocab, m->accept_part, m->G, m->accept_ticket, m->accept_choice, s));
  AcceptParams p;
  std::memset(&p, 0, sizeof(p));
  p.choice = m->accept_choice;
  if (state) {
    p.state = state;
  } else {
    std::memcpy(p.parent, parent, sizeof(p.parent));
    std::memcpy(p.tokens, tokens, sizeof(p.tokens));
    p.pos0 = pos0;
  }
  p.status = m->status;
  p.vocab = dm.vocab;
  p.n_kv_heads = dm.hkv;
  p.head_dim = dm.hd;
  p.max_ctx = dm.max_ctx;
  for (int l0 = 0; l0 < dm.n_layers; l0 += kAcceptLayers) {
    p.n_layers = std::min(kAcceptLayers, dm.n_layers - l0);
    for (int l = 0; l < p.n_layers; ++l) {
      p.kc[l] = static_cast<uint16_t*>(k_cache[l0 + l]);
      p.vc[l] = static_cast<uint16_t*>(v_cache[l0 + l]);
    }
    p.result = l0 == 0 ? result : nullptr;
    const int cols = p.n_layers * 2 * dm.hkv * (dm.hd / 8);
    const int blocks = std::max(1, std::min(m->G, (cols + 255) / 256));  // 256 threads per block
    CK(launch_accept_walk(p, blocks, s));
  }
  return MSM_OK;
}
}  // namespace

extern "C" {

msm_status msm_accept(msm_model* m, const float* logits, const int32_t* tokens, const int32_t* parent,
                      int32_t pos0, void* const* k_cache, void* const* v_cache, int32_t* result, void* stream) {
  return enqueue_accept(m, logits, tokens, parent, pos0, nullptr, k_cache, v_cache, result, stream);
}

msm_status msm_accept_dev(msm_model* m, const float* logits, const int32_t* state, void* const* k_cache,
                          void* const* v_cache, int32_t* result, void* stream) {
  if (!state) return fail(MSM_ERR_INVALID_ARG, "state is NULL");
  return enqueue_accept(m, logits, nullptr, nullptr, 0, state, k_cache, v_cache, result, stream);
}

struct msm_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = 0;
};

void msm_graph_destroy(msm_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

}  // extern "C"

namespace {
// the draft model's part of a speculative-step graph
struct SpecArgs {
  msm_model* draft;
  const void* draft_hidden_in;
  void* const* dk;
  void* const* dv;
  float* draft_logits;
  const void* embed_table;
  int32_t* state;
};

msm_status capture_step(msm_model* m, const void* hidden_in, const int32_t* parent, const int32_t* tokens,
                        int32_t pos0, const int32_t* state, void* const* k_cache, void* const* v_cache,
                        float* logits_out, void* hidden_out, int32_t* accept_result, msm_graph** out,
                        const SpecArgs* spec = nullptr) {
  if (!out) return fail(MSM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  if (spec && spec->draft->device != m->device)
    return fail(MSM_ERR_INVALID_ARG, "the draft and target models must be on one device");
  CK(cudaSetDevice(m->device));
  cudaStream_t cs = nullptr;
  CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "cudaStreamBeginCapture");
  }
  // the graph arms both parities of the exchange buffers before its launches and
  // again after them, so a replay neither depends on nor leaves behind state that
  // an eager step of either launch parity (odd layer counts) could trip over; the
  // capture leaves the model's launch counters as they were
  msm_model* const dr = spec ? spec->draft : nullptr;
  const uint64_t launches0 = m->launch_count, steps0 = m->step_count, run0 = m->launches_run;
  uint8_t* const last_x0 = m->last_x;
  const uint64_t d_launches0 = dr ? dr->launch_count : 0, d_steps0 = dr ? dr->step_count : 0,
                 d_run0 = dr ? dr->launches_run : 0;
  uint8_t* const d_last_x0 = dr ? dr->last_x : nullptr;
  msm_status st = rearm_all(m, cs);
  if (st == MSM_OK && dr) {
    // draft -> its proposal in the state -> the tokens' embedding rows -> verify -> accept
    st = rearm_all(dr, cs);
    if (st == MSM_OK)
      st = enqueue_draft(dr, spec->draft_hidden_in, 0, spec->state, spec->dk, spec->dv, spec->draft_logits, nullptr,
                         cs);
    if (st == MSM_OK) st = enqueue_embed(m, spec->embed_table, spec->state, const_cast<void*>(hidden_in), cs);
  }
  if (st == MSM_OK)
    st = enqueue_verify(m, own_buffers(m), hidden_in, parent, pos0, state, k_cache, v_cache, logits_out, hidden_out,
                        cs);
  if (st == MSM_OK && accept_result)
    st = enqueue_accept(m, logits_out, tokens, parent, pos0, state, k_cache, v_cache, accept_result, cs);
  if (st == MSM_OK) st = rearm_all(m, cs);
  if (st == MSM_OK && dr) st = rearm_all(dr, cs);
  // recording runs nothing: the model's launch parity must keep following the
  // launches that did run (a replay arms both parities, so it needs no count)
  m->launch_count = launches0;
  m->step_count = steps0;
  m->launches_run = run0;
  m->last_x = last_x0;
  if (dr) {
    dr->launch_count = d_launches0;
    dr->step_count = d_steps0;
    dr->launches_run = d_run0;
    dr->last_x = d_last_x0;
  }
  std::string msg = st == MSM_OK ? std::string() : std::string(msm_last_error());
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cs, &graph);
  cudaStreamDestroy(cs);
  if (st != MSM_OK) {
    if (graph) cudaGraphDestroy(graph);
    return fail(st, msg);
  }
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return cuda_fail(e, "cudaStreamEndCapture");
  }
  msm_graph* g = new msm_graph;
  g->graph = graph;
  g->device = m->device;
  e = cudaGraphInstantiate(&g->exec, graph, 0);
  if (e != cudaSuccess) {
    msm_graph_destroy(g);
    return cuda_fail(e, "cudaGraphInstantiate");
  }
  *out = g;
  return MSM_OK;
}
}  // namespace

extern "C" {

msm_status msm_graph_create(msm_model* m, const void* hidden_in, const int32_t* parent, const int32_t* tokens,
                            int32_t pos0, void* const* k_cache, void* const* v_cache, float* logits_out,
                            void* hidden_out, int32_t* accept_result, msm_graph** out) {
  return capture_step(m, hidden_in, parent, tokens, pos0, nullptr, k_cache, v_cache, logits_out, hidden_out,
                      accept_result, out);
}

msm_status msm_graph_create_dev(msm_model* m, const void* hidden_in, const int32_t* state, void* const* k_cache,
                                void* const* v_cache, float* logits_out, void* hidden_out, int32_t* accept_result,
                                msm_graph** out) {
  if (!state) {
    if (out) *out = nullptr;
    return fail(MSM_ERR_INVALID_ARG, "state is NULL");
  }
  return capture_step(m, hidden_in, nullptr, nullptr, 0, state, k_cache, v_cache, logits_out, hidden_out,
                      accept_result, out);
}

msm_status msm_graph_launch(msm_graph* g, void* stream) {
  if (!g) return fail(MSM_ERR_INVALID_ARG, "graph is NULL");
  CK(cudaSetDevice(g->device));
  CK(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)));
  return MSM_OK;
}

msm_status msm_draft_step(msm_model* m, const void* hidden_in, int32_t pos0, void* const* k_cache,
                          void* const* v_cache, float* logits_out, int32_t* tokens_out, void* stream) {
  return enqueue_draft(m, hidden_in, pos0, nullptr, k_cache, v_cache, logits_out, tokens_out, stream);
}

msm_status msm_draft_step_dev(msm_model* m, const void* hidden_in, int32_t* state, void* const* k_cache,
                              void* const* v_cache, float* logits_out, void* stream) {
  if (!state) return fail(MSM_ERR_INVALID_ARG, "state is NULL");
  return enqueue_draft(m, hidden_in, 0, state, k_cache, v_cache, logits_out, nullptr, stream);
}

msm_status msm_embed_dev(msm_model* m, const void* table, const int32_t* state, void* hidden_out, void* stream) {
  return enqueue_embed(m, table, state, hidden_out, stream);
}

msm_status msm_graph_create_spec(msm_model* target, msm_model* draft, const void* draft_hidden_in,
                                 void* const* draft_k_cache, void* const* draft_v_cache, float* draft_logits,
                                 const void* embed_table, void* hidden_buf, int32_t* state, void* const* k_cache,
                                 void* const* v_cache, float* logits_out, int32_t* accept_result, msm_graph** out) {
  if (out) *out = nullptr;
  if (!draft || !embed_table || !hidden_buf || !state || !accept_result)
    return fail(MSM_ERR_INVALID_ARG, "draft, embed_table, hidden_buf, state and accept_result are required");
  SpecArgs sa{draft, draft_hidden_in, draft_k_cache, draft_v_cache, draft_logits, embed_table, state};
  return capture_step(target, hidden_buf, nullptr, nullptr, 0, state, k_cache, v_cache, logits_out, nullptr,
                      accept_result, out, &sa);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// verify step on static scratch (msm_verify_step_noalloc)
// ---------------------------------------------------------------------------
// The per-step scratch of the layer kernel (exchange buffers of both parities,
// attention and expert partials, the layer-to-layer q / hidden hand-off) lives
// in this array instead of model-owned allocations.  One array per device,
// shared by every model: overlapping calls race on it (stated in msm.h).
static __device__ __align__(256) unsigned char msm_noalloc_scratch[MSM_NOALLOC_SCRATCH_BYTES];

namespace {
msm_status noalloc_lookup(unsigned char** base) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, msm_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  if (!p) return fail(MSM_ERR_CUDA, "cudaGetSymbolAddress(static scratch) returned NULL");
  *base = static_cast<unsigned char*>(p);
  return MSM_OK;
}
}  // namespace

extern "C" msm_status msm_verify_step_noalloc(msm_model* m, const void* hidden_in, const int32_t* parent,
                                              int32_t pos0, void* const* k_cache, void* const* v_cache,
                                              float* logits_out, void* hidden_out, void* stream) {
  if (!m) return fail(MSM_ERR_INVALID_ARG, "model is NULL");
  const Dims& dm = m->dm;
  msm_status vst = validate_step(m, hidden_in, parent, pos0, nullptr, k_cache, v_cache, logits_out, hidden_out);
  if (vst != MSM_OK) return vst;
  if (m->noalloc_need > (uint64_t)MSM_NOALLOC_SCRATCH_BYTES) {
    char buf[200];
    std::snprintf(buf, sizeof(buf),
                  "msm_verify_step_noalloc: this model's step needs %llu bytes of scratch; the static array holds "
                  "%llu (MSM_NOALLOC_SCRATCH_BYTES)",
                  (unsigned long long)m->noalloc_need, (unsigned long long)MSM_NOALLOC_SCRATCH_BYTES);
    return fail(MSM_ERR_UNSUPPORTED, buf);
  }
  // carve: x[0] | x[1] | partials | in_q[0] | in_q[1] | in_h[0] | in_h[1]
  const uint64_t q_bytes = align256((uint64_t)T * dm.hq * dm.hd * 2), h_bytes = align256((uint64_t)T * dm.d * 2);
  unsigned char* base = m->noalloc;
  StepBuffers B;
  B.x[0] = base;
  B.x[1] = base + m->xo.total;
  B.sbuf = base + 2 * m->xo.total;
  B.in_q[0] = reinterpret_cast<uint16_t*>(B.sbuf + m->so.total);
  B.in_q[1] = reinterpret_cast<uint16_t*>(B.sbuf + m->so.total + q_bytes);
  B.in_h[0] = reinterpret_cast<uint16_t*>(B.sbuf + m->so.total + 2 * q_bytes);
  B.in_h[1] = reinterpret_cast<uint16_t*>(B.sbuf + m->so.total + 2 * q_bytes + h_bytes);
  B.tma_act = m->act_tma_na ? m->tma_act_na : nullptr;
  B.model_owned = false;
  CK(cudaSetDevice(m->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the last call's contents: arm the exchange part (sentinels, zeroed
  // counters) and the partials on the caller's stream before the launches
  for (int c = 0; c < 2; ++c) {
    msm_status st = arm_exchange(B.x[c], m->xo, s);
    if (st != MSM_OK) return st;
  }
  CK(launch_fill_u32(B.sbuf, m->so.y / 4, 0x80000000u, s));
  CK(launch_fill_u32(B.sbuf + m->so.y, (m->so.total - m->so.y) / 4, 0xFFFFFFFFu, s));
  return enqueue_verify(m, B, hidden_in, parent, pos0, nullptr, k_cache, v_cache, logits_out, hidden_out, stream);
}
