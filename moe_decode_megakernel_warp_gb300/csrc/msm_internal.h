// Internal definitions shared by the host runtime (msm_api.cu) and the kernels
// (msm_kernel.cu, msm_pack.cu) of libmsm.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace msm {

constexpr int T = 16;                 // tree tokens per verify step
constexpr int kThreads = 384;         // 12 warps per persistent block
constexpr int kLoaderWarp = 0;        // TMA producer of the shared-memory weight ring
constexpr int kPrefetchWarp = 3;      // L2 prefetch of the previous step's hot experts
constexpr int kFirstCompute = 4;      // warps 4..11: attention / GEMM / expert workers
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kSlots = 12;            // descriptors of the variable-size ring
constexpr int kDenseTileSteps = 64;   // 16-row x 1024-column bf16 tiles: 64 k-steps x 512 B
constexpr int kKStepBytes = 512;      // one 16x16 bf16 block: its 32 threads' m16n8k16 A fragments
constexpr int kDenseTmemSlots = 8;    // dense weight tiles held in tensor memory at once
// NVFP4 expert tiles: 128 rows x tk columns (tk = 512 where the width allows, else 256):
// tk / 256 column blocks of 128 rows x 128 code bytes in the 128-byte swizzle layout
// (16 KB each), then the UE4M3 block scales as tk / 64 groups of 512 bytes, one per K=64
// step: the word of row m's four scales at byte (m % 32) * 16 + (m / 32) * 4 of its group
constexpr int kExpTileRows = 128;
constexpr int kExpBlockK = 256;                                  // columns per 16 KB code block
constexpr int kExpBlockBytes = kExpTileRows * kExpBlockK / 2;
__host__ __device__ constexpr int exp_tile_k(int K) { return K % 512 == 0 ? 512 : 256; }
__host__ __device__ constexpr int exp_tile_bytes(int K) { return exp_tile_k(K) / kExpBlockK * kExpBlockBytes + kExpTileRows * exp_tile_k(K) / 16; }
__host__ __device__ constexpr int exp_scale_off(int K) { return exp_tile_k(K) / kExpBlockK * kExpBlockBytes; }
constexpr int kSmallBytes = 16 * 1024; // barriers, routing tables, scratch, dense partials
constexpr int kMaxSmem = 232448;      // 227 KB opt-in dynamic shared memory per block
constexpr int kTimingEvents = 192;
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;

// self-timing events of one launch (per block): *_IN = the phase's input is staged
enum TimingEvent : int {
  EV_START = 0, EV_PRO_IN = 1, EV_PRO_DONE = 2, EV_ATTN_IN = 3, EV_ATTN_DONE = 4, EV_MERGE_DONE = 5,
  EV_OPROJ_IN = 6, EV_OPROJ_DONE = 7, EV_POOL_IN = 8, EV_POOL_DONE = 9, EV_ROUTER_IN = 10, EV_ROUTER_DONE = 11,
  EV_ROUTE_TOPK = 12, EV_ROUTE_DONE = 13, EV_GEMM1_DONE = 14, EV_GEMM2_IN = 15, EV_GEMM2_DONE = 16,
  EV_COMBINE_DONE = 17, EV_UNPOOL_IN = 18, EV_UNPOOL_DONE = 19, EV_TAIL_IN = 20, EV_TAIL_DONE = 21, EV_END = 22,
  EV_LOADER_ROUTED = 23, EV_LOADER_END = 24, EV_ROUTE_DISPATCH = 25,
  EV_POOL_STAGED = 26, EV_SPLIT_DONE = 27, EV_B1_ISSUED = 28, EV_B1_LANDED = 29,
  EV_POOL_NORMED = 30, EV_POOL_GAIN = 31,
  // finer stamps: o_proj units 0 / 1 of the block (first tile ready, last tile ready,
  // partial sums stored, epilogue done), GEMM1 of the first compute warp, and the loader
  EV_OP_U0_FIRST = 32, EV_OP_U0_LAST = 33, EV_OP_U0_RED = 34, EV_OP_U0_EPI = 35,
  EV_OP_U1_FIRST = 36, EV_OP_U1_LAST = 37, EV_OP_U1_RED = 38, EV_OP_U1_EPI = 39,
  EV_G1_FIRST_READY = 40, EV_G1_FIRST_DONE = 41, EV_G1_LAST_READY = 42, EV_G1_LAST_DONE = 43,
  EV_LD_OP_FIRST = 44, EV_LD_OP_LAST = 45, EV_LD_G1_FIRST = 46, EV_LD_G1_LAST = 47,
  // GEMM2 of the first compute warp pair (first / last unit: tile ready, unit done) and
  // the staging of the block's second expert (start, done)
  EV_G2_FIRST_READY = 48, EV_G2_FIRST_DONE = 49, EV_G2_LAST_READY = 50, EV_G2_LAST_DONE = 51,
  EV_G2_STAGE2_IN = 52, EV_G2_STAGE2_DONE = 53,
  EV_LD_OP_U1 = 54,  // loader issued the first tile of the block's second o_proj unit
  // the block's poller saw a phase-completion counter reach the grid size
  EV_SEEN_MERGE = 55, EV_SEEN_OPROJ = 56, EV_SEEN_POOL = 57, EV_SEEN_ROUTER = 58, EV_SEEN_ROUTE = 59,
  EV_SEEN_COMBINE = 60, EV_SEEN_UNPOOL = 61, EV_SEEN_TAIL = 62,
  // per-tile trace of the expert GEMMs (the block's first tiles): the tensor-core warp
  // saw tile i's operands ready / had issued its MMAs; GEMM1 epilogue of unit i done
  EV_TC_G1_READY = 64,   // + i, i < 16
  EV_TC_G1_ISSUED = 80,  // + i, i < 16
  EV_G1_EPI_DONE = 96,   // + i, i < 16
  EV_TC_G2_READY = 112,  // + i, i < 8
  EV_TC_G2_ISSUED = 120, // + i, i < 8
  EV_LD_G1_ISSUED = 128, // + i, i < 16: the loader issued the copy of GEMM1 tile i
  EV_LD_RING_GROWN = 144, // the loader's ring grew into the activation buffer
  EV_LD_G1_NEXT = 160,    // + i, i < 16: the loader had GEMM1 tile i's source (after the stream step)
  EV_LD_G1_PLACED = 176   // + i, i < 16: ... and its ring space
};

// phases of one layer launch (recorded in the status word on a timeout)
enum Phase : int {
  PH_START = 0, PH_PROLOGUE = 1, PH_ATTN = 2, PH_ATTN_MERGE = 3, PH_OPROJ = 4, PH_POOL = 5,
  PH_ROUTER = 6, PH_ROUTE = 7, PH_GEMM1 = 8, PH_GEMM2 = 9, PH_COMBINE = 10, PH_UNPOOL = 11,
  PH_TAIL = 12, PH_END = 13,
  PH_TC_DENSE = 14  // the tensor-core warp moving dense weight tiles into tensor memory
};

// device status word
struct DevStatus {
  int code;    // 0 or msm_status
  int phase;   // Phase where the first failure was seen
  int block;
  int layer;
  int abort;   // set by the first failing block; every wait gives up once it is set
  int pad[3];
};

// Exchange buffers of one launch parity (byte offsets into the parity's region).
struct XOffsets {
  uint64_t o, h1, u, logits, a, z, h2, q0, tkv0;  // re-armed by the next launch
  uint64_t cnt;                                   // phase-completion counters, zeroed likewise
  uint64_t b1;    // GEMM1 operand B of the launch (written whole by the router phase)
  uint64_t total;
};
// Phase-completion counters of one launch: every block adds 1 to counter i once it
// has stored its share of phase i; a consumer of the phase's output waits until the
// counter equals the grid size, then reads the output without sentinel checks.
enum PhaseCounter : int {
  CNT_ATTN = 0,    // attention partials (m, l, acc) of every (kv head, split)
  CNT_MERGE = 1,   // attention output o
  CNT_OPROJ = 2,   // h1
  CNT_POOL = 3,    // pooled u
  CNT_ROUTER = 4,  // router logits
  CNT_GEMM2 = 5,   // expert outputs y
  CNT_COMBINE = 6, // combined z
  CNT_UNPOOL = 7,  // h2
  kPhaseCounters = 8
};
constexpr int kCounterBytes = 256;
// Buffers drained by their single consumer (never double-buffered).
struct SOffsets {
  uint64_t part, ml, y;
  uint64_t total;
};

struct Dims {
  int d, hq, hkv, hd, p, f, e, k, vocab, max_ctx, window, n_layers;
  int nqkv;        // (hq + 2 hkv) hd
  int group;       // hq / hkv
  int attn_rows;   // R: KV rows per attention tile
  int kv_rows;     // KV rows per ring tile: R, or 2R for a draft model (two attention tiles)
  int attn_nk;     // keys per warp per tile
  int attn_wph;    // warps per q head
  int splits;      // attention splits per kv head
  float rms_eps;
  int draft;       // a draft model: dense SwiGLU FFN layers (f = ffn_dim), attention to the whole block
};

struct LaunchParams {
  Dims dm;
  // packed weights
  const uint8_t* w_qkv_pro;   // layer 0 QKV (prologue of launch 0) or null
  const uint16_t* g_attn_pro; // layer 0 attention norm gain
  const uint8_t* w_o;
  const uint8_t* w_pool;
  const uint8_t* w_router;
  const float* b_router;
  const uint8_t* w_unpool;
  const uint16_t* g_moe;
  const uint8_t* w1;
  const uint8_t* w2;
  const float* w1_gs;
  const float* w2_gs;
  const uint8_t* w_up;        // draft models: FFN gate + up (paired rows), FFN down
  const uint8_t* w_down;
  const uint8_t* w_tail;      // next layer's QKV, or the LM head on the last layer
  const uint16_t* g_tail;     // next layer's attention gain, or the final gain
  // caller buffers
  const uint16_t* hidden_in;  // launch 0
  uint16_t* hidden_out;       // last launch (optional)
  float* logits;              // last launch with vocab > 0
  uint16_t* kc;               // this layer's caches
  uint16_t* vc;
  uint16_t* kc_next;          // next layer's caches (tail writes the tree rows)
  uint16_t* vc_next;
  const uint16_t* kc_pf;      // next layer's caches for the KV L2 prefetch
  const uint16_t* vc_pf;
  // model buffers
  uint8_t* x_cur;             // exchange region of this launch's parity
  uint8_t* x_next;            // the other parity: re-armed here
  uint8_t* s_buf;             // single-consumer buffers
  XOffsets xo;
  SOffsets so;
  const uint16_t* in_q;       // Q / residual handed over by the previous launch
  const uint16_t* in_h;
  uint16_t* out_q;            // ... and to the next launch
  uint16_t* out_h;
  float* rope;                // [16 depth][hd/2][2] cos, sin (filled by launch 0)
  const double* inv_freq;     // [hd/2]
  int32_t* routing_idx;       // [16][k] of this layer
  float* routing_w;
  uint32_t* hist_cur;         // [e] expert usage of this layer in this step
  const uint32_t* hist_prev;  // [e] ... in the previous step
  uint32_t* tree_dbg;         // [32]: anc[16], tpos[16]
  uint64_t* timing;           // [grid][kTimingEvents] of this layer
  DevStatus* status;
  // scalars
  int layer, first, last, is_global, next_global, pos0;
  int ring_bytes, act_bytes;
  // expert phases: GEMM1's operand B (the split pooled vectors and their scales) and
  // the GEMM2 operands sit at these offsets at the top of the activation buffer; from
  // the end of routing to the unpooler the weight ring may grow by ring_ext bytes into
  // the bottom of it
  int g1_b_off, g2_off, ring_ext;
  int sfb_ext;  // bytes the expert ring may grow by once GEMM1's operand-B scales are in tensor memory
  // the unpooler's activation sits at this offset (the top of the buffer), and its
  // weight tiles may take unpool_ext bytes of the bottom
  int unpool_act_off, unpool_ext;
  int attn_act_off;  // attention's Q, tree rows and merge scratch: the top of the activation buffer
  int kv_ext;        // ... below it, ring space for the KV tiles (launches after the first)
  uint32_t flags;
  uint32_t timeout_ns_lo, timeout_ns_hi;
  int prefetch_experts;
  uint32_t runahead_bytes;  // L2 run-ahead of the loader's stream; 0 = off
  int phase_rot;
  int32_t parent[16];
  // device-resident step inputs, or null: int32 [34] = pos0, parent[16], draft
  // tokens[16], spare; when set, pos0 and parent above are unused and each
  // launch validates the state at entry (a bad one fails the launch with code 1)
  const int32_t* state;
  // KV cache tensor maps of this layer: 3-D {hd, max_ctx, hkv}, 128-byte swizzle
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  // the five dense activations of this launch's exchange buffer (ActMap order) as
  // 3-D tensor maps {64 columns, 16 rows, K / 64 blocks} with the 128-byte swizzle,
  // which is the shared-memory activation layout; act_tma == 0: plain loads
  CUtensorMap tmap_act[5];
  int act_tma;
  int act_box[5];  // 64-column blocks per copy
};
enum ActMap : int { ACT_O = 0, ACT_H1 = 1, ACT_U = 2, ACT_Z = 3, ACT_H2 = 4 };

// packed sizes
__host__ __device__ inline uint64_t dense_unit_bytes(int K) { return (uint64_t)K * 32; }  // 16 rows x K bf16
// an expert unit: 128 rows x K columns = K / exp_tile_k(K) tiles (W1: 64 gate rows and the
// 64 matching up rows, interleaved gate, up, gate, ...; W2: 128 rows)
__host__ __device__ inline uint64_t exp_unit_bytes(int K) { return (uint64_t)(K / exp_tile_k(K)) * exp_tile_bytes(K); }
__host__ __device__ inline int w1_units(int f) { return f / 64; }
__host__ __device__ inline int w2_units(int p) { return p / kExpTileRows; }
// GEMM1 operand B: the 16 pooled vectors, each as the sum of kSplitTerms NVFP4 terms,
// one B row per (term, token) pair, row n = term * 16 + token: first p / 64 scale groups
// of 512 bytes, one per K=64 step, for the tensor-memory copy (32 lines of 16 bytes; line
// l: the scale words of rows l and l + 32, two zero words) -- the part a block no longer
// needs once they are copied; then p / 256 column blocks of 64 rows x 128 code bytes
// (128-byte swizzle, 8 KB each, 1 KB aligned); then the 16 tokens' fp32 row scales
constexpr int kSplitTerms = 4;
constexpr int kSplitRows = kSplitTerms * T;
__host__ __device__ inline uint64_t b1_sfb_bytes(int p) { return (uint64_t)p / 64 * 512; }
__host__ __device__ inline uint64_t b1_code_off(int p) { return b1_sfb_bytes(p); }
__host__ __device__ inline uint64_t b1_code_bytes(int p) { return (uint64_t)p / 256 * kSplitRows * 128; }
__host__ __device__ inline uint64_t b1_ts_off(int p) { return b1_code_off(p) + b1_code_bytes(p); }
__host__ __device__ inline uint64_t b1_bytes(int p) { return b1_ts_off(p) + 256; }

// kernel entry points (defined in msm_kernel.cu / msm_pack.cu)
const void* layer_kernel(bool timing, bool draft);  // the layer kernel's four instantiations

// accept step (msm_accept.cu): argmax partials [16][parts] of the 16 logit rows
// reduced by the last block to the 16 choices, then the walk + K/V compaction, up to kAcceptLayers layers per launch (the
// per-layer cache pointers travel in the kernel parameters, so a stream capture
// needs no host-to-device copy)
constexpr int kAcceptLayers = 64;
struct AcceptParams {
  const int32_t* choice;  // [16] greedy choice per tree node (launch 1's output)
  int32_t parent[16];
  int32_t tokens[16];
  int32_t pos0, n_kv_heads, head_dim, max_ctx, n_layers, vocab;
  int32_t* result;  // written by block 0 of the launch that carries it, else nullptr
  const int32_t* state;  // device-resident pos0 / parent / tokens (then the fields above are unused), or null
  DevStatus* status;     // where a launch reports an invalid device-resident state
  uint16_t* kc[kAcceptLayers];
  uint16_t* vc[kAcceptLayers];
};
cudaError_t launch_accept_argmax(const float* logits, int vocab, uint64_t* part, int parts, uint32_t* ticket,
                                 int32_t* choice, cudaStream_t s);
cudaError_t launch_accept_walk(const AcceptParams& p, int blocks, cudaStream_t s);
cudaError_t launch_draft_propose(const int32_t* choice, int32_t* state, cudaStream_t s);
cudaError_t launch_embed(const void* table, int vocab, int d, const int32_t* state, void* out, DevStatus* status,
                         cudaStream_t s);

}  // namespace msm
