/*
 * msm.h — C ABI of libmsm: one speculative-decoding verify step of a batch-1
 * mixture-of-experts decoder on one GB300 GPU, one persistent kernel launch per
 * decoder layer.
 *
 * The method (LMSYS/SGLang megakernel for "Muse Spark Open", as reported by the
 * alphasignal.ai article "LMSYS Doubles Muse Spark Open Speed to 1,109 Tokens per
 * Second" and the orcarouter.ai article "Muse Spark Open: 1,109 tokens/s is a
 * kernel-level change"):
 *   - the target model verifies a 16-token tree proposed by a draft model in one
 *     pass (alphasignal.ai, § "Draft and verify share one graph"; orcarouter.ai,
 *     § on the draft model: the candidates form a tree, not a linear chain);
 *   - each launch covers one decoder layer's attention through the next layer's
 *     QKV projection and KV-cache write (alphasignal.ai, § "Launch boundaries
 *     leave hardware idle"; orcarouter.ai, § "where the kernel boundary sits");
 *   - the layer: tree-masked attention over the KV history (46 sliding-window
 *     layers over the last 2,048 tokens, 16 global), output projection, pooler,
 *     router top-8 of 256, two NVFP4 expert GEMMs, unpooler and combine
 *     (orcarouter.ai, § "where the kernel boundary sits").
 *
 * Conventions
 *   - Every call is host-synchronous in its validation and asynchronous on the
 *     stream it is given for GPU work.  Host-detectable errors (null pointers,
 *     invalid parent array, positions out of range, unsupported widths) return
 *     at once without enqueuing anything.
 *   - Device pointers are passed as plain pointers; `stream` is a cudaStream_t
 *     passed as void* (NULL = legacy default stream).
 *   - The caller owns every buffer it passes: weights (only read during
 *     msm_model_create, which copies them into a packed, model-owned layout —
 *     they may be freed once it returns), KV caches, hidden states, logits.
 *   - The model owns its packed weights, exchange buffers, routing records,
 *     timing buffer and device status word.
 *   - Bounded device waits: every in-kernel wait gives up after
 *     msm_config.timeout_us, records MSM_ERR_DEVICE_TIMEOUT in the model's status
 *     word and lets the launch finish; msm_sync() reports it and re-arms the
 *     model.  Nothing traps.
 *   - A model is not thread-safe; one model may be used by one host thread at a
 *     time.  Two steps of one model must not overlap on the GPU.
 *   - Co-residency: the blocks of a layer launch (one per SM, grid_blocks of them)
 *     wait on each other, so all of them must be resident at once.  The model checks
 *     at creation that the grid fits the device (one 384-thread block with ~227 KB
 *     of shared memory per SM); while steps run, nothing else may occupy the SMs
 *     (another kernel, another model's step, MPS or MIG clients).  If blocks cannot
 *     be co-resident, the bounded waits run out and the step reports
 *     MSM_ERR_DEVICE_TIMEOUT instead of hanging.
 *
 * Layouts (row-major; "bf16" is the 16-bit brain-float bit pattern)
 *   hidden state      bf16 [16][d_model]        (tree token i in row i)
 *   parent            int32 [16] host array: parent[0] == -1, 0 <= parent[i] < i
 *   KV cache (layer)  bf16 [n_kv_heads][max_ctx][head_dim]; rows [0, pos0) hold
 *                     the history (K already rotated); the step writes the K/V of
 *                     tree token i to row pos0 + i
 *   logits            fp32 [16][vocab]
 *   w_qkv             bf16 [(n_q_heads + 2 n_kv_heads) head_dim][d_model]
 *                     (rows: q heads, then k heads, then v heads)
 *   w_o               bf16 [d_model][n_q_heads head_dim]
 *   w_pool            bf16 [pool_dim][d_model]
 *   w_router          bf16 [n_experts][pool_dim];  b_router fp32 [n_experts]
 *   w_unpool          bf16 [d_model][pool_dim]
 *   norm_attn/norm_moe/norm_final  bf16 [d_model] RMSNorm gains
 *   w1 (NVFP4)        codes uint8 [n_experts][2 ffn_dim][pool_dim/2] (two E2M1
 *                     codes per byte, low nibble = even column), block scales
 *                     unsigned E4M3 (UE4M3: bit 7 must be 0 and is ignored)
 *                     [n_experts][2 ffn_dim][pool_dim/16], tensor scale fp32
 *                     [n_experts]; rows [0, ffn_dim) = SwiGLU gate, the rest = up
 *   w2 (NVFP4)        codes [n_experts][pool_dim][ffn_dim/2], scales
 *                     [n_experts][pool_dim][ffn_dim/16], tensor scale [n_experts]
 *   w_lm              bf16 [vocab][d_model]
 */
#ifndef MSM_H
#define MSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSM_TREE_TOKENS 16

typedef enum {
  MSM_OK = 0,
  MSM_ERR_INVALID_ARG = 1,    /* bad pointer, parent array, position or config */
  MSM_ERR_CUDA = 2,           /* a CUDA runtime call failed (see msm_last_error) */
  MSM_ERR_OOM = 3,            /* device allocation failed */
  MSM_ERR_DEVICE_TIMEOUT = 4, /* a bounded in-kernel wait expired */
  MSM_ERR_UNSUPPORTED = 5     /* widths / features this library does not implement */
} msm_status;

/* msm_config.flags */
#define MSM_FLAG_SELF_TIMING 0x1u      /* %globaltimer stamps per block and phase (the
                                          orcarouter.ai article, § "where the 5.9 ms
                                          still goes": the kernel times itself) */
#define MSM_FLAG_EXPERT_PREFETCH 0x2u  /* L2 prefetch of the previous step's most-used
                                          experts (alphasignal.ai, § "Four mechanisms
                                          keep work moving") */
#define MSM_FLAG_KV_PREFETCH 0x4u      /* L2 prefetch of the next layer's KV history at
                                          combine time (orcarouter.ai, § "where the
                                          5.9 ms still goes") */
#define MSM_FLAG_PDL 0x8u              /* chain layer launches with programmatic
                                          dependent launch */
#define MSM_FLAG_DRAFT 0x20u           /* the model is the draft model of the decode
                                          step (alphasignal.ai, § "Draft and verify share
                                          one graph"): each layer's MoE half is a dense
                                          SwiGLU FFN (w_gate, w_up, w_down; norm_moe is
                                          its RMSNorm gain), every layer attends to its
                                          whole KV history and to all 16 slots of the
                                          block (no tree mask, no window); pool_dim,
                                          n_experts and top_k are 0 and the expert,
                                          pooler, router and unpooler weights NULL;
                                          vocab > 0.  Run with msm_draft_step. */
#define MSM_FLAG_TEST_DROP_HANDOFF 0x10000u /* test hook: one block never signals that
                                          its share of h1 is stored, so the pooler's
                                          consumers time out */

typedef struct {
  int d_model, n_q_heads, n_kv_heads, head_dim;
  int pool_dim, ffn_dim, n_experts, top_k;
  int n_layers;
  int vocab;        /* 0: no LM head; the step then returns the final hidden state */
  int window;       /* sliding window (keys r with tpos - r < window) of non-global layers */
  int max_ctx;      /* KV rows per layer and head */
  const uint8_t* layer_is_global; /* host [n_layers]: 1 = global attention */
  float rms_eps, rope_theta;
  uint32_t flags;   /* MSM_FLAG_* */
  int grid_blocks;  /* persistent blocks per launch; 0 = one per SM */
  int attn_splits;  /* KV splits per kv head; 0 = automatic */
  int prefetch_experts; /* experts prefetched by MSM_FLAG_EXPERT_PREFETCH; 0 = 14 */
  uint32_t timeout_us;  /* bounded-wait limit; 0 = 200000 */
  int l2_runahead_kb;   /* L2 prefetch distance of each block's dense-weight / KV
                           stream (expert tiles are not prefetched), KiB; 0 = off
                           (alphasignal.ai, § "Four mechanisms keep work moving":
                           weights for the next operation are fetched while the
                           current one runs, partly staged in L2).  Measured slower
                           than off on the 62-layer workload (32 KiB: +7 %), hence off. */
} msm_config;

/* Device pointers, one per layer (host arrays of n_layers entries). */
typedef struct {
  const void* const* w_qkv;
  const void* const* w_o;
  const void* const* w_pool;
  const void* const* w_router;
  const float* const* b_router;
  const void* const* w_unpool;
  const void* const* norm_attn;
  const void* const* norm_moe;
  const uint8_t* const* w1_codes;
  const uint8_t* const* w1_scales;
  const float* const* w1_tensor_scale;
  const uint8_t* const* w2_codes;
  const uint8_t* const* w2_scales;
  const float* const* w2_tensor_scale;
  const void* norm_final; /* required when vocab > 0 */
  const void* w_lm;       /* required when vocab > 0 */
  /* MSM_FLAG_DRAFT models only (NULL otherwise): bf16 [ffn_dim][d_model] gate and up
     projections and bf16 [d_model][ffn_dim] down projection of each layer's FFN */
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
} msm_weights;

typedef struct msm_model msm_model;

/* Statistics of the model and of its last step (host struct). */
typedef struct {
  int grid_blocks, threads_per_block, smem_bytes, attn_splits;
  int launches_per_step;         /* kernel launches one msm_verify_step enqueues */
  int cooperative;               /* 1 if launches are cooperative (co-residency guaranteed) */
  uint64_t packed_weight_bytes;  /* model-owned packed weights */
  uint64_t exchange_bytes;       /* model-owned exchange buffers */
  int tma_act_staging;           /* 1 if dense activations are staged by tensor copies
                                    (msm_verify_step / _dev), 0 if by plain loads */
  uint64_t launches_run;         /* layer-kernel launches enqueued so far by every verify
                                    entry point (a graph capture records, not runs) */
  uint64_t noalloc_scratch_bytes;  /* static scratch one msm_verify_step_noalloc call needs */
} msm_stats;

/*
 * Create a model on `device`: validate the config, pack the caller's weights
 * into the model's layout (GPU kernels on an internal stream, completed before
 * return) and allocate the exchange buffers.
 * Errors: MSM_ERR_INVALID_ARG (null pointer, bad config), MSM_ERR_UNSUPPORTED
 * (widths outside what the kernels implement: d_model and n_q_heads*head_dim
 * multiples of 64, pool_dim and ffn_dim multiples of 256 with pool_dim <= 2048
 * and ffn_dim <= 1024, head_dim 64 or 128, n_q_heads/n_kv_heads in {1,2,4,8},
 * top_k <= 8, n_experts <= 256 and a multiple of 16, vocab a multiple of 16; a
 * grid larger than the device keeps resident), MSM_ERR_OOM, MSM_ERR_CUDA.  On
 * error *out is NULL.
 */
msm_status msm_model_create(const msm_config* config, const msm_weights* weights, int device,
                            msm_model** out);

/* Free every model-owned buffer.  Waits for the model's work to finish.  NULL is ignored. */
void msm_model_destroy(msm_model* model);

/*
 * One verify step: for every layer in order, tree attention over the cache rows
 * [0, pos0) and the tree's own rows, then the MoE block; writes the K/V rows of
 * the 16 tree tokens to rows pos0..pos0+15 of every layer's cache, and the
 * logits of all 16 tree tokens (vocab > 0) and/or the final hidden state.
 *   hidden_in   device bf16 [16][d_model] (read)
 *   parent      host int32 [16]; parent[0] == -1, 0 <= parent[i] < i
 *   pos0        first tree row; 0 <= pos0 and pos0 + 16 <= max_ctx
 *   k_cache, v_cache  host arrays of n_layers device pointers (see layout)
 *   logits_out  device fp32 [16][vocab] or NULL (must be non-NULL if vocab > 0)
 *   hidden_out  device bf16 [16][d_model] or NULL (must be non-NULL if vocab == 0)
 * Enqueues n_layers launches on `stream`.  Device-side failures are reported
 * by the next msm_sync().
 */
msm_status msm_verify_step(msm_model* model, const void* hidden_in, const int32_t* parent,
                           int32_t pos0, void* const* k_cache, void* const* v_cache,
                           float* logits_out, void* hidden_out, void* stream);

/*
 * The same step with hidden_in / logits_out / hidden_out in HOST memory: copies
 * the input to the device, runs the step, copies the results back and waits
 * for the stream.  Returns the step's device status as msm_sync() would.
 * Host buffers may be pageable; pinned buffers make the copies asynchronous.
 */
msm_status msm_verify_step_host(msm_model* model, const void* hidden_in_host,
                                const int32_t* parent, int32_t pos0, void* const* k_cache,
                                void* const* v_cache, float* logits_host, void* hidden_out_host,
                                void* stream);

/*
 * msm_verify_step_noalloc: the verify step of msm_verify_step (same arguments,
 * same results, bit for bit) with its per-step scratch taken from a fixed
 * static device array instead of the model's own buffers.  The pages describe
 * no such entry point; it has no counterpart there.
 *
 * Who needs it: callers that must not allocate device memory at the time they
 * run a step -- for instance code under a strict device-memory budget, or code
 * that pre-plans all of its memory and forbids allocation on the decode path.
 * On success this call allocates nothing: no cudaMalloc / cudaFree, no
 * allocating library call.  (msm_verify_step allocates nothing per step either,
 * but it uses exchange buffers that msm_model_create allocated for the model;
 * this entry point uses the static array instead.)
 *
 * Scratch: MSM_NOALLOC_SCRATCH_BYTES (10 MiB) of __device__ memory per device,
 * shared by every model on that device.  A step needs
 *   2 * (exchange buffers + 256 bytes of phase counters) + attention/expert
 *   partials + 2 * (16 n_q_heads head_dim * 2) + 2 * (16 d_model * 2) bytes
 * (each part rounded up to 256 bytes), about 8.4 MiB at d_model 4096, 32/8
 * heads of 128, pool_dim 2048, ffn_dim 1024, top-8 on 152 SMs; the exact
 * figure of a model is msm_stats.noalloc_scratch_bytes.  A model whose step
 * needs more is rejected with MSM_ERR_UNSUPPORTED and a message giving both
 * sizes; nothing is launched.
 * The exchange part must hold its empty sentinels when a step starts; every
 * call arms it on `stream` before its first layer launch, so no state carries
 * over from an earlier call, a failed step or another model.
 *
 * Set-up: msm_model_create looks up the array's device address
 * (cudaGetSymbolAddress, with the model's device current), which loads the code
 * module that holds the array and so gives the array its device memory then, at
 * creation, not at the first call; the calls themselves do no set-up.
 *
 * Concurrency: the scratch is one array per device.  Calls that overlap on the
 * device (from other threads, or on other streams of the same device before the
 * previous call's work has finished) race on it and give wrong results.
 * Serialise them, e.g. by issuing them on one stream.
 *
 * Device-side failures are reported by the next msm_sync(), as for
 * msm_verify_step.
 */
#define MSM_NOALLOC_SCRATCH_BYTES (10u << 20)
msm_status msm_verify_step_noalloc(msm_model* model, const void* hidden_in, const int32_t* parent,
                                   int32_t pos0, void* const* k_cache, void* const* v_cache,
                                   float* logits_out, void* hidden_out, void* stream);

/* Wait for `stream`, then return (and clear) the device status latched by the
 * model's launches.  After MSM_ERR_DEVICE_TIMEOUT the model re-arms its exchange
 * buffers, so the next step starts clean. */
msm_status msm_sync(msm_model* model, void* stream);

/* Routing of the last completed step: idx int32 [n_layers][16][top_k] (expert
 * indices, larger logit first, ties to the lower index) and w fp32
 * [n_layers][16][top_k] (softmax over the selected logits).  Host buffers; either
 * may be NULL.  Synchronises the device. */
msm_status msm_get_routing(msm_model* model, int32_t* idx, float* w);

/* Tree as computed on the device in the last step: anc uint32 [16]
 * (ancestor-or-self bitmask), tpos int32 [16] (pos0 + depth).  Host buffers. */
msm_status msm_get_tree(msm_model* model, uint32_t* anc, int32_t* tpos);

/* Self-timing stamps of the last step (MSM_FLAG_SELF_TIMING):
 * uint64 [n_layers][grid_blocks][MSM_TIMING_EVENTS] %globaltimer values (ns), 0
 * where an event did not occur.  Event ids (per block of a launch; "_IN" = the
 * phase's input has been received and staged):
 *   0 start, 1 prologue in, 2 prologue done, 3 attention in, 4 attention done,
 *   5 split merge done, 6 o_proj in, 7 o_proj done, 8 pooler in, 9 pooler done,
 *   10 router in, 11 router done, 12 top-k done, 13 routing done, 14 GEMM1 done,
 *   15 GEMM2 in, 16 GEMM2 done, 17 combine done, 18 unpooler in, 19 unpooler done,
 *   20 tail in, 21 tail done, 22 end, 23 loader saw the routing, 24 loader done,
 *   25 expert dispatch built, 26 pooler input staged (before its norm), 27 first
 *   pooled row read for GEMM1, 28 / 29 first / second GEMM1 input row of the
 *   first compute warp staged, 30 pooler input normalised by the first compute
 *   warp, 31 pooler norm gain in shared memory; 32-39 o_proj units 0 and 1 of the block (first tile ready, last tile
 *   ready, partial sums stored, epilogue done), 40-43 GEMM1 of the first compute
 *   warp (first unit's tile ready / unit done, last unit's tile ready / done),
 *   44 / 45 loader issued the first / last o_proj tile, 46 / 47 the first / last
 *   GEMM1 tile; 48-51 GEMM2 of the first compute warp pair (first unit's tile ready
 *   / unit done, last unit's tile ready / done), 52 / 53 second GEMM2 staging
 *   round (experts 3-4 of a block; two per round) begun / done, 54 loader issued the first tile of the
 *   block's second o_proj unit; 55-62 the block's poller saw the phase-completion
 *   counter that releases the split merge, o_proj, pooler, router, top-k, combine,
 *   unpooler and tail reach the grid size.
 * `n` is the capacity of `buf` in elements. */
#define MSM_TIMING_EVENTS 192
msm_status msm_get_timing(msm_model* model, uint64_t* buf, size_t n);

msm_status msm_get_stats(const msm_model* model, msm_stats* out);

/* Diagnostic: copy an exchange buffer of the last launch of the last step to host
 * memory.  `name` is one of "o" (attention output, bf16 [16][n_q_heads head_dim]),
 * "h1" (residual after attention, bf16 [16][d_model]), "u" (pooled, bf16
 * [16][pool_dim]), "logits" (router logits, fp32 [16][n_experts]), "a" (SwiGLU
 * activations, fp32 [16 top_k][ffn_dim]), "z" (combined expert output, bf16
 * [16][pool_dim]), "h2" (layer output, bf16 [16][d_model]).  Slots a launch never
 * filled keep their sentinels (0xFFFF / -0.0).  `bytes` is the capacity of `host`.
 * Synchronises the device. */
msm_status msm_get_exchange(msm_model* model, const char* name, void* host, size_t bytes);

/*
 * Accept step after a verify step: the target's greedy choice at each tree node,
 * the walk down the tree, and KV-cache compaction (alphasignal.ai, § "Draft and
 * verify share one graph": candidates the target agrees with become output
 * tokens, rejected branches are dropped; orcarouter.ai, closing figure: greedy
 * decoding, accept inside the step's CUDA graph).
 *   logits   device fp32 [16][vocab], the verify step's logits_out (read)
 *   tokens   host int32 [16]: the draft token of each tree node; tokens[0] (the
 *            root) is not checked; every id must lie in [0, vocab)
 *   parent   host int32 [16], the verify step's tree
 *   pos0, k_cache, v_cache   as passed to the verify step
 *   result   device int32 [MSM_ACCEPT_RESULT_INTS] (written):
 *            [0] a = number of accepted nodes, root included (1..16)
 *            [1] the bonus token: the greedy choice at the last accepted node
 *            [2 + j] path[j], the j-th accepted node (path[0] = 0), -1 for j >= a
 *            [18 + i] the greedy choice (argmax of the logits) at node i
 * Greedy choice: the largest logit, the smallest index among equal ones; a NaN
 * ranks above every number.  Walk: from the root, move to the child (smallest
 * tree index first) whose token is the current node's choice; stop when none is.
 * Compaction: for j < a, cache row pos0 + j of every layer, K and V, every KV head
 * receives row pos0 + path[j]; no other row is written.  Everything runs on the
 * device (two launches on `stream`, no host round trip), so a stream capture
 * records it.  It uses model-owned scratch (argmax partials, a ticket counter), so
 * accept calls of one model must not overlap on the GPU, like its steps.
 * Errors: MSM_ERR_UNSUPPORTED when vocab == 0, MSM_ERR_INVALID_ARG
 * for NULL or misaligned buffers, an invalid parent array, token ids or pos0;
 * nothing is enqueued then.
 */
#define MSM_ACCEPT_RESULT_INTS 34
msm_status msm_accept(msm_model* model, const float* logits, const int32_t* tokens, const int32_t* parent,
                      int32_t pos0, void* const* k_cache, void* const* v_cache, int32_t* result, void* stream);

/*
 * One CUDA graph per decode step (alphasignal.ai, § "Draft and verify share one
 * graph"; orcarouter.ai, closing figure): msm_graph_create captures the arming of
 * the model's exchange buffers, the verify step's n_layers launches, if
 * accept_result is not NULL msm_accept's launches, and a second arming (so eager
 * steps and replays may be mixed freely), and instantiates the graph.
 * Arguments are those of msm_verify_step and msm_accept; the tree, the tokens and
 * pos0 are recorded in the graph, as are all buffer addresses, so a replay reads
 * the buffers' current contents at those addresses.  msm_graph_launch replays it
 * on `stream`; every replay computes what the captured calls compute.
 * (msm_graph_create_dev below records a device-resident state instead of the tree,
 * tokens and pos0; msm_graph_create_spec adds the draft step and the embedding of
 * its proposal, so one graph holds the whole speculative step.)  The model must outlive its graphs;
 * replays of one model must not overlap on the GPU.  msm_graph_destroy frees the
 * graph (NULL is ignored).  Errors: those of the captured calls (nothing is
 * recorded then), MSM_ERR_CUDA for a failed capture or instantiation.
 */
typedef struct msm_graph msm_graph;

/*
 * Device-resident step inputs, so that one graph can serve every decode step
 * (the pages' plugin replays one graph per step; orcarouter.ai, closing figure):
 * a device int32 [MSM_STEP_STATE_INTS] array
 *   [0] pos0, [1 + i] parent[i], [17 + i] the draft token of tree node i, [33] unused
 * read by the kernels when they run, not when the call is made.  The caller
 * writes it (for instance with cudaMemcpyAsync on the same stream) before each
 * step.  The kernels check it (parent[0] == -1, 0 <= parent[i] < i, token ids in
 * [0, vocab), 0 <= pos0 <= max_ctx - 16); an invalid state makes every launch of
 * the step give up at entry without touching the caches or outputs, and the next
 * msm_sync() returns MSM_ERR_INVALID_ARG (msm_accept_dev then also writes a = 0
 * and -1 elsewhere in `result`).
 *   msm_verify_step_dev  = msm_verify_step with the tree and pos0 from `state`
 *   msm_accept_dev       = msm_accept with tree, tokens and pos0 from `state`
 *   msm_graph_create_dev = msm_graph_create capturing those two: a replay reads the
 *                          state's current contents, so one graph serves any tree
 *                          and position
 * Host errors as for the host-parameter calls, plus MSM_ERR_INVALID_ARG for a NULL
 * or misaligned state.
 */
#define MSM_STEP_STATE_INTS 34
msm_status msm_verify_step_dev(msm_model* model, const void* hidden_in, const int32_t* state, void* const* k_cache,
                               void* const* v_cache, float* logits_out, void* hidden_out, void* stream);
msm_status msm_accept_dev(msm_model* model, const float* logits, const int32_t* state, void* const* k_cache,
                          void* const* v_cache, int32_t* result, void* stream);
msm_status msm_graph_create_dev(msm_model* model, const void* hidden_in, const int32_t* state, void* const* k_cache,
                                void* const* v_cache, float* logits_out, void* hidden_out, int32_t* accept_result,
                                msm_graph** out);

msm_status msm_graph_create(msm_model* model, const void* hidden_in, const int32_t* parent, const int32_t* tokens,
                            int32_t pos0, void* const* k_cache, void* const* v_cache, float* logits_out,
                            void* hidden_out, int32_t* accept_result, msm_graph** out);
msm_status msm_graph_launch(msm_graph* graph, void* stream);
void msm_graph_destroy(msm_graph* graph);

/*
 * msm_draft_step: one pass of the draft model (a model created with
 * MSM_FLAG_DRAFT) over a block of 16 slots, proposing 15 tokens at once
 * (alphasignal.ai, § "Draft and verify share one graph": a 5-layer draft, one
 * launch per layer, its 15 candidates from one pass).  The pages give only the
 * widths; the layer follows the target layer's conventions:
 *   slot i sits at position pos0 + i (RoPE) and writes its K/V rows to cache row
 *   pos0 + i; it attends to every history row [0, pos0) and to all 16 slots;
 *   h1 = bf16(h + bf16(attn W_o^T)); z = bf16(silu(x W_gate^T) * (x W_up^T)) with
 *   x = RMSNorm(h1); h2 = bf16(h1 + bf16(z W_down^T)); after the last layer the
 *   final RMSNorm and the LM head give fp32 logits.
 *   hidden_in  device bf16 [16][d_model]: the block's input rows
 *   pos0       first cache row of the block: 0 <= pos0 <= max_ctx - 16
 *   k_cache / v_cache  host arrays of n_layers device pointers, bf16
 *              [n_kv_heads][max_ctx][head_dim] each (the draft's own caches)
 *   logits_out device fp32 [16][vocab] (required)
 *   tokens_out device int32 [16]: tokens_out[0] = -1 (slot 0 holds the caller's
 *              known token), tokens_out[i] = the argmax of slot i's logits (the
 *              smallest index among equal maxima): the proposal for position
 *              pos0 + i.  The proposal is a chain, parent[i] = i - 1.
 * Launches n_layers layer-kernel launches and two reduction launches on `stream`;
 * returns after enqueueing.  Errors: MSM_ERR_INVALID_ARG (NULL pointer, pos0 out
 * of range, model not a draft model); a failing launch reports at msm_sync.
 */
msm_status msm_draft_step(msm_model* draft, const void* hidden_in, int32_t pos0, void* const* k_cache,
                          void* const* v_cache, float* logits_out, int32_t* tokens_out, void* stream);

/*
 * msm_draft_step_dev: msm_draft_step with pos0 read from a device-resident step
 * state (MSM_STEP_STATE_INTS ints, as for msm_verify_step_dev) when the kernels run;
 * the proposal goes into the state: parent[i] = i - 1 (the chain) for every i, and
 * the token of node i = the argmax of slot i for i = 1..15.  The root's token
 * (state[17]) is the caller's and is not written.  An invalid pos0 makes the layer
 * launches give up at entry (msm_sync then returns MSM_ERR_INVALID_ARG); the state
 * is still written, from whatever logits_out held.
 */
msm_status msm_draft_step_dev(msm_model* draft, const void* hidden_in, int32_t* state, void* const* k_cache,
                              void* const* v_cache, float* logits_out, void* stream);

/*
 * msm_embed_dev: the verify step's input rows from an embedding table, read from a
 * step state when the kernel runs: hidden_out[i] = table[state[17 + i]] (the token
 * of tree node i).  The verify step takes its 16 input rows as given (the embedding
 * precedes it in the pages' decoder); this call lets one graph go from the draft's
 * proposal to the verify step's input without a host round trip.
 *   model      the target model (vocab > 0; its d_model and vocab size the table)
 *   table      device bf16 [vocab][d_model], caller-owned, 16-byte aligned
 *   hidden_out device bf16 [16][d_model], 16-byte aligned
 * One launch of 16 blocks on `stream`.  A token id outside [0, vocab) gives a zero
 * row and MSM_ERR_INVALID_ARG at the next msm_sync (the verify step's own state
 * check rejects the step then).  Host errors: MSM_ERR_INVALID_ARG (NULL or
 * misaligned pointers), MSM_ERR_UNSUPPORTED (vocab == 0).
 */
msm_status msm_embed_dev(msm_model* model, const void* table, const int32_t* state, void* hidden_out, void* stream);

/*
 * msm_graph_create_spec: one CUDA graph holding a whole speculative decode step on
 * a device-resident state (alphasignal.ai, § "Draft and verify share one graph"):
 *   msm_draft_step_dev(draft, draft_hidden_in, state, draft caches, draft_logits)
 *   msm_embed_dev(target, embed_table, state, hidden_buf)
 *   msm_verify_step_dev(target, hidden_buf, state, k_cache, v_cache, logits_out)
 *   msm_accept_dev(target, logits_out, state, k_cache, v_cache, accept_result)
 * with both models' exchange buffers armed before and after.  Before each replay
 * the caller sets state[0] (pos0) and state[17] (the root token, e.g. the previous
 * step's bonus token) and fills draft_hidden_in; the graph writes the rest of the
 * state, hidden_buf, both logits and accept_result.  Both models must be on one
 * device and outlive the graph; replays must not overlap.  Errors: those of the
 * captured calls, MSM_ERR_INVALID_ARG for a NULL draft, table, hidden_buf, state or
 * accept_result or models on different devices.
 */
msm_status msm_graph_create_spec(msm_model* target, msm_model* draft, const void* draft_hidden_in,
                                 void* const* draft_k_cache, void* const* draft_v_cache, float* draft_logits,
                                 const void* embed_table, void* hidden_buf, int32_t* state, void* const* k_cache,
                                 void* const* v_cache, float* logits_out, int32_t* accept_result, msm_graph** out);

/* Message of the last error on the calling thread ("" if none). */
const char* msm_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MSM_H */
