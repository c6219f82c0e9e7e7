// msm_accept.cu — the accept step after a verify step: the target's greedy
// choice at every tree node, the walk down the tree, and the move of the accepted
// nodes' K/V rows to the front of the tree's rows.
//
// alphasignal.ai, "LMSYS Doubles Muse Spark Open Speed to 1,109 Tokens per
// Second", § "Draft and verify share one graph": candidates the target agrees with
// become output tokens, rejected branches are dropped; orcarouter.ai, "Muse Spark
// Open: 1,109 tokens/s is a kernel-level change", closing figure (the repository
// screenshot): greedy decoding at batch 1, accept inside the step's CUDA graph.
//
// Two launches, both free of host round trips (so a stream capture records them):
//   1. accept_argmax_kernel: block b scans a contiguous slice of all 16 logit rows
//      and leaves one 64-bit key per row, value-ordered bits above the complement
//      of the index, so that the largest key is the largest logit with the
//      smallest index (a NaN ranks above +inf, -0 equals +0); the last block to
//      finish (a ticket counter after a gpu-scope fence) reduces the 16 x G keys
//      to the 16 choices and re-zeroes the counter;
//   2. accept_walk_kernel: every block walks the tree (the same walk in every
//      block) and copies its share of the K/V columns: one thread owns a 16-byte
//      column of one (layer, K|V, head), loads every moved row of it, then stores
//      them, so row pos0 + j receives the old row pos0 + path[j] whatever the path.
#include "msm_internal.h"

namespace msm {
namespace {

constexpr int kAcceptThreads = 256;
constexpr int kRowsPerThread = 16;

__device__ __forceinline__ uint64_t argmax_key(float x, uint32_t idx) {
  uint32_t b = __float_as_uint(x);
  if (x != x) b = 0x7FFFFFFFu;      // every NaN ranks above +inf
  else if (x == 0.0f) b = 0u;       // -0 == +0
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - idx);
}

__device__ __forceinline__ uint64_t max_u64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__global__ void __launch_bounds__(kAcceptThreads) accept_argmax_kernel(const float* __restrict__ logits,
                                                                        int vocab, uint64_t* part,
                                                                        uint32_t* ticket, int32_t* choice) {
  __shared__ uint64_t red[kRowsPerThread][kAcceptThreads / 32];
  __shared__ bool last;
  const int G = gridDim.x, b = blockIdx.x;
  const int n4 = vocab / 4;
  const int per = (n4 + G - 1) / G;
  const int c0 = min(n4, b * per), c1 = min(n4, c0 + per);
  uint64_t best[kRowsPerThread];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) best[r] = 0ull;  // below every element's key
  for (int c = c0 + (int)threadIdx.x; c < c1; c += kAcceptThreads) {
    float4 v[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) v[r] = __ldcs(reinterpret_cast<const float4*>(logits + (size_t)r * vocab) + c);
    const uint32_t i0 = (uint32_t)c * 4u;
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      best[r] = max_u64(best[r], max_u64(max_u64(argmax_key(v[r].x, i0), argmax_key(v[r].y, i0 + 1)),
                                         max_u64(argmax_key(v[r].z, i0 + 2), argmax_key(v[r].w, i0 + 3))));
    }
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    uint64_t x = best[r];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x = max_u64(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) red[r][wid] = x;
  }
  __syncthreads();
  if (threadIdx.x < kRowsPerThread) {
    uint64_t x = 0ull;
#pragma unroll
    for (int w = 0; w < kAcceptThreads / 32; ++w) x = max_u64(x, red[threadIdx.x][w]);
    part[(size_t)threadIdx.x * G + b] = x;
  }
  // the last block reduces every block's keys
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == (uint32_t)G - 1u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int r = threadIdx.x >> 4, sub = threadIdx.x & 15;  // 16 threads per row
  uint64_t x = 0ull;
  for (int i0 = 0; i0 < G; i0 += 16 * 8) {  // eight loads in flight per thread
    uint64_t y[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = i0 + q * 16 + sub;
      y[q] = i < G ? __ldcg(part + (size_t)r * G + i) : 0ull;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) x = max_u64(x, y[q]);
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) x = max_u64(x, __shfl_xor_sync(0xffffffffu, x, o));
  if (sub == 0) choice[r] = (int32_t)(0xFFFFFFFFu - (uint32_t)x);
  if (threadIdx.x == 0) *ticket = 0u;
}

__global__ void __launch_bounds__(kAcceptThreads) accept_walk_kernel(const AcceptParams p) {
  __shared__ int32_t s_arg[kRowsPerThread];
  __shared__ int32_t s_path[kRowsPerThread];
  __shared__ int32_t s_n, s_pos0;
  __shared__ int32_t s_par[kRowsPerThread], s_tok[kRowsPerThread];
  __shared__ int s_ok;
  if (threadIdx.x < 32) {
    // the tree, the draft tokens and pos0: launch parameters, or the device-resident
    // state checked here (parent[0] == -1, 0 <= parent[i] < i, tokens in [0, vocab),
    // 0 <= pos0 <= max_ctx - 16)
    const int i = threadIdx.x;
    int pv = 0, tv = 0, pos0 = p.pos0;
    if (i < kRowsPerThread) {
      pv = p.state ? p.state[1 + i] : p.parent[i];
      tv = p.state ? p.state[1 + kRowsPerThread + i] : p.tokens[i];
      s_arg[i] = p.choice[i];
      s_par[i] = pv;
      s_tok[i] = tv;
    }
    if (p.state) pos0 = p.state[0];
    const bool ok = __all_sync(0xffffffffu, i >= kRowsPerThread ||
                                                ((i == 0 ? pv == -1 : (pv >= 0 && pv < i)) && tv >= 0 && tv < p.vocab)) &&
                    pos0 >= 0 && pos0 <= p.max_ctx - kRowsPerThread;
    if (i == 0) {
      s_ok = ok;
      s_pos0 = pos0;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int cur = 0, n = 1;
    s_path[0] = 0;
    if (s_ok) {
      // from the root, the first child (in tree order) whose draft token is the
      // parent's greedy choice; stop at the first node without one
      for (;;) {
        int nxt = -1;
        for (int c = cur + 1; c < kRowsPerThread; ++c)
          if (s_par[c] == cur && s_tok[c] == s_arg[cur]) {
            nxt = c;
            break;
          }
        if (nxt < 0) break;
        s_path[n++] = nxt;
        cur = nxt;
      }
    } else {
      n = 0;  // nothing accepted, nothing moved
      if (blockIdx.x == 0 && p.status) atomicCAS(&p.status->code, 0, 1 /* MSM_ERR_INVALID_ARG */);
    }
    s_n = n;
    if (p.result != nullptr && blockIdx.x == 0) {
      p.result[0] = n;
      p.result[1] = n ? s_arg[cur] : -1;
      for (int j = 0; j < kRowsPerThread; ++j) {
        p.result[2 + j] = j < n ? s_path[j] : -1;
        p.result[2 + kRowsPerThread + j] = s_arg[j];
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  if (n <= 1) return;
  const int chunks = p.head_dim / 8;  // 16-byte chunks per row
  const int per_layer = 2 * p.n_kv_heads * chunks;
  const int cols = p.n_layers * per_layer;
  for (int col = blockIdx.x * kAcceptThreads + threadIdx.x; col < cols; col += gridDim.x * kAcceptThreads) {
    const int l = col / per_layer, rem = col - l * per_layer;
    const int kv = rem / (p.n_kv_heads * chunks), rem2 = rem - kv * (p.n_kv_heads * chunks);
    const int h = rem2 / chunks, ch = rem2 - h * chunks;
    uint16_t* base = (kv ? p.vc[l] : p.kc[l]) + ((size_t)h * p.max_ctx + s_pos0) * p.head_dim + ch * 8;
    uint4 v[kRowsPerThread - 1];
#pragma unroll
    for (int j = 1; j < kRowsPerThread; ++j)
      if (j < n && s_path[j] != j) v[j - 1] = *reinterpret_cast<const uint4*>(base + (size_t)s_path[j] * p.head_dim);
#pragma unroll
    for (int j = 1; j < kRowsPerThread; ++j)
      if (j < n && s_path[j] != j) *reinterpret_cast<uint4*>(base + (size_t)j * p.head_dim) = v[j - 1];
  }
}

// The draft's proposal into a device-resident step state: the tree becomes the chain
// (parent[i] = i - 1) and node i >= 1 takes slot i's greedy choice; the root's token
// (state[17]) is the caller's and stays.
__global__ void draft_propose_kernel(const int32_t* __restrict__ choice, int32_t* state) {
  const int i = threadIdx.x;
  if (i < kRowsPerThread) {
    state[1 + i] = i - 1;
    if (i > 0) state[1 + kRowsPerThread + i] = choice[i];
  }
}

// Rows of an embedding table for the 16 tree tokens of a step state: out[i] =
// table[state[17 + i]]; an id outside [0, vocab) gives a zero row and reports
// MSM_ERR_INVALID_ARG through the status (the verify step's own state check then
// gives the step up).  One block per token, 16-byte chunks.
__global__ void embed_kernel(const uint16_t* __restrict__ table, int vocab, int d, const int32_t* __restrict__ state,
                             uint16_t* __restrict__ out, DevStatus* status) {
  const int i = blockIdx.x;
  const int id = state[1 + kRowsPerThread + i];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && threadIdx.x == 0 && status) atomicCAS(&status->code, 0, 1 /* MSM_ERR_INVALID_ARG */);
  const uint4* src = reinterpret_cast<const uint4*>(table + (size_t)(ok ? id : 0) * d);
  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)i * d);
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) dst[c] = ok ? src[c] : make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_draft_propose(const int32_t* choice, int32_t* state, cudaStream_t s) {
  draft_propose_kernel<<<1, 32, 0, s>>>(choice, state);
  return cudaGetLastError();
}

cudaError_t launch_embed(const void* table, int vocab, int d, const int32_t* state, void* out, DevStatus* status,
                         cudaStream_t s) {
  embed_kernel<<<kRowsPerThread, 256, 0, s>>>(static_cast<const uint16_t*>(table), vocab, d, state,
                                              static_cast<uint16_t*>(out), status);
  return cudaGetLastError();
}

cudaError_t launch_accept_argmax(const float* logits, int vocab, uint64_t* part, int parts, uint32_t* ticket,
                                 int32_t* choice, cudaStream_t s) {
  accept_argmax_kernel<<<parts, kAcceptThreads, 0, s>>>(logits, vocab, part, ticket, choice);
  return cudaGetLastError();
}

cudaError_t launch_accept_walk(const AcceptParams& p, int blocks, cudaStream_t s) {
  accept_walk_kernel<<<blocks, kAcceptThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace msm
