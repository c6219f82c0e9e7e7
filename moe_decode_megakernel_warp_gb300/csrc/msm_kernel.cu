// The per-layer persistent kernel of the verify step (sm_103a).
//
// One launch runs, on every SM, one 384-thread block with fixed warp roles
// (alphasignal.ai, "LMSYS Doubles Muse Spark Open Speed to 1,109 Tokens per
// Second", § "A 12-warp pipeline takes over scheduling"; orcarouter.ai,
// "Muse Spark Open: 1,109 tokens/s is a kernel-level change", § "where the
// kernel boundary sits"):
//   warp 0      TMA producer: streams the block's weight tiles (and KV tiles)
//               into a shared-memory ring, running ahead into the next op's
//               weights while the current op waits for its inputs
//   warps 1-2   re-arm the exchange buffers the next launch will use
//   warp 3      L2 prefetch of the previous step's most-used experts
//   warps 4-11  attention, dense GEMMs, expert GEMMs, combines
// The launch covers layer l's attention through layer l+1's QKV projection and
// KV-cache write (alphasignal.ai, § "Launch boundaries leave hardware idle").
// Blocks hand each phase's output to each other through global memory. Every
// block, once it has stored its share, adds 1 to that phase's counter after a
// gpu-scope fence, and consumers wait for the counter to reach the grid size:
// on one GPU every dense phase's output is read by all blocks, and polling each
// element while producers write held consumers far longer than one counter.
// The expert GEMM1 -> GEMM2 rows and the prologue's Q / tree K/V keep the
// pages' data-as-flag slots: empty while they hold a sentinel (0xFFFF for bf16,
// an all-ones NaN no rounding produces; -0.0 for fp32, since writers store
// x+0.0), polled in the payload itself (alphasignal.ai, § "Four mechanisms keep
// work moving"; orcarouter.ai, § "three bills").  Every wait is bounded by
// %globaltimer.
#include "msm_device.cuh"
#include "msm_internal.h"

namespace msm {

// ---------------------------------------------------------------------------
// shared memory carve-up
// ---------------------------------------------------------------------------
struct Smem {
  uint8_t* ring;
  uint8_t* act;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* route_bar;
  uint32_t* slot_off;
  volatile int* abort;
  int* n_active;
  int* pos0;          // first tree row of this step (the launch parameter or the device state)
  uint64_t* stage_bar;  // completion of the activation tensor copies
  uint32_t* anc;
  int32_t* tpos;
  int32_t* depth;
  int32_t* topk_idx;  // [16][8]
  float* topk_w;      // [16][8]
  int16_t* act_e;     // [128]
  uint8_t* act_n;     // [128]
  uint8_t* act_tok;   // [128][16]
  uint8_t* act_slot;  // [128][16]
  float* x_ts;        // [16]
  float* a_ts;        // [2][16]
  float* red;         // [8][16]
  volatile uint32_t* slot_tile;  // [kSlots] index of the tile the loader last put in each slot
  struct RunAhead* ring_state;    // the loader's L2 run-ahead lists
  float* dred;        // [8][16][16] dense-phase cross-warp partial sums
  uint64_t* tcbar;    // tensor-core pipeline barriers (TcBar)
  uint32_t* tmem_base;  // tensor-memory columns of the block (written by the allocating warp)
  uint32_t* tc_ti;      // [1]: first ring tile of GEMM2 (for the tensor-core warp)
  uint32_t* dq_e;       // [kDenseQ] the loader's hand-over queue to the tensor-core warp:
  volatile uint32_t* dq_seq;  // dense tiles (ring index | 2 KB chunks << 24) and markers
};
constexpr int kDenseQ = 32;
constexpr uint32_t kDqRoute = 0xFFFFFFFEu;  // marker: the loader waits for the routing now
constexpr uint32_t kDqEnd = 0xFFFFFFFFu;    // marker: the launch's stream is done

// Tensor-core pipeline of the expert GEMMs: mbarriers between the tensor-core warp (MMA
// and scale-copy issue) and the compute warp groups (operand staging, epilogues).
enum TcBar : int {
  TB_D1_FULL = 0,    // [2 parities] a unit's GEMM1 accumulator complete (commit)
  TB_D1_FREE = 2,    // [2] ... read by the unit's epilogue (4 warps)
  TB_SFA_DONE = 4,   // [4] the MMAs that read a weight-scale buffer are done (commit)
  TB_D2_FULL = 8,    // [2]
  TB_D2_FREE = 10,   // [2] (4 warps)
  TB_G2_STAGE = 12,  // a GEMM2 round's activations and their block scales staged
  TB_DONE = 13,      // the compute warps are done with tensor memory (8 warps)
  TB_DRAIN = 14,     // every MMA of the tensor-core warp has completed
  TB_ROUTED = 15,    // the block's routing (expert list, first expert tile) is in shared memory
  TB_B1 = 16,        // GEMM1's operand B has landed in the activation buffer (transaction count)
  TB_SFA_FULL = 17,  // [4] a tile's weight scales are in a scale buffer (4 warps)
  TB_SFB1 = 21,      // GEMM1's operand-B scales are in tensor memory (commit)
  TB_SLOT = 22,      // [kSlots] the tensor-core reads of the weight tile in a ring slot are
                     // done (commit): the loader's release of expert and dense tiles (one
                     // commit; the KV tiles' consumers arrive on the slot's `empty` barrier)
  TB_TFULL = TB_SLOT + kSlots,           // [kDenseTmemSlots] a dense tile is in tensor memory (commit)
  TB_TFREE = TB_TFULL + kDenseTmemSlots,  // [kDenseTmemSlots] ... read by the 4 warps of its group
  TB_XDONE = TB_TFREE + kDenseTmemSlots,  // the expert phases' tensor-memory reads are done (8 warps)
  kTcBars
};
// tensor-memory columns (512 allocated: one block per SM).  GEMM2 reuses GEMM1's
// operand-scale and accumulator columns: its first tensor-memory write follows every
// GEMM1 epilogue, and so every GEMM1 MMA.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_SFB1 = 0;    // GEMM1 operand-B scales: 4 columns per K=64 step (p / 64 steps)
constexpr uint32_t TM_SFA = 128;   // 4 x 32: weight scales of a tile (up to 8 K=64 steps x 4 columns)
constexpr uint32_t TM_D1 = 256;    // 2 x 64: GEMM1 accumulators, column term * 16 + token
constexpr uint32_t TM_SFB2 = 0;    // 2 x 64: GEMM2 activation scales of a round's two experts
constexpr uint32_t TM_D2 = 256;    // 2 x 16: GEMM2 accumulators
// Outside the expert phases all 512 columns hold dense weight tiles: slot j (64 columns)
// takes the block's dense tiles di = j, j + 8, ...; lane 32 q + t, columns 4c .. 4c + 3
// hold the A fragment of k-step 4c + q as thread t of warp q reads it (the packed layout)
constexpr uint32_t kDenseTmemCols = 64;
static_assert(kDenseTmemSlots * kDenseTmemCols == kTmemCols, "dense tiles fill the tensor memory");

constexpr int kRingStateOff = 6656;  // in the small area, below the GEMM2 row scales
constexpr int kATsOff = 7936;        // [2][16] floats, below the reduction scratch at 8192
__device__ __forceinline__ Smem carve(uint8_t* base, const LaunchParams& P) {
  Smem s;
  s.ring = base;
  s.act = base + P.ring_bytes;
  uint8_t* sm = s.act + P.act_bytes;
  s.full = reinterpret_cast<uint64_t*>(sm + 0);
  s.empty = reinterpret_cast<uint64_t*>(sm + 96);
  s.route_bar = reinterpret_cast<uint64_t*>(sm + 192);
  s.slot_off = reinterpret_cast<uint32_t*>(sm + 200);
  s.abort = reinterpret_cast<volatile int*>(sm + 248);
  s.n_active = reinterpret_cast<int*>(sm + 252);
  s.anc = reinterpret_cast<uint32_t*>(sm + 256);
  s.tpos = reinterpret_cast<int32_t*>(sm + 320);
  s.depth = reinterpret_cast<int32_t*>(sm + 384);
  s.topk_idx = reinterpret_cast<int32_t*>(sm + 448);
  s.topk_w = reinterpret_cast<float*>(sm + 960);
  s.act_e = reinterpret_cast<int16_t*>(sm + 1472);
  s.act_n = sm + 1728;
  s.act_tok = sm + 1856;
  s.act_slot = sm + 3904;
  s.x_ts = reinterpret_cast<float*>(sm + 5952);
  s.a_ts = reinterpret_cast<float*>(sm + kATsOff);
  s.red = reinterpret_cast<float*>(sm + 6080);
  s.slot_tile = reinterpret_cast<volatile uint32_t*>(sm + 6592);
  s.pos0 = reinterpret_cast<int*>(sm + 6640);
  s.stage_bar = reinterpret_cast<uint64_t*>(sm + 6648);
  s.ring_state = reinterpret_cast<struct RunAhead*>(sm + kRingStateOff);
  s.dred = reinterpret_cast<float*>(sm + 8192);
  s.tc_ti = reinterpret_cast<uint32_t*>(sm + 7416);
  s.tmem_base = reinterpret_cast<uint32_t*>(sm + 7420);
  s.tcbar = reinterpret_cast<uint64_t*>(sm + 7424);
  s.dq_e = reinterpret_cast<uint32_t*>(sm + 7040);
  s.dq_seq = reinterpret_cast<volatile uint32_t*>(sm + 7168);
  return s;
}

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// A bounded wait ran out: record it in the status word and make every wait give up.
// Out of line, and with no pointer to the context: a call that took the context's
// address would keep the whole context in local memory for the launch.
__device__ __noinline__ void fail_timeout(const LaunchParams* P, volatile int* abort, int block, int phase) {
  *abort = 1;
  if (atomicCAS(&P->status->code, 0, 4 /* MSM_ERR_DEVICE_TIMEOUT */) == 0) {
    P->status->phase = phase;
    P->status->block = block;
    P->status->layer = P->layer;
  }
  atomicExch(&P->status->abort, 1);
}
struct Ctx {
  const LaunchParams* P;
  Smem S;
  uint64_t deadline;
  int pos0;  // copy of *S.pos0
  uint32_t stage_n = 0;  // activation stagings by tensor copies so far (stage_bar's phase)
  uint64_t next_abort_check = 0;
  int block;

  __device__ __forceinline__ void fail(int phase) { fail_timeout(P, S.abort, block, phase); }
  // true when the caller must give up.  The grid-wide abort word lives in global
  // memory: it is read at most every 4 us per thread, since a global round trip in
  // a spin loop would delay the caller's notice of the very data it waits for.
  __device__ __forceinline__ bool expired(int phase) {
    if (*S.abort) return true;
    const uint64_t now = globaltimer();
    if (now > deadline) {
      fail(phase);
      return true;
    }
    if (now >= next_abort_check) {
      next_abort_check = now + 4000;
      if (ld_relaxed_u32(&P->status->abort) != 0) {
        *S.abort = 1;
        return true;
      }
    }
    return false;
  }
};

__device__ __forceinline__ bool wait_bar(Ctx& cx, uint64_t* bar, uint32_t parity, int phase) {
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 15) == 0 && cx.expired(phase)) return false;
  }
  return true;
}

// Wait until tile t of the block's sequence has landed.  A slot's mbarrier only
// tells phases apart by parity, so a consumer first waits until the loader has
// put tile t in its slot (the slot then cannot move on before t is released) and
// only then tests the parity of t's phase.
__device__ __forceinline__ bool wait_tile(Ctx& cx, uint32_t t, int phase) {
  const uint32_t s = t % kSlots;
  uint32_t n = 0;
  while (cx.S.slot_tile[s] != t) {
    if ((++n & 15) == 0 && cx.expired(phase)) return false;
  }
  return wait_bar(cx, &cx.S.full[s], (t / kSlots) & 1, phase);
}

// poll a 16-byte bf16 chunk until none of its 8 elements is the sentinel
__device__ __forceinline__ bool poll_bf16x8(Ctx& cx, const void* p, uint4& v, int phase) {
  uint32_t n = 0;
  v = ld_relaxed_v4(p);
  while (!bf16x8_ready(v)) {
    if ((++n & 31) == 0 && cx.expired(phase)) return false;
    v = ld_relaxed_v4(p);
  }
  return true;
}

// Poll up to N 16-byte chunks together: every pending chunk is re-read in the same
// round, so a consumer that arrives before its producers keeps N loads in flight
// instead of waiting out one round trip per chunk.  `ready` tells whether a chunk
// holds no sentinel; returns false if the block gave up.
template <int N, class Ready>
__device__ __forceinline__ bool poll_batch(Ctx& cx, const uint4* base, int stride, uint4 (&v)[N], uint32_t pending,
                                           Ready ready, int phase) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    if ((pending >> i) & 1u) v[i] = ld_relaxed_v4(base + i * stride);
  uint32_t n = 0;
  for (;;) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (((pending >> i) & 1u) && ready(v[i])) pending &= ~(1u << i);
    if (!pending) return true;
    if ((++n & 7) == 0 && cx.expired(phase)) return false;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((pending >> i) & 1u) v[i] = ld_relaxed_v4(base + i * stride);
  }
}

// one thread per block records: the first compute thread, or the loader lane
template <bool kTiming>
__device__ __forceinline__ void stamp(const LaunchParams& P, int block, int ev) {
  if (kTiming && (threadIdx.x == kFirstCompute * 32 || threadIdx.x == 0))
    P.timing[(size_t)block * kTimingEvents + ev] = globaltimer();
}

// stamp of any one thread (runtime flag)
__device__ __forceinline__ void stamp_any(const LaunchParams& P, int ev) {
  if (P.flags & 0x1u) P.timing[(size_t)blockIdx.x * kTimingEvents + ev] = globaltimer();
}
// sub-phase stamps inside helpers shared by both kernel variants (runtime flag)
__device__ __forceinline__ void stamp_rt(const LaunchParams& P, int ev) {
  if ((P.flags & 0x1u) && threadIdx.x == kFirstCompute * 32)
    P.timing[(size_t)blockIdx.x * kTimingEvents + ev] = globaltimer();
}

// ---------------------------------------------------------------------------
// work split (identical in the loader and the consumers)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void unit_range(int n_units, int bb, int G, int& lo, int& hi) {
  // 32-bit: n_units * G stays far below 2^32 for every shape the host accepts (a
  // 64-bit division is a long subroutine, inlined at every call site)
  lo = (int)(((uint32_t)n_units * (uint32_t)bb) / (uint32_t)G);
  hi = (int)(((uint32_t)n_units * (uint32_t)(bb + 1)) / (uint32_t)G);
}
__device__ __forceinline__ int rot_block(int b, int rot, int G) { return (b + rot) % G; }
// The expert units: n / G units per block, the n % G extra ones on the first blocks for
// GEMM1 (so its later-finishing sixth units all belong to the first experts) and on the
// last blocks for GEMM2 (whose first experts' inputs are then the late ones, on blocks
// with one unit less)
__device__ __forceinline__ void expert_units(int n_units, int bb, int G, bool gemm2, int& lo, int& hi) {
  const int q = n_units / G, x = n_units - q * G;
  if (!gemm2) {
    lo = bb * q + min(bb, x);
    hi = lo + q + (bb < x ? 1 : 0);
  } else {
    lo = bb * q + max(0, bb - (G - x));
    hi = lo + q + (bb >= G - x ? 1 : 0);
  }
}

// attention unit of block bb: kv head, split, row range
struct AttnUnit {
  int valid, hk, s, r0, r1, n_sub, tree;
};
__device__ __forceinline__ AttnUnit attn_unit(const LaunchParams& P, int pos0, int bb, int is_global) {
  const Dims& dm = P.dm;
  AttnUnit u;
  u.valid = bb < dm.hkv * dm.splits;
  u.hk = u.valid ? bb / dm.splits : 0;
  u.s = u.valid ? bb % dm.splits : 0;
  int lo = is_global ? 0 : max(0, pos0 - dm.window + 1);
  int n = pos0 - lo;
  int chunk = (n + dm.splits - 1) / dm.splits;
  chunk = ((chunk + dm.kv_rows - 1) / dm.kv_rows) * dm.kv_rows;
  if (chunk < dm.kv_rows) chunk = dm.kv_rows;
  u.r0 = min(pos0, lo + u.s * chunk);
  u.r1 = min(pos0, u.r0 + chunk);
  u.n_sub = u.valid ? (u.r1 - u.r0 + dm.kv_rows - 1) / dm.kv_rows : 0;
  u.tree = u.valid && (u.s == dm.splits - 1);
  return u;
}

// ---------------------------------------------------------------------------
// the variable-size shared-memory ring (producer side)
// ---------------------------------------------------------------------------
// L2 run-ahead: the byte ranges the block's loader will stream, in stream order.
// A cursor keeps cp.async.bulk.prefetch.L2 requests up to `ahead` bytes in front
// of what the ring has issued, so HBM keeps streaming while the ring waits on
// its consumers (weights and KV history do not depend on the computation; the
// expert ranges are appended once the routing is known).  A hint only: ranges
// that do not fit the table are simply not prefetched.
constexpr int kMaxRanges = 24;
struct RunAhead {
  const uint8_t* p[kMaxRanges];
  uint32_t n[kMaxRanges];
  int count, i;
  uint32_t off;
  uint64_t pref, used;
  uint32_t ahead;  // 0 = off
  __device__ void init(uint32_t a) {
    count = i = 0;
    off = 0;
    pref = used = 0;
    ahead = a;
  }
  // (ptr == nullptr: bytes the ring streams that are not prefetched)
  __device__ void add(const void* ptr, uint64_t bytes) {
    if (!ahead || bytes == 0 || count == kMaxRanges) return;
    p[count] = static_cast<const uint8_t*>(ptr);
    n[count] = (uint32_t)bytes;
    ++count;
  }
  __device__ void pump() {
    while (i < count && pref < used + ahead) {
      const uint32_t c = min(n[i] - off, 65536u);
      if (p[i]) prefetch_l2(p[i] + off, c);
      off += c;
      pref += c;
      if (off == n[i]) {
        ++i;
        off = 0;
      }
    }
  }
};

// The loader's view of the ring: a FIFO of tiles laid out circularly.  Only scalars,
// so that they stay in the loader lane's registers; a tile's offset is read back from
// the slot table in shared memory once, when the tile before it is released.
struct Ring {
  uint32_t cap;       // bytes the ring may use now (grows during the expert phases)
  uint32_t xmask;     // bit s: slot s holds an expert tile (released through TB_SLOT + s)
  uint32_t par_e;     // bit s: parity of slot s's next `empty` phase
  uint32_t par_x;     // bit s: ... of its next TB_SLOT phase
  uint32_t issued;    // tiles issued
  uint32_t tail;      // oldest tile not known to be released
  uint32_t head;      // end of the newest tile
  uint32_t tail_off;  // start of the oldest outstanding tile (tail < issued)
  bool wrapped;       // the outstanding tiles run to the top and continue at 0
  bool ra_on;         // L2 run-ahead enabled
  bool routed;        // the block's routing is done: expert tiles may use the bottom of the activation buffer
  bool sfb_free;      // ... and GEMM1's operand-B scale groups above it
  RunAhead* ra;       // L2 run-ahead state (shared memory)
};
static_assert(kRingStateOff + sizeof(RunAhead) <= 7040, "run-ahead state overlaps the dense hand-over queue");
static_assert(7168 + kDenseQ * 4 <= 7416, "dense hand-over queue overlaps the tensor-core barriers");
static_assert(7424 + kTcBars * 8 <= kATsOff, "tensor-core barriers overlap the GEMM2 row scales");
static_assert(TM_SFB1 + 2048 / 64 * 4 <= TM_SFA && TM_SFB2 + 2 * 64 <= TM_SFA && TM_SFA + 4 * 32 <= TM_D1 &&
              TM_D1 + 2 * kSplitRows <= kTmemCols && TM_D2 + 32 <= kTmemCols, "tensor-memory map");

// a free run of `bytes` (1 KB granules) after the newest tile, at the bottom once the
// top is too short; waits for the oldest tiles' release until there is one
__device__ __forceinline__ bool ring_place(Ctx& cx, Ring& r, uint32_t bytes, uint32_t& off_out) {
  const uint32_t cap = r.cap;
  const uint32_t need = (bytes + 1023u) & ~1023u;
  uint32_t off = 0;
  for (;;) {
    if (r.issued - r.tail < (uint32_t)kSlots) {
      if (r.tail == r.issued) {  // empty: start again at the bottom
        r.wrapped = false;
        off = 0;
        r.tail_off = 0;
        break;
      }
      if (!r.wrapped) {  // occupied: [tail_off, head)
        if (r.head + need <= cap) { off = r.head; break; }
        if (need <= r.tail_off) { off = 0; r.wrapped = true; break; }
      } else if (r.head + need <= r.tail_off && r.head + need <= cap) {  // occupied: [tail_off, top) and [0, head)
        off = r.head;
        break;
      }
    }
    const uint32_t s = r.tail % kSlots, bit = 1u << s;
    if (r.xmask & bit) {
      if (!wait_bar(cx, &cx.S.tcbar[TB_SLOT + s], (r.par_x & bit) ? 1u : 0u, 99)) return false;
      r.par_x ^= bit;
    } else {
      if (!wait_bar(cx, &cx.S.empty[s], (r.par_e & bit) ? 1u : 0u, 99)) return false;
      r.par_e ^= bit;
    }
    ++r.tail;
    if (r.tail != r.issued) {
      const uint32_t next = cx.S.slot_off[r.tail % kSlots];
      if (next < r.tail_off) r.wrapped = false;  // the span no longer crosses the top
      r.tail_off = next;
    }
  }
  off_out = off;
  r.head = off + need;
  return true;
}

// the contiguous bytes of this block's units of a dense weight (run-ahead lists)
__device__ void add_dense_range(RunAhead& ra, const uint8_t* W, int K, int N, int rot) {
  int lo, hi;
  unit_range(N / 16, rot_block(blockIdx.x, rot, gridDim.x), gridDim.x, lo, hi);
  const uint64_t ub = dense_unit_bytes(K);
  ra.add(W + (uint64_t)lo * ub, (uint64_t)(hi - lo) * ub);
}

// L2 run-ahead lists (off by default): kept out of line, so that the loader's hot
// path stays small in the instruction cache
__device__ __noinline__ void ra_front(const LaunchParams& P, RunAhead* ra, int block, int r0, int r1, int hk) {
  const Dims& dm = P.dm;
  // everything up to the routing decision, in the order the ring streams it
  if (P.first) add_dense_range(*ra, P.w_qkv_pro, dm.d, dm.nqkv, P.phase_rot * 1);
  if (r1 > r0) {
    const uint64_t off = ((uint64_t)hk * dm.max_ctx + r0) * dm.hd, bytes = (uint64_t)(r1 - r0) * dm.hd * 2;
    ra->add(P.kc + off, bytes);
    ra->add(P.vc + off, bytes);
  }
  add_dense_range(*ra, P.w_o, dm.hq * dm.hd, dm.d, P.phase_rot * 3);
  if (dm.draft) {
    // a draft model's whole stream: the FFN, then the next layer's QKV or the LM head
    add_dense_range(*ra, P.w_up, dm.d, 2 * dm.f, P.phase_rot * 4);
    add_dense_range(*ra, P.w_down, dm.f, dm.d, P.phase_rot * 5);
    if (!P.last) add_dense_range(*ra, P.w_tail, dm.d, dm.nqkv, P.phase_rot * 9);
    else add_dense_range(*ra, P.w_tail, dm.d, dm.vocab, P.phase_rot * 9);
  } else {
    add_dense_range(*ra, P.w_pool, dm.d, dm.p, P.phase_rot * 4);
    add_dense_range(*ra, P.w_router, dm.p, dm.e, P.phase_rot * 5);
  }
  if (block == 0) {
    prefetch_l2(P.g_moe, (uint32_t)dm.d * 2);
    if (P.g_tail) prefetch_l2(P.g_tail, (uint32_t)dm.d * 2);
  }
  ra->pump();
}
__device__ __noinline__ void ra_back(const LaunchParams& P, RunAhead* ra, int block, int na) {
  const Dims& dm = P.dm;
  const int G = gridDim.x;
  const int u1pe = w1_units(dm.f), u2pe = w2_units(dm.p);
  const uint64_t ub1 = exp_unit_bytes(dm.p), ub2 = exp_unit_bytes(dm.f);
  // the rest of the launch's stream: this block's expert units (runs of one expert
  // are contiguous), the unpooler, then the next layer's QKV or the LM head
  for (int pass = 0; pass < 2; ++pass) {
    const int upe = pass ? u2pe : u1pe;
    const uint64_t ub = pass ? ub2 : ub1;
    int lo, hi;
    expert_units(na * upe, rot_block(block, P.phase_rot * (pass ? 7 : 6), G), G, pass != 0, lo, hi);
    for (int gu = lo; gu < hi;) {
      const int run = min(hi, (gu / upe + 1) * upe) - gu;
      ra->add(nullptr, (uint64_t)run * ub);  // expert tiles: streamed, not prefetched
      gu += run;
    }
  }
  add_dense_range(*ra, P.w_unpool, dm.p, dm.d, P.phase_rot * 8);
  if (!P.last) add_dense_range(*ra, P.w_tail, dm.d, dm.nqkv, P.phase_rot * 9);
  else if (dm.vocab > 0) add_dense_range(*ra, P.w_tail, dm.d, dm.vocab, P.phase_rot * 9);
  ra->pump();
}
__device__ __noinline__ void ra_pump(RunAhead* ra, uint32_t bytes) {
  ra->used += bytes;
  ra->pump();
}

// The launch's tile stream in consumption order, produced one tile per call of next()
// (one copy of the issue path, instead of one inlined per weight): segment 0 the
// prologue QKV (launch 0), 1 this block's KV tiles, 2 the dependency wait, 3 o_proj,
// 4 pooler, 5 router, 6 this block's routing decision, 7 GEMM1 units, 8 GEMM2 units,
// 9 unpooler, 10 the next layer's QKV or the LM head.  Only scalars (registers).
enum : int { TS_TILE = 0, TS_KV = 1, TS_DEP_WAIT = 2, TS_ROUTE_WAIT = 3, TS_END = 4 };
struct TileStream {
  int seg;
  int lo, hi, u;     // units of the segment; u: unit of the next tile (dense: of its pair)
  int half;          // dense: the next tile is of unit u + half (units go in pairs, tiles alternating)
  int k0, steps;     // dense: next k-step within unit u; k-steps per unit
  int kb;            // dense: first k-step of the streamed range (a K half of the unit)
  int upe;           // experts: units per expert
  uint64_t ub;       // bytes per unit
  const uint8_t* W;  // weights of the segment
  int kv_r0, kv_hk;  // KV: first row, kv head
  // the tile just produced: its unit and first k-step (for the loader's stamps)
  int t_u, t_k0;

  __device__ void dense(const uint8_t* w, int K, int N, int rot) {
    unit_range(N / 16, rot_block(blockIdx.x, rot, gridDim.x), gridDim.x, lo, hi);
    u = lo;
    half = 0;
    k0 = 0;
    kb = 0;
    steps = K / 16;
    ub = dense_unit_bytes(K);
    W = w;
  }
  // K half h of every unit (a draft model's FFN down projection, its input staged in halves)
  __device__ void dense_half(const uint8_t* w, int K, int N, int rot, int h) {
    dense(w, K, N, rot);
    steps = K / 32;
    kb = h * steps;
  }
  // expert units: 128 rows x K as K / exp_tile_k(K) tiles of exp_tile_bytes(K) each
  __device__ void experts(const uint8_t* w, int n_units, int per_expert, int K, int rot, bool gemm2) {
    expert_units(n_units, rot_block(blockIdx.x, rot, gridDim.x), gridDim.x, gemm2, lo, hi);
    u = lo;
    k0 = 0;
    steps = K / exp_tile_k(K);
    upe = per_expert;
    ub = (uint64_t)exp_tile_bytes(K);
    W = w;
  }
  // the launch's stream starts with segment 0: the prologue QKV (launch 0 only)
  __device__ void begin(const LaunchParams& P) {
    seg = 0;
    lo = hi = u = k0 = half = kb = 0;
    if (P.first) dense(P.w_qkv_pro, P.dm.d, P.dm.nqkv, P.phase_rot * 1);
  }
  // TS_TILE: src / bytes set; TS_KV: kv_row set; else a wait or the end.  kDraft: the
  // stream of a draft model's launch (a separate kernel, so that the target's carries
  // none of the draft's code)
  template <bool kDraft>
  __device__ __forceinline__ int next(const Ctx& cx, const uint8_t*& src, uint32_t& bytes, int& kv_row) {
    const LaunchParams& P = *cx.P;
    const Dims& dm = P.dm;
    for (;;) {
      if (u < hi) {
        t_u = u;
        t_k0 = k0;
        if (seg == 1) {
          kv_row = kv_r0 + (u - lo) * dm.kv_rows;
          bytes = (uint32_t)dm.kv_rows * dm.hd * 2 * 2;
          ++u;
          return TS_KV;
        }
        if (seg == 7 || seg == 8) {
          const int e = cx.S.act_e[u / upe];
          src = W + (((uint64_t)e * upe + u % upe) * steps + k0) * ub;
          bytes = (uint32_t)ub;
          if (++k0 == steps) {
            k0 = 0;
            ++u;
          }
          return TS_TILE;
        }
        // dense: the block's units in pairs (u, u + 1), their tiles alternating, so the two
        // compute warp groups (one unit each) stream side by side
        const int uu = u + half, ns = min(kDenseTileSteps, steps - k0);
        t_u = uu;
        src = W + (uint64_t)uu * ub + (uint64_t)(kb + k0) * kKStepBytes;
        bytes = (uint32_t)ns * kKStepBytes;
        if (half == 0 && u + 1 < hi) {
          half = 1;
        } else {
          half = 0;
          k0 += kDenseTileSteps;
          if (k0 >= steps) {
            k0 = 0;
            u += 2;
          }
        }
        return TS_TILE;
      }
      ++seg;
      lo = hi = u = k0 = half = kb = 0;
      switch (seg) {
        case 1: {
          const AttnUnit au = attn_unit(P, cx.pos0, rot_block(cx.block, P.phase_rot * 2, gridDim.x), P.is_global);
          hi = au.n_sub;
          kv_r0 = au.r0;
          kv_hk = au.hk;
          break;
        }
        case 2: return TS_DEP_WAIT;
        case 3: dense(P.w_o, dm.hq * dm.hd, dm.d, P.phase_rot * 3); break;
        // a draft model: 4 = the FFN's paired gate/up rows, 5 and 6 = the two K halves of
        // its down projection; no expert segments and no unpooler
        case 4:
          if (kDraft) dense(P.w_up, dm.d, 2 * dm.f, P.phase_rot * 4);
          else dense(P.w_pool, dm.d, dm.p, P.phase_rot * 4);
          break;
        case 5:
          if (kDraft) dense_half(P.w_down, dm.f, dm.d, P.phase_rot * 5, 0);
          else dense(P.w_router, dm.p, dm.e, P.phase_rot * 5);
          break;
        case 6:
          if (!kDraft) return TS_ROUTE_WAIT;
          dense_half(P.w_down, dm.f, dm.d, P.phase_rot * 5, 1);
          break;
        case 7:
          if (!kDraft) experts(P.w1, *cx.S.n_active * w1_units(dm.f), w1_units(dm.f), dm.p, P.phase_rot * 6, false);
          break;
        case 8:
          if (!kDraft) experts(P.w2, *cx.S.n_active * w2_units(dm.p), w2_units(dm.p), dm.f, P.phase_rot * 7, true);
          break;
        case 9:
          if (!kDraft) dense(P.w_unpool, dm.p, dm.d, P.phase_rot * 8);
          break;
        case 10:
          if (!P.last) dense(P.w_tail, dm.d, dm.nqkv, P.phase_rot * 9);
          else if (dm.vocab > 0) dense(P.w_tail, dm.d, dm.vocab, P.phase_rot * 9);
          break;
        default: return TS_END;
      }
    }
  }
};

// an entry of the dense hand-over queue (the loader's q-th): written, then published
__device__ __forceinline__ void dq_push(Ctx& cx, uint32_t& q, uint32_t e) {
  const uint32_t k = q % kDenseQ;
  cx.S.dq_e[k] = e;
  __threadfence_block();
  cx.S.dq_seq[k] = ++q;
}

template <bool kTiming, bool kDraft>
__device__ void loader(Ctx& cx) {
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const uint64_t pol = policy_evict_first();
  prefetch_tensormap(&P.tmap_k);
  prefetch_tensormap(&P.tmap_v);
  // the run-ahead lists live in shared memory: as local arrays they would sit in the
  // small L1 left beside a 227 KB carve-out, and their lines, evicted by the compute
  // warps' traffic, would cost the loader an L2 round trip per access
  Ring r;
  r.cap = (uint32_t)P.ring_bytes;
  r.xmask = r.par_e = r.par_x = 0u;
  r.routed = r.sfb_free = false;
  r.issued = r.tail = r.head = r.tail_off = 0;
  r.wrapped = false;
  r.ra = cx.S.ring_state;
  r.ra->init(P.runahead_bytes);
  r.ra_on = P.runahead_bytes != 0;
  // segment 0: the prologue QKV (launch 0); weights and KV rows do not depend on the
  // previous launch, so they stream before the dependency wait
  TileStream ts;
  ts.begin(P);
  if (r.ra_on) {
    const AttnUnit au = attn_unit(P, cx.pos0, rot_block(cx.block, P.phase_rot * 2, gridDim.x), P.is_global);
    ra_front(P, r.ra, cx.block, au.valid ? au.r0 : 0, au.valid ? au.r1 : 0, au.hk);
  }
  bool ok = true;
  int g1_last = -1;
  uint32_t dq = 0;  // entries of the dense hand-over queue
  while (ok) {
    const uint8_t* src = nullptr;
    uint32_t bytes = 0;
    int kv_row = 0;
    const int st = ts.template next<kDraft>(cx, src, bytes, kv_row);
    if (st == TS_END) break;
    if (st == TS_DEP_WAIT) {
      // the deadline of the bounded waits starts once the previous launch is done
      pdl_wait();
      cx.deadline = globaltimer() + (((uint64_t)P.timeout_ns_hi << 32) | P.timeout_ns_lo);
      continue;
    }
    if (st == TS_ROUTE_WAIT) {
      // expert tiles wait for this block's routing decision
      dq_push(cx, dq, kDqRoute);
      ok = wait_bar(cx, cx.S.route_bar, 0, PH_ROUTE);
      stamp<kTiming>(P, cx.block, EV_LOADER_ROUTED);
      if (ok && r.ra_on) ra_back(P, r.ra, cx.block, *cx.S.n_active);
      continue;
    }
    // the expert tiles may also use the bottom of the activation buffer once routing is
    // done with the pooled vectors staged there, and so may the unpooler's tiles (its
    // activation is staged at the top); the next layer's QKV tiles may not
    // (set for every tile from the tile's own segment: a block may have no tiles at all in
    // the segments between two that grow the ring)
    r.cap = (uint32_t)P.ring_bytes;
    if (ts.seg == 7 || ts.seg == 8) {
      if (!r.routed && P.ring_ext > 0 && mbar_try_wait(&cx.S.tcbar[TB_ROUTED], 0)) {
        r.routed = true;
        stamp_any(P, EV_LD_RING_GROWN);
      }
      if (r.routed) {
        r.cap += (uint32_t)P.ring_ext;
        // GEMM1's operand-B scales sit right above the extension: free once copied
        if (!r.sfb_free && P.sfb_ext > 0 && mbar_try_wait(&cx.S.tcbar[TB_SFB1], 0)) r.sfb_free = true;
        if (r.sfb_free) r.cap += (uint32_t)P.sfb_ext;
      }
    } else if (ts.seg == 9) {
      r.cap += (uint32_t)P.unpool_ext;
    } else if (ts.seg == 1 && !P.first) {
      // KV tiles: the activation buffer below attention's region is free until o_proj
      // staging (launch 0 stages its prologue input there first)
      r.cap += (uint32_t)P.kv_ext;
    }
    const int g1i = ts.seg == 7 ? (ts.t_u - ts.lo) * ts.steps + ts.t_k0 : 99;
    if (g1i < 16) stamp_any(P, EV_LD_G1_NEXT + g1i);
    uint32_t off;
    if (!ring_place(cx, r, bytes, off)) {
      ok = false;
      break;
    }
    if (g1i < 16) stamp_any(P, EV_LD_G1_PLACED + g1i);
    const uint32_t s = r.issued % kSlots;
    if (st == TS_TILE) r.xmask |= 1u << s;  // weight tiles: released by the tensor-core warp
    else r.xmask &= ~(1u << s);
    cx.S.slot_off[s] = off;
    cx.S.slot_tile[s] = r.issued;
    mbar_expect_tx(&cx.S.full[s], bytes);
    if (st == TS_KV) {
      const int R = dm.kv_rows, halves = dm.hd / 64;
      uint8_t* dst = cx.S.ring + off;
      for (int h = 0; h < halves; ++h) {
        tma_load_3d(dst + h * R * 128, &P.tmap_k, h * 64, kv_row, ts.kv_hk, &cx.S.full[s]);
        tma_load_3d(dst + (halves + h) * R * 128, &P.tmap_v, h * 64, kv_row, ts.kv_hk, &cx.S.full[s]);
      }
    } else {
      bulk_g2s(cx.S.ring + off, src, bytes, &cx.S.full[s], pol);
      // a dense tile goes on to tensor memory through the tensor-core warp
      if (ts.seg != 7 && ts.seg != 8) dq_push(cx, dq, r.issued | ((bytes / 2048u) << 24));
    }
    ++r.issued;
    if (g1i < 16) stamp_any(P, EV_LD_G1_ISSUED + g1i);
    if (r.ra_on) ra_pump(r.ra, bytes);
    if (kTiming) {
      if (ts.seg == 3) {
        if (ts.t_u == ts.lo && ts.t_k0 == 0) stamp<kTiming>(P, cx.block, EV_LD_OP_FIRST);
        if (ts.t_u == ts.lo + 1 && ts.t_k0 == 0) stamp<kTiming>(P, cx.block, EV_LD_OP_U1);
        if (ts.u >= ts.hi) stamp<kTiming>(P, cx.block, EV_LD_OP_LAST);
      } else if (ts.seg == 7) {
        if (ts.t_u == ts.lo && ts.t_k0 == 0) stamp<kTiming>(P, cx.block, EV_LD_G1_FIRST);
        if (ts.u == ts.hi) g1_last = ts.t_u;
        if (ts.t_u == g1_last && ts.u == ts.hi) stamp<kTiming>(P, cx.block, EV_LD_G1_LAST);
      }
    }
  }
  stamp<kTiming>(P, cx.block, EV_LOADER_END);
  dq_push(cx, dq, kDqEnd);
  if (!ok) {
    // give every copy still in flight a chance to land before the block exits
    cx.deadline = globaltimer() + 20000000ull;
    *cx.S.abort = 1;
    for (uint32_t j = r.tail; j < r.issued; ++j) {
      uint32_t s = j % kSlots, n = 0;
      while (!mbar_try_wait(&cx.S.full[s], (j / kSlots) & 1)) {
        if ((++n & 15) == 0 && globaltimer() > cx.deadline) break;
      }
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------
struct Worker {
  Ctx* cx;
  int cw, lane, g, q;
  uint32_t ti;  // next tile index of the block's sequence
  uint32_t di;  // next dense tile (tensor-memory hand-over) of the block's sequence
  bool ok;
  bool b1;      // this thread issued the copy of GEMM1's operand B
  uint32_t xseq;  // expert tiles of the block before GEMM2's first (weight-scale buffer rotation)
};

__device__ __forceinline__ void cbar() { named_bar(1, kComputeThreads); }

__device__ __forceinline__ uint32_t* phase_counter(const LaunchParams& P, int i) {
  return reinterpret_cast<uint32_t*>(P.x_cur + P.xo.cnt) + i;
}

// The block has stored its share of phase i: the named barrier orders every compute
// thread's stores before one thread's gpu-scope fence, and the counter add after it.
// (Test hook: block 0 never signals the o_proj phase, so its consumers time out.)
__device__ void publish(Worker& w, int i) {
  cbar();
  if (w.cw == 0 && w.lane == 0) {
    const LaunchParams& P = *w.cx->P;
    if ((P.flags & 0x10000u) && i == CNT_OPROJ && blockIdx.x == 0) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(phase_counter(P, i)) : "memory");
  }
}

// Wait until every block has published phase i.  One thread polls the counter with
// acquire loads; the named barrier then orders the other compute threads' loads of
// the phase's output after that observation.  The outputs are read with relaxed
// (L2-coherent) loads and no sentinel checks.  A wait that runs out sets the abort.
__device__ bool await_phase(Worker& w, int i, int phase) {
  Ctx& cx = *w.cx;
  if (w.cw == 0 && w.lane == 0 && !*cx.S.abort) {
    const uint32_t* c = phase_counter(*cx.P, i);
    const uint32_t target = gridDim.x;
    uint32_t n = 0;
    for (;;) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
      if (v >= target) break;
      if ((++n & 15) == 0 && cx.expired(phase)) break;
    }
    const int ev = phase == PH_ATTN_MERGE ? EV_SEEN_MERGE : phase == PH_OPROJ ? EV_SEEN_OPROJ
                 : phase == PH_POOL ? EV_SEEN_POOL : phase == PH_ROUTER ? EV_SEEN_ROUTER
                 : phase == PH_ROUTE ? EV_SEEN_ROUTE : phase == PH_COMBINE ? EV_SEEN_COMBINE
                 : phase == PH_UNPOOL ? EV_SEEN_UNPOOL : EV_SEEN_TAIL;
    stamp_rt(*cx.P, ev);
  }
  cbar();
  if (*cx.S.abort) w.ok = false;
  return w.ok;
}

// B-operand layout of a [16 tokens][K] activation: blocks of 64 columns, each 16
// rows (tokens) of 128 bytes; the 16-byte chunk c of row t sits at slot c ^ (t & 7)
// of its row.  This is the tensor-memory-access 128-byte swizzle of a {64, 16} box,
// and ldmatrix reads any 8x8 matrix (8 tokens, 8 columns) from 8 different bank
// groups.
constexpr uint32_t kActBlockBytes = 2048;  // 16 rows x 64 bf16 columns
__device__ __forceinline__ uint32_t act_chunk(int t, int c) {  // c: 16-byte chunk (8 columns) of row t
  return (uint32_t)(c >> 3) * kActBlockBytes + (uint32_t)t * 128u + ((((uint32_t)c & 7u) ^ ((uint32_t)t & 7u)) << 4);
}
__device__ __forceinline__ uint32_t act_off(int t, int k) { return act_chunk(t, k >> 3); }

// Stage a [16][K] bf16 activation from global memory into the B layout, optionally
// applying RMSNorm with `gain`.  cnt >= 0: wait for every block to publish that
// phase counter first; else, with `poll`, poll each chunk's sentinels; else plain loads.
__device__ bool stage_act(Worker& w, const uint16_t* src, int K, int cnt, bool poll, const uint16_t* gain,
                                       float eps, int phase, int map = -1, uint32_t aoff = 0) {
  Ctx& cx = *w.cx;
  uint8_t* const act = cx.S.act + aoff;  // where the activation goes in the buffer (1 KB aligned)
  const int tid = w.cw * 32 + w.lane;
  const int t = tid >> 4, sub = tid & 15;
  const int nch = K / 8;
  float2 ss2 = make_float2(0.f, 0.f);  // sums of squares of even / odd elements
  bool ok = w.ok;
  // the norm gain does not depend on the producers: fetch the two chunks this thread
  // normalises now
  const bool gain_pre = gain != nullptr && nch <= 2 * kComputeThreads;
  uint4 gpre[2];
  if (gain_pre) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (tid + j * kComputeThreads < nch) gpre[j] = ld_nc_v4_early(reinterpret_cast<const uint4*>(gain) + tid + j * kComputeThreads);
  }
  if (map >= 0 && cx.P->act_tma && cnt >= 0 && !poll) {
    // tensor copies of the whole [16][K] activation in the act layout: one thread
    // issues them once every block has published the phase and every compute warp is
    // done with the buffer (its generic accesses ordered before the copies' writes)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    await_phase(w, cnt, phase);
    ok = w.ok;
    const bool issuer = tid == 0 && ok;
    if (issuer) {
      asm volatile("fence.proxy.async.global;" ::: "memory");  // the producers' stores, acquired above
      const int nblk = K / 64, nb = cx.P->act_box[map];
      mbar_expect_tx(cx.S.stage_bar, (uint32_t)K * 32u);
      for (int z = 0; z < nblk; z += nb)
        tma_load_3d(act + (size_t)z * kActBlockBytes, &cx.P->tmap_act[map], 0, 0, z, cx.S.stage_bar);
    }
    const uint32_t par = cx.stage_n & 1u;
    ++cx.stage_n;
    if (ok) ok = wait_bar(cx, cx.S.stage_bar, par, phase);
    if (issuer && !ok) {
      // the block gives up (another block failed): the copies read valid memory and
      // land within microseconds, but must land before this block may exit
      for (uint32_t n = 0; n < (1u << 24) && !mbar_try_wait(cx.S.stage_bar, par); ++n) {
      }
    }
    if (ok && gain != nullptr) {
      // the row's sum of squares in the order of the load path below (bitwise the same)
#pragma unroll 4
      for (int c = sub; c < nch; c += 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(act + act_off(t, c * 8));
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 x2 = make_float2(__uint_as_float(wd[i] << 16), __uint_as_float(wd[i] & 0xFFFF0000u));
          ss2 = __ffma2_rn(x2, x2, ss2);
        }
      }
    }
  } else {
  // every compute warp is done with the act buffer (and, with a counter, the producers are done)
  if (cnt >= 0) await_phase(w, cnt, phase);
  else cbar();
  ok = w.ok;
  // loads are issued in batches of 16 before any is inspected, so their latencies overlap
  constexpr int kB = 16;
  for (int c0 = sub; c0 < nch && ok; c0 += 16 * kB) {
    uint4 v[kB];
    const uint4* base = reinterpret_cast<const uint4*>(src + (size_t)t * K + c0 * 8);  // chunk j at base + 16 j
    uint32_t pending = 0;
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (c0 + 16 * j < nch) pending |= 1u << j;
    if (poll) {
      ok = poll_batch<kB>(cx, base, 16, v, pending, [](const uint4& x) { return bf16x8_ready(x); }, phase);
    } else if (cnt >= 0) {
#pragma unroll
      for (int j = 0; j < kB; ++j)
        if ((pending >> j) & 1u) v[j] = ld_relaxed_v4(base + 16 * j);
    } else {
#pragma unroll
      for (int j = 0; j < kB; ++j)
        if ((pending >> j) & 1u) v[j] = base[16 * j];
    }
    if (!ok) break;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int c = c0 + 16 * j;
      if (c >= nch) continue;
      const uint32_t wd[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x2 = make_float2(__uint_as_float(wd[i] << 16), __uint_as_float(wd[i] & 0xFFFF0000u));
        ss2 = __ffma2_rn(x2, x2, ss2);
      }
      *reinterpret_cast<uint4*>(act + act_off(t, c * 8)) = v[j];
    }
  }
  }
  if (gain != nullptr && phase == PH_POOL) stamp_rt(*cx.P, EV_POOL_STAGED);
  ok = __all_sync(0xffffffffu, ok);
  if (gain != nullptr) {
    // 1 / rms of each row: the row's 16 threads reduce their partial sums of squares,
    // one of them leaves the factor in the (then unused) scan scratch
    float ss = ss2.x + ss2.y;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    float* inv_s = cx.S.red;
    if (sub == 0) inv_s[t] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps)));
    cbar();
    if (phase == PH_POOL) stamp_rt(*cx.P, EV_POOL_GAIN);
    if (ok) {
      // thread tid owns chunk columns tid, tid + 256, ...: one gain chunk, then the 16
      // rows, four at a time (all loads before any store).  A compact loop: this code
      // runs once per phase, cold in the instruction cache.
#pragma unroll 1
      for (int j = 0, c = tid; c < nch; ++j, c += kComputeThreads) {
        const uint4 gv = (gain_pre && j < 2) ? (j == 0 ? gpre[0] : gpre[1])
                                             : __ldg(reinterpret_cast<const uint4*>(gain + c * 8));
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        float2 g2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) g2[i] = make_float2(__uint_as_float(gw[i] << 16), __uint_as_float(gw[i] & 0xFFFF0000u));
#pragma unroll 1
        for (int r0 = 0; r0 < 16; r0 += 4) {
          uint4 v[4];
          uint32_t off[4];
          float iv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            off[q] = act_off(r0 + q, c * 8);
            v[q] = *reinterpret_cast<const uint4*>(act + off[q]);
            iv[q] = inv_s[r0 + q];
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t wd[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
            const float2 inv2 = make_float2(iv[q], iv[q]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              // (x * inv) * g per element in fp32, two elements per instruction; the
              // result stays in shared memory, so no sentinel mapping is needed
              const float2 xs = __fmul2_rn(make_float2(__uint_as_float(wd[i] << 16), __uint_as_float(wd[i] & 0xFFFF0000u)), inv2);
              const float2 y = __fmul2_rn(xs, g2[i]);
              const __nv_bfloat162 h = __floats2bfloat162_rn(y.x, y.y);
              wd[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(act + off[q]) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          }
        }
      }
    }
  }
  if (gain != nullptr && phase == PH_POOL) stamp_rt(*cx.P, EV_POOL_NORMED);
  w.ok = ok;
  cbar();
  // all compute warps must agree (a failure anywhere aborts the block)
  if (*cx.S.abort) w.ok = false;
  return w.ok;
}

__device__ __forceinline__ uint32_t lane_mat_off(int lane) {
  return (uint32_t)(lane >> 3) * 128u + (uint32_t)(lane & 7) * 16u;
}

struct QkvDst {
  uint16_t* q;         // [16][hq*hd]
  bool q_relaxed;
  uint16_t* kc;        // caches of the layer whose rows are written
  uint16_t* vc;
  uint16_t* tkv;       // optional sentinel copy [2][hkv][16][hd]
};

__device__ __forceinline__ void qkv_epilogue(const LaunchParams& P, const Smem& S, const QkvDst& dst, int u, int p,
                                             int t, float vlo, float vhi) {
  const Dims& dm = P.dm;
  const int D = dm.hd, upd = D / 16;
  const int nQ = dm.hq * upd, nK = dm.hkv * upd;
  if (u < nQ + nK) {
    // rows p and p+8 of the unit are dims (j*8+p) and (j*8+p + D/2) of one head
    const bool isq = u < nQ;
    const int hu = isq ? u : u - nQ, h = hu / upd, j = hu % upd;
    const int dim = j * 8 + p;
    const float* cs = P.rope + ((size_t)S.depth[t] * (D / 2) + dim) * 2;
    const float c = cs[0], s = cs[1];
    const uint16_t xr = bf16_bits_rn(vlo * c - vhi * s), yr = bf16_bits_rn(vhi * c + vlo * s);
    if (isq) {
      uint16_t* q = dst.q + (size_t)t * dm.hq * D + (size_t)h * D + dim;
      if (dst.q_relaxed) { st_relaxed_u16(q, xr); st_relaxed_u16(q + D / 2, yr); }
      else { q[0] = xr; q[D / 2] = yr; }
    } else {
      uint16_t* k = dst.kc + ((size_t)h * dm.max_ctx + *S.pos0 + t) * D + dim;
      k[0] = xr;
      k[D / 2] = yr;
      if (dst.tkv) {
        uint16_t* tp = dst.tkv + ((size_t)h * 16 + t) * D + dim;
        st_relaxed_u16(tp, xr);
        st_relaxed_u16(tp + D / 2, yr);
      }
    }
  } else {
    const int hu = u - nQ - nK, h = hu / upd, j = hu % upd;
    const uint16_t a = bf16_bits_rn(vlo), b = bf16_bits_rn(vhi);
    uint16_t* v = dst.vc + ((size_t)h * dm.max_ctx + *S.pos0 + t) * D + j * 16 + p;
    v[0] = a;
    v[8] = b;
    if (dst.tkv) {
      uint16_t* tp = dst.tkv + (((size_t)dm.hkv + h) * 16 + t) * D + j * 16 + p;
      st_relaxed_u16(tp, a);
      st_relaxed_u16(tp + 8, b);
    }
  }
}

// what a dense phase does with its outputs (one copy of the phase loop serves all)
enum EpiKind {
  EPI_QKV = 0, EPI_OPROJ = 1, EPI_POOL = 2, EPI_ROUTER = 3, EPI_UNPOOL = 4, EPI_LMHEAD = 5,
  EPI_SWIGLU = 6,   // dense FFN: z = bf16(silu(gate) * up) from a unit's paired rows
  EPI_PARTIAL = 7   // fp32 partial sums of a K half (the other half adds them)
};
struct EpiArgs {
  int kind;
  QkvDst dq;               // EPI_QKV
  const uint16_t* res;     // residual input (EPI_OPROJ: h, EPI_UNPOOL: h1)
  uint16_t* out;           // bf16 output (h1, u, z, h2)
  uint16_t* out2;          // optional second copy of h2 (next launch / caller)
  float* out32;            // fp32 output (router logits, LM-head logits, EPI_PARTIAL's sums)
  const float* part;       // EPI_UNPOOL: optional fp32 partial sums added before rounding
};

// epilogue of output rows u*16 + p and u*16 + p + 8 for token t (values lo, hi)
// (res2: the residual pair of rows p, p+8 when has_res, else read here)
__device__ void dense_epi(const LaunchParams& P, const Smem& S, const EpiArgs& ea, int u, int p, int t,
                                       float lo, float hi, bool has_res = false, uint32_t res2 = 0) {
  const Dims& dm = P.dm;
  switch (ea.kind) {
    case EPI_QKV:
      qkv_epilogue(P, S, ea.dq, u, p, t, lo, hi);
      break;
    case EPI_OPROJ:
    case EPI_UNPOOL: {
      const float v2[2] = {lo, hi};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int n = u * 16 + p + hf * 8;
        const float o = bf16_to_f32(bf16_bits_rn(ea.part ? v2[hf] + ea.part[(size_t)t * dm.d + n] : v2[hf]));
        const uint16_t r = has_res ? (uint16_t)(hf ? res2 >> 16 : res2 & 0xFFFFu)
                           : ea.kind == EPI_OPROJ ? ea.res[(size_t)t * dm.d + n]
                                                  : ld_relaxed_u16(ea.res + (size_t)t * dm.d + n);
        const uint16_t v = bf16_bits_rn(bf16_to_f32(r) + o);
        st_relaxed_u16(ea.out + (size_t)t * dm.d + n, v);
        if (ea.out2) ea.out2[(size_t)t * dm.d + n] = v;
      }
      break;
    }
    case EPI_SWIGLU: {
      // rows p / p+8 of unit u are gate and up row 8u + p; z is kept as its two K halves,
      // [2][16][f/2], so each half stages like a [16][f/2] activation
      const int n = u * 8 + p, fh = dm.f >> 1, hf = n >= fh ? 1 : 0;
      const float zv = lo / (1.0f + expf(-lo)) * hi;
      st_relaxed_u16(ea.out + ((size_t)hf * 16 + t) * fh + (n - hf * fh), bf16_bits_rn(zv));
      break;
    }
    case EPI_PARTIAL:
      // read back by this same thread in the second half's epilogue (same units, group, lane)
      ea.out32[(size_t)t * dm.d + u * 16 + p] = lo;
      ea.out32[(size_t)t * dm.d + u * 16 + p + 8] = hi;
      break;
    case EPI_POOL:
      st_relaxed_u16(ea.out + (size_t)t * dm.p + u * 16 + p, bf16_bits_rn(lo));
      st_relaxed_u16(ea.out + (size_t)t * dm.p + u * 16 + p + 8, bf16_bits_rn(hi));
      break;
    case EPI_ROUTER: {
      const int n = u * 16 + p;
      st_relaxed_u32(ea.out32 + (size_t)t * dm.e + n, __float_as_uint(f32_canon(lo + P.b_router[n])));
      st_relaxed_u32(ea.out32 + (size_t)t * dm.e + n + 8, __float_as_uint(f32_canon(hi + P.b_router[n + 8])));
      break;
    }
    default:  // EPI_LMHEAD
      ea.out32[(size_t)t * dm.vocab + u * 16 + p] = lo;
      ea.out32[(size_t)t * dm.vocab + u * 16 + p + 8] = hi;
      break;
  }
}

// Dense phase: out[16 tokens][N] = act[16][K] . W[N][K]^T over this block's
// 16-row units.  The two warp groups take alternate units (unit lo + i by group i & 1),
// so one group's cross-warp sum and epilogue overlap the other group's MMAs on the
// next unit.  The weight tiles come from tensor memory, where the tensor-core warp
// copies each one as it lands (so the ring's space goes back to the loader at once and
// the block holds up to 8 tiles beyond it): warp wi of the group reads its lane quadrant
// of the tile's slot, the A fragments of k-steps wi, wi + 4, ... (tcgen05.ld), and runs
// their MMAs against the staged activation; each unit ends with the sum of the group's
// four partials in fixed warp order (the result does not depend on the grid size or the
// group) and an epilogue over (row pair, token): dense_epi(unit, p, t, row p value,
// row p+8 value), run by the group's 128 threads.
__device__ void dense_phase(Worker& w, const int K, const int N, const int rot, const EpiArgs& ea,
                                         int trace, uint32_t aoff = 0) {
  Ctx& cx = *w.cx;
  const int G = gridDim.x;
  int lo, hi;
  unit_range(N / 16, rot_block(cx.block, rot, G), G, lo, hi);
  const int steps = K / 16;
  const int ktiles = (steps + kDenseTileSteps - 1) / kDenseTileSteps;
  // The compute warps form two groups of four; group g takes the units lo + g, lo + g + 2,
  // ... and warp wi of the group k-steps 16 wi .. 16 wi + 15 of each of their tiles (a
  // tile held by all eight warps at once would be released only after one warp's whole
  // dependent MMA chain).  k-step & 3 is the loop index & 3.
  const int group = w.cw >> 2, wi = w.cw & 3;
  // lane l addresses row l & 7 of matrix m = l >> 3 (tokens 8 (m >> 1) .., columns
  // 8 (m & 1) .. of the k-step); k-step ks sits at 16-column position ks & 3 (= wi for
  // this warp's k-steps) of 64-column block ks >> 2
  uint32_t act_lane;
  {
    const int m = w.lane >> 3, t = (m >> 1) * 8 + (w.lane & 7);
    act_lane = smem_u32(cx.S.act + aoff) + act_chunk(t, wi * 2 + (m & 1));
  }
  // this warp's lane quadrant of the dense slots
  const uint32_t tq = *cx.S.tmem_base + ((uint32_t)(wi * 32) << 16);
  float* red = cx.S.dred;  // [8 warps][16 rows][16 tokens]
  const int tig = wi * 32 + w.lane;  // thread in group
  // the residual inputs of the o_proj / unpooler epilogues do not depend on this phase:
  // read them for the group's first units now, while the tiles stream in
  constexpr int kPreUnits = 2;
  uint32_t pre[kPreUnits];
  const bool pre_res = ea.kind == EPI_OPROJ || ea.kind == EPI_UNPOOL;
  if (pre_res) {
    const int d = cx.P->dm.d, p = tig >> 4, tok = tig & 15;
#pragma unroll
    for (int i = 0; i < kPreUnits; ++i) {
      pre[i] = 0u;
      const int u = lo + group + 2 * i;
      if (u < hi) {
        const uint16_t* r = ea.res + (size_t)tok * d + u * 16 + p;
        const uint32_t a = ea.kind == EPI_OPROJ ? r[0] : ld_relaxed_u16(r);
        const uint32_t b = ea.kind == EPI_OPROJ ? r[8] : ld_relaxed_u16(r + 8);
        pre[i] = a | (b << 16);
      }
    }
  }
  for (int u = lo + group; u < hi; u += 2) {
    const int loc = u - lo;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // odd k-steps
    // the loader streams the units in pairs, their tiles alternating
    const bool paired = (loc | 1) < hi - lo;
    const uint32_t d0 = w.di + (uint32_t)((loc >> 1) * 2 * ktiles + (paired ? (loc & 1) : 0));
    for (int kt = 0; kt < ktiles; ++kt) {
      const uint32_t dd = d0 + (uint32_t)(paired ? 2 * kt : kt);
      const uint32_t j = dd % kDenseTmemSlots;
      if (w.ok) w.ok = wait_bar(cx, &cx.S.tcbar[TB_TFULL + j], (dd / kDenseTmemSlots) & 1, 50);
      if (trace >= 0 && loc < 2 && tig == 0 && (kt == 0 || kt + 1 == ktiles)) stamp_any(*cx.P, trace + loc * 4 + (kt == 0 ? 0 : 1));
      if (w.ok) {
        tc_fence_after();
        const int k0 = kt * kDenseTileSteps;
        const int nc = min(kDenseTileSteps, steps - k0) >> 2;  // k-steps of this warp in the tile
        const uint32_t bb = act_lane + (uint32_t)(k0 >> 2) * kActBlockBytes;
        // two halves of 8 k-steps: the slot goes back once both are in registers
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[32];
          if (h == 0 || nc > 8) {
            tmem_ld32(tq + j * kDenseTmemCols + 32 * h, a);
            tmem_ld_wait();
          }
          if (h == (nc > 8 ? 1 : 0)) {  // the tile's last tensor-memory read by this warp
            tc_fence_before();
            __syncwarp();
            if (w.lane == 0) mbar_arrive(&cx.S.tcbar[TB_TFREE + j], 1);
          }
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const int c = h * 8 + c8;
            if (c >= nc) break;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(bb + (uint32_t)c * kActBlockBytes, b0, b1, b2, b3);
            float(&cc)[2][4] = (c8 & 1) ? acc2 : acc;
            mma_bf16(cc[0], a[4 * c8], a[4 * c8 + 1], a[4 * c8 + 2], a[4 * c8 + 3], b0, b1);
            mma_bf16(cc[1], a[4 * c8], a[4 * c8 + 1], a[4 * c8 + 2], a[4 * c8 + 3], b2, b3);
          }
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] += acc2[nt][i];
    // partials -> shared memory: rows g / g+8, tokens nt*8 + 2q (+1)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = w.g + ((i >> 1) << 3), tok = nt * 8 + 2 * w.q + (i & 1);
        red[(w.cw * 16 + row) * 16 + tok] = acc[nt][i];
      }
    if (trace >= 0 && loc < 2 && tig == 0) stamp_any(*cx.P, trace + loc * 4 + 2);
    named_bar(2 + group, 128);
    if (w.ok) {
      const int p = tig >> 4, tok = tig & 15;
      float vlo = 0.f, vhi = 0.f;
#pragma unroll
      for (int ww = 4 * group; ww < 4 * group + 4; ++ww) {
        vlo += red[(ww * 16 + p) * 16 + tok];
        vhi += red[(ww * 16 + p + 8) * 16 + tok];
      }
      uint32_t r2 = 0u;
#pragma unroll
      for (int i = 0; i < kPreUnits; ++i)
        if (loc == group + 2 * i) r2 = pre[i];
      dense_epi(*cx.P, cx.S, ea, u, p, tok, vlo, vhi, pre_res && loc < group + 2 * kPreUnits, r2);
    }
    named_bar(2 + group, 128);  // the group's partial sums may be overwritten
    if (trace >= 0 && loc < 2 && tig == 0) stamp_any(*cx.P, trace + loc * 4 + 3);
    if (*cx.S.abort) w.ok = false;
  }
  // both groups' epilogues are stored before the phase is published
  cbar();
  w.ti += (uint32_t)((hi - lo) * ktiles);
  w.di += (uint32_t)((hi - lo) * ktiles);
}

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
// physical byte offset of (row, d) inside a tile loaded with the 128-byte swizzle
// (two 64-column halves of `rows` rows each)
__device__ __forceinline__ uint32_t swz(int row, int d, int rows) {
  return (uint32_t)(d >> 6) * rows * 128u + (uint32_t)row * 128u + ((((d & 63) >> 3) ^ (row & 7)) << 4);
}

template <int D>
struct AttnState {
  float m[2], l[2];
  float o[D / 8][4];
};

// process 16 keys [kb, kb+16) of a K/V tile for head fragments qa
template <int D, class Vis>
__device__ __forceinline__ void attn_keys16(AttnState<D>& st, const uint32_t (&qa)[D / 16][4],
                                            uint32_t kbase, uint32_t vbase, int rows, int kb, int lane,
                                            float scale_log2, Vis vis) {
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
  }
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int key = kb + nt * 8 + r8;
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      const int d0 = (ks + (mi >> 1)) * 16 + (mi & 1) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + swz(key, d0, rows), b0, b1, b2, b3);
      mma_bf16(s[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_bf16(s[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
    }
  }
  const int g = lane >> 2, q = lane & 3;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = g + ((i >> 1) << 3);     // token
      const int key = kb + nt * 8 + 2 * q + (i & 1);
      float v = vis(row, key) ? s[nt][i] * scale_log2 : -INFINITY;
      s[nt][i] = v;
      mx[i >> 1] = fmaxf(mx[i >> 1], v);
    }
  }
  float alpha[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    const float mnew = fmaxf(st.m[r], mx[r]);
    const float muse = (mnew == -INFINITY) ? 0.f : mnew;
    alpha[r] = exp2f(st.m[r] - muse);
    st.m[r] = mnew;
    mx[r] = muse;
  }
  float rs[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float p = exp2f(s[nt][i] - mx[i >> 1]);
      s[nt][i] = p;
      rs[i >> 1] += p;
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) st.l[r] = st.l[r] * alpha[r] + rs[r];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    st.o[n][0] *= alpha[0];
    st.o[n][1] *= alpha[0];
    st.o[n][2] *= alpha[1];
    st.o[n][3] *= alpha[1];
  }
  // P as two bf16 terms, P = hi + lo (about 16 significant bits): with P in one bf16
  // term the attention output carried ~2e-3 relative error, which its own bf16 rounding
  // then spread to most elements, and through h1 and the pooled vector to the router
  // logits (a few 1e-3, above the top-8 margin of the inputs)
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = s[i >> 1][(i & 1) * 2], b = s[i >> 1][(i & 1) * 2 + 1];
    ph[i] = pack_bf16x2(a, b);
    pl[i] = pack_bf16x2(a - bf16_to_f32((uint16_t)(ph[i] & 0xFFFFu)), b - bf16_to_f32((uint16_t)(ph[i] >> 16)));
  }
#pragma unroll
  for (int n = 0; n < D / 8; n += 2) {
    const int key = kb + (mi & 1) * 8 + r8;
    const int d0 = (n + (mi >> 1)) * 8;
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vbase + swz(key, d0, rows), b0, b1, b2, b3);
    mma_bf16(st.o[n], ph[0], ph[1], ph[2], ph[3], b0, b1);
    mma_bf16(st.o[n + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
    mma_bf16(st.o[n], pl[0], pl[1], pl[2], pl[3], b0, b1);
    mma_bf16(st.o[n + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
  }
}

// NKEYS keys (a multiple of 16, from key kb of a tile of `rows` rows) in one online-softmax
// update: the whole-tile form the draft model's attention uses (one query head per KV
// head, so the block's warps split the tiles of that head among themselves)
template <int D, int NKEYS, class Vis>
__device__ __forceinline__ void attn_keys_n(AttnState<D>& st, const uint32_t (&qa)[D / 16][4],
                                            uint32_t kbase, uint32_t vbase, int rows, int kb, int lane,
                                            float scale_log2, Vis vis) {
  constexpr int NT = NKEYS / 8;
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
  }
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int ks = 0; ks < D / 16; ks += 2) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int key = kb + nt * 8 + r8;
      const int d0 = (ks + (mi >> 1)) * 16 + (mi & 1) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + swz(key, d0, rows), b0, b1, b2, b3);
      mma_bf16(s[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_bf16(s[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
    }
  }
  const int g = lane >> 2, q = lane & 3;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = g + ((i >> 1) << 3);     // token
      const int key = kb + nt * 8 + 2 * q + (i & 1);
      float v = vis(row, key) ? s[nt][i] * scale_log2 : -INFINITY;
      s[nt][i] = v;
      mx[i >> 1] = fmaxf(mx[i >> 1], v);
    }
  }
  float alpha[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    const float mnew = fmaxf(st.m[r], mx[r]);
    const float muse = (mnew == -INFINITY) ? 0.f : mnew;
    alpha[r] = exp2f(st.m[r] - muse);
    st.m[r] = mnew;
    mx[r] = muse;
  }
  float rs[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float p = exp2f(s[nt][i] - mx[i >> 1]);
      s[nt][i] = p;
      rs[i >> 1] += p;
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) st.l[r] = st.l[r] * alpha[r] + rs[r];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    st.o[n][0] *= alpha[0];
    st.o[n][1] *= alpha[0];
    st.o[n][2] *= alpha[1];
    st.o[n][3] *= alpha[1];
  }
  // P as two bf16 terms (as in attn_keys16); k-step kk of P.V covers keys 16 kk ..
  // 16 kk + 15, the score columns of nt = 2 kk and 2 kk + 1
#pragma unroll
  for (int kk = 0; kk < NKEYS / 16; ++kk) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = s[2 * kk + (i >> 1)][(i & 1) * 2], b = s[2 * kk + (i >> 1)][(i & 1) * 2 + 1];
      ph[i] = pack_bf16x2(a, b);
      pl[i] = pack_bf16x2(a - bf16_to_f32((uint16_t)(ph[i] & 0xFFFFu)), b - bf16_to_f32((uint16_t)(ph[i] >> 16)));
    }
#pragma unroll
    for (int n = 0; n < D / 8; n += 2) {
      const int key = kb + kk * 16 + (mi & 1) * 8 + r8;
      const int d0 = (n + (mi >> 1)) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vbase + swz(key, d0, rows), b0, b1, b2, b3);
      mma_bf16(st.o[n], ph[0], ph[1], ph[2], ph[3], b0, b1);
      mma_bf16(st.o[n + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
      mma_bf16(st.o[n], pl[0], pl[1], pl[2], pl[3], b0, b1);
      mma_bf16(st.o[n + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
  }
}

// kTiles: the WPH warps of a head take alternate KV tiles, all rows of each in one update
// (the draft model); else each takes its NK keys of every tile (the target model)
template <int D, bool kTiles>
__device__ void attention_phase(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int G = gridDim.x;
  const AttnUnit au = attn_unit(P, cx.pos0, rot_block(cx.block, P.phase_rot * 2, G), P.is_global);
  if (!au.valid) return;
  const int group = dm.group, R = dm.attn_rows, NK = dm.attn_nk, WPH = dm.attn_wph;
  const int KR = dm.kv_rows, nsub = KR / R;  // rows of a ring tile, attention tiles in it
  // act buffer regions at its top: Q fragments source, tree K/V, merge scratch (the KV
  // tiles may use the buffer below them)
  uint8_t* qsm = cx.S.act + P.attn_act_off;
  uint8_t* tk = qsm + group * (D / 16) * kKStepBytes;
  uint8_t* tv = tk + 16 * D * 2;
  float* scratch = reinterpret_cast<float*>(tv + 16 * D * 2);
  const int tid = w.cw * 32 + w.lane;
  // stage Q of this kv head's query heads (A operand layout)
  {
    const uint16_t* qsrc = P.first ? reinterpret_cast<const uint16_t*>(P.x_cur + P.xo.q0) : P.in_q;
    const int nch = T * group * D / 8;
    constexpr int kB = 4;
    for (int c0 = tid; c0 < nch && w.ok; c0 += kComputeThreads * kB) {
      uint4 v[kB];
      const uint16_t* src[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const int c = c0 + i * kComputeThreads;
        if (c >= nch) continue;
        const int t = c / (group * D / 8), rem = c % (group * D / 8), j = rem / (D / 8), d = (rem % (D / 8)) * 8;
        src[i] = qsrc + (size_t)t * dm.hq * D + (size_t)(au.hk * group + j) * D + d;
        v[i] = P.first ? ld_relaxed_v4(src[i]) : *reinterpret_cast<const uint4*>(src[i]);
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const int c = c0 + i * kComputeThreads;
        if (c >= nch || !w.ok) continue;
        if (P.first && !bf16x8_ready(v[i])) w.ok = poll_bf16x8(cx, src[i], v[i], PH_ATTN);
        const int t = c / (group * D / 8), rem = c % (group * D / 8), j = rem / (D / 8), d = (rem % (D / 8)) * 8;
        const int m = ((d >> 3) & 1) * 2 + (t >> 3);
        *reinterpret_cast<uint4*>(qsm + j * (D / 16) * kKStepBytes + (d >> 4) * kKStepBytes + m * 128 + (t & 7) * 16) = v[i];
      }
    }
    if (au.tree) {
      for (int c = tid; c < 2 * 16 * D / 8 && w.ok; c += kComputeThreads) {
        const int kv = c / (16 * D / 8), rem = c % (16 * D / 8), row = rem / (D / 8), d = (rem % (D / 8)) * 8;
        uint4 v;
        if (P.first) {
          const uint16_t* p = reinterpret_cast<const uint16_t*>(P.x_cur + P.xo.tkv0) +
                              (((size_t)kv * dm.hkv + au.hk) * 16 + row) * D + d;
          w.ok = poll_bf16x8(cx, p, v, PH_ATTN);
        } else {
          const uint16_t* cache = kv ? P.vc : P.kc;
          v = *reinterpret_cast<const uint4*>(cache + ((size_t)au.hk * dm.max_ctx + cx.pos0 + row) * D + d);
        }
        *reinterpret_cast<uint4*>((kv ? tv : tk) + swz(row, d, 16)) = v;
      }
    }
  }
  w.ok = __all_sync(0xffffffffu, w.ok);
  cbar();
  stamp_rt(P, EV_ATTN_IN);
  if (*cx.S.abort) w.ok = false;
  const int j = w.cw / WPH, part = w.cw % WPH;
  const bool active = j < group;
  uint32_t qa[D / 16][4];
  AttnState<D> st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
  if (active) {
    const uint32_t qb = smem_u32(qsm) + j * (D / 16) * kKStepBytes + lane_mat_off(w.lane);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(qb + ks * kKStepBytes, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
  }
  const float scale_log2 = 1.4426950408889634f * rsqrtf((float)D);
  const int pos0 = cx.pos0, window = dm.window, glob = P.is_global;
  const int32_t* tpos = cx.S.tpos;
  for (int i = 0; i < au.n_sub; ++i) {
    const uint32_t t = w.ti + (uint32_t)i;
    const uint32_t s = t % kSlots;
    if (w.ok) w.ok = wait_tile(cx, t, PH_ATTN);
    if (!w.ok) break;
    if (active) {
      const uint32_t kb_ = smem_u32(cx.S.ring + cx.S.slot_off[s]);
      const uint32_t vb_ = kb_ + (uint32_t)KR * D * 2;
      const int row0 = au.r0 + i * KR, r1 = au.r1;
      auto vis = [&](int tok, int key) {
        const int r = row0 + key;
        return r < r1 && (glob || tpos[tok] - r < window);
      };
      if constexpr (kTiles) {
        // attention tile i nsub + sb (keys sb R .. of the ring tile), while it holds rows
        for (int sb = 0; sb < nsub && row0 + sb * R < r1; ++sb) {
          if ((i * nsub + sb) % WPH != part) continue;
          if (R == 32) attn_keys_n<D, 32>(st, qa, kb_, vb_, KR, sb * R, w.lane, scale_log2, vis);
          else attn_keys_n<D, 64>(st, qa, kb_, vb_, KR, sb * R, w.lane, scale_log2, vis);
        }
      } else {
        for (int sb = 0; sb < nsub && row0 + sb * R < r1; ++sb)
          for (int kb = part * NK; kb < (part + 1) * NK; kb += 16)
            attn_keys16<D>(st, qa, kb_, vb_, KR, sb * R + kb, w.lane, scale_log2, vis);
      }
    }
    __syncwarp();
    if (w.lane == 0) mbar_arrive(&cx.S.empty[s], 1);
  }
  w.ti += (uint32_t)au.n_sub;
  // the tree rows: part 0, or with whole tiles the part after the last history tile's
  const int tree_part = kTiles ? ((au.r1 - au.r0 + R - 1) / R) % WPH : 0;
  if (w.ok && active && au.tree && part == tree_part) {
    const uint32_t* anc = cx.S.anc;
    auto vis = [&](int tok, int key) { return ((anc[tok] >> key) & 1u) != 0u; };
    attn_keys16<D>(st, qa, smem_u32(tk), smem_u32(tv), 16, 0, w.lane, scale_log2, vis);
  }
  (void)pos0;
  // finish the row sums across the quad
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
  }
  // merge the WPH warps of each head through shared memory
  const int g = w.g, q = w.q;
  const int per_warp = 2 + 2 + D / 8 * 4;  // m[2], l[2], o
  if (WPH > 1) {
    if (active && part > 0) {
      float* sc = scratch + ((size_t)(j * WPH + part) * 32 + w.lane) * per_warp;
      sc[0] = st.m[0]; sc[1] = st.m[1]; sc[2] = st.l[0]; sc[3] = st.l[1];
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        for (int i = 0; i < 4; ++i) sc[4 + n * 4 + i] = st.o[n][i];
    }
    cbar();
    if (active && part == 0) {
      for (int pp = 1; pp < WPH; ++pp) {
        const float* sc = scratch + ((size_t)(j * WPH + pp) * 32 + w.lane) * per_warp;
        float al[2], be[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float mn = fmaxf(st.m[r], sc[r]);
          const float mu = (mn == -INFINITY) ? 0.f : mn;
          al[r] = exp2f(st.m[r] - mu);
          be[r] = exp2f(sc[r] - mu);
          st.m[r] = mn;
          st.l[r] = st.l[r] * al[r] + sc[2 + r] * be[r];
        }
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          st.o[n][0] = st.o[n][0] * al[0] + sc[4 + n * 4 + 0] * be[0];
          st.o[n][1] = st.o[n][1] * al[0] + sc[4 + n * 4 + 1] * be[0];
          st.o[n][2] = st.o[n][2] * al[1] + sc[4 + n * 4 + 2] * be[1];
          st.o[n][3] = st.o[n][3] * al[1] + sc[4 + n * 4 + 3] * be[1];
        }
      }
    }
  }
  if (w.ok && active && part == 0) {
    // partial of (kv head, split): acc [16][group][D], (m, l) [16][group] in log2 units
    float* part_acc = reinterpret_cast<float*>(P.s_buf + P.so.part) +
                      ((size_t)(au.hk * dm.splits + au.s) * T) * group * D;
    float* part_ml = reinterpret_cast<float*>(P.s_buf + P.so.ml) + ((size_t)(au.hk * dm.splits + au.s) * T) * group * 2;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int tok = g + r * 8;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        float* dst = part_acc + ((size_t)tok * group + j) * D + n * 8 + 2 * q;
        uint2 v = make_uint2(__float_as_uint(f32_canon(st.o[n][2 * r])), __float_as_uint(f32_canon(st.o[n][2 * r + 1])));
        asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%2};" ::"l"(dst), "r"(v.x), "r"(v.y) : "memory");
      }
      if (q == 0) {
        float* dst = part_ml + ((size_t)tok * group + j) * 2;
        asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%2};" ::"l"(dst), "r"(__float_as_uint(f32_canon(st.m[r]))),
                     "r"(__float_as_uint(f32_canon(st.l[r])))
                     : "memory");
      }
    }
  }
}

// merge the split partials of every (token, q head): O = bf16(sum_s 2^(m_s-M) acc_s / L)
template <int D>
__device__ void attn_merge_phase(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int G = gridDim.x;
  const int group = dm.group, S = dm.splits;
  const int gw = rot_block(cx.block, P.phase_rot * 2, G) * kComputeWarps + w.cw;
  constexpr int PER = D / 32;  // floats per lane
  const float* part_acc = reinterpret_cast<const float*>(P.s_buf + P.so.part);
  const float* part_ml = reinterpret_cast<const float*>(P.s_buf + P.so.ml);
  uint16_t* o_out = reinterpret_cast<uint16_t*>(P.x_cur + P.xo.o);
  // two warps per merged row (warps 2i and 2i + 1 of a block, i = pair): each takes half
  // the splits, all of its loads in flight at once, and the odd warp hands its (M, L,
  // acc) to the even one through the activation buffer (free between the attention and
  // the o_proj staging)
  const int half = w.cw & 1, pair = w.cw >> 1;
  float* xs = reinterpret_cast<float*>(cx.S.act) + pair * 32 * (PER + 2);
  const int s_mid = (S + 1) / 2, s_lo = half ? s_mid : 0, s_hi = half ? S : s_mid;
  if (!await_phase(w, CNT_ATTN, PH_ATTN_MERGE)) return;
  for (int it = gw >> 1; it < T * dm.hq; it += G * kComputeWarps / 2) {
    const int t = it / dm.hq, h = it % dm.hq, hk = h / group, j = h % group;
    auto mlp = [&](int s) { return part_ml + (((size_t)(hk * S + s) * T + t) * group + j) * 2; };
    auto accp = [&](int s) { return part_acc + (((size_t)(hk * S + s) * T + t) * group + j) * D + w.lane * PER; };
    // splits in batches of 10 (one batch for up to 20 splits), every load of a batch in
    // flight together; a batch's partials are rescaled to the running maximum (M, L, acc
    // in log2 units)
    constexpr int kB = 10;
    float M = -INFINITY, L = 0.f, acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int s0 = s_lo; s0 < s_hi; s0 += kB) {
      uint2 mv[kB];
      float av[kB][PER];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (s0 + i >= s_hi) continue;
        mv[i] = ld_relaxed_v2(mlp(s0 + i));
        if constexpr (PER == 4) {
          const uint4 q4 = ld_relaxed_v4(accp(s0 + i));
          av[i][0] = __uint_as_float(q4.x); av[i][1 % PER] = __uint_as_float(q4.y);
          av[i][2 % PER] = __uint_as_float(q4.z); av[i][3 % PER] = __uint_as_float(q4.w);
        } else {
          const uint2 q2 = ld_relaxed_v2(accp(s0 + i));
          av[i][0] = __uint_as_float(q2.x); av[i][1 % PER] = __uint_as_float(q2.y);
        }
      }
      float Mb = M;
#pragma unroll
      for (int i = 0; i < kB; ++i)
        if (s0 + i < s_hi) Mb = fmaxf(Mb, __uint_as_float(mv[i].x));
      const float Mu = (Mb == -INFINITY) ? 0.f : Mb;
      const float al = exp2f(M - Mu);  // 0 while M is still -inf
      L *= al;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] *= al;
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (s0 + i >= s_hi) continue;
        const float ws = exp2f(__uint_as_float(mv[i].x) - Mu);
        L += ws * __uint_as_float(mv[i].y);
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] += ws * av[i][e];
      }
      M = Mb;
    }
    if (half) {
      float* x = xs + w.lane * (PER + 2);
      x[0] = M;
      x[1] = L;
#pragma unroll
      for (int e = 0; e < PER; ++e) x[2 + e] = acc[e];
    }
    named_bar(4 + pair, 64);
    if (!half) {
      // the two halves: the even warp's, then the odd warp's, at their common maximum
      const float* x = xs + w.lane * (PER + 2);
      const float M1 = x[0], L1 = x[1];
      const float Mm = fmaxf(M, M1), Mu = (Mm == -INFINITY) ? 0.f : Mm;
      const float a0 = exp2f(M - Mu), a1 = exp2f(M1 - Mu);
      L = L * a0 + L1 * a1;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = acc[e] * a0 + x[2 + e] * a1;
      const float inv = 1.f / L;
      uint16_t* dst = o_out + (size_t)t * dm.hq * D + (size_t)h * D + w.lane * PER;
      if constexpr (PER == 4) {
        uint2 v = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2 % PER] * inv, acc[3 % PER] * inv));
        asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%2};" ::"l"(dst), "r"(v.x), "r"(v.y) : "memory");
      } else {
        st_relaxed_u32(dst, pack_bf16x2(acc[0] * inv, acc[1 % PER] * inv));
      }
    }
    named_bar(4 + pair, 64);  // the exchange slot may be reused
  }
}

// ---------------------------------------------------------------------------
// routing: top-k per token, expert dispatch, GEMM1 input (orcarouter.ai, § "where
// the kernel boundary sits": top-8 of 256, experts in NVFP4)
// ---------------------------------------------------------------------------
// GEMM1's operand B: each pooled vector u_t as a sum of kSplitTerms NVFP4 terms,
// u_t[k] ~ ts_t sum_j 4^-j S_tj[k / 16] c_tj[k], with ts_t = amax_t / 2688 rounded up to a
// power of two; term j quantises what the terms before it left (block scale S_tj =
// E4M3(bmax / (6 ts_t 4^-j)), E2M1 codes c_tj).  A term leaves at most ~0.18 of its
// block's largest residual, so four leave ~1e-3 of the block's largest magnitude, below
// bf16's own rounding of the larger elements.  With u in this form the GEMM1 products
// run on the block-scaled tensor cores straight from the weights' E2M1 codes in the ring
// (one B row per (term, token)); the 4^-j ts_t factors go in per accumulator column in
// the epilogue.  The blocks without router work split the 16 x p/16 (token, 16-column
// block) pairs among themselves, 16 threads per pair, and store their share (and the
// row scales of the tokens whose first pair they own) in the launch's exchange buffer;
// the router counter publishes it and every block then copies the whole operand in.
__device__ void split_pooled(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const int p = P.dm.p, G = gridDim.x;
  const int tid = w.cw * 32 + w.lane;
  // the router phase's units go one per block (fewer units than blocks): the others split
  const int n_router = P.dm.e / 16, bb = rot_block(cx.block, P.phase_rot * 5, G);
  int rlo, rhi, idx = cx.block, nfree = G;
  unit_range(n_router, bb, G, rlo, rhi);
  if (n_router < G) {
    if (rhi > rlo) return;
    idx = bb - rlo;  // blocks before this one took one unit each
    nfree = G - n_router;
  }
  const int nb = p / 16;
  int lo, hi;
  unit_range(T * nb, idx, nfree, lo, hi);
  if (lo >= hi) return;
  // the row scales of this block's tokens (at most two: a block has fewer than nb pairs;
  // a warp that failed still passes the barriers)
  const int t0 = lo / nb, t1 = (hi - 1) / nb;
  float* red = cx.S.red;
  for (int t = t0; t <= t1 && w.ok; ++t) {
    uint32_t am = 0u;  // |x| of non-negative floats orders like its bits
    for (int c = tid; c < p / 8; c += kComputeThreads) {
      const uint4 v = *reinterpret_cast<const uint4*>(cx.S.act + act_off(t, c * 8));
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) am = max(am, max((wd[j] & 0x7FFFu) << 16, wd[j] & 0x7FFF0000u));
    }
    am = __reduce_max_sync(0xffffffffu, am);
    if (w.lane == 0) reinterpret_cast<uint32_t*>(red)[(t - t0) * kComputeWarps + w.cw] = am;
  }
  cbar();
  if (tid <= t1 - t0 && !*cx.S.abort) {
    uint32_t am = 0u;
    for (int i = 0; i < kComputeWarps; ++i) am = max(am, reinterpret_cast<uint32_t*>(red)[tid * kComputeWarps + i]);
    float ts = __fdiv_rn(__uint_as_float(am), 2688.0f);  // amax / (6 * 448), up to a power of two
    if (ts > 0.f) {
      int ex;
      if (frexpf(ts, &ex) != 0.5f) ts = ldexpf(1.0f, ex);
    }
    cx.S.x_ts[t0 + tid] = ts;
  }
  cbar();
  if (!w.ok || *cx.S.abort) return;
  const int h = tid >> 4, i = tid & 15;
  const uint32_t hmask = 0xFFFFu << (w.lane & 16);  // this half-warp's lanes
  uint8_t* sfimg = P.x_cur + P.xo.b1;
  uint8_t* img = sfimg + b1_code_off(p);
  float* tsimg = reinterpret_cast<float*>(sfimg + b1_ts_off(p));
  for (int pr = lo + h; pr < hi; pr += 16) {
    const int t = pr / nb, c = pr % nb, k = c * 16 + i;
    float x = bf16_to_f32(*reinterpret_cast<const uint16_t*>(cx.S.act + act_off(t, k) + (k & 7) * 2));
    float ts = cx.S.x_ts[t];
    if (c == 0 && i == 0) tsimg[t] = ts;
    // (a compact loop: this code runs once per launch, cold in the instruction cache;
    // the quotients are the kernel's own choice of split, so reciprocals serve)
    float inv6 = ts > 0.f ? __frcp_rn(6.0f * ts) : 0.f;
#pragma unroll 1
    for (int j = 0; j < kSplitTerms; ++j, ts *= 0.25f, inv6 *= 4.0f) {
      float bmax = fabsf(x);
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(hmask, bmax, o));
      const uint32_t sc = ts > 0.f ? f32_to_e4m3(bmax * inv6) : 0u;
      const float den = e4m3_to_f32(sc) * ts;
      const float qx = sc != 0u ? x * __frcp_rn(den) : 0.f;
      const float qn = __shfl_xor_sync(hmask, qx, 1);
      const uint32_t byte = (i & 1) ? f32x2_to_e2m1x2(qn, qx) : f32x2_to_e2m1x2(qx, qn);  // even element low
      const uint32_t h2 = e2m1x2_to_f16x2(byte);
      const float mine = __half2float(__ushort_as_half((unsigned short)((i & 1) ? (h2 >> 16) : (h2 & 0xFFFFu))));
      x -= mine * den;  // the residual for the next term
      const int n = j * T + t;  // operand row
      if (!(i & 1)) {
        const int bi = (k & 255) >> 1;  // byte of the 128-byte row
        img[(k >> 8) * 8192 + n * 128 + (((bi >> 4) ^ (n & 7)) << 4) + (bi & 15)] = (uint8_t)byte;
      }
      if (i == 0) sfimg[(c >> 2) * 512 + (n & 31) * 16 + (n >> 5) * 4 + (c & 3)] = (uint8_t)sc;
    }
    if (t == 0 && (c & 3) == 0) {
      // the scale group's words of rows 64..127 (no such rows): zero
      uint32_t* g = reinterpret_cast<uint32_t*>(sfimg + (c >> 2) * 512);
      g[(2 * i) * 4 + 2] = 0u; g[(2 * i) * 4 + 3] = 0u;
      g[(2 * i + 1) * 4 + 2] = 0u; g[(2 * i + 1) * 4 + 3] = 0u;
    }
  }
}

__device__ void route_phase(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int E = dm.e, K = dm.k;
  const float* logits = reinterpret_cast<const float*>(P.x_cur + P.xo.logits);
  // top-k: warp cw takes tokens 2cw and 2cw+1, both at once (independent chains).
  // Logits become order-preserving unsigned keys (router logits are canonical: never
  // -0.0); each round takes the warp-wide largest key, ties to the lowest expert
  // index, with two warp reductions.  Lane c keeps round c's pick; the softmax of the
  // K picks is then one expf per lane and a fixed-order butterfly sum.
  const int per = (E + 31) / 32;
  if (w.cw == 0 && w.lane == 0 && w.ok) {
    // GEMM1's operand B (every block's share is published with the router counter seen
    // above) -> the top of the activation buffer, whose generic reads every thread
    // fenced before that wait; it lands while routing runs
    asm volatile("fence.proxy.async.global;" ::: "memory");
    const uint32_t bytes = (uint32_t)b1_bytes(dm.p);
    const uint8_t* src = P.x_cur + P.xo.b1;
    mbar_expect_tx(&cx.S.tcbar[TB_B1], bytes);
    for (uint32_t o = 0; o < bytes; o += 16384)
      bulk_g2s_plain(cx.S.act + P.g1_b_off + o, src + o, min(16384u, bytes - o), &cx.S.tcbar[TB_B1]);
    w.b1 = true;
    stamp_rt(P, EV_B1_ISSUED);
  }
  {
    const int t0 = w.cw * 2;
    uint32_t key[2][kMaxExperts / 32];
    // (every block published its router logits before this phase began)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = w.lane + 32 * i;
        key[tt][i] = (i < per && e < E) ? ld_relaxed_u32(logits + (t0 + tt) * E + e) : 0u;
      }
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = w.lane + 32 * i;
        const uint32_t b = key[tt][i];
        key[tt][i] = (i < per && e < E) ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;  // 0: below every key
      }
    uint32_t taken[2] = {0u, 0u};  // bit i: key[tt][i] of this lane already selected
    float my_v[2] = {0.f, 0.f};    // lane c < K: round c's logit
    int my_e[2] = {0, 0};          // and expert
    for (int c = 0; c < K; ++c) {
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        // this lane's best unselected key (lowest i among equal keys)
        uint32_t bk = 0u;
        int bi = 0;
#pragma unroll
        for (int i = kMaxExperts / 32 - 1; i >= 0; --i)
          if (!((taken[tt] >> i) & 1u) && key[tt][i] >= bk && i < per) { bk = key[tt][i]; bi = i; }
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t e_me = (bk == wk) ? (uint32_t)(w.lane + 32 * bi) : 0xFFFFFFFFu;
        uint32_t e = __reduce_min_sync(0xffffffffu, e_me);
        if (e >= (uint32_t)E) e = 0;  // only for NaN logits, which are outside the contract
        if ((int)(e & 31) == w.lane) taken[tt] |= 1u << (e >> 5);
        if (w.lane == c) {
          my_v[tt] = __uint_as_float((wk & 0x80000000u) ? (wk & 0x7FFFFFFFu) : ~wk);
          my_e[tt] = (int)e;
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      const float v0 = __shfl_sync(0xffffffffu, my_v[tt], 0);  // the largest
      const float ex = w.lane < K ? expf(my_v[tt] - v0) : 0.f;
      float sum = ex;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (w.lane < K && w.ok) {
        cx.S.topk_idx[(t0 + tt) * kMaxTopK + w.lane] = my_e[tt];
        cx.S.topk_w[(t0 + tt) * kMaxTopK + w.lane] = ex / sum;
      }
    }
  }
  cbar();
  stamp_rt(P, EV_ROUTE_TOPK);
  if (*cx.S.abort) w.ok = false;
  // dispatch: every (token, slot) pair sets its bit in its expert's 128-bit mask, thread
  // e counts its bits, then a block-wide scan compacts the active experts
  const int tid = w.cw * 32 + w.lane;
  uint32_t* bits = reinterpret_cast<uint32_t*>(cx.S.dred);  // [E][4], bit s = t K + c
  for (int i = tid; i < E * 4; i += kComputeThreads) bits[i] = 0u;
  cbar();
  if (w.ok && tid < T * K) {
    // (after a failed wait topk_idx was never written: the index is range-checked)
    const int e = cx.S.topk_idx[(tid / K) * kMaxTopK + tid % K];
    if ((unsigned)e < (unsigned)E) atomicOr(&bits[e * 4 + (tid >> 5)], 1u << (tid & 31));
  }
  cbar();
  int cnt = 0;
  uint32_t b4[4] = {0u, 0u, 0u, 0u};
  if (tid < E) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      b4[j] = bits[tid * 4 + j];
      cnt += __popc(b4[j]);
    }
    cnt = min(cnt, 16);  // a token picks an expert at most once (NaN logits aside)
  }
  const int act = cnt > 0;
  int incl = act;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (w.lane >= o) incl += y;
  }
  float* red = cx.S.red;
  if (w.lane == 31) reinterpret_cast<int*>(red)[w.cw] = incl;
  cbar();
  int base = 0;
  for (int i = 0; i < w.cw; ++i) base += reinterpret_cast<int*>(red)[i];
  const int rank = base + incl - act;
  if (act) {
    cx.S.act_e[rank] = (int16_t)tid;
    cx.S.act_n[rank] = (uint8_t)cnt;
    int n = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      for (uint32_t m = b4[j]; m && n < 16; m &= m - 1u) {  // slots in increasing (token, slot) order
        const int sl = j * 32 + __ffs(m) - 1;
        cx.S.act_tok[rank * 16 + n] = (uint8_t)(sl / K);
        cx.S.act_slot[rank * 16 + n] = (uint8_t)sl;
        ++n;
      }
  }
  if (tid == kComputeThreads - 1) {
    int tot = 0;
    for (int i = 0; i < kComputeWarps; ++i) tot += reinterpret_cast<int*>(red)[i];
    *cx.S.n_active = tot;
  }
  // routing record and expert usage (block 0)
  if (cx.block == 0) {
    if (tid < T * K) {
      const int t = tid / K, c = tid % K;
      P.routing_idx[tid] = cx.S.topk_idx[t * kMaxTopK + c];
      P.routing_w[tid] = cx.S.topk_w[t * kMaxTopK + c];
    }
    if (tid < E) P.hist_cur[tid] = (uint32_t)cnt;
    if (tid < T) {
      P.tree_dbg[tid] = cx.S.anc[tid];
      P.tree_dbg[16 + tid] = (uint32_t)cx.S.tpos[tid];
    }
  }
  stamp_rt(P, EV_ROUTE_DISPATCH);
  // the dispatch tables are complete: the loader may stream this block's expert tiles
  // while the rows below are converted
  cbar();
  if (tid == 0) mbar_arrive(cx.S.route_bar, 1);
  cbar();
  if (tid == 0) {
    // the tensor-core warp's first GEMM1 tile of the ring, then its go
    *cx.S.tc_ti = w.ti;
    mbar_arrive(&cx.S.tcbar[TB_ROUTED], 1);
  }
  if (*cx.S.abort) w.ok = false;
}

// ---------------------------------------------------------------------------
// expert GEMMs on the tensor cores (tcgen05, accumulators in tensor memory)
// ---------------------------------------------------------------------------
// Work split: the block's expert units (128 rows x K, streamed as tiles of 512 or 256
// columns) are multiplied by one thread of the tensor-core warp (warp 2), which issues
// every MMA of the block in tile order, so each accumulator sums its K steps in a fixed
// order, and hands each ring slot back (one commit) once the tile's MMAs are done.  Both
// GEMMs run kind::mxf4nvf4 (E2M1 x E2M1, UE4M3 scales per 16 elements) with A the weight
// tile in the ring.  GEMM1's B is the split pooled vectors (64 rows: 4 terms x 16
// tokens, copied in once per launch); GEMM2's B is the expert's NVFP4 activation rows.
// The compute warp groups put each tile's weight scales into one of four scale buffers
// in tensor memory (the block's expert tile n by group n & 1, into buffer n & 3) and run
// the epilogues (tensor memory -> registers -> global), unit u by group u & 1; the
// accumulators alternate by unit.  (The tensor-core warp could copy the scales itself,
// but eight copies cost it as much issue time as the tile's eight MMAs.)

__device__ __forceinline__ uint32_t tm_lane(int quadrant) { return (uint32_t)(quadrant * 32) << 16; }

// GEMM1 epilogue of block-local unit `loc`: the unit's 128 accumulator rows are 64
// (gate, up) row pairs, interleaved, so lane pairs hold the two halves of one output
// column; h = silu(gate) * up for the expert's tokens goes to fp32 rows of `a` (the
// GEMM2 input; the consumer polls the -0.0 sentinel).  The accumulator is released
// whatever failed, so the tensor-core warp never waits on a skipped epilogue.
__device__ void g1_epilogue(Worker& w, int lo, int loc, uint32_t tm) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int upe = w1_units(dm.f);
  const int gu = lo + loc, a = gu / upe, jg = gu % upe;
  const int q = w.cw & 3, m = q * 32 + w.lane;
  const int d = loc & 1;
  float v[T];
  const bool ok = __all_sync(0xffffffffu, w.ok && wait_bar(cx, &cx.S.tcbar[TB_D1_FULL + d], (loc >> 1) & 1, PH_GEMM1));
  if (ok) {
    tc_fence_after();
    uint32_t r[kSplitTerms][16];
#pragma unroll
    for (int j = 0; j < kSplitTerms; ++j) tmem_ld16(tm + tm_lane(q) + TM_D1 + d * kSplitRows + j * 16, r[j]);
    tmem_ld_wait();
    // sum_j 4^-j D[term j][t], smallest term first (the factors are exact)
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float acc = __uint_as_float(r[kSplitTerms - 1][t]);
#pragma unroll
      for (int j = kSplitTerms - 2; j >= 0; --j) acc = fmaf(acc, 0.25f, __uint_as_float(r[j][t]));
      v[t] = acc;
    }
  }
  tc_fence_before();
  __syncwarp();
  if (w.lane == 0) mbar_arrive(&cx.S.tcbar[TB_D1_FREE + d], 1);
  if (!ok) {
    w.ok = false;
    return;
  }
  const int e = cx.S.act_e[a], n = cx.S.act_n[a];
  float* aout = reinterpret_cast<float*>(P.x_cur + P.xo.a);
  const float gs = P.w1_gs[e];
  const float* ts1 = reinterpret_cast<const float*>(cx.S.act + P.g1_b_off + b1_ts_off(dm.p));  // row scales
  for (int pi = 0; pi < n; ++pi) {
    const int tok = cx.S.act_tok[a * 16 + pi], slot = cx.S.act_slot[a * 16 + pi];
    float mine = 0.f;
#pragma unroll
    for (int t = 0; t < T; ++t) mine = t == tok ? v[t] : mine;
    const float sc = ts1[tok] * gs;
    const float up = __shfl_xor_sync(0xffffffffu, mine, 1) * sc;  // (odd lanes: the gate, unused)
    if (!(w.lane & 1)) {
      const float gate = mine * sc;
      const float av = gate / (1.0f + expf(-gate)) * up;
      st_relaxed_u32(aout + (size_t)slot * dm.f + jg * 64 + (m >> 1), __float_as_uint(f32_canon(av)));
    }
  }
  if (loc < 16 && q == 0 && w.lane == 0) stamp_any(P, EV_G1_EPI_DONE + loc);
}

// Expert tile n of the block (ring tile t): its weight scales -> scale buffer n & 3 of
// tensor memory once the MMAs of tile n - 4 are done with it, one word (a K=64 step's
// four scales) per row in four columns, lane m = row m.  The buffer's barrier is
// arrived at whatever failed (the tensor-core warp then gives up on its own waits).
__device__ void stage_sfa(Worker& w, uint32_t n, uint32_t t, int K, int phase) {
  Ctx& cx = *w.cx;
  const int q = w.cw & 3, m = q * 32 + w.lane;
  const uint32_t b = n & 3;
  bool ok = w.ok && !*cx.S.abort;
  if (n >= 4) ok = __all_sync(0xffffffffu, ok && wait_bar(cx, &cx.S.tcbar[TB_SFA_DONE + b], ((n >> 2) - 1) & 1, phase));
  ok = __all_sync(0xffffffffu, ok && wait_tile(cx, t, phase));
  if (ok) {
    tc_fence_after();
    const uint8_t* sc = cx.S.ring + cx.S.slot_off[t % kSlots] + exp_scale_off(K) + (m & 31) * 16 + (m >> 5) * 4;
    const uint32_t dst = *cx.S.tmem_base + tm_lane(q) + TM_SFA + 32 * b;
    for (int h = 0; h < exp_tile_k(K) / 256; ++h) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(sc + (4 * h + j) * 512);
        v[4 * j] = v[4 * j + 1] = v[4 * j + 2] = v[4 * j + 3] = wd;
      }
      tmem_st16(dst + 16 * h, v);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncwarp();
  if (w.lane == 0) mbar_arrive(&cx.S.tcbar[TB_SFA_FULL + b], 1);
  if (!ok) w.ok = false;
}

// GEMM1 on the compute side: group 1 stages the weight scales of every tile, group 0 runs
// the epilogue of every unit (the tensor-core warp does the rest).
__device__ void gemm1_phase(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int G = gridDim.x;
  const int NT = dm.p / exp_tile_k(dm.p);
  const int na = *cx.S.n_active, upe = w1_units(dm.f);
  int lo, hi;
  expert_units(na * upe, rot_block(cx.block, P.phase_rot * 6, G), G, false, lo, hi);
  // the operand (its row scales are read by the epilogues) has landed; the thread that
  // issued the copy waits for it whatever failed, before the top of the buffer is used
  // again (GEMM2) or the block exits
  if (!wait_bar(cx, &cx.S.tcbar[TB_B1], 0, PH_GEMM1)) w.ok = false;
  if (w.b1) {
    for (uint32_t it = 0; it < (1u << 24) && !mbar_try_wait(&cx.S.tcbar[TB_B1], 0); ++it) {
    }
  }
  const uint32_t tm = *cx.S.tmem_base;
  const int wg = w.cw >> 2;
  const int ntiles = (hi - lo) * NT;
  if (hi > lo) stamp_rt(P, EV_G1_FIRST_READY);
  if (wg == 1) {
    // group 1 puts every tile's weight scales in place as the tile lands (never held up
    // by an epilogue), group 0 runs every unit's epilogue
    for (int i = 0; i < ntiles; ++i) stage_sfa(w, (uint32_t)i, w.ti + (uint32_t)i, dm.p, PH_GEMM1);
  } else {
    for (int loc = 0; loc < hi - lo; ++loc) g1_epilogue(w, lo, loc, tm);
  }
  if (hi > lo) stamp_rt(P, EV_G1_LAST_DONE);
  w.ti += (uint32_t)ntiles;
  w.xseq = (uint32_t)ntiles;
}

// every MMA this thread issued has completed (bounded wait) before tensor memory is freed
__device__ void tc_drain(uint64_t* bar) {
  tc_commit(bar);
  const uint64_t dl = globaltimer() + 50000000ull;
  for (uint32_t it = 0; !mbar_try_wait(bar, 0); ++it)
    if ((it & 15) == 0 && globaltimer() > dl) break;
}

// GEMM2 epilogue of block-local unit `loc` (expert a of the round starting at a0):
// y rows of the expert's token slots, bf16
__device__ void g2_epilogue(Worker& w, int lo, int loc, int a0, uint32_t tm) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int upe = w2_units(dm.p);
  const int gu = lo + loc, a = gu / upe, pr = gu % upe, ea = a - a0;
  const int e = cx.S.act_e[a], n = cx.S.act_n[a];
  const int q = w.cw & 3, m = q * 32 + w.lane;
  const int d = loc & 1;
  uint32_t r[16];
  const bool ok = __all_sync(0xffffffffu, w.ok && wait_bar(cx, &cx.S.tcbar[TB_D2_FULL + d], (loc >> 1) & 1, PH_GEMM2));
  if (ok) {
    tc_fence_after();
    tmem_ld16(tm + tm_lane(q) + TM_D2 + d * 16, r);
    tmem_ld_wait();
  }
  tc_fence_before();
  __syncwarp();
  if (w.lane == 0) mbar_arrive(&cx.S.tcbar[TB_D2_FREE + d], 1);
  if (ok) {
    uint16_t* yout = reinterpret_cast<uint16_t*>(P.s_buf + P.so.y);
    const float gs = P.w2_gs[e];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      if (p < n) {
        const int slot = cx.S.act_slot[a * 16 + p];
        const float sc = cx.S.a_ts[ea * 16 + p] * gs;
        st_relaxed_u16(yout + (size_t)slot * dm.p + pr * kExpTileRows + m, bf16_bits_rn(__uint_as_float(r[p]) * sc));
      }
    }
  } else {
    w.ok = false;
  }
}

__device__ void gemm2_phase(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int G = gridDim.x;
  const int na = *cx.S.n_active, upe = w2_units(dm.p), NT = dm.f / exp_tile_k(dm.f);
  int lo, hi;
  expert_units(na * upe, rot_block(cx.block, P.phase_rot * 7, G), G, true, lo, hi);
  const float* ain = reinterpret_cast<const float*>(P.x_cur + P.xo.a);
  const uint32_t region = (uint32_t)dm.f * 8;  // one expert's 16 activation rows, E2M1, B layout
  uint8_t* g2b = cx.S.act + P.g2_off;          // the round's two experts' B operands
  uint8_t* sfb_stage = g2b + 2 * region;       // [2][16][F/16] UE4M3 block scales
  const int wg = w.cw >> 2, q = w.cw & 3;
  const uint32_t tm = *cx.S.tmem_base, tl = tm + tm_lane(q);
  const int tid = w.cw * 32 + w.lane;
  if (hi > lo) {
    const int a_first = lo / upe, a_last = (hi - 1) / upe;
    int epi = wg;  // next unit whose epilogue this group runs
    // the block's experts two at a time (one round unless its units span more than two)
    for (int a0 = a_first; a0 <= a_last; a0 += 2) {
      const int a1 = min(a0 + 1, a_last);
      cbar();  // the previous round's MMAs and epilogues are done with the staged operands
      if (a0 != a_first) stamp_rt(P, EV_G2_STAGE2_IN);
      if (*cx.S.abort) w.ok = false;
      // NVFP4 of every activation row of the round: row p of expert a = its p-th token
      const int n0 = cx.S.act_n[a0], nrows = n0 + (a1 > a0 ? cx.S.act_n[a1] : 0);
      float* rowbuf = reinterpret_cast<float*>(g2b + ((2 * region + 2 * dm.f + 1023) & ~1023u)) + (size_t)w.cw * dm.f;
      for (int r = w.cw; r < nrows && w.ok; r += kComputeWarps) {
        const int ea = r < n0 ? 0 : 1, p = r - ea * n0;
        const float* row = ain + (size_t)cx.S.act_slot[(a0 + ea) * 16 + p] * dm.f;
        // poll the row into shared memory (every pending chunk of a batch is re-read in
        // the same round), tracking the row's largest magnitude on the way
        const int nch4 = dm.f / 4;
        uint32_t amax_bits = 0u;  // |x| of non-negative floats orders like its bits
        constexpr int kB = 8;
        for (int c0 = w.lane; c0 < nch4 && w.ok; c0 += 32 * kB) {
          uint4 v[kB];
          uint32_t pending = 0;
#pragma unroll
          for (int j = 0; j < kB; ++j)
            if (c0 + 32 * j < nch4) pending |= 1u << j;
          w.ok = poll_batch<kB>(cx, reinterpret_cast<const uint4*>(row) + c0, 32, v, pending,
                                [](const uint4& x) { return f32x4_ready(x); }, PH_GEMM2);
          if (!w.ok) break;
#pragma unroll
          for (int j = 0; j < kB; ++j) {
            if (c0 + 32 * j >= nch4) continue;
            *reinterpret_cast<uint4*>(rowbuf + (c0 + 32 * j) * 4) = v[j];
            amax_bits = max(max(amax_bits, max(v[j].x & 0x7FFFFFFFu, v[j].y & 0x7FFFFFFFu)),
                            max(v[j].z & 0x7FFFFFFFu, v[j].w & 0x7FFFFFFFu));
          }
        }
        w.ok = __all_sync(0xffffffffu, w.ok);
        if (!w.ok) break;
        amax_bits = __reduce_max_sync(0xffffffffu, amax_bits);
        __syncwarp();
        // NVFP4 of the row: per-row fp32 scale amax / (6 * 448) rounded up to a power of
        // two, E4M3 block scale per 16 elements, E2M1 codes, every decision in fp32
        // (the same steps as the oracle's quantiser); four lanes per 16-element block
        const float amax = __uint_as_float(amax_bits);
        float ts = __fdiv_rn(amax, 2688.0f);  // amax / (6 * 448), rounded up to a power of two
        if (ts > 0.f) {
          int ex;
          const float mn = frexpf(ts, &ex);
          if (mn != 0.5f) ts = ldexpf(1.0f, ex);
        }
        uint8_t* bq = g2b + ea * region;
        for (int base = 0; base < dm.f; base += 128) {
          const int k = base + w.lane * 4;
          const bool in = k < dm.f;
          const float4 x = in ? *reinterpret_cast<const float4*>(rowbuf + k) : make_float4(0.f, 0.f, 0.f, 0.f);
          float bmax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
          bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
          bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 2));
          uint32_t sc = 0;
          if (ts > 0.f) sc = f32_to_e4m3(__fdiv_rn(bmax, __fmul_rn(6.0f, ts)));
          const float denom = __fmul_rn(e4m3_to_f32(sc), ts);
          uint32_t c01 = 0, c23 = 0;
          if (sc != 0) {
            c01 = f32x2_to_e2m1x2(__fdiv_rn(x.x, denom), __fdiv_rn(x.y, denom));
            c23 = f32x2_to_e2m1x2(__fdiv_rn(x.z, denom), __fdiv_rn(x.w, denom));
          }
          if (in) {
            // row p, byte k / 2 of the B operand: 256-column blocks of 16 rows x 128 bytes
            const int kb = k >> 8, bir = (k & 255) >> 1;
            *reinterpret_cast<uint16_t*>(bq + kb * 2048 + p * 128 + ((((bir >> 4) ^ (p & 7))) << 4) + (bir & 15)) =
                (uint16_t)(c01 | (c23 << 8));
            if ((w.lane & 3) == 0) sfb_stage[(ea * 16 + p) * (dm.f / 16) + (k >> 4)] = (uint8_t)sc;
          }
        }
        __syncwarp();  // the warp's next row reuses rowbuf
        if (w.lane == 0) cx.S.a_ts[ea * 16 + p] = ts;
      }
      w.ok = __all_sync(0xffffffffu, w.ok);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B rows -> the MMAs
      cbar();
      // activation block scales -> tensor memory: lane p of every quadrant, per K=64 step
      // one word (its four scales) in four columns; rows past the expert's tokens hold 0
      if (wg == 0 && w.ok) {
        const int nk = dm.f / 64;
        for (int ea = 0; ea <= a1 - a0; ++ea) {
          const int na_rows = cx.S.act_n[a0 + ea];
          for (int g = 0; g < nk; g += 4) {
            uint32_t v[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t wd = (w.lane < na_rows && g + j < nk)
                                      ? *reinterpret_cast<const uint32_t*>(sfb_stage + (ea * 16 + w.lane) * (dm.f / 16) + 4 * (g + j))
                                      : 0u;
              v[4 * j] = v[4 * j + 1] = v[4 * j + 2] = v[4 * j + 3] = wd;
            }
            tmem_st16(tl + TM_SFB2 + ea * 64 + g * 4, v);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      cbar();
      if (tid == 0) mbar_arrive(&cx.S.tcbar[TB_G2_STAGE], 1);
      if (a0 == a_first) stamp_rt(P, EV_GEMM2_IN);
      else stamp_rt(P, EV_G2_STAGE2_DONE);
      if (*cx.S.abort) w.ok = false;
      // this round's tiles: weight scales of the group's tiles (expert tile n = xseq + i
      // by group n & 1), epilogues interleaved
      const int u_lo = max(lo, a0 * upe), u_hi = min(hi, (a1 + 1) * upe);
      const int i_lo = (u_lo - lo) * NT, i_hi = (u_hi - lo) * NT;
      for (int i = i_lo + ((int)((w.xseq + (uint32_t)i_lo) & 1u) != wg ? 1 : 0); i < i_hi; i += 2) {
        for (; epi <= i / NT - 2 && w.ok; epi += 2) g2_epilogue(w, lo, epi, a0, tm);
        stage_sfa(w, w.xseq + (uint32_t)i, w.ti + (uint32_t)i, dm.f, PH_GEMM2);
        if (i < 2 && a0 == a_first) stamp_rt(P, EV_G2_FIRST_READY);
      }
      // every epilogue of the round before its operands are replaced
      for (; epi < u_hi - lo && w.ok; epi += 2) g2_epilogue(w, lo, epi, a0, tm);
    }
    stamp_rt(P, EV_G2_LAST_DONE);
  }
  w.ti += (uint32_t)((hi - lo) * NT);
}

// The tensor-core warp: one thread issues every expert MMA of the block in tile order
// (orcarouter.ai, § "where the kernel boundary sits": warps dedicated to driving the
// tensor cores) and hands each ring slot back to the loader when the tile's MMAs are done.

// expert tile seq's weight scales are in scale buffer seq & 3 and the tile has landed
__device__ __forceinline__ bool tile_ready(Ctx& cx, uint32_t seq, uint32_t t, int phase) {
  return wait_bar(cx, &cx.S.tcbar[TB_SFA_FULL + (seq & 3)], (seq >> 2) & 1, phase) && wait_tile(cx, t, phase);
}
// a tile's MMAs are issued: its scale buffer and its ring slot are released when they are done
__device__ __forceinline__ void tile_done(Ctx& cx, uint32_t seq, uint32_t t) {
  tc_commit(&cx.S.tcbar[TB_SFA_DONE + (seq & 3)]);
  tc_commit(&cx.S.tcbar[TB_SLOT + t % kSlots]);
}

// The block's dense weight tiles, in the loader's order (its hand-over queue): each goes
// from its ring slot to tensor-memory slot di % 8 with 128x256b copies as soon as it
// lands, which releases the ring slot (one commit) and hands the tile to its consumers
// (another); the slot is reused once the tile eight before has been read.  Returns at
// the loader's routing-wait or end marker.
__device__ uint32_t dense_queue(Ctx& cx, uint32_t& q, uint32_t& di, bool& ok) {
  uint64_t* tb = cx.S.tcbar;
  const uint32_t tm = *cx.S.tmem_base;
  for (;;) {
    const uint32_t k = q % kDenseQ;
    uint32_t n = 0;
    while (cx.S.dq_seq[k] != q + 1) {
      __nanosleep(32);
      if ((++n & 15) == 0 && cx.expired(PH_TC_DENSE)) {
        ok = false;
        return kDqEnd;
      }
    }
    __threadfence_block();
    const uint32_t e = cx.S.dq_e[k];
    ++q;
    if (e == kDqRoute || e == kDqEnd) return e;
    const uint32_t ti = e & 0xFFFFFFu, chunks = e >> 24;
    const uint32_t j = di % kDenseTmemSlots;
    if (di >= kDenseTmemSlots) ok = wait_bar(cx, &tb[TB_TFREE + j], ((di / kDenseTmemSlots) - 1) & 1, PH_TC_DENSE);
    const uint32_t s = ti % kSlots;
    if (ok) ok = wait_bar(cx, &cx.S.full[s], (ti / kSlots) & 1, PH_TC_DENSE);
    if (!ok) return kDqEnd;
    tc_fence_after();
    const uint32_t a_s = smem_u32(cx.S.ring + cx.S.slot_off[s]);
    for (uint32_t c = 0; c < chunks; c += 2)  // two 2 KB chunks per copy
      tc_cp_128x256b(tm + j * kDenseTmemCols + 4 * c, sdesc_kmajor(a_s + c * 2048u, 2048, 128));
    tc_commit(&tb[TB_SLOT + s]);
    tc_commit(&tb[TB_TFULL + j]);
    ++di;
  }
}
// every dense tile handed over so far has been read (before other tensor-memory use)
__device__ bool dense_drain(Ctx& cx, uint32_t di) {
  for (uint32_t d = di > (uint32_t)kDenseTmemSlots ? di - kDenseTmemSlots : 0u; d < di; ++d)
    if (!wait_bar(cx, &cx.S.tcbar[TB_TFREE + d % kDenseTmemSlots], (d / kDenseTmemSlots) & 1, PH_TC_DENSE))
      return false;
  tc_fence_after();
  return true;
}

__device__ void tc_issuer(Ctx& cx) {
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  uint64_t* tb = cx.S.tcbar;
  const uint32_t tm = *cx.S.tmem_base;
  const int G = gridDim.x;
  // dense tiles up to the routing decision (a draft model: the whole launch)
  uint32_t q = 0, di = 0;
  bool ok = true;
  const uint32_t m0 = dense_queue(cx, q, di, ok);
  // the expert phases: their tensor-memory columns once every dense tile is read
  if (ok && m0 == kDqRoute) ok = dense_drain(cx, di) && wait_bar(cx, &tb[TB_ROUTED], 0, PH_ROUTE);
  if (ok && m0 == kDqRoute) {
    const int na = *cx.S.n_active;
    uint32_t seq = 0;                 // expert tiles issued so far
    const uint32_t t1 = *cx.S.tc_ti;  // ring index of the block's first expert tile
    uint32_t t2 = t1;                 // ... of its first GEMM2 tile
    // ---- GEMM1: D[128 rows][term 16 + token] += W1 tile . B^T ----
    {
      const int tk = exp_tile_k(dm.p), nst = tk / 64, NT = dm.p / tk;
      int lo, hi;
      expert_units(na * w1_units(dm.f), rot_block(cx.block, P.phase_rot * 6, G), G, false, lo, hi);
      t2 = t1 + (uint32_t)((hi - lo) * NT);
      const uint32_t sfb_s = smem_u32(cx.S.act + P.g1_b_off), b_s = sfb_s + (uint32_t)b1_code_off(dm.p);
      if (hi > lo) {
        ok = wait_bar(cx, &tb[TB_B1], 0, PH_GEMM1);
        if (ok) {
          stamp_any(P, EV_B1_LANDED);
          // the operand's scale groups -> tensor memory, one per K=64 step
          for (int s = 0; s < dm.p / 64; ++s)
            tc_cp_32x128b_x4(tm + TM_SFB1 + 4 * s, sdesc_plain(sfb_s + 512 * s, 128));
          tc_commit(&tb[TB_SFB1]);  // once copied, the scale groups' shared memory may take ring tiles
        }
      }
      for (int loc = 0; loc < hi - lo && ok; ++loc) {
        const int d = loc & 1;
        if (loc >= 2) {
          ok = wait_bar(cx, &tb[TB_D1_FREE + d], ((loc >> 1) - 1) & 1, PH_GEMM1);
          if (!ok) break;
          tc_fence_after();
        }
        for (int kt = 0; kt < NT; ++kt) {
          const int i = loc * NT + kt;
          const uint32_t t = t1 + (uint32_t)i;
          ok = tile_ready(cx, seq, t, PH_GEMM1);
          if (!ok) break;
          if (i < 16) stamp_any(P, EV_TC_G1_READY + i);
          tc_fence_after();
          const uint32_t a_s = smem_u32(cx.S.ring + cx.S.slot_off[t % kSlots]);
          const uint32_t sfa = tm + TM_SFA + 32 * (seq & 3);
          for (int j = 0; j < nst; ++j) {
            const int kg = kt * tk + 64 * j;  // first column of the step
            mma_nvf4_ss(tm + TM_D1 + d * kSplitRows, sdesc_k_sw128(a_s + (j >> 2) * kExpBlockBytes + (j & 3) * 32),
                        sdesc_k_sw128(b_s + (kg >> 8) * (kSplitRows * 128) + ((kg >> 6) & 3) * 32), idesc_nvf4(kSplitRows),
                        sfa + 4 * j, tm + TM_SFB1 + 4 * (kg >> 6), (kt | j) != 0);
          }
          tile_done(cx, seq, t);
          ++seq;
          if (i < 16) stamp_any(P, EV_TC_G1_ISSUED + i);
        }
        if (ok) tc_commit(&tb[TB_D1_FULL + d]);
      }
    }
    // ---- GEMM2: D[128 rows][token slot] += W2 tile . B^T, two experts per round ----
    if (ok) {
      const int tk = exp_tile_k(dm.f), nst = tk / 64, NT = dm.f / tk, upe = w2_units(dm.p);
      int lo, hi;
      expert_units(na * upe, rot_block(cx.block, P.phase_rot * 7, G), G, true, lo, hi);
      const uint32_t act_s = smem_u32(cx.S.act + P.g2_off), region = (uint32_t)dm.f * 8;
      if (hi > lo) {
        const int a_first = lo / upe, a_last = (hi - 1) / upe;
        int round = 0;
        for (int a0 = a_first; a0 <= a_last && ok; a0 += 2, ++round) {
          const int a1 = min(a0 + 1, a_last);
          ok = wait_bar(cx, &tb[TB_G2_STAGE], round & 1, PH_GEMM2);
          if (!ok) break;
          tc_fence_after();
          const int u_lo = max(lo, a0 * upe), u_hi = min(hi, (a1 + 1) * upe);
          for (int gu = u_lo; gu < u_hi && ok; ++gu) {
            const int loc = gu - lo, ea = gu / upe - a0, d = loc & 1;
            if (loc >= 2) {
              ok = wait_bar(cx, &tb[TB_D2_FREE + d], ((loc >> 1) - 1) & 1, PH_GEMM2);
              if (!ok) break;
              tc_fence_after();
            }
            for (int kt = 0; kt < NT; ++kt) {
              const int i = loc * NT + kt;
              const uint32_t t = t2 + (uint32_t)i;
              ok = tile_ready(cx, seq, t, PH_GEMM2);
              if (!ok) break;
              if (i < 8) stamp_any(P, EV_TC_G2_READY + i);
              tc_fence_after();
              const uint32_t a_s = smem_u32(cx.S.ring + cx.S.slot_off[t % kSlots]);
              const uint32_t sfa = tm + TM_SFA + 32 * (seq & 3);
              for (int j = 0; j < nst; ++j) {
                const int kb = j >> 2, jj = j & 3;  // 16 KB column block, K=64 step inside it
                mma_nvf4_ss(tm + TM_D2 + d * 16, sdesc_k_sw128(a_s + kb * kExpBlockBytes + jj * 32),
                            sdesc_k_sw128(act_s + ea * region + (kt * (tk / 256) + kb) * 2048 + jj * 32), idesc_nvf4(16),
                            sfa + 4 * j, tm + TM_SFB2 + ea * 64 + (kt * nst + j) * 4, (kt | j) != 0);
              }
              tile_done(cx, seq, t);
              ++seq;
              if (i < 8) stamp_any(P, EV_TC_G2_ISSUED + i);
            }
            if (ok) tc_commit(&tb[TB_D2_FULL + d]);
          }
        }
      }
    }
    // the unpooler and the next layer's QKV (or the LM head): dense tiles again, once the
    // compute warps are done with the expert phases' tensor memory
    if (ok) ok = wait_bar(cx, &tb[TB_XDONE], 0, PH_TC_DENSE);
    if (ok) {
      tc_fence_after();
      dense_queue(cx, q, di, ok);
    }
  }
  tc_drain(&tb[TB_DRAIN]);
}

// z[t] = bf16(sum_c w[t][c] * y[t*k + c]); each y element has this one consumer,
// which re-arms it after reading
__device__ void combine_phase(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int G = gridDim.x;
  uint16_t* y = reinterpret_cast<uint16_t*>(P.s_buf + P.so.y);
  uint16_t* z = reinterpret_cast<uint16_t*>(P.x_cur + P.xo.z);
  const int nch = dm.p / 8;
  const int gt = rot_block(cx.block, P.phase_rot * 10, G) * kComputeThreads + w.cw * 32 + w.lane;
  if (!await_phase(w, CNT_GEMM2, PH_COMBINE)) return;
  for (int it = gt; it < T * nch && w.ok; it += G * kComputeThreads) {
    const int t = it / nch, pc = it % nch;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint4 v[kMaxTopK];
#pragma unroll
    for (int c = 0; c < kMaxTopK; ++c)
      if (c < dm.k) v[c] = ld_relaxed_v4(y + (size_t)(t * dm.k + c) * dm.p + pc * 8);
#pragma unroll
    for (int c = 0; c < kMaxTopK; ++c) {
      if (c >= dm.k) continue;
      const float wt = cx.S.topk_w[t * kMaxTopK + c];
      const uint32_t wd[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += wt * bf16_to_f32((uint16_t)(wd[i] & 0xFFFF));
        acc[2 * i + 1] += wt * bf16_to_f32((uint16_t)(wd[i] >> 16));
      }
    }
    st_relaxed_v4(z + (size_t)t * dm.p + pc * 8,
                  make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                             pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
  }
  w.ok = __all_sync(0xffffffffu, w.ok);
}

// rotary table [depth 0..15][hd/2] (cos, sin); angle in fp64, reduced to [-pi, pi]
__device__ void rope_table(Worker& w) {
  const LaunchParams& P = *w.cx->P;
  const int half = P.dm.hd / 2;
  const int tid = w.cw * 32 + w.lane;
  for (int i = tid; i < 16 * half; i += kComputeThreads) {
    const int dep = i / half, k = i % half;
    double ang = (double)(w.cx->pos0 + dep) * P.inv_freq[k];
    const double two_pi = 6.283185307179586476925286766559;
    ang = ang - two_pi * rint(ang / two_pi);
    float s, c;
    sincosf((float)ang, &s, &c);
    P.rope[2 * i] = c;
    P.rope[2 * i + 1] = s;
  }
}

// QKV epilogue: RoPE pairs (d, d + hd/2) share a unit (rows g and g+8)
// re-arm the exchange buffers of the other parity (warps 1-2)
__device__ void rearm(const LaunchParams& P, int block, int tid, int nthreads) {
  struct R { uint64_t off, bytes; uint32_t pat; };
  const R regs[] = {
      {P.xo.o, P.xo.h1 - P.xo.o, 0xFFFFFFFFu},   {P.xo.h1, P.xo.u - P.xo.h1, 0xFFFFFFFFu},
      {P.xo.u, P.xo.logits - P.xo.u, 0xFFFFFFFFu}, {P.xo.logits, P.xo.a - P.xo.logits, kF32Empty},
      {P.xo.a, P.xo.z - P.xo.a, kF32Empty},       {P.xo.z, P.xo.h2 - P.xo.z, 0xFFFFFFFFu},
      {P.xo.h2, P.xo.q0 - P.xo.h2, 0xFFFFFFFFu},   {P.xo.q0, P.xo.tkv0 - P.xo.q0, 0xFFFFFFFFu},
      {P.xo.tkv0, P.xo.cnt - P.xo.tkv0, 0xFFFFFFFFu}, {P.xo.cnt, P.xo.b1 - P.xo.cnt, 0u}};
  const int G = gridDim.x;
#pragma unroll 1
  for (int ri = 0; ri < 10; ++ri) {
    const R& r = regs[ri];
    const uint64_t n16 = r.bytes / 16;
    const uint64_t lo = n16 * block / G, hi = n16 * (block + 1) / G;
    const uint4 v = make_uint4(r.pat, r.pat, r.pat, r.pat);
    for (uint64_t i = lo + tid; i < hi; i += nthreads)
      *reinterpret_cast<uint4*>(P.x_next + r.off + i * 16) = v;
  }
}

// A draft model's FFN half of the layer, in place of the MoE half:
//   z  = bf16(silu(x W_gate^T) * (x W_up^T)), x = bf16(RMSNorm(h1))
//   h2 = bf16(h1 + bf16(z W_down^T))
// The gate and up rows are paired in one unit (rows p / p + 8), so one dense phase
// over N = 2f gives z.  z ([16][f] bf16) is larger than the activation buffer, so the
// down projection runs as two dense phases over the two K halves of z: the first
// leaves fp32 partial sums, the second (the same units, so the same threads) adds
// them before the rounding.  The phase counters of the pooler and the unpooler mark
// z and h2.
__device__ void draft_ffn(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  uint8_t* X = P.x_cur;
  const uint16_t* h1 = reinterpret_cast<const uint16_t*>(X + P.xo.h1);
  uint16_t* z = reinterpret_cast<uint16_t*>(X + P.xo.z);
  float* part = reinterpret_cast<float*>(P.s_buf + P.so.part);
  const int fh = dm.f / 2;
  stage_act(w, h1, dm.d, CNT_OPROJ, false, P.g_moe, dm.rms_eps, PH_POOL, ACT_H1);
  {
    EpiArgs ea{};
    ea.kind = EPI_SWIGLU;
    ea.out = z;
    dense_phase(w, dm.d, 2 * dm.f, P.phase_rot * 4, ea, -1);
    publish(w, CNT_POOL);
  }
  stage_act(w, z, fh, CNT_POOL, false, nullptr, 0.f, PH_ROUTER, ACT_U);
  {
    EpiArgs ea{};
    ea.kind = EPI_PARTIAL;
    ea.out32 = part;
    dense_phase(w, fh, dm.d, P.phase_rot * 5, ea, -1);
  }
  stage_act(w, z + (size_t)16 * fh, fh, CNT_POOL, false, nullptr, 0.f, PH_UNPOOL, ACT_Z);
  {
    EpiArgs ea{};
    ea.kind = EPI_UNPOOL;
    ea.res = h1;
    ea.out = reinterpret_cast<uint16_t*>(X + P.xo.h2);
    ea.out2 = P.last ? P.hidden_out : P.out_h;
    ea.part = part;
    dense_phase(w, fh, dm.d, P.phase_rot * 5, ea, -1);
    publish(w, CNT_UNPOOL);
  }
}

// ---------------------------------------------------------------------------
// the compute warps' sequence of one launch
// ---------------------------------------------------------------------------
template <bool kTiming, bool kDraft>
__device__ void compute_main(Worker& w) {
  Ctx& cx = *w.cx;
  const LaunchParams& P = *cx.P;
  const Dims& dm = P.dm;
  const int b = blockIdx.x;
  uint8_t* X = P.x_cur;
  if (P.first) {
    // the rotary table of this step's tree positions, then the prologue:
    // RMSNorm(hidden_in) -> layer 0 QKV -> RoPE -> layer 0 KV rows and Q
    rope_table(w);
    stage_act(w, P.hidden_in, dm.d, -1, false, P.g_attn_pro, dm.rms_eps, PH_PROLOGUE);
    stamp<kTiming>(P, b, EV_PRO_IN);
    EpiArgs ea{};
    ea.kind = EPI_QKV;
    ea.dq = QkvDst{reinterpret_cast<uint16_t*>(X + P.xo.q0), true, P.kc, P.vc, reinterpret_cast<uint16_t*>(X + P.xo.tkv0)};
    dense_phase(w, dm.d, dm.nqkv, P.phase_rot * 1, ea, -1);
    stamp<kTiming>(P, b, EV_PRO_DONE);
    cbar();
  }
  // a2: tree attention (split over blocks), a3: merge of the split partials
  if (dm.hd == 128) attention_phase<128, kDraft>(w);
  else attention_phase<64, kDraft>(w);
  publish(w, CNT_ATTN);
  stamp<kTiming>(P, b, EV_ATTN_DONE);
  if (dm.hd == 128) attn_merge_phase<128>(w);
  else attn_merge_phase<64>(w);
  publish(w, CNT_MERGE);
  stamp<kTiming>(P, b, EV_MERGE_DONE);
  // a4: h1 = bf16(h + bf16(O W_o^T))
  {
    const uint16_t* hprev = P.first ? P.hidden_in : P.in_h;
    uint16_t* h1 = reinterpret_cast<uint16_t*>(X + P.xo.h1);
    stage_act(w, reinterpret_cast<const uint16_t*>(X + P.xo.o), dm.hq * dm.hd, CNT_MERGE, false, nullptr, 0.f, PH_OPROJ,
              ACT_O);
    stamp<kTiming>(P, b, EV_OPROJ_IN);
    EpiArgs ea{};
    ea.kind = EPI_OPROJ;
    ea.res = hprev;
    ea.out = h1;
    dense_phase(w, dm.hq * dm.hd, dm.d, P.phase_rot * 3, ea, EV_OP_U0_FIRST);
    publish(w, CNT_OPROJ);
    stamp<kTiming>(P, b, EV_OPROJ_DONE);
  }
  if constexpr (kDraft) {
    draft_ffn(w);
  } else {
  // a5: u = bf16(bf16(RMSNorm(h1)) W_pool^T)
  {
    uint16_t* uo = reinterpret_cast<uint16_t*>(X + P.xo.u);
    stage_act(w, reinterpret_cast<const uint16_t*>(X + P.xo.h1), dm.d, CNT_OPROJ, false, P.g_moe, dm.rms_eps, PH_POOL,
              ACT_H1);
    stamp<kTiming>(P, b, EV_POOL_IN);
    EpiArgs ea{};
    ea.kind = EPI_POOL;
    ea.out = uo;
    dense_phase(w, dm.d, dm.p, P.phase_rot * 4, ea, -1);
    publish(w, CNT_POOL);
    stamp<kTiming>(P, b, EV_POOL_DONE);
  }
  // a6: router logits = u W_r^T + b (fp32)
  {
    float* lg = reinterpret_cast<float*>(X + P.xo.logits);
    stage_act(w, reinterpret_cast<const uint16_t*>(X + P.xo.u), dm.p, CNT_POOL, false, nullptr, 0.f, PH_ROUTER, ACT_U);
    stamp<kTiming>(P, b, EV_ROUTER_IN);
    EpiArgs ea{};
    ea.kind = EPI_ROUTER;
    ea.out32 = lg;
    dense_phase(w, dm.p, dm.e, P.phase_rot * 5, ea, -1);
    // a8 (GEMM1 side): this block's share of the split pooled vectors
    split_pooled(w);
    stamp_rt(P, EV_SPLIT_DONE);
    publish(w, CNT_ROUTER);
    stamp<kTiming>(P, b, EV_ROUTER_DONE);
  }
  // a6/a7: top-k and dispatch (and the copy of GEMM1's operand B, which overwrites the
  // staged pooled vectors: every thread's generic accesses of them go first)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  await_phase(w, CNT_ROUTER, PH_ROUTE);
  route_phase(w);
  stamp<kTiming>(P, b, EV_ROUTE_DONE);
  // a9, a10: the expert GEMMs
  gemm1_phase(w);
  stamp<kTiming>(P, b, EV_GEMM1_DONE);
  gemm2_phase(w);
  // the expert phases' tensor-memory reads are done: the dense tiles may come back
  tc_fence_before();
  __syncwarp();
  if (w.lane == 0) mbar_arrive(&cx.S.tcbar[TB_XDONE], 1);
  publish(w, CNT_GEMM2);
  stamp<kTiming>(P, b, EV_GEMM2_DONE);
  // move the next layer's KV history toward L2 while the combine waits
  if ((P.flags & 0x4u) && !P.last && w.cw == 0 && w.lane == 0 && P.kc_pf != nullptr) {
    const AttnUnit au = attn_unit(P, cx.pos0, rot_block(b, P.phase_rot * 2, gridDim.x), P.next_global);
    if (au.valid && au.r1 > au.r0) {
      const size_t off = ((size_t)au.hk * dm.max_ctx + au.r0) * dm.hd;
      const uint32_t bytes = (uint32_t)((au.r1 - au.r0) * dm.hd * 2);
      prefetch_l2(P.kc_pf + off, bytes);
      prefetch_l2(P.vc_pf + off, bytes);
    }
  }
  // a11: combine, then h2 = bf16(h1 + bf16(z W_unp^T))
  combine_phase(w);
  publish(w, CNT_COMBINE);
  stamp<kTiming>(P, b, EV_COMBINE_DONE);
  {
    const uint16_t* h1 = reinterpret_cast<const uint16_t*>(X + P.xo.h1);
    uint16_t* h2 = reinterpret_cast<uint16_t*>(X + P.xo.h2);
    uint16_t* hnext = P.last ? P.hidden_out : P.out_h;
    stage_act(w, reinterpret_cast<const uint16_t*>(X + P.xo.z), dm.p, CNT_COMBINE, false, nullptr, 0.f, PH_UNPOOL, ACT_Z,
              (uint32_t)P.unpool_act_off);
    stamp<kTiming>(P, b, EV_UNPOOL_IN);
    EpiArgs ea{};
    ea.kind = EPI_UNPOOL;
    ea.res = h1;
    ea.out = h2;
    ea.out2 = hnext;
    dense_phase(w, dm.p, dm.d, P.phase_rot * 8, ea, -1, (uint32_t)P.unpool_act_off);
    publish(w, CNT_UNPOOL);
    stamp<kTiming>(P, b, EV_UNPOOL_DONE);
  }
  }
  pdl_launch_dependents();
  // a12: next layer's RMSNorm + QKV + RoPE + KV write; a12': final norm + LM head
  if (!P.last) {
    stage_act(w, reinterpret_cast<const uint16_t*>(X + P.xo.h2), dm.d, CNT_UNPOOL, false, P.g_tail, dm.rms_eps, PH_TAIL,
              ACT_H2);
    stamp<kTiming>(P, b, EV_TAIL_IN);
    EpiArgs ea{};
    ea.kind = EPI_QKV;
    ea.dq = QkvDst{P.out_q, false, P.kc_next, P.vc_next, nullptr};
    dense_phase(w, dm.d, dm.nqkv, P.phase_rot * 9, ea, -1);
  } else if (dm.vocab > 0) {
    stage_act(w, reinterpret_cast<const uint16_t*>(X + P.xo.h2), dm.d, CNT_UNPOOL, false, P.g_tail, dm.rms_eps, PH_TAIL,
              ACT_H2);
    stamp<kTiming>(P, b, EV_TAIL_IN);
    EpiArgs ea{};
    ea.kind = EPI_LMHEAD;
    ea.out32 = P.logits;
    dense_phase(w, dm.d, dm.vocab, P.phase_rot * 9, ea, -1);
  }
  stamp<kTiming>(P, b, EV_TAIL_DONE);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool kTiming, bool kDraft>
__global__ void __launch_bounds__(kThreads, 1) msm_layer_kernel(const __grid_constant__ LaunchParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.P = &P;
  cx.S = carve(smem, P);
  cx.block = blockIdx.x;
  cx.deadline = globaltimer() + (((uint64_t)P.timeout_ns_hi << 32) | P.timeout_ns_lo) + 1000000000ull;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&cx.S.full[i], 1);
      mbar_init(&cx.S.empty[i], kComputeWarps);
    }
    mbar_init(cx.S.route_bar, 1);
    mbar_init(cx.S.stage_bar, 1);
    for (int i = 0; i < kTcBars; ++i) {
      const bool by4 = (i >= TB_D1_FREE && i < TB_D1_FREE + 2) || (i >= TB_D2_FREE && i < TB_D2_FREE + 2) ||
                       (i >= TB_SFA_FULL && i < TB_SFA_FULL + 4) || (i >= TB_TFREE && i < TB_TFREE + kDenseTmemSlots);
      mbar_init(&cx.S.tcbar[i], (i == TB_DONE || i == TB_XDONE) ? kComputeWarps : by4 ? 4 : 1);
    }
    for (int i = 0; i < kSlots; ++i) cx.S.slot_tile[i] = 0xFFFFFFFFu;
    for (int i = 0; i < kDenseQ; ++i) cx.S.dq_seq[i] = 0u;
    *cx.S.abort = (smem_u32(smem) & 1023u) != 0u;  // the swizzled tiles need 1 KB alignment
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // a1: the tree (ancestor-or-self masks, depths, positions) from the parent array,
  // taken from the launch parameters or from the device-resident step state; a state
  // is checked first (parent[0] == -1, 0 <= parent[i] < i, 0 <= pos0 <= max_ctx - 16),
  // so the walk below always ends and every cache row stays in range
  if (warp == 1) {
    // the parents travel through the GEMM1 row-scale scratch, unused until routing
    int* par = reinterpret_cast<int*>(cx.S.x_ts);
    int pos0 = P.pos0, pv = lane < T ? P.parent[lane] : 0;
    if (P.state != nullptr) {
      // (a draft model reads only pos0: its block is always the chain)
      pos0 = P.state[0];
      pv = lane < T ? (kDraft ? lane - 1 : P.state[1 + lane]) : 0;
    }
    const bool ok = __all_sync(0xffffffffu, lane >= T || (lane == 0 ? pv == -1 : (pv >= 0 && pv < lane))) &&
                    pos0 >= 0 && pos0 <= P.dm.max_ctx - T;
    if (lane < T) par[lane] = pv;
    if (lane == 0) *cx.S.pos0 = ok ? pos0 : -1;  // -1: the block gives up below
    __syncwarp();
    if (!ok) {
      if (lane == 0) atomicCAS(&P.status->code, 0, 1 /* MSM_ERR_INVALID_ARG */);
    } else if (lane < T) {
      uint32_t m = 0;
      int dep = 0;
      for (int j = lane; j >= 0; j = par[j]) {
        m |= 1u << j;
        if (j != lane) ++dep;
      }
      // (a draft model's block is a chain whose slots all see one another)
      cx.S.anc[lane] = kDraft ? 0xFFFFu : m;
      cx.S.depth[lane] = dep;
      cx.S.tpos[lane] = pos0 + dep;
    }
  }
  if (warp == 2) {
    // the tensor-core warp holds the block's tensor memory for the whole launch (one
    // block per SM, so the columns are free once the previous launch's block has left)
    tmem_alloc(cx.S.tmem_base, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  cx.pos0 = *cx.S.pos0;
  if (*cx.S.abort || cx.pos0 < 0) {
    if (threadIdx.x == 0 && atomicCAS(&P.status->code, 0, 2) == 0) P.status->phase = PH_START;
    if (warp == 2) tmem_dealloc(*cx.S.tmem_base, kTmemCols);
    pdl_launch_dependents();
    return;
  }
  if (warp == kLoaderWarp) {
    if (lane == 0) loader<kTiming, kDraft>(cx);
    pdl_launch_dependents();
    return;
  }
  if (warp == 1) {
    pdl_wait();
    rearm(P, blockIdx.x, lane, 32);
    pdl_launch_dependents();
    return;
  }
  if (warp == 2) {
    pdl_wait();
    cx.deadline = globaltimer() + (((uint64_t)P.timeout_ns_hi << 32) | P.timeout_ns_lo);
    if (lane == 0) tc_issuer(cx);
    __syncwarp();
    // free tensor memory once the compute warps are done with it
    if (lane == 0) {
      const uint64_t dl = globaltimer() + (((uint64_t)P.timeout_ns_hi << 32) | P.timeout_ns_lo) + 50000000ull;
      for (uint32_t it = 0; !mbar_try_wait(&cx.S.tcbar[TB_DONE], 0); ++it)
        if ((it & 15) == 0 && globaltimer() > dl) break;
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*cx.S.tmem_base, kTmemCols);
    pdl_launch_dependents();
    return;
  }
  if (warp == kPrefetchWarp) {
    pdl_wait();
    if ((P.flags & 0x2u) && P.hist_prev != nullptr && P.prefetch_experts > 0) {
      // the previous step's most-used experts of this layer -> L2 (block-strided slices)
      const Dims& dm = P.dm;
      const uint64_t ub1 = exp_unit_bytes(dm.p) * w1_units(dm.f), ub2 = exp_unit_bytes(dm.f) * w2_units(dm.p);
      uint32_t taken[kMaxExperts / 32] = {0};
      for (int c = 0; c < P.prefetch_experts && c < dm.e; ++c) {
        uint32_t best = 0;
        int bi = -1;
        for (int e = lane; e < dm.e; e += 32) {
          const uint32_t h = P.hist_prev[e];
          if (!((taken[e >> 5] >> (e & 31)) & 1u) && h > 0 && (bi < 0 || h > best)) { best = h; bi = e; }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const uint32_t ob = __shfl_xor_sync(0xffffffffu, best, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (oi >= 0 && (bi < 0 || ob > best || (ob == best && oi < bi))) { best = ob; bi = oi; }
        }
        if (bi < 0) break;
        taken[bi >> 5] |= 1u << (bi & 31);
        const uint8_t* srcs[2] = {P.w1 + (uint64_t)bi * ub1, P.w2 + (uint64_t)bi * ub2};
        const uint64_t sizes[2] = {ub1, ub2};
        for (int m = 0; m < 2; ++m) {
          const uint64_t chunk = 16384;
          const uint64_t nck = (sizes[m] + chunk - 1) / chunk;
          for (uint64_t ck = (uint64_t)blockIdx.x * 32 + lane; ck < nck; ck += (uint64_t)gridDim.x * 32) {
            const uint64_t o = ck * chunk;
            prefetch_l2(srcs[m] + o, (uint32_t)min(chunk, sizes[m] - o));
          }
        }
      }
    }
    pdl_launch_dependents();
    return;
  }
  // ---- compute warps ----
  Worker w;
  w.cx = &cx;
  w.cw = warp - kFirstCompute;
  w.lane = lane;
  w.g = lane >> 2;
  w.q = lane & 3;
  w.ti = 0;
  w.di = 0;
  w.ok = true;
  w.b1 = false;
  w.xseq = 0;
  pdl_wait();
  cx.deadline = globaltimer() + (((uint64_t)P.timeout_ns_hi << 32) | P.timeout_ns_lo);
  stamp<kTiming>(P, blockIdx.x, EV_START);
  compute_main<kTiming, kDraft>(w);
  stamp<kTiming>(P, blockIdx.x, EV_END);
  // the warp's tensor-memory accesses are done before the block frees it
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&cx.S.tcbar[TB_DONE], 1);
}

const void* layer_kernel(bool timing, bool draft) {
  if (draft)
    return timing ? reinterpret_cast<const void*>(&msm_layer_kernel<true, true>)
                  : reinterpret_cast<const void*>(&msm_layer_kernel<false, true>);
  return timing ? reinterpret_cast<const void*>(&msm_layer_kernel<true, false>)
                : reinterpret_cast<const void*>(&msm_layer_kernel<false, false>);
}

}  // namespace msm
