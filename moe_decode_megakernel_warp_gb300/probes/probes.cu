// Intra-GPU microbenchmarks behind the layer kernel's design choices, on one GPU:
//
//   poll     GPU-scope acquire load: the latency of one (a dependent chain, no
//            writer); and a flag handed between two blocks on different SMs (release
//            store, acquire poll), one-way latency = elapsed / round trips / 2,
//            idle and with bulk copies (cp.async.bulk) in flight on both SMs.
//   fence    cost of one gpu-scope fence (fence.acq_rel.gpu) issued by one thread:
//            idle, right after the block stored 64 KB, and while bulk copies are in
//            flight into the block's shared memory.
//   icache   per-pass time of straight-line code blocks run in a loop: a ~100 KB
//            block alone, two ~100 KB blocks back to back, and a ~100 KB block
//            followed by a ~20 KB one.
//   handoff  grid-wide handoff of a [16][K] bf16 activation: 128 producer blocks
//            store it with 2-byte stores, all 152 blocks stage it into shared
//            memory, either polling every element's all-ones sentinel or waiting
//            on one counter that producers bump after a fence.
//
// The pages report these costs for GB300 (orcarouter.ai, "Muse Spark Open: 1,109
// tokens/s is a kernel-level change", § on the three costs of a megakernel:
// instruction cache, weight prefetch, synchronisation; alphasignal.ai, "LMSYS
// Doubles Muse Spark Open Speed to 1,109 Tokens per Second", § "Four mechanisms
// keep work moving"). Every wait below is bounded; a wait that runs out sets an
// error flag that the host reports.
//
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 probes.cu
// Usage: probes [poll|fence|icache|handoff|all] [--quick]  (one JSON line per result)
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

namespace {

constexpr uint32_t kSpinLimit = 1u << 22;  // polls before a wait gives up

__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t ph) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok)
               : "r"(su32(b)), "r"(ph)
               : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t n, uint64_t* b) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
               "l"(src), "r"(n), "r"(su32(b))
               : "memory");
}
__device__ bool mb_wait(uint64_t* b, uint32_t ph, int* err) {
  for (uint32_t n = 0; n < kSpinLimit; ++n)
    if (mb_try(b, ph)) return true;
  atomicExch(err, 1);
  return false;
}

// Warp 1 of a block keeps `rounds` rounds of 4 bulk copies of 16 KB in flight into the
// block's shared memory (two buffers) until *stop is set or the rounds run out.
__device__ void copy_loop(const uint8_t* src, uint8_t* sm, uint64_t* bars, int rounds, const volatile int* stop,
                          int* err) {
  if ((threadIdx.x & 31) != 0) return;
  int issued = 0;
  for (int r = 0; r < rounds && !*stop; ++r) {
    uint64_t* b = &bars[r & 1];
    if (r >= 2 && !mb_wait(b, ((r >> 1) - 1) & 1, err)) return;
    mb_expect(b, 4 * 16384);
    for (int i = 0; i < 4; ++i)
      bulk_load(sm + (r & 1) * 65536 + i * 16384, src + ((size_t)(r * 4 + i) % 256) * 16384, 16384, b);
    issued = r + 1;
  }
  // drain: the last rounds issued complete before the block exits
  for (int r = max(0, issued - 2); r < issued; ++r) mb_wait(&bars[r & 1], (r >> 1) & 1, err);
}

// ---- poll ---------------------------------------------------------------------------
__global__ void __launch_bounds__(64, 1) poll_kernel(uint32_t* flags, int iters, int with_copies, const uint8_t* src,
                                                     unsigned long long* out, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bars[2];
  __shared__ volatile int stop;
  const int b = blockIdx.x, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mb_init(&bars[0], 1);
    mb_init(&bars[1], 1);
    stop = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 1) {
    if (with_copies) copy_loop(src, sm, bars, 1 << 20, &stop, err);
    return;
  }
  if (threadIdx.x != 0) return;
  uint32_t* mine = flags + b * 32;        // flag this block waits on
  uint32_t* other = flags + (1 - b) * 32;  // flag the other block waits on
  const uint64_t t0 = gtime();
  for (int i = 1; i <= iters; ++i) {
    if (b == 0) st_release(other, i);
    uint32_t n = 0;
    while (ld_acquire(mine) != (uint32_t)i) {
      if (++n > kSpinLimit) {
        atomicExch(err, 1);
        stop = 1;
        return;
      }
    }
    if (b == 1) st_release(other, i);
  }
  const uint64_t t1 = gtime();
  stop = 1;
  if (b == 0) out[0] = t1 - t0;
}

// latency of one GPU-scope acquire load (a dependent chain of them, no writer)
__global__ void __launch_bounds__(32, 1) load_latency_kernel(const uint32_t* zeros, int iters, unsigned long long* out) {
  if (threadIdx.x != 0) return;
  uint32_t v = 0;
  const uint64_t t0 = gtime();
  for (int i = 0; i < iters; ++i) v = ld_acquire(zeros + (v & 1u));  // the next address waits for this value
  const uint64_t t1 = gtime();
  out[0] = (t1 - t0) + (v == 12345u ? 1u : 0u);
}

// ---- fence --------------------------------------------------------------------------
// mode 0: idle; 1: after the block's threads stored 64 KB; 2: bulk copies in flight
__global__ void __launch_bounds__(64, 1) fence_kernel(uint32_t* scratch, int mode, int reps, const uint8_t* src,
                                                      unsigned long long* out, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bars[2];
  __shared__ volatile int stop;
  __shared__ volatile int ready;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mb_init(&bars[0], 1);
    mb_init(&bars[1], 1);
    stop = 0;
    ready = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 1) {
    if (mode == 2) {
      if (lane == 0) ready = 1;
      copy_loop(src, sm, bars, 1 << 20, &stop, err);
    }
    return;
  }
  uint64_t total = 0;
  for (int r = 0; r < reps; ++r) {
    if (mode == 1) {
      // 64 KB of stores from the warp, then the fence
      for (int i = lane; i < 16384; i += 32) scratch[(size_t)r * 16384 + i] = (uint32_t)(r + i);
      __syncwarp();
    }
    if (mode == 2 && lane == 0) {
      uint32_t n = 0;
      while (!ready && ++n < kSpinLimit) {
      }
      // let the copies get going
      const uint64_t until = gtime() + 2000;
      while (gtime() < until) {
      }
    }
    if (lane == 0) {
      const uint64_t t0 = gtime();
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      const uint64_t t1 = gtime();
      total += t1 - t0;
    }
    __syncwarp();
  }
  if (lane == 0) {
    stop = 1;
    out[0] = total;
  }
}

// ---- icache -------------------------------------------------------------------------
// A straight-line block of independent FMAs: 8 chains, `n` instructions of 16 bytes.
#define FMA8                                                                                                      \
  asm volatile(                                                                                                   \
      "fma.rn.f32 %0, %0, %8, %9; fma.rn.f32 %1, %1, %8, %9; fma.rn.f32 %2, %2, %8, %9; fma.rn.f32 %3, %3, %8, %9;" \
      "fma.rn.f32 %4, %4, %8, %9; fma.rn.f32 %5, %5, %8, %9; fma.rn.f32 %6, %6, %8, %9; fma.rn.f32 %7, %7, %8, %9;" \
      : "+f"(x0), "+f"(x1), "+f"(x2), "+f"(x3), "+f"(x4), "+f"(x5), "+f"(x6), "+f"(x7)                           \
      : "f"(a), "f"(c));
#define FMA64 FMA8 FMA8 FMA8 FMA8 FMA8 FMA8 FMA8 FMA8
#define FMA512 FMA64 FMA64 FMA64 FMA64 FMA64 FMA64 FMA64 FMA64
#define FMA1024 FMA512 FMA512

template <int K1024>  // ~16 KB of code per unit
__device__ __noinline__ float code_block(float a, float c, float s) {
  float x0 = s, x1 = s + 1.f, x2 = s + 2.f, x3 = s + 3.f, x4 = s + 4.f, x5 = s + 5.f, x6 = s + 6.f, x7 = s + 7.f;
#pragma unroll
  for (int k = 0; k < K1024; ++k) {
    FMA1024
  }
  return ((x0 + x1) + (x2 + x3)) + ((x4 + x5) + (x6 + x7));
}
// A second straight-line block (a distinct function, so its code is distinct);
// code_block<6> is about 96 KB of machine code, code_block2<1> about 16 KB.
template <int K1024>
__device__ __noinline__ float code_block2(float a, float c, float s) {
  float x0 = s, x1 = s + 1.f, x2 = s + 2.f, x3 = s + 3.f, x4 = s + 4.f, x5 = s + 5.f, x6 = s + 6.f, x7 = s + 7.f;
#pragma unroll
  for (int k = 0; k < K1024; ++k) {
    FMA1024
  }
  return ((x0 + x1) + (x2 + x3)) - ((x4 + x5) + (x6 + x7));
}
// passes of block A (KA x 16 KB), then block B (KB x 16 KB) if KB > 0
template <int KA, int KB>
__global__ void __launch_bounds__(32, 1) icache2_kernel(int passes, float a, float c, float* out,
                                                        unsigned long long* t) {
  float s = (float)threadIdx.x;
  const uint64_t t0 = gtime();
  for (int p = 0; p < passes; ++p) {
    s = code_block<KA>(a, c, s);
    if (KB > 0) s = code_block2<KB>(a, c, s);
  }
  const uint64_t t1 = gtime();
  out[threadIdx.x] = s;
  if (threadIdx.x == 0) t[0] = t1 - t0;
}

// ---- handoff ------------------------------------------------------------------------
constexpr int kT = 16;
__device__ __forceinline__ uint4 ldr(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st16(uint16_t* p, uint16_t v) {
  asm volatile("st.relaxed.gpu.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}
__device__ __forceinline__ bool ready8(const uint4& x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) ok &= ((w[i] & 0xFFFFu) != 0xFFFFu) && ((w[i] >> 16) != 0xFFFFu);
  return ok;
}
// counter = 0: poll every element's sentinel; else wait on *counter >= producers
__global__ void __launch_bounds__(256, 1) handoff_kernel(uint16_t* buf, int K, unsigned* counter, unsigned producers,
                                                         unsigned long long* tm, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  const int tid = threadIdx.x, b = blockIdx.x;
  __syncthreads();
  const uint64_t t_enter = gtime();
  if (b < K / 16 && tid < 128) {
    const int p = tid >> 4, t = tid & 15;
    const uint64_t until = t_enter + 200 * (b % 11);  // a little skew between producers
    while (gtime() < until) {
    }
    for (int u = b; u < K / 16; u += gridDim.x) {
      st16(buf + (size_t)t * K + u * 16 + p, (uint16_t)(0x3F80 + p));
      st16(buf + (size_t)t * K + u * 16 + p + 8, (uint16_t)(0x3F80 + p + 8));
    }
  }
  if (counter) {
    __syncthreads();
    if (b < K / 16 && tid == 0) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
    }
  }
  const uint64_t t_prod = gtime();
  const int nch = kT * K / 8;
  if (!counter) {
    for (int c0 = tid; c0 < nch; c0 += 256 * 16) {
      uint4 v[16];
      uint32_t pending = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + 256 * j < nch) {
          pending |= 1u << j;
          v[j] = ldr(reinterpret_cast<const uint8_t*>(buf) + (size_t)(c0 + 256 * j) * 16);
        }
      for (uint32_t n = 0;; ++n) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (((pending >> j) & 1u) && ready8(v[j])) pending &= ~(1u << j);
        if (!pending) break;
        if (n > (1u << 20)) {
          atomicExch(err, 1);
          break;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if ((pending >> j) & 1u) v[j] = ldr(reinterpret_cast<const uint8_t*>(buf) + (size_t)(c0 + 256 * j) * 16);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + 256 * j < nch) *reinterpret_cast<uint4*>(sm + (size_t)(c0 + 256 * j) * 16) = v[j];
    }
  } else {
    if (tid == 0) {
      uint32_t n = 0;
      while (ld_acquire(counter) < producers) {
        if (++n > (1u << 20)) {
          atomicExch(err, 1);
          break;
        }
      }
    }
    __syncthreads();
    for (int c0 = tid; c0 < nch; c0 += 256 * 16) {
      uint4 v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + 256 * j < nch) v[j] = ldr(reinterpret_cast<const uint8_t*>(buf) + (size_t)(c0 + 256 * j) * 16);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + 256 * j < nch) *reinterpret_cast<uint4*>(sm + (size_t)(c0 + 256 * j) * 16) = v[j];
    }
  }
  __syncthreads();
  const uint64_t t_done = gtime();
  if (tid == 0) {
    tm[b * 3 + 0] = t_enter;
    tm[b * 3 + 1] = t_prod;
    tm[b * 3 + 2] = t_done;
  }
}

// ---- host ---------------------------------------------------------------------------
#define CK(x)                                                                          \
  do {                                                                                 \
    cudaError_t e_ = (x);                                                              \
    if (e_ != cudaSuccess) {                                                           \
      std::fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
      std::exit(2);                                                                    \
    }                                                                                  \
  } while (0)

double median(std::vector<double> v) {
  std::sort(v.begin(), v.end());
  return v[v.size() / 2];
}

struct Dev {
  uint8_t* src = nullptr;  // 4 MB of copy source
  unsigned long long* out = nullptr;
  int* err = nullptr;
  Dev() {
    CK(cudaMalloc(&src, 256 * 16384));
    CK(cudaMemset(src, 1, 256 * 16384));
    CK(cudaMalloc(&out, 4096 * 8));
    CK(cudaMalloc(&err, 4));
    CK(cudaMemset(err, 0, 4));
  }
  int error() {
    int e = 0;
    CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
    return e;
  }
};

void probe_poll(Dev& d, bool quick) {
  uint32_t* flags;
  CK(cudaMalloc(&flags, 64 * 4));
  {
    CK(cudaMemset(flags, 0, 64 * 4));
    const int iters = quick ? 2000 : 20000;
    std::vector<double> ns;
    for (int rep = 0; rep < 5; ++rep) {
      load_latency_kernel<<<1, 32>>>(flags, iters, d.out);
      CK(cudaDeviceSynchronize());
      unsigned long long t;
      CK(cudaMemcpy(&t, d.out, 8, cudaMemcpyDeviceToHost));
      ns.push_back((double)t / iters);
    }
    std::printf("{\"probe\": \"acquire_load\", \"ns_per_load\": %.1f, \"loads\": %d, \"error\": %d}\n", median(ns), iters,
                d.error());
  }
  CK(cudaFuncSetAttribute(poll_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 131072));
  const int iters = quick ? 2000 : 20000;
  for (int wc = 0; wc < 2; ++wc) {
    std::vector<double> ns;
    for (int rep = 0; rep < (quick ? 3 : 7); ++rep) {
      CK(cudaMemset(flags, 0, 64 * 4));
      // 2 blocks of 64 threads; 128 KB of shared memory keeps them on different SMs
      poll_kernel<<<2, 64, 131072>>>(flags, iters, wc, d.src, d.out, d.err);
      CK(cudaDeviceSynchronize());
      unsigned long long t;
      CK(cudaMemcpy(&t, d.out, 8, cudaMemcpyDeviceToHost));
      ns.push_back((double)t / iters / 2.0);
    }
    std::printf("{\"probe\": \"poll\", \"bulk_copies_in_flight\": %s, \"one_way_ns\": %.1f, \"round_trips\": %d, \"error\": %d}\n",
                wc ? "true" : "false", median(ns), iters, d.error());
  }
  CK(cudaFree(flags));
}

void probe_fence(Dev& d, bool quick) {
  uint32_t* scratch;
  const int reps = quick ? 20 : 200;
  CK(cudaMalloc(&scratch, (size_t)reps * 65536));
  CK(cudaFuncSetAttribute(fence_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 131072));
  const char* names[3] = {"idle", "after_64KB_of_stores", "bulk_copies_in_flight"};
  for (int mode = 0; mode < 3; ++mode) {
    fence_kernel<<<1, 64, 131072>>>(scratch, mode, reps, d.src, d.out, d.err);
    CK(cudaDeviceSynchronize());
    unsigned long long t;
    CK(cudaMemcpy(&t, d.out, 8, cudaMemcpyDeviceToHost));
    std::printf("{\"probe\": \"fence\", \"case\": \"%s\", \"ns_per_fence\": %.1f, \"reps\": %d, \"error\": %d}\n", names[mode],
                (double)t / reps, reps, d.error());
  }
  CK(cudaFree(scratch));
}

template <typename Kern>
double time_icache(Kern k, int passes, float* out, unsigned long long* t) {
  k<<<1, 32>>>(passes, 1.0000001f, 1e-7f, out, t);  // warm (first-launch code load)
  CK(cudaDeviceSynchronize());
  std::vector<double> us;
  for (int r = 0; r < 5; ++r) {
    k<<<1, 32>>>(passes, 1.0000001f, 1e-7f, out, t);
    CK(cudaDeviceSynchronize());
    unsigned long long v;
    CK(cudaMemcpy(&v, t, 8, cudaMemcpyDeviceToHost));
    us.push_back((double)v / 1000.0 / passes);
  }
  return median(us);
}

void probe_icache(Dev& d, bool quick) {
  float* out;
  CK(cudaMalloc(&out, 32 * 4));
  const int passes = quick ? 20 : 200;
  const double a = time_icache(icache2_kernel<6, 0>, passes, out, d.out);
  const double aa = time_icache(icache2_kernel<6, 6>, passes, out, d.out);
  const double ab = time_icache(icache2_kernel<6, 1>, passes, out, d.out);
  std::printf("{\"probe\": \"icache\", \"block_kb\": 96, \"alone_us_per_pass\": %.2f, \"two_96kb_blocks_us_per_pass\": %.2f, "
              "\"96kb_plus_16kb_us_per_pass\": %.2f, \"passes\": %d, \"error\": %d}\n",
              a, aa, ab, passes, d.error());
  CK(cudaFree(out));
}

void probe_handoff(Dev& d, bool quick) {
  const int G = 152;
  for (int K : {2048, 4096}) {
    uint16_t* buf;
    unsigned* counter;
    unsigned long long* tm;
    CK(cudaMalloc(&buf, (size_t)kT * K * 2));
    CK(cudaMalloc(&counter, 4));
    CK(cudaMalloc(&tm, G * 3 * 8));
    CK(cudaFuncSetAttribute(handoff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024));
    const unsigned producers = (unsigned)std::min(K / 16, G);
    for (int mode = 0; mode < 2; ++mode) {
      std::vector<double> first, last;
      for (int it = 0; it < (quick ? 6 : 25); ++it) {
        CK(cudaMemset(buf, 0xFF, (size_t)kT * K * 2));
        CK(cudaMemset(counter, 0, 4));
        handoff_kernel<<<G, 256, 160 * 1024>>>(buf, K, mode ? counter : nullptr, producers, tm, d.err);
        CK(cudaDeviceSynchronize());
        std::vector<unsigned long long> h(G * 3);
        CK(cudaMemcpy(h.data(), tm, h.size() * 8, cudaMemcpyDeviceToHost));
        unsigned long long pmax = 0, dmin = ~0ull, dmax = 0;
        for (int b = 0; b < G; ++b) {
          if (b < K / 16) pmax = std::max(pmax, h[b * 3 + 1]);
          dmin = std::min(dmin, h[b * 3 + 2]);
          dmax = std::max(dmax, h[b * 3 + 2]);
        }
        if (it >= 1) {
          first.push_back(((double)dmin - (double)pmax) / 1000.0);
          last.push_back(((double)dmax - (double)pmax) / 1000.0);
        }
      }
      std::printf("{\"probe\": \"handoff\", \"K\": %d, \"mode\": \"%s\", \"first_consumer_us_after_last_producer\": %.2f, "
                  "\"last_consumer_us_after_last_producer\": %.2f, \"error\": %d}\n",
                  K, mode ? "counter" : "poll_data", median(first), median(last), d.error());
    }
    CK(cudaFree(buf));
    CK(cudaFree(counter));
    CK(cudaFree(tm));
  }
}

// Clusters: how many clusters of 1, 2, 4 and 8 blocks of the layer kernel's shape (384
// threads, 227 KB of dynamic shared memory, one block per SM) can be resident at once.
// A query only: nothing is launched.
__global__ void __launch_bounds__(384, 1) cluster_shape_kernel(int* p) {
  if (p != nullptr && threadIdx.x == 0) p[blockIdx.x] = 1;
}

void probe_clusters() {
  const int smem = 232448;
  CK(cudaFuncSetAttribute(cluster_shape_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  CK(cudaFuncSetAttribute(cluster_shape_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
  for (int cs : {1, 2, 4, 8}) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs * 16);
    cfg.blockDim = dim3(384);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    CK(cudaOccupancyMaxActiveClusters(&n, cluster_shape_kernel, &cfg));
    std::printf("{\"probe\": \"clusters\", \"cluster_size\": %d, \"max_active_clusters\": %d, \"blocks\": %d, "
                "\"error\": 0}\n", cs, n, n * cs);
  }
}

}  // namespace

int main(int argc, char** argv) {
  const char* which = argc > 1 ? argv[1] : "all";
  bool quick = false;
  for (int i = 1; i < argc; ++i)
    if (!std::strcmp(argv[i], "--quick")) quick = true;
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  Dev d;
  const bool all = !std::strcmp(which, "all");
  if (all || !std::strcmp(which, "poll")) probe_poll(d, quick);
  if (all || !std::strcmp(which, "fence")) probe_fence(d, quick);
  if (all || !std::strcmp(which, "icache")) probe_icache(d, quick);
  if ((all || !std::strcmp(which, "handoff")) && sms >= 152) probe_handoff(d, quick);
  if (all || !std::strcmp(which, "clusters")) probe_clusters();
  return d.error() ? 1 : 0;
}
