// Device implementation of the synthetic input generator: the same element
// definitions as synth.c (synth_defs.h), run as CUDA kernels so the 62-layer
// workload (about 64 GB of weights) is drawn straight into device memory.
// Bit-identical to the host generator.  Input preparation only; compile with
// -fmad=false.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_defs.h"

namespace {

__global__ void normal_bf16_kernel(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std,
                                   uint16_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = synth_bf16_rne(synth_value(seed, stream, i, mean, std));
}

__global__ void normal_f32_kernel(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, float* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = (float)synth_value(seed, stream, i, mean, std);
}

// per-expert |max| of the fp32 values (non-negative floats order like their bits)
__global__ void amax_kernel(uint64_t seed, uint64_t base_stream, uint64_t per, double std, unsigned int* amax_bits) {
  const int e = blockIdx.y;
  const uint64_t stream = base_stream | ((uint64_t)(uint16_t)e << 16);
  float m = 0.f;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < per; i += (uint64_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf((float)synth_value(seed, stream, i, 0.0, std)));
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + e, __float_as_uint(m));
}

// one thread per (expert, row, 16-column block); same encoding steps as synth.c
__global__ void encode_kernel(uint64_t seed, uint64_t base_stream, int E, int64_t rows, int64_t cols, double std,
                              const unsigned int* amax_bits, uint8_t* codes, uint8_t* sf, float* gs) {
  const int64_t nb = cols / 16;
  const int64_t total = (int64_t)E * rows * nb;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = t % nb, r = (t / nb) % rows;
    const int e = (int)(t / (nb * rows));
    const uint64_t stream = base_stream | ((uint64_t)(uint16_t)e << 16);
    const float amax = __uint_as_float(amax_bits[e]);
    const float ts = amax / (6.0f * 448.0f);
    if (r == 0 && b == 0) gs[e] = ts;
    float x[16];
    float bmax = 0.0f;
    for (int j = 0; j < 16; ++j) {
      x[j] = (float)synth_value(seed, stream, (uint64_t)(r * cols + b * 16 + j), 0.0, std);
      bmax = fmaxf(bmax, fabsf(x[j]));
    }
    const uint8_t s = (ts > 0.0f) ? synth_e4m3_rne(bmax / (6.0f * ts)) : 0;
    const size_t row_off = ((size_t)e * rows + r);
    sf[row_off * nb + b] = s;
    const float denom = synth_e4m3_value(s) * ts;
    for (int j = 0; j < 16; j += 2) {
      uint8_t c0 = 0, c1 = 0;
      if (s != 0) {
        c0 = synth_e2m1_rne(x[j] / denom);
        c1 = synth_e2m1_rne(x[j + 1] / denom);
      }
      codes[(row_off * cols + b * 16 + j) / 2] = (uint8_t)(c0 | (c1 << 4));
    }
  }
}

int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  return (int)(g > 65535 * 4 ? 65535 * 4 : (g ? g : 1));
}

}  // namespace

extern "C" {

int synth_gpu_normal_bf16(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, void* dst,
                          void* cuda_stream) {
  if (n == 0) return 0;
  normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(seed, stream, n, mean, std,
                                                                         (uint16_t*)dst);
  return (int)cudaGetLastError();
}

int synth_gpu_normal_f32(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, void* dst,
                         void* cuda_stream) {
  if (n == 0) return 0;
  normal_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(seed, stream, n, mean, std, (float*)dst);
  return (int)cudaGetLastError();
}

// E matrices [rows][cols] of N(0, std^2), expert e drawn from stream base_stream | (e << 16),
// each NVFP4-encoded with its own tensor scale. scratch: E unsigned ints of device memory.
int synth_gpu_nvfp4_experts(uint64_t seed, uint64_t base_stream, int E, int64_t rows, int64_t cols, double std,
                            void* codes, void* sf, void* gs, void* scratch, void* cuda_stream) {
  cudaStream_t s = (cudaStream_t)cuda_stream;
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(unsigned int) * E, s);
  if (e != cudaSuccess) return (int)e;
  const uint64_t per = (uint64_t)rows * cols;
  dim3 g1(64, E);
  amax_kernel<<<g1, 256, 0, s>>>(seed, base_stream, per, std, (unsigned int*)scratch);
  const uint64_t total = (uint64_t)E * rows * (cols / 16);
  encode_kernel<<<grid_for(total), 256, 0, s>>>(seed, base_stream, E, rows, cols, std, (const unsigned int*)scratch,
                                                (uint8_t*)codes, (uint8_t*)sf, (float*)gs);
  return (int)cudaGetLastError();
}

}  // extern "C"
