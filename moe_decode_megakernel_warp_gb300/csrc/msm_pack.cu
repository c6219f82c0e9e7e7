// Weight packing kernels, run once at model creation, and the sentinel fill.
//
// Dense bf16 matrices W[N][K] become 16-row units; each unit holds its K columns
// as k-steps of 16 columns, each k-step four 8x8 matrices in ldmatrix order
// (rows 0-7 | k 0-7, rows 8-15 | k 0-7, rows 0-7 | k 8-15, rows 8-15 | k 8-15),
// so one contiguous bulk copy brings a tile and one ldmatrix.x4 yields the
// m16n8k16 A fragment.  Two matrices get their rows paired inside a unit so an
// epilogue thread holds both halves of a pair: the q/k rows of a head as
// (d, d + hd/2) for rotate-half RoPE, and W1 as (gate j, up j) for SwiGLU.
//
// NVFP4 expert matrices become 16-row units of 64-column groups (576 bytes):
// 512 bytes of E2M1 codes ordered [row][quad q][k-step][2 bytes: the bytes
// holding columns 2q,2q+1 and 2q+8,2q+9], then 64 bytes of E4M3 scales
// [row][k-step], so each thread loads its A-fragment codes with one 8-byte load.
#include "msm_device.cuh"
#include "msm_internal.h"

namespace msm {

// row of the source matrix held by row `r` (0..15) of unit `u`
__device__ __forceinline__ int dense_src_row(int kind, int u, int r, int hd, int hq, int hkv) {
  if (kind == 1) {  // QKV with RoPE pairing
    const int upd = hd / 16, nQ = hq * upd, nK = hkv * upd;
    if (u < nQ + nK) {
      const bool isq = u < nQ;
      const int hu = isq ? u : u - nQ, h = hu / upd, j = hu % upd;
      const int dim = (r < 8) ? j * 8 + r : hd / 2 + j * 8 + (r - 8);
      return (isq ? 0 : hq * hd) + h * hd + dim;
    }
    return (hq + hkv) * hd + (u - nQ - nK) * 16 + r;
  }
  return u * 16 + r;
}

__global__ void pack_dense_kernel(const uint16_t* __restrict__ W, uint8_t* __restrict__ out, int N, int K,
                                  int kind, int hd, int hq, int hkv) {
  const long long steps = K / 16;
  const long long total = (long long)(N / 16) * steps * 32;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(c & 7), m = (int)((c >> 3) & 3);
    const long long ks = (c >> 5) % steps, u = (c >> 5) / steps;
    const int ur = (m & 1) * 8 + r;
    const int kcol = (int)ks * 16 + (m >> 1) * 8;
    const int src = dense_src_row(kind, (int)u, ur, hd, hq, hkv);
    const uint4 v = *reinterpret_cast<const uint4*>(W + (size_t)src * K + kcol);
    *reinterpret_cast<uint4*>(out + ((size_t)u * steps + ks) * kKStepBytes + m * 128 + r * 16) = v;
  }
}

// one thread per (expert, unit, group, row)
__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                  uint8_t* __restrict__ out, int E, int rows, int K, int swiglu, int F) {
  const int units = swiglu ? F / 8 : rows / 16;
  const int ng = K / 64;
  const long long total = (long long)E * units * ng * 16;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(c & 15);
    const long long rest = c >> 4;
    const int gi = (int)(rest % ng);
    const long long eu = rest / ng;
    const int u = (int)(eu % units), e = (int)(eu / units);
    const int R = swiglu ? ((r < 8) ? u * 8 + r : F + u * 8 + (r - 8)) : u * 16 + r;
    const uint8_t* crow = codes + ((size_t)e * rows + R) * (K / 2) + gi * 32;
    const uint8_t* srow = sf + ((size_t)e * rows + R) * (K / 16) + gi * 4;
    uint8_t* gout = out + ((size_t)eu * ng + gi) * kExpGroupBytes;
    uint8_t cb[32];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        cb[q * 8 + ks * 2 + 0] = crow[ks * 8 + q];
        cb[q * 8 + ks * 2 + 1] = crow[ks * 8 + q + 4];
      }
#pragma unroll
    for (int i = 0; i < 32; i += 16)
      *reinterpret_cast<uint4*>(gout + r * 32 + i) = *reinterpret_cast<const uint4*>(cb + i);
    *reinterpret_cast<uint32_t*>(gout + 512 + r * 4) =
        (uint32_t)srow[0] | ((uint32_t)srow[1] << 8) | ((uint32_t)srow[2] << 16) | ((uint32_t)srow[3] << 24);
  }
}

__global__ void fill_u32_kernel(uint32_t* p, uint64_t n, uint32_t v) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

cudaError_t launch_pack_dense(const void* W, void* out, int N, int K, int kind, int hd, int hq, int hkv,
                              cudaStream_t s) {
  pack_dense_kernel<<<1024, 256, 0, s>>>(static_cast<const uint16_t*>(W), static_cast<uint8_t*>(out), N, K,
                                         kind, hd, hq, hkv);
  return cudaGetLastError();
}
cudaError_t launch_pack_nvfp4(const void* codes, const void* sf, void* out, int E, int rows, int K, int swiglu,
                              int F, cudaStream_t s) {
  pack_nvfp4_kernel<<<1024, 256, 0, s>>>(static_cast<const uint8_t*>(codes), static_cast<const uint8_t*>(sf),
                                         static_cast<uint8_t*>(out), E, rows, K, swiglu, F);
  return cudaGetLastError();
}
cudaError_t launch_fill_u32(void* p, uint64_t n, uint32_t v, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  fill_u32_kernel<<<512, 256, 0, s>>>(static_cast<uint32_t*>(p), n, v);
  return cudaGetLastError();
}

}  // namespace msm
