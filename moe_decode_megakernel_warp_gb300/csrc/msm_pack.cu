// Weight packing kernels, run once at model creation, and the sentinel fill.
//
// Dense bf16 matrices W[N][K] become 16-row units; each unit holds its K columns as
// tiles of 64 k-steps of 16 columns (the last tile of a unit may be shorter), laid out
// for the tensor-memory copy the dense phases read them through: the m16n8k16 A
// fragment of k-step 4c + q of a tile, as thread t of a warp holds it (four words:
// rows t/4 and t/4 + 8, columns 2(t%4) and 2(t%4) + 8 of the k-step), sits at byte
// c * 2048 + (32 q + t) * 16 of the tile.  A 128x256b tensor-memory copy of chunks c,
// c + 1 (core matrices 8 rows x 16 bytes, 2048 bytes apart along K, 128 along the rows)
// puts it in lane 32 q + t, columns 4c .. 4c + 3, so warp q of a group reads its k-steps
// q, q + 4, ... with one tcgen05.ld, and a shorter tile is a prefix of the layout.
// Two matrices get their rows paired inside a unit so an
// epilogue thread holds both halves of a pair: the q/k rows of a head as
// (d, d + hd/2) for rotate-half RoPE, and a dense FFN's stacked [gate; up] as
// (gate j, up j) for SwiGLU.
//
// NVFP4 expert matrices become 128-row units of 512-column tiles (256 where the width is
// not a multiple of 512): column blocks of 128 rows x 128 code bytes in the 128-byte
// swizzle layout the tensor cores read, then the block scales grouped per K=64 step (the
// scale word of row m at (m % 32) * 16 + (m / 32) * 4 of its 512-byte group: 128 threads
// read a step's words with 4-way bank conflicts at most).  W1 units hold 64 gate rows and
// the 64 matching up
// rows, interleaved (gate j, up j, gate j + 1, ...), so neighbouring lanes of the SwiGLU
// epilogue hold the two halves of an output.
#include "msm_device.cuh"
#include "msm_internal.h"

namespace msm {

// row of the source matrix held by row `r` (0..15) of unit `u` (N: the packed rows)
__device__ __forceinline__ int dense_src_row(int kind, int u, int r, int N, int hd, int hq, int hkv) {
  if (kind == 2)  // [gate; up] stacked: rows 0-7 gate rows 8u.., rows 8-15 the matching up rows
    return (r < 8) ? u * 8 + r : N / 2 + u * 8 + (r - 8);
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

// one thread per fragment word (unit, k-step, thread t, word j): word j of the fragment
// is rows (j & 1) * 8 + t / 4, columns (j >> 1) * 8 + 2 (t % 4) (+1) of the k-step
__global__ void pack_dense_kernel(const uint16_t* __restrict__ W, uint8_t* __restrict__ out, int N, int K,
                                  int kind, int hd, int hq, int hkv) {
  const long long steps = K / 16;
  const long long total = (long long)(N / 16) * steps * 128;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(c & 3), t = (int)((c >> 2) & 31);
    const long long ks = (c >> 7) % steps, u = (c >> 7) / steps;
    const int ur = (j & 1) * 8 + t / 4;
    const int kcol = (int)ks * 16 + (j >> 1) * 8 + 2 * (t % 4);
    const int src = dense_src_row(kind, (int)u, ur, N, hd, hq, hkv);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(W + (size_t)src * K + kcol);
    const long long kt = ks / kDenseTileSteps, kin = ks % kDenseTileSteps;
    const long long off = ((long long)u * steps + kt * kDenseTileSteps) * kKStepBytes + (kin >> 2) * 2048 +
                          ((kin & 3) * 32 + t) * 16 + j * 4;
    *reinterpret_cast<uint32_t*>(out + off) = v;
  }
}

// one thread per (expert, unit, k-tile, row): the row's code bytes of the tile go to row m
// of each 16 KB column block with 16-byte chunk c at chunk c ^ (m & 7) (the 128-byte
// swizzle of a K-major tensor-core operand), its block scales to byte (m % 32) * 16 +
// (m / 32) * 4 + b % 4 of the tile's scale group b / 4
__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                  uint8_t* __restrict__ out, int E, int rows, int K, int swiglu, int F) {
  const int units = swiglu ? w1_units(F) : w2_units(rows);
  const int tk = exp_tile_k(K), nt = K / tk, nkb = tk / kExpBlockK;
  const long long total = (long long)E * units * nt * kExpTileRows;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(c % kExpTileRows);
    const long long rest = c / kExpTileRows;
    const int kt = (int)(rest % nt);
    const long long eu = rest / nt;
    const int u = (int)(eu % units), e = (int)(eu / units);
    const int R = swiglu ? ((m & 1) ? F : 0) + u * 64 + (m >> 1) : u * kExpTileRows + m;
    const uint4* crow = reinterpret_cast<const uint4*>(codes + ((size_t)e * rows + R) * (K / 2) + (size_t)kt * (tk / 2));
    const uint8_t* srow = sf + ((size_t)e * rows + R) * (K / 16) + (size_t)kt * (tk / 16);
    uint8_t* tile = out + ((size_t)eu * nt + kt) * exp_tile_bytes(K);
    for (int kb = 0; kb < nkb; ++kb)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(tile + kb * kExpBlockBytes + m * 128 + ((ch ^ (m & 7)) << 4)) = crow[kb * 8 + ch];
    for (int b = 0; b < tk / 16; ++b)
      tile[exp_scale_off(K) + (b >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (b & 3)] = srow[b];
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
