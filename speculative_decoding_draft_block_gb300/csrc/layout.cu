// Weight layout steps: the token-major and the tile-packed copies of the Markov
// projection.
//
// DSpark summary page, 방법론 › 반자기회귀 생성: the Markov head's bias for
// token v is E[x] . P[:, v]. The tile kernels stream P row-major ([r][V]) into
// the tensor cores; the per-step draw refines 32 consecutive tokens, whose
// columns of P are r rows apart. P_t = P^T ([V][r]) puts those 32 x r weights
// in one contiguous block. It is made once per model (P is a weight).
//
// Plain tiled transpose through shared memory: a CTA moves a 64 (k) x 64 (v)
// tile; reads of P and writes of P_t are 64 consecutive elements per warp
// pair (coalesced), the padded tile keeps the transposed reads conflict-light.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ds {

namespace {

constexpr int kT = 64;

template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T* __restrict__ P, int32_t r, int32_t V,
                                                         T* __restrict__ Pt) {
  __shared__ T tile[kT][kT + 1];
  const int v0 = blockIdx.x * kT, k0 = blockIdx.y * kT;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4
  for (int i = ty; i < kT; i += 4) {
    const int k = k0 + i, v = v0 + tx;
    if (k < r && v < V) tile[i][tx] = P[(size_t)k * V + v];
  }
  __syncthreads();
  for (int i = ty; i < kT; i += 4) {
    const int v = v0 + i, k = k0 + tx;
    if (v < V && k < r) Pt[(size_t)v * r + k] = tile[tx][i];
  }
}

// Tile-packed copy of P for the tensor-core tile kernel: for each 128-token
// tile nt, its r x 128 slice of P in exactly the shared-memory image the MMA
// reads (64-row k-blocks c, each two 64-token halves h of 64 rows x 128 bytes,
// the 16-byte unit u of row m stored at unit u ^ (m & 7), the 128-byte
// swizzle), so that a stage of the tile arrives with one bulk copy instead of
// a tensor copy per row. Tokens past V are zero. One thread per 16-byte unit.
__global__ void __launch_bounds__(256) pack_kernel(const uint16_t* __restrict__ P, int32_t r, int32_t V,
                                                    int32_t n_nt, uint4* __restrict__ out) {
  const int nkb = r / 64;
  const size_t units = (size_t)n_nt * nkb * 1024;  // 16 KB = 1024 units per (tile, k-block)
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < units; q += (size_t)gridDim.x * blockDim.x) {
    const size_t blk = q >> 10;                    // (tile, k-block)
    const int nt = (int)(blk / nkb), c = (int)(blk - (size_t)nt * nkb);
    const int w = (int)(q & 1023);                 // destination unit within the 16 KB block
    const int h = w >> 9, m = (w >> 3) & 63, us = w & 7;
    const int u = us ^ (m & 7);                    // source unit stored at swizzled position us
    const int v0 = nt * 128 + h * 64 + u * 8;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (v0 < V) val = *reinterpret_cast<const uint4*>(P + (size_t)(c * 64 + m) * V + v0);
    out[q] = val;
  }
}

}  // namespace

size_t packed_projection_bytes(int32_t r, int32_t V) {
  return (size_t)((V + 127) / 128) * (size_t)(r / 64) * 16384u;
}

cudaError_t launch_pack_projection(const void* P, int32_t r, int32_t V, void* P_packed, cudaStream_t s) {
  const int n_nt = (V + 127) / 128;
  const size_t units = (size_t)n_nt * (r / 64) * 1024;
  const int blocks = (int)((units + 255) / 256 < 65535 * 8 ? (units + 255) / 256 : 65535 * 8);
  pack_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(P), r, V, n_nt, static_cast<uint4*>(P_packed));
  return cudaGetLastError();
}

cudaError_t launch_transpose(const void* P, int32_t r, int32_t V, int32_t dtype, void* P_t,
                             cudaStream_t s) {
  const dim3 grid((V + kT - 1) / kT, (r + kT - 1) / kT);
  if (dtype == DS_BF16)
    transpose_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(P), r, V,
                                                    static_cast<uint16_t*>(P_t));
  else
    transpose_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(P), r, V,
                                                 static_cast<float*>(P_t));
  return cudaGetLastError();
}

}  // namespace ds
