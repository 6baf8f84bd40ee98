// Weight layout step: the token-major copy of the Markov projection.
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

}  // namespace

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
