// Device evaluation of Philox4x32-10 (the kernels' copy), for checking it
// word for word against the host and the reference implementation.
#include <stdint.h>

#include "internal.h"
#include "philox.h"

namespace ds {

namespace {

__global__ void philox_fill_kernel(const uint4* ctr, uint32_t k0, uint32_t k1, uint4* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = ctr[i];
  const Philox4 r = philox4x32_10(c.x, c.y, c.z, c.w, k0, k1);
  out[i] = make_uint4(r.v[0], r.v[1], r.v[2], r.v[3]);
}

}  // namespace

cudaError_t launch_philox_fill(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out,
                               int32_t n, cudaStream_t s) {
  philox_fill_kernel<<<(n + 255) / 256, 256, 0, s>>>(reinterpret_cast<const uint4*>(ctr), k0, k1,
                                                     reinterpret_cast<uint4*>(out), n);
  return cudaGetLastError();
}

}  // namespace ds
