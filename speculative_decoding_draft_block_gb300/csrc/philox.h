// Philox4x32-10 counter-based generator, host and device.
//
// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): ten rounds; each multiplies counter words 0 and 2 by two round
// constants, swaps the high/low halves into place with words 1 and 3 and the
// key, and bumps the key by a Weyl increment between rounds.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define DS_HD __host__ __device__ __forceinline__
#else
#define DS_HD inline
#endif

namespace ds {

struct Philox4 {
  uint32_t v[4];
};

DS_HD uint32_t mulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return (uint32_t)(((uint64_t)a * (uint64_t)b) >> 32);
#endif
}

DS_HD Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                            uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint32_t hi0 = mulhi32(M0, c0), lo0 = M0 * c0;
    const uint32_t hi1 = mulhi32(M1, c2), lo1 = M1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  Philox4 r;
  r.v[0] = c0;
  r.v[1] = c1;
  r.v[2] = c2;
  r.v[3] = c3;
  return r;
}

// Word 0 of the stream keyed by (seed) at counter (request, position, stage, 0).
DS_HD uint32_t philox_word(uint64_t seed, uint32_t request, uint32_t position, uint32_t stage) {
  return philox4x32_10(request, position, stage, 0u, (uint32_t)(seed & 0xffffffffu),
                       (uint32_t)(seed >> 32))
      .v[0];
}

// u = (w + 1/2) * 2^-32, exact in double, strictly inside (0, 1).
DS_HD double uniform_from_word(uint32_t w) { return ((double)w + 0.5) * (1.0 / 4294967296.0); }

}  // namespace ds
