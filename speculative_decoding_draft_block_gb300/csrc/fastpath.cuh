// Fast path for the per-token weights of bf16 logits (the draft hot loop).
//
// For a bf16 logit z (8 significant bits) and g = log2(e)/T split as
// g = G + gl with G truncated to 16 significant bits, a = z*G is exact in fp32.
// With t = (z + b)*g = a + (b*g + z*gl), the bias term uses g rounded to fp32
// (its own rounding is far below the tolerance) and z*gl is folded in by FMA:
//
//   k = rint(a) via the 1.5*2^23 rounding constant, d = a - k (exact),
//   f = d + (b*g + z*gl),  p = 2^f (ex2.approx),  w = p * 2^(k - ref),
//
// the last factor applied to p's exponent field. The chunk reference ref is
// rint(max_j z_j * G). The path is taken only when every z of the chunk is
// finite and spans less than 96 / G (so 2^(k - ref) stays a normal number);
// otherwise the general path of common.cuh is used.
//
// Chunk sums on this path are exact up to ~2^-36 relative: each weight is split
// on a fixed 2^-15 grid, w = w_hi + w_lo with w_hi = (w + 384) - 384 (exact),
// the w_hi are summed exactly (multiples of 2^-15 below 512) and the small w_lo
// separately. The caller checks that the high sum stayed below 512.
//
// Two tokens are processed per instruction with the packed .f32x2 operations
// (IEEE round-to-nearest per lane, so a scalar evaluation gives identical bits).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace ds {

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kGrid = 384.0f;        // 1.5 * 2^8: ulp 2^-15 on [256, 512)
constexpr float kFastSpan = 96.0f;     // max (zmax - zmin) * G on the fast path
constexpr float kFastHiLimit = 511.0f;

struct G16 {
  float G, gl, gf;  // g = G + gl exactly to ~2^-40; gf = g rounded to fp32
};

__device__ __forceinline__ G16 make_g16(float T) {
  const Gscale g = make_gscale(T);
  const float G = __uint_as_float(__float_as_uint(g.hi) & 0xFFFFFF00u);
  return {G, __fadd_rn(__fsub_rn(g.hi, G), g.lo), g.hi};  // g.hi - G is exact
}

// Scalar weight, bit-identical to one lane of fast_w2.
__device__ __forceinline__ float fast_w1(float z, float b, G16 g, uint32_t ref23) {
  const float a = __fmul_rn(z, g.G);
  const float t = __fmul_rn(b, g.gf);
  const float tl = __fmaf_rn(z, g.gl, t);
  const float m = __fadd_rn(a, kMagic);
  const float kf = __fadd_rn(m, -kMagic);
  const float d = __fmaf_rn(kf, -1.0f, a);
  const float f = __fadd_rn(d, tl);
  const float p = ex2_approx(f);
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(m) << 23) - ref23);
}

struct FastConsts {
  float G, gl, gf;
  uint32_t ref23;
};

__device__ __forceinline__ FastConsts make_fast_consts(G16 g, int ref) {
  return {g.G, g.gl, g.gf, (uint32_t)ref << 23};
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Weights of the two tokens packed in zw, accumulated into (shi, slo).
__device__ __forceinline__ void fast_pair(uint32_t zw, float b0, float b1, const FastConsts& k,
                                          float2& shi, float2& slo) {
  const float2 z2 = unpack_bf16x2(zw);
  const float2 a2 = __fmul2_rn(z2, make_float2(k.G, k.G));
  const float2 t2 = __fmul2_rn(make_float2(b0, b1), make_float2(k.gf, k.gf));
  const float2 tl2 = __ffma2_rn(z2, make_float2(k.gl, k.gl), t2);
  const float2 m2 = __fadd2_rn(a2, make_float2(kMagic, kMagic));
  const float2 kf2 = __fadd2_rn(m2, make_float2(-kMagic, -kMagic));
  const float2 d2 = __ffma2_rn(kf2, make_float2(-1.0f, -1.0f), a2);
  const float2 f2 = __fadd2_rn(d2, tl2);
  const float p0 = ex2_approx(f2.x), p1 = ex2_approx(f2.y);
  const float2 w2 =
      make_float2(__uint_as_float(__float_as_uint(p0) + (__float_as_uint(m2.x) << 23) - k.ref23),
                  __uint_as_float(__float_as_uint(p1) + (__float_as_uint(m2.y) << 23) - k.ref23));
  const float2 tt = __fadd2_rn(w2, make_float2(kGrid, kGrid));
  const float2 wh = __fadd2_rn(tt, make_float2(-kGrid, -kGrid));
  const float2 wl = __ffma2_rn(wh, make_float2(-1.0f, -1.0f), w2);
  shi = __fadd2_rn(shi, wh);
  slo = __fadd2_rn(slo, wl);
}

// Scalar split of one weight on the same grid (for prefix sums in the locate).
__device__ __forceinline__ void fast_split(float w, float& wh, float& wl) {
  const float tt = __fadd_rn(w, kGrid);
  wh = __fadd_rn(tt, -kGrid);
  wl = __fmaf_rn(wh, -1.0f, w);
}

// Chunk predicate and reference from the packed bf16 logits of 32 tokens.
__device__ __forceinline__ bool fast_chunk_ok(const uint32_t* zp, G16 g, int& ref) {
  __nv_bfloat162 mx = *reinterpret_cast<const __nv_bfloat162*>(&zp[0]);
  __nv_bfloat162 mn = mx;
#pragma unroll
  for (int i = 1; i < 16; ++i) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&zp[i]);
    mx = __hmax2(mx, v);
    mn = __hmin2(mn, v);
  }
  const float zmax = fmaxf(__low2float(mx), __high2float(mx));
  const float zmin = fminf(__low2float(mn), __high2float(mn));
  const bool ok = (zmin > kNegInf) && ((zmax - zmin) * g.G < kFastSpan) &&
                  (fabsf(zmax * g.G) < 4.0e6f);
  ref = ok ? (int)rintf(__fmul_rn(zmax, g.G)) : 0;
  return ok;
}

}  // namespace ds
