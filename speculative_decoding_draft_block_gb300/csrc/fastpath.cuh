// Fast path for the per-token weights of bf16 logits (the draft hot loop).
//
// For a bf16 logit z (8 significant bits) and g = log2(e)/T split as
// g = G + gl with G truncated to 16 significant bits, a = z*G is exact in fp32.
// With t = (z + b)*g = a + z*gl + b*g and the chunk reference ref:
//
//   m = z*G + C with C = 1.5*2^23 - ref (one rounding: m = C + k, k an
//       integer within 1/2 of a), -k = C - m and d = a - k (both exact, FMA),
//   f = b*g + (z*gl + d),  p = 2^f (ex2.approx),
//   w = p * 2^(k - ref): the float bits of m hold 1.5*2^23 + (k - ref), so
//       bits(p) + (bits(m) << 23) adds k - ref to p's exponent field.
//
// The chunk reference is ref = rint(max_j z_j * G). The path is taken only
// when every z of the chunk is finite and spans less than 96 / G (so the
// scaled weights stay normal numbers) and |max z * G| < 4e6 (so C stays in
// [2^23, 2^24), where the float spacing is 1); otherwise the general path of
// common.cuh is used.
//
// A chunk's weights are summed in float32 (each lane of a packed pair, then the
// two lanes): a relative error of about 1e-7, the size of the weights' own
// error (ex2.approx, and the float32 tensor-core bias). The caller sends a
// chunk whose sum is not finite to the general path.
//
// Two tokens are processed per instruction with the packed .f32x2 operations
// (IEEE round-to-nearest per lane, so a scalar evaluation gives identical bits).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace ds {

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kFastSpan = 96.0f;     // max (zmax - zmin) * G on the fast path

struct G16 {
  float G, gl, gf;  // g = G + gl exactly to ~2^-40; gf = g rounded to fp32
};

__device__ __forceinline__ G16 make_g16_from(Gscale g) {
  const float G = __uint_as_float(__float_as_uint(g.hi) & 0xFFFFFF00u);
  return {G, __fadd_rn(__fsub_rn(g.hi, G), g.lo), g.hi};  // g.hi - G is exact
}

__device__ __forceinline__ G16 make_g16(float T) {
  const Gscale g = make_gscale(T);
  const float G = __uint_as_float(__float_as_uint(g.hi) & 0xFFFFFF00u);
  return {G, __fadd_rn(__fsub_rn(g.hi, G), g.lo), g.hi};  // g.hi - G is exact
}

// Scalar weight, bit-identical to one lane of fast_pair (used by the locate).
__device__ __forceinline__ float fast_w1(float z, float b, G16 g, int ref) {
  const float C = __fsub_rn(kMagic, (float)ref);
  const float m = __fmaf_rn(z, g.G, C);
  const float nk = __fmaf_rn(m, -1.0f, C);
  const float d = __fmaf_rn(z, g.G, nk);
  const float f = __fmaf_rn(b, g.gf, __fmaf_rn(z, g.gl, d));
  const float p = ex2_approx(f);
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(m) << 23));
}

struct FastConsts {
  float2 G, gl, gf, C, neg1;
};

__device__ __forceinline__ FastConsts make_fast_consts(G16 g, int ref) {
  const float C = __fsub_rn(kMagic, (float)ref);
  return {make_float2(g.G, g.G), make_float2(g.gl, g.gl), make_float2(g.gf, g.gf), make_float2(C, C),
          make_float2(-1.0f, -1.0f)};
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Weights of the two tokens packed in zw (bias b2) against the constants' reference.
__device__ __forceinline__ float2 fast_w2(uint32_t zw, float2 b2, const FastConsts& k) {
  const float2 z2 = unpack_bf16x2(zw);
  const float2 m2 = __ffma2_rn(z2, k.G, k.C);
  const float2 nk2 = __ffma2_rn(m2, k.neg1, k.C);
  const float2 d2 = __ffma2_rn(z2, k.G, nk2);
  const float2 f2 = __ffma2_rn(b2, k.gf, __ffma2_rn(z2, k.gl, d2));
  const float p0 = ex2_approx(f2.x), p1 = ex2_approx(f2.y);
  return make_float2(__uint_as_float(__float_as_uint(p0) + (__float_as_uint(m2.x) << 23)),
                     __uint_as_float(__float_as_uint(p1) + (__float_as_uint(m2.y) << 23)));
}

// Weights of the two tokens packed in zw, accumulated into s (float32, one
// rounding per addition).
__device__ __forceinline__ void fast_pair(uint32_t zw, float2 b2, const FastConsts& k, float2& s) {
  s = __fadd2_rn(s, fast_w2(zw, b2, k));
}

// Residual weight max(0, wp - R * wq) of one token, R = Rhi + Rlo (two FMAs,
// the order every side uses).
__device__ __forceinline__ float residual_w(float wp, float wq, float Rhi, float Rlo) {
  return fmaxf(__fmaf_rn(-wq, Rlo, __fmaf_rn(-wq, Rhi, wp)), 0.f);
}

// Chunk predicate against a given reference (the row-global references of the
// final draw): every logit finite, z*G within (ref - 96, ref + 1], |z*G| < 4e6.
__device__ __forceinline__ bool fast_span_ok(const uint32_t* zp, float G, int ref) {
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
  const float r = (float)ref;
  return (zmin > kNegInf) && (fabsf(zmax * G) < 4.0e6f) && (r - zmin * G < kFastSpan) &&
         (zmax * G <= r + 1.0f) && (fabsf(r) < 4.0e6f);
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
