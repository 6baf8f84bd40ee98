// Shared device numerics for the sampling kernels.
//
// Sampling by inverse CDF over a ~152k-token vocabulary must agree with a
// float64 reference on almost every draw. A per-token relative error delta in
// the weights moves the CDF by a random walk whose mean absolute size is a few
// hundred times delta at V ~ 1.5e5, so the kernels keep every weight within a
// couple of float32 ulps and never round a running sum:
//   * t = logit * log2(e) / T is carried as an unevaluated sum: the product of
//     the logit with the high part of log2(e)/T is split exactly with an FMA
//     (Dekker / Ogita-Rump-Oishi TwoProduct), the small terms are folded in.
//   * t = k + f with k = rint(t_hi) (so t_hi - k is exact), w = 2^f * 2^(k-n),
//     where n is a per-chunk integer reference: rescaling between chunks is a
//     power of two and therefore exact.
//   * Sums are double-float (Knuth's TwoSum), so accumulation adds no error
//     beyond ~2^-48 relative.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "philox.h"

namespace ds {

#define kNegInf (-__int_as_float(0x7f800000))
constexpr int kEmptyRef = -(1 << 29);  // reference of a chunk with no mass
constexpr int kChunk = 32;             // tokens per partial-sum record

enum DsStatusCode {
  kOk = 0,
  kErrInvalidArg = 1,
  kErrUnsupported = 2,
  kErrWorkspace = 3,
  kErrCuda = 4,
  kErrTimeout = 5,
  kErrBounds = 6,
  kErrNonfinite = 7
};

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---- element loads ---------------------------------------------------------

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// Load 8 consecutive elements (16-byte aligned for bf16, 32 for f32) as floats.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* o) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float* o) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// ---- double-float ----------------------------------------------------------

struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

__device__ __forceinline__ DF fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// acc += x, keeping the rounding error of the high word in the low word.
__device__ __forceinline__ void df_accumulate(DF& acc, float x) {
  const DF t = two_sum(acc.hi, x);
  acc.hi = t.hi;
  acc.lo = __fadd_rn(acc.lo, t.lo);
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  DF s = two_sum(a.hi, b.hi);
  s.lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ DF df_scale2(DF a, int e) {  // exact power-of-two scaling
  return {ldexpf(a.hi, e), ldexpf(a.lo, e)};
}

// a * b as a double-float (TwoProduct of the high words, cross terms added).
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return fast_two_sum(p, e);
}

// a < b for double-floats.
__device__ __forceinline__ bool df_lt(DF a, DF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }

// x / S for a float x and a double-float S > 0, to ~2^-23 relative.
__device__ __forceinline__ float div_by_df(float x, DF S) {
  const float q = __fdiv_rn(x, S.hi);
  return __fmaf_rn(-q, __fdiv_rn(S.lo, S.hi), q);
}

// ---- log2(e) / T as a double-float -----------------------------------------
//
// Everything on the device is float or double-float: double precision runs at
// a small fraction of the float rate on this part and sits on the latency path
// of every sampling step.

struct Gscale {
  float hi, lo;
};

// log2(e) = kLog2eHi + kLog2eLo (the float nearest, and the rest).
#define kLog2eHi __uint_as_float(0x3fb8aa3bu)
#define kLog2eLo __uint_as_float(0x32a57060u)

// g = log2(e) / T to ~2^-47 relative: q = RN(hi / T), the remainder hi - q*T
// is exact (FMA), and the remainder plus lo divided by T gives the low word.
__device__ __forceinline__ Gscale make_gscale(float T) {
  const float q = __fdiv_rn(kLog2eHi, T);
  const float rem = __fadd_rn(__fmaf_rn(-q, T, kLog2eHi), kLog2eLo);
  const float ql = __fdiv_rn(rem, T);
  const float hi = __fadd_rn(q, ql);
  return {hi, __fsub_rn(ql, __fsub_rn(hi, q))};
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// 2^(t - n) for t = (z + b) * g and an integer reference n >= rint(z * g.hi).
//   a = z*g.hi is split exactly from the product (FMA), the small terms
//   z*g.lo and b*g.hi are folded into the fraction, k = rint(a) comes from the
//   1.5*2^23 rounding trick (valid for |a| < 2^22), f = (a - k) + small lies
//   within ~[-0.5 - |b g|, 0.5 + |b g|], and 2^(k - n) is built in the exponent
//   field (flushed to 0 below 2^-126). z = -inf gives 0; NaN and +inf give NaN.
__device__ __forceinline__ float weight_rel(float z, float b, Gscale g, int n) {
  const float a = __fmul_rn(z, g.hi);
  const float ae = __fmaf_rn(z, g.hi, -a);
  float tl = __fmaf_rn(z, g.lo, ae);
  tl = __fmaf_rn(b, g.hi, tl);
  const float m = __fadd_rn(a, 12582912.f);
  const float kf = __fsub_rn(m, 12582912.f);
  const float f = __fadd_rn(__fsub_rn(a, kf), tl);
  const float p = ex2_approx(f);
  int e = (__float_as_int(m) - 0x4B400000) - n;
  e = max(e, -127);
  const float w = __fmul_rn(p, __int_as_float((e + 127) << 23));
  return z == kNegInf ? 0.f : w;
}

// Chunk reference: rint of the largest z*g.hi among finite entries.
__device__ __forceinline__ float scaled_hi(float z, Gscale g) { return __fmul_rn(z, g.hi); }

// ---- uniform ---------------------------------------------------------------

// u = (w + 1/2) * 2^-32 of the stream's first word, exactly, as a double-float:
// w = a * 2^16 + c gives u = a * 2^-16 + (c + 1/2) * 2^-32 (both terms exact).
__device__ __forceinline__ DF uniform_df(uint64_t seed, uint32_t request, uint32_t position,
                                         uint32_t stage) {
  const uint32_t w = philox_word(seed, request, position, stage);
  const float a = __uint2float_rn(w >> 16) * 1.52587890625e-05f;               // 2^-16
  const float c = (__uint2float_rn(w & 0xffffu) + 0.5f) * 2.3283064365386963e-10f;  // 2^-32
  return fast_two_sum(a, c);
}

// Non-finite check for logits: NaN or +inf is an error; -inf is allowed.
__device__ __forceinline__ bool bad_logit(float x) {
  return !(x == x) || x == __int_as_float(0x7f800000);
}

}  // namespace ds
