// Analytic per-position acceptance rate 1 - TV(p, q) = sum_i min(p_i, q_i).
//
// DSpark summary page, 방법론 › 신뢰도 기반 검증 (the STS paragraph): the STS
// temperatures are fitted against the probability that a drafted position
// passes verification; under the accept rule of the 배경 section (accept
// x ~ q with probability min(1, p(x) / q(x))) that probability is
// sum_x min(p(x), q(x)). One CTA per row: pass 1 finds both rows' maxima,
// pass 2 their normalisers, pass 3 sums min(p_i, q_i); passes 2 and 3 find
// the row in L2. Float32 arithmetic with per-thread sums over a few hundred
// tokens: the result is a soft label, so a relative error of ~1e-5 is ample.
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace ds {
namespace {

constexpr int kAccThreads = 512;

__device__ __forceinline__ void load8f(const __nv_bfloat16* p, float* o) { load8(p, o); }
__device__ __forceinline__ void load8f(const float* p, float* o) { load8(p, o); }

template <typename T>
__device__ __forceinline__ T block_reduce(T v, T (*op)(T, T), T* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();  // sh may still be read by a previous reduction
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  T r = sh[0];
  for (int w = 1; w < kAccThreads / 32; ++w) r = op(r, sh[w]);
  return r;
}

__device__ float fmax_op(float a, float b) { return fmaxf(a, b); }
__device__ float fadd_op(float a, float b) { return __fadd_rn(a, b); }

// Greedy rows: first index of the largest value (ties: lowest index).
__device__ __forceinline__ void better(float v, int i, float& bv, int& bi) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kAccThreads)
    acceptance_kernel(const Tin* __restrict__ target, const Tin* __restrict__ draft, int V,
                      const float* __restrict__ temperature, float* __restrict__ alpha, int32_t* status) {
  __shared__ float shf[kAccThreads / 32];
  __shared__ int shi[kAccThreads / 32];
  const size_t row = blockIdx.x;
  const Tin* t = target + row * (size_t)V;
  const Tin* d = draft + row * (size_t)V;
  const float T = temperature[row];
  const int tid = threadIdx.x;
  bool bad = false;
  if (T == 0.f) {
    float bt = kNegInf, bd = kNegInf;
    int it = INT_MAX, id = INT_MAX;
    for (int i = tid * 8; i < V; i += kAccThreads * 8) {
      float x[8], y[8];
      load8f(t + i, x);
      load8f(d + i, y);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        bad |= bad_logit(x[q]) || bad_logit(y[q]);
        better(x[q], i + q, bt, it);
        better(y[q], i + q, bd, id);
      }
    }
    // (value, index) reductions for both rows, lowest index on ties
    for (int pass = 0; pass < 2; ++pass) {
      float v = pass ? bd : bt;
      int ix = pass ? id : it;
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
        better(ov, oi, v, ix);
      }
      __syncthreads();
      if ((tid & 31) == 0) {
        shf[tid >> 5] = v;
        shi[tid >> 5] = ix;
      }
      __syncthreads();
      v = shf[0];
      ix = shi[0];
      for (int w = 1; w < kAccThreads / 32; ++w) better(shf[w], shi[w], v, ix);
      if (pass) id = ix; else it = ix;
    }
    if (bad) report(status, kErrNonfinite);
    if (tid == 0) alpha[row] = (it == id) ? 1.f : 0.f;
    return;
  }
  if (!(T >= 1e-3f && T <= 1e3f)) {
    if (tid == 0) {
      report(status, kErrInvalidArg);
      alpha[row] = 0.f;
    }
    return;
  }
  const float g = __fdiv_rn(kLog2eHi, T);  // log2(e) / T
  // pass 1: maxima (finite logits; -inf has zero probability)
  float mt = kNegInf, md = kNegInf;
  for (int i = tid * 8; i < V; i += kAccThreads * 8) {
    float x[8], y[8];
    load8f(t + i, x);
    load8f(d + i, y);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      bad |= bad_logit(x[q]) || bad_logit(y[q]);
      mt = fmaxf(mt, x[q]);
      md = fmaxf(md, y[q]);
    }
  }
  mt = block_reduce<float>(mt, fmax_op, shf);
  md = block_reduce<float>(md, fmax_op, shf);
  if (!(mt > kNegInf) || !(md > kNegInf)) bad = true;
  // pass 2: normalisers of 2^((x - max) g)
  const float nt = -mt * g, nd = -md * g;
  float st = 0.f, sd = 0.f;
  for (int i = tid * 8; i < V; i += kAccThreads * 8) {
    float x[8], y[8];
    load8f(t + i, x);
    load8f(d + i, y);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      st = __fadd_rn(st, ex2_approx(__fmaf_rn(x[q], g, nt)));
      sd = __fadd_rn(sd, ex2_approx(__fmaf_rn(y[q], g, nd)));
    }
  }
  st = block_reduce<float>(st, fadd_op, shf);
  sd = block_reduce<float>(sd, fadd_op, shf);
  const float it = __frcp_rn(st), id = __frcp_rn(sd);
  // pass 3: sum of min(p_i, q_i)
  float a = 0.f;
  for (int i = tid * 8; i < V; i += kAccThreads * 8) {
    float x[8], y[8];
    load8f(t + i, x);
    load8f(d + i, y);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      a = __fadd_rn(a, fminf(ex2_approx(__fmaf_rn(x[q], g, nt)) * it, ex2_approx(__fmaf_rn(y[q], g, nd)) * id));
  }
  a = block_reduce<float>(a, fadd_op, shf);
  if (bad) report(status, kErrNonfinite);
  if (tid == 0) alpha[row] = fminf(fmaxf(a, 0.f), 1.f);
}

}  // namespace

cudaError_t launch_acceptance(const void* target, const void* draft, int32_t rows, int32_t V, int32_t dtype,
                              const float* temperature, float* alpha, int32_t* status, cudaStream_t s) {
  if (dtype == DS_BF16)
    acceptance_kernel<__nv_bfloat16><<<rows, kAccThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(target), static_cast<const __nv_bfloat16*>(draft), V, temperature,
        alpha, status);
  else
    acceptance_kernel<float><<<rows, kAccThreads, 0, s>>>(static_cast<const float*>(target),
                                                          static_cast<const float*>(draft), V, temperature,
                                                          alpha, status);
  return cudaGetLastError();
}

}  // namespace ds
