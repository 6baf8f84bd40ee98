// Per-row sampling context and the per-chunk reductions shared by the tile
// kernels (tensor-core and SIMT) and the locate kernel.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace ds {
namespace {

// Everything a kernel needs to know about one row of the batch being sampled.
struct RowCtx {
  int32_t mode;
  int32_t a_token;  // E row of the bias; -1 when the row needs no bias
  const void* zrow;
  const void* trow;
  Gscale g;
  int32_t Np, Nq;
  float Rhi, Rlo;
  uint32_t upos, ustage;  // Philox position and stage of the row's draw
  int32_t out_index;      // flat index of the drawn token in tokens_out
  int32_t zk;             // draft: 0-based position of the base row; final: row index j
};

// The values a row's context is built from, loaded with no dependence on one
// another so that they travel in one round: the temperature, and the
// conditioning token (draft) or the final-draw descriptor (verify).
struct RowInputs {
  float T;
  int32_t tok;
  FinalDesc d;
};

// The tokens of earlier positions are written by other CTAs of the same
// launch in the persistent draft kernel: read them at L2 (never a stale L1
// line). `step` is the 1-based draft position (p.step outside that kernel).
__device__ __forceinline__ RowInputs load_row_inputs(const SampleParams& p, int b, int step) {
  RowInputs in;
  in.T = 0.f;
  in.tok = 0;
  in.d = FinalDesc{kSkip, 0, 0, 0, 0, 0, 0.f, 0.f};
  if (b >= p.B) return in;
  in.T = p.temperature[b];
  if (p.src == 0)
    in.tok = (step == 1) ? p.anchor[b] : __ldcg(p.draft_tokens + (size_t)b * p.K + (step - 2));
  else
    in.d = p.final_desc[b];
  return in;
}

template <typename Tin>
__device__ RowCtx make_row_ctx(const SampleParams& p, int b, const RowInputs& in, int step) {
  RowCtx c;
  c.mode = kSkip;
  c.a_token = -1;
  c.zrow = nullptr;
  c.trow = nullptr;
  c.g = {0.f, 0.f};
  c.Np = c.Nq = 0;
  c.Rhi = c.Rlo = 0.f;
  c.upos = 0;
  c.ustage = 0;
  c.out_index = 0;
  c.zk = 0;
  if (b >= p.B) return c;
  const Tin* base = reinterpret_cast<const Tin*>(p.base_logits);
  const Tin* tgt = reinterpret_cast<const Tin*>(p.target_logits);
  const float T = in.T;
  const bool greedy = (T == 0.f);
  if (!greedy && !(T >= 1e-3f && T <= 1e3f)) {
    report(p.status, kErrInvalidArg);
    return c;
  }
  if (!greedy) c.g = make_gscale(T);
  if (p.src == 0) {
    const int k = step;  // 1-based
    int tok = in.tok;
    if (tok < 0 || tok >= p.V) {
      report(p.status, kErrBounds);
      tok = 0;
    }
    c.a_token = tok;
    c.mode = greedy ? kGreedyMarkov : kSampleMarkov;
    c.zrow = base + ((size_t)b * p.K + (k - 1)) * (size_t)p.V;
    c.upos = (uint32_t)k;
    c.ustage = DS_STAGE_DRAFT;
    c.out_index = b * p.K + (k - 1);
    c.zk = k - 1;
  } else {
    const FinalDesc d = in.d;
    if (greedy || d.mode == kSkip) return c;
    c.mode = d.mode;
    c.trow = tgt + ((size_t)b * (p.K + 1) + d.row) * (size_t)p.V;
    c.Np = d.Np;
    c.upos = (uint32_t)(d.row + 1);
    c.ustage = DS_STAGE_RESAMPLE;
    c.out_index = b * (p.K + 1) + d.out_pos;
    c.zk = d.row;
    if (d.mode == kResidual) {
      int tok = d.a_token;
      if (tok < 0 || tok >= p.V) {
        report(p.status, kErrBounds);
        tok = 0;
      }
      c.a_token = tok;
      c.zrow = base + ((size_t)b * p.K + d.row) * (size_t)p.V;
      c.Nq = d.Nq;
      c.Rhi = d.Rhi;
      c.Rlo = d.Rlo;
    }
  }
  return c;
}

template <typename Tin>
__device__ RowCtx make_row_ctx(const SampleParams& p, int b, int step) {
  return make_row_ctx<Tin>(p, b, load_row_inputs(p, b, step), step);
}

template <typename Tin>
__device__ RowCtx make_row_ctx(const SampleParams& p, int b) {
  return make_row_ctx<Tin>(p, b, p.step);
}

// The r-vector whose product with P is the row's bias: E[a_token] for the
// Markov head; for the RNN head the state of the step (draft) or of row zk
// (final draw). Only meaningful when c.a_token >= 0.
template <typename Tin>
__device__ __forceinline__ const Tin* bias_row(const SampleParams& p, int b, const RowCtx& c) {
  if (p.a_rows != nullptr) {
    int j = p.src == 0 ? 0 : c.zk;
    j = j < 0 ? 0 : (j >= p.K ? p.K - 1 : j);
    return reinterpret_cast<const Tin*>(p.a_rows) + (size_t)b * p.a_rows_stride + (size_t)j * p.r;
  }
  return reinterpret_cast<const Tin*>(p.E) + (size_t)(c.a_token >= 0 ? c.a_token : 0) * p.r;
}

// Chunk reference n = rint(max_j z_j * g.hi) over finite z; kEmptyRef if none.
__device__ __forceinline__ int chunk_ref_from_max(float amax) {
  return amax == kNegInf ? kEmptyRef : (int)rintf(amax);
}

// Element sources for chunk_record: plain floats, or bf16 pairs packed in
// 32-bit words (the tensor-core epilogue keeps its logits packed to save
// registers; unpacking is a shift or a mask).
struct F32Src {
  const float* p;
  __device__ __forceinline__ float operator()(int j) const { return p[j]; }
};
struct Bf16Src {
  const uint32_t* p;
  __device__ __forceinline__ float operator()(int j) const {
    const uint32_t w = p[j >> 1];
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};

// Reduce one chunk of n (<= 32) tokens starting at token col0 to its record.
// z, bias, t give the chunk's base logits, Markov bias and target logits.
// If w_out is given, per-token weights (relative to rec.ref) are written too.
template <bool FULL, typename ZS, typename TS>
__device__ __forceinline__ void chunk_record(const RowCtx& c, ZS z, const float* bias, TS t, int n,
                                             int col0, ChunkRec& rec, int32_t* status,
                                             float* w_out = nullptr) {
  constexpr int NMAX = 32;
  rec.hi = 0.f;
  rec.lo = 0.f;
  rec.ref = 0;
  rec.idx = -1;
  bool bad = false;
  if (c.mode == kGreedyMarkov) {
    DF best = {kNegInf, 0.f};
    int bi = -1;
#pragma unroll
    for (int j = 0; j < NMAX; ++j) {
      if (FULL || j < n) {
        const float zj = z(j);
        bad |= bad_logit(zj) || !(bias[j] == bias[j]);
        DF l = (zj == kNegInf) ? DF{kNegInf, 0.f} : two_sum(zj, bias[j]);
        if (bi < 0 || l.hi > best.hi || (l.hi == best.hi && l.lo > best.lo)) {
          best = l;
          bi = col0 + j;
        }
      }
    }
    rec.hi = best.hi;
    rec.lo = best.lo;
    rec.idx = bi;
  } else if (c.mode == kSampleMarkov) {
    // NaN / +inf logits or biases make the sum non-finite; -inf weighs 0.
    float amax = kNegInf;
#pragma unroll
    for (int j = 0; j < NMAX; ++j)
      if (FULL || j < n) amax = fmaxf(amax, scaled_hi(z(j), c.g));
    const int ref = chunk_ref_from_max(amax);
    DF s = {0.f, 0.f};
    if (ref != kEmptyRef) {
#pragma unroll
      for (int j = 0; j < NMAX; ++j) {
        if (FULL || j < n) {
          const float w = weight_rel(z(j), bias[j], c.g, ref);
          df_accumulate(s, w);
          if (w_out) w_out[j] = w;
        } else if (w_out) {
          w_out[j] = 0.f;
        }
      }
    } else {
      bool any_nan = false;
#pragma unroll
      for (int j = 0; j < NMAX; ++j)
        if (FULL || j < n) any_nan |= !(z(j) == z(j));
      bad |= any_nan;
      if (w_out)
#pragma unroll
        for (int j = 0; j < NMAX; ++j) w_out[j] = 0.f;
    }
    bad |= !isfinite(s.hi);
    rec.hi = s.hi;
    rec.lo = s.lo;
    rec.ref = ref;
  } else {  // kResidual / kBonus: weights on the row's global scale
    DF s = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NMAX; ++j) {
      if (FULL || j < n) {
        float w = weight_rel(t(j), 0.f, c.g, c.Np);
        if (c.mode == kResidual) {
          const float wq = weight_rel(z(j), bias[j], c.g, c.Nq);
          float d = __fmaf_rn(-wq, c.Rhi, w);
          d = __fmaf_rn(-wq, c.Rlo, d);
          bad |= !(d == d);
          w = fmaxf(d, 0.f);
        }
        df_accumulate(s, w);
        if (w_out) w_out[j] = w;
      } else if (w_out) {
        w_out[j] = 0.f;
      }
    }
    bad |= !isfinite(s.hi);
    rec.hi = s.hi;
    rec.lo = s.lo;
    rec.ref = 0;
  }
  if (bad) report(status, kErrNonfinite);
}

// ---- group records -------------------------------------------------------
//
// A group record combines the chunk records of a contiguous token range:
//   sampling rows: ref = the largest chunk reference, hi + lo = the sum of the
//                  chunk sums each scaled by 2^(chunk ref - ref) (exact powers
//                  of two; chunks below 2^-126 relative to the group's
//                  reference are dropped, far below the sampling tolerance)
//   greedy rows:   the largest (hi, lo) with the smallest token on ties
//   residual/bonus rows: the plain double-float sum (records share ref 0)

// x * 2^e for e <= 0 without a library call (rounds only in the subnormal range).
__device__ __forceinline__ float pow2_scale(float x, int e) {
  if (e >= -126) return __fmul_rn(x, __int_as_float((e + 127) << 23));
  if (e < -252) return __fmul_rn(x, 0.f);
  return __fmul_rn(__fmul_rn(x, __int_as_float(1 << 23)), __int_as_float((e + 253) << 23));
}

// A record's mass relative to the reference N (N >= every non-empty ref).
__device__ __forceinline__ DF rec_scaled(const ChunkRec& r, int N) {
  if (r.ref == kEmptyRef) return {0.f, 0.f};
  const long long e = (long long)r.ref - N;
  const int ei = e < -300 ? -300 : (int)e;
  return {pow2_scale(r.hi, ei), pow2_scale(r.lo, ei)};
}

// Record load that bypasses L1 (records are written by the previous kernel).
__device__ __forceinline__ ChunkRec ld_rec(const ChunkRec* q) {
  const uint4 v = __ldcg(reinterpret_cast<const uint4*>(q));
  return {__uint_as_float(v.x), __uint_as_float(v.y), (int32_t)v.z, (int32_t)v.w};
}

__device__ __forceinline__ ChunkRec group_empty() { return {0.f, 0.f, kEmptyRef, -1}; }

__device__ __forceinline__ bool greedy_better(const ChunkRec& a, const ChunkRec& b) {
  if (a.idx < 0) return false;
  if (b.idx < 0) return true;
  return a.hi > b.hi || (a.hi == b.hi && (a.lo > b.lo || (a.lo == b.lo && a.idx < b.idx)));
}

// 2^e for e in [-127, 0] as a float (2^-127 -> +0: contributions below 2^-126
// relative to the group's reference are dropped).
__device__ __forceinline__ float pow2_clamped(int e) { return __int_as_float((max(e, -127) + 127) << 23); }

__device__ __forceinline__ void group_merge(int mode, ChunkRec& acc, const ChunkRec& r) {
  if (mode == kGreedyMarkov) {
    if (greedy_better(r, acc)) acc = r;
  } else if (mode == kSampleMarkov) {
    // branch-free: an empty side (ref kEmptyRef, sum 0) scales to 0
    const int R = max(acc.ref, r.ref);
    const float fa = pow2_clamped(acc.ref - R), fr = pow2_clamped(r.ref - R);
    const DF s = df_add(DF{__fmul_rn(acc.hi, fa), __fmul_rn(acc.lo, fa)},
                        DF{__fmul_rn(r.hi, fr), __fmul_rn(r.lo, fr)});
    acc.hi = s.hi;
    acc.lo = s.lo;
    acc.ref = R;
  } else {
    const DF s = df_add(DF{acc.hi, acc.lo}, DF{r.hi, r.lo});
    acc.hi = s.hi;
    acc.lo = s.lo;
    acc.ref = 0;
  }
}

__device__ __forceinline__ ChunkRec shfl_xor_rec(const ChunkRec& r, int o) {
  return {__shfl_xor_sync(0xffffffffu, r.hi, o), __shfl_xor_sync(0xffffffffu, r.lo, o),
          __shfl_xor_sync(0xffffffffu, r.ref, o), __shfl_xor_sync(0xffffffffu, r.idx, o)};
}

}  // namespace
}  // namespace ds
