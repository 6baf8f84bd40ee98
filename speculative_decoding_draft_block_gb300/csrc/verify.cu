// Verification kernels: target row statistics, accept tests and the final
// draw's set-up.
//
// DSpark summary page, 배경: verification is left to right; the first rejection
// discards everything after it, and the rejection rule keeps the target's
// distribution exactly. Per (request b, scheduled position k <= L_b + 1):
//
//   verify_rows_kernel      one CTA per target row, dispatched in position
//                           order; a request's rows after its first recorded
//                           rejection return at once; per row: streams it once
//                           with 16-byte loads, builds S_p = sum 2^(t_i g - ref)
//                           (per-thread power-of-two references merged
//                           exactly, double-float sums), evaluates p(x_k) and
//                           takes the accept decision u * q(x_k) < p(x_k) in
//                           double-float (greedy rows: target argmax and exact match);
//                           optionally stores p(x_k) itself.
//   verify_finalize_kernel  one thread per request: accepted prefix length,
//                           emitted tokens, and the descriptor of the final
//                           draw (residual at the first rejection, or bonus
//                           from row L+1), drawn by the shared sampling kernels.
#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "fastpath.cuh"
#include "internal.h"
#include "sampling.cuh"
#include "sm100.cuh"

namespace ds {

namespace {

constexpr int kRowThreads = 256;

// Row sum of one thread's 8-token groups of bf16 target logits, relative to a
// running integer reference R (the largest group reference seen so far).
//
// Only the normaliser S_p is needed here (for p(x) = w_x / S_p and the
// residual ratio S_p / S_q), not a CDF, so each weight is 2^(z g_hi - R) with
// one rounded FMA for the exponent and ex2.approx (relative error a few 1e-7
// for the weights that carry the sum, unbiased); each 8-token group is summed
// in float32 and added to a double-float total. S_p then agrees with float64
// to ~1e-7, far inside the 1e-6 accept-test margin. A group that raises R
// rescales the total by an exact power of two; a group with a non-finite or
// out-of-range logit takes the general path. Returns false if nothing was
// finite.
__device__ __forceinline__ bool row_sum_bf16(const __nv_bfloat16* row, int V, int tid, Gscale g,
                                             DF& total, int& R, bool& bad) {
  R = INT_MIN;
  total = {0.f, 0.f};
  const float2 G2 = make_float2(g.hi, g.hi);
  float2 NR2 = make_float2(0.f, 0.f);  // -R
  // move the reference up to nr: the total so far is rescaled by an exact power of two
  auto raise = [&](int nr) {
    if (R != INT_MIN) {
      const float f = pow2_clamped(R - nr);
      total = {__fmul_rn(total.hi, f), __fmul_rn(total.lo, f)};
    }
    R = nr;
    NR2 = make_float2(-(float)R, -(float)R);
  };
  auto group = [&](const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    __nv_bfloat162 mx = *reinterpret_cast<const __nv_bfloat162*>(&w[0]);
#pragma unroll
    for (int q = 1; q < 4; ++q) mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&w[q]));
    const float zmax = fmaxf(__low2float(mx), __high2float(mx));
    const float amax = __fmul_rn(zmax, g.hi);
    if (fabsf(amax) < 4.0e6f) {  // finite and in range (NaN fails too)
      const int gref = (int)rintf(amax);
      if (gref > R) raise(gref);
      // the 8 weights (each <= 2) summed in float32 (one rounding per addition,
      // relative error ~1e-7 per group, unbiased), then added exactly to the
      // double-float total
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 z2 = unpack_bf16x2(w[q]);
        const float2 a2 = __ffma2_rn(z2, G2, NR2);
        s2 = __fadd2_rn(s2, make_float2(ex2_approx(a2.x), ex2_approx(a2.y)));
      }
      df_accumulate(total, __fadd_rn(s2.x, s2.y));
      return;
    }
    // general path for this group (relative to R, or to a new R if none yet)
    float f8[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f8[2 * q] = __uint_as_float(w[q] << 16);
      f8[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
    float am = kNegInf;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      bad |= bad_logit(f8[q]);
      if (f8[q] != kNegInf) am = fmaxf(am, scaled_hi(f8[q], g));
    }
    if (am == kNegInf) return;
    const int ng = (int)rintf(am);
    if (ng > R) raise(ng);
#pragma unroll
    for (int q = 0; q < 8; ++q) df_accumulate(total, weight_rel(f8[q], 0.f, g, R));
  };
  // kLoads 16-byte loads in flight per thread
  constexpr int kStride = kRowThreads * 8, kLoads = 4;
  for (int i0 = tid * 8; i0 < V; i0 += kLoads * kStride) {
    uint4 v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u)
      if (i0 + u * kStride < V) v[u] = __ldcs(reinterpret_cast<const uint4*>(row + i0 + u * kStride));
#pragma unroll
    for (int u = 0; u < kLoads; ++u)
      if (i0 + u * kStride < V) group(v[u]);
  }
  return R != INT_MIN;
}

struct RowShared {
  float sv[kRowThreads / 32];
  int si[kRowThreads / 32];
  int sref[kRowThreads / 32];
  DF sdf[kRowThreads];
  int len, skip;  // the row's scheduled length and skip decision, from thread 0
};

// Target row j of request b (j <= L): S_p, and for j < L the accept test of
// the drafted token at position j + 1 (greedy: exact match with the argmax).
// Called by the whole CTA; returns the accept flag (thread 0's copy).
template <typename Tin>
__device__ __forceinline__ bool verify_row(const VerifyParams& p, int b, int j, int L, RowShared& sh) {
  float* sv = sh.sv;
  int* si = sh.si;
  int* sref = sh.sref;
  DF* sdf = sh.sdf;
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  const float T = p.temperature[b];
  const Tin* row = reinterpret_cast<const Tin*>(p.target_logits) + ((size_t)b * (p.K + 1) + j) * (size_t)p.V;
  VRow out;
  out.s_hi = out.s_lo = 0.f;
  out.ref = 0;
  out.argmax = -1;
  out.accept = 0;
  out.valid = 1;
  out.pad[0] = out.pad[1] = 0;
  bool bad = false;

  if (T == 0.f) {
    float best = kNegInf;
    int bi = INT_MAX;
    for (int i = tid * 8; i < p.V; i += kRowThreads * 8) {
      float v[8];
      load8(row + i, v);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        bad |= bad_logit(v[q]);
        if (v[q] > best || bi == INT_MAX) {
          best = v[q];
          bi = i + q;
        }
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) {
        best = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      sv[wid] = best;
      si[wid] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      float bb = sv[0];
      int bx = si[0];
      for (int w = 1; w < kRowThreads / 32; ++w)
        if (sv[w] > bb || (sv[w] == bb && si[w] < bx)) {
          bb = sv[w];
          bx = si[w];
        }
      out.argmax = bx;
      if (j < L) {
        out.accept = (p.draft_tokens[(size_t)b * p.K + j] == bx) ? 1 : 0;
        // the greedy target law is the point mass on its argmax
        if (p.p_token != nullptr) p.p_token[(size_t)b * p.K + j] = out.accept ? 1.f : 0.f;
      }
    }
  } else {
    if (!(T >= 1e-3f && T <= 1e3f)) {
      if (tid == 0) report(p.status, kErrInvalidArg);
      return false;
    }
    const Gscale g = make_gscale(T);
    int nt = INT_MIN;
    DF acc = {0.f, 0.f};
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
      int R;
      if (row_sum_bf16(row, p.V, tid, g, acc, R, bad)) nt = R;
    } else
    for (int i = tid * 8; i < p.V; i += kRowThreads * 8) {
      float v[8];
      load8(row + i, v);
      float amax = kNegInf;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        bad |= bad_logit(v[q]);
        if (v[q] != kNegInf) amax = fmaxf(amax, scaled_hi(v[q], g));
      }
      if (amax == kNegInf) continue;
      const int ng = (int)rintf(amax);
      if (ng > nt) {
        if (nt != INT_MIN) acc = df_scale2(acc, max(nt - ng, -300));
        nt = ng;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) df_accumulate(acc, weight_rel(v[q], 0.f, g, nt));
    }
    int m = nt;
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) sref[wid] = m;
    __syncthreads();
    int N = sref[0];
    for (int w = 1; w < kRowThreads / 32; ++w) N = max(N, sref[w]);
    sdf[tid] = (nt == INT_MIN) ? DF{0.f, 0.f} : rec_scaled(ChunkRec{acc.hi, acc.lo, nt, 0}, N);
    __syncthreads();
    // fixed-order tree reduction
    for (int s = kRowThreads / 2; s > 0; s >>= 1) {
      if (tid < s) sdf[tid] = df_add(sdf[tid], sdf[tid + s]);
      __syncthreads();
    }
    if (tid == 0) {
      const DF S = sdf[0];
      out.s_hi = S.hi;
      out.s_lo = S.lo;
      out.ref = N;
      const bool pos = S.hi > 0.f;
      if (!pos) bad = true;
      if (j < L && pos) {
        int x = p.draft_tokens[(size_t)b * p.K + j];
        if (x < 0 || x >= p.V) {
          report(p.status, kErrBounds);
          x = 0;
        }
        const float tx = to_f32(row[x]);
        // u * q(x) < p(x) = w_x / S, tested as u * q(x) * S < w_x
        const float wx = weight_rel(tx, 0.f, g, N);
        const float qx = p.q_token[(size_t)b * p.K + j];
        const uint64_t seed = p.seed_ptr != nullptr ? *p.seed_ptr : p.seed;
        const DF uq = df_mul(uniform_df(seed, (uint32_t)b, (uint32_t)(j + 1), DS_STAGE_ACCEPT),
                             DF{qx, 0.f});
        out.accept = df_lt(df_mul(uq, S), DF{wx, 0.f}) ? 1 : 0;
        if (p.p_token != nullptr) p.p_token[(size_t)b * p.K + j] = div_by_df(wx, S);
      }
    }
  }
  if (bad) report(p.status, kErrNonfinite);
  if (tid == 0) p.vrows[(size_t)b * (p.K + 1) + j] = out;
  return out.accept != 0;
}

// One CTA per target row, launched position-major (blockIdx.y is the position),
// so every request's row 0 is dispatched first, then row 1, and so on. A CTA
// whose request already recorded a rejection at an earlier position returns at
// once (verification stops at the first rejection), so the rows streamed
// approach sum_b min(a_b + 1, L_b + 1). A row started before the earlier
// result is known is still evaluated: the finalize kernel reads rows only up
// to the first rejection.
template <typename Tin>
__global__ void __launch_bounds__(kRowThreads) verify_rows_kernel(VerifyParams p) {
  __shared__ RowShared sh;
  const int tid = threadIdx.x;
  const int b = blockIdx.x, j = blockIdx.y;
  // thread 0 decides for the CTA: first_reject changes under other CTAs, so no
  // other thread reads it (every thread must take the same path)
  if (tid == 0) {
    int L = p.sched_len[b];
    if (L < 0 || L > p.K) {
      if (j == 0) report(p.status, kErrInvalidArg);
      L = L < 0 ? 0 : p.K;
    }
    int skip = 0;
    if (j > L) {
      skip = 2;  // not scheduled
    } else if (*reinterpret_cast<volatile uint32_t*>(p.first_reject + b) < (uint32_t)j) {
      skip = 1;  // an earlier row rejected
      if (j < L && p.p_token != nullptr) p.p_token[(size_t)b * p.K + j] = -1.f;  // not evaluated
    }
    sh.len = L;
    sh.skip = skip;
  }
  __syncthreads();
  const int L = sh.len;
  if (sh.skip) return;
  const bool acc = verify_row<Tin>(p, b, j, L, sh);
  if (tid == 0 && j < L && !acc) atomicMin(p.first_reject + b, (uint32_t)j);
}

// One warp per request: lane 0 walks the accept flags and writes the final
// draw's descriptor; the warp writes the emitted-token row.
__global__ void __launch_bounds__(128) verify_finalize_kernel(VerifyParams p) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (b >= p.B) return;
  const int K = p.K;
  int L = p.sched_len[b];
  L = L < 0 ? 0 : (L > K ? K : L);
  const float T = p.temperature[b];
  const VRow* vr = p.vrows + (size_t)b * (K + 1);
  int a = 0;
  while (a < L && vr[a].accept) ++a;
  int32_t* out = p.out_tokens + (size_t)b * (K + 1);
  for (int i = lane; i <= K; i += 32) out[i] = i < a ? p.draft_tokens[(size_t)b * K + i] : -1;
  if (p.p_token != nullptr)  // positions past L_b were not verified (the rows kernel wrote k < L_b)
    for (int i = L + lane; i < K; i += 32) p.p_token[(size_t)b * K + i] = -1.f;
  FinalDesc d;
  d.mode = kSkip;
  d.row = a;
  d.a_token = -1;
  d.out_pos = a;
  d.Np = d.Nq = 0;
  d.Rhi = d.Rlo = 0.f;
  if (T == 0.f) {
    __syncwarp();
    if (lane == 0) out[a] = vr[a].argmax;
  } else if (T >= 1e-3f && T <= 1e3f) {
    d.Np = vr[a].ref;
    if (a < L) {
      d.mode = kResidual;
      d.a_token = (a == 0) ? p.anchor[b] : p.draft_tokens[(size_t)b * K + (a - 1)];
      const ds_row_stats qs = p.q_stats[(size_t)b * K + a];
      d.Nq = qs.ref;
      // R = S_p / S_q as a double-float: q = RN(Sp.hi / Sq.hi) refined by one
      // correction step with the exact residual of the high words
      const DF Sp = {vr[a].s_hi, vr[a].s_lo}, Sq = {qs.sum_hi, qs.sum_lo};
      const float q = __fdiv_rn(Sp.hi, Sq.hi);
      const DF qS = df_mul(DF{q, 0.f}, Sq);
      const DF res = df_add(Sp, DF{-qS.hi, -qS.lo});
      const float ql = __fdiv_rn(res.hi, Sq.hi);
      const DF R = fast_two_sum(q, ql);
      d.Rhi = R.hi;
      d.Rlo = R.lo;
    } else {
      d.mode = kBonus;
    }
  }
  if (lane == 0) {
    p.accept_count[b] = a;
    p.num_emitted[b] = a + 1;
    p.final_desc[b] = d;
  }
}

}  // namespace

cudaError_t launch_verify_rows(const VerifyParams& p, cudaStream_t s) {
  dim3 grid(p.B, p.K + 1);  // position-major dispatch order
  if (p.dtype == DS_BF16)
    verify_rows_kernel<__nv_bfloat16><<<grid, kRowThreads, 0, s>>>(p);
  else
    verify_rows_kernel<float><<<grid, kRowThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_verify_finalize(const VerifyParams& p, cudaStream_t s) {
  verify_finalize_kernel<<<(p.B + 3) / 4, 128, 0, s>>>(p);
  return cudaGetLastError();
}

namespace {

constexpr int kFetchThreads = 256;
constexpr int kFetchChunk16 = 4096;  // 16-byte words per CTA (64 KB)

// Target rows 0..L_b of request b from host memory mapped into the device's
// address space: CTA (x, b) copies words [x * kFetchChunk16, ...) of the
// request's first L_b + 1 rows, four 16-byte loads in flight per thread.
// L_b comes from the device (the schedule's output), so no host round trip
// sits between the schedule and verify.
__global__ void __launch_bounds__(kFetchThreads)
    fetch_rows_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int K, size_t row16,
                      const int32_t* __restrict__ sched_len, unsigned long long* bytes) {
  const int b = blockIdx.y;
  int L = sched_len[b];
  L = L < 0 ? 0 : (L > K ? K : L);
  const size_t n16 = (size_t)(L + 1) * row16;
  if (bytes != nullptr && blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(bytes, (unsigned long long)n16 * 16);
  const size_t c0 = (size_t)blockIdx.x * kFetchChunk16;
  if (c0 >= n16) return;
  const size_t c1 = c0 + kFetchChunk16 < n16 ? c0 + kFetchChunk16 : n16;
  const size_t base = (size_t)b * (size_t)(K + 1) * row16;
  const uint4* sp = src + base;
  uint4* dp = dst + base;
  size_t i = c0 + threadIdx.x;
  for (; i + 3 * kFetchThreads < c1; i += 4 * kFetchThreads) {
    const uint4 v0 = sp[i], v1 = sp[i + kFetchThreads], v2 = sp[i + 2 * kFetchThreads],
                v3 = sp[i + 3 * kFetchThreads];
    dp[i] = v0;
    dp[i + kFetchThreads] = v1;
    dp[i + 2 * kFetchThreads] = v2;
    dp[i + 3 * kFetchThreads] = v3;
  }
  for (; i < c1; i += kFetchThreads) dp[i] = sp[i];
}

}  // namespace

cudaError_t launch_fetch_rows(void* dst, const void* src_dev, int32_t B, int32_t K, size_t row_bytes,
                              const int32_t* sched_len, unsigned long long* bytes, cudaStream_t s) {
  const size_t row16 = row_bytes / 16;
  const size_t req16 = (size_t)(K + 1) * row16;
  dim3 grid((unsigned)((req16 + kFetchChunk16 - 1) / kFetchChunk16), (unsigned)B);
  fetch_rows_kernel<<<grid, kFetchThreads, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src_dev),
                                                   K, row16, sched_len, bytes);
  return cudaGetLastError();
}

}  // namespace ds
