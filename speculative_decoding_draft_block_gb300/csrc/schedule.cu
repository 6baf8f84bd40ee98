// Confidence head, survival and the hardware-aware prefix scheduler.
//
// Asynchronous variant (DSpark summary page, 주요 결과 › 프로덕션 배포 결과):
// the verify budget of cycle t is the early-stop count of cycle t - 2, kept in
// a device ring {budget, budget, cycle counter, 0} that the schedule kernel
// advances itself (nothing changes on the host between cycles, so a captured
// cycle replays), and the candidates taken are the first budget-many of cycle
// t's own sorted order.
//
// DSpark summary page, 방법론 › 신뢰도 기반 검증:
//   c_k = sigmoid((w_h . h_k + w_e . E[x_{k-1}] + b) / T_k)   (STS temperature T_k)
//   s_k = c_1 * ... * c_k                                      (prefix survival)
// The scheduler sorts all (request, position) candidates by survival and adds
// them greedily while the expected throughput J = SPS(N) * A / N keeps rising,
// stopping at the first candidate that does not raise it (non-anticipation).
//
//   confidence_kernel  one warp per (b, k): two dot products (d and r long,
//                      16-byte loads, fp32 accumulation of exact bf16
//                      products), sigmoid. w_h . h_k reads only inputs of the
//                      cycle and runs before the programmatic-launch wait, so
//                      it overlaps the end of the draft.
//   schedule_kernel    one CTA: survival cumprod; a histogram of the
//                      survivals selects the largest run of top bins with at
//                      most 4B (then 1024) candidates, a prefix of the sorted
//                      order, which alone is sorted (a merge tree over the
//                      requests' runs, each already in order) when the early
//                      stop falls inside it; otherwise the full bitonic sort of 64-bit keys
//                      (survival descending, then k, then b): for 2048-8192
//                      keys each thread holds E = B*K/1024 of them in
//                      registers (small strides in registers, middle ones by
//                      warp shuffles, only strides >= 32E in shared memory);
//                      otherwise in shared memory, stages of stride <= 32
//                      synchronising one warp only;
//                      double-float prefix scan of A, first drop of J tested
//                      without division: J' > J <=> SPS(N+1) (A+s) N > SPS(N) A (N+1).
//                      (double precision runs at a small fraction of the float
//                      rate here, and this kernel is one CTA on one SM)
#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace ds {

namespace {

template <typename Tin>
__device__ __forceinline__ float dot_warp(const Tin* a, const Tin* w, int n, int lane) {
  float acc = 0.f;
  int i = lane * 8;
  for (; i + 3 * 256 < n; i += 4 * 256) {  // four groups of loads in flight
    float x[4][8], y[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      load8(a + i + u * 256, x[u]);
      load8(w + i + u * 256, y[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc = __fmaf_rn(x[u][q], y[u][q], acc);
  }
  for (; i < n; i += 32 * 8) {
    float x[8], y[8];
    load8(a + i, x);
    load8(w + i, y);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = __fmaf_rn(x[q], y[q], acc);
  }
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  return acc;
}

// w_h . h_k for bf16: w_h staged once per CTA in shared memory, eight 16-byte
// loads of h in flight per lane, two accumulators (exact bf16 products).
__device__ __forceinline__ float dot_h_bf16(const __nv_bfloat16* a, const __nv_bfloat16* sw, int n,
                                            int lane) {
  float acc0 = 0.f, acc1 = 0.f;
  int i = lane * 8;
  for (; i + 7 * 256 < n; i += 8 * 256) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldg(reinterpret_cast<const uint4*>(a + i + u * 256));
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 w = *reinterpret_cast<const uint4*>(sw + i + u * 256);
      const uint32_t xv[4] = {v[u].x, v[u].y, v[u].z, v[u].w}, wv[4] = {w.x, w.y, w.z, w.w};
      float acc = (u & 1) ? acc1 : acc0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc = __fmaf_rn(__uint_as_float(xv[q] << 16), __uint_as_float(wv[q] << 16), acc);
        acc = __fmaf_rn(__uint_as_float(xv[q] & 0xffff0000u), __uint_as_float(wv[q] & 0xffff0000u), acc);
      }
      if (u & 1) acc1 = acc; else acc0 = acc;
    }
  }
  for (; i < n; i += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a + i));
    const uint4 w = *reinterpret_cast<const uint4*>(sw + i);
    const uint32_t xv[4] = {v.x, v.y, v.z, v.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc0 = __fmaf_rn(__uint_as_float(xv[q] << 16), __uint_as_float(wv[q] << 16), acc0);
      acc0 = __fmaf_rn(__uint_as_float(xv[q] & 0xffff0000u), __uint_as_float(wv[q] & 0xffff0000u), acc0);
    }
  }
  float acc = __fadd_rn(acc0, acc1);
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  return acc;
}

// kStage: bf16 with w_h staged in shared memory (d up to kStageMaxD).
constexpr int kStageMaxD = 12288;

template <typename Tin, bool kStage>
__global__ void __launch_bounds__(256) confidence_kernel(SchedParams p) {
  extern __shared__ __align__(16) unsigned char conf_smem[];
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
  static_assert(!kStage || std::is_same<Tin, __nv_bfloat16>::value, "staging is bf16 only");
  sm100::pdl_launch_dependents();
  // w_h and h are inputs of the cycle (no kernel of the cycle writes them), so
  // w_h . h_k runs before the wait and overlaps the end of the draft.
  if constexpr (kStage) {
    const uint4* src = reinterpret_cast<const uint4*>(p.w_h);
    uint4* dst = reinterpret_cast<uint4*>(conf_smem);
    for (int i = threadIdx.x; i < p.d / 8; i += 256) dst[i] = __ldg(src + i);
    __syncthreads();
  }
  if (item >= p.B * p.K) {
    sm100::pdl_wait();
    return;
  }
  const Tin* h = reinterpret_cast<const Tin*>(p.h) + (size_t)item * p.d;
  float dh;
  if constexpr (kStage)
    dh = dot_h_bf16(h, reinterpret_cast<const __nv_bfloat16*>(conf_smem), p.d, lane);
  else
    dh = dot_warp(h, reinterpret_cast<const Tin*>(p.w_h), p.d, lane);
  sm100::pdl_wait();  // draft tokens come from the draft's kernels
  const int b = item / p.K, k = item - b * p.K;
  int prev = (k == 0) ? p.anchor[b] : p.draft_tokens[(size_t)b * p.K + k - 1];
  if (prev < 0 || prev >= p.V) {
    if (lane == 0) report(p.status, kErrBounds);
    prev = 0;
  }
  const Tin* E = reinterpret_cast<const Tin*>(p.E) + (size_t)prev * p.r;
  const float de = dot_warp(E, reinterpret_cast<const Tin*>(p.w_e), p.r, lane);
  if (lane == 0) {
    const float Tk = p.sts_temp[k];
    const float raw = __fadd_rn(__fadd_rn(dh, de), p.bias);
    const float logit = __fdiv_rn(raw, Tk);
    const float c = __frcp_rn(__fadd_rn(1.f, expf(-logit)));
    if (!(c == c) || !(Tk > 0.f)) report(p.status, kErrNonfinite);
    p.conf[item] = c;
    if (p.conf_logit) p.conf_logit[item] = raw;
  }
}

__device__ __forceinline__ float sps_at(const float* sps, int n_max, int n) {
  return sps[(n < n_max ? n : n_max) - 1];
}

__device__ __forceinline__ DF shfl_up_df2(DF v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// J = SPS(N) * A / N as a double (for the objective output only).
__device__ __forceinline__ double objective_of(float sps, DF A, int N) {
  const DF num = df_mul(DF{sps, 0.f}, A);
  const float q = __fdiv_rn(num.hi, (float)N);
  const DF back = df_mul(DF{q, 0.f}, DF{(float)N, 0.f});
  const DF res = df_add(num, DF{-back.hi, -back.lo});
  const float ql = __fdiv_rn(res.hi, (float)N);
  return (double)q + (double)ql;
}

// J(N+1, A+s) > J(N, A) without division (all factors positive).
__device__ __forceinline__ bool gains(float sps1, float sps0, DF A, float s, int N) {
  const DF A1 = df_add(A, DF{s, 0.f});
  const DF lhs = df_mul(df_mul(DF{sps1, 0.f}, A1), DF{(float)N, 0.f});
  const DF rhs = df_mul(df_mul(DF{sps0, 0.f}, A), DF{(float)(N + 1), 0.f});
  return lhs.hi > rhs.hi || (lhs.hi == rhs.hi && lhs.lo > rhs.lo);
}

constexpr int kSchedThreads = 1024;

// Shared-memory position of key w: the low four bits are XORed with bits 4-7,
// so that a warp reading 64-bit words either contiguously or E words apart
// (the blocked layout of bitonic_regs) touches each bank pair once per phase.
// Positions stay inside w's own 16-word block.
__device__ __forceinline__ int swz(int w) { return w ^ ((w >> 4) & 15); }

// One compare-exchange of pair i at the given stride, ascending within blocks
// of `size` keys whose index has the `size` bit clear.
__device__ __forceinline__ void bitonic_cx(unsigned long long* keys, int i, int stride, int size) {
  const int lo = 2 * i - (i & (stride - 1));
  const int hi = lo + stride;
  const bool asc = (lo & size) == 0;
  const unsigned long long a = keys[swz(lo)], c = keys[swz(hi)];
  if ((a > c) == asc) {
    keys[swz(lo)] = c;
    keys[swz(hi)] = a;
  }
}

// Sort key of candidate i = b*K + k: survival descending, then k, then b;
// padding (i >= n) sorts last.
__device__ __forceinline__ unsigned long long sched_key(const SchedParams& p, int i, int n, int K) {
  if (i >= n) return ~0ull;
  const int b = i / K, k = i - b * K;
  const uint32_t hi = 0xffffffffu - __float_as_uint(fmaxf(p.survival[i], 0.f));
  return ((unsigned long long)hi << 32) | ((unsigned long long)k << 16) | (unsigned long long)b;
}

// Bitonic sort of n_pad = E * kSchedThreads keys with thread t holding keys
// t*E .. t*E + E - 1 in registers (built there from the survivals): strides below E are exchanged in registers,
// strides E .. 32E - 1 between the lanes of a warp (shuffles), and only
// strides of 32E and more through shared memory. Same network, same result
// as the shared-memory sort; the keys end sorted in `keys`.
template <int E>
__device__ void bitonic_regs(unsigned long long* keys, int n_pad, int tid, const SchedParams& p, int n,
                             int K) {
  unsigned long long v[E];
#pragma unroll
  for (int j = 0; j < E; ++j) v[j] = sched_key(p, tid * E + j, n, K);
  for (int size = 2; size <= n_pad; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * E) {
#pragma unroll
      for (int j = 0; j < E; ++j) keys[swz(tid * E + j)] = v[j];
      __syncthreads();
      for (; stride >= 32 * E; stride >>= 1) {
        for (int i = tid; i < (n_pad >> 1); i += kSchedThreads) bitonic_cx(keys, i, stride, size);
        __syncthreads();
      }
#pragma unroll
      for (int j = 0; j < E; ++j) v[j] = keys[swz(tid * E + j)];
    }
    for (; stride >= E; stride >>= 1) {
      const int d = stride / E;  // partner lane distance
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int i = tid * E + j;
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[j], d);
        const bool keep_min = ((i & stride) == 0) == ((i & size) == 0);
        v[j] = keep_min ? (o < v[j] ? o : v[j]) : (o > v[j] ? o : v[j]);
      }
    }
#pragma unroll
    for (int st = E / 2; st > 0; st >>= 1) {
      if (st <= stride) {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          if ((j & st) == 0) {
            const bool asc = ((tid * E + j) & size) == 0;
            const unsigned long long a = v[j], c = v[j | st];
            if ((a > c) == asc) {
              v[j] = c;
              v[j | st] = a;
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < E; ++j) keys[swz(tid * E + j)] = v[j];
  __syncthreads();
}

// ---- select before sort ----------------------------------------------------
//
// The early stop reads the sorted order only up to its first drop, usually a
// few hundred of the B*K candidates. A histogram of the survivals' float bits
// (bin = bits >> 20: exponent and three mantissa bits, s in [0, 1] gives bins
// below 1024) picks the largest run of top bins holding at most kSelCap
// candidates. Every candidate in those bins has a larger survival than every
// candidate outside them, so they are exactly the first m_sel keys of the full
// order: sorting only them gives the same first m_sel keys, the same prefix
// sums and the same decisions. If the scan finds no drop among them (and they
// are not all the candidates), the full sort runs instead.
constexpr int kSelCap = kSchedThreads;  // candidates sorted after the selection (one per thread)
// The merge tree's two buffers of kSelCap keys follow the n_pad keys of the
// full sort in dynamic shared memory.
constexpr int kMergeOff = 16384;  // the largest n_pad (B * K <= 16384)
constexpr int kSelBins = 1024;
static_assert(kSelBins == kSchedThreads, "one histogram bin per thread in the selection scan");

__device__ __forceinline__ int surv_bin(float s) {
  return (int)(__float_as_uint(fminf(fmaxf(s, 0.f), 1.f)) >> 20);  // 0 .. 1016
}

// Bitonic sort of the first P (a power of two, 1..kSchedThreads) keys, one per
// thread: strides below 32 by warp shuffles, the others through shared memory
// with a barrier over the P sorting threads only (named barrier 1).
__device__ void bitonic_one(unsigned long long* keys, int P, int tid) {
  const bool own = tid < P;
  const int Pw = P < 32 ? 32 : P;  // whole warps take part in the shuffles
  unsigned long long v = own ? keys[swz(tid)] : ~0ull;
  for (int size = 2; size <= P && tid < Pw; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32) {  // P >= 64: whole warps
      keys[swz(tid)] = v;
      sm100::named_bar_sync(1, P);
      for (; stride >= 32; stride >>= 1) {
        if (tid < (P >> 1)) bitonic_cx(keys, tid, stride, size);
        sm100::named_bar_sync(1, P);
      }
      v = keys[swz(tid)];
    }
    for (; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_min = ((tid & stride) == 0) == ((tid & size) == 0);
      v = keep_min ? (o < v ? o : v) : (o > v ? o : v);
    }
  }
  if (own) keys[swz(tid)] = v;
  __syncthreads();
}

// The selected keys, sorted by a merge tree over the requests: request b's
// selected candidates (positions 0 .. L_b - 1, already in key order since
// survival does not rise with k) sit at off[b] .. off[b + 1] - 1 of `a`;
// level l merges the runs of request groups 2j and 2j + 1 of size 2^l, each
// key finding its place as (its index in its own run) + (the number of keys
// of the partner run below it, by binary search; keys are unique). Bp: the
// request count rounded up to a power of two (off[b] = m for b >= B). The
// result ends in `a` or `t`: the returned pointer.
__device__ unsigned long long* merge_tree(unsigned long long* a, unsigned long long* t, const int* off,
                                          int Bp, int m, int tid) {
  for (int l = 0; (1 << l) < Bp; ++l) {
    for (int i = tid; i < m; i += kSchedThreads) {
      const unsigned long long x = a[i];
      const int g = (int)(x & 0xffff) >> l;
      const int own_lo = off[g << l];
      const int pg = g ^ 1;
      int lo = off[pg << l], hi = off[(pg + 1) << l];
      while (lo < hi) {  // first partner key above x
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1; else hi = mid;
      }
      const int p_lo = off[pg << l];
      const int m_lo = off[(g >> 1) << (l + 1)];
      t[m_lo + (i - own_lo) + (lo - p_lo)] = x;
    }
    __syncthreads();
    unsigned long long* s = a;
    a = t;
    t = s;
  }
  return a;
}

// Scan of the first cnt sorted keys: A_m = B + the sum of the first m
// survivals (double-float; each thread owns a contiguous run [i0, i1)), and the
// first m at which adding candidate m does not raise J (cnt if none).
struct DropScan {
  int M, i0, i1;
  DF excl;  // the sum of the survivals before i0
};

__device__ DropScan scan_first_drop(const unsigned long long* keys, int cnt, const SchedParams& p,
                                    DF* wsum, int* red, int tid) {
  const int lane = tid & 31, wid = tid >> 5;
  const int B = p.B;
  DropScan r;
  const int per = (cnt + kSchedThreads - 1) / kSchedThreads;
  r.i0 = min(cnt, tid * per);
  r.i1 = min(cnt, r.i0 + per);
  DF local = {0.f, 0.f};
  for (int i = r.i0; i < r.i1; ++i)
    local = df_add(local, DF{__uint_as_float(0xffffffffu - (uint32_t)(keys[swz(i)] >> 32)), 0.f});
  // block exclusive scan of `local`
  DF incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const DF v = shfl_up_df2(incl, o);
    if (lane >= o) incl = df_add(v, incl);
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    DF v = wsum[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const DF u = shfl_up_df2(v, o);
      if (lane >= o) v = df_add(u, v);
    }
    wsum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  DF excl = shfl_up_df2(incl, 1);
  if (lane == 0) excl = DF{0.f, 0.f};
  if (wid > 0) excl = df_add(wsum[wid - 1], excl);
  r.excl = excl;

  int first_drop = INT_MAX;
  DF a_prev = df_add(DF{(float)B, 0.f}, excl);
  for (int i = r.i0; i < r.i1; ++i) {
    const float sv = __uint_as_float(0xffffffffu - (uint32_t)(keys[swz(i)] >> 32));
    const int nb = B + i;  // verified tokens before adding candidate i
    if (!gains(sps_at(p.sps, p.n_max, nb + 1), sps_at(p.sps, p.n_max, nb), a_prev, sv, nb)) {
      first_drop = i;
      break;
    }
    a_prev = df_add(a_prev, DF{sv, 0.f});
  }
  for (int o = 16; o > 0; o >>= 1) first_drop = min(first_drop, __shfl_xor_sync(0xffffffffu, first_drop, o));
  __syncthreads();  // red[] and wsum[] may still be read by a previous scan's callers
  if (lane == 0) red[wid] = first_drop;
  __syncthreads();
  if (wid == 0) {
    int M = red[lane];
    for (int o = 16; o > 0; o >>= 1) M = min(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[0] = M;
  }
  __syncthreads();
  r.M = (red[0] == INT_MAX) ? cnt : red[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(SchedParams p) {
  extern __shared__ unsigned long long keys[];
  __shared__ DF wsum[32];
  __shared__ int red[32];
  __shared__ int hist[kSelBins];
  __shared__ int roff[kSchedThreads + 1];  // merge tree: run offsets of the requests
  __shared__ int s_budget, s_cycle, s_cnt, s_msel;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int B = p.B, K = p.K, n = B * K;
  sm100::pdl_wait();  // confidences come from the confidence kernel
  // asynchronous mode: this cycle's budget, written two cycles ago
  if (tid == 0) {
    s_cycle = (p.mode == DS_SCHED_ASYNC) ? p.budget_ring[2] : 0;
    s_budget = (p.mode == DS_SCHED_ASYNC) ? p.budget_ring[s_cycle & 1] : 0;
    s_cnt = 0;
  }
  for (int j = tid; j < kSelBins; j += kSchedThreads) hist[j] = 0;
  const bool greedy = p.mode == DS_SCHED_GREEDY_EARLYSTOP || p.mode == DS_SCHED_ASYNC;
  __syncthreads();

  // survival (sequential over k per request, fp32); the selection's histogram
  // of the survivals' bins
  for (int b = tid; b < B; b += kSchedThreads) {
    float s = 1.f;
    int L = 0;
    for (int k0 = 0; k0 < K; k0 += 16) {  // a chunk's loads in flight together
      float c[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) c[u] = (k0 + u < K) ? p.conf[(size_t)b * K + k0 + u] : 1.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int k = k0 + u;
        if (k < K) {
          s = s * c[u];
          p.survival[(size_t)b * K + k] = s;
          if (p.mode == DS_SCHED_THRESHOLD && s >= p.threshold && L == k) L = k + 1;
          if (greedy) atomicAdd(&hist[surv_bin(s)], 1);
        }
      }
    }
    p.sched_len[b] = (p.mode == DS_SCHED_FIXED_K) ? K : (p.mode == DS_SCHED_THRESHOLD ? L : 0);
  }
  __syncthreads();
  if (p.mode != DS_SCHED_GREEDY_EARLYSTOP && p.mode != DS_SCHED_ASYNC) {
    // objective of the fixed selection: block sums of N and A (double-float)
    int nsum = 0;
    DF a = {0.f, 0.f};
    for (int b = tid; b < B; b += kSchedThreads) {
      const int L = p.sched_len[b];
      nsum += L;
      for (int k = 0; k < L; ++k) a = df_add(a, DF{p.survival[(size_t)b * K + k], 0.f});
    }
    for (int o = 16; o > 0; o >>= 1) {
      nsum += __shfl_xor_sync(0xffffffffu, nsum, o);
      a = df_add(a, DF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)});
    }
    if (lane == 0) {
      red[wid] = nsum;
      wsum[wid] = a;
    }
    __syncthreads();
    if (tid == 0) {
      int N = B;
      DF A = {(float)B, 0.f};
      for (int w = 0; w < kSchedThreads / 32; ++w) {
        N += red[w];
        A = df_add(A, wsum[w]);
      }
      p.objective[0] = objective_of(sps_at(p.sps, p.n_max, N), A, N);
    }
    return;
  }

  // ---- select: the top bins holding at most kSelCap candidates ----
  // thread t counts the candidates in bins >= kSelBins - 1 - t (inclusive scan)
  int hv = hist[kSelBins - 1 - tid];
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, hv, o);
    if (lane >= o) hv += u;
  }
  if (lane == 31) red[wid] = hv;
  __syncthreads();
  if (wid == 0) {
    int v = red[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    red[lane] = v;
  }
  __syncthreads();
  if (wid > 0) hv += red[wid - 1];
  DropScan ds;
  ds.M = -1;
  int m_prev = 0;
  // first a selection sized to the usual early stop (a few candidates per
  // request: at most 4B, from 256), then at most kSelCap
  int cap0 = 256;
  while (cap0 < 4 * B && cap0 < kSelCap) cap0 <<= 1;
  for (int cap = cap0; cap <= kSelCap && ds.M < 0; cap *= 2) {
  const int nfit = __syncthreads_count(hv <= cap);  // the counts rise with t
  if (tid == nfit - 1) s_msel = hv;
  if (nfit == 0 && tid == 0) s_msel = 0;
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  const int m_sel = s_msel;
  const int bin_lo = kSelBins - nfit;
  if (m_sel > m_prev && (m_sel == n || p.mode != DS_SCHED_ASYNC || s_budget <= m_sel)) {
    m_prev = m_sel;
    // a request's selected candidates are a prefix of its positions (survival
    // does not rise with k): its thread finds the prefix length L_b,
    // recomputing the same products from the confidences it read before
    const bool tree = B <= kSchedThreads;  // merge tree over the requests
    int Lb = 0;
    for (int b = tid; b < B; b += kSchedThreads) {
      const float* cb = p.conf + (size_t)b * K;
      int L = 0;
      float s = 1.f;
      while (L < K) {
        const float sn = s * cb[L];
        if (surv_bin(sn) < bin_lo) break;
        s = sn;
        ++L;
      }
      Lb = L;
      if (!tree && L > 0) {  // slots in any order: sorted by the network next
        const int base = atomicAdd(&s_cnt, L);
        s = 1.f;
        for (int k = 0; k < L; ++k) {
          s = s * cb[k];
          keys[swz(base + k)] = ((unsigned long long)(0xffffffffu - __float_as_uint(fmaxf(s, 0.f))) << 32) |
                                ((unsigned long long)k << 16) | (unsigned long long)b;
        }
      }
    }
    if (tree) {
      int Bp = 1;
      while (Bp < B) Bp <<= 1;
      // run offsets: exclusive scan of L_b over the (padded) requests
      int v = Lb;
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (lane == 31) red[wid] = v;
      __syncthreads();
      if (wid == 0) {
        int w = red[lane];
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += u;
        }
        red[lane] = w;
      }
      __syncthreads();
      const int incl = v + (wid > 0 ? red[wid - 1] : 0);
      if (tid < Bp) roff[tid] = incl - Lb;
      if (tid == Bp - 1) roff[Bp] = incl;  // = m_sel
      __syncthreads();
      unsigned long long* ma = keys + kMergeOff;
      unsigned long long* mb = ma + kSelCap;
      if (tid < B && Lb > 0) {
        const float* cb = p.conf + (size_t)tid * K;
        float s = 1.f;
        for (int k = 0; k < Lb; ++k) {
          s = s * cb[k];
          ma[roff[tid] + k] = ((unsigned long long)(0xffffffffu - __float_as_uint(fmaxf(s, 0.f))) << 32) |
                              ((unsigned long long)k << 16) | (unsigned long long)tid;
        }
      }
      __syncthreads();
      const unsigned long long* sorted = merge_tree(ma, mb, roff, Bp, m_sel, tid);
      for (int i = tid; i < m_sel; i += kSchedThreads) keys[swz(i)] = sorted[i];
      __syncthreads();
    } else {
      __syncthreads();
      int P = 1;
      while (P < m_sel) P <<= 1;
      for (int i = m_sel + tid; i < P; i += kSchedThreads) keys[swz(i)] = ~0ull;  // padding sorts last
      __syncthreads();
      bitonic_one(keys, P, tid);
    }
    const DropScan sel_scan = scan_first_drop(keys, m_sel, p, wsum, red, tid);
    // resolved when the early stop falls inside the selection (or it is everything)
    if (sel_scan.M < m_sel || m_sel == n) ds = sel_scan;
  }
  }
  if (ds.M < 0) {
    int n_pad = 1;
    while (n_pad < n) n_pad <<= 1;
    // Bitonic network: registers and shuffles for 2048 to 8192 keys; otherwise
    // in shared memory, where a compare-exchange of stride <= 32 pairs keys
    // inside the 64-key window of the warp that owns pairs [32j, 32j + 32), so
    // those stages synchronise the warp only.
    if (n_pad == 2 * kSchedThreads) {
      bitonic_regs<2>(keys, n_pad, tid, p, n, K);
    } else if (n_pad == 4 * kSchedThreads) {
      bitonic_regs<4>(keys, n_pad, tid, p, n, K);
    } else if (n_pad == 8 * kSchedThreads) {
      bitonic_regs<8>(keys, n_pad, tid, p, n, K);
    } else {
      for (int i = tid; i < n_pad; i += kSchedThreads) keys[swz(i)] = sched_key(p, i, n, K);
      __syncthreads();
      const int half = n_pad >> 1;
      const int local_sizes = n_pad < 64 ? n_pad : 64;
      for (int base = wid * 32; base < half; base += kSchedThreads) {
        for (int size = 2; size <= local_sizes; size <<= 1)
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (base + lane < half) bitonic_cx(keys, base + lane, stride, size);
            __syncwarp();
          }
      }
      __syncthreads();
      for (int size = 128; size <= n_pad; size <<= 1) {
        for (int stride = size >> 1; stride > 32; stride >>= 1) {
          for (int i = tid; i < half; i += kSchedThreads) bitonic_cx(keys, i, stride, size);
          __syncthreads();
        }
        for (int base = wid * 32; base < half; base += kSchedThreads)
          for (int stride = 32; stride > 0; stride >>= 1) {
            if (base + lane < half) bitonic_cx(keys, base + lane, stride, size);
            __syncwarp();
          }
        __syncthreads();
      }
    }
    ds = scan_first_drop(keys, n, p, wsum, red, tid);
  }

  int M = ds.M;
  if (p.mode == DS_SCHED_ASYNC) {
    // dynamic top-k: take the budget's worth of the current order; store this
    // cycle's early-stop count as the budget of cycle + 2
    if (tid == 0) {
      p.budget_ring[s_cycle & 1] = M;
      p.budget_ring[2] = s_cycle + 1;
    }
    M = min(max(s_budget, 0), n);
  }

  for (int i = tid; i < M; i += kSchedThreads) {
    const unsigned long long key = keys[swz(i)];
    const int k = (int)((key >> 16) & 0xffff), b = (int)(key & 0xffff);
    atomicMax(&p.sched_len[b], k + 1);
  }
  // objective at the chosen set: thread owning item M-1 (or thread 0 for M = 0)
  if (M == 0) {
    if (tid == 0) p.objective[0] = (double)sps_at(p.sps, p.n_max, B);
  } else if (M - 1 >= ds.i0 && M - 1 < ds.i1) {
    DF a = df_add(DF{(float)B, 0.f}, ds.excl);
    for (int i = ds.i0; i < M; ++i)
      a = df_add(a, DF{__uint_as_float(0xffffffffu - (uint32_t)(keys[swz(i)] >> 32)), 0.f});
    p.objective[0] = objective_of(sps_at(p.sps, p.n_max, B + M), a, B + M);
  }
}

// Launch with programmatic stream serialization: the kernel's prologue may
// overlap its predecessor; it calls griddepcontrol.wait before reading what
// earlier kernels wrote.
template <typename Kern>
cudaError_t launch_pdl(Kern kernel, int grid, int block, size_t smem, cudaStream_t s, SchedParams p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

size_t schedule_smem_bytes(int32_t B, int32_t K) {
  (void)B;
  (void)K;
  return (size_t)(kMergeOff + 2 * kSelCap) * sizeof(unsigned long long);
}

cudaError_t launch_confidence(const SchedParams& p, cudaStream_t s) {
  const int items = p.B * p.K;
  const int blocks = (items + 7) / 8;
  if (p.dtype == DS_BF16 && p.d <= kStageMaxD)  // at most 24 KB of w_h per CTA
    return launch_pdl(confidence_kernel<__nv_bfloat16, true>, blocks, 256,
                      sizeof(__nv_bfloat16) * (size_t)p.d, s, p);
  if (p.dtype == DS_BF16) return launch_pdl(confidence_kernel<__nv_bfloat16, false>, blocks, 256, 0, s, p);
  return launch_pdl(confidence_kernel<float, false>, blocks, 256, 0, s, p);
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(
      schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (kMergeOff + 2 * kSelCap) * 8);
  if (attr != cudaSuccess) return attr;
  return launch_pdl(schedule_kernel, 1, kSchedThreads, schedule_smem_bytes(p.B, p.K), s, p);
}

}  // namespace ds
