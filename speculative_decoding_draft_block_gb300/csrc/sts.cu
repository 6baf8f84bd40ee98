// Sequential Temperature Scaling (STS) fit on the GPU.
//
// [DSpark] 방법론 › 신뢰도 기반 검증 (STS paragraph): each confidence models
// P(position k accepted | every earlier position accepted), so the prefix
// acceptance probability is their cumulative product. STS calibrates that
// product left to right: at position k the temperatures of earlier positions
// stay fixed and a one-dimensional grid search picks the temperature with the
// lowest Expected Calibration Error (ECE). 주요 결과 reports raw ECE of 3-8 %
// brought to about 1 % by STS.
//
// With a_nk the raw confidence logit and y_nk the soft per-step label:
//     pred_n(T) = prod_{j<k} sigmoid(a_nj / T_j) * sigmoid(a_nk / T)
//     lab_n     = prod_{j<=k} y_nj
//     ECE(T)    = sum over n_bins equal-width bins of |sum_{n in bin} (lab_n - pred_n)| / N
// which is the usual sum over bins of (|bin| / N) * |mean label - mean prediction|.
// T_k is the first grid point with the smallest ECE.
//
// One launch per position: sts_fit_kernel, grid (chunks, ceil(G / 256)) in
// clusters of 8 CTAs along the chunks, 256 threads.
//   1. Thread t owns grid point g = 256 * blockIdx.y + t and two columns of
//      the CTA's shared histograms [copy][bin][256] (two copies: even and odd
//      samples, two independent add chains). The CTA stages 256 samples at a
//      time: the prefix prediction and prefix label (each one factor on from
//      the previous position's stored prefix), both pre-scaled by n_bins.
//   2. Every thread walks the staged samples and adds lab - pred (in units of
//      1 / n_bins) to the bin of pred.
//   3. The 8 CTAs of a cluster merge their histograms through distributed
//      shared memory in a fixed order; CTA rank r handles bins r, r + 8, ...
//      and adds each merged bin sum, as a 64-bit fixed-point integer
//      (2^-30 units), into the workspace histogram [bin][g] with an integer
//      atomic. Integer addition is associative, so the totals do not depend on
//      the order in which clusters arrive: the fit is deterministic.
//   4. The last CTA to finish (ticket counter, threadfence reduction) forms
//      ECE(g) for every grid point, takes the first arg-min, writes T_k, its
//      index, its ECE and the curve, and clears the histogram and the ticket
//      for the next position.
// Positions chain by programmatic dependent launch: the next launch zeroes
// its shared histograms and loads its grid point while this one finishes.
//
// Per evaluation: sigmoid(a / T) = 1 / (1 + 2^(a * c)), c = -log2(e) / T,
// with the ex2 and rcp approximations (two MUFU operations; relative error
// about 1e-6, and exact limits 0 and 1 for large |a / T|), then the bin by a
// round-down add against 2^23 (floor without a conversion instruction).
// Each evaluation is a handful of FP32 operations besides the two MUFU ones,
// so the kernel is bound by the MUFU rate (16 per SM per clock).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cg = cooperative_groups;

namespace ds {
namespace {

constexpr int kStsThreads = 256;
constexpr int kStsCluster = 8;
constexpr float kFix = 1073741824.0f;        // 2^30: fixed-point scale of the bin sums
constexpr float kFixInv = 9.31322574615478515625e-10f;  // 2^-30

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// sigmoid(a / T) with c = -log2(e) / T.
__device__ __forceinline__ float sts_sigmoid_c(float a, float c) {
  return rcp_approx(1.0f + ex2_approx(a * c));
}

__device__ __forceinline__ float neg_log2e_over(float T) { return __fdiv_rn(-kLog2eHi, T); }

// floor(x) for 0 <= x < 2^23, by a round-down add against 2^23.
__device__ __forceinline__ int floor_small(float x) {
  return __float_as_int(__fadd_rd(x, 8388608.0f)) - 0x4B000000;
}

__global__ void __cluster_dims__(kStsCluster, 1, 1) __launch_bounds__(kStsThreads, 5)
    sts_fit_kernel(StsParams p, int k) {
  extern __shared__ float4 sts_smem[];
  float4* samp = sts_smem;                                          // [256] {a, base*nb, lab*nb, -}
  float* hist = reinterpret_cast<float*>(sts_smem + kStsThreads);  // [2][n_bins][256]
  __shared__ float best_v[kStsThreads / 32];
  __shared__ int best_i[kStsThreads / 32];
  __shared__ int is_last;

  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const int g = blockIdx.y * kStsThreads + tid;
  const bool active = g < p.G;
  const int nb = p.n_bins;
  const float fnb = (float)nb;
  float* h0 = hist + tid;
  float* h1 = hist + nb * kStsThreads + tid;

  float c = 0.0f;
  if (active) {
    const float T = p.grid[g];
    if (!(T > 0.0f) || !isfinite(T)) {
      if (blockIdx.x == 0) report(p.status, kErrInvalidArg);
    } else {
      c = neg_log2e_over(T);
    }
  }
  for (int b = 0; b < nb; ++b) {
    h0[b * kStsThreads] = 0.0f;
    h1[b * kStsThreads] = 0.0f;
  }
  // Everything above reads only inputs; the previous position's launch may
  // still be finishing (programmatic dependent launch). From here on its
  // results (T_{k-1}, the prefixes, the cleared histogram) are needed.
  sm100::pdl_wait();
  float cprev = 0.0f;
  if (k > 0) cprev = neg_log2e_over(__ldcg(p.sts_temp + (k - 1)));

  const float* base_prev = p.base + (size_t)((k + 1) & 1) * p.N;
  const float* lab_prev = p.lab + (size_t)((k + 1) & 1) * p.N;
  float* base_cur = p.base + (size_t)(k & 1) * p.N;
  float* lab_cur = p.lab + (size_t)(k & 1) * p.N;

  const int n0 = min((int)blockIdx.x * p.chunk, p.N);
  const int n1 = min(n0 + p.chunk, p.N);
  for (int s0 = n0; s0 < n1; s0 += kStsThreads) {
    __syncthreads();  // the previous block of samples is no longer read
    const int n = s0 + tid;
    if (n < n1) {
      const float a = __ldg(p.logits + (size_t)n * p.K + k);
      const float y = __ldg(p.labels + (size_t)n * p.K + k);
      float base = 1.0f, lab = y;
      if (k > 0) {
        const float ap = __ldg(p.logits + (size_t)n * p.K + (k - 1));
        base = __ldcg(base_prev + n) * sts_sigmoid_c(ap, cprev);
        lab = __ldcg(lab_prev + n) * y;
      }
      if (blockIdx.y == 0) {
        if (!isfinite(a)) report(p.status, kErrNonfinite);
        if (!(y >= 0.0f && y <= 1.0f)) report(p.status, kErrInvalidArg);
        base_cur[n] = base;
        lab_cur[n] = lab;
      }
      samp[tid] = make_float4(a, base * fnb, lab * fnb, 0.0f);
    }
    __syncthreads();
    if (active) {
      const int cnt = min(kStsThreads, n1 - s0);
      int i = 0;
#pragma unroll 2
      for (; i + 1 < cnt; i += 2) {
        const float4 s = samp[i];
        const float4 t = samp[i + 1];
        const float ps = s.y * sts_sigmoid_c(s.x, c);  // prediction * n_bins, in [0, n_bins]
        const float pt = t.y * sts_sigmoid_c(t.x, c);
        const int bs = min(floor_small(ps), nb - 1) * kStsThreads;
        const int bt = min(floor_small(pt), nb - 1) * kStsThreads;
        const float vs = h0[bs];  // both loads before either store: two chains in flight
        const float vt = h1[bt];
        h0[bs] = vs + (s.z - ps);
        h1[bt] = vt + (t.z - pt);
      }
      if (i < cnt) {
        const float4 s = samp[i];
        const float ps = s.y * sts_sigmoid_c(s.x, c);
        h0[min(floor_small(ps), nb - 1) * kStsThreads] += s.z - ps;
      }
    }
  }
  __syncthreads();
  for (int b = 0; b < nb; ++b) h0[b * kStsThreads] += h1[b * kStsThreads];

  // Cluster merge: every CTA's histogram is complete before any is read.
  cluster.sync();
  const int rank = (int)cluster.block_rank();
  if (active) {
    for (int b = rank; b < nb; b += kStsCluster) {
      float v = 0.0f;
#pragma unroll
      for (int q = 0; q < kStsCluster; ++q) {
        const float* remote = cluster.map_shared_rank(hist, q);
        v += remote[b * kStsThreads + tid];
      }
      const long long fix = __float2ll_rn(v * kFix);  // units of 2^-30 / n_bins
      if (fix != 0)
        atomicAdd(reinterpret_cast<unsigned long long*>(p.hist64 + (size_t)b * p.G + g),
                  (unsigned long long)fix);
    }
  }
  // No CTA leaves while another may still read its shared memory.
  cluster.sync();
  // Every CTA of this launch is resident by now, so the next position's
  // launch may start its prologue; it waits for this grid before using results.
  sm100::pdl_launch_dependents();

  // Threadfence reduction: the last CTA to arrive sees every bin total. The
  // barrier orders this CTA's atomics before thread 0's fence and ticket.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned total = gridDim.x * gridDim.y;
    const bool last = (atomicAdd(p.ticket, 1u) == total - 1);
    if (last) __threadfence();
    is_last = last;
  }
  __syncthreads();
  if (!is_last) return;

  const float scale = kFixInv / (fnb * (float)p.N);
  float bv = __int_as_float(0x7f800000);
  int bi = 0x7fffffff;
  for (int gg = tid; gg < p.G; gg += kStsThreads) {
    unsigned long long acc = 0;  // sum of |bin total| in fixed point: below 2^63
    long long* col = p.hist64 + gg;
    for (int b0 = 0; b0 < nb; b0 += 8) {
      long long v[8];  // all loads of a batch are in flight before any use or store
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (b0 + j < nb) ? __ldcg(col + (size_t)(b0 + j) * p.G) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (b0 + j < nb) {
          acc += (unsigned long long)(v[j] < 0 ? -v[j] : v[j]);
          col[(size_t)(b0 + j) * p.G] = 0;  // cleared for the next position
        }
      }
    }
    const float e = (float)acc * scale;
    p.ece_all[gg] = e;
    if (p.ece_curve) p.ece_curve[(size_t)k * p.G + gg] = e;
    if (e < bv) {  // gg increases along the loop, so the first minimum stays
      bv = e;
      bi = gg;
    }
  }
  // first arg-min: smaller value, then smaller index
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov < bv || (ov == bv && oi < bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if ((tid & 31) == 0) {
    best_v[tid >> 5] = bv;
    best_i[tid >> 5] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    bv = best_v[0];
    bi = best_i[0];
    for (int w = 1; w < kStsThreads / 32; ++w) {
      if (best_v[w] < bv || (best_v[w] == bv && best_i[w] < bi)) {
        bv = best_v[w];
        bi = best_i[w];
      }
    }
    const int gi = bi;
    if (gi >= 0 && gi < p.G) {
      p.sts_temp[k] = p.grid[gi];
      p.grid_index[k] = gi;
      p.ece[k] = bv;
    } else {  // no finite ECE: only reachable after a reported input error
      p.sts_temp[k] = 1.0f;
      p.grid_index[k] = -1;
      p.ece[k] = __int_as_float(0x7fc00000);
      report(p.status, kErrNonfinite);
    }
    *p.ticket = 0u;  // ready for the next position
  }
}

}  // namespace

size_t sts_fit_smem_bytes(int32_t n_bins) {
  return sizeof(float4) * kStsThreads + 2 * sizeof(float) * (size_t)n_bins * kStsThreads;
}

cudaError_t launch_sts_fit(const StsParams& prm, cudaStream_t s) {
  StsParams p = prm;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // About four CTAs per SM in total, at least 64 samples per CTA, whole clusters.
  const int gy = (p.G + kStsThreads - 1) / kStsThreads;
  const int want = (4 * sms + gy - 1) / gy;
  const int by_n = (p.N + 63) / 64;
  int chunks = want < by_n ? want : by_n;
  chunks = ((chunks + kStsCluster - 1) / kStsCluster) * kStsCluster;
  p.n_chunks = chunks;
  p.chunk = (p.N + chunks - 1) / chunks;
  const size_t smem = sts_fit_smem_bytes(p.n_bins);
  e = cudaFuncSetAttribute(sts_fit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.ticket, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.hist64, 0, sizeof(long long) * (size_t)p.n_bins * p.G, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks, gy);
  cfg.blockDim = dim3(kStsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  for (int k = 0; k < p.K; ++k) {
    cfg.numAttrs = k > 0 ? 1 : 0;  // the first position follows the memsets in plain order
    e = cudaLaunchKernelEx(&cfg, sts_fit_kernel, p, k);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace ds
