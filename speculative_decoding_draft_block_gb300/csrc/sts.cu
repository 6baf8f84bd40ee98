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
// Two launches per position, both data-parallel over (samples, grid points):
//   sts_hist_kernel    grid (chunks, ceil(G / 256)), 256 threads. Thread t owns
//                      grid point g = 256 * blockIdx.y + t and one column of the
//                      CTA's shared histogram [bin][256]. The CTA stages 256
//                      samples at a time (prefix prediction and prefix label,
//                      each one factor on from the previous position's stored
//                      prefix), then every thread walks them and adds
//                      lab - pred to the bin of pred. Partial sums go to the
//                      workspace as [chunk][bin][g]: nothing is atomically
//                      accumulated, so results do not depend on scheduling.
//   sts_reduce_kernel  grid (ceil(G / 32), n_bins), 256 threads. Lane = grid
//                      point, warp w sums chunks w, w + 8, ... in double-float,
//                      the 8 warp sums combine in a fixed order. The last CTA
//                      to finish (ticket counter, threadfence reduction) forms
//                      ECE(g) over the bins, takes the first arg-min and writes
//                      T_k, its index, its ECE and the curve.
//
// Sigmoid: 1 / (1 + 2^(-t log2 e)) with the hardware exp2 and reciprocal
// approximations (two MUFU operations per evaluation, relative error about
// 1e-6 after clamping t to [-80, 80], where the tails are 0 and 1 to float32
// precision). That is far inside the bin width; the parity tests bound the
// effect of samples that sit on a bin edge.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace ds {
namespace {

constexpr int kStsThreads = 256;

__device__ __forceinline__ float sts_sigmoid(float t) {
  t = fminf(fmaxf(t, -80.0f), 80.0f);
  return __fdividef(1.0f, 1.0f + __expf(-t));
}

__global__ void __launch_bounds__(kStsThreads) sts_hist_kernel(StsParams p, int k) {
  extern __shared__ float4 sts_smem[];
  float4* samp = sts_smem;                                   // [256] {a, base, lab, -}
  float* hist = reinterpret_cast<float*>(sts_smem + kStsThreads);  // [n_bins][256]
  const int tid = threadIdx.x;
  const int g = blockIdx.y * kStsThreads + tid;
  const bool active = g < p.G;
  const int nb = p.n_bins;
  const float fnb = (float)nb;

  float invT = 0.0f;
  if (active) {
    const float T = p.grid[g];
    if (!(T > 0.0f) || !isfinite(T)) {
      if (blockIdx.x == 0) report(p.status, kErrInvalidArg);
    } else {
      invT = 1.0f / T;
    }
  }
  float invTprev = 0.0f;
  if (k > 0) invTprev = 1.0f / __ldcg(p.sts_temp + (k - 1));
  for (int b = 0; b < nb; ++b) hist[b * kStsThreads + tid] = 0.0f;

  const float* base_prev = p.base + (size_t)((k + 1) & 1) * p.N;
  const float* lab_prev = p.lab + (size_t)((k + 1) & 1) * p.N;
  float* base_cur = p.base + (size_t)(k & 1) * p.N;
  float* lab_cur = p.lab + (size_t)(k & 1) * p.N;

  const int n0 = blockIdx.x * p.chunk;
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
        base = __ldcg(base_prev + n) * sts_sigmoid(ap * invTprev);
        lab = __ldcg(lab_prev + n) * y;
      }
      if (blockIdx.y == 0) {
        if (!isfinite(a)) report(p.status, kErrNonfinite);
        if (!(y >= 0.0f && y <= 1.0f)) report(p.status, kErrInvalidArg);
        base_cur[n] = base;
        lab_cur[n] = lab;
      }
      samp[tid] = make_float4(a, base, lab, 0.0f);
    }
    __syncthreads();
    if (active) {
      const int cnt = min(kStsThreads, n1 - s0);
      float* col = hist + tid;
#pragma unroll 4
      for (int i = 0; i < cnt; ++i) {
        const float4 s = samp[i];
        const float pred = s.y * sts_sigmoid(s.x * invT);
        const int bin = min(max((int)(pred * fnb), 0), nb - 1);
        col[bin * kStsThreads] += s.z - pred;
      }
    }
  }
  __syncthreads();
  if (active) {
    float* out = p.part + (size_t)blockIdx.x * nb * p.G + g;
    for (int b = 0; b < nb; ++b) out[(size_t)b * p.G] = hist[b * kStsThreads + tid];
  }
}

__global__ void __launch_bounds__(kStsThreads) sts_reduce_kernel(StsParams p, int k) {
  __shared__ DF part8[8][32];
  __shared__ float best_v[kStsThreads];
  __shared__ int best_i[kStsThreads];
  __shared__ int is_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x * 32 + lane;
  const int bin = blockIdx.y;
  DF acc{0.0f, 0.0f};
  if (g < p.G) {
    const float* src = p.part + (size_t)bin * p.G + g;
    const size_t stride = (size_t)p.n_bins * p.G;
    int c = warp;
    for (; c + 24 < p.n_chunks; c += 32) {
      const float v0 = __ldcg(src + (size_t)c * stride);
      const float v1 = __ldcg(src + (size_t)(c + 8) * stride);
      const float v2 = __ldcg(src + (size_t)(c + 16) * stride);
      const float v3 = __ldcg(src + (size_t)(c + 24) * stride);
      df_accumulate(acc, v0);
      df_accumulate(acc, v1);
      df_accumulate(acc, v2);
      df_accumulate(acc, v3);
    }
    for (; c < p.n_chunks; c += 8) df_accumulate(acc, __ldcg(src + (size_t)c * stride));
  }
  part8[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && g < p.G) {
    DF s = part8[0][lane];
    for (int w = 1; w < 8; ++w) s = df_add(s, part8[w][lane]);
    p.binsum[(size_t)bin * p.G + g] = s.hi + s.lo;
  }
  // Threadfence reduction: the last CTA to arrive sees every bin sum.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned total = gridDim.x * gridDim.y;
    is_last = (atomicAdd(p.ticket, 1u) == total - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  const float invN = 1.0f / (float)p.N;
  float bv = __int_as_float(0x7f800000);
  int bi = 0x7fffffff;
  for (int gg = tid; gg < p.G; gg += kStsThreads) {
    DF e{0.0f, 0.0f};
    for (int b = 0; b < p.n_bins; ++b) df_accumulate(e, fabsf(__ldcg(p.binsum + (size_t)b * p.G + gg)));
    const float v = (e.hi + e.lo) * invN;
    p.ece_all[gg] = v;
    if (p.ece_curve) p.ece_curve[(size_t)k * p.G + gg] = v;
    if (v < bv) {  // gg increases along the loop, so the first minimum stays
      bv = v;
      bi = gg;
    }
  }
  best_v[tid] = bv;
  best_i[tid] = bi;
  __syncthreads();
  for (int s = kStsThreads / 2; s > 0; s >>= 1) {
    if (tid < s) {
      const float ov = best_v[tid + s];
      const int oi = best_i[tid + s];
      if (ov < best_v[tid] || (ov == best_v[tid] && oi < best_i[tid])) {
        best_v[tid] = ov;
        best_i[tid] = oi;
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    const int gi = best_i[0];
    if (gi >= 0 && gi < p.G) {
      p.sts_temp[k] = p.grid[gi];
      p.grid_index[k] = gi;
      p.ece[k] = best_v[0];
    } else {  // every ECE was NaN: only reachable after a reported input error
      p.sts_temp[k] = 1.0f;
      p.grid_index[k] = -1;
      p.ece[k] = __int_as_float(0x7fc00000);
      report(p.status, kErrNonfinite);
    }
    *p.ticket = 0u;  // ready for the next position
  }
}

}  // namespace

int32_t sts_num_chunks(int32_t N) {
  const int32_t blocks = (N + kStsThreads - 1) / kStsThreads;
  return blocks < kStsMaxChunks ? blocks : kStsMaxChunks;
}

int32_t sts_chunk(int32_t N) {
  const int32_t c = sts_num_chunks(N);
  return (N + c - 1) / c;
}

size_t sts_hist_smem_bytes(int32_t n_bins) {
  return sizeof(float4) * kStsThreads + sizeof(float) * (size_t)n_bins * kStsThreads;
}

cudaError_t launch_sts_fit(const StsParams& p, cudaStream_t s) {
  const size_t smem = sts_hist_smem_bytes(p.n_bins);
  cudaError_t e = cudaFuncSetAttribute(sts_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.ticket, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const dim3 hist_grid(p.n_chunks, (p.G + kStsThreads - 1) / kStsThreads);
  const dim3 red_grid((p.G + 31) / 32, p.n_bins);
  for (int k = 0; k < p.K; ++k) {
    sts_hist_kernel<<<hist_grid, kStsThreads, smem, s>>>(p, k);
    sts_reduce_kernel<<<red_grid, kStsThreads, 0, s>>>(p, k);
  }
  return cudaGetLastError();
}

}  // namespace ds
