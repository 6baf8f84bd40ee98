// Row sampling kernels shared by the draft block and the final draw of verify.
//
// DSpark summary page, 방법론 › 반자기회귀 생성: at each block position the
// Markov head adds E[x_{k-1}] . P to the backbone's logits and the position is
// sampled conditioned on the previous token. One draw needs the whole
// vocabulary's normaliser before it can be located, so a step is two kernels:
//
//   sample_tile_kernel    grid (V/256, B/32). Each CTA forms the bias of a
//                         32-row x 256-token tile (A = gathered E rows, P tile
//                         streamed through shared memory), adds the base
//                         logits, and reduces every (row, 32-token chunk) to a
//                         record: the chunk's weight sum 2^(t - ref) as a
//                         double-float with an integer reference (sampling
//                         rows), or its largest logit (greedy rows). The V-wide
//                         logits never leave registers.
//   sample_locate_kernel  grid B. Combines a row's records (exact power-of-two
//                         rescale, double-float prefix), finds the chunk where
//                         the CDF crosses u*S, recomputes that chunk's 32
//                         weights with the identical arithmetic and picks the
//                         token: x = min{i : u*S < C_i}.
//
// The same two kernels draw the verify's residual (max(0, p - q)) and bonus
// (p_{L+1}) tokens from per-request descriptors.
#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "fastpath.cuh"
#include "locate.cuh"
#include "sampling.cuh"
#include "sm100.cuh"

namespace ds {

namespace {

constexpr int kThreads = 256;
constexpr int kPsStride = 8 * 36;  // 8 chunks of 32 floats padded to 36 (bank spread)

template <typename Tin>
__device__ __forceinline__ void load_chunk(const void* row, int col0, int n, float* out) {
  const Tin* p = reinterpret_cast<const Tin*>(row) + col0;
  if (n == 32) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) load8(p + j, out + j);
  } else {
    for (int j = 0; j < n; ++j) out[j] = to_f32(p[j]);
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) sample_tile_kernel(SampleParams p) {
  extern __shared__ float smem[];
  __shared__ RowCtx rows[kTileRows];
  __shared__ int any_bias;
  const int r = p.r, rs = r + 4;
  float* As = smem;
  float* Ps = smem + kTileRows * rs;
  const int tid = threadIdx.x;
  const int row0 = blockIdx.y * kTileRows;
  const int colbase = blockIdx.x * kTileCols;
  const Tin* E = reinterpret_cast<const Tin*>(p.E);
  const Tin* P = reinterpret_cast<const Tin*>(p.P);

  sm100::pdl_launch_dependents();
  sm100::pdl_wait();
  if (tid == 0) any_bias = 0;
  __syncthreads();
  if (tid < kTileRows) {
    rows[tid] = make_row_ctx<Tin>(p, row0 + tid);
    if (rows[tid].a_token >= 0) atomicOr(&any_bias, 1);
  }
  __syncthreads();

  const int rl = tid >> 3, cl = tid & 7;
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.f;

  if (any_bias) {
    for (int i = tid; i < kTileRows * r; i += kThreads) {
      const int rr = i / r, kk = i - rr * r;
      const int tok = rows[rr].a_token;
      As[rr * rs + kk] = tok >= 0 ? to_f32(E[(size_t)tok * r + kk]) : 0.f;
    }
    for (int kb = 0; kb < r; kb += 32) {
      const int kc = min(32, r - kb);
      __syncthreads();
      for (int i = tid; i < kc * kTileCols; i += kThreads) {
        const int kk = i >> 8, cc = i & 255;
        const int col = colbase + cc;
        const float v = col < p.V ? to_f32(P[(size_t)(kb + kk) * p.V + col]) : 0.f;
        Ps[kk * kPsStride + (cc >> 5) * 36 + (cc & 31)] = v;
      }
      __syncthreads();
      for (int kk = 0; kk < kc; ++kk) {
        const float a = As[rl * rs + kb + kk];
        const float4* pp = reinterpret_cast<const float4*>(Ps + kk * kPsStride + cl * 36);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 v = pp[j];
          acc[4 * j + 0] = __fmaf_rn(a, v.x, acc[4 * j + 0]);
          acc[4 * j + 1] = __fmaf_rn(a, v.y, acc[4 * j + 1]);
          acc[4 * j + 2] = __fmaf_rn(a, v.z, acc[4 * j + 2]);
          acc[4 * j + 3] = __fmaf_rn(a, v.w, acc[4 * j + 3]);
        }
      }
    }
  }

  const int row = row0 + rl;
  const int chunk = blockIdx.x * 8 + cl;
  const RowCtx& c = rows[rl];
  const bool active = row < p.B && chunk < p.n_chunks && c.mode != kSkip;
  ChunkRec rec = group_empty();
  if (active) {
    const int col0 = chunk * 32;
    const int n = min(32, p.V - col0);
    float z[32], t[32];
    if (c.zrow) load_chunk<Tin>(c.zrow, col0, n, z);
    if (c.trow) load_chunk<Tin>(c.trow, col0, n, t);
    if (n == 32)
      chunk_record<true>(c, F32Src{z}, acc, F32Src{t}, 32, col0, rec, p.status);
    else
      chunk_record<false>(c, F32Src{z}, acc, F32Src{t}, n, col0, rec, p.status);
    p.chunks[(size_t)chunk * p.B + row] = rec;
  }
  // group record of the row's 256 tokens: the 8 lanes of a row are adjacent
  ChunkRec g = rec;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    const ChunkRec other = shfl_xor_rec(g, o);
    // merge in token order so that equal greedy logits keep the first token
    if (cl & o) {
      ChunkRec lo = other;
      group_merge(c.mode, lo, g);
      g = lo;
    } else {
      group_merge(c.mode, g, other);
    }
  }
  if (cl == 0 && row < p.B && c.mode != kSkip)
    p.supers[(size_t)row * p.sup_stride + blockIdx.x] = g;
}

struct BlockSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// One CTA per row (see locate_row).
template <typename Tin>
__global__ void __launch_bounds__(kLocThreads) sample_locate_kernel(SampleParams p) {
  extern __shared__ ChunkRec sgrp[];
  __shared__ LocShared sm;
  sm100::pdl_launch_dependents();
  sm100::pdl_wait();
  locate_row<Tin>(p, blockIdx.x, p.step, threadIdx.x, sm, sgrp, BlockSync{});
}

}  // namespace

size_t sample_tile_smem_bytes(int32_t r) {
  return sizeof(float) * ((size_t)kTileRows * (r + 4) + (size_t)32 * kPsStride);
}

cudaError_t launch_sample_tile(const SampleParams& p, cudaStream_t s) {
  const size_t smem = sample_tile_smem_bytes(p.r);
  dim3 grid((p.V + kTileCols - 1) / kTileCols, (p.B + kTileRows - 1) / kTileRows);
  if (p.dtype == DS_BF16) {
    static cudaError_t attr = cudaFuncSetAttribute(
        sample_tile_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (attr != cudaSuccess) return attr;
    sample_tile_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(p);
  } else {
    static cudaError_t attr = cudaFuncSetAttribute(
        sample_tile_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (attr != cudaSuccess) return attr;
    sample_tile_kernel<float><<<grid, kThreads, smem, s>>>(p);
  }
  return cudaGetLastError();
}

size_t locate_smem_bytes(const SampleParams& p) { return (size_t)p.sup_stride * sizeof(ChunkRec); }

void simt_group_layout(SampleParams& p) {
  p.sup_stride = sup_stride_for(p.V);
  p.sup_nt = (p.V + kTileCols - 1) / kTileCols;
  p.sup_rows = kTileRows;
  p.sup_tiles = p.sup_nt * ((p.B + kTileRows - 1) / kTileRows);
  p.sup_groups = p.sup_tiles;
  p.sup_cpt = kTileCols / 32;
}

template <typename K, typename... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_sample_locate(const SampleParams& p, cudaStream_t s) {
  const size_t smem = locate_smem_bytes(p);
  if (p.dtype == DS_BF16) {
    static cudaError_t attr = cudaFuncSetAttribute(
        sample_locate_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(sample_locate_kernel<__nv_bfloat16>, dim3(p.B), dim3(kLocThreads), smem, s, p);
  }
  static cudaError_t attr = cudaFuncSetAttribute(
      sample_locate_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr != cudaSuccess) return attr;
  return launch_pdl(sample_locate_kernel<float>, dim3(p.B), dim3(kLocThreads), smem, s, p);
}

}  // namespace ds
