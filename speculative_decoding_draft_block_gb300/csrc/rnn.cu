// RNN head of the draft block: the gated state update on the tensor cores.
//
// [DSpark] 방법론 › 반자기회귀 생성: the RNN head keeps a recurrent state over
// the whole prefix drafted so far in the block. At every step it combines the
// current state, the embedding of the previous token and the backbone hidden
// state through a gated update. The state (size r, the Markov rank) replaces
// E[x_{k-1}] as the input of the logit projection P, so the draw of position k
// uses l_k = z_k + s_k . P with the same tile and locate kernels as the Markov
// head. The update is a GRU cell (reset gate on the recurrent product, as in
// cuDNN), gate rows in the order reset, update, new:
//     g_i = W_ih [e ; h] + b_ih,   g_h = W_hh s + b_hh
//     r = sigmoid(g_i^r + g_h^r),  u = sigmoid(g_i^u + g_h^u)
//     n = tanh(g_i^n + r * g_h^n), s' = (1 - u) * n + u * s
// with s_0 = 0, e = E[x_{k-1}] (x_0 = the anchor) and h = h_k. The state is
// stored as bfloat16, the model's storage type.
//
// Work split:
//   * W_ih[:, r:] . h_k + b_ih does not depend on drafted tokens: one GEMM over
//     all B*K positions per draft call (M = B*K, N = 3r, K = d);
//   * per position, one GEMM over the B requests with the packed step matrix
//     (N = 4r, K = 2r): for each block of 32 state units its 128 rows hold the
//     reset and update rows over [e ; s], the new-gate rows over e alone and
//     over s alone. The epilogue of a 128-column tile therefore holds all four
//     pre-activations of its 32 units and writes the new state directly.
//
// rnn_gemm_kernel: 128 x 128 output tile per CTA, K in steps of 64 (one
// 128-byte swizzled TMA box per operand per stage, 4 stages), warp 0 issues
// TMA, warp 1 (one elected thread) issues tcgen05.mma kind::f16 with the
// accumulator in TMEM, warps 2..5 read TMEM back (lane quarter = warp % 4) and
// run the epilogue. Every wait is bounded; on timeout the kernel records
// DS_ERR_TIMEOUT and unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace ds {
namespace {

using namespace sm100;

constexpr int kGemmThreads = 192;
constexpr int kGemmStages = 4;
constexpr uint32_t kBoxBytes = 128 * 128;               // 128 rows x 64 bf16
constexpr uint32_t kGemmStageBytes = 2 * kBoxBytes;     // A box + W box
constexpr size_t kGemmSmem = kGemmStages * kGemmStageBytes + 1024;  // + alignment slack
constexpr uint32_t kGemmTmemCols = 128;
constexpr uint32_t kGemmWaitPolls = 1u << 16;

struct GemmShared {
  uint64_t full[kGemmStages], empty[kGemmStages], done;
  uint32_t tmem_slot;
  int abort_flag;
};

__device__ __forceinline__ bool gemm_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < kGemmWaitPolls; ++i) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((i & 15) == 15 && *abort_flag) return false;
  }
  *abort_flag = 1;
  report(status, kErrTimeout);
  return false;
}

__device__ __forceinline__ float sigmoidf_acc(float x) { return 1.0f / (1.0f + expf(-x)); }

template <int kMode>
__global__ void __launch_bounds__(kGemmThreads, 1)
    rnn_gemm_kernel(const GemmParams g, const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmW) {
  extern __shared__ uint8_t raw[];
  __shared__ GemmShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base_addr = smem_u32(raw);
  uint8_t* smem = raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  const int nt = blockIdx.x, mt = blockIdx.y;
  const int nkb = g.Kd / 64;
  volatile int* abort_flag = &sh.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGemmStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem_slot, kGemmTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    pdl_wait();  // the A rows (and, for the update, the state) come from earlier kernels
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmW);
      const uint64_t pol = policy_evict_last();
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % kGemmStages;
        if (!gemm_wait(&sh.empty[st], ((kb / kGemmStages) & 1) ^ 1, abort_flag, g.status)) break;
        uint8_t* dst = smem + st * kGemmStageBytes;
        mbar_expect_tx(&sh.full[st], kGemmStageBytes);
        tma_load_2d(dst, &tmA, &sh.full[st], kb * 64, mt * 128, pol);
        tma_load_2d(dst + kBoxBytes, &tmW, &sh.full[st], kb * 64, nt * 128, pol);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 128, false, false);  // both operands K-major
      const uint64_t bits = smem_desc_bits(16, 1024, 2);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int st = kb % kGemmStages;
        ok = gemm_wait(&sh.full[st], (kb / kGemmStages) & 1, abort_flag, g.status);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* a = smem + st * kGemmStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, smem_desc(a + kk * 32, bits), smem_desc(a + kBoxBytes + kk * 32, bits), idesc,
                   (kb | kk) != 0 ? 1u : 0u);
        mma_commit(&sh.empty[st]);
      }
      if (ok) mma_commit(&sh.done);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int m = mt * 128 + q * 32 + lane;
    if (gemm_wait(&sh.done, 0, abort_flag, g.status)) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
      if (kMode == kGemmBias) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int n0 = nt * 128 + c * 32;
          if (m < g.M) {
            float* out = g.out + (size_t)m * g.N + n0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < g.N) out[j] = v[j] + __ldg(g.bias + n0 + j);
          }
        }
      } else {
        // columns 0..31 reset, 32..63 update, 64..95 new (input part),
        // 96..127 new (recurrent part) of units u0 .. u0 + 31
        float pr[32], pu[32], pnx[32], pns[32];
        tmem_ld32(taddr, pr);
        tmem_ld32(taddr + 32, pu);
        tmem_ld32(taddr + 64, pnx);
        tmem_ld32(taddr + 96, pns);
        const int b = m, r = g.r, u0 = nt * 32;
        if (b < g.M) {
          const float* gh = g.gh + ((size_t)b * g.K + (g.p - 1)) * 3 * r;
          const __nv_bfloat16* sp = g.s_prev + (size_t)b * 2 * r + u0;
          __nv_bfloat16* sn = g.s_next + (size_t)b * 2 * r + u0;
          __nv_bfloat16* so = g.states + ((size_t)b * g.K + (g.p - 1)) * r + u0;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            __nv_bfloat162 out2;
            float res[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int u = u0 + j + t;
              const float rg = sigmoidf_acc(pr[j + t] + __ldg(gh + u) + __ldg(g.b_hh + u));
              const float ug = sigmoidf_acc(pu[j + t] + __ldg(gh + r + u) + __ldg(g.b_hh + r + u));
              const float ng = tanhf(pnx[j + t] + __ldg(gh + 2 * r + u) +
                                     rg * (pns[j + t] + __ldg(g.b_hh + 2 * r + u)));
              const float s_old = __bfloat162float(sp[j + t]);
              res[t] = (1.0f - ug) * ng + ug * s_old;
            }
            out2.x = __float2bfloat16_rn(res[0]);
            out2.y = __float2bfloat16_rn(res[1]);
            *reinterpret_cast<__nv_bfloat162*>(sn + j) = out2;
            *reinterpret_cast<__nv_bfloat162*>(so + j) = out2;
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kGemmTmemCols);
  }
}

// Input rows of the first update: [E[anchor_b] ; s_0 = 0] (one warp per row).
__global__ void __launch_bounds__(256) rnn_init_kernel(const __nv_bfloat16* E, const int32_t* anchor,
                                                       int B, int r, int V, __nv_bfloat16* gru_in,
                                                       int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();  // the buffer may still be read by the previous call's kernels
  const int b = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= B) return;
  int tok = anchor[b];
  if (tok < 0 || tok >= V) {
    if (lane == 0) report(status, kErrBounds);
    tok = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(E + (size_t)tok * r);
  uint4* dst = reinterpret_cast<uint4*>(gru_in + (size_t)b * 2 * r);
  const int n16 = r / 8;
  for (int i = lane; i < n16; i += 32) {
    dst[i] = __ldg(src + i);
    dst[n16 + i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Packed step matrix W_step [4r][2r]: unit block t (units 32t .. 32t+31) owns
// rows 128t .. 128t+127 = reset | update | new-input | new-recurrent, each 32
// rows over the 2r inputs [e ; s]:
//   reset, update:  [W_ih[g*r + u][0:r] , W_hh[g*r + u][0:r]]
//   new-input:      [W_ih[2r + u][0:r]  , 0]
//   new-recurrent:  [0                  , W_hh[2r + u][0:r]]
__global__ void __launch_bounds__(256) rnn_pack_kernel(const __nv_bfloat16* W_ih,
                                                       const __nv_bfloat16* W_hh, int r, int d,
                                                       __nv_bfloat16* W_step) {
  const size_t total = (size_t)4 * r * 2 * r;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / (2 * r)), c = (int)(i % (2 * r));
    const int t = row / 128, w = row % 128, grp = w / 32, u = t * 32 + (w % 32);
    const bool from_e = c < r;
    const int cc = from_e ? c : c - r;
    __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
    if (grp < 2) {
      v = from_e ? W_ih[(size_t)(grp * r + u) * (r + d) + cc] : W_hh[(size_t)(grp * r + u) * r + cc];
    } else if (grp == 2) {
      if (from_e) v = W_ih[(size_t)(2 * r + u) * (r + d) + cc];
    } else {
      if (!from_e) v = W_hh[(size_t)(2 * r + u) * r + cc];
    }
    W_step[i] = v;
  }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl_cfg(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
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

}  // namespace

// A: rows of Kd bf16 (a_stride elements apart), M rows; W: N rows of Kd
// (w_stride apart). Kd % 64 == 0; N % 128 == 0 for the update epilogue.
cudaError_t launch_rnn_gemm(const GemmParams& g, int mode, const void* A, int64_t a_stride,
                            const void* W, int64_t w_stride, cudaStream_t s) {
  if (g.Kd <= 0 || g.Kd % 64 != 0 || g.M <= 0 || g.N <= 0) return cudaErrorInvalidValue;
  CUtensorMap mA, mW;
  const cuuint32_t box[2] = {64, 128};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)g.Kd, (cuuint64_t)g.M};
    const cuuint64_t str[1] = {(cuuint64_t)a_stride * 2};
    if (!encode_tmap_bf16(&mA, A, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)g.Kd, (cuuint64_t)g.N};
    const cuuint64_t str[1] = {(cuuint64_t)w_stride * 2};
    if (!encode_tmap_bf16(&mW, W, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const dim3 grid((g.N + 127) / 128, (g.M + 127) / 128);
  if (mode == kGemmBias) {
    cudaError_t e = cudaFuncSetAttribute(rnn_gemm_kernel<kGemmBias>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e != cudaSuccess) return e;
    return launch_pdl_cfg(rnn_gemm_kernel<kGemmBias>, grid, dim3(kGemmThreads), kGemmSmem, s, g, mA, mW);
  }
  cudaError_t e = cudaFuncSetAttribute(rnn_gemm_kernel<kGemmGru>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl_cfg(rnn_gemm_kernel<kGemmGru>, grid, dim3(kGemmThreads), kGemmSmem, s, g, mA, mW);
}

cudaError_t launch_rnn_init(const void* E, const int32_t* anchor, int32_t B, int32_t r, int32_t V,
                            void* gru_in, int32_t* status, cudaStream_t s) {
  return launch_pdl_cfg(rnn_init_kernel, dim3((B + 7) / 8), dim3(256), 0, s,
                        reinterpret_cast<const __nv_bfloat16*>(E), anchor, (int)B, (int)r, (int)V,
                        reinterpret_cast<__nv_bfloat16*>(gru_in), status);
}

cudaError_t launch_rnn_pack(const void* W_ih, const void* W_hh, int32_t r, int32_t d, void* W_step,
                            cudaStream_t s) {
  const size_t total = (size_t)8 * r * r;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  rnn_pack_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(W_ih),
                                         reinterpret_cast<const __nv_bfloat16*>(W_hh), r, d,
                                         reinterpret_cast<__nv_bfloat16*>(W_step));
  return cudaGetLastError();
}

}  // namespace ds
