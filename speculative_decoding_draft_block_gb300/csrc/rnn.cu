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
//     all B*K positions per draft call (N = 3r, K = d). A tile is one position
//     and 128 requests (a 3-D TMA box over h), and the result is stored
//     position-major and unit-major, gh[k][n][b], so that both its stores and
//     the update's loads are coalesced across requests;
//   * per position, one GEMM over the B requests with the packed step matrix
//     (N = 4r, K = 2r): for each block of 16 state units its 64 rows hold the
//     reset and update rows over [e ; s], the new-gate rows over e alone and
//     over s alone. The epilogue of a 64-column tile therefore holds all four
//     pre-activations of its 16 units and writes the new state directly.
//
// rnn_gemm_kernel: 128 x N output tile per CTA (N = 128 for the hidden-state
// GEMM, 64 for the update), K in steps of 64 (one 128-byte swizzled TMA box
// per operand per stage), warp 0 issues TMA, warp 1 (one elected thread)
// issues tcgen05.mma kind::f16 with the accumulator in TMEM, warps 2..5 read
// TMEM back (lane quarter = warp % 4) and run the epilogue. The weight boxes
// of the first stages are requested before the dependent-launch wait (weights
// are inputs of the call); the A boxes after it. Every wait is bounded; on
// timeout the kernel records DS_ERR_TIMEOUT and unwinds.
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
constexpr int kMaxStages = 8;
constexpr uint32_t kABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kGemmWaitPolls = 1u << 16;

template <int kMode>
struct GemmCfg {
  static constexpr int kN = kMode == kGemmGru ? 64 : 128;
  static constexpr int kStages = kMode == kGemmGru ? 8 : 6;
  static constexpr uint32_t kWBytes = kN * 128;
  static constexpr uint32_t kStageBytes = kABytes + kWBytes;
  static constexpr size_t kSmem = kStages * kStageBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = kN;
  static_assert(kStages <= kMaxStages, "stage count");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

struct GemmShared {
  uint64_t full[kMaxStages], empty[kMaxStages], done;
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

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid(x) = 1 / (1 + 2^(-x log2 e)) and tanh(x) = 1 - 2 / (1 + 2^(2x log2 e)),
// with the ex2 and rcp approximations: relative error ~1e-6, exact limits for
// large |x| (ex2 saturates to 0 or +inf, rcp(+inf) = 0). The state is stored
// as bfloat16, 2^-8 relative, so this moves only values on a rounding boundary.
__device__ __forceinline__ float sigmoid_fast(float x) {
  return rcp_approx(1.0f + ex2_approx(-x * kLog2eHi));
}
__device__ __forceinline__ float tanh_fast(float x) {
  return 1.0f - 2.0f * rcp_approx(1.0f + ex2_approx(2.0f * kLog2eHi * x));
}

template <int kMode>
__global__ void __launch_bounds__(kGemmThreads, 1)
    rnn_gemm_kernel(const GemmParams g, const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmW) {
  using C = GemmCfg<kMode>;
  extern __shared__ uint8_t raw[];
  __shared__ GemmShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base_addr = smem_u32(raw);
  uint8_t* smem = raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  const int mtiles = (g.B + 127) / 128;
  const int nt = blockIdx.x;
  const int mt = blockIdx.y % mtiles;
  const int pos = blockIdx.y / mtiles;  // hidden-state GEMM: the position of this tile
  const int nkb = g.Kd / 64;
  volatile int* abort_flag = &sh.abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem_slot, C::kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmW);
      const uint64_t pol = policy_evict_last();
      auto load_a = [&](int kb, int st) {
        uint8_t* dst = smem + st * C::kStageBytes;
        if (kMode == kGemmBias)
          tma_load_3d(dst, &tmA, &sh.full[st], kb * 64, pos, mt * 128, pol);
        else
          tma_load_2d(dst, &tmA, &sh.full[st], kb * 64, mt * 128, pol);
      };
      auto load_w = [&](int kb, int st) {
        tma_load_2d(smem + st * C::kStageBytes + kABytes, &tmW, &sh.full[st], kb * 64, nt * C::kN, pol);
      };
      // weights of the first stages while the previous kernel finishes
      const int pre = nkb < C::kStages ? nkb : C::kStages;
      for (int kb = 0; kb < pre; ++kb) {
        mbar_expect_tx(&sh.full[kb], C::kStageBytes);
        load_w(kb, kb);
      }
      pdl_wait();  // A rows (the update: e and s) come from earlier kernels
      for (int kb = 0; kb < pre; ++kb) load_a(kb, kb);
      for (int kb = pre; kb < nkb; ++kb) {
        const int st = kb % C::kStages;
        if (!gemm_wait(&sh.empty[st], ((kb / C::kStages) & 1) ^ 1, abort_flag, g.status)) break;
        mbar_expect_tx(&sh.full[st], C::kStageBytes);
        load_w(kb, st);
        load_a(kb, st);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, C::kN, false, false);  // both operands K-major
      const uint64_t bits = smem_desc_bits(16, 1024, 2);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int st = kb % C::kStages;
        ok = gemm_wait(&sh.full[st], (kb / C::kStages) & 1, abort_flag, g.status);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* a = smem + st * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, smem_desc(a + kk * 32, bits), smem_desc(a + kABytes + kk * 32, bits), idesc,
                   (kb | kk) != 0 ? 1u : 0u);
        mma_commit(&sh.empty[st]);
      }
      if (ok) mma_commit(&sh.done);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int b = mt * 128 + q * 32 + lane;
    const int r = g.r, u0 = nt * 16;
    pdl_wait();
    // Update: this row's gate inputs (written by the hidden-state GEMM), the
    // recurrent biases and the old state are loaded while TMA and MMA run.
    float gin[kMode == kGemmGru ? 48 : 1], bh[kMode == kGemmGru ? 48 : 1];
    uint4 sraw[2] = {};
    if (kMode == kGemmGru && b < g.B) {
      const float* gh = g.gh + (size_t)(g.p - 1) * 3 * r * g.B + b;  // gh[p-1][n][b]
#pragma unroll
      for (int j = 0; j < 48; ++j) {
        const int n = (j >> 4) * r + u0 + (j & 15);  // gate j / 16, unit u0 + j % 16
        gin[j] = gh[(size_t)n * g.B];
        bh[j] = __ldg(g.b_hh + n);
      }
      const uint4* sp = reinterpret_cast<const uint4*>(g.s_prev + (size_t)b * 2 * r + u0);
      sraw[0] = sp[0];
      sraw[1] = sp[1];
    }
    if (gemm_wait(&sh.done, 0, abort_flag, g.status)) {
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
      if (kMode == kGemmBias) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int n0 = nt * 128 + c * 32;
          if (b < g.B) {
            // gh[pos][n][b]: for each n the warp stores 32 consecutive requests
            float* out = g.out + ((size_t)pos * g.N + n0) * g.B + b;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < g.N) out[(size_t)j * g.B] = v[j] + __ldg(g.bias + n0 + j);
          }
        }
      } else {
        // columns 0..15 reset, 16..31 update, 32..47 new (input part),
        // 48..63 new (recurrent part) of units u0 .. u0 + 15
        float v0[32], v1[32];
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 32, v1);
        if (b < g.B) {
          const __nv_bfloat16* sold = reinterpret_cast<const __nv_bfloat16*>(sraw);
          uint4 oraw[2];
          __nv_bfloat16* snew = reinterpret_cast<__nv_bfloat16*>(oraw);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float rg = sigmoid_fast(v0[j] + gin[j] + bh[j]);
            const float ug = sigmoid_fast(v0[16 + j] + gin[16 + j] + bh[16 + j]);
            const float ng = tanh_fast(v1[j] + gin[32 + j] + rg * (v1[16 + j] + bh[32 + j]));
            snew[j] = __float2bfloat16_rn((1.0f - ug) * ng + ug * __bfloat162float(sold[j]));
          }
          uint4* sn = reinterpret_cast<uint4*>(g.s_next + (size_t)b * 2 * r + u0);
          uint4* so = reinterpret_cast<uint4*>(g.states + ((size_t)b * g.K + (g.p - 1)) * r + u0);
          sn[0] = oraw[0];
          sn[1] = oraw[1];
          so[0] = oraw[0];
          so[1] = oraw[1];
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
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

// Packed step matrix W_step [4r][2r]: unit block t (units 16t .. 16t+15) owns
// rows 64t .. 64t+63 = reset | update | new-input | new-recurrent, each 16
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
    const int t = row / 64, w = row % 64, grp = w / 16, u = t * 16 + (w % 16);
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

template <int kMode>
cudaError_t launch_gemm_mode(const GemmParams& g, dim3 grid, const CUtensorMap& mA,
                             const CUtensorMap& mW, cudaStream_t s) {
  using C = GemmCfg<kMode>;
  // once per process (and so never inside a stream capture after a first call)
  static const cudaError_t attr = cudaFuncSetAttribute(
      rnn_gemm_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (attr != cudaSuccess) return attr;
  return launch_pdl_cfg(rnn_gemm_kernel<kMode>, grid, dim3(kGemmThreads), C::kSmem, s, g, mA, mW);
}

}  // namespace

// kGemmBias: A = h [B][K][Kd] (one position and 128 requests per tile), W = N
// rows of Kd, w_stride elements apart; out gh[K][N][B].
// kGemmGru: A = the input rows [e ; s] [B][Kd = 2r], W = W_step [4r][2r].
cudaError_t launch_rnn_gemm(const GemmParams& g, int mode, const void* A, const void* W,
                            int64_t w_stride, cudaStream_t s) {
  if (g.Kd <= 0 || g.Kd % 64 != 0 || g.B <= 0 || g.N <= 0 || g.K <= 0) return cudaErrorInvalidValue;
  const int mtiles = (g.B + 127) / 128;
  CUtensorMap mA, mW;
  if (mode == kGemmBias) {
    const cuuint64_t dims[3] = {(cuuint64_t)g.Kd, (cuuint64_t)g.K, (cuuint64_t)g.B};
    const cuuint64_t str[2] = {(cuuint64_t)g.Kd * 2, (cuuint64_t)g.K * g.Kd * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&mA, A, 3, dims, str, box)) return cudaErrorInvalidValue;
    const cuuint64_t wd[2] = {(cuuint64_t)g.Kd, (cuuint64_t)g.N};
    const cuuint64_t ws[1] = {(cuuint64_t)w_stride * 2};
    const cuuint32_t wb[2] = {64, 128};
    if (!encode_tmap_bf16(&mW, W, 2, wd, ws, wb)) return cudaErrorInvalidValue;
    return launch_gemm_mode<kGemmBias>(g, dim3((g.N + 127) / 128, g.K * mtiles), mA, mW, s);
  }
  if (g.N % 64 != 0) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)g.Kd, (cuuint64_t)g.B};
  const cuuint64_t str[1] = {(cuuint64_t)g.Kd * 2};
  const cuuint32_t box[2] = {64, 128};
  if (!encode_tmap_bf16(&mA, A, 2, dims, str, box)) return cudaErrorInvalidValue;
  const cuuint64_t wd[2] = {(cuuint64_t)g.Kd, (cuuint64_t)g.N};
  const cuuint64_t ws[1] = {(cuuint64_t)w_stride * 2};
  const cuuint32_t wb[2] = {64, 64};
  if (!encode_tmap_bf16(&mW, W, 2, wd, ws, wb)) return cudaErrorInvalidValue;
  return launch_gemm_mode<kGemmGru>(g, dim3(g.N / 64, mtiles), mA, mW, s);
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
