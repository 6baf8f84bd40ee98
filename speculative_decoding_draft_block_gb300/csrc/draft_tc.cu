// Tensor-core tile kernel of the draft step and of the verify's final draw.
//
// DSpark summary page, 방법론 › 반자기회귀 생성: the Markov head's bias for a
// block position is E[x_{k-1}] . P for every request at once -- a
// [B x r] x [r x V] product -- and the position is then sampled from
// softmax((z_k + bias) / T). This kernel computes that product on the 5th-gen
// tensor cores and reduces it straight out of TMEM:
//
//   warp 0      producer: TMA loads of P tiles (64 k-rows x 128 tokens per
//               stage, 128B-swizzled, MN-major, L2 evict-last: P is re-read
//               every step; it stays in L2 when the process has set aside
//               persisting L2, see ds_reserve_persisting_l2) and of the
//               staged A rows.
//   warp 1      MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> f32),
//               M = 128 requests, N = 128 tokens, K = r in steps of 16, into one
//               of two TMEM accumulators (double-buffered against the epilogue).
//   warp 2      producer of the base-logit tiles (draft steps), in their own ring
//   warp 3      idle (warpgroup 0 releases its registers to the epilogue)
//   warps 4..   epilogue (kEpiWarps warps, 112 registers each): gather the A operand (E rows of the
//               conditioning tokens, stored 128B-swizzled K-major) with 16-byte
//               loads at each M-tile; then per tile tcgen05.ld of their TMEM
//               slice, add the base logits from shared memory, and reduce every
//               (request, 32-token chunk) to its record: the double-float sum
//               of 2^(t - ref) with an integer reference (sampling rows), or
//               its largest logit (greedy rows). Nothing V-wide is stored.
//
// Tiles (M-tile of 128 requests, N-tile of 128 tokens) are split into
// contiguous ranges, one range per CTA, one CTA per SM. Consecutive steps are
// chained with programmatic dependent launch; every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "fastpath.cuh"
#include "sampling.cuh"
#include "sm100.cuh"

namespace ds {

namespace {

using namespace sm100;

constexpr int kEpiWarps = 16;                   // multiple of 4 (TMEM lane quadrants)
constexpr int kCtrlWarps = 4;                   // warpgroup 0: producer, MMA issuer, two idle warps
constexpr int kColGroups = kEpiWarps / 4;       // column groups per lane quadrant
constexpr int kChunks = 4 / kColGroups;         // 32-token chunks per thread per tile
constexpr int kTcThreads = 32 * (kCtrlWarps + kEpiWarps);
// Register split: warpgroup 0 (control) gives registers to the epilogue
// warpgroups. The block launches with kLaunchRegs per thread (65536 / 640,
// rounded down to the allocation unit of 8); the split uses exactly that pool.
constexpr uint32_t kLaunchRegs = 96, kCtrlRegs = 32, kEpiRegs = 112;
static_assert(32 * kCtrlWarps * kCtrlRegs + 32 * kEpiWarps * kEpiRegs <= kTcThreads * kLaunchRegs,
              "register split exceeds the launch pool");
static_assert(kTcThreads * kLaunchRegs <= 65536, "launch pool exceeds the register file");
constexpr int kUnrollChunks = 1;                // code size over TMEM-load overlap
constexpr int kTileN = 128;
// The P ring is kPRing bytes: kPStages stages of one 64-row k-block (16 KB,
// two tensor copies of 64 rows each), or, with the tile-packed copy of P,
// kPStages / 2 stages of two k-blocks (32 KB, one bulk copy).
constexpr int kPStages = 6;
constexpr int kZSlots = 4;            // 128 rows x 64 tokens of logits each
constexpr int kAccum = 2;             // TMEM accumulators (128 columns each)
constexpr uint32_t kASize = 65536;    // up to r = 256
constexpr uint32_t kPStage = 16384;
constexpr uint32_t kZSlot = 16384;
constexpr uint32_t kOffP = kASize;
constexpr uint32_t kOffZ = kOffP + kPStages * kPStage;
constexpr uint32_t kSmemBytes = kOffZ + kZSlots * kZSlot + 1024;
constexpr uint32_t kTmemCols = kAccum * kTileN;
// tcgen05.alloc takes a power-of-two column count from 32 to 512: three
// 128-column accumulators (384 columns) would be an illegal allocation.
static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
              "TMEM allocation must be a power of two in [32, 512] columns");

struct TcParams {
  SampleParams sp;
  int32_t n_mt, n_nt, nkb, tiles;

  int32_t packed;        // P from the tile-packed copy: 32 KB stages by bulk copy
  int32_t pring;         // stages in the P ring (6 or 3)
  int32_t pstage_bytes;  // ring stage size (16 or 32 KB)
  int32_t kb_stage;      // 64-row k-blocks per stage (1 or 2)
  int32_t pstages;       // stages per tile: ceil(nkb / kb_stage)
  uint32_t wait_polls;   // polls of a bounded wait before it gives up
  int32_t withhold_cta;  // test hook (-1: none), see set_tile_test_hooks
};

struct Shared {
  uint64_t a_full, a_empty;
  uint64_t p_full[kPStages], p_empty[kPStages];
  uint64_t z_full[kZSlots], z_empty[kZSlots];
  uint64_t t_full[kAccum], t_empty[kAccum];
  uint64_t x_bar;  // barrier of the epilogue threads (all arrive)
  uint64_t drain;  // the MMA issuer's last commit, waited for before TMEM is freed
  uint32_t tmem_slot;
  int abort_flag;
};

// Bounded wait (about a second at most with the default kWaitPolls): the
// thread sleeps in try_wait with a 20 us hint (it wakes as soon as the phase
// completes), so waiting warps do not take issue slots from the epilogue.
constexpr uint32_t kWaitPolls = 1u << 16;
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* status, uint32_t polls) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < polls; ++i) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((i & 15) == 15 && *abort_flag) return false;
  }
  *abort_flag = 1;
  report(status, kErrTimeout);
  return false;
}

// Wait for a copy or commit already issued by this thread to land, also after
// an abort, so that nothing is in flight when the CTA exits; bounded.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, uint32_t polls) {
  for (uint32_t i = 0; i <= polls; ++i)
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return;
}

// Barrier over the epilogue threads only, bounded like every other wait.
// `arrive` false withholds this thread's arrival (test hook only).
__device__ __forceinline__ bool epi_barrier(Shared& sh, uint32_t& ph, volatile int* abort_flag,
                                            int32_t* status, uint32_t polls, bool arrive = true) {
  if (arrive) mbar_arrive(&sh.x_bar);
  const bool ok = wait_bar(&sh.x_bar, ph & 1, abort_flag, status, polls);
  ++ph;
  return ok;
}

// What the epilogue keeps about its row in registers (the general path
// rebuilds the full row context itself). Np, Nq, Rhi, Rlo: final draw only.
struct EpiRow {
  int32_t mode;
  G16 g16;
  int32_t Np, Nq;
  float Rhi, Rlo;
  const __nv_bfloat16* zrow;  // final draw: the request's base and target rows
  const __nv_bfloat16* trow;
};

// Row context of a draft row from its temperature alone (no token reads), so
// it can be formed before the wait on the previous kernel.
__device__ __forceinline__ EpiRow epi_row_draft(const SampleParams& sp, int row) {
  EpiRow c;
  c.mode = kSkip;
  c.g16 = G16{0.f, 0.f, 0.f};
  c.Np = c.Nq = 0;
  c.Rhi = c.Rlo = 0.f;
  c.zrow = c.trow = nullptr;
  if (row < sp.B) {
    const float T = sp.temperature[row];
    if (T == 0.f) {
      c.mode = kGreedyMarkov;
    } else if (T >= 1e-3f && T <= 1e3f) {
      c.mode = kSampleMarkov;
      c.g16 = make_g16(T);
    } else {
      report(sp.status, kErrInvalidArg);
    }
  }
  return c;
}

// One 16-token half of a final-draw chunk's fast path (bf16; see
// fastpath.cuh): tokens 16h .. 16h + 15, tp8 / zp8 their 8 packed target and
// base logit words, b16 their bias columns. Bonus weights 2^(t g - Np), or
// residual weights max(0, 2^(t g - Np) - R 2^((z + b) g - Nq)), both against
// the rows' global references; the pairs are added in token order, as a
// whole-chunk pass would add them.
__device__ __forceinline__ void final_half(const uint32_t* tp8, const uint32_t* zp8, const uint32_t* b16,
                                           bool res, const FastConsts& kp, const FastConsts& kq, float Rhi,
                                           float Rlo, float2& s) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 wp = fast_w2(tp8[i], make_float2(0.f, 0.f), kp);
    if (res) {
      const float2 wq =
          fast_w2(zp8[i], make_float2(__uint_as_float(b16[2 * i]), __uint_as_float(b16[2 * i + 1])), kq);
      s = __fadd2_rn(s, make_float2(residual_w(wp.x, wq.x, Rhi, Rlo), residual_w(wp.y, wq.y, Rhi, Rlo)));
    } else {
      s = __fadd2_rn(s, wp);
    }
  }
}

// One 16-token half of a sampling chunk's fast path: tokens 16h .. 16h + 15,
// zp8 their 8 packed logit words, b16 their bias columns. The pairs are
// added in token order, as a whole-chunk pass would add them.
__device__ __forceinline__ void sample_half(const uint32_t* zp8, const uint32_t* b16, const FastConsts& k,
                                            float2& s) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    fast_pair(zp8[i], make_float2(__uint_as_float(b16[2 * i]), __uint_as_float(b16[2 * i + 1])), k, s);
}

// One 16-token half of a greedy chunk: the largest z + bias as a double-float
// and its first token, continuing from the previous half (j0 = 16h).
__device__ __forceinline__ void greedy_half(const uint32_t* zp8, const uint32_t* b16, int j0, DF& best,
                                            int& bj, bool& bad) {
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) {
    const uint32_t w = zp8[jj >> 1];
    const float zj = __uint_as_float((jj & 1) ? (w & 0xffff0000u) : (w << 16));
    const float bb = __uint_as_float(b16[jj]);
    bad |= bad_logit(zj) || !(bb == bb);
    const DF l = (zj == kNegInf) ? DF{kNegInf, 0.f} : two_sum(zj, bb);
    if ((j0 == 0 && jj == 0) || l.hi > best.hi || (l.hi == best.hi && l.lo > best.lo)) {
      best = l;
      bj = j0 + jj;
    }
  }
}

// The general path for the lanes with need set (greedy and sampling chunks
// the fast paths decline, ragged chunks, residual/bonus draws). Called by the
// whole warp: it reloads the bias from TMEM (a warp-collective load) and the
// logits from shared memory, so that the fast paths keep everything in
// registers. zb / tb: this row's 128-byte logit rows in the (swizzled) slots.
__device__ __noinline__ ChunkRec slow_chunk_warp(const SampleParams* sp, int row, bool need,
                                                 uint32_t taddr, const uint8_t* zb,
                                                 const uint8_t* tb, int ch0, int sw, int col0,
                                                 ChunkRec* out) {
  uint32_t braw[32];
  tmem_ld32_issue(taddr, braw);
  tmem_ld_wait(braw);
  if (!need) return group_empty();
  float bias[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) bias[e] = __uint_as_float(braw[e]);
  uint32_t zp[16], tp[16];
  const RowCtx rc = make_row_ctx<__nv_bfloat16>(*sp, row);
  const int n = min(32, sp->V - col0);
  if (zb != nullptr) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int off = ((ch0 + u) ^ sw) << 4;
      const uint4 v = *reinterpret_cast<const uint4*>(zb + off);
      const uint4 t = *reinterpret_cast<const uint4*>(tb + off);
      zp[4 * u] = v.x; zp[4 * u + 1] = v.y; zp[4 * u + 2] = v.z; zp[4 * u + 3] = v.w;
      tp[4 * u] = t.x; tp[4 * u + 1] = t.y; tp[4 * u + 2] = t.z; tp[4 * u + 3] = t.w;
    }
  } else {  // the rows in global memory (n is even: V % 8 == 0)
    const uint32_t* zr = reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const __nv_bfloat16*>(rc.zrow) + col0);
    const uint32_t* tr = reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const __nv_bfloat16*>(rc.trow) + col0);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      zp[u] = (rc.zrow && 2 * u < n) ? zr[u] : 0u;
      tp[u] = (rc.trow && 2 * u < n) ? tr[u] : 0u;
    }
  }
  ChunkRec r;
  chunk_record<false>(rc, Bf16Src{zp}, bias, Bf16Src{tp}, n, col0, r, sp->status);
  *out = r;
  return r;
}

// Token whose E row forms A-operand row b of this launch (0 for padding rows).
__device__ __forceinline__ int a_token_for_row(const SampleParams& sp, int b) {
  if (b >= sp.B) return 0;
  int tok = 0;
  if (sp.src == 0) {
    tok = (sp.step == 1) ? sp.anchor[b] : sp.draft_tokens[(size_t)b * sp.K + (sp.step - 2)];
  } else {
    const FinalDesc d = sp.final_desc[b];
    tok = (d.mode == kResidual && sp.temperature[b] != 0.f) ? d.a_token : 0;
  }
  return (tok >= 0 && tok < sp.V) ? tok : 0;  // out-of-range ids are reported by make_row_ctx
}

// Row b of the A operand: E[token] for the Markov head; for the RNN head the
// current state (draft) or the state of the final-draw row (verify).
__device__ __forceinline__ const __nv_bfloat16* a_row_src(const SampleParams& sp, int b) {
  const __nv_bfloat16* rows = reinterpret_cast<const __nv_bfloat16*>(sp.a_rows);
  if (rows == nullptr)
    return reinterpret_cast<const __nv_bfloat16*>(sp.E) + (size_t)a_token_for_row(sp, b) * sp.r;
  if (b >= sp.B) return rows;  // padding rows of the last M-tile
  if (sp.src == 0) return rows + (size_t)b * sp.a_rows_stride;
  int j = sp.final_desc[b].row;
  j = j < 0 ? 0 : (j >= sp.K ? sp.K - 1 : j);  // bonus rows (j = K) need no bias
  return rows + (size_t)b * sp.a_rows_stride + (size_t)j * sp.r;
}

template <bool kFinal>
__global__ void __launch_bounds__(kTcThreads, 1)
    tile_tc_kernel(const __grid_constant__ TcParams prm, const __grid_constant__ CUtensorMap tmP,
                   const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ CUtensorMap tmT,
                   const __grid_constant__ CUtensorMap tmA) {
  extern __shared__ uint8_t raw[];
  __shared__ Shared sh;
  const SampleParams& sp = prm.sp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base_addr = smem_u32(raw);
  uint8_t* smem = raw + (((base_addr + 1023u) & ~1023u) - base_addr);
  uint8_t* sA = smem;
  uint8_t* sP = smem + kOffP;
  uint8_t* sZ = smem + kOffZ;
  constexpr bool draft = !kFinal;
  const bool staged = (sp.a_stage_in != nullptr);  // A rows staged by the previous locate

  if (threadIdx.x == 0) {
    mbar_init(&sh.a_full, staged ? 1 : kEpiWarps);
    mbar_init(&sh.a_empty, 1);
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&sh.p_full[i], 1);
      mbar_init(&sh.p_empty[i], 1);
    }
    for (int i = 0; i < kZSlots; ++i) {
      mbar_init(&sh.z_full[i], 1);
      mbar_init(&sh.z_empty[i], kEpiWarps / 2);
    }
    for (int i = 0; i < kAccum; ++i) {
      mbar_init(&sh.t_full[i], 1);
      mbar_init(&sh.t_empty[i], kEpiWarps);
    }
    mbar_init(&sh.x_bar, 32 * kEpiWarps);
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem_slot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  pdl_launch_dependents();

  const int G = gridDim.x;
  const int t0 = (int)((long long)blockIdx.x * prm.tiles / G);
  const int t1 = (int)((long long)(blockIdx.x + 1) * prm.tiles / G);
  volatile int* abort_flag = &sh.abort_flag;

  if (warp < kCtrlWarps) {
    // warpgroup 0 hands registers to the epilogue warpgroups
    setmaxnreg_dec<kCtrlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_p = policy_evict_last();
    if (lane == 0) prefetch_tmap(&tmP);
    if (lane == 0 && staged) prefetch_tmap(&tmA);
    uint32_t pc = 0, a_loads = 0;
    int a_mt = -1;
    bool waited = draft && !staged, ok = true;  // a draft step's P and logits are inputs
    for (int t = t0, i = 0; t < t1 && ok; ++t, ++i) {
      const int mt = t / prm.n_nt, nt = t - mt * prm.n_nt;
      const int n0 = nt * kTileN;
      for (int st = 0; st < prm.pstages && ok; ++st, ++pc) {
        const uint32_t ps = pc % (uint32_t)prm.pring;
        if (lane == 0) {
          ok = wait_bar(&sh.p_empty[ps], ((pc / (uint32_t)prm.pring) & 1) ^ 1, abort_flag, sp.status,
                        prm.wait_polls);
          if (ok) {
            uint8_t* dst = sP + ps * (uint32_t)prm.pstage_bytes;
            if (prm.packed) {
              // k-blocks [st * 2, st * 2 + 1] of tile nt, contiguous in the packed copy
              const int nk = min(prm.kb_stage, prm.nkb - st * prm.kb_stage);
              const uint32_t bytes = (uint32_t)nk * 16384u;
              mbar_expect_tx(&sh.p_full[ps], bytes);
              bulk_load_hint(dst,
                             reinterpret_cast<const uint8_t*>(sp.P_packed) +
                                 ((size_t)nt * prm.nkb + (size_t)st * prm.kb_stage) * 16384u,
                             bytes, &sh.p_full[ps], pol_p);
            } else {
              mbar_expect_tx(&sh.p_full[ps], kPStage);
              tma_load_2d(dst, &tmP, &sh.p_full[ps], n0, st * 64, pol_p);
              tma_load_2d(dst + 8192, &tmP, &sh.p_full[ps], n0 + 64, st * 64, pol_p);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (!ok) break;
      if (ok && staged && mt != a_mt) {
        // this M-tile's A rows, written by the previous step's locate; issued after
        // the tile's P and logit loads so those are in flight during the wait, and
        // before anything that waits on the MMA
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        if (lane == 0) {
          ok = a_loads == 0 || wait_bar(&sh.a_empty, (a_loads - 1) & 1, abort_flag, sp.status, prm.wait_polls);
          if (ok) {
            mbar_expect_tx(&sh.a_full, (uint32_t)prm.nkb * 16384u);
            for (int c = 0; c < prm.nkb; ++c)
              tma_load_2d(sA + c * 16384, &tmA, &sh.a_full, c * 64, mt * 128, pol_p);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++a_loads;
        a_mt = mt;
      }
    }
    // nothing of this CTA may be in flight when it exits (also after an abort)
    if (lane == 0) {
      const uint32_t ring = (uint32_t)prm.pring;
      for (uint32_t j = pc > ring ? pc - ring : 0; j < pc; ++j)
        drain_bar(&sh.p_full[j % ring], (j / ring) & 1, prm.wait_polls);
      if (a_loads > 0) drain_bar(&sh.a_full, (a_loads - 1) & 1, prm.wait_polls);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ logit producer
    // the draft step's base-logit tiles (inputs: no dependent wait), in a ring
    // of their own so they run ahead of the projection stream
    if (draft) {
      const uint64_t pol_z = policy_evict_first();
      if (lane == 0) prefetch_tmap(&tmZ);
      uint32_t zc = 0;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const int mt = t / prm.n_nt, nt = t - mt * prm.n_nt;
        const int n0 = nt * kTileN;
        for (int nb = 0; nb < 2 && ok; ++nb, ++zc) {
          const uint32_t zs = zc % kZSlots;
          if (lane == 0) {
            ok = wait_bar(&sh.z_empty[zs], ((zc / kZSlots) & 1) ^ 1, abort_flag, sp.status, prm.wait_polls);
            if (ok) {
              mbar_expect_tx(&sh.z_full[zs], kZSlot);
              tma_load_3d(sZ + zs * kZSlot, &tmZ, &sh.z_full[zs], n0 + nb * 64, sp.step - 1,
                          mt * 128, pol_z);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      if (lane == 0)
        for (uint32_t j = zc > (uint32_t)kZSlots ? zc - kZSlots : 0; j < zc; ++j)
          drain_bar(&sh.z_full[j % kZSlots], (j / kZSlots) & 1, prm.wait_polls);
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, kTileN, false, true);
      const uint64_t abits = smem_desc_bits(16, 1024, 2);
      const uint64_t bbits = smem_desc_bits(8192, 1024, 2);
      int cur_mt = -1;
      uint32_t a_uses = 0, pc = 0;
      bool ok = true;
      for (int t = t0, i = 0; t < t1 && ok; ++t, ++i) {
        const int mt = t / prm.n_nt;
        if (mt != cur_mt) {
          if (cur_mt >= 0) mma_commit(&sh.a_empty);
          ok = wait_bar(&sh.a_full, a_uses & 1, abort_flag, sp.status, prm.wait_polls);
          if (!ok) break;
          ++a_uses;
          cur_mt = mt;
          tc_fence_after();
        }
        const uint32_t buf = i % kAccum;
        ok = wait_bar(&sh.t_empty[buf], ((i / kAccum) & 1) ^ 1, abort_flag, sp.status, prm.wait_polls);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * kTileN;
        for (int st = 0; st < prm.pstages && ok; ++st, ++pc) {
          const uint32_t ps = pc % (uint32_t)prm.pring;
          ok = wait_bar(&sh.p_full[ps], (pc / (uint32_t)prm.pring) & 1, abort_flag, sp.status, prm.wait_polls);
          if (!ok) break;
          tc_fence_after();
          for (int cl = 0; cl < prm.kb_stage; ++cl) {
            const int c = st * prm.kb_stage + cl;  // 64-row k-block of r
            if (c >= prm.nkb) break;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(sA + c * 16384 + kk * 32, abits);
              const uint64_t bd = smem_desc(sP + ps * (uint32_t)prm.pstage_bytes + cl * 16384 + kk * 2048, bbits);
              mma_bf16(d, ad, bd, idesc, (c | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&sh.p_empty[ps]);
        }
        if (ok) mma_commit(&sh.t_full[buf]);
      }
      // every MMA this thread issued has completed before TMEM is freed
      mma_commit(&sh.drain);
      drain_bar(&sh.drain, 0, prm.wait_polls);
    }
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<kEpiRegs>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kCtrlWarps, et = threadIdx.x - 32 * kCtrlWarps;
    const int q = warp & 3, cg = ew >> 2;
    const int r_local = q * 32 + lane;
    int cur_mt = -1, pre_mt = -1;
    uint32_t a_uses = 0, xph = 0;
    EpiRow c;
    c.mode = kSkip;
    if (draft && t0 < t1) {  // temperatures are inputs: read them before the wait
      pre_mt = t0 / prm.n_nt;
      c = epi_row_draft(sp, pre_mt * 128 + r_local);
    }
    pdl_wait();  // tokens and final-draw descriptors come from earlier kernels
    ChunkRec gacc = group_empty();  // this thread's chunks of the current M-tile
    for (int t = t0, i = 0; t < t1; ++t, ++i) {
      const int mt = t / prm.n_nt, nt = t - mt * prm.n_nt;
      const int row = mt * 128 + r_local;
      if (mt != cur_mt) {
        // A operand of this M-tile: E rows of its conditioning tokens, written
        // 128B-swizzled (16-byte chunk c of row m at c ^ (m & 7)) for the MMA.
        if (draft) {
          if (mt != pre_mt) c = epi_row_draft(sp, row);
        } else {
          const RowCtx rc = make_row_ctx<__nv_bfloat16>(sp, row);
          c.mode = rc.mode;
          c.g16 = (rc.mode == kResidual || rc.mode == kBonus) ? make_g16_from(rc.g) : G16{0.f, 0.f, 0.f};
          c.Np = rc.Np;
          c.Nq = rc.Nq;
          c.Rhi = rc.Rhi;
          c.Rlo = rc.Rlo;
          c.zrow = reinterpret_cast<const __nv_bfloat16*>(rc.zrow);
          c.trow = reinterpret_cast<const __nv_bfloat16*>(rc.trow);
        }
        if (!staged) {
          if (a_uses > 0 && !wait_bar(&sh.a_empty, (a_uses - 1) & 1, abort_flag, sp.status, prm.wait_polls)) break;
          // kThreadsPerRow threads per A row, each a contiguous run of its
          // 16-byte chunks, all loads in flight before the first store
          constexpr int kThreadsPerRow = 32 * kEpiWarps / 128;
          const int m = et / kThreadsPerRow, part = et % kThreadsPerRow;
          const int per_row = prm.nkb * 8;  // 16-byte chunks per row
          const int cpt = per_row / kThreadsPerRow;
          const uint4* src = reinterpret_cast<const uint4*>(a_row_src(sp, mt * 128 + m)) + part * cpt;
          constexpr int kMaxCpt = 32 / kThreadsPerRow;
          constexpr int kBatch = kMaxCpt < 8 ? kMaxCpt : 8;  // loads in flight per thread
#pragma unroll
          for (int u0 = 0; u0 < kMaxCpt; u0 += kBatch) {
            uint4 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
              if (u0 + u < cpt) v[u] = __ldg(src + u0 + u);
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
              if (u0 + u < cpt) {
                const int rem = part * cpt + u0 + u, kb = rem >> 3, ch = rem & 7;
                *reinterpret_cast<uint4*>(sA + kb * 16384 + m * 128 + ((ch ^ (m & 7)) << 4)) = v[u];
              }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.a_full);
          ++a_uses;
        }
        cur_mt = mt;
        gacc = group_empty();
      }
      const uint32_t buf = i % kAccum;
      // this thread's chunks: cg * kChunks .. + kChunks - 1, all in logit box nb
      const int nb = (cg * kChunks) >> 1;
      const uint32_t zc = 2u * i + nb;
      const uint32_t zs = draft ? zc % kZSlots : nb;
      const uint32_t zph = draft ? (zc / kZSlots) & 1 : (i & 1);
      if (draft && !wait_bar(&sh.z_full[zs], zph, abort_flag, sp.status, prm.wait_polls)) break;
      // final draw: each thread loads its own row's 2 x 64 tokens (base and
      // target) straight from global memory, issued before the MMA wait
      uint4 fz[kChunks][4], ft[kChunks][4];
      if (kFinal) {
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int col0 = nt * kTileN + (cg * kChunks + j) * 32;
          const bool full = row < sp.B && col0 + 32 <= sp.V;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            ft[j][u] = (full && c.trow) ? __ldcs(reinterpret_cast<const uint4*>(c.trow + col0) + u)
                                        : make_uint4(0, 0, 0, 0);
            fz[j][u] = (full && c.zrow) ? __ldcs(reinterpret_cast<const uint4*>(c.zrow + col0) + u)
                                        : make_uint4(0, 0, 0, 0);
          }
        }
      }
      if (!wait_bar(&sh.t_full[buf], (i / kAccum) & 1, abort_flag, sp.status, prm.wait_polls)) break;
      tc_fence_after();
      __syncwarp();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + buf * kTileN;
      const uint8_t* zb = sZ + zs * kZSlot + r_local * 128;  // this row's line in its logit box
      const int sw = r_local & 7;
      // the final draw indexes its prefetched rows by j: fully unrolled there
#pragma unroll(kFinal ? kChunks : kUnrollChunks)
      for (int j = 0; j < kChunks; ++j) {
        const int ch0 = ((cg * kChunks + j) & 1) * 4;
        const int col0 = nt * kTileN + (cg * kChunks + j) * 32;
        const bool active = row < sp.B && c.mode != kSkip && col0 < sp.V;
        const int n = min(32, sp.V - col0);
        ChunkRec* out = sp.chunks + (size_t)(col0 >> 5) * sp.B + row;  // chunk-major: coalesced
        bool done = !active;
        if constexpr (kFinal) {
          // the bias in two 16-column loads (warp-collective), as in the draft
          const bool fast = active && n == 32 && (c.mode == kResidual || c.mode == kBonus);
          const bool res = c.mode == kResidual;
          uint32_t zp[16], tp[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 t = ft[j][u], v = fz[j][u];
            tp[4 * u] = t.x; tp[4 * u + 1] = t.y; tp[4 * u + 2] = t.z; tp[4 * u + 3] = t.w;
            zp[4 * u] = v.x; zp[4 * u + 1] = v.y; zp[4 * u + 2] = v.z; zp[4 * u + 3] = v.w;
          }
          bool ok = fast && fast_span_ok(tp, c.g16.G, c.Np) && (!res || fast_span_ok(zp, c.g16.G, c.Nq));
          const FastConsts kp = make_fast_consts(c.g16, c.Np);
          const FastConsts kq = make_fast_consts(c.g16, c.Nq);
          float2 sum2 = make_float2(0.f, 0.f);
          const uint32_t taddr = tbase + (cg * kChunks + j) * 32;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t b16[16];
            tmem_ld16_issue(taddr + 16 * h, b16);
            tmem_ld16_wait(b16);
            if (ok) final_half(tp + 8 * h, zp + 8 * h, b16, res, kp, kq, c.Rhi, c.Rlo, sum2);
          }
          if (ok) {
            const float sum = __fadd_rn(sum2.x, sum2.y);
            ok = sum >= 0.f && isfinite(sum);
            if (ok) {
              const ChunkRec rec = {sum, 0.f, 0, -2};  // fast-path record
              *out = rec;
              group_merge(c.mode, gacc, rec);
            }
          }
          done = fast ? ok : !active;
        } else {
          // the bias in two 16-column loads (warp-collective: every lane issues
          // them), so only 16 bias registers are live
          const bool fast = active && n == 32 && (c.mode == kSampleMarkov || c.mode == kGreedyMarkov);
          const bool samp = c.mode == kSampleMarkov;
          uint32_t zp[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 v = fast ? *reinterpret_cast<const uint4*>(zb + (((ch0 + u) ^ sw) << 4))
                                 : make_uint4(0u, 0u, 0u, 0u);
            zp[4 * u] = v.x;
            zp[4 * u + 1] = v.y;
            zp[4 * u + 2] = v.z;
            zp[4 * u + 3] = v.w;
          }
          int fref = 0;
          bool ok = fast && (!samp || fast_chunk_ok(zp, c.g16, fref));
          const FastConsts k = make_fast_consts(c.g16, fref);
          float2 sum2 = make_float2(0.f, 0.f);
          DF best = {kNegInf, 0.f};
          int bj = 0;
          bool bad = false;
          const uint32_t taddr = tbase + (cg * kChunks + j) * 32;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t b16[16];
            tmem_ld16_issue(taddr + 16 * h, b16);
            tmem_ld16_wait(b16);
            if (ok) {
              if (samp)
                sample_half(zp + 8 * h, b16, k, sum2);
              else
                greedy_half(zp + 8 * h, b16, 16 * h, best, bj, bad);
            }
          }
          if (ok) {
            ChunkRec rec;
            if (samp) {
              const float sum = __fadd_rn(sum2.x, sum2.y);
              ok = sum >= 0.f && isfinite(sum);
              rec = {sum, 0.f, fref, -2};  // fast-path record
            } else {
              ok = !bad;
              rec = {best.hi, best.lo, 0, col0 + bj};
            }
            if (ok) {
              *out = rec;
              group_merge(c.mode, gacc, rec);
            }
          }
          done = !active || ok;
        }
        if (__any_sync(0xffffffffu, !done)) {
          const ChunkRec rec = slow_chunk_warp(&sp, row, !done, tbase + (cg * kChunks + j) * 32,
                                               kFinal ? nullptr : zb, kFinal ? nullptr : zb, ch0, sw,
                                               col0, out);
          if (!done) group_merge(c.mode, gacc, rec);
        }
      }
      if (t + 1 == t1 || (t + 1) / prm.n_nt != mt) {
        // Group record of each row over this CTA's tiles of the M-tile: the
        // column groups' partial records meet in the row's line of the tile's
        // first logit slot (consumed, and not released until after this).
        uint8_t* xb = sZ + (draft ? (2u * i) % kZSlots : 0u) * kZSlot + r_local * 128;
        // test hook: one warp of one CTA withholds its arrival here, at a point
        // where every copy and MMA of the CTA has completed (this is its last
        // tile and its accumulator and logits were waited for), so the others'
        // bounded wait runs out and the CTA returns with nothing in flight
        const bool withhold = blockIdx.x == prm.withhold_cta && ew == 0 && t + 1 == t1;
        if (!epi_barrier(sh, xph, abort_flag, sp.status, prm.wait_polls, !withhold)) break;
        if (cg > 0) *reinterpret_cast<ChunkRec*>(xb + 16 * cg) = gacc;
        if (!epi_barrier(sh, xph, abort_flag, sp.status, prm.wait_polls)) break;
        if (cg == 0 && row < sp.B && c.mode != kSkip) {
          ChunkRec g = gacc;
#pragma unroll
          for (int k = 1; k < kColGroups; ++k)
            group_merge(c.mode, g, *reinterpret_cast<const ChunkRec*>(xb + 16 * k));
          sp.supers[(size_t)row * sp.sup_stride + (blockIdx.x - first_group(sp, mt))] = g;
        }
        // The exchange line lies in the first logit slot of the tile. Only the
        // column groups that read that slot release it (z_empty counts their
        // warps), column group 0 among them, after these reads; the other
        // groups wrote their records between the two barriers.
        static_assert(kColGroups <= 8, "one 128-byte line holds the exchanged records");
      }
      // this warp is done with the tile's accumulator and logit slots
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.t_empty[buf]);
        if (draft) mbar_arrive(&sh.z_empty[zs]);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  return encode_tmap_bf16(m, ptr, rank, dims, strides, box);
}

cudaError_t register_split_ok(const void* fn) {
  cudaFuncAttributes a;
  const cudaError_t e = cudaFuncGetAttributes(&a, fn);
  if (e != cudaSuccess) return e;
  const long long pool = (long long)kTcThreads * a.numRegs;
  const long long need = 32LL * kCtrlWarps * kCtrlRegs + 32LL * kEpiWarps * kEpiRegs;
  return (a.numRegs == (int)kLaunchRegs && need <= pool) ? cudaSuccess : cudaErrorInvalidConfiguration;
}

std::atomic<uint32_t> g_wait_polls{kWaitPolls};
std::atomic<int32_t> g_withhold_cta{-1};

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

bool encode_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = get_encoder();
  if (!fn) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};  // up to rank 5
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void tc_group_layout(SampleParams& p) {
  static const int sms = num_sms();
  p.sup_stride = sup_stride_for(p.V);
  p.sup_nt = (p.V + kTileN - 1) / kTileN;
  p.sup_rows = 128;
  p.sup_tiles = p.sup_nt * ((p.B + 127) / 128);
  int g = sms < kMaxTcGroups ? sms : kMaxTcGroups;
  p.sup_groups = p.sup_tiles < g ? p.sup_tiles : g;
  p.sup_cpt = kTileN / 32;
}

void set_tile_test_hooks(uint32_t wait_polls, int32_t withhold_cta) {
  g_wait_polls.store(wait_polls == 0 ? kWaitPolls : wait_polls, std::memory_order_relaxed);
  g_withhold_cta.store(withhold_cta < 0 ? -1 : withhold_cta, std::memory_order_relaxed);
}

bool tc_path_supported(int32_t dtype, int32_t r, int32_t V) {
  (void)V;  // any V % 8 == 0 (the ABI's rule)
  return dtype == DS_BF16 && r % 64 == 0 && r >= 64 && r <= 256;
}

cudaError_t launch_tile_tc(const SampleParams& p, cudaStream_t s) {
  static cudaError_t attr_d = cudaFuncSetAttribute(
      tile_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  static cudaError_t attr_f = cudaFuncSetAttribute(
      tile_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (attr_d != cudaSuccess) return attr_d;
  if (attr_f != cudaSuccess) return attr_f;
  // the register split inside the kernel needs exactly the launch pool it was
  // planned for: refuse to launch a build whose launch count differs (an
  // increase that cannot be satisfied would never return)
  static cudaError_t regs_d = register_split_ok(reinterpret_cast<const void*>(tile_tc_kernel<false>));
  static cudaError_t regs_f = register_split_ok(reinterpret_cast<const void*>(tile_tc_kernel<true>));
  if (regs_d != cudaSuccess) return regs_d;
  if (regs_f != cudaSuccess) return regs_f;
  TcParams prm;
  prm.sp = p;
  prm.n_mt = (p.B + 127) / 128;
  prm.n_nt = (p.V + kTileN - 1) / kTileN;
  prm.nkb = p.r / 64;
  prm.packed = p.P_packed != nullptr ? 1 : 0;
  prm.kb_stage = prm.packed ? 2 : 1;
  prm.pstage_bytes = (int32_t)kPStage * prm.kb_stage;
  prm.pring = kPStages / prm.kb_stage;
  prm.pstages = (prm.nkb + prm.kb_stage - 1) / prm.kb_stage;
  if (p.r % 64 != 0 || p.r > 256) return cudaErrorInvalidValue;
  prm.tiles = prm.n_mt * prm.n_nt;
  prm.wait_polls = g_wait_polls.load(std::memory_order_relaxed);
  prm.withhold_cta = g_withhold_cta.load(std::memory_order_relaxed);

  CUtensorMap mP, mZ, mT;
  const cuuint64_t V = (cuuint64_t)p.V;
  {
    const cuuint64_t dims[2] = {V, (cuuint64_t)p.r};
    const cuuint64_t str[1] = {V * 2};
    const cuuint32_t box[2] = {64, 64};
    if (!encode(&mP, p.P, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {V, (cuuint64_t)p.K, (cuuint64_t)p.B};
    const cuuint64_t str[2] = {V * 2, V * 2 * (cuuint64_t)p.K};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)(p.src == 0 ? 128 : 1)};  // final draw: plain loads
    if (!encode(&mZ, p.base_logits, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  mT = mZ;  // the final draw reads its rows with ordinary loads
  CUtensorMap mA = mP;  // unused unless A rows are staged
  if (p.a_stage_in != nullptr) {
    const cuuint64_t dims[2] = {(cuuint64_t)p.r, (cuuint64_t)p.B};
    const cuuint64_t str[1] = {(cuuint64_t)p.a_stage_stride * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!encode(&mA, p.a_stage_in, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const int grid = p.sup_groups;
  if (p.sup_tiles != prm.tiles || grid < 1 || grid > prm.tiles) return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;

  if (p.src == 0) return cudaLaunchKernelEx(&cfg, tile_tc_kernel<false>, prm, mP, mZ, mT, mA);
  return cudaLaunchKernelEx(&cfg, tile_tc_kernel<true>, prm, mP, mZ, mT, mA);
}

}  // namespace ds
