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
  if (row >= p.B || chunk >= p.n_chunks) return;
  const RowCtx& c = rows[rl];
  if (c.mode == kSkip) return;
  const int col0 = chunk * 32;
  const int n = min(32, p.V - col0);
  float z[32], t[32];
  if (c.zrow) load_chunk<Tin>(c.zrow, col0, n, z);
  if (c.trow) load_chunk<Tin>(c.trow, col0, n, t);
  ChunkRec rec;
  if (n == 32)
    chunk_record<true>(c, F32Src{z}, acc, F32Src{t}, 32, col0, rec, p.status);
  else
    chunk_record<false>(c, F32Src{z}, acc, F32Src{t}, n, col0, rec, p.status);
  p.chunks[(size_t)row * p.n_chunks + chunk] = rec;
}

// ---- locate ------------------------------------------------------------------

__device__ __forceinline__ DF shfl_up_df(DF v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

__device__ __forceinline__ bool df_gt(DF a, DF b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ DF scaled_rec(const ChunkRec& r, int N) {
  const int e = (r.ref == kEmptyRef) ? -300 : max(r.ref - N, -300);
  return df_scale2(DF{r.hi, r.lo}, e);
}

// One CTA per row: combine the row's chunk records, locate the chunk where the
// CDF crosses u*S, recompute its 32 weights and pick the token. The records
// are staged once with independent 16-byte loads; the E row of the bias is
// prefetched alongside, and the P column loads of the crossing chunk are all
// issued before they are consumed, so the row costs few dependent round trips.
template <typename Tin>
__global__ void __launch_bounds__(kThreads) sample_locate_kernel(SampleParams p) {
  extern __shared__ ChunkRec srec[];
  __shared__ int s_int[kThreads / 32];
  __shared__ DF s_df[kThreads / 32];
  __shared__ float s_arow[1024];
  __shared__ float s_part[kThreads / 32][32];
  __shared__ int s_found;
  __shared__ DF s_excl;
  sm100::pdl_launch_dependents();
  sm100::pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const RowCtx c = make_row_ctx<Tin>(p, b);
  if (c.mode == kSkip) return;
  const int nc = p.n_chunks;
  const int r = p.r;
  const Tin* Erow = reinterpret_cast<const Tin*>(p.E) + (size_t)(c.a_token >= 0 ? c.a_token : 0) * r;
  float erow[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = tid + q * kThreads;
    erow[q] = (c.a_token >= 0 && k < r) ? to_f32(Erow[k]) : 0.f;
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.chunks + (size_t)b * nc);
    uint4* dst = reinterpret_cast<uint4*>(srec);
    for (int i0 = 0; i0 < nc; i0 += kThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kThreads + tid;
        if (i < nc) v[u] = __ldcg(src + i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kThreads + tid;
        if (i < nc) dst[i] = v[u];
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = tid + q * kThreads;
    if (k < r) s_arow[k] = erow[q];
  }
  __syncthreads();
  const int seg = (nc + kThreads - 1) / kThreads;
  const int c0 = min(nc, tid * seg), c1 = min(nc, c0 + seg);

  if (c.mode == kGreedyMarkov) {
    DF best = {kNegInf, 0.f};
    int bi = INT_MAX;
    for (int i = c0; i < c1; ++i) {
      const ChunkRec rr = srec[i];
      if (rr.idx < 0) continue;
      if (bi == INT_MAX || rr.hi > best.hi || (rr.hi == best.hi && rr.lo > best.lo)) {
        best = {rr.hi, rr.lo};
        bi = rr.idx;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const DF ov = {__shfl_xor_sync(0xffffffffu, best.hi, o), __shfl_xor_sync(0xffffffffu, best.lo, o)};
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool take = (oi != INT_MAX) &&
                        (bi == INT_MAX || ov.hi > best.hi || (ov.hi == best.hi && ov.lo > best.lo) ||
                         (ov.hi == best.hi && ov.lo == best.lo && oi < bi));
      if (take) {
        best = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      s_df[wid] = best;
      s_int[wid] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      DF bb = {kNegInf, 0.f};
      int bx = INT_MAX;
      for (int w = 0; w < kThreads / 32; ++w) {
        const DF v = s_df[w];
        const int iw = s_int[w];
        if (iw == INT_MAX) continue;
        if (bx == INT_MAX || v.hi > bb.hi || (v.hi == bb.hi && v.lo > bb.lo) ||
            (v.hi == bb.hi && v.lo == bb.lo && iw < bx)) {
          bb = v;
          bx = iw;
        }
      }
      if (bx == INT_MAX) {
        bx = 0;
        report(p.status, kErrNonfinite);
      }
      p.tokens_out[c.out_index] = bx;
      if (p.src == 0) {
        p.q_token[c.out_index] = 1.f;
        ds_row_stats st;
        st.sum_hi = 1.f;
        st.sum_lo = 0.f;
        st.ref = 0;
        st.argmax = bx;
        p.q_stats[c.out_index] = st;
      }
    }
    return;
  }

  // ---- sampling rows: global reference, prefix sums, crossing chunk ----
  int lm = INT_MIN;
  if (c.mode == kSampleMarkov)
    for (int i = c0; i < c1; ++i) lm = max(lm, srec[i].ref);
  for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, o));
  if (lane == 0) s_int[wid] = lm;
  __syncthreads();
  int N = 0;
  if (c.mode == kSampleMarkov) {
    N = s_int[0];
    for (int w = 1; w < kThreads / 32; ++w) N = max(N, s_int[w]);
  }
  DF tot = {0.f, 0.f};
  for (int i = c0; i < c1; ++i) tot = df_add(tot, scaled_rec(srec[i], N));
  DF inc = tot;
  for (int o = 1; o < 32; o <<= 1) {
    const DF v = shfl_up_df(inc, o);
    if (lane >= o) inc = df_add(v, inc);
  }
  DF prev = shfl_up_df(inc, 1);
  if (lane == 0) prev = DF{0.f, 0.f};
  if (lane == 31) s_df[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    DF wv = lane < kThreads / 32 ? s_df[lane] : DF{0.f, 0.f};
    for (int o = 1; o < 32; o <<= 1) {
      const DF v = shfl_up_df(wv, o);
      if (lane >= o) wv = df_add(v, wv);
    }
    if (lane < kThreads / 32) s_df[lane] = wv;
    if (lane == 0) s_found = INT_MAX;
  }
  __syncthreads();
  const DF wexcl = wid > 0 ? s_df[wid - 1] : DF{0.f, 0.f};
  const DF excl = df_add(wexcl, prev);
  const DF S = s_df[kThreads / 32 - 1];
  const double Sd = df_to_double(S);
  if (!(Sd > 0.0) || !isfinite(Sd)) {
    if (tid == 0) {
      report(p.status, kErrNonfinite);
      p.tokens_out[c.out_index] = 0;
    }
    return;
  }
  const double u = uniform_dev(p.seed, (uint32_t)b, c.upos, c.ustage);
  const double theta_d = u * Sd;
  const float th_hi = (float)theta_d;
  const DF theta = {th_hi, (float)(theta_d - (double)th_hi)};
  DF run = excl;
  int my_found = INT_MAX;
  DF my_excl = {0.f, 0.f};
  for (int i = c0; i < c1; ++i) {
    const DF incl = df_add(run, scaled_rec(srec[i], N));
    if (df_gt(incl, theta)) {
      my_found = i;
      my_excl = run;
      break;
    }
    run = incl;
  }
  if (my_found != INT_MAX) atomicMin(&s_found, my_found);
  __syncthreads();
  if (my_found != INT_MAX && my_found == s_found) s_excl = my_excl;
  if (tid == 0 && s_found == INT_MAX) {  // u*S at the very top: last chunk with mass
    int ch = nc - 1;
    while (ch > 0 && !(srec[ch].hi > 0.f)) --ch;
    s_found = ch;
    const DF sc = scaled_rec(srec[ch], N);
    s_excl = df_add(S, DF{-sc.hi, -sc.lo});
  }
  __syncthreads();
  const int chunk = s_found;
  const int col0 = chunk * 32;
  const int n = min(32, p.V - col0);

  // ---- recompute the crossing chunk: logits first, then the bias (k split over warps) ----
  float zl = 0.f, tl = 0.f;
  if (wid == 0) {
    zl = (c.zrow && lane < n) ? to_f32(reinterpret_cast<const Tin*>(c.zrow)[col0 + lane]) : 0.f;
    tl = (c.trow && lane < n) ? to_f32(reinterpret_cast<const Tin*>(c.trow)[col0 + lane]) : 0.f;
  }
  {
    float acc = 0.f;
    if (c.a_token >= 0) {
      const int per = r / (kThreads / 32);
      const int k0 = wid * per;
      const Tin* P = reinterpret_cast<const Tin*>(p.P) + (size_t)k0 * p.V + col0 + (lane < n ? lane : 0);
      for (int kb = 0; kb < per; kb += 32) {
        float pv[32];
#pragma unroll
        for (int u8 = 0; u8 < 32; ++u8) pv[u8] = (kb + u8 < per) ? to_f32(P[(size_t)(kb + u8) * p.V]) : 0.f;
#pragma unroll
        for (int u8 = 0; u8 < 32; ++u8)
          if (kb + u8 < per) acc = __fmaf_rn(s_arow[k0 + kb + u8], pv[u8], acc);
      }
    }
    s_part[wid][lane] = acc;
  }
  __syncthreads();
  if (wid == 0) {
    float bsum = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) bsum = __fadd_rn(bsum, s_part[w][lane]);
    // weights with the arithmetic of the chunk's record (idx -2: tensor-core fast path)
    float w = 0.f;
    int e = 0;
    if (c.mode == kSampleMarkov) {
      const ChunkRec cr = srec[chunk];
      const int ref = cr.ref;
      if (lane < n && ref != kEmptyRef) {
        if (cr.idx == -2)
          w = fast_w1(zl, bsum, make_g16(p.temperature[b]), (uint32_t)ref << 23);
        else
          w = weight_rel(zl, bsum, c.g, ref);
      }
      e = (ref == kEmptyRef) ? -300 : max(ref - N, -300);
    } else if (lane < n) {
      w = weight_rel(tl, 0.f, c.g, c.Np);
      if (c.mode == kResidual) {
        const float wq = weight_rel(zl, bsum, c.g, c.Nq);
        float d = __fmaf_rn(-wq, c.Rhi, w);
        d = __fmaf_rn(-wq, c.Rlo, d);
        w = fmaxf(d, 0.f);
      }
    }
    if (!(w >= 0.f) || !isfinite(w)) w = 0.f;
    DF pre = {ldexpf(w, e), 0.f};
    for (int o = 1; o < 32; o <<= 1) {
      const DF v = shfl_up_df(pre, o);
      if (lane >= o) pre = df_add(v, pre);
    }
    const DF incl = df_add(s_excl, pre);
    const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && df_gt(incl, theta));
    const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
    const int xl = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
    const float wx = __shfl_sync(0xffffffffu, w, xl);
    if (lane == 0) {
      if (!pos) report(p.status, kErrNonfinite);
      p.tokens_out[c.out_index] = col0 + xl;
      if (p.src == 0) {
        p.q_token[c.out_index] = (float)(ldexp((double)wx, e) / Sd);
        ds_row_stats st;
        st.sum_hi = S.hi;
        st.sum_lo = S.lo;
        st.ref = N;
        st.argmax = -1;
        p.q_stats[c.out_index] = st;
      }
    }
  }
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

size_t locate_smem_bytes(int32_t V) { return (size_t)num_chunks(V) * sizeof(ChunkRec); }

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
  const size_t smem = locate_smem_bytes(p.V);
  if (p.dtype == DS_BF16) {
    static cudaError_t attr = cudaFuncSetAttribute(
        sample_locate_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(sample_locate_kernel<__nv_bfloat16>, dim3(p.B), dim3(kThreads), smem, s, p);
  }
  static cudaError_t attr = cudaFuncSetAttribute(
      sample_locate_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr != cudaSuccess) return attr;
  return launch_pdl(sample_locate_kernel<float>, dim3(p.B), dim3(kThreads), smem, s, p);
}

}  // namespace ds
