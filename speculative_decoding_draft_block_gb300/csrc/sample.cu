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

namespace ds {

namespace {

constexpr int kThreads = 256;
constexpr int kPsStride = 8 * 36;  // 8 chunks of 32 floats padded to 36 (bank spread)

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
};

template <typename Tin>
__device__ RowCtx make_row_ctx(const SampleParams& p, int b) {
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
  if (b >= p.B) return c;
  const Tin* base = reinterpret_cast<const Tin*>(p.base_logits);
  const Tin* tgt = reinterpret_cast<const Tin*>(p.target_logits);
  const float T = p.temperature[b];
  const bool greedy = (T == 0.f);
  if (!greedy && !(T >= 1e-3f && T <= 1e3f)) {
    report(p.status, kErrInvalidArg);
    return c;
  }
  if (!greedy) c.g = make_gscale(T);
  if (p.src == 0) {
    const int k = p.step;  // 1-based
    int tok = (k == 1) ? p.anchor[b] : p.draft_tokens[(size_t)b * p.K + (k - 2)];
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
  } else {
    const FinalDesc d = p.final_desc[b];
    if (greedy || d.mode == kSkip) return c;
    c.mode = d.mode;
    c.trow = tgt + ((size_t)b * (p.K + 1) + d.row) * (size_t)p.V;
    c.Np = d.Np;
    c.upos = (uint32_t)(d.row + 1);
    c.ustage = DS_STAGE_RESAMPLE;
    c.out_index = b * (p.K + 1) + d.out_pos;
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

// Reduce one chunk of n (<= 32) tokens starting at token col0 to its record.
// z, bias, t hold the chunk's base logits, Markov bias and target logits.
// If w_out is given, the per-token weights (relative to rec.ref) and the
// running double-float prefix after each token are written too.
__device__ __forceinline__ void chunk_record(const RowCtx& c, const float* z, const float* bias,
                                             const float* t, int n, int col0, ChunkRec& rec,
                                             int32_t* status, float* w_out = nullptr,
                                             DF* prefix_out = nullptr) {
  rec.hi = 0.f;
  rec.lo = 0.f;
  rec.ref = 0;
  rec.idx = -1;
  bool bad = false;
  if (c.mode == kGreedyMarkov) {
    DF best = {kNegInf, 0.f};
    int bi = -1;
    for (int j = 0; j < n; ++j) {
      bad |= bad_logit(z[j]) || !(bias[j] == bias[j]);
      DF l = (z[j] == kNegInf) ? DF{kNegInf, 0.f} : two_sum(z[j], bias[j]);
      if (bi < 0 || l.hi > best.hi || (l.hi == best.hi && l.lo > best.lo)) {
        best = l;
        bi = col0 + j;
      }
    }
    rec.hi = best.hi;
    rec.lo = best.lo;
    rec.idx = bi;
  } else if (c.mode == kSampleMarkov) {
    float amax = kNegInf;
    for (int j = 0; j < n; ++j) {
      bad |= bad_logit(z[j]) || !(bias[j] == bias[j]);
      if (z[j] != kNegInf) amax = fmaxf(amax, scaled_hi(z[j], c.g));
    }
    if (amax == kNegInf) {
      rec.ref = kEmptyRef;
      if (w_out)
        for (int j = 0; j < n; ++j) {
          w_out[j] = 0.f;
          prefix_out[j] = {0.f, 0.f};
        }
    } else {
      const int ref = (int)rintf(amax);
      DF s = {0.f, 0.f};
      for (int j = 0; j < n; ++j) {
        const float w = exp2_rel(z[j], bias[j], c.g, ref);
        df_accumulate(s, w);
        if (w_out) {
          w_out[j] = w;
          prefix_out[j] = s;
        }
      }
      rec.hi = s.hi;
      rec.lo = s.lo;
      rec.ref = ref;
    }
  } else {  // kResidual / kBonus: weights on the row's global scale
    DF s = {0.f, 0.f};
    for (int j = 0; j < n; ++j) {
      bad |= bad_logit(t[j]);
      float w = exp2_rel(t[j], 0.f, c.g, c.Np);
      if (c.mode == kResidual) {
        bad |= bad_logit(z[j]) || !(bias[j] == bias[j]);
        const float wq = exp2_rel(z[j], bias[j], c.g, c.Nq);
        float d = __fmaf_rn(-wq, c.Rhi, w);
        d = __fmaf_rn(-wq, c.Rlo, d);
        w = fmaxf(d, 0.f);
      }
      df_accumulate(s, w);
      if (w_out) {
        w_out[j] = w;
        prefix_out[j] = s;
      }
    }
    rec.hi = s.hi;
    rec.lo = s.lo;
    rec.ref = 0;
  }
  if (bad) report(status, kErrNonfinite);
}

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
  chunk_record(c, z, acc, t, n, col0, rec, p.status);
  p.chunks[(size_t)row * p.n_chunks + chunk] = rec;
}

// ---- block helpers --------------------------------------------------------

__device__ __forceinline__ int block_max_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : INT_MIN;
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

__device__ __forceinline__ int block_min_int(int v, int* red) {
  return -block_max_int(-v, red);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) sample_locate_kernel(SampleParams p) {
  __shared__ int red[32];
  __shared__ DF tot_s[kThreads];
  __shared__ DF excl_s[kThreads];
  __shared__ float arow[1024];
  __shared__ float zs[32], bs[32], ts[32];
  __shared__ int found_s;
  __shared__ DF found_excl;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const RowCtx c = make_row_ctx<Tin>(p, b);
  if (c.mode == kSkip) return;
  const ChunkRec* rec = p.chunks + (size_t)b * p.n_chunks;
  const int nc = p.n_chunks;
  const int seg = (nc + kThreads - 1) / kThreads;
  const int c0 = min(nc, tid * seg), c1 = min(nc, c0 + seg);

  if (c.mode == kGreedyMarkov) {
    // argmax over chunk records, lowest token on ties
    DF best = {kNegInf, 0.f};
    int bi = INT_MAX;
    for (int i = c0; i < c1; ++i) {
      const ChunkRec r = rec[i];
      if (bi == INT_MAX || r.hi > best.hi || (r.hi == best.hi && r.lo > best.lo)) {
        best = {r.hi, r.lo};
        bi = r.idx;
      }
    }
    tot_s[tid] = best;
    red[0] = 0;
    __shared__ int idx_s[kThreads];
    idx_s[tid] = bi;
    __syncthreads();
    if (tid == 0) {
      DF bb = {kNegInf, 0.f};
      int bx = INT_MAX;
      for (int i = 0; i < kThreads; ++i) {
        if (idx_s[i] == INT_MAX) continue;
        const DF v = tot_s[i];
        if (bx == INT_MAX || v.hi > bb.hi || (v.hi == bb.hi && v.lo > bb.lo) ||
            (v.hi == bb.hi && v.lo == bb.lo && idx_s[i] < bx)) {
          bb = v;
          bx = idx_s[i];
        }
      }
      if (bx == INT_MAX || bx < 0) bx = 0;
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
  int local_max = INT_MIN;
  if (c.mode == kSampleMarkov)
    for (int i = c0; i < c1; ++i) local_max = max(local_max, rec[i].ref);
  const int N = (c.mode == kSampleMarkov) ? block_max_int(local_max, red) : 0;

  DF tot = {0.f, 0.f};
  for (int i = c0; i < c1; ++i) {
    const ChunkRec r = rec[i];
    const int e = (r.ref == kEmptyRef) ? -1000 : r.ref - N;
    tot = df_add(tot, df_scale2(DF{r.hi, r.lo}, max(e, -300)));
  }
  tot_s[tid] = tot;
  __syncthreads();
  if (tid == 0) {
    DF run = {0.f, 0.f};
    for (int i = 0; i < kThreads; ++i) {
      excl_s[i] = run;
      run = df_add(run, tot_s[i]);
    }
    tot_s[0] = run;  // total S
    found_s = INT_MAX;
  }
  __syncthreads();
  const DF S = tot_s[0];
  const double Sd = df_to_double(S);
  if (!(Sd > 0.0)) {
    if (tid == 0) {
      report(p.status, kErrNonfinite);
      p.tokens_out[c.out_index] = 0;
    }
    return;
  }
  const double u = uniform_dev(p.seed, (uint32_t)b, c.upos, c.ustage);
  const double theta = u * Sd;

  DF run = excl_s[tid];
  int my_found = INT_MAX;
  DF my_excl = {0.f, 0.f};
  for (int i = c0; i < c1; ++i) {
    const ChunkRec r = rec[i];
    const int e = (r.ref == kEmptyRef) ? -1000 : r.ref - N;
    const DF incl = df_add(run, df_scale2(DF{r.hi, r.lo}, max(e, -300)));
    if (df_to_double(incl) > theta) {
      my_found = i;
      my_excl = run;
      break;
    }
    run = incl;
  }
  const int cfound = block_min_int(my_found, red);
  if (my_found == cfound && cfound != INT_MAX) found_excl = my_excl;
  __syncthreads();

  int chunk = cfound;
  if (chunk == INT_MAX) {  // rounding left u*S at the very top: take the last chunk with mass
    if (tid == 0) {
      chunk = nc - 1;
      while (chunk > 0 && rec[chunk].hi == 0.f) --chunk;
      found_s = chunk;
      found_excl = df_add(S, DF{-rec[chunk].hi, -rec[chunk].lo});
    }
    __syncthreads();
    chunk = found_s;
  }

  // ---- recompute the crossing chunk with the tile kernel's arithmetic ----
  const int col0 = chunk * 32;
  const int n = min(32, p.V - col0);
  if (c.a_token >= 0) {
    const Tin* E = reinterpret_cast<const Tin*>(p.E);
    for (int k = tid; k < p.r; k += kThreads) arow[k] = to_f32(E[(size_t)c.a_token * p.r + k]);
  }
  __syncthreads();
  if (tid < 32) {
    const int col = col0 + tid;
    float acc = 0.f;
    if (c.a_token >= 0 && tid < n) {
      const Tin* P = reinterpret_cast<const Tin*>(p.P);
      for (int k = 0; k < p.r; ++k) acc = __fmaf_rn(arow[k], to_f32(P[(size_t)k * p.V + col]), acc);
    }
    bs[tid] = acc;
    zs[tid] = (c.zrow && tid < n) ? to_f32(reinterpret_cast<const Tin*>(c.zrow)[col]) : 0.f;
    ts[tid] = (c.trow && tid < n) ? to_f32(reinterpret_cast<const Tin*>(c.trow)[col]) : 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    float w[32];
    DF pre[32];
    ChunkRec chk;
    RowCtx cc = c;
    chunk_record(cc, zs, bs, ts, n, col0, chk, p.status, w, pre);
    const int e = (chk.ref == kEmptyRef) ? -1000 : chk.ref - N;
    const DF ex = found_excl;
    int x = -1;
    int last_pos = -1;
    for (int j = 0; j < n; ++j) {
      if (w[j] > 0.f) last_pos = j;
      const DF incl = df_add(ex, df_scale2(pre[j], max(e, -300)));
      if (w[j] > 0.f && df_to_double(incl) > theta) {
        x = j;
        break;
      }
    }
    if (x < 0) x = last_pos >= 0 ? last_pos : 0;  // recompute drifted from the record
    const int tok = col0 + x;
    p.tokens_out[c.out_index] = tok;
    if (p.src == 0) {
      const double q = ldexp((double)w[x], e) / Sd;
      p.q_token[c.out_index] = (float)q;
      ds_row_stats st;
      st.sum_hi = S.hi;
      st.sum_lo = S.lo;
      st.ref = N;
      st.argmax = -1;
      p.q_stats[c.out_index] = st;
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

cudaError_t launch_sample_locate(const SampleParams& p, cudaStream_t s) {
  if (p.dtype == DS_BF16)
    sample_locate_kernel<__nv_bfloat16><<<p.B, kThreads, 0, s>>>(p);
  else
    sample_locate_kernel<float><<<p.B, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ds
