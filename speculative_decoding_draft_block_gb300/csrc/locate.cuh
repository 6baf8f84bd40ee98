// Draw of one row from its chunk and group records (the "locate"), run by
// sample_locate_kernel with one CTA per row.
#pragma once
#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include "common.cuh"
#include "fastpath.cuh"
#include "internal.h"
#include "sampling.cuh"

namespace ds {
namespace {

constexpr int kLocThreads = 256;  // threads drawing one row

struct LocShared {
  float arow[1024];
  float part[kLocThreads / 32][32];
  float bias[32];
  int found;
  int N;
  DF excl, S, theta;
  ChunkRec crec;
};


__device__ __forceinline__ DF shfl_up_df(DF v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

__device__ __forceinline__ bool df_gt(DF a, DF b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

// The drawn token's E row into the staged A operand of the next step (warp).
template <typename Tin>
__device__ __forceinline__ void stage_e_row(const SampleParams& p, int b, int tok, int lane) {
  if (p.a_stage_out == nullptr) return;
  const int n16 = p.r * (int)sizeof(Tin) / 16;
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const Tin*>(p.E) + (size_t)tok * p.r);
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<Tin*>(p.a_stage_out) + (size_t)b * p.a_stage_stride);
  for (int i = lane; i < n16; i += 32) dst[i] = __ldg(src + i);
}

// Warp-wide inclusive double-float prefix sum.
__device__ __forceinline__ DF warp_incl_scan(DF v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF w = shfl_up_df(v, o);
    if (lane >= o) v = df_add(w, v);
  }
  return v;
}

__device__ __forceinline__ DF shfl_df(DF v, int l) {
  return {__shfl_sync(0xffffffffu, v.hi, l), __shfl_sync(0xffffffffu, v.lo, l)};
}

// One row, in three levels: (1) combine the row's group records (exact
// power-of-two rescale, double-float prefix) and find the group where the CDF
// crosses u*S; (2) scan that group's chunk records to find the crossing chunk;
// (3) recompute that chunk's 32 weights with the arithmetic its record used
// and pick the token: x = min{i : u*S < C_i}. Levels 1 and 2 run in warp 0
// alone. Every load that does not depend on an earlier result is issued
// together at the start (group records, seed, the row's token and temperature;
// then the E row of the bias, only stored for level 3), so that each level
// costs one round of loads. Called by kLocThreads threads (tid), with `sync` a
// barrier over exactly those threads; sgrp holds the row's group records
// (up to sup_stride). `step` is the 1-based draft position (p.step outside
// the persistent draft kernel).
template <typename Tin, typename Sync>
__device__ __forceinline__ void locate_row(const SampleParams& p, int b, int step, int tid,
                                           LocShared& sm, ChunkRec* sgrp, Sync sync) {
  const int lane = tid & 31, wid = tid >> 5;
  const int nc = p.n_chunks;
  const int r = p.r;
  const int mt = b / p.sup_rows;
  const int g_lo = first_group(p, mt);
  const int ng = last_group(p, mt) - g_lo + 1;
  // group records and the seed first: they do not depend on the row's context
  const uint4* gsrc = reinterpret_cast<const uint4*>(p.supers + (size_t)b * p.sup_stride);
  uint4 gv[8];
  uint64_t seed = p.seed;
  if (wid == 0) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = u * 32 + lane;
      if (i < ng) gv[u] = __ldcg(gsrc + i);
    }
    if (p.seed_ptr != nullptr) seed = *p.seed_ptr;  // after the dependent wait
  }
  const RowInputs rin = load_row_inputs(p, b, step);  // in flight with the records
  const RowCtx c = make_row_ctx<Tin>(p, b, rin, step);
  if (c.mode == kSkip) return;
  const Tin* Erow = bias_row<Tin>(p, b, c);
  float erow[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = tid + q * kLocThreads;
    erow[q] = (c.a_token >= 0 && k < r) ? to_f32(Erow[k]) : 0.f;
  }
  if (wid == 0) {
    uint4* dst = reinterpret_cast<uint4*>(sgrp);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = u * 32 + lane;
      if (i < ng) dst[i] = gv[u];
    }
    for (int i0 = 32 * 8; i0 < ng; i0 += 32 * 8) {  // more than 256 groups (SIMT tiles)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < ng) gv[u] = __ldcg(gsrc + i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < ng) dst[i] = gv[u];
      }
    }
  }

  if (wid == 0) {
    const DF u01 = uniform_df(seed, (uint32_t)b, c.upos, c.ustage);
    __syncwarp();
    const int seg = (ng + 31) / 32;
    const int c0 = min(ng, lane * seg), c1 = min(ng, c0 + seg);
    if (c.mode == kGreedyMarkov) {
      ChunkRec best = group_empty();
      for (int i = c0; i < c1; ++i) {
        const ChunkRec rr = sgrp[i];
        if (greedy_better(rr, best)) best = rr;
      }
      for (int o = 16; o > 0; o >>= 1) {
        const ChunkRec ov = shfl_xor_rec(best, o);
        if (greedy_better(ov, best)) best = ov;
      }
      const bool bad_idx = best.idx < 0 || best.idx >= p.V;  // no finite logit (or a bad record)
      const int bx = bad_idx ? 0 : best.idx;
      stage_e_row<Tin>(p, b, bx, lane);
      if (lane == 0) {
        if (bad_idx) report(p.status, kErrNonfinite);
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
      sm.found = -1;
    } else {
      // ---- level 1: global reference, prefix over the groups, crossing group ----
      int N = 0;
      if (c.mode == kSampleMarkov) {
        int lm = INT_MIN;
        for (int i = c0; i < c1; ++i) lm = max(lm, sgrp[i].ref);
        for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, o));
        N = lm;
      }
      DF tot = {0.f, 0.f};
      for (int i = c0; i < c1; ++i) tot = df_add(tot, rec_scaled(sgrp[i], N));
      const DF inc = warp_incl_scan(tot, lane);
      DF excl = shfl_up_df(inc, 1);
      if (lane == 0) excl = DF{0.f, 0.f};
      const DF S = shfl_df(inc, 31);
      int gsel = -1;
      DF gexcl = {0.f, 0.f}, theta = {0.f, 0.f};
      if (S.hi > 0.f && isfinite(S.hi)) {
        theta = df_mul(u01, S);
        const unsigned hit = __ballot_sync(0xffffffffu, c1 > c0 && df_gt(inc, theta));
        if (hit) {
          // the crossing group is within the first lane whose prefix passes u*S
          const int l = __ffs(hit) - 1;
          if (lane == l) {
            DF run = excl;
            for (int i = c0; i < c1; ++i) {
              const DF incl = df_add(run, rec_scaled(sgrp[i], N));
              if (df_gt(incl, theta)) {
                gsel = i;
                gexcl = run;
                break;
              }
              run = incl;
            }
          }
          gsel = __shfl_sync(0xffffffffu, gsel, l);
          gexcl = shfl_df(gexcl, l);
        }
        if (gsel < 0) {  // u*S at the very top (or rounding): last group with mass
          int gi = ng - 1;
          while (gi > 0 && !(rec_scaled(sgrp[gi], N).hi > 0.f)) --gi;
          gsel = gi;
          const DF sc = rec_scaled(sgrp[gi], N);
          gexcl = df_add(S, DF{-sc.hi, -sc.lo});
        }
      }
      if (gsel < 0) {
        stage_e_row<Tin>(p, b, 0, lane);
        if (lane == 0) {
          report(p.status, kErrNonfinite);
          p.tokens_out[c.out_index] = 0;
        }
        sm.found = -1;
      } else {
        // ---- level 2: the chunks of the crossing group ----
        const int g = g_lo + gsel;
        const int mt0 = mt * p.sup_nt;
        const int ta = max(group_tile0(p, g), mt0), tb = min(group_tile0(p, g + 1), mt0 + p.sup_nt);
        const int ch_lo = (ta - mt0) * p.sup_cpt, ch_hi = min((tb - mt0) * p.sup_cpt, nc);
        const ChunkRec* crow = p.chunks + b;  // chunk i of row b at crow[i * B]
        DF run = gexcl, fexcl = gexcl, lexcl = gexcl;
        int found = -1, last = -1;
        ChunkRec frec = group_empty(), lrec = group_empty();
        for (int base = ch_lo; base < ch_hi && found < 0; base += 128) {
          ChunkRec rr[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = base + 32 * u + lane;
            rr[u] = i < ch_hi ? ld_rec(crow + (size_t)i * p.B) : group_empty();
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (found >= 0) break;
            const int i = base + 32 * u + lane;
            const DF v = rec_scaled(rr[u], N);
            const DF ic = warp_incl_scan(v, lane);
            DF ex = shfl_up_df(ic, 1);
            if (lane == 0) ex = DF{0.f, 0.f};
            const DF incl = df_add(run, ic);
            const DF exa = df_add(run, ex);
            const unsigned hit = __ballot_sync(0xffffffffu, i < ch_hi && df_gt(incl, theta));
            const unsigned mass = __ballot_sync(0xffffffffu, i < ch_hi && v.hi > 0.f);
            if (hit) {
              const int l = __ffs(hit) - 1;
              found = base + 32 * u + l;
              fexcl = shfl_df(exa, l);
              frec = {__shfl_sync(0xffffffffu, rr[u].hi, l), 0.f, __shfl_sync(0xffffffffu, rr[u].ref, l),
                      __shfl_sync(0xffffffffu, rr[u].idx, l)};
            } else {
              if (mass) {
                const int l = 31 - __clz(mass);
                last = base + 32 * u + l;
                lexcl = shfl_df(exa, l);
                lrec = {0.f, 0.f, __shfl_sync(0xffffffffu, rr[u].ref, l), __shfl_sync(0xffffffffu, rr[u].idx, l)};
              }
              run = shfl_df(incl, 31);
            }
          }
        }
        if (found < 0) {  // rounding left u*S past the group's in-order total
          found = last >= 0 ? last : ch_lo;
          fexcl = last >= 0 ? lexcl : gexcl;
          frec = last >= 0 ? lrec : ld_rec(crow + (size_t)found * p.B);
        }
        if (lane == 0) {
          sm.found = found;
          sm.excl = fexcl;
          sm.crec = frec;
          sm.N = N;
          sm.S = S;
          sm.theta = theta;
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = tid + q * kLocThreads;
    if (k < r) sm.arow[k] = erow[q];
  }
  sync();
  if (sm.found < 0) return;  // greedy row done, or no mass
  const int chunk = sm.found;
  const int col0 = chunk * 32;
  const int n = min(32, p.V - col0);
  const int N = sm.N;
  const DF S = sm.S, theta = sm.theta;

  // ---- level 3: recompute the crossing chunk: logits first, then the bias (k split over warps) ----
  float zl = 0.f, tl = 0.f;
  if (wid == 0) {
    zl = (c.zrow && lane < n) ? to_f32(reinterpret_cast<const Tin*>(c.zrow)[col0 + lane]) : 0.f;
    tl = (c.trow && lane < n) ? to_f32(reinterpret_cast<const Tin*>(c.trow)[col0 + lane]) : 0.f;
  }
  const bool token_major = p.P_t != nullptr;
  if (token_major) {
    // 8 threads per token, each over 8-element groups part, part + 8, ...
    const int j = tid >> 3, part = tid & 7;
    float acc = 0.f;
    if (c.a_token >= 0 && j < n) {
      const Tin* row = reinterpret_cast<const Tin*>(p.P_t) + (size_t)(col0 + j) * r;
      const int groups = r >> 3;
      for (int g0 = part; g0 < groups; g0 += 32) {
        float v[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (g0 + 8 * u < groups) load8(row + (g0 + 8 * u) * 8, v[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (g0 + 8 * u < groups) {
            const float* a = sm.arow + (g0 + 8 * u) * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = __fmaf_rn(a[e], v[u][e], acc);
          }
      }
    }
    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
    if (part == 0) sm.bias[j] = acc;
  } else {
    float acc = 0.f;
    if (c.a_token >= 0) {
      const int per = r / (kLocThreads / 32);
      const int k0 = wid * per;
      const Tin* P = reinterpret_cast<const Tin*>(p.P) + (size_t)k0 * p.V + col0 + (lane < n ? lane : 0);
      for (int kb = 0; kb < per; kb += 32) {
        float pv[32];
#pragma unroll
        for (int u8 = 0; u8 < 32; ++u8) pv[u8] = (kb + u8 < per) ? to_f32(P[(size_t)(kb + u8) * p.V]) : 0.f;
#pragma unroll
        for (int u8 = 0; u8 < 32; ++u8)
          if (kb + u8 < per) acc = __fmaf_rn(sm.arow[k0 + kb + u8], pv[u8], acc);
      }
    }
    sm.part[wid][lane] = acc;
  }
  sync();
  if (wid == 0) {
    float bsum = 0.f;
    if (token_major)
      bsum = sm.bias[lane];
    else
      for (int w = 0; w < kLocThreads / 32; ++w) bsum = __fadd_rn(bsum, sm.part[w][lane]);
    // weights with the arithmetic of the chunk's record (idx -2: tensor-core fast path)
    float w = 0.f;
    int e = 0;
    if (c.mode == kSampleMarkov) {
      const ChunkRec cr = sm.crec;
      const int ref = cr.ref;
      if (lane < n && ref != kEmptyRef) {
        if (cr.idx == -2)
          w = fast_w1(zl, bsum, make_g16_from(c.g), ref);
        else
          w = weight_rel(zl, bsum, c.g, ref);
      }
      e = (ref == kEmptyRef) ? -300 : max(ref - N, -300);
    } else if (lane < n) {
      if (sm.crec.idx == -2) {  // fast-path record of the final draw
        const G16 g16 = make_g16_from(c.g);
        w = fast_w1(tl, 0.f, g16, c.Np);
        if (c.mode == kResidual) w = residual_w(w, fast_w1(zl, bsum, g16, c.Nq), c.Rhi, c.Rlo);
      } else {
        w = weight_rel(tl, 0.f, c.g, c.Np);
        if (c.mode == kResidual) {
          const float wq = weight_rel(zl, bsum, c.g, c.Nq);
          float d = __fmaf_rn(-wq, c.Rhi, w);
          d = __fmaf_rn(-wq, c.Rlo, d);
          w = fmaxf(d, 0.f);
        }
      }
    }
    if (!(w >= 0.f) || !isfinite(w)) w = 0.f;
    DF pre = {pow2_scale(w, e), 0.f};
    for (int o = 1; o < 32; o <<= 1) {
      const DF v = shfl_up_df(pre, o);
      if (lane >= o) pre = df_add(v, pre);
    }
    const DF incl = df_add(sm.excl, pre);
    const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && df_gt(incl, theta));
    const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
    const int xl = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
    const float wx = __shfl_sync(0xffffffffu, w, xl);
    stage_e_row<Tin>(p, b, col0 + xl, lane);
    if (lane == 0) {
      if (!pos) report(p.status, kErrNonfinite);
      p.tokens_out[c.out_index] = col0 + xl;
      if (p.src == 0) {
        p.q_token[c.out_index] = pow2_scale(div_by_df(wx, S), e);
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
}  // namespace ds
