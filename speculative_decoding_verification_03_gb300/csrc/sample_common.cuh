// Residual / bonus weights and the per-sequence inverse-CDF finalisation,
// shared by the fused row-pass kernel and the standalone sampler.
//
// "Speculative Decoding: Draft, EAGLE, MTP", section "one speculative step":
// at the first rejection a the emitted token is drawn from the normalised
// positive residual max(p_a - q_a, 0); when every verified draft passed, the
// bonus token is drawn from p_k.  The token is the smallest v with
// C(v) > u * R, C the running sum of the weights in vocabulary order and R
// their total.  Weights: p_v = 2^(z_t c + nbt) up to a common factor (which
// cancels in C(v) / R); residual r_v = p_v * (1 - e^delta_v) where
// delta_v = ln q_v - ln p_v < 0, with 1 - e^delta from a Taylor polynomial
// near 0 so that nearly equal p and q do not cancel.
#pragma once

#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

// -(e^d - 1) for |d| <= 0.25 from the Taylor series of e^d - 1 truncated
// after d^7 / 7! (relative truncation error below 4e-9 on that interval).
__device__ __forceinline__ float one_minus_exp_small(float d) {
  float p = 1.f / 5040.f;
  p = fmaf(p, d, 1.f / 720.f);
  p = fmaf(p, d, 1.f / 120.f);
  p = fmaf(p, d, 1.f / 24.f);
  p = fmaf(p, d, 1.f / 6.f);
  p = fmaf(p, d, 0.5f);
  p = fmaf(p, d, 1.f);
  return -(p * d);
}

// Eight logits v0..v0+7 of a row as raw bits (bf16: one uint4; fp32: two).
struct Raw8 {
  uint4 a, b;
};

template <int kDtype>
__device__ __forceinline__ Raw8 load8(const void *base, long long row_off, int v0, int V, bool vec_ok) {
  Raw8 r;
  if (kDtype == SV_BF16) {
    const unsigned short *p = reinterpret_cast<const unsigned short *>(base) + row_off;
    if (vec_ok && v0 + 8 <= V) {
      r.a = __ldg(reinterpret_cast<const uint4 *>(p + v0));
    } else {
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = (v0 + k < V) ? (uint32_t)__ldg(p + v0 + k) : 0u;
      r.a = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    }
    r.b = make_uint4(0, 0, 0, 0);
  } else {
    const float *p = reinterpret_cast<const float *>(base) + row_off;
    if (vec_ok && v0 + 8 <= V) {
      r.a = __ldg(reinterpret_cast<const uint4 *>(p + v0));
      r.b = __ldg(reinterpret_cast<const uint4 *>(p + v0 + 4));
    } else {
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = (v0 + k < V) ? __float_as_uint(__ldg(p + v0 + k)) : 0u;
      r.a = make_uint4(h[0], h[1], h[2], h[3]);
      r.b = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
  return r;
}

template <int kDtype>
__device__ __forceinline__ float raw_at(const Raw8 &r, int k) {
  if (kDtype == SV_BF16) {
    const uint32_t w = (k >> 1) == 0 ? r.a.x : (k >> 1) == 1 ? r.a.y : (k >> 1) == 2 ? r.a.z : r.a.w;
    return (k & 1) ? bf16hi(w) : bf16lo(w);
  }
  const uint4 &q = k < 4 ? r.a : r.b;
  const int kk = k & 3;
  return __uint_as_float(kk == 0 ? q.x : kk == 1 ? q.y : kk == 2 ? q.z : q.w);
}

// A task written by another SM during the same kernel: read it from L2.
__device__ __forceinline__ SampleTask load_task_cg(const SampleTask *p) {
  static_assert(sizeof(SampleTask) % 8 == 0, "SampleTask is read as 8-byte words");
  SampleTask t;
  const int2 *src = reinterpret_cast<const int2 *>(p);
  int2 *dst = reinterpret_cast<int2 *>(&t);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(SampleTask) / 8); ++i) dst[i] = __ldcg(src + i);
  return t;
}

struct RowPtrs {
  long long t_off, d_off;
  bool t_vec, d_vec;
};

// Weights of the eight elements v0..v0+7.
template <int kDtype>
__device__ __forceinline__ void weights_from(const SampleTask &t, int kind, int v0, int V, const Raw8 &zt,
                                             const Raw8 &zd, float (&r)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float a = raw_at<kDtype>(zt, k);
    const float p = ex2_approx(fmaf(a, t.c, t.nbt));
    float w = p;
    if (kind == kTaskResidual) {
      const float delta = fmaf(raw_at<kDtype>(zd, k) - a, t.invtau, t.k0_hi) + t.k0_lo;
      const float om = delta > -0.25f ? one_minus_exp_small(delta) : 1.f - ex2_approx(delta * kLog2e);
      w = (p > 0.f && delta < 0.f) ? p * om : 0.f;
    }
    r[k] = (v0 + k < V) ? w : 0.f;
  }
}

// The sum of the weights of the eight elements v0..v0+7, two elements per
// packed fp32x2 instruction (each lane the same operations as weights_from).
template <int kDtype>
__device__ __forceinline__ float weights_sum8(const SampleTask &t, int kind, int v0, int V, const Raw8 &zt,
                                              const Raw8 &zd) {
  const float2 cc = make_float2(t.c, t.c), nb = make_float2(t.nbt, t.nbt);
  float2 acc = make_float2(0.f, 0.f);
  if (kind == kTaskResidual) {
    const float2 it = make_float2(t.invtau, t.invtau), kh = make_float2(t.k0_hi, t.k0_hi);
    const float2 kl = make_float2(t.k0_lo, t.k0_lo), l2e = make_float2(kLog2e, kLog2e);
    const float2 c7 = make_float2(1.f / 5040.f, 1.f / 5040.f), c6 = make_float2(1.f / 720.f, 1.f / 720.f);
    const float2 c5 = make_float2(1.f / 120.f, 1.f / 120.f), c4 = make_float2(1.f / 24.f, 1.f / 24.f);
    const float2 c3 = make_float2(1.f / 6.f, 1.f / 6.f), c2 = make_float2(0.5f, 0.5f), one = make_float2(1.f, 1.f);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const float2 a = make_float2(raw_at<kDtype>(zt, k), raw_at<kDtype>(zt, k + 1));
      const float2 b = make_float2(raw_at<kDtype>(zd, k), raw_at<kDtype>(zd, k + 1));
      float2 p = __ffma2_rn(a, cc, nb);
      p.x = ex2_approx(p.x);
      p.y = ex2_approx(p.y);
      const float2 d = __fadd2_rn(__ffma2_rn(__fadd2_rn(b, make_float2(-a.x, -a.y)), it, kh), kl);
      float2 q = c7;  // -(e^d - 1) by the truncated Taylor series (one_minus_exp_small)
      q = __ffma2_rn(q, d, c6);
      q = __ffma2_rn(q, d, c5);
      q = __ffma2_rn(q, d, c4);
      q = __ffma2_rn(q, d, c3);
      q = __ffma2_rn(q, d, c2);
      q = __ffma2_rn(q, d, one);
      const float2 sm = __fmul2_rn(q, d);
      float2 ex = __fmul2_rn(d, l2e);
      ex.x = ex2_approx(ex.x);
      ex.y = ex2_approx(ex.y);
      const float omx = d.x > -0.25f ? -sm.x : 1.f - ex.x, omy = d.y > -0.25f ? -sm.y : 1.f - ex.y;
      const float wx = (p.x > 0.f && d.x < 0.f && v0 + k < V) ? p.x * omx : 0.f;
      const float wy = (p.y > 0.f && d.y < 0.f && v0 + k + 1 < V) ? p.y * omy : 0.f;
      acc = __fadd2_rn(acc, make_float2(wx, wy));
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      float2 p = __ffma2_rn(make_float2(raw_at<kDtype>(zt, k), raw_at<kDtype>(zt, k + 1)), cc, nb);
      p.x = v0 + k < V ? ex2_approx(p.x) : 0.f;
      p.y = v0 + k + 1 < V ? ex2_approx(p.y) : 0.f;
      acc = __fadd2_rn(acc, p);
    }
  }
  return acc.x + acc.y;
}

template <int kDtype>
__device__ __forceinline__ void weights8(const SampleParams &P, const SampleTask &t, int kind, const RowPtrs &R, int j,
                                         int lane, float (&r)[8]) {
  const int v0 = j * kSubChunk + lane * 8;
  const Raw8 zt = load8<kDtype>(P.target, R.t_off, v0, P.V, R.t_vec);
  Raw8 zd;
  zd.a = zd.b = make_uint4(0, 0, 0, 0);
  if (kind == kTaskResidual) zd = load8<kDtype>(P.draft, R.d_off, v0, P.V, R.d_vec);
  weights_from<kDtype>(t, kind, v0, P.V, zt, zd, r);
}

__device__ __forceinline__ float sum8(const float (&r)[8]) {
  return ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
}

// Double-float numbers: an unevaluated sum hi + lo of two fp32 values, about
// 48 bits of significand (Dekker, "A floating-point technique for extending
// the available precision", 1971; Knuth's two-sum).  Used for the prefix sums
// of the draw, where fp64 would run at a small fraction of the fp32 rate on
// this GPU.  __fadd_rn keeps the compiler from reassociating the error terms.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fadd_rn(s, -a);
  const float e = __fadd_rn(__fadd_rn(a, -__fadd_rn(s, -bb)), __fadd_rn(b, -bb));
  return {s, e};
}

__device__ __forceinline__ DF fast_two_sum(float a, float b) {  // |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return {s, __fadd_rn(b, -__fadd_rn(s, -a))};
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ DF df_add_f(DF a, float b) {
  const DF s = two_sum(a.hi, b);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}

// a > b, decided on the double-float values
__device__ __forceinline__ bool df_gt(DF a, DF b) {
  return __fadd_rn(__fadd_rn(a.hi, -b.hi), __fadd_rn(a.lo, -b.lo)) > 0.f;
}

// u * R for an fp32 u, as a double-float (the product's error by an FMA)
__device__ __forceinline__ DF df_scale(float u, DF r) {
  const float p = __fmul_rn(u, r.hi);
  const float e = __fmaf_rn(u, r.hi, -p);
  return fast_two_sum(p, __fmaf_rn(u, r.lo, e));
}

__device__ __forceinline__ DF warp_incl_scan_df(DF v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    DF n;
    n.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
    n.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
    if (lane >= o) v = df_add(v, n);
  }
  return v;
}

__device__ __forceinline__ RowPtrs row_ptrs(const SampleParams &P, const SampleTask &t, int b, int esz) {
  RowPtrs R;
  R.t_off = ((long long)b * (P.K + 1) + t.a) * (long long)P.V;
  R.d_off = ((long long)b * P.K + t.a) * (long long)P.V;
  R.t_vec = ((reinterpret_cast<uintptr_t>(P.target) + (uintptr_t)R.t_off * esz) & 15) == 0;
  R.d_vec = t.kind == kTaskResidual && ((reinterpret_cast<uintptr_t>(P.draft) + (uintptr_t)R.d_off * esz) & 15) == 0;
  return R;
}

// One warp: sums of sub-chunks [j0, j1) (at most kSampleUnroll), loads first.
template <int kDtype>
__device__ __forceinline__ void group_sums(const SampleParams &P, const SampleTask &t, int kind, const RowPtrs &R,
                                           int j0, int j1, int lane, float *subsum) {
  Raw8 zt[kSampleUnroll], zd[kSampleUnroll];
#pragma unroll
  for (int u = 0; u < kSampleUnroll; ++u) {
    const int v0 = (j0 + u) * kSubChunk + lane * 8;
    zd[u].a = zd[u].b = zt[u].a = zt[u].b = make_uint4(0, 0, 0, 0);
    if (j0 + u < j1) {
      zt[u] = load8<kDtype>(P.target, R.t_off, v0, P.V, R.t_vec);
      if (kind == kTaskResidual) zd[u] = load8<kDtype>(P.draft, R.d_off, v0, P.V, R.d_vec);
    }
  }
#pragma unroll
  for (int u = 0; u < kSampleUnroll; ++u) {
    if (j0 + u < j1) {
      const float s = warp_sum(weights_sum8<kDtype>(t, kind, (j0 + u) * kSubChunk + lane * 8, P.V, zt[u], zd[u]));
      if (lane == 0) subsum[j0 + u] = s;
    }
  }
}

// One warp locates the token of sequence b from its sub-chunk sums.  Lane l
// owns sub-chunks [l q, l q + q); when q <= kFinalRegs they are read once into
// registers.  Prefix sums across sub-chunks are double-float (a prefix error
// of 1e-7 R would move the crossing at large V); inside the crossing
// sub-chunk the prefix is fp32 from the lane's start.
constexpr int kFinalRegs = 24;

template <int kDtype>
__device__ void finalize_warp(const SampleParams &P, const SampleTask &t, int b, const RowPtrs &R, int lane) {
  float *sub = P.subsum + (size_t)b * P.nsub;
  const int nsub = P.nsub;
  const int q = (nsub + 31) / 32;
  const int ja = min(nsub, lane * q), jb = min(nsub, ja + q);
  const bool in_regs = q <= kFinalRegs;
  const float u = (float)t.u;  // 24-bit uniform: exact
  int kind = t.kind;
  for (int attempt = 0; attempt < 2; ++attempt) {
    float v[kFinalRegs];
    DF mine = {0.f, 0.f};
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < kFinalRegs; ++k) v[k] = (ja + k < jb) ? __ldcg(sub + ja + k) : 0.f;
#pragma unroll
      for (int k = 0; k < kFinalRegs; ++k) mine = df_add_f(mine, v[k]);
    } else {
      for (int j = ja; j < jb; ++j) mine = df_add_f(mine, __ldcg(sub + j));
    }
    const DF incl = warp_incl_scan_df(mine, lane);
    DF Rtot;
    Rtot.hi = __shfl_sync(0xffffffffu, incl.hi, 31);
    Rtot.lo = __shfl_sync(0xffffffffu, incl.lo, 31);
    if (!(Rtot.hi > 0.f) && kind == kTaskResidual && attempt == 0) {
      // Zero residual mass (rounding only): sample p_a instead, and say so.
      if (lane == 0) atomicOr(P.status, SV_FLAG_ZERO_RESIDUAL);
      kind = kTaskBonus;
      for (int j0 = 0; j0 < nsub; j0 += kSampleUnroll)
        group_sums<kDtype>(P, t, kind, R, j0, min(nsub, j0 + kSampleUnroll), lane, sub);
      __syncwarp();
      __threadfence_block();
      continue;
    }
    const DF T = df_scale(u, Rtot);
    // the crossing sub-chunk: the first j with prefix(j) + s_j > T
    int cand = INT_MAX, last_pos = -1;
    DF pe = {0.f, 0.f};
    DF run = df_add(incl, {-mine.hi, -mine.lo});  // exclusive prefix of this lane
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < kFinalRegs; ++k) {
        if (ja + k < jb) {
          const float sj = v[k];
          if (sj > 0.f) last_pos = ja + k;
          const DF nxt = df_add_f(run, sj);
          if (cand == INT_MAX && df_gt(nxt, T)) {
            cand = ja + k;
            pe = run;
          }
          run = nxt;
        }
      }
    } else {
      for (int j = ja; j < jb; ++j) {
        const float sj = __ldcg(sub + j);
        if (sj > 0.f) last_pos = j;
        const DF nxt = df_add_f(run, sj);
        if (cand == INT_MAX && df_gt(nxt, T)) {
          cand = j;
          pe = run;
        }
        run = nxt;
      }
    }
    int jstar = warp_min_i(cand);
    DF pexcl;
    if (jstar != INT_MAX) {
      const int owner = __ffs(__ballot_sync(0xffffffffu, cand == jstar)) - 1;
      pexcl.hi = __shfl_sync(0xffffffffu, pe.hi, owner);
      pexcl.lo = __shfl_sync(0xffffffffu, pe.lo, owner);
    } else {
      // u * R at or past the total by rounding: the last sub-chunk with mass.
      int lp = last_pos;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
      jstar = lp < 0 ? 0 : lp;
      pexcl = df_add_f(Rtot, -__ldcg(sub + jstar));
    }
    // Prefix sum over the 256 weights of sub-chunk jstar (8 per lane).
    float r[8];
    weights8<kDtype>(P, t, kind, R, jstar, lane, r);
    float pre[8];
    pre[0] = r[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) pre[k] = pre[k - 1] + r[k];
    const DF incl2 = warp_incl_scan_df({pre[7], 0.f}, lane);
    const DF base = df_add(pexcl, df_add_f(incl2, -pre[7]));  // prefix before this lane's 8
    const int v0 = jstar * kSubChunk + lane * 8;
    int c2 = INT_MAX, back = -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (c2 == INT_MAX && r[k] > 0.f && df_gt(df_add_f(base, pre[k]), T)) c2 = v0 + k;
      if (r[k] > 0.f) back = v0 + k;
    }
    c2 = warp_min_i(c2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) back = max(back, __shfl_xor_sync(0xffffffffu, back, o));
    if (lane == 0) {
      int tok = c2 != INT_MAX ? c2 : (back >= 0 ? back : t.argmax_t);
      if (tok < 0 || tok >= P.V) tok = t.argmax_t;
      P.out_tokens[(size_t)b * (P.K + 1) + t.a] = tok;
    }
    break;
  }
}

}  // namespace sv
