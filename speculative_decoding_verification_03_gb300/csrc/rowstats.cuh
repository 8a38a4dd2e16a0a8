// Row statistics and per-position decisions of the streaming row pass
// (rowpass.cu).
//
// Per vocabulary row ("Speculative Decoding: Draft, EAGLE, MTP", section "one
// speculative step"): the raw maximum m, the first argmax, and
// E = sum_{v != argmax} exp((z_v - m) / tau), so that ln S = log1p(E) and the
// AV feature logit(q_max) = -ln E ("Adaptive Verification without a
// confidence head", section "Scoring the distribution").
#pragma once

#include <cfloat>
#include <climits>

#include "avfit_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr uint32_t kNegInfBf16x2 = 0xff80ff80u;
constexpr uint32_t kNegInfF32 = 0xff800000u;

struct alignas(16) Part {
  float m;
  float E;
  int arg;
  uint32_t flags;
};

__device__ __forceinline__ int kept_len_of(const RowPassParams &P, int b) {
  if (!P.draft_len) return P.K;
  int k = __ldg(P.draft_len + b);
  return k < 0 ? 0 : (k > P.K ? P.K : k);
}

__device__ __forceinline__ float row_scale(const RowPassParams &P, int b) {
  const float tau = __ldg(P.temperature + b);
  return tau > 0.f ? kLog2e / tau : kLog2e;  // greedy (and invalid) rows at tau = 1
}

__device__ __forceinline__ Part load_stats_cg(const sv_row_stats_t *p) {
  const int4 v = __ldcg(reinterpret_cast<const int4 *>(p));
  Part r;
  r.m = __int_as_float(v.x);
  r.E = __int_as_float(v.y);
  r.arg = v.z;
  r.flags = (uint32_t)v.w;
  return r;
}

__device__ __forceinline__ void store_stats(sv_row_stats_t *p, const Part &s) {
  int4 v;
  v.x = __float_as_int(s.m);
  v.y = __float_as_int(s.E);
  v.z = s.arg;
  v.w = (int)s.flags;
  *reinterpret_cast<int4 *>(p) = v;
}

// Combine the partial statistics of two disjoint element sets of one row.
__device__ __forceinline__ Part combine(Part A, Part B, float c) {
  const bool b_empty = (B.arg == INT_MAX);
  const bool a_empty = (A.arg == INT_MAX);
  if (b_empty) {
    A.flags |= B.flags;
    if (isnan(B.E)) A.flags |= SV_FLAG_NONFINITE;
    return A;
  }
  if (a_empty) {
    B.flags |= A.flags;
    if (isnan(A.E)) B.flags |= SV_FLAG_NONFINITE;
    return B;
  }
  const bool a_wins = (A.m > B.m) || (A.m == B.m && A.arg < B.arg);
  Part W = a_wins ? A : B;
  const Part L = a_wins ? B : A;
  W.E = W.E + (L.E + 1.0f) * ex2_approx((L.m - W.m) * c);
  W.flags |= L.flags;
  return W;
}

// The math warps' partials of one item, lane w holding warp w's (the other
// lanes hold empty partials), combined across the warp.  The result is the
// same as combining them one by one (up to rounding):
//   M = the largest max; the winner = the lowest argmax attaining it;
//   E = the winner's own sum plus, for every other partial,
//       (E_w + 1) 2^((m_w - M) c), its maximum re-admitted as an ordinary
//       element.
// The exponentials are evaluated in parallel and summed in a fixed butterfly
// order, so the item's latency does not grow with a chain of dependent
// shuffles and MUFU operations (the pipes the math warps keep busy).
// Warps cover disjoint elements, so argmaxes differ between partials.
__device__ __forceinline__ Part combine_warp(const Part mine, float c) {
  const bool empty = mine.arg == INT_MAX;
  Part R;
  R.flags = __reduce_or_sync(0xffffffffu, mine.flags | ((empty && isnan(mine.E)) ? (uint32_t)SV_FLAG_NONFINITE : 0u));
  R.m = warp_max(empty ? -INFINITY : mine.m);
  R.arg = warp_min_i((!empty && mine.m == R.m) ? mine.arg : INT_MAX);
  float term = 0.f;
  if (!empty) term = mine.arg == R.arg ? mine.E : (mine.E + 1.0f) * ex2_approx((mine.m - R.m) * c);
  R.E = __shfl_sync(0xffffffffu, warp_sum(term), 0);
  return R;
}

__device__ __forceinline__ float logit_at(const void *base, int dtype, long long idx) {
  if (dtype == SV_BF16) {
    const uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(base) + idx);
    return __uint_as_float(((uint32_t)h) << 16);
  }
  return __ldg(reinterpret_cast<const float *>(base) + idx);
}

// ---------------------------------------------------------------------------
// Math-warp state and the running-max update.
// ---------------------------------------------------------------------------
struct WarpState {
  float M;    // warp-uniform running max of the raw logits
  float nbh;  // fl(-M * c)
  float nbl;  // -M * c - nbh, exactly
  int arg;    // warp-uniform index of the excluded first max
  float A;    // this lane's sum of 2^(z * c + nbh)
  uint32_t flags;
};

__device__ __forceinline__ void state_reset(WarpState &s) {
  s.M = -INFINITY;
  s.nbh = 0.f;
  s.nbl = 0.f;
  s.arg = INT_MAX;
  s.A = 0.f;
  s.flags = 0;
}

// The warp max rose to wm, attained first at element gidx (already excluded
// by its owner lane).  Rescale the lane sums to the new max:
//   A' = (A * 2^nbl_old + [lane 0] * 1) * 2^((M_old - M_new) c - nbl_new)
// where the "+1" re-admits the previous first max, now an ordinary element.
__device__ __forceinline__ void state_rise(WarpState &s, float wm, int gidx, float c, int lane) {
  const float Mold = s.M, nbl_old = s.nbl;
  s.M = wm;
  s.nbh = __fmul_rn(-wm, c);
  s.nbl = fmaf(-wm, c, -s.nbh);
  const float scale = ex2_approx((Mold - wm) * c - s.nbl);
  const float fold = fmaf(nbl_old, kLn2, 1.0f);
  s.A = fmaf(s.A, fold, lane == 0 ? 1.0f : 0.0f) * scale;
  s.arg = gidx;
}

template <int kDtype>
struct Elems;

template <>
struct Elems<SV_BF16> {
  static constexpr int kPerVec = 8;
  __device__ __forceinline__ static float get(const uint4 &w, int k) {
    const uint32_t x = (k >> 1) == 0 ? w.x : (k >> 1) == 1 ? w.y : (k >> 1) == 2 ? w.z : w.w;
    return (k & 1) ? bf16hi(x) : bf16lo(x);
  }
  __device__ __forceinline__ static void kill(uint4 &w, int k) {
    const uint32_t mask = (k & 1) ? 0xffff0000u : 0x0000ffffu;
    const uint32_t ninf = kNegInfBf16x2 & mask;
    switch (k >> 1) {
      case 0: w.x = (w.x & ~mask) | ninf; break;
      case 1: w.y = (w.y & ~mask) | ninf; break;
      case 2: w.z = (w.z & ~mask) | ninf; break;
      default: w.w = (w.w & ~mask) | ninf; break;
    }
  }
  __device__ __forceinline__ static uint4 neg_inf() { return make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2); }
  __device__ __forceinline__ static float vmax1(const uint4 &v) {
    const uint32_t m = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
    return fmaxf(bf16lo(m), bf16hi(m));
  }
  // a vector's maximum kept packed (as a bf16 pair), and its value
  using PM = uint32_t;
  __device__ __forceinline__ static PM pmax(const uint4 &v) { return bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w)); }
  __device__ __forceinline__ static PM pmax2(PM a, PM b) { return bf16x2_max(a, b); }
  __device__ __forceinline__ static float pval(PM m) { return fmaxf(bf16lo(m), bf16hi(m)); }
  // element `local` of the staged data := -inf
  __device__ __forceinline__ static void kill_smem(uint4 *ring, int local) {
    reinterpret_cast<unsigned short *>(ring)[local] = (unsigned short)0xff80u;
  }
  __device__ __forceinline__ static float vmax(const uint4 (&w)[kVecPerThread]) {
    uint32_t m0 = bf16x2_max(w[0].x, w[0].y), m1 = bf16x2_max(w[0].z, w[0].w);
#pragma unroll
    for (int j = 1; j < kVecPerThread; ++j) {
      m0 = bf16x2_max(m0, bf16x2_max(w[j].x, w[j].y));
      m1 = bf16x2_max(m1, bf16x2_max(w[j].z, w[j].w));
    }
    const uint32_t m = bf16x2_max(m0, m1);
    return fmaxf(bf16lo(m), bf16hi(m));
  }
};

template <>
struct Elems<SV_FP32> {
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static float get(const uint4 &w, int k) {
    const uint32_t x = k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w;
    return __uint_as_float(x);
  }
  __device__ __forceinline__ static void kill(uint4 &w, int k) {
    switch (k) {
      case 0: w.x = kNegInfF32; break;
      case 1: w.y = kNegInfF32; break;
      case 2: w.z = kNegInfF32; break;
      default: w.w = kNegInfF32; break;
    }
  }
  __device__ __forceinline__ static uint4 neg_inf() { return make_uint4(kNegInfF32, kNegInfF32, kNegInfF32, kNegInfF32); }
  __device__ __forceinline__ static float vmax1(const uint4 &v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  using PM = float;
  __device__ __forceinline__ static PM pmax(const uint4 &v) { return vmax1(v); }
  __device__ __forceinline__ static PM pmax2(PM a, PM b) { return fmaxf(a, b); }
  __device__ __forceinline__ static float pval(PM m) { return m; }
  __device__ __forceinline__ static void kill_smem(uint4 *ring, int local) {
    reinterpret_cast<uint32_t *>(ring)[local] = kNegInfF32;
  }
  __device__ __forceinline__ static float vmax(const uint4 (&w)[kVecPerThread]) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(w[j].x), __uint_as_float(w[j].y)),
                         fmaxf(__uint_as_float(w[j].z), __uint_as_float(w[j].w))));
    return m;
  }
};

// The running-max raise.  pm[j] is the max of this lane's vector j from the
// first pass (kept in registers; -inf past the stage's end), so the lane's
// first element equal to wm lies in its first vector with pm[j] == wm, and
// only that vector is read again.  The lane owning the first copy of wm
// overwrites it with -inf in shared memory (the stage is this warp's until
// released, and only this lane reads that vector), then the lane sums are
// rescaled.
template <int kDtype>
__device__ __forceinline__ void stage_rise(WarpState &s, uint4 *ring, int tid, int lane, int e0, float c, float wm,
                                                const typename Elems<kDtype>::PM (&pm)[kVecPerThread]) {
  using E = Elems<kDtype>;
  int jv = -1;
#pragma unroll
  for (int j = kVecPerThread - 1; j >= 0; --j)
    if (E::pval(pm[j]) == wm) jv = j;
  int cand = INT_MAX;
  if (jv >= 0) {
    const int vi = tid + jv * kConsumers;
    const uint4 v = ring[vi];
    int k0 = E::kPerVec - 1;
#pragma unroll
    for (int k = E::kPerVec - 2; k >= 0; --k)
      if (E::get(v, k) == wm) k0 = k;
    cand = e0 + vi * E::kPerVec + k0;
  }
  const int gidx = warp_min_i(cand);
  if (cand == gidx) E::kill_smem(ring, gidx - e0);
  __syncwarp();
  state_rise(s, wm, gidx, c, lane);
}

// exp2 terms of one 16-byte vector in packed pairs: fma2 for the arguments,
// two MUFU ex2, add2 into four pair accumulators.
template <int kDtype>
__device__ __forceinline__ void vec_exp_acc(const uint4 &v, float2 cc, float2 nb, float2 (&acc)[4]) {
  using E = Elems<kDtype>;
#pragma unroll
  for (int p = 0; p < E::kPerVec / 2; ++p) {
    float2 t = __ffma2_rn(make_float2(E::get(v, 2 * p), E::get(v, 2 * p + 1)), cc, nb);
    t.x = ex2_approx(t.x);
    t.y = ex2_approx(t.y);
    acc[p & 3] = __fadd2_rn(acc[p & 3], t);
  }
}

// One stage in shared memory, read twice: vector j of this lane is vector
// vi = tid + j * kConsumers of the stage, its element k sits at row index
// e0 + vi * kPerVec + k.  Pass 1 takes the stage max (and raises the warp max
// when needed, see stage_rise), pass 2 sums the exp2 terms.  Full stages take
// a path without per-vector bounds checks.
template <int kDtype>
__device__ __forceinline__ void consume_stage(WarpState &s, uint4 *ring, int nvec, int tid, int lane, int e0,
                                              float c) {
  using E = Elems<kDtype>;
  const uint4 *base = ring + tid;
  const bool full = nvec == kVecPerStage;
  if (full) {
    // per-vector maxima kept for a raise (about half of a row's stages raise
    // some warp's running max)
    typename E::PM pm[kVecPerThread];
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) pm[j] = E::pmax(base[j * kConsumers]);
    typename E::PM m = pm[0];
#pragma unroll
    for (int j = 1; j < kVecPerThread; ++j) m = E::pmax2(m, pm[j]);
    const float wm = warp_max(E::pval(m));
    if (wm > s.M) stage_rise<kDtype>(s, ring, tid, lane, e0, c, wm, pm);  // warp-uniform
  } else {
    // a row's last stage: vectors past nvec count as -inf
    typename E::PM pm[kVecPerThread];
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) pm[j] = E::pmax(tid + j * kConsumers < nvec ? base[j * kConsumers] : E::neg_inf());
    typename E::PM m = pm[0];
#pragma unroll
    for (int j = 1; j < kVecPerThread; ++j) m = E::pmax2(m, pm[j]);
    const float wm = warp_max(E::pval(m));
    if (wm > s.M) stage_rise<kDtype>(s, ring, tid, lane, e0, c, wm, pm);  // warp-uniform
  }
  const float2 cc = make_float2(c, c), nb = make_float2(s.nbh, s.nbh);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if (full) {
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) vec_exp_acc<kDtype>(base[j * kConsumers], cc, nb, acc);
  } else {
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j)
      if (tid + j * kConsumers < nvec) vec_exp_acc<kDtype>(base[j * kConsumers], cc, nb, acc);
  }
  s.A += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
}

// Scalar elements (ragged row ends): one value per lane, index idx.
__device__ __forceinline__ void consume_scalar(WarpState &s, float v, int idx, int lane, float c) {
  const float wm = warp_max(v);
  if (wm > s.M) {
    const int cand = (v == wm) ? idx : INT_MAX;
    const int gidx = warp_min_i(cand);
    if (cand == gidx) v = -INFINITY;
    state_rise(s, wm, gidx, c, lane);
  }
  s.A += ex2_approx(fmaf(v, c, s.nbh));
}


// ---------------------------------------------------------------------------
// Decisions and the refit terms.
// ---------------------------------------------------------------------------
// q * 2^32 rounded to the nearest integer (ties away from zero), by integer
// operations on the fp32 encoding; |q| < 2^30.  The fused refit's sums are
// exact in this fixed point, so they do not depend on the order of the adds.
__device__ __forceinline__ long long fixed_2p32(float q) {
  const uint32_t bits = __float_as_uint(q);
  const int e = (int)((bits >> 23) & 0xffu);
  if (e == 0 || e == 0xff) return 0;  // zero, subnormal (< 2^-126) or not finite
  const long long m = (long long)((bits & 0x7fffffu) | 0x800000u);
  const int sh = e - 118;  // q * 2^32 = m * 2^(e - 150 + 32)
  long long v;
  if (sh >= 0) v = m << (sh < 38 ? sh : 38);
  else if (sh > -26) v = (m + (1ll << (-sh - 1))) >> (-sh);
  else v = 0;
  return (bits >> 31) ? -v : v;
}

// Acceptance test u < p(d)/q(d) at one position, in fp64 ("Accelerating
// Large Language Model Decoding with Speculative Sampling", Algorithm 2):
// ln p(d) = (z_t(d) - m_t) / tau - ln S_t and likewise for q.  The fp32 fast
// path below defers to this one whenever it is not certain.
__device__ __forceinline__ bool reject_fp64(float zt, float zd, const Part &T, const Part &D, double invtau,
                                            double u) {
  const double lnSt = log1p((double)T.E), lnSd = log1p((double)D.E);
  const double lq = ((double)zd - (double)D.m) * invtau - lnSd;
  double ratio;
  if (lq == -INFINITY) {
    ratio = INFINITY;
  } else {
    const double lp = ((double)zt - (double)T.m) * invtau - lnSt;
    ratio = exp(lp - lq);
  }
  return !(u < ratio);
}

// fp32 acceptance test u < p(d)/q(d) from the two logits at the drafted
// token and the rows' statistics (tau > 0, d in range); inside an error band
// around the boundary it defers to the exact fp64 test.
__device__ __forceinline__ bool reject_pre(float u, float lu, float zt, float zd, const Part &T, const Part &D,
                                           float lnSt, float lnSd, float inv_f, float tau_f) {
  const float A = (zt - T.m) * inv_f, Bq = (zd - D.m) * inv_f;
  const float dl = (A - lnSt) - (Bq - lnSd);
  const float band = 2e-6f + 4e-7f * (fabsf(A) + fabsf(Bq) + lnSt + lnSd + fabsf(lu));
  if (u != 0.f && fabsf(dl - lu) > band) return !(lu < dl);
  return reject_fp64(zt, zd, T, D, 1.0 / (double)tau_f, (double)u);
}
// the same test with its logarithms taken here: ln S = log1p(E), ln u
__device__ __forceinline__ bool reject_values(float u, float zt, float zd, const Part &T, const Part &D, float tau_f) {
  return reject_pre(u, logf(u), zt, zd, T, D, log1pf(T.E), log1pf(D.E), 1.f / tau_f, tau_f);
}

// AV feature and confidence of a draft row (fp32, as in finish_verify).
__device__ __forceinline__ float av_feature(float E) {
  float x = E > 0.f ? -logf(E) : 30.f;
  return x > 30.f ? 30.f : (x < -30.f ? -30.f : x);
}
__device__ __forceinline__ float av_conf(const RowPassParams &P, int i, float x) {
  return 1.0f / (1.0f + expf(-fmaf(__ldcg(P.theta), x, __ldcg(P.theta + 1 + i))));
}

// One label's refit terms as 2^-32 fixed point (one lane).
__device__ __forceinline__ void fit_label(const RowPassParams &P, int i, float x, float conf, bool accepted) {
  const float y = accepted ? 1.0f : 0.0f;
  const float r = conf - y, w = conf * (1.0f - conf);
  const float q[kFitQ] = {r * x, w * x * x, r, w * x, w, 1.0f};
#pragma unroll
  for (int j = 0; j < kFitQ; ++j) atomicAdd(P.fitacc + i * kFitQ + j, (unsigned long long)fixed_2p32(q[j]));
}

}  // namespace sv
