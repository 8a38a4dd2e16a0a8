// Residual / bonus sampling by inverse CDF.
//
// "Speculative Decoding: Draft, EAGLE, MTP", section "one speculative step":
// at the first rejection a the emitted token is drawn from the normalised
// positive residual max(p_a - q_a, 0); when every verified draft passed, the
// bonus token is drawn from p_k.  The worked two-token example of footnote 1
// of "Adaptive Verification without a confidence head" (residual [1, 0]) is
// the same rule.  The token is the smallest v with C(v) > u * R, where C is
// the running sum of the weights in vocabulary order and R their total.
//
// Two phases, all on the device:
//   1. per_cta CTAs per sequence; each warp sums the weights of 256-element
//      sub-chunks (8 per lane, four sub-chunks' 16-byte loads in flight per
//      lane, shuffle reduction, no block barrier) into subsum[b][j];
//   2. the last CTA to finish (atomic counter) scans the sub-chunk sums in
//      fp64 (block-wide prefix sum), finds the sub-chunk where the CDF
//      crosses u * R, and one warp recomputes its 256 weights and locates the
//      token with a warp prefix sum.
// Weights: p_v = 2^(z_t c + nbt) up to a common factor (which cancels in
// C(v) / R); residual r_v = p_v * (1 - e^delta_v) where
// delta_v = ln q_v - ln p_v < 0, with 1 - e^delta from a Taylor polynomial
// near 0 so that nearly equal p and q do not cancel.
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

// -(e^d - 1) for |d| <= 0.5 from the Taylor series of e^d - 1 truncated
// after d^8 / 8! (relative truncation error below 1e-8 on that interval).
__device__ __forceinline__ float one_minus_exp_small(float d) {
  float p = 1.f / 40320.f;
  p = fmaf(p, d, 1.f / 5040.f);
  p = fmaf(p, d, 1.f / 720.f);
  p = fmaf(p, d, 1.f / 120.f);
  p = fmaf(p, d, 1.f / 24.f);
  p = fmaf(p, d, 1.f / 6.f);
  p = fmaf(p, d, 0.5f);
  p = fmaf(p, d, 1.f);
  return -(p * d);
}

template <int kDtype>
__device__ __forceinline__ void load8(const void *base, long long row_off, int v0, int V, bool vec_ok, float (&z)[8]) {
  if (kDtype == SV_BF16) {
    const unsigned short *p = reinterpret_cast<const unsigned short *>(base) + row_off;
    if (vec_ok && v0 + 8 <= V) {
      const uint4 w = __ldg(reinterpret_cast<const uint4 *>(p + v0));
      z[0] = bf16lo(w.x); z[1] = bf16hi(w.x); z[2] = bf16lo(w.y); z[3] = bf16hi(w.y);
      z[4] = bf16lo(w.z); z[5] = bf16hi(w.z); z[6] = bf16lo(w.w); z[7] = bf16hi(w.w);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) z[k] = (v0 + k < V) ? __uint_as_float(((uint32_t)__ldg(p + v0 + k)) << 16) : 0.f;
    }
  } else {
    const float *p = reinterpret_cast<const float *>(base) + row_off;
    if (vec_ok && v0 + 8 <= V) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(p + v0));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(p + v0 + 4));
      z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w; z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) z[k] = (v0 + k < V) ? __ldg(p + v0 + k) : 0.f;
    }
  }
}

struct RowPtrs {
  long long t_off, d_off;
  bool t_vec, d_vec;
};

// Weights of the eight elements v0..v0+7 given their logits.
__device__ __forceinline__ void weights_from(const SampleTask &t, int kind, int v0, int V, const float (&zt)[8],
                                             const float (&zd)[8], float (&r)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float w = 0.f;
    if (v0 + k < V) {
      const float p = ex2_approx(fmaf(zt[k], t.c, t.nbt));
      if (kind == kTaskResidual) {
        const float delta = fmaf(zd[k] - zt[k], t.invtau, t.k0_hi) + t.k0_lo;
        if (p > 0.f && delta < 0.f) {
          const float om = delta > -0.5f ? one_minus_exp_small(delta) : 1.f - ex2_approx(delta * kLog2e);
          w = p * om;
        }
      } else {
        w = p;
      }
    }
    r[k] = w;
  }
}

// The eight weights of `lane` in sub-chunk j (elements j*256 + lane*8 ..).
template <int kDtype>
__device__ __forceinline__ void weights8(const SampleParams &P, const SampleTask &t, int kind, const RowPtrs &R, int j,
                                         int lane, float (&r)[8]) {
  const int v0 = j * kSubChunk + lane * 8;
  float zt[8], zd[8];
  load8<kDtype>(P.target, R.t_off, v0, P.V, R.t_vec, zt);
  if (kind == kTaskResidual) load8<kDtype>(P.draft, R.d_off, v0, P.V, R.d_vec, zd);
  weights_from(t, kind, v0, P.V, zt, zd, r);
}

__device__ __forceinline__ float sum8(const float (&r)[8]) {
  return ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
}

// Sub-chunk sums of sub-chunks [j0, j1): warp w takes groups of kSampleUnroll
// consecutive sub-chunks and issues all their loads before reducing.
template <int kDtype>
__device__ __forceinline__ void subchunk_sums(const SampleParams &P, const SampleTask &t, int kind, const RowPtrs &R,
                                              int j0, int j1, float *subsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int jb = j0 + warp * kSampleUnroll; jb < j1; jb += kSampleWarps * kSampleUnroll) {
    float zt[kSampleUnroll][8], zd[kSampleUnroll][8];
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) {
      const int v0 = (jb + u) * kSubChunk + lane * 8;
      if (jb + u < j1) {
        load8<kDtype>(P.target, R.t_off, v0, P.V, R.t_vec, zt[u]);
        if (kind == kTaskResidual) load8<kDtype>(P.draft, R.d_off, v0, P.V, R.d_vec, zd[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) {
      if (jb + u >= j1) break;
      float r[8];
      weights_from(t, kind, (jb + u) * kSubChunk + lane * 8, P.V, zt[u], zd[u], r);
      const float s = warp_sum(sum8(r));
      if (lane == 0) subsum[jb + u] = s;
    }
  }
}

// Exclusive prefix of v over the block in thread order (fp64); total returned via *tot.
__device__ __forceinline__ double block_excl_scan_d(double v, double *red, double *tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  double base = 0.0, all = 0.0;
  for (int w = 0; w < kSampleWarps; ++w) {
    if (w < warp) base += red[w];
    all += red[w];
  }
  __syncthreads();
  *tot = all;
  return base + inc - v;
}

template <int kDtype>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleParams P) {
  __shared__ double red_d[kSampleWarps];
  __shared__ int s_last, s_jstar;
  __shared__ double s_pexcl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / P.per_cta;
  const int part = blockIdx.x - b * P.per_cta;
  const SampleTask t = P.tasks[b];
  if (t.kind == kTaskNone) return;
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;
  int kind = t.kind;

  RowPtrs R;
  R.t_off = ((long long)b * (P.K + 1) + t.a) * (long long)P.V;
  R.d_off = ((long long)b * P.K + t.a) * (long long)P.V;
  R.t_vec = ((reinterpret_cast<uintptr_t>(P.target) + (uintptr_t)R.t_off * kEsz) & 15) == 0;
  R.d_vec = kind == kTaskResidual && ((reinterpret_cast<uintptr_t>(P.draft) + (uintptr_t)R.d_off * kEsz) & 15) == 0;
  float *subsum = P.subsum + (size_t)b * P.nsub;

  // Phase 1: sub-chunk sums of this CTA's share of the row.
  const int per = (P.nsub + P.per_cta - 1) / P.per_cta;
  const int j0 = part * per, j1 = min(P.nsub, j0 + per);
  subchunk_sums<kDtype>(P, t, kind, R, j0, j1, subsum);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(P.smp_cnt + b, 1u);
    s_last = (old == (uint32_t)P.per_cta - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Phase 2 (last CTA of this sequence): locate the crossing of u * R.
  const int q = (P.nsub + kSampleThreads - 1) / kSampleThreads;
  const int ja = tid * q, jb = min(P.nsub, ja + q);
  for (int attempt = 0; attempt < 2; ++attempt) {
    double mine = 0.0;
    for (int j = ja; j < jb; ++j) mine += (double)__ldcg(subsum + j);
    double Rtot;
    const double excl = block_excl_scan_d(mine, red_d, &Rtot);
    if (!(Rtot > 0.0) && kind == kTaskResidual && attempt == 0) {
      // Zero residual mass (rounding only): sample p_a instead, and say so.
      if (tid == 0) atomicOr(P.status, SV_FLAG_ZERO_RESIDUAL);
      kind = kTaskBonus;
      subchunk_sums<kDtype>(P, t, kind, R, 0, P.nsub, subsum);
      __syncthreads();
      __threadfence();
      continue;
    }
    const double T = t.u * Rtot;
    if (tid == 0) s_jstar = INT_MAX;
    __syncthreads();
    double run = excl;
    for (int j = ja; j < jb; ++j) {
      const double nxt = run + (double)__ldcg(subsum + j);
      if (nxt > T) {
        atomicMin(&s_jstar, j);
        break;
      }
      run = nxt;
    }
    __syncthreads();
    if (s_jstar == INT_MAX) {
      // u * R at or past the total by rounding: the last sub-chunk with mass.
      if (tid == 0) {
        int jl = P.nsub - 1;
        while (jl > 0 && !(__ldcg(subsum + jl) > 0.f)) --jl;
        s_jstar = jl;
      }
      __syncthreads();
    }
    const int jstar = s_jstar;
    if (tid == jstar / q) {
      double pe = excl;
      for (int j = ja; j < jstar; ++j) pe += (double)__ldcg(subsum + j);
      s_pexcl = pe;
    }
    __syncthreads();
    if (warp == 0) {
      // Prefix sum over the 256 weights of sub-chunk jstar (8 per lane).
      float r[8];
      weights8<kDtype>(P, t, kind, R, jstar, lane, r);
      float pre[8];
      pre[0] = r[0];
#pragma unroll
      for (int k = 1; k < 8; ++k) pre[k] = pre[k - 1] + r[k];
      double inc = (double)pre[7];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
      }
      const double base = s_pexcl + inc - (double)pre[7];
      const int v0 = jstar * kSubChunk + lane * 8;
      int cand = INT_MAX, back = -1;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (cand == INT_MAX && r[k] > 0.f && base + (double)pre[k] > T) cand = v0 + k;
        if (r[k] > 0.f) back = v0 + k;
      }
      cand = warp_min_i(cand);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) back = max(back, __shfl_xor_sync(0xffffffffu, back, o));
      if (lane == 0) {
        int tok = cand != INT_MAX ? cand : (back >= 0 ? back : t.argmax_t);
        if (tok < 0 || tok >= P.V) tok = t.argmax_t;
        P.out_tokens[(size_t)b * (P.K + 1) + t.a] = tok;
      }
    }
    break;
  }
}

}  // namespace

cudaError_t launch_sample(const SampleParams &P, int grid, cudaStream_t stream) {
  if (P.dtype == SV_BF16) sample_kernel<SV_BF16><<<grid, kSampleThreads, 0, stream>>>(P);
  else sample_kernel<SV_FP32><<<grid, kSampleThreads, 0, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
