// AV refit: one IRLS / Newton step per round of decode steps.
//
// "Adaptive Verification without a confidence head", section "Fitting the
// coefficients": only drafts up to and including the first rejection carry a
// label (accepted = 1, the rejected one = 0); the log-likelihood loss is
// minimised by a second-order Taylor step H * delta = g with H of size
// (K+1)x(K+1) over the shared slope omega and the per-position intercepts
// beta_i; gradient and Hessian are accumulated over a round of N decode
// steps (O(K^2) memory), solved at the round's last step; each coefficient's
// step is damped by n / (n + c).
//
// With one shared slope and one intercept per position the Hessian is an
// arrow matrix: H_ww, a row H_wb[i] = sum w x over position i, and a diagonal
// H_bb[i] = sum w.  The solve is the Schur complement on omega:
//   delta_w = (g_w - sum_i H_wb[i] g_b[i] / d_i) / (H_ww - sum_i H_wb[i]^2 / d_i)
//   delta_b[i] = (g_b[i] - H_wb[i] delta_w) / d_i,  d_i = H_bb[i] (+ ridge)
// Layout: grid of G CTAs over the sequences; warp i of a CTA owns position i;
// lanes stride over the CTA's sequences and accumulate six fp64 sums; CTA
// partials go to the state buffer; the last CTA (atomic counter) adds them in
// CTA order (deterministic), updates the round accumulators and, at the end
// of the round, solves and writes theta.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

__global__ void avfit_kernel(const FitParams P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = P.K;
  const int G = gridDim.x;
  AvStateHeader *hdr = reinterpret_cast<AvStateHeader *>(P.state);
  double *acc = reinterpret_cast<double *>(P.state + kAvAccOff);
  double *parts = reinterpret_cast<double *>(P.state + kAvPartOff);
  __shared__ int s_last;

  const int per = (P.B + G - 1) / G;
  const int b0 = blockIdx.x * per, b1 = min(P.B, b0 + per);
  const int i = warp;
  double q[kFitQ] = {0, 0, 0, 0, 0, 0};
  if (i < K) {
    const double om = (double)__ldg(P.theta), be = (double)__ldg(P.theta + 1 + i);
    for (int b = b0 + lane; b < b1; b += 32) {
      int k = P.kept_len ? __ldg(P.kept_len + b) : K;
      k = k < 0 ? 0 : (k > K ? K : k);
      int a = __ldg(P.accept_len + b);
      a = a < 0 ? 0 : (a > k ? k : a);
      const bool labelled = (i < a) || (i == a && a < k);
      if (!labelled) continue;
      const double y = i < a ? 1.0 : 0.0;
      const double x = (double)__ldg(P.feature + (size_t)b * K + i);
      const double s = 1.0 / (1.0 + exp(-(om * x + be)));
      const double w = s * (1.0 - s);
      q[0] += (s - y) * x;
      q[1] += w * x * x;
      q[2] += (s - y);
      q[3] += w * x;
      q[4] += w;
      q[5] += 1.0;
    }
#pragma unroll
    for (int j = 0; j < kFitQ; ++j) q[j] = warp_sum_d(q[j]);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kFitQ; ++j) parts[((size_t)blockIdx.x * SV_MAX_K + i) * kFitQ + j] = q[j];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&hdr->cta_done, 1u);
    s_last = (old == (uint32_t)G - 1u);
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  hdr->cta_done = 0u;

  // acc layout: g[0..K] (g[0] = slope), Hww, Hwb[K], Hbb[K], n[K]
  double *g = acc;
  double *Hww = acc + (K + 1);
  double *Hwb = Hww + 1;
  double *Hbb = Hwb + K;
  double *n = Hbb + K;
  for (int ii = 0; ii < K; ++ii) {
    double t[kFitQ] = {0, 0, 0, 0, 0, 0};
    for (int c = 0; c < G; ++c)
      for (int j = 0; j < kFitQ; ++j) t[j] += __ldcg(parts + ((size_t)c * SV_MAX_K + ii) * kFitQ + j);
    g[0] += t[0];
    *Hww += t[1];
    g[1 + ii] += t[2];
    Hwb[ii] += t[3];
    Hbb[ii] += t[4];
    n[ii] += t[5];
  }
  hdr->step += 1u;
  if ((int)hdr->step < P.round_len) return;

  // End of round: damped Newton step over omega and the labelled intercepts.
  double ntot = 0.0, trace = *Hww;
  for (int ii = 0; ii < K; ++ii) {
    ntot += n[ii];
    trace += Hbb[ii];
  }
  if (ntot > 0.0) {
    const double ridge = 1e-9 * trace / (double)(K + 1);
    double a = *Hww + ridge, rhs = g[0];
    for (int ii = 0; ii < K; ++ii) {
      if (!(n[ii] > 0.0)) continue;
      const double d = Hbb[ii] + ridge;
      a -= Hwb[ii] * Hwb[ii] / d;
      rhs -= Hwb[ii] * g[1 + ii] / d;
    }
    if (a > 0.0 && isfinite(rhs)) {
      const double dw = rhs / a;
      const double c = (double)P.damping_c;
      P.theta[0] = (float)((double)P.theta[0] - ntot / (ntot + c) * dw);
      for (int ii = 0; ii < K; ++ii) {
        if (!(n[ii] > 0.0)) continue;
        const double db = (g[1 + ii] - Hwb[ii] * dw) / (Hbb[ii] + ridge);
        P.theta[1 + ii] = (float)((double)P.theta[1 + ii] - n[ii] / (n[ii] + c) * db);
      }
    } else {
      atomicOr(&hdr->status, SV_FLAG_FIT_SINGULAR);
    }
  }
  for (int j = 0; j < (int)kAvAccDoubles; ++j) acc[j] = 0.0;
  hdr->step = 0u;
}

__global__ void philox_kernel(uint64_t seed, int nb, int npos, uint32_t *out) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (long long)nb * npos) return;
  const int b = (int)(t / npos), pos = (int)(t - (long long)b * npos);
  const U32x4 r = philox4x32_10((uint32_t)b, (uint32_t)pos, 0u, 0u, (uint32_t)(seed & 0xffffffffu),
                                (uint32_t)(seed >> 32));
  uint4 v = make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]);
  reinterpret_cast<uint4 *>(out)[t] = v;
}

}  // namespace

cudaError_t launch_avfit(const FitParams &P, int grid, cudaStream_t stream) {
  const int block = 32 * (P.K > 0 ? P.K : 1);
  avfit_kernel<<<grid, block, 0, stream>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_philox(uint64_t seed, int nb, int npos, uint32_t *out, cudaStream_t stream) {
  const long long n = (long long)nb * npos;
  const int grid = (int)((n + 255) / 256);
  philox_kernel<<<grid, 256, 0, stream>>>(seed, nb, npos, out);
  return cudaGetLastError();
}

}  // namespace sv
