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
// lanes stride over the CTA's sequences and accumulate six sums; CTA
// partials go to the state buffer; in the last CTA (atomic counter) warp 0
// adds them in CTA order (deterministic), lane i owning position i, updates
// the fp64 round accumulators and, at the end of the round, solves with warp
// reductions for the Schur terms and writes theta.
#include "avfit_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

__global__ void avfit_kernel(const FitParams P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = P.K;
  const int G = gridDim.x;
  AvStateHeader *hdr = reinterpret_cast<AvStateHeader *>(P.state);
  float *parts = reinterpret_cast<float *>(P.state + kAvPartOff);
  __shared__ int s_last;

  // Per-label terms in fp32 (fp64 issues at a small fraction of the fp32 rate
  // on this GPU); per-CTA sums of at most a few hundred labels stay well
  // inside fp32 precision.  The round accumulators and the solve are fp64.
  const int per = (P.B + G - 1) / G;
  const int b0 = blockIdx.x * per, b1 = min(P.B, b0 + per);
  const int i = warp;
  if (i < K) {
    float q[kFitQ] = {0, 0, 0, 0, 0, 0};
    const float om = __ldg(P.theta), be = __ldg(P.theta + 1 + i);
    for (int b = b0 + lane; b < b1; b += 32) {
      int k = P.kept_len ? __ldg(P.kept_len + b) : K;
      k = k < 0 ? 0 : (k > K ? K : k);
      int a = __ldg(P.accept_len + b);
      a = a < 0 ? 0 : (a > k ? k : a);
      const bool labelled = (i < a) || (i == a && a < k);
      if (!labelled) continue;
      const float x = __ldg(P.feature + (size_t)b * K + i);
      const float sg = 1.0f / (1.0f + expf(-fmaf(om, x, be)));
      const float y = i < a ? 1.0f : 0.0f;
      const float w = sg * (1.0f - sg);
      q[0] = fmaf(sg - y, x, q[0]);
      q[1] = fmaf(w * x, x, q[1]);
      q[2] += sg - y;
      q[3] = fmaf(w, x, q[3]);
      q[4] += w;
      q[5] += 1.0f;
    }
#pragma unroll
    for (int j = 0; j < kFitQ; ++j) q[j] = warp_sum(q[j]);
    if (lane < kFitQ) {
      float v = q[0];
#pragma unroll
      for (int j = 1; j < kFitQ; ++j)
        if (lane == j) v = q[j];
      parts[((size_t)blockIdx.x * SV_MAX_K + i) * kFitQ + lane] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&hdr->cta_done, 1u);
    s_last = (old == (uint32_t)G - 1u);
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();

  // Last CTA, warp 0, lane i = position i: add the CTA partials (in CTA
  // order) and update the round.
  double t[kFitQ] = {0, 0, 0, 0, 0, 0};
  if (lane < K) {
    for (int c = 0; c < G; ++c)
#pragma unroll
      for (int j = 0; j < kFitQ; ++j) t[j] += (double)__ldcg(parts + ((size_t)c * SV_MAX_K + lane) * kFitQ + j);
  }
  av_round_update(P.state, P.theta, K, P.round_len, P.damping_c, t, lane);
  if (lane == 0) hdr->cta_done = 0u;
}

// End of an externally managed round: solve from the accumulators as they
// stand (for a batch sharded over several GPUs, the caller has replaced them
// by their sum over the shards) and clear them.  One warp.
__global__ void avsolve_kernel(unsigned char *state, float *theta, int K, float damping_c) {
  const double t[kFitQ] = {0, 0, 0, 0, 0, 0};
  av_round_update(state, theta, K, 1, damping_c, t, (int)threadIdx.x);
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

cudaError_t launch_avsolve(unsigned char *state, float *theta, int K, float damping_c, cudaStream_t stream) {
  avsolve_kernel<<<1, 32, 0, stream>>>(state, theta, K, damping_c);
  return cudaGetLastError();
}

cudaError_t launch_philox(uint64_t seed, int nb, int npos, uint32_t *out, cudaStream_t stream) {
  const long long n = (long long)nb * npos;
  const int grid = (int)((n + 255) / 256);
  philox_kernel<<<grid, 256, 0, stream>>>(seed, nb, npos, out);
  return cudaGetLastError();
}

}  // namespace sv
