// The end of one AV refit step, shared by the standalone refit kernel and
// the verify kernel's fused refit: add this step's per-position sums to the
// fp64 round accumulators and, at the end of the round, solve the arrow-shaped
// Newton system by the Schur complement on omega and update theta ("Adaptive
// Verification without a confidence head", "Fitting the coefficients").
#pragma once

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

// One warp; lane i < K holds t = the step's sums at position i:
// (sum (s-y) x, sum w x^2, sum (s-y), sum w x, sum w, label count).
// State layout: acc = [g (K+1; g[0] = slope), Hww, Hwb[K], Hbb[K], n[K]].
__device__ __forceinline__ void av_round_update(unsigned char *state, float *theta, int K, int round_len,
                                                float damping_c, const double (&t)[kFitQ], int lane) {
  AvStateHeader *hdr = reinterpret_cast<AvStateHeader *>(state);
  double *acc = reinterpret_cast<double *>(state + kAvAccOff);
  double *g = acc;
  double *Hww = acc + (K + 1);
  double *Hwb = Hww + 1;
  double *Hbb = Hwb + K;
  double *n = Hbb + K;
  double gb = 0, hwb = 0, hbb = 0, nn = 0;
  if (lane < K) {
    gb = __ldcg(g + 1 + lane) + t[2];
    hwb = __ldcg(Hwb + lane) + t[3];
    hbb = __ldcg(Hbb + lane) + t[4];
    nn = __ldcg(n + lane) + t[5];
  }
  const double gw = __ldcg(g) + warp_sum_d(lane < K ? t[0] : 0.0);
  const double hww = __ldcg(Hww) + warp_sum_d(lane < K ? t[1] : 0.0);
  const uint32_t step = hdr->step + 1u;
  bool solved = false;
  // round_len == 0: accumulate only; the caller ends the round (sv_av_solve)
  if (round_len > 0 && (int)step >= round_len) {
    const double ntot = warp_sum_d(nn);
    const double trace = hww + warp_sum_d(hbb);
    if (ntot > 0.0) {
      const double ridge = 1e-9 * trace / (double)(K + 1);
      const bool has = lane < K && nn > 0.0;
      const double d = hbb + ridge;
      const double s1 = warp_sum_d(has ? hwb * hwb / d : 0.0);
      const double s2 = warp_sum_d(has ? hwb * gb / d : 0.0);
      const double a = hww + ridge - s1, rhs = gw - s2;
      if (a > 0.0 && isfinite(rhs)) {
        const double dw = rhs / a;
        const double c = (double)damping_c;
        if (lane == 0) theta[0] = (float)((double)theta[0] - ntot / (ntot + c) * dw);
        if (has) {
          const double db = (gb - hwb * dw) / d;
          theta[1 + lane] = (float)((double)theta[1 + lane] - nn / (nn + c) * db);
        }
      } else if (lane == 0) {
        atomicOr(&hdr->status, SV_FLAG_FIT_SINGULAR);
      }
    }
    solved = true;
  }
  if (lane < K) {
    g[1 + lane] = solved ? 0.0 : gb;
    Hwb[lane] = solved ? 0.0 : hwb;
    Hbb[lane] = solved ? 0.0 : hbb;
    n[lane] = solved ? 0.0 : nn;
  }
  if (lane == 0) {
    g[0] = solved ? 0.0 : gw;
    *Hww = solved ? 0.0 : hww;
    hdr->step = solved ? 0u : step;
  }
}

// Fixed-point scale of the fused refit's integer accumulators: sums of the
// per-label terms are exact and independent of the order of the atomic adds.
constexpr double kFitFixedScale = 4294967296.0;  // 2^32

}  // namespace sv
