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
// Two phases, all on the device, warp-level (no block barrier):
//   1. a grid-stride loop over groups (sequence b, four consecutive
//      256-element sub-chunks); a warp issues all of a group's 16-byte loads
//      (target and draft rows), then reduces each sub-chunk's weights with
//      shuffles into subsum[b][j];
//   2. the warp that completes a sequence's last group (atomic counter)
//      scans the sub-chunk sums in fp64, finds the sub-chunk where the CDF
//      crosses u * R, recomputes its 256 weights and locates the token with a
//      warp prefix sum.
// Weights: p_v = 2^(z_t c + nbt) up to a common factor (which cancels in
// C(v) / R); residual r_v = p_v * (1 - e^delta_v) where
// delta_v = ln q_v - ln p_v < 0, with 1 - e^delta from a Taylor polynomial
// near 0 so that nearly equal p and q do not cancel.
#include "sample_common.cuh"

namespace sv {

namespace {

// Grid-stride over groups (sequence b, kSampleUnroll consecutive sub-chunks);
// the warp that completes a sequence's last group finalises it.
template <int kDtype>
__global__ void __launch_bounds__(kSampleThreads, kSampleCtasPerSm) sample_kernel(const SampleParams P) {
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;
  const int lane = threadIdx.x & 31;
  const long long gwarp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int gps = (P.nsub + kSampleUnroll - 1) / kSampleUnroll;
  const long long ngroups = (long long)P.B * gps;
  // a row pass that gave up on a wait may have left tasks unwritten: draw
  // nothing (the status word already reports the time-out)
  if (__ldcg(P.status) & SV_FLAG_TIMEOUT) return;
  for (long long g = gwarp; g < ngroups; g += nwarps) {
    const int b = (int)(g / gps);
    const int jg = (int)(g - (long long)b * gps);
    const SampleTask t = P.tasks[b];
    if (t.kind == kTaskNone) continue;
    if (!((t.kind == kTaskResidual && t.a >= 0 && t.a < P.K) || (t.kind == kTaskBonus && t.a >= 0 && t.a <= P.K)))
      continue;  // never written by this launch's scans
    const RowPtrs R = row_ptrs(P, t, b, kEsz);
    const int j0 = jg * kSampleUnroll;
    group_sums<kDtype>(P, t, t.kind, R, j0, min(P.nsub, j0 + kSampleUnroll), lane, P.subsum + (size_t)b * P.nsub);
    int last = 0;
    if (lane == 0) {
      __threadfence();
      last = atomicAdd(P.smp_cnt + b, 1u) == (uint32_t)gps - 1u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      finalize_warp<kDtype>(P, t, b, R, lane);
    }
  }
}

}  // namespace

cudaError_t launch_sample(const SampleParams &P, int grid, cudaStream_t stream) {
  if (P.dtype == SV_BF16) sample_kernel<SV_BF16><<<grid, kSampleThreads, 0, stream>>>(P);
  else sample_kernel<SV_FP32><<<grid, kSampleThreads, 0, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
