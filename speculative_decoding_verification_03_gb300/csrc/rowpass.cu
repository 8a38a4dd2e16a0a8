// Row pass: one streaming read of every verified target and draft row.
//
// What it computes, per vocabulary row ("Speculative Decoding: Draft, EAGLE,
// MTP", section "one speculative step": both models return a distribution per
// drafted position): the raw maximum m, the first argmax, and
// E = sum_{v != argmax} exp((z_v - m) / tau), so that ln S = log1p(E) and the
// AV feature logit(q_max) = -ln E ("Adaptive Verification without a confidence
// head", section "Scoring the distribution").  When the last row of a sequence
// is done, the same CTA runs the sequence's left-to-right acceptance scan
// (section "algorithm loop in code" of the cheatsheet) and writes the
// sampling task for the residual or bonus row.
//
// GB300 design: a persistent grid, one CTA per SM, warp-specialised:
//   warp 12 (producer)    takes work items -- queued target rows and sample
//                         items first, then static rows from a global
//                         ticket -- and streams them with 1-D TMA bulk copies
//                         into a 4-stage shared-memory ring (54 KB stages,
//                         mbarrier complete_tx);
//   warps 0-11 (math)     read 16-byte vectors from shared memory, keep a
//                         warp-uniform running max (bf16x2 max + redux) and
//                         a per-lane sum of exp2 terms (packed fp32x2),
//                         exclude exactly one copy of the max, and publish one
//                         partial per warp and item; sample stages sum the
//                         residual / bonus weights per 256-element sub-chunk;
//   warps 13-15 (epilogue) take finished items from a shared counter, combine
//                         the 12 partials, merge row chunks, and run the
//                         early-exit walk of the sequence whose row they
//                         completed (decisions, AV scores and refit labels,
//                         queueing the next target row or the draw).
// Every wait is bounded (2 s by default); a time-out sets SV_FLAG_TIMEOUT,
// drains this CTA's in-flight copies and returns.
#include <cfloat>
#include <climits>

#include "avfit_common.cuh"
#include "rowstats.cuh"
#include "sample_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

namespace {

constexpr int kFlagFirst = 1;
constexpr int kFlagLast = 2;
constexpr int kFlagDone = 4;
constexpr int kFlagSample = 8;     // a residual/bonus item of the fused sampler
constexpr int kFlagResidual = 16;  // ... whose stage also holds the draft row
constexpr int kSampleHalfBytes = kStageBytes / 2;
constexpr int kItemSample = -2;    // PartInfo.item of a finished sample item
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp0 = kConsumerWarps + 1;  // .. + kEpiWarps - 1

// Per stage: the fields every math warp reads (one 16-byte shared load), the
// sample parameters (sample stages only) and the item's metadata, read only
// on the item's last stage.  A sample stage holds
// target elements [e0, e0 + n) in its first half and, for a residual, the
// draft row's same elements in its second half (n = nvec * 16 / esz).
struct StageHot {
  int e0;       // row element index of the first staged element
  int nvec;     // staged 16-byte vectors (per half for a sample stage)
  int flags;    // kFlagFirst | kFlagLast | kFlagDone | kFlagSample | kFlagResidual
  float c;      // log2(e) / tau
};

struct StageSample {  // sample stages only
  float nbt;    // weights 2^(z_t c + nbt)
  float invtau;
  float k0_hi, k0_lo;
  int b;        // the sequence
  int pad[3];
};

// Eight staged elements starting at element offset `off` of a stage half.
template <int kDtype>
__device__ __forceinline__ Raw8 smem_raw8(const uint8_t *half, int off) {
  Raw8 r;
  if (kDtype == SV_BF16) {
    r.a = *reinterpret_cast<const uint4 *>(half + off * 2);
    r.b = make_uint4(0, 0, 0, 0);
  } else {
    r.a = *reinterpret_cast<const uint4 *>(half + off * 4);
    r.b = *reinterpret_cast<const uint4 *>(half + off * 4 + 16);
  }
  return r;
}

struct StageCold {
  int item;
  int b;
  int sidx;   // statistics index inside the sequence: 2j (target j) or 2i+1 (draft i)
  int chunk;
  int x0, xn0, x1, xn1;  // elements read with plain loads on the LAST stage
  long long row_off;     // element offset of the row inside its tensor
  int is_target;
  int pad;
};

struct PartInfo {
  int item;
  int b;
  int sidx;
  int chunk;
  float c;
  int pad[3];
};


struct __align__(128) Smem {
  uint8_t ring[kStages][kStageBytes];
  StageHot hot[kStages];
  StageSample smpl[kStages];
  StageCold cold[kStages];
  PartInfo pinfo[kPartSlots];
  Part part[kPartSlots][kConsumerWarps];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t pfull[kPartSlots];
  uint64_t pempty[kPartSlots];
  int abort_flag;
  int epi_next;  // next partial item for the epilogue warps
};


// Slot -> (is_target, position) for the streaming mode.  Verify modes stream a
// sequence's rows from the highest position down: the rows a residual or a
// bonus re-reads are most often the low positions (a rejection at position i
// needs the first i drafts accepted), so those are read last and are still
// in L2 when the sequence completes.
__device__ __forceinline__ void slot_kind(int mode, int K, int slot, int &is_target, int &pos) {
  if (mode == kVerifyFull) {
    // slots: tK, d(K-1), t(K-1), ..., d0, t0
    is_target = !(slot & 1);
    pos = K - ((slot + 1) >> 1);
  } else if (mode == kVerifyTargets) {
    is_target = 1;
    pos = K - slot;
  } else {
    is_target = 0;
    pos = slot;
  }
}

__device__ __forceinline__ int rows_needed(const RowPassParams &P, int k) {
  if (P.mode == kVerifyFull) return 2 * k + 1;
  if (P.mode == kVerifyTargets) return k + 1;
  return P.K;
}

// ---------------------------------------------------------------------------
// Per-sequence completion (epilogue warp, all 32 lanes).
// ---------------------------------------------------------------------------

__device__ void finish_verify(const RowPassParams &P, int b, int lane) {
  const int K = P.K;
  const int k = kept_len_of(P, b);
  const float tau_f = __ldg(P.temperature + b);
  const bool bad_tau = !(tau_f >= 0.f);
  const bool greedy = !(tau_f > 0.f);
  // fp32 1/tau and log2(e)/tau, both correctly rounded (the row pass uses the
  // same scale for its statistics)
  const float inv_f = greedy ? 1.f : 1.f / tau_f;
  const float c_f = greedy ? kLog2e : kLog2e / tau_f;
  const size_t rowb = (size_t)P.V;
  uint32_t flags = 0;
  if (lane == 0) {
    if (bad_tau) flags |= SV_FLAG_BAD_TEMP;
    if (P.draft_len) {
      const int kr = __ldg(P.draft_len + b);
      if (kr < 0 || kr > K) flags |= SV_FLAG_BAD_LEN;
    }
  }
  const sv_row_stats_t *st = P.stats + (size_t)b * (2 * K + 1);

  // Lane i <= k: statistics of target row i; lane i < k: those of draft row
  // i and the acceptance test at position i.  The test runs in fp32 and is
  // kept when |ln u - ln(p/q)| exceeds a bound on its rounding error (a few
  // fp32 ulps of each term); otherwise the warp redoes it in fp64.
  bool reject = false, unsure = false, in_range = false;
  int d = -1;
  float u = 0.f, zt = 0.f, zd = 0.f;
  float lnSt = 0.f;
  Part T, D;
  T.m = D.m = 0.f;
  T.E = D.E = 0.f;
  T.arg = D.arg = 0;
  T.flags = D.flags = 0u;
  if (lane <= k) {
    T = load_stats_cg(st + 2 * lane);
    lnSt = log1pf(T.E);
    flags |= T.flags & SV_FLAG_NONFINITE;
  }
  if (lane < k) {
    const int i = lane;
    D = P.draft_stats_in ? load_stats_cg(P.draft_stats_in + (size_t)b * K + i) : load_stats_cg(st + 2 * i + 1);
    flags |= D.flags & SV_FLAG_NONFINITE;
    d = __ldg(P.draft_tokens + (size_t)b * K + i);
    in_range = d >= 0 && d < P.V;
    if (!in_range) flags |= SV_FLAG_TOKEN_RANGE;
    if (greedy) {
      reject = !(in_range && d == T.arg);
    } else {
      u = uniform24f(P.seed, (uint32_t)b, (uint32_t)i, 0);
      reject = true;  // p/q = 0 for an out-of-range token
      if (in_range) {
        const long long trow = ((long long)b * (K + 1) + i) * (long long)rowb;
        const long long drow = ((long long)b * K + i) * (long long)rowb;
        zt = logit_at(P.target, P.dtype, trow + d);
        zd = logit_at(P.draft, P.dtype, drow + d);
        const float lnSd = log1pf(D.E);
        const float A = (zt - T.m) * inv_f, Bq = (zd - D.m) * inv_f;
        const float dl = (A - lnSt) - (Bq - lnSd);  // ln(p/q)
        const float lu = logf(u);
        const float band = 2e-6f + 4e-7f * (fabsf(A) + fabsf(Bq) + lnSt + lnSd + fabsf(lu));
        unsure = u == 0.f || !(fabsf(dl - lu) > band);  // also NaN
        reject = !(lu < dl);
      }
    }
  }
  if (__any_sync(0xffffffffu, unsure)) {
    if (lane < k && !greedy && in_range) reject = reject_fp64(zt, zd, T, D, 1.0 / (double)tau_f, (double)u);
  }
  const unsigned rej = __ballot_sync(0xffffffffu, reject);
  const int a = rej ? (__ffs(rej) - 1) : k;

  // Row a's statistics from lane a.
  const float Ta_m = __shfl_sync(0xffffffffu, T.m, a);
  const float Ta_E = __shfl_sync(0xffffffffu, T.E, a);
  const int Ta_arg = __shfl_sync(0xffffffffu, T.arg, a);
  const float lnSt_a = __shfl_sync(0xffffffffu, lnSt, a);
  const float Da_m = __shfl_sync(0xffffffffu, D.m, a);
  const float Da_E = __shfl_sync(0xffffffffu, D.E, a);

  // The sample task first (the sampler waits for it), then the outputs.
  if (lane == 0) {
    SampleTask t;
    t.kind = greedy ? kTaskNone : (a < k ? kTaskResidual : kTaskBonus);
    t.a = a;
    t.argmax_t = (Ta_arg >= 0 && Ta_arg < P.V) ? Ta_arg : 0;
    t.c = c_f;
    t.invtau = inv_f;
    // p(v) = 2^(z(v) c + nbt): an overall scale of the weights, which the
    // draw does not depend on, so fp32 suffices
    t.nbt = -fmaf(Ta_m, c_f, lnSt_a * kLog2e);
    t.k0_hi = 0.f;
    t.k0_lo = 0.f;
    if (t.kind == kTaskResidual) {
      // q(v)/p(v) = exp((z_d(v) - z_t(v)) / tau + k0); k0 sets where the
      // residual p - q changes sign and is kept to fp64 precision:
      // k0 = (m_t - m_d) / tau + ln(S_t / S_d), S = 1 + E
      const double lnr = log1p(((double)Ta_E - (double)Da_E) / (1.0 + (double)Da_E));
      const double k0 = ((double)Ta_m - (double)Da_m) / (double)tau_f + lnr;
      t.k0_hi = (float)k0;
      t.k0_lo = (float)(k0 - (double)t.k0_hi);
    }
    t.u = greedy ? 0.0 : (double)uniform24f(P.seed, (uint32_t)b, (uint32_t)a, 1);
    P.tasks[b] = t;
    if (P.fused) {
      // hand the sequence's sample items to the producers (all sp of them,
      // also for greedy rows, so that every slot gets an item); the fence
      // orders the task before the entries
      __threadfence();
      const uint32_t base = atomicAdd(P.dq_tail, (uint32_t)P.sp);
      for (int q = 0; q < P.sp; ++q) st_relaxed_gpu(P.dq + base + q, b * P.sp + q + 1);
    }
    P.out_accept_len[b] = a;
  }

  // Emitted tokens: accepted drafts, the position-a token (written here for
  // greedy rows, by the sampler otherwise), then -1.
  if (lane <= K) {
    int32_t v = -1;
    if (lane < a) v = d;
    else if (lane == a && greedy) v = (Ta_arg >= 0 && Ta_arg < P.V) ? Ta_arg : 0;
    P.out_tokens[(size_t)b * (K + 1) + lane] = v;
  }

  // AV feature x = -ln E = logit(q_max) of the draft row and the confidence
  // sigmoid(omega x + beta_i) ("Adaptive Verification without a confidence
  // head"), fp32; theta through L2 (the fused refit rewrites it).
  // (theta may be null when only features are asked for; the fused refit
  // and out_conf require it)
  float x = 0.f, conf = 0.f;
  if (lane < k && (P.out_feature || P.out_conf || P.fit)) {
    x = D.E > 0.f ? -logf(D.E) : 30.f;
    x = x > 30.f ? 30.f : (x < -30.f ? -30.f : x);
    if (P.theta) conf = 1.0f / (1.0f + expf(-fmaf(__ldcg(P.theta), x, __ldcg(P.theta + 1 + lane))));
  }
  if (lane < K) {
    const float nan = __int_as_float(0x7fc00000);
    if (P.out_feature) P.out_feature[(size_t)b * K + lane] = lane < k ? x : nan;
    if (P.out_conf) P.out_conf[(size_t)b * K + lane] = lane < k ? conf : nan;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(P.status, flags);

  if (P.fit) {
    // Fused refit: this sequence's labelled drafts (up to and including the
    // first rejection) add their log-loss gradient and Hessian terms
    // ("Fitting the coefficients").
    const int nlab = min(a + 1, k);
    if (lane < nlab) {
      const float y = lane < a ? 1.0f : 0.0f;
      const float r = conf - y, w = conf * (1.0f - conf);
      const float q[kFitQ] = {r * x, w * x * x, r, w * x, w, 1.0f};
#pragma unroll
      for (int j = 0; j < kFitQ; ++j)
        atomicAdd(P.fitacc + lane * kFitQ + j, (unsigned long long)fixed_2p32(q[j]));
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence();
      last = atomicAdd(P.scans_done, 1u) == (uint32_t)P.B - 1u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      // every scan has read theta: the round update may now change it
      __threadfence();
      double t[kFitQ] = {0, 0, 0, 0, 0, 0};
      if (lane < K) {
#pragma unroll
        for (int j = 0; j < kFitQ; ++j)
          t[j] = (double)(long long)__ldcg(P.fitacc + lane * kFitQ + j) * (1.0 / kFitFixedScale);
      }
      av_round_update(P.av_state, P.theta_rw, K, P.round_len, P.damping_c, t, lane);
    }
  }
}

// ---------------------------------------------------------------------------
// Early exit: the acceptance walk one position at a time, as the rows of that
// position finish (fused verify modes).
// ---------------------------------------------------------------------------

// A sequence finished one of its theta-reading events (a draft row's score,
// or the final decision).  The event that completes the last sequence of the
// launch runs the refit round update (warp-wide).
__device__ void seq_event(const RowPassParams &P, int b, int k, int lane) {
  const int need = (P.mode == kVerifyFull ? k : 0) + 1;
  int last = 0;
  if (lane == 0) {
    __threadfence();
    const bool done = atomicAdd(P.seq_cnt + b, 1u) == (uint32_t)need - 1u;
    if (done && P.fit) last = atomicAdd(P.scans_done, 1u) == (uint32_t)P.B - 1u;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) {
    __threadfence();
    double t[kFitQ] = {0, 0, 0, 0, 0, 0};
    if (lane < P.K) {
#pragma unroll
      for (int j = 0; j < kFitQ; ++j)
        t[j] = (double)(long long)__ldcg(P.fitacc + lane * kFitQ + j) * (1.0 / kFitFixedScale);
    }
    av_round_update(P.av_state, P.theta_rw, P.K, P.round_len, P.damping_c, t, lane);
  }
}

// Target rows the walk queued when its accepted positions were 0..a-1 (see
// rows_on_accept): rows 1..min(a + D, k) with a look-ahead of D rows.
__device__ __forceinline__ int rows_queued(const RowPassParams &P, int a, int k) {
  if (a == 0) return 0;
  return min(a + P.spec, k);
}

// The walk ended at position a (a < k: first rejection; a == k: all
// accepted, bonus): tokens after a, the sampling task and its queue entries
// (plus fillers for the target rows never queued), the remaining outputs.
__device__ void lazy_finalize(const RowPassParams &P, int b, int a, int k, int lane) {
  const int K = P.K;
  const float tau_f = __ldg(P.temperature + b);
  const bool greedy = !(tau_f > 0.f);
  const sv_row_stats_t *st = P.stats + (size_t)b * (2 * K + 1);
  uint32_t flags = 0;
  if (lane == 0) {
    if (!(tau_f >= 0.f)) flags |= SV_FLAG_BAD_TEMP;
    if (P.draft_len) {
      const int kr = __ldg(P.draft_len + b);
      if (kr < 0 || kr > K) flags |= SV_FLAG_BAD_LEN;
    }
  }
  if (lane < k) {  // every verified draft token is range-checked, as in the full scan
    const int d = __ldg(P.draft_tokens + (size_t)b * K + lane);
    if (d < 0 || d >= P.V) flags |= SV_FLAG_TOKEN_RANGE;
  }
  // outputs of the positions the walk did not use
  if (lane < K) {
    const float nan = __int_as_float(0x7fc00000);
    if (lane >= k) {
      if (P.out_feature) P.out_feature[(size_t)b * K + lane] = nan;
      if (P.out_conf) P.out_conf[(size_t)b * K + lane] = nan;
    } else if (P.mode == kVerifyTargets && (P.out_feature || P.out_conf)) {
      const Part D = load_stats_cg(P.draft_stats_in + (size_t)b * K + lane);
      const float x = av_feature(D.E);
      if (P.out_feature) P.out_feature[(size_t)b * K + lane] = x;
      if (P.out_conf) P.out_conf[(size_t)b * K + lane] = av_conf(P, lane, x);
    }
  }
  if (lane <= K && lane > a) P.out_tokens[(size_t)b * (K + 1) + lane] = -1;
  if (lane == 0) {
    const Part T = load_stats_cg(st + 2 * a);
    if (a == k && (T.flags & SV_FLAG_NONFINITE)) flags |= SV_FLAG_NONFINITE;  // the bonus row
    Part D;
    D.m = 0.f;
    D.E = 0.f;
    if (a < k) D = P.draft_stats_in ? load_stats_cg(P.draft_stats_in + (size_t)b * K + a) : load_stats_cg(st + 2 * a + 1);
    const int argmax_t = (T.arg >= 0 && T.arg < P.V) ? T.arg : 0;
    if (greedy) P.out_tokens[(size_t)b * (K + 1) + a] = argmax_t;
    SampleTask t;
    t.kind = greedy ? kTaskNone : (a < k ? kTaskResidual : kTaskBonus);
    t.a = a;
    t.argmax_t = argmax_t;
    const float inv_f = greedy ? 1.f : 1.f / tau_f;
    const float c_f = greedy ? kLog2e : kLog2e / tau_f;
    t.c = c_f;
    t.invtau = inv_f;
    t.nbt = -fmaf(T.m, c_f, log1pf(T.E) * kLog2e);
    t.k0_hi = 0.f;
    t.k0_lo = 0.f;
    if (t.kind == kTaskResidual) {
      const double lnr = log1p(((double)T.E - (double)D.E) / (1.0 + (double)D.E));
      const double k0 = ((double)T.m - (double)D.m) / (double)tau_f + lnr;
      t.k0_hi = (float)k0;
      t.k0_lo = (float)(k0 - (double)t.k0_hi);
    }
    t.u = greedy ? 0.0 : (double)uniform24f(P.seed, (uint32_t)b, (uint32_t)a, 1);
    P.tasks[b] = t;
    // the sample items (the task is visible first), then fillers in the
    // target-row queue for the rows that were never queued (every queued
    // target row, including one queued ahead and not needed, counts against
    // the sequence's K)
    __threadfence();
    const int nfill = (K - rows_queued(P, a, k)) * P.nch_dyn;
    const uint32_t base = atomicAdd(P.dq_tail, (uint32_t)P.sp);
    const uint32_t fbase = nfill > 0 ? atomicAdd(P.tq_tail, (uint32_t)nfill) : 0u;
    for (int q = 0; q < P.sp; ++q) st_relaxed_gpu(P.dq + base + q, b * P.sp + q + 1);
    for (int q = 0; q < nfill; ++q) st_relaxed_gpu(P.tq + fbase + q, kQueueNop);
    P.out_accept_len[b] = a;
  }
  if (P.fit) {
    // the labelled drafts (up to and including the first rejection) add
    // their refit terms ("Fitting the coefficients"), one lane per position
    const int nlab = min(a + 1, k);
    if (lane < nlab) {
      const Part D = P.draft_stats_in ? load_stats_cg(P.draft_stats_in + (size_t)b * K + lane)
                                      : load_stats_cg(st + 2 * lane + 1);
      const float x = av_feature(D.E);
      fit_label(P, lane, x, av_conf(P, lane, x), lane < a);
    }
    __syncwarp();  // the labels before seq_event's fence
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(P.status, flags);
  seq_event(P, b, k, lane);
}

// Events of position i: reached (i >= 1: position i - 1 accepted), its target
// row done, its draft row done (i < k), each one atomicAdd on the position's
// counter.  The event that completes them decides the position (or, at
// i == k, finalizes with the bonus row), after a fence.
__device__ __forceinline__ uint32_t pos_need(int i, int k) {
  return (i >= 1 ? 1u : 0u) + 1u + (i < k ? 1u : 0u);
}
// Target rows queued when position i is accepted, [*j0, *j1] (empty when
// j1 < j0).  Each row is queued exactly once, by a fixed rule with a
// look-ahead of D = P.spec rows: the acceptance of position 0 queues rows
// 1 .. 1 + D and that of position i >= 1 row i + 1 + D (rows up to i + D
// came with earlier positions); rows past k are never queued.
__device__ __forceinline__ void rows_on_accept(const RowPassParams &P, int i, int k, int *j0, int *j1) {
  const int last = i + 1 + P.spec;
  *j0 = i == 0 ? 1 : last;
  *j1 = min(last, k);
}
// lane 0: publish target rows j0..j1 of sequence b in the target-row queue
// slots from base
__device__ __forceinline__ void publish_targets(const RowPassParams &P, int b, int j0, int j1, uint32_t base) {
  int q = 0;
  for (int j = j0; j <= j1; ++j) {
    const int code0 = (b * P.K + (j - 1)) * P.nch_dyn + 1;
    for (int c = 0; c < P.nch_dyn; ++c) st_relaxed_gpu(P.tq + base + q++, code0 + c);
  }
}

// Inputs of the decision at position i that no other row's completion
// changes: the drafted token d and the two logits at it (loaded while the
// position's event counter is updated, so that the latencies overlap).
struct PosInputs {
  int d;
  float zt, zd;
};
__device__ __forceinline__ PosInputs pos_logits(const RowPassParams &P, int b, int i, int d) {
  PosInputs in;
  in.d = d;
  in.zt = in.zd = 0.f;
  if (in.d >= 0 && in.d < P.V) {
    const long long rowb = (long long)P.V;
    in.zt = logit_at(P.target, P.dtype, ((long long)b * (P.K + 1) + i) * rowb + in.d);
    in.zd = logit_at(P.draft, P.dtype, ((long long)b * P.K + i) * rowb + in.d);
  }
  return in;
}

// fp32 acceptance test of position i with the exact fp64 fallback (one lane).
__device__ __forceinline__ bool reject_in(const RowPassParams &P, int b, int i, const Part &T, const Part &D,
                                          float tau_f, bool greedy, const PosInputs &in) {
  const bool in_range = in.d >= 0 && in.d < P.V;
  if (greedy) return !(in_range && in.d == T.arg);
  if (!in_range) return true;
  const float u = uniform24f(P.seed, (uint32_t)b, (uint32_t)i, 0);
  return reject_values(u, in.zt, in.zd, T, D, tau_f);
}

// The walk from position i (all of whose events are in; `known` holds the
// statistics of the row whose completion got here: sidx_known = 2 i (target)
// or 2 i + 1 (draft), -1 when both rows must be loaded; `in` the position's
// inputs).  An accepted position queues the rows of rows_on_accept, then
// reaches i + 1, continuing while that position's rows are done.
__device__ void lazy_walk(const RowPassParams &P, int b, int i, int k, int lane, const Part known, int sidx_known,
                          PosInputs in) {
  const int K = P.K;
  const float tau_f = __ldg(P.temperature + b);
  const bool greedy = !(tau_f > 0.f);
  for (;;) {
    int rej = 0, cont = 0;
    if (lane == 0) {
      const sv_row_stats_t *st = P.stats + (size_t)b * (2 * K + 1);
      const Part T = sidx_known == 2 * i ? known : load_stats_cg(st + 2 * i);
      const Part D = sidx_known == 2 * i + 1 ? known
                     : (P.draft_stats_in ? load_stats_cg(P.draft_stats_in + (size_t)b * K + i)
                                         : load_stats_cg(st + 2 * i + 1));
      const bool reject = reject_in(P, b, i, T, D, tau_f, greedy, in);
      if (T.flags & SV_FLAG_NONFINITE) atomicOr(P.status, SV_FLAG_NONFINITE);
      rej = reject;
      if (!reject) {
        // Issued in this order so that the round trips overlap: the next
        // drafted token, the queue reservation for the next target rows, the
        // "reached" event of position i + 1; then the queue entries (their
        // slots are reserved, so a walk that races ahead cannot take them)
        // and the logits at the next token.
        P.out_tokens[(size_t)b * (K + 1) + i] = in.d;
        const int dn = i + 1 < K ? __ldg(P.draft_tokens + (size_t)b * K + i + 1) : 0;
        int j0, j1;
        rows_on_accept(P, i, k, &j0, &j1);
        uint32_t base = 0;
        if (j1 >= j0) base = atomicAdd(P.tq_tail, (uint32_t)((j1 - j0 + 1) * P.nch_dyn));
        const uint32_t old = atomicAdd(P.pos_cnt + (size_t)b * (K + 1) + i + 1, 1u);
        if (j1 >= j0) publish_targets(P, b, j0, j1, base);
        if (i + 1 < k) in = pos_logits(P, b, i + 1, dn);
        cont = old == pos_need(i + 1, k) - 1u;
        if (cont) __threadfence();
      }
    }
    rej = __shfl_sync(0xffffffffu, rej, 0);
    cont = __shfl_sync(0xffffffffu, cont, 0);
    if (rej) {
      lazy_finalize(P, b, i, k, lane);
      return;
    }
    if (!cont) return;
    ++i;
    sidx_known = -1;
    if (i == k) {  // every draft accepted and the bonus row is done
      lazy_finalize(P, b, k, k, lane);
      return;
    }
  }
}

// A row of sequence b finished (sidx = 2 i: target row i, 2 i + 1: draft row
// i); R (lane 0) holds its statistics, already stored.
__device__ __noinline__ void lazy_row_done(const RowPassParams &P, int b, int sidx, const Part R, int lane) {
  const int k = kept_len_of(P, b);
  const int i = sidx >> 1;
  int ready = 0;
  PosInputs in;
  in.d = 0;
  in.zt = in.zd = 0.f;
  if (lane == 0) {
    // the drafted token and this row's event first, so that their round
    // trips overlap each other and the work below
    const int d = i < P.K ? __ldg(P.draft_tokens + (size_t)b * P.K + i) : 0;
    const uint32_t old = atomicAdd(P.pos_cnt + (size_t)b * (P.K + 1) + i, 1u);
    // a draft row is always used (its AV score); a target row's flags are
    // raised when its position is decided (it may have been read ahead)
    if ((sidx & 1) && (R.flags & SV_FLAG_NONFINITE)) atomicOr(P.status, SV_FLAG_NONFINITE);
    if (i < P.K) in = pos_logits(P, b, i, d);
    if ((sidx & 1) && (P.out_feature || P.out_conf)) {  // a draft row's score
      const float x = av_feature(R.E);
      if (P.out_feature) P.out_feature[(size_t)b * P.K + i] = x;
      if (P.out_conf) P.out_conf[(size_t)b * P.K + i] = av_conf(P, i, x);
    }
    ready = old == pos_need(i, k) - 1u;
    if (ready) __threadfence();
  }
  ready = __shfl_sync(0xffffffffu, ready, 0);
  if (ready) {
    if (i == k) lazy_finalize(P, b, k, k, lane);  // every draft accepted: bonus from row k
    else lazy_walk(P, b, i, k, lane, R, sidx, in);
  }
  if (sidx & 1) seq_event(P, b, k, lane);
}

__device__ void finish_score(const RowPassParams &P, int b, int lane) {
  const int K = P.K;
  const sv_row_stats_t *st = P.stats + (size_t)b * (2 * K + 1);
  uint32_t flags = 0;
  double conf = 1.0;
  if (lane < K) {
    const Part D = load_stats_cg(st + 2 * lane + 1);
    flags |= D.flags & SV_FLAG_NONFINITE;
    const double E = (double)D.E;
    double x = E > 0.0 ? -log(E) : 30.0;
    x = x > 30.0 ? 30.0 : (x < -30.0 ? -30.0 : x);
    const double z = (double)__ldg(P.theta) * x + (double)__ldg(P.theta + 1 + lane);
    conf = 1.0 / (1.0 + exp(-z));
    P.out_feature[(size_t)b * K + lane] = (float)x;
    P.out_conf[(size_t)b * K + lane] = (float)conf;
    if (P.out_draft_stats) store_stats(P.out_draft_stats + (size_t)b * K + lane, D);
  }
  // survival = cumulative product of the confidences, in position order
  int kept = K;
  if (P.keep_threshold > 0.f) {
    double surv = 1.0;
    kept = 0;
    bool stop = false;
    for (int i = 0; i < K; ++i) {
      const double ci = __shfl_sync(0xffffffffu, conf, i);
      if (!stop) {
        surv *= ci;
        if (surv >= (double)P.keep_threshold) kept = i + 1;
        else stop = true;
      }
    }
  }
  if (lane == 0 && P.out_kept_len) P.out_kept_len[b] = kept;
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// Producer helpers: queue claims.
// ---------------------------------------------------------------------------
// The entry of a claimed slot (its publisher writes it right after the
// reservation): wait (bounded) until it is nonzero.
__device__ __forceinline__ bool wait_entry(const RowPassParams &P, const int *slot, volatile int *abort_flag,
                                           int *out) {
  int code = ld_acquire_gpu(slot);
  if (code == 0) {
    const uint64_t t0 = global_ns();
    while ((code = ld_acquire_gpu(slot)) == 0) {
      if (*abort_flag) break;
      if (global_ns() - t0 > P.timeout_ns) {
        *abort_flag = 1;
        atomicOr(P.status, SV_FLAG_TIMEOUT);
        break;
      }
      __nanosleep(200);
    }
  }
  *out = code;
  return code != 0;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int kDtype>
__global__ void __launch_bounds__(kRowThreads, 1) rowpass_kernel(const RowPassParams P) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem &S = *reinterpret_cast<Smem *>(smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    for (int s = 0; s < kPartSlots; ++s) {
      mbar_init(&S.pfull[s], kConsumerWarps);
      mbar_init(&S.pempty[s], 1);
    }
    S.abort_flag = 0;
    S.epi_next = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int *abort_flag = &S.abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    // (failure-detection tests: staging nothing leaves every consumer wait to
    // run out; no copy is ever in flight)
    if (lane != 0 || P.withhold) return;
    int s = 0;
    uint32_t phase = 0;
    uint32_t nfull[kStages];
#pragma unroll
    for (int i = 0; i < kStages; ++i) nfull[i] = 0;
    int cached_b = -1, cached_k = 0;
    float cached_c = 1.f;
    bool ok = true;
    const int K = P.K;
    // Order of the claims.  Early exit: a target row some walk queued (its
    // chain of decisions waits on it), else a static item (every first
    // target row, then every draft row, position-major), else a sample item
    // of a draw.  Each queue is claimed one slot at a time with atomicAdd
    // (a unique slot, no contention on retries); a claimed slot stays
    // pending until its entry is published and the producer looks at it
    // between items, so it never waits for work that only other producers'
    // rows could publish, and every published entry is staged by the
    // producer holding its slot.  Without early exit: the static items, then
    // the sample items in order (each is published by the scan of rows
    // already staged).
    bool static_left = true, dyn_left = P.fused != 0;
    uint64_t idle_t0 = 0;
    int tq_pend = -1, dq_pend = -1;
    bool tq_left = P.lazy != 0, dq_left = P.lazy != 0;
    // a share of the CTAs serve the draws' sample items before static items
    const bool draws_first = P.draw_every > 0 && (int)blockIdx.x % P.draw_every == 0;
    uint32_t backoff = 0;
    for (;;) {
      int row_b = 0, row_chunk = 0, row_target = 0, row_pos = 0;
      int item = -1;
      int code = 0;  // a sample item's 1-based code
      if (P.lazy) {
        if (tq_pend < 0 && tq_left) {
          const int n = (int)atomicAdd(P.tq_head, 1u);
          if (n < P.ntq) tq_pend = n;
          else tq_left = false;
        }
        int tcode = tq_pend >= 0 ? ld_acquire_gpu(P.tq + tq_pend) : 0;
        if (tcode != 0) {
          item = P.nstatic + tq_pend;
          tq_pend = -1;
          idle_t0 = 0;
          backoff = 0;
          if (tcode == kQueueNop) continue;
          // a queued target row: (b K + i - 1) nch + chunk
          const int r = tcode - 1;
          row_chunk = r % P.nch_dyn;
          const int q = r / P.nch_dyn;
          row_b = q / K;
          row_pos = q - row_b * K + 1;
          row_target = 1;
        } else {
          // then a static item and a published sample item of a draw, in
          // this CTA's order (draws_first: a sample item first)
          bool have = false;
          for (int pass = 0; pass < 2 && !have; ++pass) {
            if ((pass == 0) == draws_first) {
              if (dq_pend < 0 && dq_left) {
                const int n = (int)atomicAdd(P.dq_head, 1u);
                if (n < P.ndyn) dq_pend = n;
                else dq_left = false;
              }
              code = dq_pend >= 0 ? ld_acquire_gpu(P.dq + dq_pend) : 0;
              if (code != 0) {
                dq_pend = -1;
                have = true;
              }
            } else if (static_left) {
              item = (int)atomicAdd(P.ticket, 1u);
              if (item < P.nstatic) {
                // static items, position-major: group 0 = every first target
                // row, group g >= 1 = every draft row g - 1 (measured: pairing
                // each sequence's target and draft row 0 in one group is slower)
                const int per_group = P.B * P.nch;
                const int g = item / per_group;
                const int rem = item - g * per_group;
                row_b = rem / P.nch;
                row_chunk = rem - row_b * P.nch;
                row_target = g == 0;
                row_pos = g == 0 ? 0 : g - 1;
                have = true;
              } else {
                static_left = false;
              }
            }
          }
          if (have) {
            idle_t0 = 0;
            backoff = 0;
          } else {
            if (!static_left && !tq_left && !dq_left && tq_pend < 0 && dq_pend < 0) break;  // all claimed and staged
            // the pending slots are not published yet: look again shortly
            if (*abort_flag) {
              ok = false;
              break;
            }
            const uint64_t now = global_ns();
            if (idle_t0 == 0) {
              idle_t0 = now;
            } else if (now - idle_t0 > P.timeout_ns) {
              *abort_flag = 1;
              atomicOr(P.status, SV_FLAG_TIMEOUT);
              ok = false;
              break;
            }
            backoff = backoff ? min(2 * backoff, 1024u) : 64u;
            __nanosleep(backoff);
            continue;
          }
        }
      } else if (static_left) {
        item = (int)atomicAdd(P.ticket, 1u);
        if (item >= P.nstatic) {
          static_left = false;
          continue;
        }
        const int per_seq = P.nslot * P.nch;
        row_b = item / per_seq;
        const int rem = item - row_b * per_seq;
        const int slot = rem / P.nch;
        row_chunk = rem - slot * P.nch;
        slot_kind(P.mode, K, slot, row_target, row_pos);
      } else if (dyn_left) {
        const int c = (int)atomicAdd(P.dq_head, 1u);
        if (c >= P.ndyn) {
          dyn_left = false;
          continue;
        }
        if (!wait_entry(P, P.dq + c, abort_flag, &code)) {
          ok = false;
          break;
        }
      } else {
        break;
      }
      if (code) {
        // ---- a sample item (b, part) of a draw
        --code;
        {
        const int b = code / P.sp, part = code - (code / P.sp) * P.sp;
        const SampleTask t = load_task_cg(P.tasks + b);
        if (t.kind == kTaskNone) continue;
        const bool resid = t.kind == kTaskResidual;
        const long long t_off = ((long long)b * (K + 1) + t.a) * (long long)P.V;
        const long long d_off = ((long long)b * K + t.a) * (long long)P.V;
        const int j0 = part * P.spc, j1 = min(P.smp.nsub, j0 + P.spc);
        const int e_beg = min(P.V, j0 * kSubChunk), e_end = min(P.V, j1 * kSubChunk);
        const int half_elems = kSampleHalfBytes / kEsz;
        const int nst = e_end > e_beg ? (e_end - e_beg + half_elems - 1) / half_elems : 1;
        for (int st = 0; st < nst; ++st) {
          if (!mbar_wait_bounded(&S.empty[s], phase ^ 1u, abort_flag, P.status, P.timeout_ns)) {
            ok = false;
            break;
          }
          const int e = e_beg + st * half_elems;
          const int n = max(0, min(half_elems, e_end - e));
          const int bytes = n * kEsz;  // a multiple of 16: rows are 16-byte aligned on this path
          StageHot &h = S.hot[s];
          h.e0 = e;
          h.nvec = bytes / 16;
          h.flags = kFlagSample | (resid ? kFlagResidual : 0) | (st == 0 ? kFlagFirst : 0) |
                    (st == nst - 1 ? kFlagLast : 0);
          h.c = t.c;
          StageSample &hs = S.smpl[s];
          hs.nbt = t.nbt;
          hs.invtau = t.invtau;
          hs.k0_hi = t.k0_hi;
          hs.k0_lo = t.k0_lo;
          hs.b = b;
          ++nfull[s];
          if (bytes > 0) {
            mbar_arrive_expect_tx(&S.full[s], (uint32_t)(resid ? 2 * bytes : bytes));
            bulk_g2s(S.ring[s], reinterpret_cast<const char *>(P.target) + (t_off + e) * kEsz, (uint32_t)bytes,
                     &S.full[s]);
            if (resid)
              bulk_g2s(S.ring[s] + kSampleHalfBytes, reinterpret_cast<const char *>(P.draft) + (d_off + e) * kEsz,
                       (uint32_t)bytes, &S.full[s]);
          } else {
            mbar_arrive(&S.full[s]);
          }
          if (++s == kStages) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        continue;
        }
      }
      const int b = row_b, chunk = row_chunk, is_target = row_target, pos = row_pos;
      if (b != cached_b) {
        cached_b = b;
        cached_k = kept_len_of(P, b);
        cached_c = row_scale(P, b);
      }
      if (P.mode != kScore) {
        if (is_target ? (pos > cached_k) : (pos >= cached_k)) continue;
      }
      const long long row = is_target ? ((long long)b * (K + 1) + pos) : ((long long)b * K + pos);
      const long long row_off = row * (long long)P.V;
      const char *base = reinterpret_cast<const char *>(is_target ? P.target : P.draft);
      // queued target rows (early exit) have their own, finer chunks
      const int celems = (P.lazy && is_target && pos > 0) ? P.chunk_elems_dyn : P.chunk_elems;
      const int e_beg = chunk * celems;
      const int e_end = min(P.V, e_beg + celems);
      const uintptr_t a_beg = reinterpret_cast<uintptr_t>(base) + (uintptr_t)(row_off + e_beg) * kEsz;
      const uintptr_t a_end = reinterpret_cast<uintptr_t>(base) + (uintptr_t)(row_off + e_end) * kEsz;
      int a0 = e_beg + (int)(((16 - (a_beg & 15)) & 15) / kEsz);
      int a1 = e_end - (int)((a_end & 15) / kEsz);
      int x0, xn0, x1, xn1;
      if (a1 <= a0) {  // no whole aligned vector: every element by plain loads
        a0 = a1 = e_beg;
        x0 = e_beg;
        xn0 = e_end - e_beg;
        x1 = e_end;
        xn1 = 0;
      } else {
        x0 = e_beg;
        xn0 = a0 - e_beg;
        x1 = a1;
        xn1 = e_end - a1;
      }
      const long long mid_bytes = (long long)(a1 - a0) * kEsz;
      const int nst = mid_bytes > 0 ? (int)((mid_bytes + kStageBytes - 1) / kStageBytes) : 1;
      const int sidx = is_target ? 2 * pos : 2 * pos + 1;
      for (int st = 0; st < nst; ++st) {
        if (!mbar_wait_bounded(&S.empty[s], phase ^ 1u, abort_flag, P.status, P.timeout_ns)) {
          ok = false;
          break;
        }
        const long long off_b = (long long)st * kStageBytes;
        const int bytes = mid_bytes > 0 ? (int)min((long long)kStageBytes, mid_bytes - off_b) : 0;
        StageHot &h = S.hot[s];
        h.e0 = a0 + (int)(off_b / kEsz);
        h.nvec = bytes / 16;
        h.flags = (st == 0 ? kFlagFirst : 0) | (st == nst - 1 ? kFlagLast : 0);
        h.c = cached_c;
        if (st == nst - 1) {
          StageCold &cd = S.cold[s];
          cd.item = item;
          cd.b = b;
          cd.sidx = sidx;
          cd.chunk = chunk;
          cd.x0 = x0;
          cd.xn0 = xn0;
          cd.x1 = x1;
          cd.xn1 = xn1;
          cd.row_off = row_off;
          cd.is_target = is_target;
        }
        ++nfull[s];
        if (bytes > 0) {
          mbar_arrive_expect_tx(&S.full[s], (uint32_t)bytes);
          // the rows' statistics read each row once: the copies stream through
          // L2 marked evict-first, which leaves L2 to the draws (whose rows
          // are read in parts, and whose crossing sub-chunk is read again by
          // the final search); C3 138.2 -> 131.5 us a launch
          bulk_g2s_hint(S.ring[s], base + (row_off + a0) * kEsz + off_b, (uint32_t)bytes, &S.full[s],
                        policy_evict_first());
        } else {
          mbar_arrive(&S.full[s]);
        }
        if (++s == kStages) {
          s = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    if (ok && mbar_wait_bounded(&S.empty[s], phase ^ 1u, abort_flag, P.status, P.timeout_ns)) {
      S.hot[s].flags = kFlagDone;
      ++nfull[s];
      mbar_arrive(&S.full[s]);
    } else {
      // Gave up: wait (bounded) for this CTA's copies still in flight.
      const uint64_t t0 = global_ns();
      for (int i = 0; i < kStages; ++i) {
        if (nfull[i] == 0) continue;
        while (!mbar_try_wait(&S.full[i], (nfull[i] - 1u) & 1u)) {
          if (global_ns() - t0 > P.timeout_ns) break;
        }
      }
    }
    return;
  }

  if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------------------ epilogue
    const int K = P.K;
    // Each epilogue warp takes the next item n (slot n % kPartSlots) from a
    // shared counter, so a warp busy with a sequence's scan or draw does not
    // hold up the items behind it.  Items are produced in order and a slot
    // is refilled only after its item was read, so the parity of n / kPartSlots
    // names the right phase of the slot's barrier.  Every warp leaves on the
    // first end-of-work marker it takes; there is one marker per warp.
    for (;;) {
      int it = 0;
      if (lane == 0) it = atomicAdd(&S.epi_next, 1);
      it = __shfl_sync(0xffffffffu, it, 0);
      const int slot = it % kPartSlots;
      if (!mbar_wait_bounded(&S.pfull[slot], (uint32_t)((it / kPartSlots) & 1), abort_flag, P.status, P.timeout_ns)) break;
      const PartInfo info = S.pinfo[slot];
      if (info.item == kItemSample) {
        // a sample item of sequence info.b finished: the last of its sp items
        // locates the token
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pempty[slot]);
        int last = 0;
        if (lane == 0) {
          __threadfence();
          last = atomicAdd(P.smp.smp_cnt + info.b, 1u) == (uint32_t)P.sp - 1u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const SampleTask t = load_task_cg(P.tasks + info.b);
          const RowPtrs R = row_ptrs(P.smp, t, info.b, P.esz);
          if (P.dtype == SV_BF16) finalize_warp<SV_BF16>(P.smp, t, info.b, R, lane);
          else finalize_warp<SV_FP32>(P.smp, t, info.b, R, lane);
        }
        continue;
      }
      if (info.item < 0) break;
      Part mine = {-INFINITY, 0.f, INT_MAX, 0u};
      if (lane < kConsumerWarps) mine = S.part[slot][lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pempty[slot]);
      int seq_done = 0;
      // the math warps' partials, combined across this warp's lanes
      Part R = combine_warp(mine, info.c);
      if (lane == 0) {
        const size_t row = (size_t)info.b * (2 * K + 1) + info.sidx;
        bool row_done = true;
        const int nch_row = (P.lazy && !(info.sidx & 1) && info.sidx > 0) ? P.nch_dyn : P.nch;
        if (nch_row > 1) {
          store_stats(P.chunk_part + row * kMaxChunks + info.chunk, R);
          __threadfence();
          const uint32_t old = atomicAdd(P.row_cnt + row, 1u);
          row_done = (old == (uint32_t)nch_row - 1u);
          if (row_done) {
            __threadfence();
            R = load_stats_cg(P.chunk_part + row * kMaxChunks + 0);
            for (int c = 1; c < nch_row; ++c) R = combine(R, load_stats_cg(P.chunk_part + row * kMaxChunks + c), info.c);
          }
        }
        if (row_done) {
          if (R.arg == INT_MAX || !(fabsf(R.m) <= FLT_MAX) || isnan(R.E)) R.flags |= SV_FLAG_NONFINITE;
          store_stats(P.stats + row, R);
          __threadfence();
          if (P.lazy) {
            seq_done = 2;  // hand the finished row to the walk below
          } else {
            const int k = kept_len_of(P, info.b);
            const uint32_t old = atomicAdd(P.seq_cnt + info.b, 1u);
            seq_done = (old == (uint32_t)rows_needed(P, k) - 1u);
            if (seq_done) __threadfence();
          }
        }
      }
      seq_done = __shfl_sync(0xffffffffu, seq_done, 0);
      if (seq_done == 2) {
        lazy_row_done(P, info.b, info.sidx, R, lane);
      } else if (seq_done) {
        __threadfence();
        if (P.mode == kScore) finish_score(P, info.b, lane);
        else finish_verify(P, info.b, lane);
      }
    }
    return;
  }

  // -------------------------------------------------------------------- math warps
  WarpState st;
  state_reset(st);
  int s = 0;
  uint32_t phase = 0;
  int it = 0;
  float c = 1.f;
  int rot = 0;  // sample stages: which warps take the extra sub-chunk alternates
  for (;;) {
    if (!mbar_wait_bounded(&S.full[s], phase, abort_flag, P.status, P.timeout_ns)) break;
    const StageHot h = S.hot[s];
    if (h.flags & kFlagDone) {
      // propagate the end of work to the epilogue warp
      // one end-of-work marker for each epilogue warp (consecutive items)
      for (int e = 0; e < kEpiWarps; ++e, ++it) {
        const int slot = it % kPartSlots;
        if (!mbar_wait_bounded(&S.pempty[slot], (uint32_t)(((it / kPartSlots) & 1) ^ 1), abort_flag, P.status,
                               P.timeout_ns))
          break;
        if (warp == 0 && lane == 0) S.pinfo[slot].item = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pfull[slot]);
      }
      break;
    }
    if (h.flags & kFlagSample) {
      // Residual / bonus weights of the staged elements, summed per 256-element
      // sub-chunk (one sub-chunk per warp pass, 8 elements per lane).
      const StageSample hs = S.smpl[s];
      SampleTask t;
      t.kind = (h.flags & kFlagResidual) ? kTaskResidual : kTaskBonus;
      t.c = h.c;
      t.nbt = hs.nbt;
      t.invtau = hs.invtau;
      t.k0_hi = hs.k0_hi;
      t.k0_lo = hs.k0_lo;
      const int n = h.nvec * 16 / kEsz;
      const int nsc = (n + kSubChunk - 1) / kSubChunk;
      float *sub = P.smp.subsum + (size_t)hs.b * P.smp.nsub + h.e0 / kSubChunk;
      // 54 sub-chunks per full stage over 12 warps: half of the warps take a
      // fifth one, alternately, so that no warp falls behind over a draw
      for (int q = (warp + rot) % kConsumerWarps; q < nsc; q += kConsumerWarps) {
        const int off = q * kSubChunk + lane * 8;  // element offset inside the stage
        const Raw8 zt = smem_raw8<kDtype>(S.ring[s], off);
        Raw8 zd;
        zd.a = zd.b = make_uint4(0, 0, 0, 0);
        if (t.kind == kTaskResidual) zd = smem_raw8<kDtype>(S.ring[s] + kSampleHalfBytes, off);
        const float sm = warp_sum(weights_sum8<kDtype>(t, t.kind, off, n, zt, zd));
        if (lane == 0) sub[q] = sm;
      }
      rot ^= kConsumerWarps / 2;
      const bool last = (h.flags & kFlagLast) != 0;
      const int bb = hs.b;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
      if (last) {
        if (lane == 0) __threadfence();  // sub-chunk sums visible before the completion count
        const int slot = it % kPartSlots;
        if (!mbar_wait_bounded(&S.pempty[slot], (uint32_t)(((it / kPartSlots) & 1) ^ 1), abort_flag, P.status,
                               P.timeout_ns))
          break;
        if (warp == 0 && lane == 0) {
          PartInfo pi;
          pi.item = kItemSample;
          pi.b = bb;
          pi.sidx = 0;
          pi.chunk = 0;
          pi.c = 0.f;
          S.pinfo[slot] = pi;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pfull[slot]);
        ++it;
      }
      if (++s == kStages) {
        s = 0;
        phase ^= 1u;
      }
      continue;
    }
    if (h.flags & kFlagFirst) {
      state_reset(st);
      c = h.c;
    }
    StageCold cd;
    if (h.flags & kFlagLast) cd = S.cold[s];
    if (h.nvec > 0) consume_stage<kDtype>(st, reinterpret_cast<uint4 *>(S.ring[s]), h.nvec, tid, lane, h.e0, c);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);

    if (h.flags & kFlagLast) {
      if (warp == 0) {
        const int nx = cd.xn0 + cd.xn1;
        if (nx > 0) {
          const int idx = lane < cd.xn0 ? cd.x0 + lane : cd.x1 + (lane - cd.xn0);
          const void *base = cd.is_target ? P.target : P.draft;
          const float v = lane < nx ? logit_at(base, kDtype, cd.row_off + idx) : -INFINITY;
          consume_scalar(st, v, idx, lane, c);
        }
      }
      // warp partial: lane sums in true units, then across the warp
      const float T = st.A * fmaf(st.nbl, kLn2, 1.0f);
      const float Ew = warp_sum(T);
      const int slot = it % kPartSlots;
      if (!mbar_wait_bounded(&S.pempty[slot], (uint32_t)(((it / kPartSlots) & 1) ^ 1), abort_flag, P.status,
                             P.timeout_ns))
        break;
      if (lane == 0) {
        Part pr;
        pr.m = st.M;
        pr.E = Ew;
        pr.arg = st.arg;
        pr.flags = st.flags;
        S.part[slot][warp] = pr;
        if (warp == 0) {
          PartInfo pi;
          pi.item = cd.item;
          pi.b = cd.b;
          pi.sidx = cd.sidx;
          pi.chunk = cd.chunk;
          pi.c = c;
          S.pinfo[slot] = pi;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull[slot]);
      ++it;
    }
    if (++s == kStages) {
      s = 0;
      phase ^= 1u;
    }
  }
}

}  // namespace

size_t rowpass_smem_bytes() { return sizeof(Smem) + 128; }

cudaError_t launch_rowpass(const RowPassParams &P, int grid, cudaStream_t stream) {
  const size_t smem = rowpass_smem_bytes();
  if (P.dtype == SV_BF16) {
    cudaFuncSetAttribute(rowpass_kernel<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    rowpass_kernel<SV_BF16><<<grid, kRowThreads, smem, stream>>>(P);
  } else {
    cudaFuncSetAttribute(rowpass_kernel<SV_FP32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    rowpass_kernel<SV_FP32><<<grid, kRowThreads, smem, stream>>>(P);
  }
  return cudaGetLastError();
}

}  // namespace sv
