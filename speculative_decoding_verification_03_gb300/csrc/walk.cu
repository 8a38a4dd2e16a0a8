// Cluster walk: the fused verification step ("Speculative Decoding: Draft,
// EAGLE, MTP", section "one speculative step": accept drafts left to right
// with probability min(1, p/q), draw the first rejected position's token
// from the normalised positive residual, a bonus token when every draft
// passed), the AV scores of the verified drafts ("Adaptive Verification
// without a confidence head", sections "Solution" and "Scoring the
// distribution") and, with a refit state, one refit step (section "Fitting
// the coefficients"), with each sequence's walk kept inside one
// thread-block cluster.
//
// Why: the walk is a chain -- target row i + 1 is needed only when position
// i is accepted -- and a row streamed by one SM arrives at that SM's share of
// the HBM bandwidth.  Here every row is cut into `cs` slices, one per CTA of
// the cluster, so a row the chain waits for arrives `cs` times sooner, and a
// cluster walks several sequences at once to keep its SMs streaming while
// their chains wait.
//
// Roles (every CTA): 12 math warps compute a slice's partial statistics
// (max, first argmax, sum of exp terms: the same arithmetic as the
// streaming row pass) from a TMA-filled shared-memory ring; a producer warp
// issues the bulk copies; an epilogue warp combines the math warps' partials
// and sends the CTA's partial to the leader (CTA 0) through distributed
// shared memory.  The leader's control warp owns the walk: it decides which
// row or draw comes next, writes that entry into every CTA's schedule ring,
// consumes the cluster's partials in schedule order, makes the decisions and
// writes the outputs.  Every CTA handles the schedule's entries in the same
// order, so rows, slots and partial buffers line up without further
// agreement.
//
// Draws: a residual or bonus draw is two entries.  "Mass": each CTA sums the
// weights of its slice per 256-element sub-chunk (rows re-read from L2) and
// sends its slice total; the leader forms u * R and finds the CTA whose
// slice holds the crossing.  "Find": that CTA locates the token inside its
// slice (double-float prefix over its sub-chunk sums, then within the
// sub-chunk) and writes it.
//
// Every wait is bounded; a time-out sets SV_FLAG_TIMEOUT, the other waits of
// the grid give up when they see it, and every thread still meets the final
// cluster barrier, so no CTA leaves while another may write to its shared
// memory.
#include <cfloat>
#include <climits>

#include "avfit_common.cuh"
#include "rowstats.cuh"
#include "sample_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kWMath = kConsumerWarps;         // math warps (the row pass's stage layout)
constexpr int kWProd = kWMath;                 // producer warp
constexpr int kWEpi = kWMath + 1;              // epilogue warp
constexpr int kWCtl = kWMath + 2;              // control warp (leader CTA)
constexpr int kWComb = kWMath + 3;             // combiner warp (leader CTA)
constexpr int kWThreads = (kWMath + 4) * 32;   // 512
constexpr int kWEnt = 16;                      // schedule ring entries
constexpr int kWParts = 4;                     // partial buffers between math and epilogue
constexpr int kWMaxSub = kStageBytes / 2 / kSubChunk;  // sub-chunks of a slice (<= 96)
constexpr int kDraftLookahead = 1;             // draft rows appended ahead of the decision frontier
constexpr int kWBatch = 4;                     // entries the leader publishes per pass

enum EntryKind : int { kEntRow = 1, kEntMass = 2, kEntFind = 3, kEntEnd = 4 };

// One schedule entry (64 bytes, written by the leader into every CTA).
struct alignas(16) Entry {
  int kind;
  int b;          // sequence
  int pos;        // row position, or the drawn position a
  int is_target;  // row entries: target row pos (else draft row pos)
  float c;        // log2(e) / tau (tau = 1 for greedy rows)
  int d;          // the drafted token whose logit the row reports, or -1
  int seq;        // the leader's sequence slot (also names the sub-chunk buffer)
  int draw_kind;  // kTaskResidual or kTaskBonus
  float nbt, invtau, k0_hi, k0_lo;  // draw weights (SampleTask)
  int rank;       // find: the CTA that searches
  float t_hi, t_lo;  // find: u R minus the mass of the lower ranks
  int argmax_t;   // find: fallback token
};
static_assert(sizeof(Entry) == 64, "Entry is copied as four 16-byte words");

// A CTA's partial for one entry (32 bytes, sent to the leader).
struct alignas(16) XPart {
  float m, E;
  int arg;
  uint32_t flags;
  float z;      // logit at the entry's token when it lies in this CTA's slice
  int has_z;
  float mass_hi, mass_lo;  // mass entries: the slice's weight total
};
static_assert(sizeof(XPart) == 32, "XPart is copied as two 16-byte words");

enum SeqPhase : int {
  kSWalk = 0,      // deciding positions
  kSNeedMass = 1,  // draw: mass entry to append
  kSMass = 2,
  kSNeedFind = 3,  // draw: find entry to append
  kSFind = 4,
  kSDrawn = 5      // token emitted; waiting for the remaining entries
};

// The walk's state of one sequence: scalars in the registers of the control
// warp's lane s (slot s), per-position values in shared memory.
struct SeqState {
  int b, k, i;       // sequence (-1: free slot), verified drafts, decision frontier
  int t_app, d_app;  // target / draft rows appended so far
  int t_ok;          // target row i's statistics are in
  int phase, a, pending, greedy, draw_kind;
  uint32_t d_have;   // draft rows whose statistics are in
  uint32_t flags;
  float tau, inv_tau, c, zt, lnSt;
  Part T;            // target row i
  float nbt, k0_hi, k0_lo;
  int argmax_t;
  int f_rank;
  float f_hi, f_lo;
};
struct SeqArr {
  int tok[SV_MAX_K];
  float zd[SV_MAX_K];
  float xs[SV_MAX_K];
  float cf[SV_MAX_K];
  float lnSd[SV_MAX_K];
  float u0[SV_MAX_K + 1];   // acceptance uniform of each position
  float lu0[SV_MAX_K + 1];  // its logarithm
  float u1[SV_MAX_K + 1];   // draw uniform of each position
  Part D[SV_MAX_K];
};

// An entry's partials merged by the combiner (leader CTA).
struct Res {
  Part st;                // rows: the row's statistics
  float z, lnS, x, conf;  // logit at the token, ln S, AV feature and confidence (draft rows)
  int zero, rs;           // mass: no mass at all; the slice holding the crossing
  float t_hi, t_lo;       // ... and u R minus the mass before it
};

struct __align__(128) WalkSmem {
  Entry ent[kWEnt];
  XPart xp[kWEnt][kWalkMaxCs];  // leader: the CTAs' partials per entry
  Part wpart[kWParts][kWMath];
  float xz[kWParts];
  float subsum[kWalkSeqs][kWMaxSub];
  SeqArr sa[kWalkSeqs];         // leader only
  float theta[SV_MAX_K + 1];    // leader only
  uint64_t sfull[kWEnt];        // entry in: this CTA's arrival (armed for 64 bytes) + the leader's st.async
  uint64_t xfull[kWEnt];        // leader: partials in (its arrival, armed for cs x 32 bytes)
  Entry lent[kWEnt];            // leader: its own copy of each entry in flight
  Res res[kWEnt];               // leader: merged partials
  unsigned long long fit[SV_MAX_K * kFitQ];  // leader: this cluster's refit sums (2^-32 fixed point)
  uint64_t full[kWalkMaxSlots];
  uint64_t empty[kWalkMaxSlots];
  uint64_t pfull[kWParts];
  uint64_t pempty[kWParts];
  int stage_x[kWBatch];   // leader: schedule slots of the entries being published
  int res_count;          // leader: entries merged by the combiner
  int abort_flag;
  int prod_e;  // entries the producer has read (an entry is acknowledged only after)
};

// Bounded wait on a local barrier phase (cluster-scope acquire when other
// CTAs release into it).  Gives up on the CTA's abort flag, on a time-out
// anywhere in the grid (the status word), or after limit_ns.
__device__ __noinline__ bool wwait(uint64_t *bar, uint32_t parity, bool cl, volatile int *abort_flag,
                                   uint32_t *status, uint64_t limit_ns) {
  if (cl ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (cl ? mbar_try_wait_cl_sleep(bar, parity, 20000u) : mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (*reinterpret_cast<volatile uint32_t *>(status) & SV_FLAG_TIMEOUT) {
      *abort_flag = 1;
      return false;
    }
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, SV_FLAG_TIMEOUT);
      return false;
    }
  }
}

// The same wait by every lane of a warp, with one result for all of them:
// lanes that disagreed (one saw the phase, another gave up) would otherwise
// part at the next warp-synchronous step.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity, bool cl, volatile int *abort_flag,
                                         const RowPassParams &P) {
  return __all_sync(0xffffffffu, wwait(bar, parity, cl, abort_flag, P.status, P.timeout_ns)) != 0;
}

// After a time-out: the entry a role of this CTA stopped at.
__device__ __forceinline__ void record_giveup(const WalkParams &W, int role, int e) {
  const int idx = 96 + ((int)blockIdx.x * 4 + role);
  if (W.giveup && idx < W.giveup_cap) W.giveup[idx] = e + 1;
}

// ---------------------------------------------------------------------------
// Producer: one bulk copy per row entry, this CTA's slice of the row.
// ---------------------------------------------------------------------------
__device__ void walk_producer(const WalkParams &W, WalkSmem &S, uint8_t *ring, int rank, volatile int *abort_flag) {
  const RowPassParams &P = W.R;
  const int e_lo = rank * W.slice;
  const int n_r = max(0, min(W.slice, P.V - e_lo));
  const uint32_t bytes = (uint32_t)n_r * (uint32_t)P.esz;  // a multiple of 16 on this path
  uint32_t nfull[kWalkMaxSlots];
#pragma unroll
  for (int i = 0; i < kWalkMaxSlots; ++i) nfull[i] = 0;
  int nrow = 0;
  bool ok = true;
  for (int e = 0;; ++e) {
    const int x = e % kWEnt;
    if (!wwait(&S.sfull[x], (uint32_t)((e / kWEnt) & 1), false, abort_flag, P.status, P.timeout_ns)) {
      ok = false;
      break;
    }
    const int kind = S.ent[x].kind;
    const int b = S.ent[x].b, pos = S.ent[x].pos, is_t = S.ent[x].is_target;
    __threadfence_block();
    *reinterpret_cast<volatile int *>(&S.prod_e) = e + 1;
    if (kind == kEntEnd) break;
    if (kind != kEntRow) continue;
    const int slot = nrow % W.nslot;
    if (!wwait(&S.empty[slot], (uint32_t)(((nrow / W.nslot) & 1) ^ 1), false, abort_flag, P.status, P.timeout_ns)) {
      ok = false;
      break;
    }
    const long long row = is_t ? ((long long)b * (P.K + 1) + pos) : ((long long)b * P.K + pos);
    const char *src = reinterpret_cast<const char *>(is_t ? P.target : P.draft) +
                      (row * (long long)P.V + e_lo) * (long long)P.esz;
    ++nfull[slot];
    if (bytes > 0) {
      mbar_arrive_expect_tx(&S.full[slot], bytes);
      bulk_g2s(ring + (size_t)slot * W.slot_bytes, src, bytes, &S.full[slot]);
    } else {
      mbar_arrive(&S.full[slot]);
    }
    ++nrow;
  }
  if (!ok) {
    record_giveup(W, 1, S.prod_e);
    // gave up: wait (bounded) for this CTA's copies still in flight
    const uint64_t t0 = global_ns();
    for (int i = 0; i < W.nslot; ++i) {
      if (nfull[i] == 0) continue;
      while (!mbar_try_wait(&S.full[i], (nfull[i] - 1u) & 1u)) {
        if (global_ns() - t0 > P.timeout_ns) break;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Math warps.
// ---------------------------------------------------------------------------
template <int kDtype>
__device__ void walk_math(const WalkParams &W, WalkSmem &S, uint8_t *ring, int rank, int tid, int warp, int lane,
                          volatile int *abort_flag) {
  const RowPassParams &P = W.R;
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;
  constexpr int kPerVec = 16 / kEsz;
  const int e_lo = rank * W.slice;
  const int n_r = max(0, min(W.slice, P.V - e_lo));
  const int nvec = n_r * kEsz / 16;
  const int nsub = (n_r + kSubChunk - 1) / kSubChunk;
  int nrow = 0;
  int e = 0;
  for (;; ++e) {
    const int x = e % kWEnt;
    if (!wait_all(&S.sfull[x], (uint32_t)((e / kWEnt) & 1), false, abort_flag, P)) break;
    const Entry E = S.ent[x];
    const int p = e % kWParts;
    const uint32_t pe_par = (uint32_t)(((e / kWParts) & 1) ^ 1);
    if (E.kind == kEntRow) {
      const int slot = nrow % W.nslot;
      if (!wait_all(&S.full[slot], (uint32_t)((nrow / W.nslot) & 1), false, abort_flag, P)) break;
      const uint8_t *buf = ring + (size_t)slot * W.slot_bytes;
      // the logit at the drafted token, read by the thread that owns its
      // vector before the statistics pass may overwrite the first max
      const int dl = E.d - e_lo;
      const bool own = E.d >= 0 && dl >= 0 && dl < n_r && (dl / kPerVec) % kConsumers == tid;
      float zsel = 0.f;
      if (own) {
        zsel = kDtype == SV_BF16 ? __uint_as_float(((uint32_t)reinterpret_cast<const unsigned short *>(buf)[dl]) << 16)
                                 : reinterpret_cast<const float *>(buf)[dl];
      }
      WarpState st;
      state_reset(st);
      if (nvec > 0)
        consume_stage<kDtype>(st, reinterpret_cast<uint4 *>(const_cast<uint8_t *>(buf)), nvec, tid, lane, e_lo, E.c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      ++nrow;
      const float Tq = st.A * fmaf(st.nbl, kLn2, 1.0f);
      const float Ew = warp_sum(Tq);
      if (!wait_all(&S.pempty[p], pe_par, false, abort_flag, P)) break;
      if (lane == 0) {
        Part pr;
        pr.m = st.M;
        pr.E = Ew;
        pr.arg = st.arg;
        pr.flags = st.flags;
        S.wpart[p][warp] = pr;
      }
      if (own) S.xz[p] = zsel;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull[p]);
    } else if (E.kind == kEntMass) {
      // residual / bonus weights of this slice per 256-element sub-chunk
      // (8 per lane), rows re-read from L2
      SampleTask t;
      t.kind = E.draw_kind;
      t.a = E.pos;
      t.c = E.c;
      t.invtau = E.invtau;
      t.nbt = E.nbt;
      t.k0_hi = E.k0_hi;
      t.k0_lo = E.k0_lo;
      t.argmax_t = E.argmax_t;
      t.u = 0.0;
      const bool resid = t.kind == kTaskResidual;
      const long long t_off = ((long long)E.b * (P.K + 1) + E.pos) * (long long)P.V;
      const long long d_off = ((long long)E.b * P.K + E.pos) * (long long)P.V;
      for (int q0 = warp; q0 < nsub; q0 += kWMath * kSampleUnroll) {
        Raw8 zt[kSampleUnroll], zd[kSampleUnroll];
#pragma unroll
        for (int u = 0; u < kSampleUnroll; ++u) {
          const int q = q0 + u * kWMath;
          zt[u].a = zt[u].b = zd[u].a = zd[u].b = make_uint4(0, 0, 0, 0);
          if (q < nsub) {
            const int v0 = e_lo + q * kSubChunk + lane * 8;
            zt[u] = load8<kDtype>(P.target, t_off, v0, P.V, true);
            if (resid) zd[u] = load8<kDtype>(P.draft, d_off, v0, P.V, true);
          }
        }
#pragma unroll
        for (int u = 0; u < kSampleUnroll; ++u) {
          const int q = q0 + u * kWMath;
          if (q < nsub) {
            float r[8];
            weights_from<kDtype>(t, t.kind, e_lo + q * kSubChunk + lane * 8, P.V, zt[u], zd[u], r);
            const float sm = warp_sum(sum8(r));
            if (lane == 0) S.subsum[E.seq][q] = sm;
          }
        }
      }
      if (!wait_all(&S.pempty[p], pe_par, false, abort_flag, P)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull[p]);
    } else {
      // find and end entries: the epilogue's; pass the partial buffer on
      if (!wait_all(&S.pempty[p], pe_par, false, abort_flag, P)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pfull[p]);
      if (E.kind == kEntEnd) return;
    }
  }
  if (lane == 0 && warp == 0) record_giveup(W, 0, e);
}

// ---------------------------------------------------------------------------
// Epilogue warp: this CTA's partial per entry, and the find entries' search.
// ---------------------------------------------------------------------------
// Locate the drawn token inside this CTA's slice: the smallest v with
// prefix(v) > T (T relative to the slice's start), from the slice's
// sub-chunk sums, then inside the crossing sub-chunk (one warp).
template <int kDtype>
__device__ void find_in_slice(const WalkParams &W, const WalkSmem &S, const Entry &E, int e_lo, int nsub, int lane) {
  const RowPassParams &P = W.R;
  const float *sub = S.subsum[E.seq];
  const int q = (nsub + 31) / 32;
  const int ja = min(nsub, lane * q), jb = min(nsub, ja + q);
  DF mine = {0.f, 0.f};
  for (int j = ja; j < jb; ++j) mine = df_add_f(mine, sub[j]);
  const DF incl = warp_incl_scan_df(mine, lane);
  DF Rtot;
  Rtot.hi = __shfl_sync(0xffffffffu, incl.hi, 31);
  Rtot.lo = __shfl_sync(0xffffffffu, incl.lo, 31);
  const DF T = {E.t_hi, E.t_lo};
  int cand = INT_MAX, last_pos = -1;
  DF pe = {0.f, 0.f};
  DF run = df_add(incl, {-mine.hi, -mine.lo});
  for (int j = ja; j < jb; ++j) {
    const float sj = sub[j];
    if (sj > 0.f) last_pos = j;
    const DF nxt = df_add_f(run, sj);
    if (cand == INT_MAX && df_gt(nxt, T)) {
      cand = j;
      pe = run;
    }
    run = nxt;
  }
  int jstar = warp_min_i(cand);
  DF pexcl;
  if (jstar != INT_MAX) {
    const int owner = __ffs(__ballot_sync(0xffffffffu, cand == jstar)) - 1;
    pexcl.hi = __shfl_sync(0xffffffffu, pe.hi, owner);
    pexcl.lo = __shfl_sync(0xffffffffu, pe.lo, owner);
  } else {
    // u R at or past the slice's total by rounding: its last sub-chunk with mass
    int lp = last_pos;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    jstar = lp < 0 ? 0 : lp;
    pexcl = df_add_f(Rtot, -sub[jstar]);
  }
  SampleTask t;
  t.kind = E.draw_kind;
  t.a = E.pos;
  t.c = E.c;
  t.invtau = E.invtau;
  t.nbt = E.nbt;
  t.k0_hi = E.k0_hi;
  t.k0_lo = E.k0_lo;
  t.argmax_t = E.argmax_t;
  t.u = 0.0;
  const long long t_off = ((long long)E.b * (P.K + 1) + E.pos) * (long long)P.V;
  const long long d_off = ((long long)E.b * P.K + E.pos) * (long long)P.V;
  const int v0 = e_lo + jstar * kSubChunk + lane * 8;
  const Raw8 zt = load8<kDtype>(P.target, t_off, v0, P.V, true);
  Raw8 zd;
  zd.a = zd.b = make_uint4(0, 0, 0, 0);
  if (t.kind == kTaskResidual) zd = load8<kDtype>(P.draft, d_off, v0, P.V, true);
  float r[8];
  weights_from<kDtype>(t, t.kind, v0, P.V, zt, zd, r);
  float pre[8];
  pre[0] = r[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) pre[k] = pre[k - 1] + r[k];
  const DF incl2 = warp_incl_scan_df({pre[7], 0.f}, lane);
  const DF base = df_add(pexcl, df_add_f(incl2, -pre[7]));
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
    int tok = c2 != INT_MAX ? c2 : (back >= 0 ? back : E.argmax_t);
    if (tok < 0 || tok >= P.V) tok = E.argmax_t;
    P.out_tokens[(size_t)E.b * (P.K + 1) + E.pos] = tok;
  }
}

template <int kDtype>
__device__ void walk_epilogue(const WalkParams &W, WalkSmem &S, int rank, int lane, volatile int *abort_flag) {
  const RowPassParams &P = W.R;
  const int e_lo = rank * W.slice;
  const int n_r = max(0, min(W.slice, P.V - e_lo));
  const int nsub = (n_r + kSubChunk - 1) / kSubChunk;
  const uint32_t xp_base = mapa_shared(&S.xp[0][rank], 0);  // the leader's copy of this CTA's partials
  const uint32_t xf_base = mapa_shared(&S.xfull[0], 0);
  int e = 0;
  for (;; ++e) {
    const int x = e % kWEnt;
    if (!wait_all(&S.sfull[x], (uint32_t)((e / kWEnt) & 1), false, abort_flag, P)) break;
    const Entry E = S.ent[x];
    const int p = e % kWParts;
    if (!wait_all(&S.pfull[p], (uint32_t)((e / kWParts) & 1), false, abort_flag, P)) break;
    XPart xo;
    xo.m = -INFINITY;
    xo.E = 0.f;
    xo.arg = INT_MAX;
    xo.flags = 0u;
    xo.z = 0.f;
    xo.has_z = 0;
    xo.mass_hi = 0.f;
    xo.mass_lo = 0.f;
    if (E.kind == kEntRow) {
      Part mine = {-INFINITY, 0.f, INT_MAX, 0u};
      if (lane < kWMath) mine = S.wpart[p][lane];
      const int dl = E.d - e_lo;
      const bool has = E.d >= 0 && dl >= 0 && dl < n_r;
      const float z = has ? S.xz[p] : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pempty[p]);
      Part R;
      R.m = __shfl_sync(0xffffffffu, mine.m, 0);
      R.E = __shfl_sync(0xffffffffu, mine.E, 0);
      R.arg = __shfl_sync(0xffffffffu, mine.arg, 0);
      R.flags = __shfl_sync(0xffffffffu, mine.flags, 0);
      for (int w = 1; w < kWMath; ++w) {
        Part o;
        o.m = __shfl_sync(0xffffffffu, mine.m, w);
        o.E = __shfl_sync(0xffffffffu, mine.E, w);
        o.arg = __shfl_sync(0xffffffffu, mine.arg, w);
        o.flags = __shfl_sync(0xffffffffu, mine.flags, w);
        R = combine(R, o, E.c);
      }
      xo.m = R.m;
      xo.E = R.E;
      xo.arg = R.arg;
      xo.flags = R.flags;
      xo.z = z;
      xo.has_z = has ? 1 : 0;
    } else if (E.kind == kEntMass) {
      // the slice's total in double-float, sub-chunks in order
      const int q = (nsub + 31) / 32;
      const int ja = min(nsub, lane * q), jb = min(nsub, ja + q);
      DF mine = {0.f, 0.f};
      for (int j = ja; j < jb; ++j) mine = df_add_f(mine, S.subsum[E.seq][j]);
      const DF incl = warp_incl_scan_df(mine, lane);
      xo.mass_hi = __shfl_sync(0xffffffffu, incl.hi, 31);
      xo.mass_lo = __shfl_sync(0xffffffffu, incl.lo, 31);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pempty[p]);
    } else {
      if (E.kind == kEntFind && E.rank == rank) find_in_slice<kDtype>(W, S, E, e_lo, nsub, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.pempty[p]);
    }
    if (lane == 0) {
      // the entry's slot may be rewritten once acknowledged: the producer
      // (normally ahead) must have read it
      if (*reinterpret_cast<volatile int *>(&S.prod_e) <= e) {
        const uint64_t t0 = global_ns();
        while (*reinterpret_cast<volatile int *>(&S.prod_e) <= e) {
          if (*abort_flag || global_ns() - t0 > P.timeout_ns) {
            *abort_flag = 1;
            break;
          }
          __nanosleep(32);
        }
      }
      // every role of this CTA is done with the entry: arm its slot for the
      // next one, then send the partial (its bytes complete the leader's barrier)
      mbar_arrive_expect_tx(&S.sfull[x], (uint32_t)sizeof(Entry));
      const uint32_t dst = xp_base + (uint32_t)(x * kWalkMaxCs * sizeof(XPart));
      const uint32_t bar = xf_base + (uint32_t)(x * sizeof(uint64_t));
      const uint4 *w = reinterpret_cast<const uint4 *>(&xo);
      st_async_v4(dst, w[0], bar);
      st_async_v4(dst + 16, w[1], bar);
    }
    __syncwarp();
    if (E.kind == kEntEnd) return;
  }
  if (lane == 0) record_giveup(W, 2, e);
}

// ---------------------------------------------------------------------------
// The leader CTA's two control warps.  The combiner merges the cluster's
// partials of each entry (lanes in parallel) and precomputes what the walk
// reads (ln S, the AV feature and confidence, the draw's crossing slice); the
// control warp's lane 0 owns the walk's state machine, and the warp publishes
// entries (lane 1 + r writes CTA r's copy) and starts sequences (lane j:
// position j).
// ---------------------------------------------------------------------------
struct Leader {  // identical in every lane of the control warp
  int app, con;          // entries appended / consumed
  int rows_app, rows_con;
  int rr;                // round-robin start over the sequence slots
  int static_next;       // next slot whose first sequence is static
  int nstage;            // entries staged in this pass
  bool tickets_left;
  bool ended;
};

enum LeaderAct : int { kActNone = 0, kActStage = 1, kActStart = 2 };

__device__ __forceinline__ Entry blank_entry(int kind) {
  Entry E;
  E.kind = kind;
  E.b = 0;
  E.pos = 0;
  E.is_target = 0;
  E.c = 1.f;
  E.d = -1;
  E.seq = 0;
  E.draw_kind = kTaskNone;
  E.nbt = 0.f;
  E.invtau = 1.f;
  E.k0_hi = 0.f;
  E.k0_lo = 0.f;
  E.rank = -1;
  E.t_hi = 0.f;
  E.t_lo = 0.f;
  E.argmax_t = 0;
  return E;
}

// Warp: lane 1 + r (r < cs) copies the n staged entries into CTA r; each
// copy's bytes complete the entry's barrier there.
__device__ __forceinline__ void warp_publish(const WalkParams &W, WalkSmem &S, int n, int lane) {
  __syncwarp();
  const int r = lane - 1;
  if (r >= 0 && r < W.cs) {
    for (int j = 0; j < n; ++j) {
      const int x = S.stage_x[j];
      const uint4 *w = reinterpret_cast<const uint4 *>(&S.lent[x]);
      const uint32_t dst = mapa_shared(&S.ent[x], (uint32_t)r);
      const uint32_t bar = mapa_shared(&S.sfull[x], (uint32_t)r);
#pragma unroll
      for (int q = 0; q < 4; ++q) st_async_v4(dst + 16 * q, w[q], bar);
    }
  }
  __syncwarp();
}

// Warp: sequence b into slot s (lane s's registers) -- its verified length,
// temperature, drafted tokens (lane j: token j) and the Philox block of each
// position (lane j: word 0 = the acceptance uniform and its logarithm, word
// 1 = the draw's uniform).
__device__ __forceinline__ void warp_start(const WalkParams &W, WalkSmem &S, SeqState &q, int s, int b, int lane) {
  const RowPassParams &P = W.R;
  SeqArr &A = S.sa[s];
  const int kr = P.draft_len ? __ldg(P.draft_len + b) : P.K;
  const int k = kr < 0 ? 0 : (kr > P.K ? P.K : kr);
  const float tau = __ldg(P.temperature + b);
  int d = 0;
  if (lane < k) d = __ldg(P.draft_tokens + (size_t)b * P.K + lane);
  const bool bad_tok = lane < k && (d < 0 || d >= P.V);
  const bool any_bad = __any_sync(0xffffffffu, bad_tok);
  if (lane < k) A.tok[lane] = d;
  if (lane <= k) {
    const U32x4 r = philox4x32_10((uint32_t)b, (uint32_t)lane, 0u, 0u, (uint32_t)(P.seed & 0xffffffffu),
                                  (uint32_t)(P.seed >> 32));
    const float u0 = (float)(r.w[0] >> 8) * (1.0f / 16777216.0f);
    A.u0[lane] = u0;
    A.lu0[lane] = logf(u0);
    A.u1[lane] = (float)(r.w[1] >> 8) * (1.0f / 16777216.0f);
  }
  if (lane == s) {
    uint32_t flags = 0u;
    if (P.draft_len && (kr < 0 || kr > P.K)) flags |= SV_FLAG_BAD_LEN;
    if (!(tau >= 0.f)) flags |= SV_FLAG_BAD_TEMP;
    if (any_bad) flags |= SV_FLAG_TOKEN_RANGE;
    q.b = b;
    q.k = k;
    q.flags = flags;
    q.greedy = !(tau > 0.f);
    q.tau = tau;
    q.inv_tau = q.greedy ? 1.f : 1.f / tau;
    q.c = q.greedy ? kLog2e : kLog2e / tau;
    q.i = 0;
    q.t_app = 0;
    q.d_app = 0;
    q.t_ok = 0;
    q.d_have = 0u;
    q.phase = kSWalk;
    q.a = 0;
    q.pending = 0;
    q.draw_kind = kTaskNone;
  }
  __syncwarp();
}

// Draw parameters of position a (residual when a < k, else the bonus row),
// as the streaming row pass computes them (lane s).
__device__ __forceinline__ void setup_draw(const WalkParams &W, const SeqArr &A, SeqState &q, int kind) {
  const Part &T = q.T;
  q.draw_kind = kind;
  q.nbt = -fmaf(T.m, q.c, q.lnSt * kLog2e);
  q.k0_hi = 0.f;
  q.k0_lo = 0.f;
  if (kind == kTaskResidual) {
    const Part D = A.D[q.a];
    const double lnr = log1p(((double)T.E - (double)D.E) / (1.0 + (double)D.E));
    const double k0 = ((double)T.m - (double)D.m) / (double)q.tau + lnr;
    q.k0_hi = (float)k0;
    q.k0_lo = (float)(k0 - (double)q.k0_hi);
  }
  q.argmax_t = (T.arg >= 0 && T.arg < W.R.V) ? T.arg : 0;
  q.phase = kSNeedMass;
}

// Decide every position whose rows are in, from the frontier on (lane s).
__device__ __forceinline__ void try_decide(const WalkParams &W, const SeqArr &A, SeqState &q) {
  const RowPassParams &P = W.R;
  while (q.phase == kSWalk && q.t_ok && (q.i == q.k || ((q.d_have >> q.i) & 1u))) {
    const int i = q.i;
    if (q.T.flags & SV_FLAG_NONFINITE) q.flags |= SV_FLAG_NONFINITE;
    if (i == q.k) {  // every verified draft accepted: the bonus from target row k
      q.a = i;
      if (q.greedy) {
        P.out_tokens[(size_t)q.b * (P.K + 1) + i] = (q.T.arg >= 0 && q.T.arg < P.V) ? q.T.arg : 0;
        q.phase = kSDrawn;
      } else {
        setup_draw(W, A, q, kTaskBonus);
      }
      return;
    }
    const int d = A.tok[i];
    const bool in_range = d >= 0 && d < P.V;
    bool reject;
    if (q.greedy) reject = !(in_range && d == q.T.arg);
    else if (!in_range) reject = true;
    else reject = reject_pre(A.u0[i], A.lu0[i], q.zt, A.zd[i], q.T, A.D[i], q.lnSt, A.lnSd[i], q.inv_tau, q.tau);
    if (!reject) {
      P.out_tokens[(size_t)q.b * (P.K + 1) + i] = d;
      q.i = i + 1;
      q.t_ok = 0;
      continue;
    }
    q.a = i;
    if (q.greedy) {
      P.out_tokens[(size_t)q.b * (P.K + 1) + i] = (q.T.arg >= 0 && q.T.arg < P.V) ? q.T.arg : 0;
      q.phase = kSDrawn;
    } else {
      setup_draw(W, A, q, kTaskResidual);
    }
    return;
  }
}

// Warp: sequence in slot s is complete -- its labels' refit terms (lane j:
// position j; labels are the drafts up to and including the first
// rejection), the tokens after a, the outputs of unverified positions, the
// accept length and status bits.
__device__ __forceinline__ void warp_finish(const WalkParams &W, WalkSmem &S, SeqState &q, int s, int lane) {
  const RowPassParams &P = W.R;
  const int K = P.K;
  const int a = __shfl_sync(0xffffffffu, q.a, s);
  const int k = __shfl_sync(0xffffffffu, q.k, s);
  const size_t b = (size_t)__shfl_sync(0xffffffffu, q.b, s);
  const uint32_t flags = __shfl_sync(0xffffffffu, q.flags, s);
  const SeqArr &A = S.sa[s];
  if (P.fit && lane < k && lane <= a) {
    const float x = A.xs[lane], conf = A.cf[lane];
    const float y = lane < a ? 1.0f : 0.0f;
    const float r = conf - y, w = conf * (1.0f - conf);
    const float qv[kFitQ] = {r * x, w * x * x, r, w * x, w, 1.0f};
#pragma unroll
    for (int j = 0; j < kFitQ; ++j) S.fit[lane * kFitQ + j] += (unsigned long long)fixed_2p32(qv[j]);
  }
  if (lane <= K && lane > a) P.out_tokens[b * (K + 1) + lane] = -1;
  if (lane < K && lane >= k) {
    const float nan = __int_as_float(0x7fc00000);
    if (P.out_feature) P.out_feature[b * K + lane] = nan;
    if (P.out_conf) P.out_conf[b * K + lane] = nan;
  }
  if (lane == 0) {
    P.out_accept_len[b] = a;
    if (flags) atomicOr(P.status, flags);
  }
  if (lane == s) q.b = -1;
  __syncwarp();
}

// Combiner warp (leader CTA): entry by entry, the cluster's partials merged
// (rows: lane r holds CTA r's partial, merged pairwise in rank order; draws:
// double-float prefix over the CTAs' masses) into S.res, then published
// through S.res_count.
__device__ void walk_combiner(const WalkParams &W, WalkSmem &S, int lane, volatile int *abort_flag) {
  const RowPassParams &P = W.R;
  int e = 0;
  for (;; ++e) {
    const int x = e % kWEnt;
    const uint32_t par = (uint32_t)((e / kWEnt) & 1);
    if (!wait_all(&S.sfull[x], par, false, abort_flag, P)) break;
    const Entry E = S.ent[x];
    if (!wait_all(&S.xfull[x], par, false, abort_flag, P)) break;
    Res R;
    R.st.m = -INFINITY;
    R.st.E = 0.f;
    R.st.arg = INT_MAX;
    R.st.flags = 0u;
    R.z = 0.f;
    R.lnS = 0.f;
    R.x = 0.f;
    R.conf = 0.f;
    R.zero = 0;
    R.rs = 0;
    R.t_hi = 0.f;
    R.t_lo = 0.f;
    if (E.kind == kEntRow) {
      Part mine = {-INFINITY, 0.f, INT_MAX, 0u};
      float z = 0.f;
      if (lane < W.cs) {
        const XPart &xp = S.xp[x][lane];
        mine.m = xp.m;
        mine.E = xp.E;
        mine.arg = xp.arg;
        mine.flags = xp.flags;
        z = xp.z;
      }
      for (int o = 1; o < W.cs; o <<= 1) {
        Part ot;
        ot.m = __shfl_down_sync(0xffffffffu, mine.m, o);
        ot.E = __shfl_down_sync(0xffffffffu, mine.E, o);
        ot.arg = __shfl_down_sync(0xffffffffu, mine.arg, o);
        ot.flags = __shfl_down_sync(0xffffffffu, mine.flags, o);
        if ((lane & (2 * o - 1)) == 0 && lane + o < W.cs) mine = combine(mine, ot, E.c);
      }
      const int owner = E.d >= 0 ? E.d / W.slice : 0;
      z = __shfl_sync(0xffffffffu, z, owner < W.cs ? owner : 0);
      if (lane == 0) {
        if (mine.arg == INT_MAX || !(fabsf(mine.m) <= FLT_MAX) || isnan(mine.E)) mine.flags |= SV_FLAG_NONFINITE;
        R.st = mine;
        R.z = E.d >= 0 ? z : 0.f;
        R.lnS = log1pf(mine.E);
        if (!E.is_target) {
          const float xf = av_feature(mine.E);
          float cf = 0.f;
          if (P.theta) cf = 1.0f / (1.0f + expf(-fmaf(S.theta[0], xf, S.theta[1 + E.pos])));
          R.x = xf;
          R.conf = cf;
          if (P.out_feature) P.out_feature[(size_t)E.b * P.K + E.pos] = xf;
          if (P.out_conf) P.out_conf[(size_t)E.b * P.K + E.pos] = cf;
        }
      }
    } else if (E.kind == kEntMass) {
      DF m = {0.f, 0.f};
      if (lane < W.cs) m = DF{S.xp[x][lane].mass_hi, S.xp[x][lane].mass_lo};
      const DF incl = warp_incl_scan_df(m, lane);
      DF Rt;
      Rt.hi = __shfl_sync(0xffffffffu, incl.hi, W.cs - 1);
      Rt.lo = __shfl_sync(0xffffffffu, incl.lo, W.cs - 1);
      if (!(Rt.hi > 0.f)) {
        R.zero = 1;
      } else {
        const DF T = df_scale(E.t_hi, Rt);  // the draw's uniform rides in t_hi
        const DF excl = df_add(incl, {-m.hi, -m.lo});
        const uint32_t hit = __ballot_sync(0xffffffffu, lane < W.cs && df_gt(incl, T));
        int rs;
        DF pre;
        if (hit) {
          rs = __ffs(hit) - 1;
          pre.hi = __shfl_sync(0xffffffffu, excl.hi, rs);
          pre.lo = __shfl_sync(0xffffffffu, excl.lo, rs);
        } else {  // u R at or past the total by rounding: the last slice with mass
          const uint32_t pos = __ballot_sync(0xffffffffu, lane < W.cs && m.hi > 0.f);
          rs = 31 - __clz(pos);
          DF mr;
          mr.hi = __shfl_sync(0xffffffffu, m.hi, rs);
          mr.lo = __shfl_sync(0xffffffffu, m.lo, rs);
          pre = df_add(Rt, {-mr.hi, -mr.lo});
        }
        const DF Trel = df_add(T, {-pre.hi, -pre.lo});
        R.rs = rs;
        R.t_hi = Trel.hi;
        R.t_lo = Trel.lo;
      }
    }
    if (lane == 0) {
      S.res[x] = R;
      st_release_cta_shared(&S.res_count, e + 1);
    }
    __syncwarp();
    if (E.kind == kEntEnd) return;
  }
  if (lane == 0) record_giveup(W, 3, e);
}

// Warp: consume entry number n (its merged partials are in S.res); lane
// E.seq updates its sequence and decides.
__device__ __forceinline__ void consume(const WalkParams &W, WalkSmem &S, Leader &L, SeqState &q, int n, int lane) {
  const RowPassParams &P = W.R;
  const int x = n % kWEnt;
  const int kind = S.lent[x].kind;
  if (kind == kEntEnd) return;
  const int s = S.lent[x].seq;
  if (kind == kEntRow) ++L.rows_con;
  int fin = 0;
  if (lane == s) {
    const Entry &E = S.lent[x];
    const Res &R = S.res[x];
    SeqArr &A = S.sa[s];
    --q.pending;
    if (kind == kEntRow) {
      if (E.is_target) {
        q.T = R.st;
        q.zt = R.z;
        q.lnSt = R.lnS;
        q.t_ok = 1;
      } else {
        const int i = E.pos;
        A.D[i] = R.st;
        A.zd[i] = R.z;
        A.lnSd[i] = R.lnS;
        A.xs[i] = R.x;
        A.cf[i] = R.conf;
        q.d_have |= 1u << i;
        if (R.st.flags & SV_FLAG_NONFINITE) q.flags |= SV_FLAG_NONFINITE;
      }
      try_decide(W, A, q);
    } else if (kind == kEntMass) {
      if (R.zero) {
        if (q.draw_kind == kTaskResidual) {
          // zero residual mass (rounding only): draw from p_a instead, and say so
          q.flags |= SV_FLAG_ZERO_RESIDUAL;
          setup_draw(W, A, q, kTaskBonus);
        } else {
          P.out_tokens[(size_t)q.b * (P.K + 1) + q.a] = q.argmax_t;
          q.phase = kSDrawn;
        }
      } else {
        q.f_rank = R.rs;
        q.f_hi = R.t_hi;
        q.f_lo = R.t_lo;
        q.phase = kSNeedFind;
      }
    } else if (kind == kEntFind) {
      q.phase = kSDrawn;
    }
    fin = q.phase == kSDrawn && q.pending == 0 && q.d_app == q.k;
  }
  if (__shfl_sync(0xffffffffu, fin, s)) warp_finish(W, S, q, s, lane);
}

// Warp: lane 0 arms the entry's partial barrier and records its slot; the
// entry itself is already in S.lent[x].
__device__ __forceinline__ void stage_slot(const WalkParams &W, WalkSmem &S, Leader &L, int lane) {
  const int x = L.app % kWEnt;
  if (lane == 0) {
    S.stage_x[L.nstage] = x;
    // the CTAs' partials for this entry complete the barrier's next phase
    mbar_arrive_expect_tx(&S.xfull[x], (uint32_t)(W.cs * sizeof(XPart)));
  }
  ++L.nstage;
  ++L.app;
}

// Warp: stage the next entry -- a target row the walk waits for first, then
// a draw, then a draft row, then a new sequence -- picked by one warp-wide
// minimum over the slots (ties in round-robin order).
__device__ __forceinline__ int choose_step(const WalkParams &W, WalkSmem &S, Leader &L, SeqState &q, int lane) {
  const RowPassParams &P = W.R;
  if (L.app - L.con >= kWEnt) return kActNone;
  const bool row_room = (L.rows_app - L.rows_con) < W.window;
  int cls = 0;
  if (lane < kWalkSeqs) {
    if (q.b >= 0) {
      if (row_room && q.phase == kSWalk && q.t_app == q.i && q.i <= q.k) cls = 1;
      else if (q.phase == kSNeedMass || q.phase == kSNeedFind) cls = 2;
      else if (row_room && q.d_app < q.k && (q.phase != kSWalk || q.d_app <= q.i + kDraftLookahead)) cls = 3;
    } else if (L.static_next < kWalkSeqs || L.tickets_left) {
      cls = 4;
    }
  }
  const int key = cls ? (cls << 6) | ((lane - L.rr) & 31) : INT_MAX;
  const int best = warp_min_i(key);
  if (best == INT_MAX) return kActNone;
  const int win = (L.rr + (best & 31)) & 31;
  cls = best >> 6;
  if (cls == 4) {
    // the first kWalkSeqs * nclusters sequences are dealt round-robin over
    // the clusters (slot-major, so small batches spread out); then tickets
    int b = -1, sn = L.static_next, tl = L.tickets_left ? 1 : 0;
    if (lane == 0) {
      if (sn < kWalkSeqs) {
        const int sb = sn * W.nclusters + (int)cluster_id_x();
        ++sn;
        if (sb < P.B) b = sb;
        else sn = kWalkSeqs;
      }
      if (b < 0 && tl) {
        const long long t = (long long)kWalkSeqs * W.nclusters + (long long)atomicAdd(W.seq_ticket, 1u);
        if (t < P.B) b = (int)t;
        else tl = 0;
      }
    }
    b = __shfl_sync(0xffffffffu, b, 0);
    L.static_next = __shfl_sync(0xffffffffu, sn, 0);
    L.tickets_left = __shfl_sync(0xffffffffu, tl, 0) != 0;
    if (b < 0) return kActNone;
    warp_start(W, S, q, win, b, lane);
    return kActStart;
  }
  const int x = L.app % kWEnt;
  if (lane == win) {
    Entry E;
    if (cls == 2) {
      E = blank_entry(q.phase == kSNeedMass ? kEntMass : kEntFind);
      E.b = q.b;
      E.pos = q.a;
      E.c = q.c;
      E.seq = win;
      E.draw_kind = q.draw_kind;
      E.nbt = q.nbt;
      E.invtau = q.inv_tau;
      E.k0_hi = q.k0_hi;
      E.k0_lo = q.k0_lo;
      E.argmax_t = q.argmax_t;
      if (q.phase == kSNeedFind) {
        E.rank = q.f_rank;
        E.t_hi = q.f_hi;
        E.t_lo = q.f_lo;
        q.phase = kSFind;
      } else {
        E.t_hi = S.sa[win].u1[q.a];  // the draw's uniform, for the combiner
        q.phase = kSMass;
      }
    } else {
      const int is_t = cls == 1;
      const int pos = is_t ? q.i : q.d_app;
      E = blank_entry(kEntRow);
      E.b = q.b;
      E.pos = pos;
      E.is_target = is_t;
      E.c = q.c;
      E.seq = win;
      const int d = pos < q.k ? S.sa[win].tok[pos] : -1;
      E.d = (d >= 0 && d < P.V) ? d : -1;
      if (is_t) ++q.t_app;
      else ++q.d_app;
    }
    ++q.pending;
    S.lent[x] = E;
  }
  __syncwarp();
  if (cls != 2) {
    ++L.rows_app;
    L.rr = (win + 1) % kWalkSeqs;
  }
  stage_slot(W, S, L, lane);
  return kActStage;
}

__device__ void walk_leader(const WalkParams &W, WalkSmem &S, int lane, volatile int *abort_flag) {
  const RowPassParams &P = W.R;
  Leader L;
  L.app = L.con = 0;
  L.rows_app = L.rows_con = 0;
  L.rr = 0;
  L.static_next = 0;
  L.nstage = 0;
  L.tickets_left = true;
  L.ended = false;
  SeqState q;  // lane s < kWalkSeqs: slot s
  q.b = -1;
  q.phase = kSWalk;
  bool failed = false;
  uint64_t t_prog = global_ns();
  for (;;) {
    bool prog = false;
    const int ncomb = ld_acquire_cta_shared(&S.res_count);
    while (L.con < ncomb) {
      consume(W, S, L, q, L.con, lane);
      ++L.con;
      prog = true;
    }
    if (L.ended) {
      if (L.con == L.app) break;
    } else {
      L.nstage = 0;
      int starts = 0;
      while (L.nstage < kWBatch) {
        const int a = choose_step(W, S, L, q, lane);
        if (a == kActNone) break;
        if (a == kActStart && ++starts >= 2) break;
        prog = true;
      }
      if (L.nstage == 0 && starts == 0 && L.app - L.con < kWEnt && !L.tickets_left && L.static_next >= kWalkSeqs &&
          __all_sync(0xffffffffu, lane >= kWalkSeqs || q.b == -1)) {
        L.ended = true;
        if (lane == 0) S.lent[L.app % kWEnt] = blank_entry(kEntEnd);
        __syncwarp();
        stage_slot(W, S, L, lane);
      }
      if (L.nstage > 0) {
        warp_publish(W, S, L.nstage, lane);
        prog = true;
      }
      if (starts) prog = true;
    }
    if (prog) {
      t_prog = global_ns();
      continue;
    }
    int stop = 0;
    if (lane == 0) {
      if (*abort_flag || (*reinterpret_cast<volatile uint32_t *>(P.status) & SV_FLAG_TIMEOUT)) {
        stop = 1;
      } else if (global_ns() - t_prog > P.timeout_ns) {
        atomicOr(P.status, SV_FLAG_TIMEOUT);
        stop = 1;
      }
      if (stop) *abort_flag = 1;
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) {
      failed = true;
      if (lane == 0) {
        record_giveup(W, 3, L.con);
        if (W.giveup && W.giveup_cap >= 96 && atomicCAS(W.giveup, 0, 1) == 0) {
          int *g = W.giveup;
          g[1] = (int)cluster_id_x();
          g[2] = L.app;
          g[3] = L.con;
          g[4] = L.rows_app;
          g[5] = L.rows_con;
          g[6] = L.static_next;
          g[7] = L.tickets_left;
          g[8] = L.ended;
        }
      }
      if (W.giveup && W.giveup_cap >= 96 && lane < kWalkSeqs) {
        int *h = W.giveup + 12 + 12 * lane;
        h[0] = q.b;
        h[1] = q.k;
        h[2] = q.i;
        h[3] = q.phase;
        h[4] = q.pending;
        h[5] = q.t_app;
        h[6] = q.d_app;
        h[7] = q.t_ok;
        h[8] = (int)q.d_have;
        h[9] = q.a;
        h[10] = q.draw_kind;
        h[11] = q.greedy;
      }
      break;
    }
    __nanosleep(32);
  }
  // this cluster's refit sums, then its completion count: the cluster that
  // completes the launch (every cluster has read theta) runs the update
  if (P.fit && !failed) {
    __syncwarp();
    for (int j = lane; j < P.K * kFitQ; j += 32)
      if (S.fit[j]) atomicAdd(P.fitacc + j, S.fit[j]);
    __threadfence();
    int last = 0;
    if (lane == 0) last = atomicAdd(P.scans_done, 1u) == (uint32_t)W.nclusters - 1u;
    if (__shfl_sync(0xffffffffu, last, 0)) {
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
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int kDtype>
__global__ void __launch_bounds__(kWThreads, 1) walk_kernel(const WalkParams W) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  WalkSmem &S = *reinterpret_cast<WalkSmem *>(base);
  uint8_t *ring = base + ((sizeof(WalkSmem) + 127) / 128) * 128;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int rank = (int)cluster_ctarank();
  const RowPassParams &P = W.R;

  if (tid == 0) {
    for (int i = 0; i < kWEnt; ++i) {
      mbar_init(&S.sfull[i], 1);
      mbar_init(&S.xfull[i], 1);
      mbar_arrive_expect_tx(&S.sfull[i], (uint32_t)sizeof(Entry));  // armed for the first entry
    }
    for (int j = 0; j < SV_MAX_K * kFitQ; ++j) S.fit[j] = 0ull;
    for (int i = 0; i < kWalkMaxSlots; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kWMath);
    }
    for (int i = 0; i < kWParts; ++i) {
      mbar_init(&S.pfull[i], kWMath);
      mbar_init(&S.pempty[i], 1);
    }
    S.abort_flag = 0;
    S.prod_e = 0;
    S.res_count = 0;
    fence_barrier_init();
  }
  if (warp == kWCtl && rank == 0 && P.theta && lane <= P.K) S.theta[lane] = __ldg(P.theta + lane);
  __syncwarp();
  // every CTA's barriers are initialised before any CTA arrives on them
  cluster_sync();
  volatile int *abort_flag = &S.abort_flag;

  if (warp < kWMath) {
    walk_math<kDtype>(W, S, ring, rank, tid, warp, lane, abort_flag);
  } else if (warp == kWProd) {
    if (lane == 0) walk_producer(W, S, ring, rank, abort_flag);
    __syncwarp();
  } else if (warp == kWEpi) {
    walk_epilogue<kDtype>(W, S, rank, lane, abort_flag);
  } else if (warp == kWCtl) {
    if (rank == 0) walk_leader(W, S, lane, abort_flag);
  } else if (rank == 0) {
    walk_combiner(W, S, lane, abort_flag);
  }
  __syncwarp();
  // no CTA leaves while another may still write into its shared memory
  cluster_sync();
}

}  // namespace

size_t walk_smem_head() { return ((sizeof(WalkSmem) + 127) / 128) * 128 + 128; }

const void *walk_kernel_fn(int dtype) {
  return dtype == SV_BF16 ? (const void *)walk_kernel<SV_BF16> : (const void *)walk_kernel<SV_FP32>;
}

int walk_threads() { return kWThreads; }

cudaError_t launch_walk(const WalkParams &W, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(W.nclusters * W.cs), 1, 1);
  lc.blockDim = dim3(kWThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = W.cs;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  lc.attrs = &attr;
  lc.numAttrs = 1;
  return W.R.dtype == SV_BF16 ? cudaLaunchKernelEx(&lc, walk_kernel<SV_BF16>, W)
                              : cudaLaunchKernelEx(&lc, walk_kernel<SV_FP32>, W);
}

}  // namespace sv
