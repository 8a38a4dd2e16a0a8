// Internal definitions shared by the host API and the kernels: launch
// parameters, the per-sequence sampling task, and the workspace layout.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// ---- row pass geometry -----------------------------------------------------
constexpr int kStageBytes = 55296;                 // one TMA bulk copy (9 x 384 threads x 16 B)
constexpr int kStages = 4;                         // ring depth (216 KB in flight per SM)
constexpr int kConsumerWarps = 12;
constexpr int kConsumers = kConsumerWarps * 32;    // 384 math threads
constexpr int kEpiWarps = 3;                       // epilogue warps (take items from a shared counter)
constexpr int kPartSlots = 8;                      // finished items the math warps may run ahead
constexpr int kRowThreads = kConsumers + 32 + 32 * kEpiWarps;  // + producer warp + epilogue warps
constexpr int kVecPerStage = kStageBytes / 16;     // 3456 16-byte vectors
constexpr int kVecPerThread = kVecPerStage / kConsumers;  // 9
static_assert(kVecPerStage % kConsumers == 0, "a stage is a whole number of vectors per math thread");
constexpr int kMaxChunks = 16;                     // chunks a row may be split into
constexpr int kChunkAlignElems = 512;              // chunk starts stay 16-byte aligned within a row

// Row pass modes: which rows of a sequence are streamed.
enum RowMode : int {
  kVerifyFull = 0,     // slots t0 d0 t1 d1 ... tK (target and draft rows)
  kVerifyTargets = 1,  // slots t0 .. tK (draft statistics supplied by the caller)
  kScore = 2           // slots d0 .. d{K-1} (AV scoring only)
};

// ---- sampling ----------------------------------------------------------------
constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSubChunk = 32 * 8;                  // 256 elements per partial sum (one warp, 8 per lane)
constexpr int kSampleUnroll = 4;                   // sub-chunks a warp loads before reducing
constexpr int kSampleCtasPerSm = 3;                // grid of the grid-stride sampler

enum TaskKind : int { kTaskNone = 0, kTaskResidual = 1, kTaskBonus = 2 };
constexpr int kQueueNop = 0x7fffffff;

// Everything the sampler needs for sequence b, written by the acceptance scan.
//   p_v  proportional to 2^(z_t[v] * c + nbt)
//   delta_v = ln q_v - ln p_v = (z_d[v] - z_t[v]) * invtau + (k0_hi + k0_lo)
//   residual weight r_v = p_v * (1 - e^delta_v) where delta_v < 0, else 0
struct SampleTask {
  int32_t kind;
  int32_t a;       // position whose row is sampled
  float c;         // log2(e) / tau
  float invtau;    // 1 / tau
  float nbt;       // -(m_t * c + ln S_t * log2 e), rounded
  float k0_hi;     // (m_t - m_d) / tau + ln S_t - ln S_d, split in two floats
  float k0_lo;
  int32_t argmax_t;  // fallback token
  double u;        // U(seed, b, a, 1)
};

struct SampleParams {
  const void *target;
  const void *draft;
  int B, K, V, esz, dtype;
  int nsub;       // sub-chunks per row
  int32_t *out_tokens;
  uint32_t *status;
  uint32_t *smp_cnt;  // [B]
  float *subsum;      // [B][nsub]
  const SampleTask *tasks;
};

struct RowPassParams {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  const int32_t *draft_len;
  const float *temperature;
  const float *theta;
  const sv_row_stats_t *draft_stats_in;
  int B, K, V, esz, dtype;
  int mode;
  int nslot;        // row slots per sequence in this mode
  int nch;          // chunks per row
  int chunk_elems;  // elements per chunk (multiple of kChunkAlignElems unless nch == 1)
  int nitems;       // B * nslot * nch
  uint64_t seed;
  float keep_threshold;
  // outputs
  int32_t *out_tokens;
  int32_t *out_accept_len;
  float *out_feature;
  float *out_conf;
  int32_t *out_kept_len;
  sv_row_stats_t *out_draft_stats;
  // workspace
  uint32_t *status;
  uint32_t *ticket;
  uint32_t *row_cnt;       // [B][2K+1]
  uint32_t *seq_cnt;       // [B]
  sv_row_stats_t *stats;   // [B][2K+1]: target j at 2j, draft i at 2i+1
  sv_row_stats_t *chunk_part;  // [B][2K+1][kMaxChunks]
  SampleTask *tasks;       // [B]
  unsigned long long timeout_ns;
  // fused sampling: after a sequence's scan, `sp` sample items (b, part) are
  // published in dq; tickets nstatic .. nstatic + ndyn - 1 take them in order
  int fused;
  int sp;        // sample parts per sequence
  int spc;       // sub-chunks per part
  int nstatic;   // static row items (= nitems)
  int ndyn;      // B * sp
  int *dq;       // [ndyn]: b * sp + part + 1 once published, 0 before
  uint32_t *dq_tail;   // slots reserved by publishers
  uint32_t *dq_head;   // slots claimed by producers
  SampleParams smp;
  // fused AV refit (sv_verify_fit): every scan adds its labels' terms to
  // fitacc as 2^-32 fixed point; the last scan updates the round
  int fit;
  int round_len;
  float damping_c;
  float *theta_rw;
  unsigned char *av_state;
  unsigned long long *fitacc;  // [SV_MAX_K][kFitQ]
  uint32_t *scans_done;
  // early exit (fused verify modes): the static items are every sequence's
  // first target row and its draft rows, position-major (all t0, all d0,
  // all d1, ...); target row i + 1 of a sequence is queued when position i
  // is accepted, so no target row past the first rejection is read.  Queued
  // target rows have a queue of their own, which producers serve before
  // anything else: tq codes 1 + (b K + i - 1) nch_dyn + chunk (target row i)
  // or kQueueNop (fillers for the rows a sequence never queued, which keep
  // the queue's length at ntq = B K nch_dyn).  dq then holds only the sample
  // items, 1 + b sp + part (ndyn = B sp).  A producer claims a slot of either
  // queue only once it has been reserved, so no producer waits for work that
  // only another producer's rows could publish.
  int *tq;
  uint32_t *tq_tail;
  uint32_t *tq_head;
  int ntq;
  int lazy;
  int ngroups;        // static groups: first target rows, then draft rows of each position
  int nch_dyn;        // chunks of a queued target row (shortens the chain of decisions)
  int chunk_elems_dyn;
  uint32_t *pos_cnt;  // [B][K+1]: events of position i (reached, target row, draft row)
  int spec;           // look-ahead D: position i >= 1 accepted queues target row i + 1 + D
  int draw_every;     // CTAs with blockIdx % draw_every == 0 take sample items before static items (0: none)
  int withhold;       // failure-detection tests: the producers stage nothing (sv_set_wait_test)
};


// ---- workspace layout --------------------------------------------------------
constexpr int kMaxSampleParts = 16;

struct WsLayout {
  size_t counters_off, counters_bytes;  // zeroed by every call
  size_t ticket_off, fitacc_off, row_cnt_off, seq_cnt_off, smp_cnt_off, pos_cnt_off, dq_off, tq_off;
  size_t stats_off, chunk_off, task_off, subsum_off;
  size_t total;
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int B, int K, int V) {
  WsLayout L{};
  const size_t nrow = (size_t)B * (size_t)(2 * K + 1);
  const size_t nsub = ((size_t)V + kSubChunk - 1) / kSubChunk;
  size_t off = 256;  // status word and spare header
  L.counters_off = off;
  L.ticket_off = off;  // ticket, dq_tail, dq_head, scans_done, tq_tail, tq_head
  off += 32;
  L.fitacc_off = off;  // [SV_MAX_K][6] 64-bit fixed point
  off += (size_t)SV_MAX_K * 6 * 8;
  L.row_cnt_off = off;
  off += nrow * 4;
  L.seq_cnt_off = off;
  off += (size_t)B * 4;
  L.smp_cnt_off = off;
  off += (size_t)B * 4;
  L.pos_cnt_off = off;
  off += (size_t)B * (K + 1) * 4;
  L.dq_off = off;  // sample items [B][kMaxSampleParts]
  off += (size_t)B * kMaxSampleParts * 4;
  L.tq_off = off;  // last: a call clears only the entries it uses
  off += (size_t)B * K * kMaxChunks * 4;
  off = align_up(off, 256);
  L.counters_bytes = off - L.counters_off;
  L.stats_off = off;
  off = align_up(off + nrow * sizeof(sv_row_stats_t), 256);
  L.chunk_off = off;
  off = align_up(off + nrow * kMaxChunks * sizeof(sv_row_stats_t), 256);
  L.task_off = off;
  off = align_up(off + (size_t)B * sizeof(SampleTask), 256);
  L.subsum_off = off;
  off = align_up(off + (size_t)B * nsub * sizeof(float), 256);
  L.total = off;
  return L;
}

// ---- AV refit state ------------------------------------------------------------
constexpr int kFitSeqPerCta = 64;
constexpr int kFitMaxCtas = 64;
constexpr int kFitQ = 6;  // per position: g_w part, H_ww part, g_b, H_wb, H_bb, n

struct AvStateHeader {
  uint32_t status;
  uint32_t step;       // decode steps accumulated in the current round
  uint32_t cta_done;   // arrivals of the current launch (self-resetting)
  uint32_t K;
};

// Layout inside the AV state buffer:
//   [header 256 B] [acc (doubles): g (K+1), Hww (1), Hwb (K), Hbb (K), n (K)]
//   [partials (floats): kFitMaxCtas x SV_MAX_K x kFitQ]
constexpr size_t kAvAccOff = 256;
constexpr size_t kAvAccDoubles = 4 * SV_MAX_K + 2;
constexpr size_t kAvPartOff = align_up(kAvAccOff + kAvAccDoubles * 8, 256);

// ---- host helpers shared by the entry points (api.cu) ------------------------
// SM count of the current device; SV_ERR_UNSUPPORTED unless it is sm_103.
sv_status_t host_device_info(int *sms);
// The calling host thread's sv_set_wait_test settings (limit 0 = default).
void host_wait_test(unsigned long long *limit_ns, int *withhold);
inline sv_status_t host_cuda_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }
inline bool host_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct FitParams {
  int B, K, round_len;
  float damping_c;
  float *theta;
  const float *feature;
  const int32_t *accept_len;
  const int32_t *kept_len;
  unsigned char *state;
};

}  // namespace sv
