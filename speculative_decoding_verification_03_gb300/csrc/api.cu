// Host side of the C ABI: argument checks, workspace layout, launches.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "specverify.h"
#include "sv_internal.h"

namespace sv {
size_t rowpass_smem_bytes();
cudaError_t launch_rowpass(const RowPassParams &P, int grid, cudaStream_t stream);
cudaError_t launch_sample(const SampleParams &P, int grid, cudaStream_t stream);
cudaError_t launch_avfit(const FitParams &P, int grid, cudaStream_t stream);
cudaError_t launch_philox(uint64_t seed, int nb, int npos, uint32_t *out, cudaStream_t stream);
cudaError_t launch_avsolve(unsigned char *state, float *theta, int K, float damping_c, cudaStream_t stream);
}  // namespace sv

using namespace sv;

namespace {
sv_status_t device_info(int *sms);
}

sv_status_t sv::host_device_info(int *sms) { return device_info(sms); }

namespace {

constexpr int kMaxB = 1 << 20;
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per wait

struct DevInfo {
  bool filled;
  sv_status_t status;
  int sms;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

// SM count of the current device; SV_ERR_UNSUPPORTED unless it is sm_103.
sv_status_t device_info(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo &d = g_dev[dev];
  if (!d.filled) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SV_ERR_CUDA;
    d.status = (major == 10 && minor == 3) ? SV_OK : SV_ERR_UNSUPPORTED;
    d.sms = n;
    d.filled = true;
  }
  *sms = d.sms;
  return d.status;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool shape_ok(int B, int K, int V) {
  return B >= 0 && B <= kMaxB && K >= 0 && K <= SV_MAX_K && V >= 1 && V <= SV_MAX_V;
}

int esize(sv_dtype_t dt) { return dt == SV_BF16 ? 2 : 4; }

// Chunks per row: split rows when there are too few rows to keep every SM busy.
void choose_chunks(int rows, int V, int sms, int &nch, int &chunk_elems) {
  nch = 1;
  if (rows > 0 && rows < 4 * sms) nch = (4 * sms + rows - 1) / rows;
  if (nch > kMaxChunks) nch = kMaxChunks;
  int ce = (V + nch - 1) / nch;
  ce = (ce + kChunkAlignElems - 1) / kChunkAlignElems * kChunkAlignElems;
  if (ce >= V) {
    nch = 1;
    chunk_elems = V;
    return;
  }
  chunk_elems = ce;
  nch = (V + ce - 1) / ce;
}

// Failure-detection test hook (sv_set_wait_test): per host thread.
thread_local unsigned long long t_wait_limit_ns = 0;
thread_local int t_withhold = 0;
}  // namespace

void sv::host_wait_test(unsigned long long *limit_ns, int *withhold) {
  *limit_ns = t_wait_limit_ns;
  *withhold = t_withhold;
}

namespace {

void fill_ws(RowPassParams &P, void *ws, const WsLayout &L) {
  unsigned char *w = static_cast<unsigned char *>(ws);
  P.status = reinterpret_cast<uint32_t *>(w);
  P.ticket = reinterpret_cast<uint32_t *>(w + L.ticket_off);
  P.row_cnt = reinterpret_cast<uint32_t *>(w + L.row_cnt_off);
  P.seq_cnt = reinterpret_cast<uint32_t *>(w + L.seq_cnt_off);
  P.stats = reinterpret_cast<sv_row_stats_t *>(w + L.stats_off);
  P.chunk_part = reinterpret_cast<sv_row_stats_t *>(w + L.chunk_off);
  P.tasks = reinterpret_cast<SampleTask *>(w + L.task_off);
  P.timeout_ns = t_wait_limit_ns ? t_wait_limit_ns : kTimeoutNs;
  P.withhold = t_withhold;
}

sv_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

// Measurement hook (sv_set_launch_events): per host thread.
thread_local cudaEvent_t t_ev_begin = nullptr, t_ev_end = nullptr;

cudaError_t rowpass_timed(const RowPassParams &P, int grid, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (t_ev_begin && (e = cudaEventRecord(t_ev_begin, st)) != cudaSuccess) return e;
  e = launch_rowpass(P, grid, st);
  if (e != cudaSuccess) return e;
  if (t_ev_end) e = cudaEventRecord(t_ev_end, st);
  return e;
}

}  // namespace

extern "C" {

size_t sv_workspace_bytes(int B, int K, int V) {
  if (!shape_ok(B, K, V)) return 0;
  return ws_layout(B, K, V).total;
}

}  // extern "C"

namespace {

struct FitArgs {
  float *theta;
  void *av_state;
  size_t av_state_bytes;
  int round_len;
  float damping_c;
};

sv_status_t verify_impl(int B, int K, int V, sv_dtype_t dtype, const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, const int32_t *draft_len, const float *temperature,
                        uint64_t seed, const float *theta, const sv_row_stats_t *draft_stats, int32_t *out_tokens,
                        int32_t *out_accept_len, float *out_feature, float *out_conf, void *workspace,
                        size_t workspace_bytes, void *stream, const FitArgs *fit) {
  if (!shape_ok(B, K, V) || (dtype != SV_BF16 && dtype != SV_FP32)) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  const int esz = esize(dtype);
  if (!target_logits || !temperature || !out_tokens || !out_accept_len) return SV_ERR_INVALID;
  if (K > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_INVALID;
  if (out_conf && !theta) return SV_ERR_INVALID;
  if (!aligned(target_logits, esz) || (draft_logits && !aligned(draft_logits, esz))) return SV_ERR_INVALID;
  if (!aligned(draft_tokens, 4) || !aligned(draft_len, 4) || !aligned(temperature, 4) || !aligned(theta, 4) ||
      !aligned(draft_stats, 16) || !aligned(out_tokens, 4) || !aligned(out_accept_len, 4) || !aligned(out_feature, 4) ||
      !aligned(out_conf, 4))
    return SV_ERR_INVALID;
  const WsLayout L = ws_layout(B, K, V);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return SV_ERR_WORKSPACE;
  int sms = 0;
  const sv_status_t ds = device_info(&sms);
  if (ds != SV_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  RowPassParams P{};
  std::memset(&P, 0, sizeof P);
  P.target = target_logits;
  P.draft = draft_logits;
  P.draft_tokens = draft_tokens;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.theta = theta;
  P.draft_stats_in = (K > 0) ? draft_stats : nullptr;
  P.B = B;
  P.K = K;
  P.V = V;
  P.esz = esz;
  P.dtype = dtype;
  P.mode = P.draft_stats_in ? kVerifyTargets : kVerifyFull;
  P.nslot = P.draft_stats_in ? (K + 1) : (2 * K + 1);
  choose_chunks(B * P.nslot, V, sms, P.nch, P.chunk_elems);
  P.nitems = B * P.nslot * P.nch;
  P.seed = seed;
  P.out_tokens = out_tokens;
  P.out_accept_len = out_accept_len;
  P.out_feature = out_feature;
  P.out_conf = out_conf;
  fill_ws(P, workspace, L);
  if (fit) {
    P.fit = 1;
    P.round_len = fit->round_len;
    P.damping_c = fit->damping_c;
    P.theta_rw = fit->theta;
    P.av_state = static_cast<unsigned char *>(fit->av_state);
    P.fitacc = reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(workspace) + L.fitacc_off);
    P.scans_done = P.ticket + 3;
  }

  unsigned char *w = static_cast<unsigned char *>(workspace);
  SampleParams S{};
  std::memset(&S, 0, sizeof S);
  S.target = target_logits;
  S.draft = draft_logits;
  S.B = B;
  S.K = K;
  S.V = V;
  S.esz = esz;
  S.dtype = dtype;
  S.nsub = (V + kSubChunk - 1) / kSubChunk;
  S.out_tokens = out_tokens;
  S.status = P.status;
  S.smp_cnt = reinterpret_cast<uint32_t *>(w + L.smp_cnt_off);
  S.subsum = reinterpret_cast<float *>(w + L.subsum_off);
  S.tasks = P.tasks;

  // Sampling runs inside the row pass (residual and bonus rows re-read while
  // L2-resident) when every row starts on a 16-byte boundary; otherwise a
  // separate sampler kernel follows the row pass.
  P.nstatic = P.nitems;
  P.fused = ((size_t)V * esz) % 16 == 0 && aligned(target_logits, 16) && (!draft_logits || aligned(draft_logits, 16));
  size_t clear = L.counters_off + L.counters_bytes;
  if (P.fused) {
    int sp = (S.nsub + 255) / 256;  // parts of up to 256 sub-chunks (measured: fewer, larger parts are faster)
    sp = sp < 1 ? 1 : (sp > kMaxSampleParts ? kMaxSampleParts : sp);
    P.sp = sp;
    P.spc = (S.nsub + sp - 1) / sp;
    P.dq = reinterpret_cast<int *>(w + L.dq_off);
    P.dq_tail = P.ticket + 1;
    P.dq_head = P.ticket + 2;
    P.smp = S;
    // early exit: target rows past a sequence's first rejection are not
    // read.  Used when the draft rows are streamed as well: their reads keep
    // the GPU busy while each sequence's chain of target rows advances one
    // decision at a time (with precomputed draft statistics the chain would
    // run alone, and reading every verified target row at once is faster)
    const bool early_exit = P.mode == kVerifyFull;
    P.nch_dyn = 1;  // queued target rows stay whole (chunking them measured slower)
    P.chunk_elems_dyn = (V + kChunkAlignElems - 1) / kChunkAlignElems * kChunkAlignElems;
    if (early_exit) {
      P.lazy = 1;
      P.ngroups = K + 1;
      P.nstatic = P.nitems = P.ngroups * B * P.nch;
      P.ndyn = B * sp;
      P.ntq = B * K * P.nch_dyn;
      P.tq = reinterpret_cast<int *>(w + L.tq_off);
      P.tq_tail = P.ticket + 4;
      P.tq_head = P.ticket + 5;
      // Reading target rows D positions ahead costs the rows of positions
      // that are rejected before them and shortens each sequence's chain of
      // decisions.  Measured (launch us, bf16): 64 x 5 x 32000 (37 MB of
      // first-pass rows) D = 1 / 2 / 3: 62.3 / 57.4 / 56.5; 256 x 6 x 128256
      // (722 MB) D = 0 / 1 / 2 / 3: 166 / 144.7 / 149.8 / 152.9; 1024 x 8 x
      // 151936 (4.7 GB) D = 0 faster than D = 1.  The chains, not the bytes,
      // bound the small launches.
      const double first_pass = (double)B * (2 * K + 1) * V * esz;
      P.spec = first_pass < 1.28e8 ? 3 : (first_pass < 1.0e9 ? 1 : 0);
      // a share of the CTAs serve the draws' sample items before static
      // items, so the draws of sequences decided early do not all queue up
      // behind the static rows (measured at 256 x 6 x 128256: 1 in 8 145.1 ->
      // 143.3 us, 1 in 4 145.3, 1 in 2 157.9, every CTA 154.8; at 1024 x 8 x
      // 151936: 1 in 4 682 us against 689 us for 1 in 8)
      P.draw_every = first_pass < 1.0e9 ? 8 : 4;
    } else {
      P.ndyn = B * sp;
    }
    P.pos_cnt = reinterpret_cast<uint32_t *>(w + L.pos_cnt_off);
    clear = P.lazy ? L.tq_off + (size_t)P.ntq * 4 : L.dq_off + (size_t)P.ndyn * 4;
  }

  // status word (offset 0) and the per-call counters, in one clear
  cudaError_t e = cudaMemsetAsync(w, 0, clear, st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  const long long tickets = (long long)P.nitems + (P.fused ? P.ndyn : 0) + P.ntq;
  const int grid = tickets < sms ? (int)tickets : sms;
  e = rowpass_timed(P, grid, st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  if (P.fused) return SV_OK;

  const long long groups = (long long)B * ((S.nsub + kSampleUnroll - 1) / kSampleUnroll);
  long long sgrid = (long long)sms * kSampleCtasPerSm;
  const long long need = (groups + kSampleWarps - 1) / kSampleWarps;
  if (need < sgrid) sgrid = need;
  e = launch_sample(S, (int)sgrid, st);
  return cuda_status(e);
}

}  // namespace

extern "C" {

sv_status_t sv_verify(int B, int K, int V, sv_dtype_t dtype, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const int32_t *draft_len, const float *temperature, uint64_t seed,
                      const float *theta, const sv_row_stats_t *draft_stats, int32_t *out_tokens,
                      int32_t *out_accept_len, float *out_feature, float *out_conf, void *workspace,
                      size_t workspace_bytes, void *stream) {
  return verify_impl(B, K, V, dtype, target_logits, draft_logits, draft_tokens, draft_len, temperature, seed, theta,
                     draft_stats, out_tokens, out_accept_len, out_feature, out_conf, workspace, workspace_bytes,
                     stream, nullptr);
}

sv_status_t sv_verify_fit(int B, int K, int V, sv_dtype_t dtype, const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const int32_t *draft_len, const float *temperature,
                          uint64_t seed, float *theta, const sv_row_stats_t *draft_stats, int32_t *out_tokens,
                          int32_t *out_accept_len, float *out_feature, float *out_conf, void *av_state,
                          size_t av_state_bytes, int round_len, float damping_c, void *workspace,
                          size_t workspace_bytes, void *stream) {
  if (!theta || !aligned(theta, 4) || round_len < 0 || !(damping_c >= 0.f)) return SV_ERR_INVALID;
  if (K < 0 || K > SV_MAX_K) return SV_ERR_INVALID;
  if (!av_state || !aligned(av_state, 256) || av_state_bytes < sv_av_state_bytes(K)) return SV_ERR_WORKSPACE;
  if (B == 0)  // no sequences: the round still advances by one step
    return sv_av_fit_step(0, K, theta, av_state, av_state_bytes, round_len, damping_c, nullptr, nullptr, nullptr,
                          stream);
  FitArgs f{theta, av_state, av_state_bytes, round_len, damping_c};
  return verify_impl(B, K, V, dtype, target_logits, draft_logits, draft_tokens, draft_len, temperature, seed, theta,
                     draft_stats, out_tokens, out_accept_len, out_feature, out_conf, workspace, workspace_bytes,
                     stream, &f);
}

sv_status_t sv_av_score(int B, int K, int V, sv_dtype_t dtype, const void *draft_logits, const float *temperature,
                        const float *theta, float keep_threshold, float *out_feature, float *out_conf,
                        int32_t *out_kept_len, sv_row_stats_t *out_draft_stats, void *workspace,
                        size_t workspace_bytes, void *stream) {
  if (!shape_ok(B, K, V) || (dtype != SV_BF16 && dtype != SV_FP32)) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  const int esz = esize(dtype);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!temperature || !theta) return SV_ERR_INVALID;
  if (K > 0 && (!draft_logits || !out_feature || !out_conf)) return SV_ERR_INVALID;
  if ((draft_logits && !aligned(draft_logits, esz)) || !aligned(temperature, 4) || !aligned(theta, 4) ||
      !aligned(out_feature, 4) || !aligned(out_conf, 4) || !aligned(out_kept_len, 4) || !aligned(out_draft_stats, 16))
    return SV_ERR_INVALID;
  if (!(keep_threshold == keep_threshold)) return SV_ERR_INVALID;
  const WsLayout L = ws_layout(B, K, V);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return SV_ERR_WORKSPACE;
  int sms = 0;
  const sv_status_t ds = device_info(&sms);
  if (ds != SV_OK) return ds;
  if (K == 0) {
    if (out_kept_len) return cuda_status(cudaMemsetAsync(out_kept_len, 0, (size_t)B * 4, st));
    return SV_OK;
  }
  RowPassParams P{};
  std::memset(&P, 0, sizeof P);
  P.draft = draft_logits;
  P.temperature = temperature;
  P.theta = theta;
  P.B = B;
  P.K = K;
  P.V = V;
  P.esz = esz;
  P.dtype = dtype;
  P.mode = kScore;
  P.nslot = K;
  choose_chunks(B * K, V, sms, P.nch, P.chunk_elems);
  P.nitems = B * K * P.nch;
  P.keep_threshold = keep_threshold;
  P.nstatic = P.nitems;
  P.out_feature = out_feature;
  P.out_conf = out_conf;
  P.out_kept_len = out_kept_len;
  P.out_draft_stats = out_draft_stats;
  fill_ws(P, workspace, L);
  unsigned char *w = static_cast<unsigned char *>(workspace);
  cudaError_t e = cudaMemsetAsync(w, 0, L.counters_off + L.counters_bytes, st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  const int grid = P.nitems < sms ? P.nitems : sms;
  return cuda_status(rowpass_timed(P, grid, st));
}

size_t sv_av_state_bytes(int K) {
  if (K < 0 || K > SV_MAX_K) return 0;
  return kAvPartOff + (size_t)kFitMaxCtas * SV_MAX_K * kFitQ * sizeof(double);
}

sv_status_t sv_av_reset(int K, void *av_state, size_t av_state_bytes, void *stream) {
  if (K < 0 || K > SV_MAX_K) return SV_ERR_INVALID;
  if (!av_state || !aligned(av_state, 256) || av_state_bytes < sv_av_state_bytes(K)) return SV_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(av_state, 0, sv_av_state_bytes(K), static_cast<cudaStream_t>(stream)));
}

sv_status_t sv_av_fit_step(int B, int K, float *theta, void *av_state, size_t av_state_bytes, int round_len,
                           float damping_c, const float *feature, const int32_t *accept_len, const int32_t *kept_len,
                           void *stream) {
  if (B < 0 || B > kMaxB || K < 0 || K > SV_MAX_K || round_len < 0 || !(damping_c >= 0.f)) return SV_ERR_INVALID;
  if (!theta || !aligned(theta, 4)) return SV_ERR_INVALID;
  if (B > 0 && K > 0 && (!feature || !accept_len)) return SV_ERR_INVALID;
  if (!aligned(feature, 4) || !aligned(accept_len, 4) || !aligned(kept_len, 4)) return SV_ERR_INVALID;
  if (!av_state || !aligned(av_state, 256) || av_state_bytes < sv_av_state_bytes(K)) return SV_ERR_WORKSPACE;
  int sms = 0;
  const sv_status_t ds = device_info(&sms);
  if (ds != SV_OK) return ds;
  FitParams F{};
  F.B = B;
  F.K = K;
  F.round_len = round_len;
  F.damping_c = damping_c;
  F.theta = theta;
  F.feature = feature;
  F.accept_len = accept_len;
  F.kept_len = kept_len;
  F.state = static_cast<unsigned char *>(av_state);
  int grid = (B + kFitSeqPerCta - 1) / kFitSeqPerCta;  // about 64 sequences per CTA
  if (grid < 1) grid = 1;
  if (grid > kFitMaxCtas) grid = kFitMaxCtas;
  return cuda_status(launch_avfit(F, grid, static_cast<cudaStream_t>(stream)));
}

size_t sv_av_accum_offset(void) { return kAvAccOff; }

size_t sv_av_accum_bytes(int K) {
  if (K < 0 || K > SV_MAX_K) return 0;
  return (size_t)(4 * K + 2) * sizeof(double);
}

sv_status_t sv_av_solve(int K, float *theta, void *av_state, size_t av_state_bytes, float damping_c, void *stream) {
  if (K < 0 || K > SV_MAX_K || !(damping_c >= 0.f)) return SV_ERR_INVALID;
  if (!theta || !aligned(theta, 4)) return SV_ERR_INVALID;
  if (!av_state || !aligned(av_state, 256) || av_state_bytes < sv_av_state_bytes(K)) return SV_ERR_WORKSPACE;
  int sms = 0;
  const sv_status_t ds = device_info(&sms);
  if (ds != SV_OK) return ds;
  return cuda_status(launch_avsolve(static_cast<unsigned char *>(av_state), theta, K, damping_c,
                                    static_cast<cudaStream_t>(stream)));
}

sv_status_t sv_philox(uint64_t seed, int nb, int npos, uint32_t *out, void *stream) {
  if (nb < 0 || npos < 0 || (long long)nb * npos > (1ll << 30)) return SV_ERR_INVALID;
  if ((long long)nb * npos == 0) return SV_OK;
  if (!out || !aligned(out, 16)) return SV_ERR_INVALID;
  int sms = 0;
  const sv_status_t ds = device_info(&sms);
  if (ds != SV_OK) return ds;
  return cuda_status(launch_philox(seed, nb, npos, out, static_cast<cudaStream_t>(stream)));
}

sv_status_t sv_status(void *status_holder, void *stream, uint32_t *flags_out) {
  if (!status_holder) return SV_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  uint32_t flags = 0;
  if (cudaMemcpy(&flags, status_holder, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
  if (flags && cudaMemset(status_holder, 0, 4) != cudaSuccess) return SV_ERR_CUDA;
  if (flags_out) *flags_out = flags;
  if (flags & SV_FLAG_TIMEOUT) return SV_ERR_TIMEOUT;
  if (flags & SV_FLAG_NONFINITE) return SV_ERR_NONFINITE;
  if (flags & SV_FLAG_TOKEN_RANGE) return SV_ERR_TOKEN_RANGE;
  if (flags & SV_FLAG_BAD_LEN) return SV_ERR_BAD_LEN;
  if (flags & SV_FLAG_BAD_TEMP) return SV_ERR_BAD_TEMP;
  return SV_OK;
}

sv_status_t sv_set_wait_test(uint64_t limit_ns, int withhold) {
  t_wait_limit_ns = limit_ns;
  t_withhold = withhold != 0;
  return SV_OK;
}

sv_status_t sv_set_launch_events(void *begin_event, void *end_event) {
  if ((begin_event == nullptr) != (end_event == nullptr)) return SV_ERR_INVALID;
  t_ev_begin = static_cast<cudaEvent_t>(begin_event);
  t_ev_end = static_cast<cudaEvent_t>(end_event);
  return SV_OK;
}

}  // extern "C"

namespace {

// Scratch for sv_verify_noalloc: a file-scope device array, so the entry
// point needs no allocation.  Host code cannot use the symbol as a device
// address; noalloc_scratch() looks the address up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];
unsigned long long g_noalloc_ctx[64];

// A process-unique id of the current CUDA context (0 if it cannot be read),
// from the driver's cuCtxGetCurrent / cuCtxGetId, looked up through the
// runtime so that the library does not link the driver library.  A device
// reset replaces the context, and with it the scratch array's address.
unsigned long long current_context_id() {
  using GetCurrent = int (*)(void **);
  using GetId = int (*)(void *, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    looked_up = true;
  }
  void *ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == 0 && ctx && get_id(ctx, &id) == 0) return id;
  return 0;
}

// The device address of the scratch array in the current context: looked up
// once per device and context (cudaGetSymbolAddress), again after a device
// reset created a new context, and on every call if the context's id cannot
// be read.  The caller holds g_noalloc_mu.
sv_status_t noalloc_scratch_locked(int dev, void **out) {
  const unsigned long long ctx = current_context_id();
  if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      g_noalloc_ptr[dev] = nullptr;
      return SV_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = ptr;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return SV_OK;
}

sv_status_t noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  return noalloc_scratch_locked(dev, out);
}

}  // namespace

extern "C" {

sv_status_t sv_verify_noalloc(int B, int K, int V, sv_dtype_t dtype, const void *target_logits,
                              const void *draft_logits, const int32_t *draft_tokens, const int32_t *draft_len,
                              const float *temperature, uint64_t seed, const float *theta,
                              const sv_row_stats_t *draft_stats, int32_t *out_tokens, int32_t *out_accept_len,
                              float *out_feature, float *out_conf, void *stream) {
  if (!shape_ok(B, K, V)) return SV_ERR_INVALID;
  if (sv_workspace_bytes(B, K, V) > (size_t)SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;
  void *scratch = nullptr;
  const sv_status_t st = noalloc_scratch(&scratch);
  if (st != SV_OK) return st;
  return sv_verify(B, K, V, dtype, target_logits, draft_logits, draft_tokens, draft_len, temperature, seed, theta,
                   draft_stats, out_tokens, out_accept_len, out_feature, out_conf, scratch,
                   (size_t)SV_NOALLOC_SCRATCH_BYTES, stream);
}

void *sv_noalloc_status_holder(void) {
  void *ptr = nullptr;
  return noalloc_scratch(&ptr) == SV_OK ? ptr : nullptr;
}

const char *sv_strerror(sv_status_t s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_NONFINITE: return "non-finite logits";
    case SV_ERR_TOKEN_RANGE: return "drafted token out of range";
    case SV_ERR_TIMEOUT: return "device wait timed out";
    case SV_ERR_WORKSPACE: return "workspace too small or misaligned";
    case SV_ERR_BAD_LEN: return "draft_len outside [0, K]";
    case SV_ERR_BAD_TEMP: return "negative or NaN temperature";
  }
  return "unknown status";
}

}  // extern "C"
