/*
 * specverify -- batched speculative-decoding verification with the
 * Adaptive-Verification (AV) acceptance estimator, for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; no CUDA or framework types.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Device pointers point to memory of the current CUDA device; the caller
 *    owns every buffer (inputs, outputs, workspace, AV state).  The library
 *    never allocates and never frees.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call only enqueues work on it and returns without
 *    waiting; only sv_status() synchronises.
 *  - Arguments the host can check (sizes, NULL pointers, alignment, workspace
 *    size) are checked before anything is enqueued; a failed check returns an
 *    error and enqueues nothing.
 *  - Conditions only the GPU can see (NaN logits, out-of-range drafted tokens,
 *    draft_len outside [0, K], negative temperatures, a wait that timed out)
 *    set bits of a 32-bit status word held in the first 4 bytes of the
 *    workspace (or of the AV state); sv_status() reads and clears it.  A call
 *    that uses a workspace clears its status word first, so the word reports
 *    the most recent call; the AV state's word accumulates across refit steps
 *    until it is read.  The
 *    kernels never trap: the affected sequence still gets outputs, produced
 *    by the rules stated at each flag.
 *  - The verification and TTS kernels are persistent (one CTA per SM) and
 *    their CTAs hand work to one another through bounded waits, so a launch
 *    expects its CTAs to be resident together: with other kernels holding
 *    the SMs, a wait can give up (SV_FLAG_TIMEOUT) instead of completing.
 *  - Logits are row-major, the vocabulary innermost and contiguous.  Any
 *    V in [1, SV_MAX_V] is accepted; rows need not be 16-byte aligned (the
 *    ragged ends are read with plain loads), but each logit pointer must be
 *    aligned to its element size.
 *
 * Notation (as in the AV article): p = target (verifier) distribution,
 * q = draft distribution.  B sequences, K drafted tokens each, vocabulary V.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_MAX_K 16
#define SV_MAX_V (1 << 24)

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID = 1,      /* a host-checkable argument is wrong              */
    SV_ERR_UNSUPPORTED = 2,  /* device is not sm_103 / feature not available    */
    SV_ERR_CUDA = 3,         /* a CUDA runtime call failed                      */
    SV_ERR_NONFINITE = 4,    /* device: NaN in a row, or a row's max not finite */
    SV_ERR_TOKEN_RANGE = 5,  /* device: a drafted token outside [0, V)          */
    SV_ERR_TIMEOUT = 6,      /* device: a bounded wait gave up                  */
    SV_ERR_WORKSPACE = 7,    /* workspace (or AV state) too small or misaligned */
    SV_ERR_BAD_LEN = 8,      /* device: draft_len[b] outside [0, K]             */
    SV_ERR_BAD_TEMP = 9      /* device: temperature[b] negative or NaN          */
} sv_status_t;

typedef enum { SV_BF16 = 0, SV_FP32 = 1 } sv_dtype_t;

/* Bits of the device status word (sv_status maps them to sv_status_t). */
#define SV_FLAG_NONFINITE      (1u << 0)
#define SV_FLAG_TOKEN_RANGE    (1u << 1)
#define SV_FLAG_TIMEOUT        (1u << 2)
#define SV_FLAG_BAD_LEN        (1u << 3)
#define SV_FLAG_BAD_TEMP       (1u << 4)
#define SV_FLAG_ZERO_RESIDUAL  (1u << 5) /* warning only: residual mass 0 by rounding, p sampled */
#define SV_FLAG_FIT_SINGULAR   (1u << 6) /* warning only: refit system not positive definite, theta kept */

/* Softmax statistics of one vocabulary row, 16 bytes.
 *   m      max_v z_v of the raw logits (before the temperature)
 *   E      sum over v != argmax of exp((z_v - m) / tau)  (exactly one copy of
 *          the max excluded); so S = 1 + E, ln S = log1p(E), q_max = 1 / S,
 *          logit(q_max) = -ln E
 *   argmax lowest index attaining m
 *   flags  SV_FLAG_* bits seen on this row
 * Greedy rows (tau == 0) are summarised at tau = 1. */
typedef struct {
    float m;
    float E;
    int32_t argmax;
    uint32_t flags;
} sv_row_stats_t;

/* ------------------------------------------------------------------------
 * sv_workspace_bytes -- size of the scratch buffer sv_verify and sv_av_score
 * need for this shape (row statistics, per-call counters, sampling partial
 * sums, status word).  The buffer must be 256-byte aligned.  Its contents
 * need no initialisation: each call clears what it uses on `stream`.  Calls
 * that share one workspace must be ordered (same stream, or events).
 * Returns 0 for an invalid shape.
 * ---------------------------------------------------------------------- */
size_t sv_workspace_bytes(int B, int K, int V);

/* ------------------------------------------------------------------------
 * sv_verify -- one batched verification step.
 *
 * Defined by "Speculative Decoding: Draft, EAGLE, MTP" (cheatsheet), section
 * "one speculative step" and its "algorithm loop in code": drafts d_i are
 * accepted left to right with probability min(1, p_i(d_i) / q_i(d_i)); at
 * the first rejection a token is drawn from the normalised positive residual
 * max(p_a - q_a, 0); if every verified draft is accepted a bonus token is
 * drawn from the next target row.  With theta != NULL the AV score of every
 * verified draft is computed in the same pass ("Adaptive Verification
 * without a confidence head", sections "Solution" and "Scoring the
 * distribution"): x_i = logit(q_max) of draft row i, conf_i =
 * sigmoid(omega * x_i + beta_i).
 *
 *   B, K, V         sequences, drafts per sequence (0..SV_MAX_K), vocabulary
 *   dtype           SV_BF16 or SV_FP32 logits
 *   target_logits   device [B][K+1][V]; row j = target logits at draft
 *                   position j (row K follows the last draft)
 *   draft_logits    device [B][K][V] (required when K > 0; with draft_stats
 *                   only the residual rows are read from it)
 *   draft_tokens    device int32 [B][K], the drafted tokens
 *   draft_len       device int32 [B] or NULL (= K): k_b drafts of sequence b
 *                   are verified; target rows j > k_b and draft rows i >= k_b
 *                   are not read.  Out-of-range values set SV_FLAG_BAD_LEN and
 *                   are clamped to [0, K].
 *   temperature     device float [B]; tau_b > 0 divides both rows' logits;
 *                   0 makes the row greedy: draft i is accepted iff it equals
 *                   the target argmax of row i (lowest index on ties) and the
 *                   emitted token is that argmax; no uniforms are drawn.
 *                   Negative or NaN values set SV_FLAG_BAD_TEMP and act as 0.
 *   seed            Philox4x32-10 key.  Acceptance at position i uses
 *                   U(seed, b, i, 0); the residual/bonus draw at position a
 *                   uses U(seed, b, a, 1), where U(seed, b, pos, draw) is the
 *                   top 24 bits of output word (draw % 4) of Philox4x32-10
 *                   with key (seed & 0xffffffff, seed >> 32) and counter
 *                   (b, pos, draw / 4, 0), times 2^-24.
 *   theta           device float [K+1] (omega, beta_0..beta_{K-1}) or NULL
 *   draft_stats     device [B][K] statistics from sv_av_score, or NULL: when
 *                   given, draft rows are not re-read for their statistics
 *   out_tokens      device int32 [B][K+1]: accepted drafts, then the
 *                   residual/bonus token, then -1
 *   out_accept_len  device int32 [B]: number of accepted drafts a_b
 *   out_feature     device float [B][K] or NULL: x_i for i < k_b, NaN beyond
 *   out_conf        device float [B][K] or NULL (requires theta): conf_i for
 *                   i < k_b, NaN beyond
 *   workspace       device, >= sv_workspace_bytes(B, K, V), 256-byte aligned
 * Out-of-range drafted tokens set SV_FLAG_TOKEN_RANGE and are rejected.
 * NaN logits set SV_FLAG_NONFINITE; that sequence's outputs are unspecified
 * but in range.
 * Target rows after a sequence's first rejection do not affect any output.
 * When the draft rows are streamed (draft_stats == NULL) they are not read
 * either, apart from rows read ahead of the walk (up to three when the
 * launch streams under 128 MB of first-pass rows, one under 1 GB, none
 * above), whose flags are ignored.
 * ---------------------------------------------------------------------- */
sv_status_t sv_verify(int B, int K, int V, sv_dtype_t dtype,
                      const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const int32_t *draft_len,
                      const float *temperature, uint64_t seed,
                      const float *theta, const sv_row_stats_t *draft_stats,
                      int32_t *out_tokens, int32_t *out_accept_len,
                      float *out_feature, float *out_conf,
                      void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * sv_av_score -- AV scoring of the drafts alone, before the target forward
 * pass ("Adaptive Verification without a confidence head", sections
 * "Background", "Scoring the distribution" and "Other features considered":
 * survival = cumulative product of the confidences).
 *
 *   draft_logits    device [B][K][V]
 *   temperature     device float [B] (0 = greedy: features at tau = 1)
 *   theta           device float [K+1]
 *   keep_threshold  > 0: k_b = number of leading drafts whose survival
 *                   prod_{j<=i} conf_j is >= keep_threshold; <= 0: k_b = K
 *   out_feature     device float [B][K] (x = -ln E, clamped to [-30, 30])
 *   out_conf        device float [B][K]
 *   out_kept_len    device int32 [B] (may be NULL)
 *   out_draft_stats device [B][K] or NULL: statistics to hand to sv_verify
 *   workspace       as for sv_verify
 * ---------------------------------------------------------------------- */
sv_status_t sv_av_score(int B, int K, int V, sv_dtype_t dtype,
                        const void *draft_logits, const float *temperature,
                        const float *theta, float keep_threshold,
                        float *out_feature, float *out_conf, int32_t *out_kept_len,
                        sv_row_stats_t *out_draft_stats,
                        void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * AV refit ("Adaptive Verification without a confidence head", section
 * "Fitting the coefficients").
 *
 * sv_av_state_bytes(K)  size of the refit state (256-byte aligned buffer):
 *   status word, round step counter, and fp64 accumulators of the gradient g
 *   (K+1), the arrow-shaped Hessian (H_ww, H_wb[K], H_bb[K]) and the label
 *   counts n[K].  Zero it once (sv_av_reset) before the first step.
 *
 * sv_av_fit_step -- one decode step of the refit.  Labels are the drafts up
 *   to and including the first rejection: y = 1 for i < accept_len[b], y = 0
 *   at i = accept_len[b] if that is < kept_len[b].  The gradient and Hessian
 *   of the summed log-loss at the current theta are added to the state; on
 *   the round_len-th step of a round the system H * delta = g is solved over
 *   the slope and the intercepts that have labels (ridge 1e-9 * trace(H) /
 *   (K+1) on the diagonal) and theta_j -= n_j / (n_j + damping_c) * delta_j
 *   (n_omega = all labels of the round); then the accumulators are cleared.
 *
 *   theta       device float [K+1], read, and updated at round end
 *   av_state    device, >= sv_av_state_bytes(K)
 *   round_len   N >= 1 decode steps per refit; 0 = accumulate only, never
 *               solve: the caller ends each round with sv_av_solve (the
 *               sharded refit below)
 *   damping_c   constant of the damping n / (n + c), >= 0
 *   feature     device float [B][K] (from sv_verify or sv_av_score)
 *   accept_len  device int32 [B] (from sv_verify)
 *   kept_len    device int32 [B] or NULL (= K)
 * ---------------------------------------------------------------------- */
size_t sv_av_state_bytes(int K);
sv_status_t sv_av_reset(int K, void *av_state, size_t av_state_bytes, void *stream);
sv_status_t sv_av_fit_step(int B, int K, float *theta, void *av_state, size_t av_state_bytes,
                           int round_len, float damping_c,
                           const float *feature, const int32_t *accept_len,
                           const int32_t *kept_len, void *stream);

/* ------------------------------------------------------------------------
 * The refit over a batch sharded across GPUs ("Adaptive Verification without
 * a confidence head", section "Fitting the coefficients": one theta fitted
 * from every label of the round, from gradient and Hessian sums of O(K^2)
 * size).  The sums are additive over sequences, so a batch split over G
 * GPUs reaches the single-GPU round update by one sum all-reduce of the
 * accumulator block before the solve:
 *   1. every GPU runs sv_av_fit_step or sv_verify_fit on its own sequences
 *      with round_len = 0 (accumulate only);
 *   2. at the round's end the caller sums the accumulator block of every
 *      GPU's AV state in place (e.g. ncclAllReduce, ncclFloat64, ncclSum, on
 *      av_state + sv_av_accum_offset(), sv_av_accum_bytes(K) / 8 values);
 *   3. every GPU calls sv_av_solve with the same theta, and all get the same
 *      update (identical fp64 inputs, identical arithmetic).
 * With G = 1 this is exactly the round_len path.  Sums over G shards differ
 * from the single-GPU sums only by the order of fp64 additions.
 *
 * sv_av_accum_offset()  byte offset of the block inside the AV state (a
 *   multiple of 256).
 * sv_av_accum_bytes(K)  its size: 4K + 2 fp64 values, in this order:
 *   g[0] (slope), g[1..K] (intercepts), H_ww, H_wb[K], H_bb[K], n[K]
 *   (H_wb[i] = sum of w x over position i's labels, H_bb[i] = sum of w,
 *   n[i] = label count; w = s (1 - s)).  Returns 0 for K outside [0, 16].
 * sv_av_solve -- end the round now: solve the arrow system from the block as
 *   it stands, update theta as sv_av_fit_step does at a round's end
 *   (damping n / (n + damping_c)), clear the block and the step counter.  A
 *   round without labels leaves theta unchanged.  Asynchronous on `stream`;
 *   SV_FLAG_FIT_SINGULAR in the AV state's status word as for
 *   sv_av_fit_step.
 * ---------------------------------------------------------------------- */
size_t sv_av_accum_offset(void);
size_t sv_av_accum_bytes(int K);
sv_status_t sv_av_solve(int K, float *theta, void *av_state, size_t av_state_bytes, float damping_c,
                        void *stream);

/* ------------------------------------------------------------------------
 * sv_verify_fit -- sv_verify and one sv_av_fit_step in a single launch.
 * Same arguments as sv_verify (theta is required and is updated at the end
 * of a round), plus the refit state of sv_av_fit_step; kept_len is
 * draft_len.  Each sequence's acceptance scan adds its labelled drafts'
 * gradient and Hessian terms (as 2^-32 fixed point, so the sums do not
 * depend on the order of the additions); the scan that finishes last -- after
 * every scan has read theta -- performs the round update exactly as
 * sv_av_fit_step does ("Adaptive Verification without a confidence head",
 * section "Fitting the coefficients").  The results equal sv_verify followed
 * by sv_av_fit_step on the same stream up to the rounding of those sums.
 * ---------------------------------------------------------------------- */
sv_status_t sv_verify_fit(int B, int K, int V, sv_dtype_t dtype,
                          const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const int32_t *draft_len,
                          const float *temperature, uint64_t seed,
                          float *theta, const sv_row_stats_t *draft_stats,
                          int32_t *out_tokens, int32_t *out_accept_len,
                          float *out_feature, float *out_conf,
                          void *av_state, size_t av_state_bytes, int round_len, float damping_c,
                          void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * sv_av_budget -- AV's global draft budget, the step before verification.
 *
 * Defined by "Adaptive Verification without a confidence head", section
 * "Other features considered": drafts are ranked by survival (the running
 * product of the confidences along each request), the estimated number of
 * accepted tokens of a budget of n drafts is n_req plus the n largest
 * survivals, and the budget is the n maximising that estimate divided by the
 * cost of drafting and verifying n tokens; the n best drafts are kept.
 *
 *   conf          device float [B][K]: per-position confidences (sv_av_score
 *                 or sv_verify); survival s[b][i] = fl32 running product in
 *                 position order; NaN survivals are not candidates, values
 *                 at or below 0 count as 0
 *   draft_len     device int32 [B] or NULL: only positions i < draft_len[b]
 *                 are candidates (clamped to [0, K])
 *   n_req         number of sampling requests (est[0])
 *   draft_cost, verify_cost  device float [N + 1] at least (N = number of
 *                 candidates <= B*K): cost of n drafted / verified tokens
 *   out_budget    device int32 [1]: the first n maximising est[n] / cost[n]
 *                 over the n with cost[n] > 0 and a finite ratio (0 if none);
 *                 est[n] sums the ranked survivals in fp64 (ranking: survival
 *                 descending, then b*K + i ascending)
 *   out_kept_len  device int32 [B]: drafts of request b among the n best; they
 *                 are its first out_kept_len[b] positions
 * B*K <= SV_BUDGET_MAX.  One CTA; returns after enqueueing.
 * ---------------------------------------------------------------------- */
#define SV_BUDGET_MAX 16384
sv_status_t sv_av_budget(int B, int K, const float *conf, const int32_t *draft_len, int n_req,
                         const float *draft_cost, const float *verify_cost,
                         int32_t *out_budget, int32_t *out_kept_len, void *stream);

/* ------------------------------------------------------------------------
 * sv_tts_signal -- the test-time-speculation distillation signal on the
 * verified rows.
 *
 * Defined by "Technical summary: Test-Time Speculation (TTS)", section
 * "Algorithm", step 3 "Distillation loss": after verification the drafter
 * takes a gradient step on KL~(p || q) + lambda KL~(q_t || q) over the
 * canvas with position weights w_k; at q = q_t the second term and its
 * gradient vanish.  For request b and canvas position k < K, with
 * p = softmax(target row k / tau_b), q = softmax(draft row k / tau_b)
 * (tau_b <= 0 counts as 1):
 *   out_kl[b][k]      = w_k * sum_v p_v (ln p_v - ln q_v)
 *   out_grad[b][k][v] = w_k * (q_v - p_v) / tau_b     (bf16, round to nearest
 *                       even: the gradient of out_kl with respect to the
 *                       draft logits)
 *
 *   target_logits  device [B][K+1][V] (the sv_verify layout; rows 0..K-1 read)
 *   draft_logits   device [B][K][V]
 *   temperature    device float [B]
 *   weights        device float [K]
 *   out_kl         device float [B][K]
 *   out_grad       device bf16 bits [B][K][V] or NULL (KL only)
 *   workspace      device, >= sv_tts_workspace_bytes(), 256-byte aligned:
 *                  the status word and the exchange between the CTAs that
 *                  share a row pair; calls that share one workspace must be
 *                  ordered (same stream, or events)
 * With 16-byte aligned rows (V * element size a multiple of 16, and V a
 * multiple of 8 when out_grad is given) every row pair is read from HBM
 * once: a group of CTAs holds it in shared memory across both passes.
 * Otherwise one CTA per pair reads it twice (the second time mostly from
 * L2).  The gradient is written once.  A bounded wait that gives up sets
 * SV_FLAG_TIMEOUT in the workspace's status word and the affected out_kl
 * values are NaN.  Returns after enqueueing.
 * ---------------------------------------------------------------------- */
size_t sv_tts_workspace_bytes(void);
sv_status_t sv_tts_signal(int B, int K, int V, sv_dtype_t dtype, const void *target_logits,
                          const void *draft_logits, const float *temperature, const float *weights,
                          float *out_kl, uint16_t *out_grad, void *workspace, size_t workspace_bytes,
                          void *stream);

/* ------------------------------------------------------------------------
 * sv_verify_tree -- verification of a token tree (several draft branches per
 * request) in one call: the acceptance walk only (the target's tree
 * attention mask is the caller's).
 *
 * Defined by "Accelerating Sonar through Speculation", section "EAGLE" (the
 * drafter explores a tree of candidates; the target scores it in one pass;
 * the best-fitting branch is kept and one target token appended), with the
 * rule of the "Speculative Decoding: Draft, EAGLE, MTP" cheatsheet, "one
 * speculative step", applied at every node: at the current node c the
 * children are tried in ascending node order; child j with token x is
 * accepted iff U < p_j(x) / q(x), where p_0 = softmax(target row c / tau),
 * q = softmax(draft row c / tau), and after each rejected child
 * p_{j+1} = max(p_j - q, 0) normalised.  An accepted child becomes the
 * current node; when no child is accepted, or c is a leaf, one token is
 * drawn from the last p_j (smallest v whose cumulative mass exceeds U' times
 * the total) and the walk ends.  Children are assumed drawn independently
 * from the draft distribution at their parent (with replacement), the
 * setting in which this rule is lossless.  Greedy rows (tau <= 0): the first
 * child equal to the target argmax (lowest index on ties) is accepted; else,
 * and at a leaf, the argmax is emitted.
 *
 *   N             nodes per request (1..SV_TREE_MAX_NODES); node 0 is the last
 *                 committed token, node n >= 1 carries tokens[b][n] and has
 *                 parents[b][n] in [0, n)
 *   target_logits device [B][N][V]: row n = the target's next-token logits
 *                 after node n
 *   draft_logits  device [B][N][V]: row n = the draft logits after node n,
 *                 from which node n's children were drawn
 *   n_nodes       device int32 [B] or NULL (= N): nodes in use per request
 *   temperature   device float [B]
 *   seed          Philox4x32-10 key: the test of child j at depth t uses word 0
 *                 of block (b, t, j, 0); the final draw at depth t word 1 of
 *                 block (b, t, 0, 0) -- a chain tree reproduces sv_verify
 *   out_tokens    device int32 [B][N]: emitted tokens, then -1
 *   out_accept_len device int32 [B]: accepted draft tokens (the path depth)
 *   out_path      device int32 [B][max(N-1,1)] or NULL: accepted node indices
 *   out_flags     device uint32 [B] or NULL: SV_TREE_* bits; a request with
 *                 SV_TREE_BAD (a parent outside [0, n), n_nodes outside
 *                 [1, N]) emits nothing (all -1, accept_len 0)
 * One CTA per request; every row read stays in L2 for its later passes.
 * ---------------------------------------------------------------------- */
#define SV_TREE_MAX_NODES 64
#define SV_TREE_ZERO_RESIDUAL (1u << 0) /* a residual had no mass (rounding); the previous p kept */
#define SV_TREE_BAD           (1u << 1)
sv_status_t sv_verify_tree(int B, int N, int V, sv_dtype_t dtype, const void *target_logits,
                           const void *draft_logits, const int32_t *tokens, const int32_t *parents,
                           const int32_t *n_nodes, const float *temperature, uint64_t seed,
                           int32_t *out_tokens, int32_t *out_accept_len, int32_t *out_path,
                           uint32_t *out_flags, void *stream);

/* ------------------------------------------------------------------------
 * sv_post_verify -- the step after verification, on the device, so that the
 * host never waits for the accepted lengths.
 *
 * Defined by "Accelerating Sonar through Speculation", section "MTP schedule
 * for one token" (a kernel shifts the target's input tokens and plugs the
 * target's next token into its position; the draft then re-runs on the same
 * batch layout) and the "Speculative Decoding: Draft, EAGLE, MTP" cheatsheet,
 * "algorithm loop in code" (the key-value cache grows by one entry per
 * accepted draft; at the first rejection it is cut back to the prefix length
 * plus the number of emitted tokens).  For sequence b with a = accept_len[b]
 * and k = draft_len[b] (K when NULL):
 *   next_in[b][j] = out_tokens[b][j]        for j <= a
 *                 = in_tokens[b][j + 1]     for a < j < k  (drafts the next
 *                                           step recomputes and discards)
 *                 = -1                      otherwise
 *   history[b][seq_len[b] + j] = out_tokens[b][j] for j <= a (positions at or
 *                 beyond history_cap are skipped: SV_PV_OVERFLOW)
 *   seq_len[b] += a + 1
 *   kv_len[b]  += a + 1 when a < k (rejection), k when all were accepted
 *                 (the bonus token has no cache entry yet)
 *
 *   in_tokens    device int32 [B][K+1]: the verify input, [t_last, d_0 ..
 *                d_{K-1}]; required when next_in is given
 *   out_tokens   device int32 [B][K+1]: sv_verify's emitted tokens
 *   accept_len   device int32 [B]: sv_verify's accept lengths
 *   draft_len    device int32 [B] or NULL: as given to sv_verify
 *   seq_len, kv_len  device int32 [B], updated in place
 *   history      device int32 [B][history_cap] or NULL, updated in place
 *   next_in      device int32 [B][K+1] or NULL (must not alias in_tokens)
 *   flags        device uint32 [B] or NULL: SV_PV_* bits of each sequence;
 *                a sequence with SV_PV_BAD_INPUT (accept_len outside
 *                [0, k], or out_tokens[b][a] < 0) is left unchanged and its
 *                next_in row is all -1.
 * One warp per sequence; returns after enqueueing.
 * ---------------------------------------------------------------------- */
#define SV_PV_OVERFLOW  (1u << 0)
#define SV_PV_BAD_INPUT (1u << 1)
sv_status_t sv_post_verify(int B, int K, const int32_t *in_tokens, const int32_t *out_tokens,
                           const int32_t *accept_len, const int32_t *draft_len,
                           int32_t *seq_len, int32_t *kv_len, int32_t *history, int history_cap,
                           int32_t *next_in, uint32_t *flags, void *stream);

/* ------------------------------------------------------------------------
 * sv_philox -- the uniform stream itself, for checking: out[b][pos][w] =
 * word w of Philox4x32-10 with key (seed & 0xffffffff, seed >> 32) and
 * counter (b, pos, 0, 0) (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11), for b < nb, pos < npos.
 *   out  device uint32 [nb][npos][4]
 * ---------------------------------------------------------------------- */
sv_status_t sv_philox(uint64_t seed, int nb, int npos, uint32_t *out, void *stream);

/* ------------------------------------------------------------------------
 * sv_status -- synchronise `stream`, read and clear the status word in the
 * first 4 bytes of `status_holder` (a workspace or an AV state).  Returns
 * SV_OK, or the most severe error among the bits that were set (TIMEOUT,
 * NONFINITE, TOKEN_RANGE, BAD_LEN, BAD_TEMP, in that order); the raw bits
 * go to *flags_out when it is not NULL.  The warning bits SV_FLAG_ZERO_RESIDUAL
 * and SV_FLAG_FIT_SINGULAR alone map to SV_OK.
 * ---------------------------------------------------------------------- */
sv_status_t sv_status(void *status_holder, void *stream, uint32_t *flags_out);

/* ------------------------------------------------------------------------
 * sv_verify_noalloc -- sv_verify for callers that cannot allocate device
 * memory.  (This entry point has no counterpart in the pages; it is a
 * deployment convenience.)  Some callers hold no device allocator of their
 * own: a plain C host that only receives pointers to tensors owned by
 * another framework, or a serving runtime that reserves all device memory
 * up front for its KV-cache pool and forbids later cudaMalloc (which can
 * fail under a full pool and synchronises the device).  This entry point
 * takes the same arguments as sv_verify minus the workspace and uses a
 * scratch array of SV_NOALLOC_SCRATCH_BYTES compiled into the library
 * instead; every GPU that loads the library holds that array until the
 * process exits.  It allocates nothing: no cudaMalloc, no cudaFree.
 *  - Shapes needing more than SV_NOALLOC_SCRATCH_BYTES of scratch
 *    (sv_workspace_bytes(B, K, V) > SV_NOALLOC_SCRATCH_BYTES) are rejected
 *    with SV_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (once per device and CUDA context: again after
 *    a device reset has replaced the context); make that first call before
 *    any stream capture.
 *  - All calls share the one array, and the array keeps the last call's
 *    contents (each call clears what must start at zero).  Calls that
 *    overlap on the GPU -- on different streams, or from different host
 *    threads without ordering -- race on it: order them.
 *  - sv_status(sv_noalloc_status_holder(), stream, ...) reads its status
 *    word.
 * ---------------------------------------------------------------------- */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
sv_status_t sv_verify_noalloc(int B, int K, int V, sv_dtype_t dtype,
                              const void *target_logits, const void *draft_logits,
                              const int32_t *draft_tokens, const int32_t *draft_len,
                              const float *temperature, uint64_t seed,
                              const float *theta, const sv_row_stats_t *draft_stats,
                              int32_t *out_tokens, int32_t *out_accept_len,
                              float *out_feature, float *out_conf, void *stream);

/* Device address of the scratch array's status word on the current device
 * and context (looked up as by sv_verify_noalloc; NULL on error). */
void *sv_noalloc_status_holder(void);

/* ------------------------------------------------------------------------
 * sv_set_launch_events -- measurement hook.  For the calling host thread,
 * every later sv_verify / sv_av_score call records `begin_event` on its
 * stream immediately before launching the row-pass kernel (the streaming
 * read of all verified rows) and `end_event` immediately after it, so the
 * caller can time that kernel alone with cudaEventElapsedTime.  Events are
 * cudaEvent_t passed as void*, owned by the caller; NULL, NULL turns the
 * hook off.  Nothing else about the calls changes.
 * ---------------------------------------------------------------------- */
sv_status_t sv_set_launch_events(void *begin_event, void *end_event);

/* ------------------------------------------------------------------------
 * sv_set_wait_test -- a test hook for failure detection (the pages have no
 * counterpart).  Applies to the later sv_verify, sv_verify_fit, sv_av_score
 * and sv_tts_signal calls made from the calling host thread until it is
 * called again:
 *   limit_ns  the limit of every device-side wait of their kernels, in ns
 *             (0 = the default, 2 s);
 *   withhold  nonzero: the kernels' producer warps stage no rows, so the
 *             other warps' first waits can only end by running out (no copy
 *             is ever in flight).  The call then writes no outputs and its
 *             workspace status reports SV_FLAG_TIMEOUT (sv_status returns
 *             SV_ERR_TIMEOUT) once limit_ns has passed; the device stays
 *             usable, and the next call on the same workspace runs normally.
 *             sv_tts_signal (rows held in shared memory, i.e. 16-byte
 *             aligned): no row copy is issued, every out_kl value is NaN and
 *             out_grad is not written; the kernel for other rows has no
 *             waits and ignores the hook.
 * For tests of the time-out path only.  Always returns SV_OK.
 * ---------------------------------------------------------------------- */
sv_status_t sv_set_wait_test(uint64_t limit_ns, int withhold);

/* Static description of a status code; never NULL. */
const char *sv_strerror(sv_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
