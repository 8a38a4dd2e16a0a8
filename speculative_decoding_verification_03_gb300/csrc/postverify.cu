// Post-verification update on the device: the next draft input row (shifted
// target input with the target's token plugged in), the token history, and
// the sequence and key-value cache lengths -- so that the host needs no
// synchronisation on the accepted lengths ("Accelerating Sonar through
// Speculation", "MTP schedule for one token"; cache bookkeeping as in the
// "Speculative Decoding: Draft, EAGLE, MTP" cheatsheet, "algorithm loop in
// code").  One warp per sequence; lanes cover the K + 1 slots.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

struct PostParams {
  int B, K, history_cap;
  const int32_t *in_tokens, *out_tokens, *accept_len, *draft_len;
  int32_t *seq_len, *kv_len, *history, *next_in;
  uint32_t *flags;
};

__global__ void post_verify_kernel(const PostParams P) {
  const int lane = threadIdx.x & 31;
  const int b = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  if (b >= P.B) return;
  const int K = P.K, K1 = K + 1;
  int k = P.draft_len ? __ldg(P.draft_len + b) : K;
  k = k < 0 ? 0 : (k > K ? K : k);
  const int a = __ldg(P.accept_len + b);
  const int32_t *out = P.out_tokens + (size_t)b * K1;
  const bool ok = a >= 0 && a <= k && __ldg(out + (a >= 0 && a <= K ? a : 0)) >= 0;
  uint32_t fl = ok ? 0u : SV_PV_BAD_INPUT;
  if (ok) {
    const int32_t sl = __ldg(P.seq_len + b);
    for (int j = lane; j < K1; j += 32) {
      if (P.next_in) {
        int32_t v = -1;
        if (j <= a) v = __ldg(out + j);
        else if (j < k) v = __ldg(P.in_tokens + (size_t)b * K1 + j + 1);
        P.next_in[(size_t)b * K1 + j] = v;
      }
      if (P.history && j <= a) {
        const long long pos = (long long)sl + j;
        if (pos >= 0 && pos < P.history_cap) P.history[(size_t)b * P.history_cap + pos] = __ldg(out + j);
        else fl |= SV_PV_OVERFLOW;
      }
    }
    // all lanes have read seq_len before lane 0 rewrites it
    __syncwarp();
    if (lane == 0) {
      P.seq_len[b] = sl + a + 1;
      P.kv_len[b] = P.kv_len[b] + (a < k ? a + 1 : k);
    }
  } else if (P.next_in) {
    for (int j = lane; j < K1; j += 32) P.next_in[(size_t)b * K1 + j] = -1;
  }
  fl = __reduce_or_sync(0xffffffffu, fl);
  if (lane == 0 && P.flags) P.flags[b] = fl;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status_t sv_post_verify(int B, int K, const int32_t *in_tokens, const int32_t *out_tokens,
                                      const int32_t *accept_len, const int32_t *draft_len, int32_t *seq_len,
                                      int32_t *kv_len, int32_t *history, int history_cap, int32_t *next_in,
                                      uint32_t *flags, void *stream) {
  if (B < 0 || B > (1 << 20) || K < 0 || K > SV_MAX_K || history_cap < 0) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!out_tokens || !accept_len || !seq_len || !kv_len) return SV_ERR_INVALID;
  if (next_in && (!in_tokens || next_in == in_tokens)) return SV_ERR_INVALID;
  if (history && history_cap == 0) return SV_ERR_INVALID;
  const void *ptrs[] = {in_tokens, out_tokens, accept_len, draft_len, seq_len, kv_len, history, next_in, flags};
  for (const void *p : ptrs)
    if (!host_aligned(p, 4)) return SV_ERR_INVALID;
  int sms = 0;
  const sv_status_t ds = host_device_info(&sms);
  if (ds != SV_OK) return ds;
  PostParams P{B, K, history_cap, in_tokens, out_tokens, accept_len, draft_len,
               seq_len, kv_len, history, next_in, flags};
  const int threads = 256;
  const long long warps = B;
  const int grid = (int)((warps * 32 + threads - 1) / threads);
  post_verify_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(P);
  return host_cuda_status(cudaGetLastError());
}
