// AV global draft budget ("Adaptive Verification without a confidence
// head", section "Other features considered"): rank every draft by its
// survival probability (running product of the confidences along its
// request), estimate the accepted tokens of a budget of n drafts as the
// number of requests plus the n largest survivals, and keep the n that
// maximises estimate / (draft cost + verify cost).  One CTA: survivals and
// 64-bit sort keys in shared memory, a bitonic sort, a double-float block
// scan of the ranked survivals, an argmax (coarse in fp32, exact in fp64
// near the maximum), and per-request kept counts.
#include <cfloat>

#include "sample_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kBudgetThreads = 1024;
constexpr int kBudgetWarps = kBudgetThreads / 32;

struct BudgetParams {
  int B, K, n_req, npad;
  const float *conf;
  const int32_t *draft_len;
  const float *draft_cost, *verify_cost;
  int32_t *out_budget, *out_kept;
};

// Key of a candidate: survival descending (its fp32 bits, non-negative, so
// the bit pattern orders like the value), then flat index ascending.
// Non-candidates get the largest key.
__device__ __forceinline__ uint64_t budget_key(float s, int idx) {
  const uint32_t bits = s > 0.f ? __float_as_uint(s) : 0u;
  return ((uint64_t)(0xffffffffu - bits) << 32) | (uint32_t)idx;
}
__device__ __forceinline__ float key_survival(uint64_t key) {
  return __uint_as_float(0xffffffffu - (uint32_t)(key >> 32));
}

// Bitonic sort of npad = 1024 E keys in shared memory (ascending), E keys
// per thread in registers (thread t holds keys t E .. t E + E - 1).
template <int E>
__device__ void bitonic_sort(uint64_t *keys, int npad) {
  const int tid = threadIdx.x;
  uint64_t r[E];
#pragma unroll
  for (int e = 0; e < E; ++e) r[e] = keys[tid * E + e];
  for (int size = 2; size <= npad; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * E) {  // partners in other warps: through shared memory
#pragma unroll
      for (int e = 0; e < E; ++e) keys[tid * E + e] = r[e];
      __syncthreads();
      for (; stride >= 32 * E; stride >>= 1) {
        const int sh = __ffs(stride) - 1;
        for (int q = tid; q < (npad >> 1); q += kBudgetThreads) {
          const int lo = ((q >> sh) << (sh + 1)) + (q & (stride - 1)), hi = lo + stride;
          const bool up = (lo & size) == 0;
          const uint64_t x = keys[lo], y = keys[hi];
          if ((x > y) == up) {
            keys[lo] = y;
            keys[hi] = x;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < E; ++e) r[e] = keys[tid * E + e];
    }
    for (; stride >= E; stride >>= 1) {  // partners in the same warp: shuffles
      const int lm = stride / E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, r[e], lm);
        const int i = tid * E + e;
        const bool keep_min = ((i & stride) == 0) == ((i & size) == 0);
        r[e] = keep_min ? (o < r[e] ? o : r[e]) : (o > r[e] ? o : r[e]);
      }
    }
#pragma unroll
    for (int st = E / 2; st >= 1; st >>= 1) {  // partners in the same thread
      if (st <= stride) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & st) continue;
          const bool up = ((tid * E + e) & size) == 0;
          if ((r[e] > r[e + st]) == up) {
            const uint64_t t = r[e];
            r[e] = r[e + st];
            r[e + st] = t;
          }
        }
      }
    }
  }
  __syncthreads();  // every thread is done reading keys before they are rewritten
#pragma unroll
  for (int e = 0; e < E; ++e) keys[tid * E + e] = r[e];
  __syncthreads();
}

__global__ void __launch_bounds__(kBudgetThreads, 1) av_budget_kernel(const BudgetParams P) {
  extern __shared__ uint64_t keys[];
  __shared__ float s_whi[kBudgetWarps], s_wlo[kBudgetWarps], s_bf[kBudgetWarps];
  __shared__ double s_bratio[kBudgetWarps];
  __shared__ int s_bn[kBudgetWarps];
  __shared__ int s_ncand;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, K = P.K, NK = B * K, npad = P.npad;

  float *cf = reinterpret_cast<float *>(keys + npad);  // the confidences, staged
  if (tid == 0) s_ncand = 0;
  for (int b = tid; b < B; b += kBudgetThreads) P.out_kept[b] = 0;
  for (int j = tid; j < NK; j += kBudgetThreads) cf[j] = __ldg(P.conf + j);  // coalesced
  __syncthreads();
  // 1. survivals (fp32 running product in position order) and keys
  for (int b = tid; b < B; b += kBudgetThreads) {
    int k = P.draft_len ? __ldg(P.draft_len + b) : K;
    k = k < 0 ? 0 : (k > K ? K : k);
    float run = 1.f;
    for (int i = 0; i < K; ++i) {
      run = __fmul_rn(run, cf[b * K + i]);
      const bool cand = i < k && !isnan(run);
      keys[b * K + i] = cand ? budget_key(run, b * K + i) : ~0ull;
    }
  }
  for (int j = NK + tid; j < npad; j += kBudgetThreads) keys[j] = ~0ull;
  __syncthreads();

  // 2. bitonic sort, ascending keys: each thread holds npad / 1024 keys in
  //    registers; strides below that stay in registers, strides up to 32x
  //    that go through warp shuffles, larger ones through shared memory
  switch (npad >> 10) {
    case 2: bitonic_sort<2>(keys, npad); break;
    case 4: bitonic_sort<4>(keys, npad); break;
    case 8: bitonic_sort<8>(keys, npad); break;
    default: bitonic_sort<16>(keys, npad); break;
  }

  // 3. number of candidates: the first non-candidate key
  for (int j = tid; j < npad; j += kBudgetThreads)
    if (keys[j] != ~0ull && (j + 1 == npad || keys[j + 1] == ~0ull)) s_ncand = j + 1;
  __syncthreads();
  const int N = s_ncand;

  // 4. est[n] = n_req + sum of the n first ranked survivals, as double-float
  //    (two fp32 numbers, ~48 bits; fp64 runs at a small fraction of the fp32
  //    rate on this GPU): each thread a contiguous segment, block scan
  const int per = (N + kBudgetThreads - 1) / kBudgetThreads;
  const int j0 = min(N, tid * per), j1 = min(N, j0 + per);
  DF seg = {0.f, 0.f};
  for (int j = j0; j < j1; ++j) seg = df_add_f(seg, key_survival(keys[j]));
  const DF incl = warp_incl_scan_df(seg, lane);
  if (lane == 31) {
    s_whi[warp] = incl.hi;
    s_wlo[warp] = incl.lo;
  }
  __syncthreads();
  if (warp == 0) {
    const DF w = warp_incl_scan_df(DF{s_whi[lane], s_wlo[lane]}, lane);
    s_whi[lane] = w.hi;
    s_wlo[lane] = w.lo;
  }
  __syncthreads();
  DF start = DF{(float)P.n_req, 0.f};  // exact for n_req < 2^24
  if (warp > 0) start = df_add(start, DF{s_whi[warp - 1], s_wlo[warp - 1]});
  start = df_add(start, df_add(incl, DF{-seg.hi, -seg.lo}));  // + this warp's exclusive prefix

  // 5. the first n maximising est[n] / cost[n] over the n with cost > 0:
  //    a coarse fp32 maximum first, then every n within rounding of it
  //    compared exactly in fp64 (a handful of divisions instead of N)
  float bestf = -FLT_MAX;
  {
    DF run = start;
    if (tid == 0) {
      const float cf = __ldg(P.draft_cost) + __ldg(P.verify_cost);
      if (cf > 0.f && isfinite((float)P.n_req / cf)) bestf = (float)P.n_req / cf;
    }
    for (int j = j0; j < j1; ++j) {
      run = df_add_f(run, key_survival(keys[j]));
      const float cf = __ldg(P.draft_cost + j + 1) + __ldg(P.verify_cost + j + 1);
      const float r = run.hi / cf;
      if (cf > 0.f && isfinite(r) && r > bestf) bestf = r;
    }
  }
  bestf = warp_max(bestf);
  if (lane == 0) s_bf[warp] = bestf;
  __syncthreads();
  bestf = s_bf[0];
  for (int w = 1; w < kBudgetWarps; ++w) bestf = fmaxf(bestf, s_bf[w]);
  const float thr = bestf - fabsf(bestf) * 1e-6f;  // fp32 ratios are within ~3 ulps
  double best = -DBL_MAX;
  int bn = INT_MAX;
  auto consider = [&](int n, const DF &est, float rf) {
    if (!(rf >= thr)) return;
    const double cost = (double)__ldg(P.draft_cost + n) + (double)__ldg(P.verify_cost + n);
    if (!(cost > 0.0)) return;
    const double r = ((double)est.hi + (double)est.lo) / cost;
    if (isfinite(r) && (r > best || (r == best && n < bn))) {
      best = r;
      bn = n;
    }
  };
  {
    DF run = start;
    if (tid == 0) {
      const float cf = __ldg(P.draft_cost) + __ldg(P.verify_cost);
      consider(0, DF{(float)P.n_req, 0.f}, (float)P.n_req / cf);
    }
    for (int j = j0; j < j1; ++j) {
      run = df_add_f(run, key_survival(keys[j]));
      const float cf = __ldg(P.draft_cost + j + 1) + __ldg(P.verify_cost + j + 1);
      consider(j + 1, run, run.hi / cf);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int on = __shfl_xor_sync(0xffffffffu, bn, o);
    if (ob > best || (ob == best && on < bn)) {
      best = ob;
      bn = on;
    }
  }
  if (lane == 0) {
    s_bratio[warp] = best;
    s_bn[warp] = bn;
  }
  __syncthreads();
  if (warp == 0) {
    best = lane < kBudgetWarps ? s_bratio[lane] : -DBL_MAX;
    bn = lane < kBudgetWarps ? s_bn[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int on = __shfl_xor_sync(0xffffffffu, bn, o);
      if (ob > best || (ob == best && on < bn)) {
        best = ob;
        bn = on;
      }
    }
    if (lane == 0) s_bn[0] = bn == INT_MAX ? 0 : bn;
  }
  __syncthreads();
  const int budget = s_bn[0];
  if (tid == 0) P.out_budget[0] = budget;
  // 6. kept drafts per request
  for (int j = tid; j < budget; j += kBudgetThreads) atomicAdd(P.out_kept + (int)(uint32_t)keys[j] / K, 1);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status_t sv_av_budget(int B, int K, const float *conf, const int32_t *draft_len, int n_req,
                                    const float *draft_cost, const float *verify_cost, int32_t *out_budget,
                                    int32_t *out_kept_len, void *stream) {
  if (B < 0 || K < 0 || K > SV_MAX_K || (long long)B * K > SV_BUDGET_MAX) return SV_ERR_INVALID;
  if (!out_budget || !out_kept_len || !draft_cost || !verify_cost || (B * K > 0 && !conf)) return SV_ERR_INVALID;
  const void *ptrs[] = {conf, draft_len, draft_cost, verify_cost, out_budget, out_kept_len};
  for (const void *p : ptrs)
    if (!host_aligned(p, 4)) return SV_ERR_INVALID;
  int sms = 0;
  const sv_status_t ds = host_device_info(&sms);
  if (ds != SV_OK) return ds;
  int npad = 2048;  // at least two keys per thread of the sort
  while (npad < B * K) npad <<= 1;
  const size_t smem = (size_t)npad * sizeof(uint64_t) + (size_t)B * K * sizeof(float);
  const cudaError_t e = cudaFuncSetAttribute(av_budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(SV_BUDGET_MAX * (sizeof(uint64_t) + sizeof(float))));
  if (e != cudaSuccess) return SV_ERR_CUDA;
  BudgetParams P{B, K, n_req, npad, conf, draft_len, draft_cost, verify_cost, out_budget, out_kept_len};
  av_budget_kernel<<<1, kBudgetThreads, smem, static_cast<cudaStream_t>(stream)>>>(P);
  return host_cuda_status(cudaGetLastError());
}
