// AV global draft budget ("Adaptive Verification without a confidence head",
// section "Other features considered"): rank every draft by its survival
// probability (running product of the confidences along its request),
// estimate the accepted tokens of a budget of n drafts as the number of
// requests plus the n largest survivals, and keep the n that maximises
// estimate / (draft cost + verify cost).
//
// One CTA of 1024 threads, everything in shared memory:
//   1. confidences staged with an odd row stride (conflict-free per-request
//      reads), survivals as fp32 running products, one thread per request;
//   2. a sort of 32-bit keys (survival descending; the prefix sums need only
//      the values, so no index rides along): every warp sorts its 32 E keys
//      with a bitonic network in registers and shuffles, then five rounds of
//      merge path join the 32 runs;
//   3. a double-float block scan of the ranked survivals and the argmax of
//      est / cost: coarse in fp32 over the staged cost table, then the few n
//      within rounding of the maximum compared exactly in fp64;
//   4. kept counts per request: drafts above the budget's last survival, plus
//      the ties at that value in flat-index order (a block scan of tie counts).
#include <cfloat>

#include "sample_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kBudgetThreads = 1024;
constexpr int kBudgetWarps = kBudgetThreads / 32;
constexpr uint32_t kNonCand = 0xffffffffu;  // sorts after every candidate
constexpr uint32_t kInfBits = 0x7f800000u;  // bits of +inf

struct BudgetParams {
  int B, K, n_req, npad, stride;  // stride: row stride of the staged confidences (K, or K rounded up to odd)
  const float *conf;
  const int32_t *draft_len;
  const float *draft_cost, *verify_cost;
  int32_t *out_budget, *out_kept;
};

// Key of a candidate: ascending key = descending survival.  A survival at or
// below 0 counts as 0; non-negative fp32 bit patterns order like the values,
// and +inf (the largest) maps to 0.  Non-candidates take kNonCand.
__device__ __forceinline__ uint32_t budget_key(float s) {
  return kInfBits - (s > 0.f ? __float_as_uint(s) : 0u);
}
__device__ __forceinline__ float key_survival(uint32_t key) { return __uint_as_float(kInfBits - key); }

// With 16 keys per thread the sort's buffers hold rank i at word i + i / 32:
// in a merge round the lanes of a warp read positions about 8 apart, which
// without the padding word would put lanes 4 apart in one bank, and a
// thread's 16 ranks never straddle a padding word.  With fewer keys per
// thread the padding's address arithmetic cost more than the conflicts it
// removes (measured), so ranks sit at their own index.
template <int E>
__device__ __forceinline__ int padded(int i) {
  return E >= 16 ? i + (i >> 5) : i;
}
__host__ __device__ constexpr int padded_words(int npad) {  // npad = 1024 E
  return npad >= 16 * 1024 ? npad + npad / 32 : npad;
}

template <int E>
__device__ __forceinline__ void store_blocked(const uint32_t (&r)[E], uint32_t *p) {
  if constexpr (E >= 16) {
    uint32_t *q = p + padded<E>(threadIdx.x * E);
#pragma unroll
    for (int e = 0; e < E; ++e) q[e] = r[e];
  } else if constexpr (E % 4 == 0) {
#pragma unroll
    for (int v = 0; v < E / 4; ++v)
      reinterpret_cast<uint4 *>(p + threadIdx.x * E)[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
  } else {
#pragma unroll
    for (int v = 0; v < E / 2; ++v) reinterpret_cast<uint2 *>(p + threadIdx.x * E)[v] = make_uint2(r[2 * v], r[2 * v + 1]);
  }
}
template <int W>
__device__ __forceinline__ void load_words(const uint32_t *p, uint32_t (&c)[W]) {
  static_assert(W == 4 || W == 2, "four or two words");
  if constexpr (W == 4) {
    const uint4 x = *reinterpret_cast<const uint4 *>(p);
    c[0] = x.x;
    c[1] = x.y;
    c[2] = x.z;
    c[3] = x.w;
  } else {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    c[0] = x.x;
    c[1] = x.y;
  }
}

// Ascending sort of npad = 1024 E keys.  On entry r[] holds this thread's E
// keys (any order); on exit thread t holds ranks t E .. t E + E - 1 in r[]
// and keys[] the sorted array, rank i at padded<E>(i).  tmp: padded_words(npad)
// words of scratch.
//   (a) every warp sorts the 32 E keys of its threads: a bitonic network,
//       strides below E inside a thread, strides E .. 16 E through shuffles;
//   (b) merge path, runs of 32 E doubling to npad (five rounds): thread t
//       writes outputs t E .. t E + E - 1 of its pair of runs, finding where
//       they start by a binary search along the diagonal, then merging E
//       steps.
template <int E>
__device__ void block_sort(uint32_t (&r)[E], uint32_t *keys, uint32_t *tmp) {
  const int tid = threadIdx.x, i0 = tid * E;
  for (int size = 2; size <= 32 * E; size <<= 1) {
    const int dir = size == 32 * E ? 0 : size;  // the last merge runs ascending in every warp
    for (int stride = size >> 1; stride >= E; stride >>= 1) {
      const int lm = stride / E;
      // the direction is the same for all of a thread's keys (stride >= E
      // leaves the low bits of the rank alone)
      const bool keep_min = ((i0 & stride) == 0) == ((i0 & dir) == 0);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, r[e], lm);
        r[e] = keep_min ? min(o, r[e]) : max(o, r[e]);
      }
    }
#pragma unroll
    for (int st = E / 2; st >= 1; st >>= 1) {
      if (st < size) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & st) continue;
          const bool up = ((i0 + e) & dir) == 0;
          const uint32_t mn = min(r[e], r[e + st]), mx = max(r[e], r[e + st]);
          r[e] = up ? mn : mx;
          r[e + st] = up ? mx : mn;
        }
      }
    }
  }
  // five rounds: tmp -> keys -> tmp -> keys -> tmp -> keys
  const int npad = kBudgetThreads * E;
  uint32_t *src = tmp, *dst = keys;
  store_blocked(r, src);
  __syncthreads();
  for (int L = 32 * E; L < npad; L <<= 1) {
    const int base = i0 & ~(2 * L - 1), diag = i0 - base;
    const int a0 = base, b0 = base + L;  // the two runs: ranks a0 .. a0 + L - 1, b0 .. b0 + L - 1
    int lo = diag > L ? diag - L : 0, hi = diag < L ? diag : L;
    while (lo < hi) {  // i = how many of the first diag outputs come from A
      const int mid = (lo + hi) >> 1;
      if (src[padded<E>(a0 + mid)] <= src[padded<E>(b0 + diag - 1 - mid)]) lo = mid + 1;
      else hi = mid;
    }
    int i = lo, j = diag - lo;
    uint32_t a = i < L ? src[padded<E>(a0 + i)] : 0u, b = j < L ? src[padded<E>(b0 + j)] : 0u;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool take_a = i < L && (j >= L || a <= b);
      r[e] = take_a ? a : b;
      if (take_a) {
        ++i;
        a = i < L ? src[padded<E>(a0 + i)] : 0u;
      } else {
        ++j;
        b = j < L ? src[padded<E>(b0 + j)] : 0u;
      }
    }
    store_blocked(r, dst);
    __syncthreads();
    uint32_t *t = src;
    src = dst;
    dst = t;
  }
}

// Exclusive scan of one value per thread over the block, in thread order,
// and the block's total (two barriers; s_w holds kBudgetWarps words).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *s_w, uint32_t &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  uint32_t t = s_w[lane];  // kBudgetWarps == 32: lane w holds warp w's total
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, t, o);
    if (lane >= o) t += n;
  }
  const uint32_t before = __shfl_sync(0xffffffffu, t - s_w[lane], warp);  // warps before this one
  total = __shfl_sync(0xffffffffu, t, 31);
  __syncthreads();  // s_w is free again
  return before + x - v;
}

// (q, n) beats (best, bn) when its ratio is larger, or equal with a smaller
// n; bn == INT_MAX marks "none yet" (no fp64 compare against a sentinel).
__device__ __forceinline__ void take_better(double q, int n, double &best, int &bn) {
  if (n != INT_MAX && (bn == INT_MAX || q > best || (q == best && n < bn))) {
    best = q;
    bn = n;
  }
}
// The best of a warp's candidates, visiting only the lanes that hold one
// (usually none or one: fp64 is slow on this GPU).
__device__ __forceinline__ void warp_best(double &best, int &bn) {
  unsigned m = __ballot_sync(0xffffffffu, bn != INT_MAX);
  double wb = 0.0;
  int wn = INT_MAX;
  while (m) {
    const int l = __ffs(m) - 1;
    m &= m - 1;
    take_better(__shfl_sync(0xffffffffu, best, l), __shfl_sync(0xffffffffu, bn, l), wb, wn);
  }
  best = wb;
  bn = wn;
}

template <int E>
__global__ void __launch_bounds__(kBudgetThreads, 1) av_budget_kernel(const BudgetParams P) {
  extern __shared__ __align__(16) uint32_t smem[];
  __shared__ float s_whi[kBudgetWarps], s_wlo[kBudgetWarps], s_bf[kBudgetWarps];
  __shared__ double s_bratio[kBudgetWarps];
  __shared__ int s_bn[kBudgetWarps];
  __shared__ uint32_t s_w[kBudgetWarps];
  __shared__ int s_ncand;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, K = P.K, NK = B * K, npad = P.npad, S = P.stride;

  const int nw = padded_words(npad);
  uint32_t *keys = smem;                          // [nw] sort input, then the ranked keys (rank i at padded<E>(i))
  uint32_t *tmp = smem + nw;                      // [nw] the sort's scratch, then
  float *costr = reinterpret_cast<float *>(tmp);  //      the cost of n = rank + 1 drafts (unpadded)
  uint32_t *cfk = smem + 2 * nw;                  // [B][S] confidences, then the keys by (b, i)

  if (tid == 0) s_ncand = 0;
  for (int j = tid; j < NK; j += kBudgetThreads) {  // coalesced reads
    const int b = j / K;
    cfk[b * S + (j - b * K)] = __float_as_uint(__ldg(P.conf + j));
  }
  for (int j = NK + tid; j < npad; j += kBudgetThreads) keys[j] = kNonCand;
  __syncthreads();

  // 1. survivals (fp32 running product in position order); the sort's input
  //    is position-major, any order will do
  int ncand = 0;
  for (int b = tid; b < B; b += kBudgetThreads) {
    int k = P.draft_len ? __ldg(P.draft_len + b) : K;
    k = k < 0 ? 0 : (k > K ? K : k);
    float run = 1.f;
    for (int i = 0; i < K; ++i) {
      run = __fmul_rn(run, __uint_as_float(cfk[b * S + i]));
      const bool cand = i < k && !isnan(run);
      const uint32_t key = cand ? budget_key(run) : kNonCand;
      cfk[b * S + i] = key;
      keys[i * B + b] = key;
      ncand += cand;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ncand += __shfl_xor_sync(0xffffffffu, ncand, o);
  if (lane == 0 && ncand) atomicAdd(&s_ncand, ncand);
  __syncthreads();
  const int N = s_ncand;
  // the cost table: N + 1 entries (the caller's arrays may be no longer).
  // Up to 8 per thread are fetched (coalesced) before the sort and land while
  // it runs; they are stored after it, as the table shares the sort's scratch.
  constexpr bool kEarlyCost = E <= 8;
  float dpre[kEarlyCost ? E : 1], vpre[kEarlyCost ? E : 1];
  if constexpr (kEarlyCost) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int j = tid + e * kBudgetThreads;
      dpre[e] = j < N ? __ldg(P.draft_cost + j + 1) : 0.f;
      vpre[e] = j < N ? __ldg(P.verify_cost + j + 1) : 0.f;
    }
  }

  // 2. the ranking
  uint32_t r[E];
  {
    constexpr int W = E % 4 == 0 ? 4 : 2;  // words per vector load
    uint32_t c[W];
#pragma unroll
    for (int v = 0; v < E / W; ++v) {
      load_words(keys + tid * E + v * W, c);
#pragma unroll
      for (int u = 0; u < W; ++u) r[v * W + u] = c[u];
    }
  }
  block_sort<E>(r, keys, tmp);  // ends with a barrier: tmp[] is free again
  if constexpr (kEarlyCost) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int j = tid + e * kBudgetThreads;
      if (j < N) costr[j] = dpre[e] + vpre[e];
    }
  } else {
    for (int j = tid; j < N; j += kBudgetThreads) costr[j] = __ldg(P.draft_cost + j + 1) + __ldg(P.verify_cost + j + 1);
  }
  // (the scan's barriers below make costr[] visible before it is read)

  // 3. est[n] = n_req + sum of the n first ranked survivals, as double-float
  //    (two fp32 numbers, ~48 bits; fp64 runs at a small fraction of the fp32
  //    rate on this GPU): thread t holds ranks t E .. t E + E - 1
  const int j0 = tid * E;
  DF seg = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (j0 + e < N) seg = df_add_f(seg, key_survival(r[e]));
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

  // 4. the first n maximising est[n] / cost[n] over the n with cost > 0: a
  //    coarse fp32 maximum first, then every n within rounding of it compared
  //    exactly in fp64
  constexpr int kCw = E % 4 == 0 ? 4 : 2;  // staged costs per vector load
  const float cost0 = __ldg(P.draft_cost) + __ldg(P.verify_cost);
  const float q0 = (float)P.n_req / cost0;
  float bestf = -FLT_MAX;
  {
    if (tid == 0 && cost0 > 0.f && isfinite(q0)) bestf = q0;
    DF run = start;
#pragma unroll
    for (int v = 0; v < E / kCw; ++v) {
      uint32_t c[kCw];
      load_words(reinterpret_cast<const uint32_t *>(costr) + j0 + v * kCw, c);
#pragma unroll
      for (int u = 0; u < kCw; ++u) {
        const int e = v * kCw + u;
        if (j0 + e < N) {
          run = df_add_f(run, key_survival(r[e]));
          const float cf = __uint_as_float(c[u]);
          const float q = run.hi / cf;
          if (cf > 0.f && isfinite(q) && q > bestf) bestf = q;
        }
      }
    }
  }
  bestf = warp_max(bestf);
  if (lane == 0) s_bf[warp] = bestf;
  __syncthreads();
  bestf = warp_max(s_bf[lane]);  // kBudgetWarps == 32
  const float thr = bestf - fabsf(bestf) * 1e-6f;  // fp32 ratios are within ~3 ulps
  double best = 0.0;
  int bn = INT_MAX;
  auto consider = [&](int n, const DF &est) {
    const double cost = (double)__ldg(P.draft_cost + n) + (double)__ldg(P.verify_cost + n);
    if (!(cost > 0.0)) return;
    const double q = ((double)est.hi + (double)est.lo) / cost;
    if (isfinite(q)) take_better(q, n, best, bn);
  };
  {
    if (tid == 0 && q0 >= thr) consider(0, DF{(float)P.n_req, 0.f});
    DF run = start;
#pragma unroll
    for (int v = 0; v < E / kCw; ++v) {
      uint32_t c[kCw];
      load_words(reinterpret_cast<const uint32_t *>(costr) + j0 + v * kCw, c);
#pragma unroll
      for (int u = 0; u < kCw; ++u) {
        const int e = v * kCw + u;
        if (j0 + e < N) {
          run = df_add_f(run, key_survival(r[e]));
          if (run.hi / __uint_as_float(c[u]) >= thr) consider(j0 + e + 1, run);
        }
      }
    }
  }
  warp_best(best, bn);
  if (lane == 0) {
    s_bratio[warp] = best;
    s_bn[warp] = bn;
  }
  __syncthreads();
  if (warp == 0) {
    best = s_bratio[lane];
    bn = s_bn[lane];
    warp_best(best, bn);
    if (lane == 0) s_bn[0] = bn == INT_MAX ? 0 : bn;
  }
  __syncthreads();
  const int budget = s_bn[0];
  if (tid == 0) P.out_budget[0] = budget;

  // 5. kept drafts per request.  The n best are every draft whose key is
  //    below kth (the budget's last ranked key) and the first `need` drafts
  //    with key == kth in flat-index order (b K + i: request-major).
  uint32_t kth = 0;
  int need = 0;
  if (budget > 0) {
    kth = keys[padded<E>(budget - 1)];
    int lo = 0, hi = budget - 1;  // first rank holding kth
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (keys[padded<E>(mid)] < kth) lo = mid + 1;
      else hi = mid;
    }
    need = budget - lo;
  }
  int carry = 0;  // ties in the requests of earlier rows
  for (int b0 = 0; b0 < B; b0 += kBudgetThreads) {
    const int b = b0 + tid;
    int lt = 0, eq = 0;
    if (b < B) {
      for (int i = 0; i < K; ++i) {
        const uint32_t key = cfk[b * S + i];
        lt += key < kth;
        eq += key == kth;
      }
    }
    uint32_t total;
    const int before = carry + (int)block_excl_scan((uint32_t)eq, s_w, total);
    if (b < B) P.out_kept[b] = lt + min(max(need - before, 0), eq);
    carry += (int)total;
  }
}

template <int E>
sv_status_t launch_budget(const BudgetParams &P, size_t smem, cudaStream_t stream) {
  const cudaError_t e = cudaFuncSetAttribute(av_budget_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  av_budget_kernel<E><<<1, kBudgetThreads, smem, stream>>>(P);
  return host_cuda_status(cudaGetLastError());
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
  // staged confidences: an odd row stride where it fits (conflict-free reads
  // of one position across requests); K == 0: no candidates and no staged
  // rows (B may then be any size)
  const size_t kSmemCap = 227 * 1024 - 1024;  // the opt-in limit less the kernel's static arrays
  const size_t sort_words = 2 * (size_t)padded_words(npad);
  int stride = K == 0 ? 0 : (K | 1);
  if ((sort_words + (size_t)B * stride) * sizeof(uint32_t) > kSmemCap) stride = K;
  const size_t smem = (sort_words + (size_t)B * stride) * sizeof(uint32_t);
  const BudgetParams P{B, K, n_req, npad, stride, conf, draft_len, draft_cost, verify_cost, out_budget, out_kept_len};
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (npad >> 10) {
    case 2: return launch_budget<2>(P, smem, st);
    case 4: return launch_budget<4>(P, smem, st);
    case 8: return launch_budget<8>(P, smem, st);
    default: return launch_budget<16>(P, smem, st);
  }
}
