// Test-time speculation (TTS) distillation signal ("Technical summary:
// Test-Time Speculation (TTS)", section "Algorithm", step 3): for every
// canvas position k of request b, with p = softmax(z_target / tau) and
// q = softmax(z_draft / tau),
//   kl[b][k]      = w_k * KL(p || q)
//   grad[b][k][v] = w_k * (q_v - p_v) / tau        (bf16; the gradient of
//                   that term with respect to the draft logits)
// Two passes over each row pair: the rows' (max, sum) statistics, then the
// per-element KL terms and the gradient.  tts_group_kernel (16-byte aligned
// rows) holds each pair in the shared memory of a group of CTAs across both
// passes, so every row is read from HBM once; tts_kernel (any alignment) runs
// one CTA per pair and re-reads the pair from L2 in the second pass.  KL is
// summed as p (e^-d - 1 + d) with d = ln p - ln q, a sum of non-negative
// terms taken by a short series for small |d|, so it keeps its relative
// precision when q is close to p.
#include <atomic>
#include <cfloat>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTtsThreads = 256;
constexpr int kTtsWarps = kTtsThreads / 32;
constexpr int kTtsUnroll = 4;

struct TtsParams {
  int B, K, V, dtype;
  const void *target;  // [B][K+1][V]
  const void *draft;   // [B][K][V]
  const float *temperature;
  const float *weights;
  float *out_kl;
  uint16_t *out_grad;  // [B][K][V] bf16 or null
};

template <int kDtype>
struct TtsElems;
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <>
struct TtsElems<SV_BF16> {
  static constexpr int kPer = 8;
  __device__ __forceinline__ static float get(const uint4 &w, int k) {
    const uint32_t x = (k >> 1) == 0 ? w.x : (k >> 1) == 1 ? w.y : (k >> 1) == 2 ? w.z : w.w;
    return (k & 1) ? bf16hi(x) : bf16lo(x);
  }
  // elements e, e + 1 (e even): both halves of one word
  __device__ __forceinline__ static float2 pair(const uint4 &w, int e) {
    const uint32_t x = (e >> 1) == 0 ? w.x : (e >> 1) == 1 ? w.y : (e >> 1) == 2 ? w.z : w.w;
    return make_float2(bf16lo(x), bf16hi(x));
  }
  // vector maximum / running minimum on the packed pairs
  __device__ __forceinline__ static float vmax(const uint4 &w) {
    const uint32_t m = bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w));
    return fmaxf(bf16lo(m), bf16hi(m));
  }
  using MinT = uint32_t;
  __device__ __forceinline__ static MinT min_init() { return 0x7f807f80u; }  // (+inf, +inf)
  __device__ __forceinline__ static MinT min_acc(MinT a, const uint4 &w) {
    return bf16x2_min(a, bf16x2_min(bf16x2_min(w.x, w.y), bf16x2_min(w.z, w.w)));
  }
  __device__ __forceinline__ static float min_fin(MinT a) { return fminf(bf16lo(a), bf16hi(a)); }
  __device__ __forceinline__ static float scalar(const void *row, int v) {
    return __uint_as_float(((uint32_t)reinterpret_cast<const uint16_t *>(row)[v]) << 16);
  }
};
template <>
struct TtsElems<SV_FP32> {
  static constexpr int kPer = 4;
  __device__ __forceinline__ static float get(const uint4 &w, int k) {
    return __uint_as_float(k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w);
  }
  __device__ __forceinline__ static float2 pair(const uint4 &w, int e) {
    return e == 0 ? make_float2(__uint_as_float(w.x), __uint_as_float(w.y))
                  : make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
  __device__ __forceinline__ static float vmax(const uint4 &w) {
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
  using MinT = float;
  __device__ __forceinline__ static MinT min_init() { return INFINITY; }
  __device__ __forceinline__ static MinT min_acc(MinT a, const uint4 &w) {
    return fminf(a, fminf(fminf(__uint_as_float(w.x), __uint_as_float(w.y)),
                          fminf(__uint_as_float(w.z), __uint_as_float(w.w))));
  }
  __device__ __forceinline__ static float min_fin(MinT a) { return a; }
  __device__ __forceinline__ static float scalar(const void *row, int v) {
    return reinterpret_cast<const float *>(row)[v];
  }
};

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// two fp32 -> packed bf16x2, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t bf16_rn(float f) { return (uint16_t)(bf16x2_rn(f, 0.f) & 0xffffu); }

// Online statistics of one lane: running max m and s = sum of
// 2^(fl(z c + nbh)) with nbh = fl(-m c) and nbl = -m c - nbh exactly, so the
// sum of 2^((z - m) c) is s 2^nbl (the rounding of -m c does not enter as a
// common offset of every term).
struct Online {
  float m, s, nbh, nbl;
};
__device__ __forceinline__ void online_raise(Online &o, float vm, float c) {
  const float nbh = __fmul_rn(-vm, c);
  const float nbl = fmaf(-vm, c, -nbh);
  // old terms 2^(z c + nbh_old) become 2^(z c + nbh): the factor 2^(nbh - nbh_old)
  // is exact (the nbl parts cancel)
  o.s = o.m == -INFINITY ? 0.f : o.s * ex2_approx(nbh - o.nbh);
  o.m = vm;
  o.nbh = nbh;
  o.nbl = nbl;
}
// The same statistics for tts_kernel, where one thread sums up to ~65K terms
// of a row (V = 2^24 over 256 threads): each vector's eight terms are added
// pairwise, and the vector sums go into s with Kahan's compensated addition
// (cmp holds the low-order part lost by the previous addition), so the
// thread's sum keeps fp32 precision whatever the row length.
struct OnlineK {
  float m, s, cmp, nbh, nbl;
};
__device__ __forceinline__ OnlineK onlinek_init() { return {-INFINITY, 0.f, 0.f, 0.f, 0.f}; }
__device__ __forceinline__ void onlinek_raise(OnlineK &o, float vm, float c) {
  const float nbh = __fmul_rn(-vm, c);
  const float nbl = fmaf(-vm, c, -nbh);
  const float f = o.m == -INFINITY ? 0.f : ex2_approx(nbh - o.nbh);
  o.s = o.m == -INFINITY ? 0.f : o.s * f;
  o.cmp = o.m == -INFINITY ? 0.f : o.cmp * f;
  o.m = vm;
  o.nbh = nbh;
  o.nbl = nbl;
}
__device__ __forceinline__ void onlinek_add(OnlineK &o, float z, float c) {
  if (z > o.m) onlinek_raise(o, z, c);
  if (o.m > -INFINITY) kahan_add(o.s, o.cmp, ex2_approx(fmaf(z, c, o.nbh)));
}
template <typename E>
__device__ __forceinline__ void onlinek_add_vec(OnlineK &o, const uint4 &x, float c) {
  float vm = E::get(x, 0);
#pragma unroll
  for (int e = 1; e < E::kPer; ++e) vm = fmaxf(vm, E::get(x, e));
  if (vm > o.m) onlinek_raise(o, vm, c);
  if (o.m > -INFINITY) {
    float t[E::kPer];
#pragma unroll
    for (int e = 0; e < E::kPer; ++e) t[e] = ex2_approx(fmaf(E::get(x, e), c, o.nbh));
#pragma unroll
    for (int h = 1; h < E::kPer; h <<= 1)
#pragma unroll
      for (int e = 0; e + h < E::kPer; e += 2 * h) t[e] += t[e + h];
    kahan_add(o.s, o.cmp, t[0]);
  }
}
// Lazy reference for the row-pass statistics held in shared memory: the
// terms are 2^(z c + nbh) with nbh = -m c for a reference m that is raised
// only when a vector's terms would pass 2^64, which keeps any row's sum far
// inside the fp32 range.  The reference is a logit of the row, so terms far
// below the maximum underflow no earlier than with a running maximum; almost
// every vector costs its exponentials and one compare, and the vector's
// maximum is taken only on a raise.  The state starts at nbh = +inf, so the
// first vector holding a finite logit raises (its sum is NaN or +inf).
__device__ __forceinline__ Online lazy_init() { return {-INFINITY, 0.f, INFINITY, 0.f}; }
template <typename E>
__device__ __forceinline__ float lazy_terms(const uint4 &x, float c, float nbh) {
  const float2 cc = make_float2(c, c), nb = make_float2(nbh, nbh);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < E::kPer; e += 2) {
    float2 t = __ffma2_rn(E::pair(x, e), cc, nb);
    t.x = ex2_approx(t.x);
    t.y = ex2_approx(t.y);
    acc = __fadd2_rn(acc, t);
  }
  return acc.x + acc.y;
}
// set the reference from a vector's maximum before its terms are added
template <typename E>
__device__ __forceinline__ void lazy_seed(Online &o, const uint4 &x, float c) {
  const float vm = E::vmax(x);
  if (vm > -INFINITY) online_raise(o, vm, c);
}
template <typename E>
__device__ __forceinline__ void lazy_add_vec2(Online &o, const uint4 &x, float c) {
  float v = lazy_terms<E>(x, c, o.nbh);
  if (!(v <= 0x1p64f)) {
    const float vm = E::vmax(x);
    v = 0.f;
    if (vm > -INFINITY) {
      online_raise(o, vm, c);
      v = lazy_terms<E>(x, c, o.nbh);
    }
  }
  o.s += v;
}

// (m, S = sum of 2^((z - m) c)) pairs for the cross-lane merge
struct MS {
  float m, S;
};
__device__ __forceinline__ MS online_final(const Online &o) { return {o.m, o.s * fmaf(o.nbl, kLn2, 1.f)}; }
__device__ __forceinline__ MS onlinek_final(const OnlineK &o) {
  return {o.m, __fsub_rn(o.s, o.cmp) * fmaf(o.nbl, kLn2, 1.f)};
}
__device__ __forceinline__ MS ms_merge(MS a, MS b, float c) {
  if (b.m > a.m) {
    const MS t = a;
    a = b;
    b = t;
  }
  if (b.m == -INFINITY) return a;
  a.S += b.S * ex2_approx((b.m - a.m) * c);
  return a;
}

// Per-pair constants of d_v = ln p_v - ln q_v = (z_t - z_d) / tau - K0 with
// K0 = (M_t - M_d) / tau + ln(S_t / S_d), and 1/tau, each as hi + lo in fp32
// (fp64 runs at a small fraction of the fp32 rate on this GPU): an error e in
// K0 moves every d by e, i.e. the gradient by p_v e and KL only at second order.
struct PairConst {
  float K0h, K0l, invh, invl;
};
__device__ __forceinline__ PairConst pair_constants(const MS &mt, const MS &md, float tau) {
  PairConst c;
  c.invh = 1.f / tau;
  c.invl = fmaf(-c.invh, tau, 1.f) * c.invh;
  const float dm = mt.m - md.m;  // exact for logits of one format and similar size
  c.K0h = fmaf(dm, c.invh, logf(mt.S / md.S));
  c.K0l = dm * c.invl;
  return c;
}

template <int kDtype>
__global__ void __launch_bounds__(kTtsThreads, 1) tts_kernel(const TtsParams P) {
  using E = TtsElems<kDtype>;
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;
  constexpr int kPer = E::kPer;
  __shared__ MS s_t[kTtsWarps], s_d[kTtsWarps];
  __shared__ float s_kl[kTtsWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, K = P.K;
  const int npairs = P.B * K;
  for (int pair = blockIdx.x; pair < npairs; pair += gridDim.x) {
    const int b = pair / K, k = pair - b * K;
    const float tau_in = __ldg(P.temperature + b);
    const float tau = tau_in > 0.f ? tau_in : 1.f;
    const float c = kLog2e / tau, invtau = 1.f / tau;
    const float w = __ldg(P.weights + k);
    const char *trow = reinterpret_cast<const char *>(P.target) + ((size_t)b * (K + 1) + k) * (size_t)V * kEsz;
    const char *drow = reinterpret_cast<const char *>(P.draft) + ((size_t)b * K + k) * (size_t)V * kEsz;
    // aligned vector span [v0, v1) common to both rows (same offset mod 16)
    const bool same_align = ((reinterpret_cast<uintptr_t>(trow) ^ reinterpret_cast<uintptr_t>(drow)) & 15) == 0;
    int v0 = V, v1 = V;
    if (same_align) {
      v0 = (int)(((16 - (reinterpret_cast<uintptr_t>(trow) & 15)) & 15) / kEsz);
      v0 = min(v0, V);
      v1 = v0 + (V - v0) / kPer * kPer;
    }
    const int nvec = (v1 - v0) / kPer;
    const uint4 *tv = reinterpret_cast<const uint4 *>(trow + (size_t)v0 * kEsz);
    const uint4 *dv = reinterpret_cast<const uint4 *>(drow + (size_t)v0 * kEsz);

    // ---- pass 1: online statistics of both rows
    OnlineK ot = onlinek_init(), od = onlinek_init();
    for (int base = 0; base < nvec; base += kTtsThreads * kTtsUnroll) {
      uint4 xt[kTtsUnroll], xd[kTtsUnroll];
#pragma unroll
      for (int u = 0; u < kTtsUnroll; ++u) {
        const int j = base + u * kTtsThreads + tid;
        if (j < nvec) {
          xt[u] = ld_stream(tv + j);
          xd[u] = ld_stream(dv + j);
        }
      }
#pragma unroll
      for (int u = 0; u < kTtsUnroll; ++u) {
        const int j = base + u * kTtsThreads + tid;
        if (j < nvec) {
          onlinek_add_vec<E>(ot, xt[u], c);
          onlinek_add_vec<E>(od, xd[u], c);
        }
      }
    }
    const int nh = v0, nrest = v0 + (V - v1);  // elements outside the vector span
    for (int i = tid; i < nrest; i += kTtsThreads) {
      const int v = i < nh ? i : v1 + (i - nh);
      onlinek_add(ot, E::scalar(trow, v), c);
      onlinek_add(od, E::scalar(drow, v), c);
    }
    MS mt = onlinek_final(ot), md = onlinek_final(od);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const MS a = {__shfl_xor_sync(0xffffffffu, mt.m, o), __shfl_xor_sync(0xffffffffu, mt.S, o)};
      const MS d = {__shfl_xor_sync(0xffffffffu, md.m, o), __shfl_xor_sync(0xffffffffu, md.S, o)};
      mt = ms_merge(mt, a, c);
      md = ms_merge(md, d, c);
    }
    if (lane == 0) {
      s_t[warp] = mt;
      s_d[warp] = md;
    }
    __syncthreads();
    mt = s_t[0];
    md = s_d[0];
    for (int i = 1; i < kTtsWarps; ++i) {
      mt = ms_merge(mt, s_t[i], c);
      md = ms_merge(md, s_d[i], c);
    }
    const float Mt = mt.m, Md = md.m;
    const float l2St = log2f(mt.S), l2Sd = log2f(md.S);
    // d_v = ln p_v - ln q_v = (z_t - z_d) / tau - K0 with the per-pair
    // constant K0 = (M_t - M_d) / tau + ln(S_t / S_d) taken in fp64 once and
    // split hi + lo, and 1/tau split likewise: d keeps its relative
    // precision when p_v and q_v nearly coincide.
    const PairConst pc = pair_constants(mt, md, tau);
    const float K0h = pc.K0h, K0l = pc.K0l, invh = pc.invh, invl = pc.invl;

    // ---- pass 2: KL terms and the gradient
    // log2 p_v = z_t c + at, log2 q_v = z_d c + ad (one FMA each)
    const float at = -fmaf(Mt, c, l2St), ad = -fmaf(Md, c, l2Sd);
    const float wg = w * invtau;
    float acc = 0.f, acc_c = 0.f;  // Kahan-compensated sum of the thread's KL terms
    // Per element: d = ln p - ln q; the KL term p (e^-d - 1 + d) and the
    // gradient w (q - p) / tau = w p (e^-d - 1) / tau.  For |d| < 1/4 both
    // come from series in d (no cancellation), else from e^-d directly.
    auto element = [&](float zt, float zd, float &g) -> float {
      const float p = ex2_approx(fmaf(zt, c, at));
      const float q = ex2_approx(fmaf(zd, c, ad));
      const float dz = zt - zd;
      const float d = fmaf(dz, invh, -K0h) + fmaf(dz, invl, -K0l);
      const float d2 = d * d;
      // e^-d - 1 + d = d^2 (1/2 - d/6 + d^2/24 - d^3/120)
      const float phi_s = d2 * fmaf(d, fmaf(d, fmaf(d, -1.f / 120.f, 1.f / 24.f), -1.f / 6.f), 0.5f);
      // e^-d - 1 = -d (1 - d/2 + d^2/6 - d^3/24 + d^4/120 - d^5/720)
      const float em1_s = -d * fmaf(d, fmaf(d, fmaf(d, fmaf(d, fmaf(d, -1.f / 720.f, 1.f / 120.f), -1.f / 24.f),
                                                      1.f / 6.f), -0.5f), 1.f);
      const float e = ex2_approx(-d * kLog2e);
      const bool small = fabsf(d) < 0.25f;
      const float em1 = small ? em1_s : e - 1.f;
      const float phi = small ? phi_s : em1 + d;
      // p = 0 (z_t = -inf): the term's limit is q
      g = wg * (p > 0.f ? p * em1 : q);
      return p > 0.f ? p * phi : q;
    };
    uint16_t *grow = P.out_grad ? P.out_grad + ((size_t)b * K + k) * (size_t)V : nullptr;
    const bool gvec = grow && ((reinterpret_cast<uintptr_t>(grow + v0) & 15) == 0);
    for (int base = 0; base < nvec; base += kTtsThreads * kTtsUnroll) {
      uint4 xt[kTtsUnroll], xd[kTtsUnroll];
#pragma unroll
      for (int u = 0; u < kTtsUnroll; ++u) {
        const int j = base + u * kTtsThreads + tid;
        if (j < nvec) {
          xt[u] = ld_stream(tv + j);
          xd[u] = ld_stream(dv + j);
        }
      }
#pragma unroll
      for (int u = 0; u < kTtsUnroll; ++u) {
        const int j = base + u * kTtsThreads + tid;
        if (j < nvec) {
          float g[kPer], kv = 0.f;
#pragma unroll
          for (int e = 0; e < kPer; ++e) kv += element(E::get(xt[u], e), E::get(xd[u], e), g[e]);
          kahan_add(acc, acc_c, kv);
          if (grow) {
            const int v = v0 + j * kPer;
            if (gvec && kPer == 8) {
              uint4 o;
              o.x = bf16x2_rn(g[0], g[1]);
              o.y = bf16x2_rn(g[2], g[3]);
              o.z = bf16x2_rn(g[4], g[5]);
              o.w = bf16x2_rn(g[6], g[7]);
              __stcs(reinterpret_cast<uint4 *>(grow + v), o);
            } else {
#pragma unroll
              for (int e = 0; e < kPer; ++e) grow[v + e] = bf16_rn(g[e]);
            }
          }
        }
      }
    }
    for (int i = tid; i < nrest; i += kTtsThreads) {
      const int v = i < nh ? i : v1 + (i - nh);
      float g;
      kahan_add(acc, acc_c, element(E::scalar(trow, v), E::scalar(drow, v), g));
      if (grow) grow[v] = bf16_rn(g);
    }
    acc = warp_sum(__fsub_rn(acc, acc_c));
    if (lane == 0) s_kl[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      float s = 0.f;
      for (int i = 0; i < kTtsWarps; ++i) s += s_kl[i];
      P.out_kl[(size_t)b * K + k] = w * s;
    }
    __syncthreads();  // shared statistics are rewritten by the next pair
  }
}

// ---------------------------------------------------------------------------
// Shared-memory kernel: a group of CTAs shares a row pair, each holding a
// slice of both rows in shared memory, so the second pass reads shared
// memory instead of re-reading the rows.  A slice is loaded by TMA bulk
// copies in kTtsChunks chunks with one mbarrier each.  Rows must be 16-byte
// aligned with V * esz a multiple of 16 (the host falls back to tts_kernel
// otherwise).
// ---------------------------------------------------------------------------
constexpr int kTtsChunks = 2;
constexpr unsigned long long kTtsWaitNs = 2000000000ull;

// one vector's gradient values -> bf16 (streaming store)
template <int kPer>
__device__ __forceinline__ void store_grad(uint16_t *grow, int j, const float *g) {
  if (kPer == 8) {
    uint4 o;
    o.x = bf16x2_rn(g[0], g[1]);
    o.y = bf16x2_rn(g[2], g[3]);
    o.z = bf16x2_rn(g[4], g[5]);
    o.w = bf16x2_rn(g[6], g[7]);
    __stcs(reinterpret_cast<uint4 *>(grow) + j, o);
  } else {
    uint2 o;
    o.x = bf16x2_rn(g[0], g[1]);
    o.y = bf16x2_rn(g[2], g[3]);
    __stcs(reinterpret_cast<uint2 *>(grow) + j, o);
  }
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_cta(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
  return old;
}

// butterfly merge of the lanes' (m, S) pairs; the pairwise merge is
// symmetric, so every lane ends with the same value
__device__ __forceinline__ void warp_merge2(MS &mt, MS &md, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const MS a = {__shfl_xor_sync(0xffffffffu, mt.m, o), __shfl_xor_sync(0xffffffffu, mt.S, o)};
    const MS d = {__shfl_xor_sync(0xffffffffu, md.m, o), __shfl_xor_sync(0xffffffffu, md.S, o)};
    mt = ms_merge(mt, a, c);
    md = ms_merge(md, d, c);
  }
}
// Pass 1 over the vectors [v0, v1) of a chunk that fall to this thread
// (stride kThreads): lazy statistics of both rows and the running minimum of
// the target logits.  `seed` takes the reference from the thread's first
// vector, so that vector's terms are not computed twice.
template <typename E, int kThreads>
__device__ __forceinline__ void pass1_chunk(const uint4 *tv, const uint4 *dv, int v0, int v1, int tid, bool seed,
                                            float c, Online &ot, Online &od, typename E::MinT &zmin) {
  int j = v0 + tid;
  if (seed && j < v1) {
    lazy_seed<E>(ot, tv[j], c);
    lazy_seed<E>(od, dv[j], c);
  }
  for (; j < v1; j += kThreads) {
    const uint4 xt = tv[j], xd = dv[j];
    zmin = E::min_acc(zmin, xt);
    lazy_add_vec2<E>(ot, xt, c);
    lazy_add_vec2<E>(od, xd, c);
  }
}

// Per-pair constants of the second pass.
struct Pass2Const {
  float c, at, ad, wg;  // log2 e / tau; log2 p = z_t c + at, log2 q = z_d c + ad; w / tau
  float atf;            // at + log2(w / tau) (fast path)
  float invh, nK0;      // 1 / tau and -K0 (d = (z_t - z_d) / tau - K0)
  bool fold;            // w / tau in [2^-20, 2^20]: the fast path may fold it into p
};
__device__ __forceinline__ Pass2Const pass2_constants(const MS &mt, const MS &md, float tau, float c, float w) {
  const PairConst pc = pair_constants(mt, md, tau);
  Pass2Const k;
  k.c = c;
  k.at = -fmaf(mt.m, c, log2f(mt.S));
  k.ad = -fmaf(md.m, c, log2f(md.S));
  k.wg = w * pc.invh;
  k.fold = k.wg >= 0x1p-20f && k.wg <= 0x1p20f;
  k.atf = k.fold ? k.at + log2f(k.wg) : k.at;
  k.invh = pc.invh;
  k.nK0 = -(pc.K0h + pc.K0l);
  return k;
}
// Warp-uniform choice of the fast path: w / tau folds into p, and every
// target logit of the warp's vectors gives p' = (w / tau) p >= 2^-100, so p'
// never underflows and e^-d = q / p stays finite (at most 2^120).
template <typename E>
__device__ __forceinline__ bool pass2_fast_ok(const Pass2Const &k, typename E::MinT zmin) {
  const bool ok_t = fmaf(E::min_fin(zmin), k.c, k.atf) >= -100.f;  // +inf (no vectors) passes, -inf / NaN fail
  return k.fold && __all_sync(0xffffffffu, ok_t);
}

// Pass 2 over the thread's vectors of [v0, v1).  Per element, with
// d = ln p - ln q: the KL term p (e^-d - 1 + d) (by its series for |d| < 1/4,
// where the direct form cancels) and the gradient (w / tau) (q - p) =
// (w / tau) p (e^-d - 1).  The fast path works with p' = (w / tau) p, so its
// KL sum carries the factor w / tau; the general path also covers p = 0
// (z_t = -inf or an underflow), where both terms tend to q.
template <typename E, int kThreads, bool kFast>
__device__ __forceinline__ void pass2_chunk(const uint4 *tv, const uint4 *dv, int v0, int v1, int tid,
                                            const Pass2Const &k, float2 &acc2, uint16_t *grow) {
  constexpr int kPer = E::kPer;
  const float2 cc2 = make_float2(k.c, k.c), invh2 = make_float2(k.invh, k.invh);
  const float2 nK0 = make_float2(k.nK0, k.nK0), neg1 = make_float2(-1.f, -1.f);
  const float2 c120 = make_float2(-1.f / 120.f, -1.f / 120.f), c24 = make_float2(1.f / 24.f, 1.f / 24.f);
  const float2 c6 = make_float2(-1.f / 6.f, -1.f / 6.f), half2 = make_float2(0.5f, 0.5f);
  const float2 nlog2e = make_float2(-kLog2e, -kLog2e);
  const float a = kFast ? k.atf : k.at;
  const float2 at2 = make_float2(a, a), wg2 = make_float2(k.wg, k.wg);
  for (int j = v0 + tid; j < v1; j += kThreads) {
    const uint4 xt = tv[j], xd = dv[j];
    float g[kPer];
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const float2 zt = E::pair(xt, e), zd = E::pair(xd, e);
      float2 p = __ffma2_rn(zt, cc2, at2);
      p.x = ex2_approx(p.x);
      p.y = ex2_approx(p.y);
      const float2 d = __ffma2_rn(__ffma2_rn(zd, neg1, zt), invh2, nK0);
      float2 ex = __fmul2_rn(d, nlog2e);  // e^-d = q / p
      ex.x = ex2_approx(ex.x);
      ex.y = ex2_approx(ex.y);
      float2 poly = __ffma2_rn(d, c120, c24);
      poly = __ffma2_rn(d, poly, c6);
      poly = __ffma2_rn(d, poly, half2);  // (e^-d - 1 + d) / d^2 to fifth order
      if (kFast) {
        // scalar from here: the exponentials come out of the SFU one by one
        const float2 dp = __fmul2_rn(d, poly);
        const float tgx = fmaf(p.x, ex.x, -p.x), tgy = fmaf(p.y, ex.y, -p.y);  // (w / tau) (q - p)
        const float tx = p.x * d.x, ty = p.y * d.y;
        acc2.x += fabsf(d.x) < 0.25f ? tx * dp.x : tx + tgx;
        acc2.y += fabsf(d.y) < 0.25f ? ty * dp.y : ty + tgy;
        g[e] = tgx;
        g[e + 1] = tgy;
      } else {
        const float2 phi_s = __fmul2_rn(__fmul2_rn(d, d), poly);
        const float2 em1 = __fadd2_rn(ex, neg1);  // e^-d - 1
        const float2 phl = __fadd2_rn(em1, d);
        const float2 phi = make_float2(fabsf(d.x) < 0.25f ? phi_s.x : phl.x, fabsf(d.y) < 0.25f ? phi_s.y : phl.y);
        float2 tkl = __fmul2_rn(p, phi), tg = __fmul2_rn(p, em1);
        if (!(p.x > 0.f) || !(p.y > 0.f)) {  // p = 0: the limits of both terms are q
          if (!(p.x > 0.f)) tkl.x = tg.x = ex2_approx(fmaf(zd.x, k.c, k.ad));
          if (!(p.y > 0.f)) tkl.y = tg.y = ex2_approx(fmaf(zd.y, k.c, k.ad));
        }
        acc2 = __fadd2_rn(acc2, tkl);
        const float2 gg = __fmul2_rn(wg2, tg);
        g[e] = gg.x;
        g[e + 1] = gg.y;
      }
    }
    if (grow) store_grad<kPer>(grow, j, g);
  }
}

// ---------------------------------------------------------------------------
// Group kernel: G CTAs (one per SM, any G up to 32, no cluster) share a row
// pair, each holding a slice of S elements of both rows; nb = 2 or 3 pair
// slices stay resident per CTA.  The slice is copied in kTtsChunks chunks,
// each owned by kGrpWarps / kTtsChunks compute warps, so a warp waits for
// one copy and releases one chunk per pair.  Per pair i a compute thread
// runs the statistics of pair i + 1 (left in shared memory), then the
// second pass of pair i (its KL partial left in shared memory); a chunk
// released by all its warps is refilled with pair i + nb.  A coordinator
// warp merges the threads' statistics into the CTA's entry and publishes it
// in the workspace; it gathers the group's G entries of a pair, merges them
// in rank order and derives the row constants once for the CTA; it sums the
// threads' KL partials, and on rank 0 sums the group's partials in rank
// order into out_kl two pairs later.  No compute warp waits on another SM.
// Every 64-bit word of the exchange holds a 32-bit value and a 32-bit tag
// (the call's generation and the pair's use of the slot), and each word is
// stored and loaded whole, so one relaxed load both tests and reads an
// entry; words of an earlier call or an earlier use of the slot never
// match.
// ---------------------------------------------------------------------------
constexpr int kGrpWarps = 16;                        // compute warps
constexpr int kGrpCompute = kGrpWarps * 32;
constexpr int kGrpThreads = kGrpCompute + 32;        // + the coordinator warp
constexpr int kGrpMinBlocks = kGrpWarps >= 16 ? 1 : 16 / kGrpWarps;  // CTAs per SM the registers must allow
constexpr int kChunkWarps = kGrpWarps / kTtsChunks;  // warps that own a chunk
constexpr int kChunkThreads = kChunkWarps * 32;
constexpr int kGrpMaxNb = 3;
constexpr int kGrpSlots = 4;                         // pairs whose exchange may be in flight
constexpr int kTtsMaxGroup = 32;
constexpr int kTtsMaxCtas = 1024;
static_assert(kGrpWarps % kTtsChunks == 0, "whole warps per chunk");
constexpr size_t kTtsWsHeader = 256;                 // status word and spare
// workspace: header, then per slot and CTA the statistics entry (four tagged
// words: m_t, S_t, m_d, S_d), then per slot and CTA the tagged KL partial
constexpr size_t kTtsWsStat = kTtsWsHeader;
constexpr size_t kTtsWsKl = kTtsWsStat + (size_t)kGrpSlots * kTtsMaxCtas * 32;
constexpr size_t kTtsWsBytes = kTtsWsKl + (size_t)kGrpSlots * kTtsMaxCtas * 8;

struct GroupArgs {
  int G, S, nb;
  uint32_t gen;         // call generation (tags)
  unsigned char *ws;    // workspace (kTtsWsBytes)
  unsigned long long wait_ns;  // limit of every wait (2 s, or sv_set_wait_test's)
  int withhold;         // sv_set_wait_test: no row copies are issued
};

struct GroupSmem {
  uint64_t full[kGrpMaxNb][kTtsChunks];
  uint64_t stat_bar[2];            // the compute threads' statistics of pairs of even / odd order
  uint64_t kl_bar[2];              // their KL partials
  uint64_t const_bar[kGrpSlots];   // a pair's constants are ready (coordinator)
  uint32_t released[kGrpMaxNb][kTtsChunks];
  uint32_t issued[kGrpMaxNb][kTtsChunks];
  Pass2Const pc[kGrpSlots];
  float scale[kGrpSlots];          // out_kl = scale * (sum of the partials)
  int pc_ok[kGrpSlots];
  int abort;                       // a wait timed out: no further copies, outputs of later pairs are NaN
  float4 tstat[2][kGrpCompute];    // per thread (m_t, S_t, m_d, S_d)
  float tkl[2][kGrpCompute];       // per thread KL partial
};

// tagged words: value bits low, tag high
__device__ __forceinline__ unsigned long long tagged(float v, uint32_t tag) {
  return ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
}
__device__ __forceinline__ float untag(unsigned long long w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ bool tag_is(unsigned long long w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }
__device__ __forceinline__ void st_words2(unsigned long long *p, unsigned long long a, unsigned long long b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ld_words2(const unsigned long long *p, unsigned long long &a, unsigned long long &b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned long long ld_word(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_word(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Waits of the group kernel poll a barrier between sleeps that double from
// 32 ns up to max_ns, so a waiting warp leaves its scheduler's issue slots
// to the warps that compute.  Both are bounded by the launch's limit (2 s,
// or the one sv_set_wait_test sets) and set
// SV_FLAG_TIMEOUT when they give up.
// Chunk copies: also gives up as soon as another thread set the abort flag.
__device__ __forceinline__ bool wait_copy(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *status, uint32_t max_ns, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t ns = 32;; ns = ns < max_ns ? 2 * ns : max_ns) {
    __nanosleep(ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, SV_FLAG_TIMEOUT);
      return false;
    }
  }
}
// CTA-local barriers: every arrival on them happens even after an abort, so
// they always complete; time-bounded only
__device__ __forceinline__ bool mbar_wait_local(uint64_t *bar, uint32_t parity, uint32_t *status, uint32_t max_ns,
                                                unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t ns = 32;; ns = ns < max_ns ? 2 * ns : max_ns) {
    __nanosleep(ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(status, SV_FLAG_TIMEOUT);
      return false;
    }
  }
}
// lanes < n read their record (nw = 4: a statistics entry, 1: a KL partial)
// until every word carries `tag` (warp-uniform result, bounded; nanosleep
// back-off between polls)
template <int nw>
__device__ __forceinline__ bool poll_records(const unsigned long long *rec, int n, int lane, uint32_t tag,
                                             unsigned long long (&w)[4], uint32_t *status,
                                             unsigned long long limit_ns) {
  auto load = [&]() {
    if (lane >= n) return true;
    if (nw == 4) {
      ld_words2(rec + 4 * lane, w[0], w[1]);
      ld_words2(rec + 4 * lane + 2, w[2], w[3]);
      return tag_is(w[0], tag) && tag_is(w[1], tag) && tag_is(w[2], tag) && tag_is(w[3], tag);
    }
    w[0] = ld_word(rec + lane);
    return tag_is(w[0], tag);
  };
  bool mine = load();
  if (__all_sync(0xffffffffu, mine)) return true;
  const uint64_t t0 = __shfl_sync(0xffffffffu, global_ns(), 0);
  uint32_t ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
    if (!mine) mine = load();
    if (__all_sync(0xffffffffu, mine)) return true;
    if (__shfl_sync(0xffffffffu, global_ns() - t0 > limit_ns ? 1 : 0, 0)) {
      if (lane == 0) atomicOr(status, SV_FLAG_TIMEOUT);
      return false;
    }
  }
}

template <int kDtype>
__global__ void __launch_bounds__(kGrpThreads, kGrpMinBlocks) tts_group_kernel(const TtsParams P, const GroupArgs A) {
  using E = TtsElems<kDtype>;
  using MinT = typename E::MinT;
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;
  constexpr int kPer = E::kPer;
  extern __shared__ __align__(128) uint8_t tts_smem[];
  GroupSmem &R = *reinterpret_cast<GroupSmem *>(tts_smem);
  uint8_t *ring = tts_smem + ((sizeof(GroupSmem) + 127) / 128) * 128;
  const size_t slice_bytes = (size_t)A.S * kEsz;  // per buffer: target slice, then draft slice
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, K = P.K, G = A.G, nb = A.nb;
  const int cta = (int)blockIdx.x, grp = cta / G, rank = cta - grp * G;
  const int ngroups = (int)gridDim.x / G;
  const int npairs = P.B * K;
  const int npairs_g = grp < npairs ? (npairs - grp + ngroups - 1) / ngroups : 0;  // pairs of this group
  const int e0 = rank * A.S, e1 = min(V, e0 + A.S);
  const int nel = max(0, e1 - e0);
  const int nvec = nel / kPer;
  const int cvec = (nvec + kTtsChunks - 1) / kTtsChunks;
  uint32_t *status = reinterpret_cast<uint32_t *>(A.ws);
  unsigned long long *g_stat = reinterpret_cast<unsigned long long *>(A.ws + kTtsWsStat);
  unsigned long long *g_kl = reinterpret_cast<unsigned long long *>(A.ws + kTtsWsKl);
  // a slot's previous content is from the same call four pairs earlier (other
  // phase bit) or from an earlier call (other generation)
  auto tag_of = [&](int it) { return (A.gen << 1) | (uint32_t)((it >> 2) & 1); };

  if (tid == 0) {
    for (int bi = 0; bi < kGrpMaxNb; ++bi)
      for (int ch = 0; ch < kTtsChunks; ++ch) {
        mbar_init(&R.full[bi][ch], 1);
        R.released[bi][ch] = 0;
        R.issued[bi][ch] = 0;
      }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&R.stat_bar[s], kGrpCompute);
      mbar_init(&R.kl_bar[s], kGrpCompute);
    }
    for (int s = 0; s < kGrpSlots; ++s) mbar_init(&R.const_bar[s], 1);
    R.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // request chunk ch of the it-th pair of this group into buffer it % nb
  auto issue = [&](int it, int ch) {
    if (it >= npairs_g || A.withhold) return;
    const int pair = grp + it * ngroups;
    const int bi = it % nb;
    const int b = pair / K, k = pair - b * K;
    const int v0 = min(nvec, ch * cvec), v1 = min(nvec, v0 + cvec);
    const uint32_t bytes = (uint32_t)(v1 - v0) * 16u;
    uint8_t *buf = ring + (size_t)bi * 2 * slice_bytes;
    R.issued[bi][ch] += 1;
    mbar_arrive_expect_tx(&R.full[bi][ch], 2 * bytes);
    if (bytes) {
      const char *trow = reinterpret_cast<const char *>(P.target) + ((size_t)b * (K + 1) + k) * (size_t)V * kEsz;
      const char *drow = reinterpret_cast<const char *>(P.draft) + ((size_t)b * K + k) * (size_t)V * kEsz;
      const size_t off = (size_t)e0 * kEsz + (size_t)v0 * 16;
      bulk_g2s(buf + (size_t)v0 * 16, trow + off, bytes, &R.full[bi][ch]);
      bulk_g2s(buf + slice_bytes + (size_t)v0 * 16, drow + off, bytes, &R.full[bi][ch]);
    }
  };
  if (tid == 0)
    for (int i = 0; i < nb; ++i)
      for (int ch = 0; ch < kTtsChunks; ++ch) issue(i, ch);

  volatile int *abort_flag = &R.abort;
  auto pair_c = [&](int it) {
    const float tau_in = __ldg(P.temperature + (grp + it * ngroups) / K);
    return kLog2e / (tau_in > 0.f ? tau_in : 1.f);
  };

  if (warp < kGrpWarps) {
    // ---------------- compute warps: chunk cw, thread ct of its owners
    const int cw = warp / kChunkWarps;
    const int ct = tid - cw * kChunkThreads;
    const int v0 = min(nvec, cw * cvec), v1 = min(nvec, v0 + cvec);
    auto stats = [&](int it) -> MinT {  // pass 1 of pair it over this thread's vectors
      const float c = pair_c(it);
      const int bi = it % nb;
      const uint4 *tv = reinterpret_cast<const uint4 *>(ring + (size_t)bi * 2 * slice_bytes);
      const uint4 *dv = reinterpret_cast<const uint4 *>(ring + (size_t)bi * 2 * slice_bytes + slice_bytes);
      Online ot = lazy_init(), od = lazy_init();
      MinT zmin = E::min_init();
      if (!*abort_flag) wait_copy(&R.full[bi][cw], (uint32_t)((it / nb) & 1), abort_flag, status, 256u, A.wait_ns);
      if (!*abort_flag) pass1_chunk<E, kChunkThreads>(tv, dv, v0, v1, ct, true, c, ot, od, zmin);
      const MS mt = online_final(ot), md = online_final(od);
      R.tstat[it & 1][tid] = make_float4(mt.m, mt.S, md.m, md.S);
      mbar_arrive(&R.stat_bar[it & 1]);
      return zmin;
    };
    MinT zcur = npairs_g > 0 ? stats(0) : E::min_init();
    for (int it = 0; it < npairs_g; ++it) {
      const MinT znext = it + 1 < npairs_g ? stats(it + 1) : E::min_init();
      const int pair = grp + it * ngroups;
      const int b = pair / K, k = pair - b * K;
      const int slot = it & (kGrpSlots - 1);
      mbar_wait_local(&R.const_bar[slot], (uint32_t)((it / kGrpSlots) & 1), status, 256u, A.wait_ns);
      const Pass2Const pk = R.pc[slot];
      const bool ok = R.pc_ok[slot] != 0 && !*abort_flag;
      const bool fast = pass2_fast_ok<E>(pk, zcur);
      float2 acc2 = make_float2(0.f, 0.f);
      const int bi = it % nb;
      const uint4 *tv = reinterpret_cast<const uint4 *>(ring + (size_t)bi * 2 * slice_bytes);
      const uint4 *dv = reinterpret_cast<const uint4 *>(ring + (size_t)bi * 2 * slice_bytes + slice_bytes);
      uint16_t *grow = P.out_grad ? P.out_grad + ((size_t)b * K + k) * (size_t)V + e0 : nullptr;
      if (ok && fast) pass2_chunk<E, kChunkThreads, true>(tv, dv, v0, v1, ct, pk, acc2, grow);
      else if (ok) pass2_chunk<E, kChunkThreads, false>(tv, dv, v0, v1, ct, pk, acc2, grow);
      __syncwarp();
      if (lane == 0) {  // this warp is done with its chunk; the last owner refills it
        const uint32_t done = atom_add_acq_rel_cta(&R.released[bi][cw], 1u);
        if (done == (uint32_t)kChunkWarps * (uint32_t)(it / nb + 1) - 1u && !*abort_flag) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue(it + nb, cw);
        }
      }
      float part = acc2.x + acc2.y;
      if (!fast && pk.fold) part *= pk.wg;  // the scale of the fast path's terms
      if (!ok) part = __int_as_float(0x7fc00000);
      R.tkl[it & 1][tid] = part;
      mbar_arrive(&R.kl_bar[it & 1]);
      zcur = znext;
    }
  } else {
    // ---------------- coordinator warp
    auto publish = [&](int it) {  // the CTA's entry of pair it
      const float c = pair_c(it);
      mbar_wait_local(&R.stat_bar[it & 1], (uint32_t)((it >> 1) & 1), status, 512u, A.wait_ns);
      // lane l merges the threads l + 32 j, j < 16, as a tree (depth 4)
      constexpr int kPerLane = kGrpCompute / 32;
      MS t[kPerLane], d[kPerLane];
#pragma unroll
      for (int j = 0; j < kPerLane; ++j) {
        const float4 v = R.tstat[it & 1][lane + 32 * j];
        t[j] = MS{v.x, v.y};
        d[j] = MS{v.z, v.w};
      }
#pragma unroll
      for (int h = 1; h < kPerLane; h <<= 1)
#pragma unroll
        for (int j = 0; j + h < kPerLane; j += 2 * h) {
          t[j] = ms_merge(t[j], t[j + h], c);
          d[j] = ms_merge(d[j], d[j + h], c);
        }
      MS mt = t[0], md = d[0];
      warp_merge2(mt, md, c);
      unsigned long long *rec = g_stat + ((size_t)(it & (kGrpSlots - 1)) * kTtsMaxCtas + cta) * 4;
      if (lane == 0) {
        const float nan = __int_as_float(0x7fc00000);  // after an abort: the group's constants become NaN
        const uint32_t tg = tag_of(it);
        const bool bad = *abort_flag != 0;
        st_words2(rec, tagged(bad ? nan : mt.m, tg), tagged(bad ? nan : mt.S, tg));
        st_words2(rec + 2, tagged(bad ? nan : md.m, tg), tagged(bad ? nan : md.S, tg));
      }
    };
    auto gather = [&](int it) {  // the group's entries of pair it -> the CTA's constants
      const int pair = grp + it * ngroups;
      const int b = pair / K, k = pair - b * K;
      const float tau_in = __ldg(P.temperature + b);
      const float tau = tau_in > 0.f ? tau_in : 1.f;
      const float c = kLog2e / tau;
      const float w = __ldg(P.weights + k);
      const int slot = it & (kGrpSlots - 1);
      unsigned long long rw[4];
      const bool got =
          poll_records<4>(g_stat + ((size_t)slot * kTtsMaxCtas + (size_t)grp * G) * 4, G, lane, tag_of(it), rw, status,
                          A.wait_ns);
      MS mt = {-INFINITY, 0.f}, md = {-INFINITY, 0.f};
      if (lane < G) {
        mt = MS{untag(rw[0]), untag(rw[1])};
        md = MS{untag(rw[2]), untag(rw[3])};
      }
      warp_merge2(mt, md, c);
      if (lane == 0) {
        const Pass2Const pk = pass2_constants(mt, md, tau, c, w);
        R.pc[slot] = pk;
        R.scale[slot] = pk.fold ? w / pk.wg : w;
        R.pc_ok[slot] = got ? 1 : 0;
        if (!got) *abort_flag = 1;
        mbar_arrive(&R.const_bar[slot]);
      }
    };
    auto klsum = [&](int it) {  // the CTA's KL partial of pair it
      mbar_wait_local(&R.kl_bar[it & 1], (uint32_t)((it >> 1) & 1), status, 512u, A.wait_ns);
      constexpr int kPerLane = kGrpCompute / 32;
      float v[kPerLane];
#pragma unroll
      for (int j = 0; j < kPerLane; ++j) v[j] = R.tkl[it & 1][lane + 32 * j];
#pragma unroll
      for (int h = 1; h < kPerLane; h <<= 1)
#pragma unroll
        for (int j = 0; j + h < kPerLane; j += 2 * h) v[j] += v[j + h];
      const float s = warp_sum(v[0]);
      if (lane == 0) st_word(g_kl + (size_t)(it & (kGrpSlots - 1)) * kTtsMaxCtas + cta, tagged(s, tag_of(it)));
    };
    auto klgather = [&](int it) {  // rank 0: the group's partials of pair it -> out_kl
      const int slot = it & (kGrpSlots - 1);
      unsigned long long w[4];
      const bool got = poll_records<1>(g_kl + (size_t)slot * kTtsMaxCtas + (size_t)grp * G, G, lane, tag_of(it), w,
                                       status, A.wait_ns);
      const float s = warp_sum(lane < G ? untag(w[0]) : 0.f);
      if (lane == 0) P.out_kl[grp + it * ngroups] = got ? R.scale[slot] * s : __int_as_float(0x7fc00000);
    };
    if (npairs_g > 0) publish(0);
    for (int it = 0; it < npairs_g; ++it) {
      gather(it);
      if (it + 1 < npairs_g) publish(it + 1);
      if (it >= 1) klsum(it - 1);
      if (rank == 0 && it >= 2) klgather(it - 2);
    }
    if (npairs_g > 0) klsum(npairs_g - 1);
    if (rank == 0)
      for (int it = max(0, npairs_g - 2); it < npairs_g; ++it) klgather(it);
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) {  // copies that were never waited for (bounded)
    const uint64_t t0 = global_ns();
    for (int bi = 0; bi < nb; ++bi)
      for (int ch = 0; ch < kTtsChunks; ++ch)
        if (R.issued[bi][ch])
          while (!mbar_try_wait(&R.full[bi][ch], (R.issued[bi][ch] - 1u) & 1u) && global_ns() - t0 < A.wait_ns) {
          }
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

namespace {
// Launch configuration for one (V, dtype): groups whose slices fit three
// resident buffers (else two), as many CTAs per SM as the occupancy query
// allows, the grid a whole number of groups.  Among the group sizes that
// fit, the one with the least estimated time per pair and group: a pair
// costs each CTA about 0.4 us per 16-byte vector step of its slowest thread
// (ceil(vectors per chunk / threads per chunk), per pass) plus about 2.3 us
// of per-pair latency (measured on the C3 rows, B=256 K=5 V=128256 bf16:
// G = 8, three slices, 4 steps: 267 us; G = 10, four slices, 4 steps:
// 322 us; G = 19, four slices, 2 steps: 501 us).
struct TtsCfg {
  int G, S, nb, ctas;
  size_t smem;
};

bool tts_group_cfg_uncached(int V, int esz, int dtype, int sms, TtsCfg *out) {
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  const size_t kSmemMax = (size_t)optin;
  const int unit = 16 / esz;
  const size_t head = ((sizeof(GroupSmem) + 127) / 128) * 128;
  const void *fn = dtype == SV_BF16 ? (const void *)tts_group_kernel<SV_BF16> : (const void *)tts_group_kernel<SV_FP32>;
  for (int nb : {3, 2}) {
    TtsCfg best{0, 0, 0, 0, 0};
    double best_cost = 0.0;
    for (int G = 1; G <= kTtsMaxGroup; ++G) {
      const int S = ((V + G - 1) / G + unit - 1) / unit * unit;
      if ((long long)(G - 1) * S >= V) continue;  // every rank holds part of the row
      const size_t smem = head + (size_t)nb * 2 * (size_t)S * esz;
      if (smem > kSmemMax) continue;
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
      }
      int nper = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nper, fn, kGrpThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
      }
      long long slots = (long long)nper * sms;
      if (slots > kTtsMaxCtas) slots = kTtsMaxCtas;
      const long long ctas = slots / G * G;
      if (ctas < G) continue;
      const int cvec = (S / unit + kTtsChunks - 1) / kTtsChunks;  // 16-byte vectors per chunk
      const int steps = (cvec + kChunkThreads - 1) / kChunkThreads;
      const double cost = (0.4 * steps + 2.3) / (double)(ctas / G);
      if (!best.G || cost < best_cost) {
        best_cost = cost;
        best = TtsCfg{G, S, nb, (int)ctas, smem};
      }
    }
    if (best.G) {
      *out = best;
      return true;
    }
  }
  return false;
}

// small per-process cache keyed by (device, V, dtype)
std::mutex g_tts_mu;
struct TtsCacheEnt {
  int dev, V, dtype, ok;
  TtsCfg cfg;
};
TtsCacheEnt g_tts_cache[16];
int g_tts_n = 0;
std::atomic<uint32_t> g_tts_gen{0};

bool tts_group_cfg(int V, int esz, int dtype, int sms, TtsCfg *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(g_tts_mu);
  for (int i = 0; i < g_tts_n; ++i)
    if (g_tts_cache[i].dev == dev && g_tts_cache[i].V == V && g_tts_cache[i].dtype == dtype) {
      *out = g_tts_cache[i].cfg;
      return g_tts_cache[i].ok != 0;
    }
  TtsCfg cfg{};
  const bool ok = tts_group_cfg_uncached(V, esz, dtype, sms, &cfg);
  TtsCacheEnt &e = g_tts_cache[g_tts_n < 16 ? g_tts_n++ : 15];
  e = TtsCacheEnt{dev, V, dtype, ok ? 1 : 0, cfg};
  *out = cfg;
  return ok;
}
}  // namespace

extern "C" size_t sv_tts_workspace_bytes(void) { return kTtsWsBytes; }

extern "C" sv_status_t sv_tts_signal(int B, int K, int V, sv_dtype_t dtype, const void *target_logits,
                                     const void *draft_logits, const float *temperature, const float *weights,
                                     float *out_kl, uint16_t *out_grad, void *workspace, size_t workspace_bytes,
                                     void *stream) {
  if (B < 0 || B > (1 << 20) || K < 0 || K > SV_MAX_K || V < 1 || V > SV_MAX_V) return SV_ERR_INVALID;
  if (dtype != SV_BF16 && dtype != SV_FP32) return SV_ERR_INVALID;
  if (!workspace || workspace_bytes < kTtsWsBytes || !host_aligned(workspace, 256)) return SV_ERR_WORKSPACE;
  if ((long long)B * K == 0) return SV_OK;
  if (!target_logits || !draft_logits || !temperature || !weights || !out_kl) return SV_ERR_INVALID;
  const int esz = dtype == SV_BF16 ? 2 : 4;
  if (!host_aligned(target_logits, esz) || !host_aligned(draft_logits, esz) || !host_aligned(temperature, 4) ||
      !host_aligned(weights, 4) || !host_aligned(out_kl, 4) || !host_aligned(out_grad, 2))
    return SV_ERR_INVALID;
  int sms = 0;
  const sv_status_t ds = host_device_info(&sms);
  if (ds != SV_OK) return ds;
  TtsParams P{B, K, V, (int)dtype, target_logits, draft_logits, temperature, weights, out_kl, out_grad};
  const long long pairs = (long long)B * K;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, 4, st);  // this call's status word
  if (e != cudaSuccess) return host_cuda_status(e);
  // the group kernel wants 16-byte aligned rows and slices
  const bool aligned16 = ((size_t)V * esz) % 16 == 0 && host_aligned(target_logits, 16) &&
                         host_aligned(draft_logits, 16) && (!out_grad || (host_aligned(out_grad, 16) && V % 8 == 0));
  TtsCfg cfg;
  if (aligned16 && tts_group_cfg(V, esz, (int)dtype, sms, &cfg)) {
    const long long ngroups = pairs < cfg.ctas / cfg.G ? pairs : cfg.ctas / cfg.G;
    const void *fn =
        dtype == SV_BF16 ? (const void *)tts_group_kernel<SV_BF16> : (const void *)tts_group_kernel<SV_FP32>;
    // the occupancy queries of other configurations may have left a smaller limit
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.smem);
    if (e != cudaSuccess) return host_cuda_status(e);
    uint32_t gen = g_tts_gen.fetch_add(1u) + 1u;
    while ((uint32_t)(gen << 1) == 0u) gen = g_tts_gen.fetch_add(1u) + 1u;  // tag 0 would match a zeroed workspace
    unsigned long long wait_ns = 0;
    int withhold = 0;
    host_wait_test(&wait_ns, &withhold);
    const GroupArgs A{cfg.G,  cfg.S,  cfg.nb, gen, static_cast<unsigned char *>(workspace),
                      wait_ns ? wait_ns : kTtsWaitNs, withhold};
    const unsigned grid = (unsigned)(ngroups * cfg.G);
    if (dtype == SV_BF16) tts_group_kernel<SV_BF16><<<grid, kGrpThreads, cfg.smem, st>>>(P, A);
    else tts_group_kernel<SV_FP32><<<grid, kGrpThreads, cfg.smem, st>>>(P, A);
    return host_cuda_status(cudaGetLastError());
  }
  const int grid = (int)(pairs < sms ? pairs : sms);
  if (dtype == SV_BF16) tts_kernel<SV_BF16><<<grid, kTtsThreads, 0, st>>>(P);
  else tts_kernel<SV_FP32><<<grid, kTtsThreads, 0, st>>>(P);
  return host_cuda_status(cudaGetLastError());
}
