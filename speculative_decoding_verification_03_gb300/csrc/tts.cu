// Test-time speculation (TTS) distillation signal ("Technical summary:
// Test-Time Speculation (TTS)", section "Algorithm", step 3): for every
// canvas position k of request b, with p = softmax(z_target / tau) and
// q = softmax(z_draft / tau),
//   kl[b][k]      = w_k * KL(p || q)
//   grad[b][k][v] = w_k * (q_v - p_v) / tau        (bf16; the gradient of
//                   that term with respect to the draft logits)
// One CTA per (b, k) row pair at a time, two passes over the pair: online
// max/sum statistics of both rows, then the per-element KL terms and the
// gradient; the second pass re-reads the pair from L2.  KL is summed as
// p (e^-d - 1 + d) with d = ln p - ln q, a sum of non-negative terms taken
// by a short series for small |d|, so it keeps its relative precision when
// q is close to p.
#include <cfloat>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTtsThreads = 512;
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
template <>
struct TtsElems<SV_BF16> {
  static constexpr int kPer = 8;
  __device__ __forceinline__ static float get(const uint4 &w, int k) {
    const uint32_t x = (k >> 1) == 0 ? w.x : (k >> 1) == 1 ? w.y : (k >> 1) == 2 ? w.z : w.w;
    return (k & 1) ? bf16hi(x) : bf16lo(x);
  }
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

// round to nearest even fp32 -> bf16 bits (finite inputs; NaN stays NaN)
__device__ __forceinline__ uint32_t bf16_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  return (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
}

// Online statistics of one lane: running max m and s = sum of
// 2^(fl(z c + nbh)) with nbh = fl(-m c) and nbl = -m c - nbh exactly, so the
// sum of 2^((z - m) c) is s 2^nbl (the rounding of -m c does not enter as a
// common offset of every term).
struct Online {
  float m, s, nbh, nbl;
};
__device__ __forceinline__ Online online_init() { return {-INFINITY, 0.f, 0.f, 0.f}; }
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
__device__ __forceinline__ void online_add(Online &o, float z, float c) {
  if (z > o.m) online_raise(o, z, c);
  if (o.m > -INFINITY) o.s += ex2_approx(fmaf(z, c, o.nbh));
}
// one 16-byte vector: raise once to the vector's max, then add its terms
template <typename E>
__device__ __forceinline__ void online_add_vec(Online &o, const uint4 &x, float c) {
  float vm = E::get(x, 0);
#pragma unroll
  for (int e = 1; e < E::kPer; ++e) vm = fmaxf(vm, E::get(x, e));
  if (vm > o.m) online_raise(o, vm, c);
  if (o.m > -INFINITY) {
#pragma unroll
    for (int e = 0; e < E::kPer; ++e) o.s += ex2_approx(fmaf(E::get(x, e), c, o.nbh));
  }
}
// (m, S = sum of 2^((z - m) c)) pairs for the cross-lane merge
struct MS {
  float m, S;
};
__device__ __forceinline__ MS online_final(const Online &o) { return {o.m, o.s * fmaf(o.nbl, kLn2, 1.f)}; }
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

// KL term p (e^-d - 1 + d) for one element, d = ln p - ln q (every term a
// multiple of p, so an error in p's normalisation only scales the sum)
__device__ __forceinline__ float kl_term(float p, float q, float d) {
  if (fabsf(d) < 0.25f) {
    const float poly = fmaf(d, fmaf(d, fmaf(d, -1.f / 120.f, 1.f / 24.f), -1.f / 6.f), 0.5f);
    return p * d * d * poly;
  }
  // p = 0 (d not finite): the term's limit is q
  if (!(p > 0.f)) return q;
  return p * ((ex2_approx(-d * kLog2e) - 1.f) + d);
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
    Online ot = online_init(), od = online_init();
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
          online_add_vec<E>(ot, xt[u], c);
          online_add_vec<E>(od, xd[u], c);
        }
      }
    }
    const int nh = v0, nrest = v0 + (V - v1);  // elements outside the vector span
    for (int i = tid; i < nrest; i += kTtsThreads) {
      const int v = i < nh ? i : v1 + (i - nh);
      online_add(ot, E::scalar(trow, v), c);
      online_add(od, E::scalar(drow, v), c);
    }
    MS mt = online_final(ot), md = online_final(od);
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
    const double inv_d = 1.0 / (double)tau;
    const double K0 = ((double)Mt - (double)Md) * inv_d + log((double)mt.S / (double)md.S);
    const float K0h = (float)K0, K0l = (float)(K0 - (double)K0h);
    const float invh = (float)inv_d, invl = (float)(inv_d - (double)invh);

    // ---- pass 2: KL terms and the gradient
    float acc = 0.f;
    auto element = [&](float zt, float zd, float &g) {
      const float dt = zt - Mt, dd = zd - Md;
      const float p = ex2_approx(fmaf(dt, c, -l2St));
      const float q = ex2_approx(fmaf(dd, c, -l2Sd));
      const float dz = zt - zd;
      const float d = fmaf(dz, invh, -K0h) + fmaf(dz, invl, -K0l);
      acc += kl_term(p, q, d);
      // q - p = p (e^-d - 1): for small |d| from the series of e^-d - 1,
      // which keeps its relative precision when q and p nearly cancel
      const float x = -d;
      const float em1 = x * fmaf(x, fmaf(x, fmaf(x, fmaf(x, fmaf(x, 1.f / 720.f, 1.f / 120.f), 1.f / 24.f),
                                                  1.f / 6.f), 0.5f), 1.f);
      g = w * (fabsf(d) < 0.25f ? p * em1 : q - p) * invtau;
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
          float g[kPer];
#pragma unroll
          for (int e = 0; e < kPer; ++e) element(E::get(xt[u], e), E::get(xd[u], e), g[e]);
          if (grow) {
            const int v = v0 + j * kPer;
            if (gvec && kPer == 8) {
              uint4 o;
              o.x = bf16_bits(g[0]) | (bf16_bits(g[1]) << 16);
              o.y = bf16_bits(g[2]) | (bf16_bits(g[3]) << 16);
              o.z = bf16_bits(g[4]) | (bf16_bits(g[5]) << 16);
              o.w = bf16_bits(g[6]) | (bf16_bits(g[7]) << 16);
              __stcs(reinterpret_cast<uint4 *>(grow + v), o);
            } else {
#pragma unroll
              for (int e = 0; e < kPer; ++e) grow[v + e] = (uint16_t)bf16_bits(g[e]);
            }
          }
        }
      }
    }
    for (int i = tid; i < nrest; i += kTtsThreads) {
      const int v = i < nh ? i : v1 + (i - nh);
      float g;
      element(E::scalar(trow, v), E::scalar(drow, v), g);
      if (grow) grow[v] = (uint16_t)bf16_bits(g);
    }
    acc = warp_sum(acc);
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

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status_t sv_tts_signal(int B, int K, int V, sv_dtype_t dtype, const void *target_logits,
                                     const void *draft_logits, const float *temperature, const float *weights,
                                     float *out_kl, uint16_t *out_grad, void *stream) {
  if (B < 0 || B > (1 << 20) || K < 0 || K > SV_MAX_K || V < 1 || V > SV_MAX_V) return SV_ERR_INVALID;
  if (dtype != SV_BF16 && dtype != SV_FP32) return SV_ERR_INVALID;
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
  const int grid = (int)(pairs < sms ? pairs : sms);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16) tts_kernel<SV_BF16><<<grid, kTtsThreads, 0, st>>>(P);
  else tts_kernel<SV_FP32><<<grid, kTtsThreads, 0, st>>>(P);
  return host_cuda_status(cudaGetLastError());
}
