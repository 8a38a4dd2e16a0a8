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
#include <mutex>

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
// the same with packed fp32x2 arithmetic (pairs of elements per instruction)
template <typename E>
__device__ __forceinline__ void online_add_vec2(Online &o, const uint4 &x, float c) {
  float vm = E::get(x, 0);
#pragma unroll
  for (int e = 1; e < E::kPer; ++e) vm = fmaxf(vm, E::get(x, e));
  if (vm > o.m) online_raise(o, vm, c);
  if (o.m > -INFINITY) {
    const float2 cc = make_float2(c, c), nb = make_float2(o.nbh, o.nbh);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E::kPer; e += 2) {
      float2 t = __ffma2_rn(make_float2(E::get(x, e), E::get(x, e + 1)), cc, nb);
      t.x = ex2_approx(t.x);
      t.y = ex2_approx(t.y);
      acc = __fadd2_rn(acc, t);
    }
    o.s += acc.x + acc.y;
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
    const PairConst pc = pair_constants(mt, md, tau);
    const float K0h = pc.K0h, K0l = pc.K0l, invh = pc.invh, invl = pc.invl;

    // ---- pass 2: KL terms and the gradient
    // log2 p_v = z_t c + at, log2 q_v = z_d c + ad (one FMA each)
    const float at = -fmaf(Mt, c, l2St), ad = -fmaf(Md, c, l2Sd);
    const float wg = w * invtau;
    float acc = 0.f;
    // Per element: d = ln p - ln q; the KL term p (e^-d - 1 + d) and the
    // gradient w (q - p) / tau = w p (e^-d - 1) / tau.  For |d| < 1/4 both
    // come from series in d (no cancellation), else from e^-d directly.
    auto element = [&](float zt, float zd, float &g) {
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
      acc += p > 0.f ? p * phi : q;
      g = wg * (p > 0.f ? p * em1 : q);
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
      element(E::scalar(trow, v), E::scalar(drow, v), g);
      if (grow) grow[v] = bf16_rn(g);
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

// ---------------------------------------------------------------------------
// Cluster kernel: the CTAs of one cluster share a row pair, each holding a
// slice of both rows in shared memory, so the second pass reads shared
// memory instead of re-reading the rows.  Each slice is loaded by TMA bulk
// copies in kTtsChunks chunks with one mbarrier each; as soon as the second
// pass has finished a chunk, the same chunk of the next pair is requested,
// so loads overlap compute with a single buffer.  Slice statistics are
// exchanged through distributed shared memory (one cluster barrier per
// pair); the KL partials of pair i are summed by rank 0 after the next
// pair's barrier.  Rows must be 16-byte aligned with V * esz a multiple of 16
// (the host falls back to tts_kernel otherwise).
// ---------------------------------------------------------------------------
constexpr int kTtsChunks = 4;

struct ClusterSmem {
  uint64_t full[kTtsChunks];
  float4 stats[2];   // this CTA's slice statistics (m_t, S_t, m_d, S_d) of even / odd pairs
  float4 klpart[2];  // this CTA's KL partial of pairs of even / odd order (x), abort mark (y)
  MS wt[kTtsWarps], wd[kTtsWarps];
  float wk[kTtsWarps];
  int abort;
  uint32_t status;  // timeout bit of a bounded wait (the pair's KL is then NaN)
};

template <int kDtype>
__global__ void __launch_bounds__(kTtsThreads, 1) tts_cluster_kernel(const TtsParams P, int S) {
  using E = TtsElems<kDtype>;
  constexpr int kEsz = kDtype == SV_BF16 ? 2 : 4;
  constexpr int kPer = E::kPer;
  extern __shared__ __align__(128) uint8_t tts_smem[];
  ClusterSmem &C = *reinterpret_cast<ClusterSmem *>(tts_smem);
  uint8_t *buf = tts_smem + ((sizeof(ClusterSmem) + 127) / 128) * 128;
  const size_t slice_bytes = (size_t)S * kEsz;  // target slice, then draft slice
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V, K = P.K;
  const uint32_t rank = cluster_ctarank();
  const int cs = (int)(gridDim.x / ncluster_x());
  const int cid = (int)cluster_id_x(), ncl = (int)ncluster_x();
  const int npairs = P.B * K;
  const int e0 = (int)rank * S, e1 = min(V, e0 + S);
  const int nel = max(0, e1 - e0);
  const int nvec = nel / kPer;                                 // 16-byte vectors of the slice
  const int cvec = (nvec + kTtsChunks - 1) / kTtsChunks;       // vectors per chunk

  if (tid == 0) {
    for (int ch = 0; ch < kTtsChunks; ++ch) mbar_init(&C.full[ch], 1);
    C.abort = 0;
    C.status = 0;
    C.klpart[0] = C.klpart[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    fence_barrier_init();
  }
  __syncthreads();

  // thread 0: request chunk ch of the it-th pair of this cluster
  auto issue = [&](int it, int ch) {
    const int pair = cid + it * ncl;
    if (pair >= npairs) return;
    const int b = pair / K, k = pair - b * K;
    const int v0 = min(nvec, ch * cvec), v1 = min(nvec, v0 + cvec);
    const uint32_t bytes = (uint32_t)(v1 - v0) * 16u;
    mbar_arrive_expect_tx(&C.full[ch], 2 * bytes);
    if (bytes) {
      const char *trow = reinterpret_cast<const char *>(P.target) + ((size_t)b * (K + 1) + k) * (size_t)V * kEsz;
      const char *drow = reinterpret_cast<const char *>(P.draft) + ((size_t)b * K + k) * (size_t)V * kEsz;
      const size_t off = (size_t)e0 * kEsz + (size_t)v0 * 16;
      bulk_g2s(buf + (size_t)v0 * 16, trow + off, bytes, &C.full[ch]);
      bulk_g2s(buf + slice_bytes + (size_t)v0 * 16, drow + off, bytes, &C.full[ch]);
    }
  };
  if (tid == 0)
    for (int ch = 0; ch < kTtsChunks; ++ch) issue(0, ch);

  volatile int *abort_flag = &C.abort;
  const uint4 *tv = reinterpret_cast<const uint4 *>(buf);
  const uint4 *dv = reinterpret_cast<const uint4 *>(buf + slice_bytes);
  int it = 0, prev_b = -1, prev_k = 0;
  float prev_w = 0.f;
  for (int pair = cid; pair < npairs; pair += ncl, ++it) {
    const int b = pair / K, k = pair - b * K;
    const float tau_in = __ldg(P.temperature + b);
    const float tau = tau_in > 0.f ? tau_in : 1.f;
    const float c = kLog2e / tau;
    const float w = __ldg(P.weights + k);
    const uint32_t parity = (uint32_t)(it & 1);

    // ---- pass 1: slice statistics, chunk by chunk as the copies land
    Online ot = online_init(), od = online_init();
    for (int ch = 0; ch < kTtsChunks; ++ch) {
      if (!*abort_flag) mbar_wait_bounded(&C.full[ch], parity, abort_flag, &C.status, 2000000000ull);
      if (*abort_flag) break;
      const int v0 = min(nvec, ch * cvec), v1 = min(nvec, v0 + cvec);
      for (int j = v0 + tid; j < v1; j += kTtsThreads) {
        online_add_vec2<E>(ot, tv[j], c);
        online_add_vec2<E>(od, dv[j], c);
      }
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
      C.wt[warp] = mt;
      C.wd[warp] = md;
    }
    __syncthreads();
    if (tid == 0) {
      MS a = C.wt[0], d = C.wd[0];
      for (int i = 1; i < kTtsWarps; ++i) {
        a = ms_merge(a, C.wt[i], c);
        d = ms_merge(d, C.wd[i], c);
      }
      C.stats[it & 1] = make_float4(a.m, a.S, d.m, d.S);
    }
    // every slice's statistics of this pair, and every KL partial of the
    // previous pair, are published
    cluster_sync();
    if (rank == 0 && tid == 0 && prev_b >= 0) {
      float sum = 0.f, bad = 0.f;
      for (int r = 0; r < cs; ++r) {
        const float4 v = ld_shared_cluster_f4(mapa_shared(&C.klpart[(it - 1) & 1], (uint32_t)r));
        sum += v.x;
        bad += v.y;
      }
      P.out_kl[(size_t)prev_b * K + prev_k] = bad > 0.f ? __int_as_float(0x7fc00000) : prev_w * sum;
    }
    mt = {-INFINITY, 0.f};
    md = {-INFINITY, 0.f};
    for (int r = 0; r < cs; ++r) {  // rank order: identical in every CTA
      const float4 v = ld_shared_cluster_f4(mapa_shared(&C.stats[it & 1], (uint32_t)r));
      mt = ms_merge(mt, MS{v.x, v.y}, c);
      md = ms_merge(md, MS{v.z, v.w}, c);
    }
    const PairConst pc = pair_constants(mt, md, tau);
    const float at = -fmaf(mt.m, c, log2f(mt.S)), ad = -fmaf(md.m, c, log2f(md.S));
    const float wg = w * pc.invh;
    const bool ok = !*abort_flag;
    // packed constants; the lo parts of 1/tau and K0 move d by at most a few
    // fp32 ulps of |z_t - z_d| / tau, i.e. the gradient by that times p_v
    const float2 cc2 = make_float2(c, c), at2 = make_float2(at, at), invh2 = make_float2(pc.invh, pc.invh);
    const float2 nK0 = make_float2(-(pc.K0h + pc.K0l), -(pc.K0h + pc.K0l)), neg1 = make_float2(-1.f, -1.f);
    const float2 c120 = make_float2(-1.f / 120.f, -1.f / 120.f), c24 = make_float2(1.f / 24.f, 1.f / 24.f);
    const float2 c6 = make_float2(-1.f / 6.f, -1.f / 6.f), half2 = make_float2(0.5f, 0.5f);
    const float2 nlog2e = make_float2(-kLog2e, -kLog2e), wg2 = make_float2(wg, wg);
    float2 acc2 = make_float2(0.f, 0.f);

    // ---- pass 2: KL terms and the gradient from shared memory, chunk by
    // chunk; each finished chunk is handed to the next pair's copy
    uint16_t *grow = P.out_grad ? P.out_grad + ((size_t)b * K + k) * (size_t)V + e0 : nullptr;
    for (int ch = 0; ch < kTtsChunks; ++ch) {
      const int v0 = min(nvec, ch * cvec), v1 = min(nvec, v0 + cvec);
      if (ok)
        for (int j = v0 + tid; j < v1; j += kTtsThreads) {
          const uint4 xt = tv[j], xd = dv[j];
          float g[kPer];
#pragma unroll
          for (int e = 0; e < kPer; e += 2) {
            // two elements per instruction; d = ln p - ln q, p e^-d = q
            const float2 zt = make_float2(E::get(xt, e), E::get(xt, e + 1));
            const float2 zd = make_float2(E::get(xd, e), E::get(xd, e + 1));
            float2 p = __ffma2_rn(zt, cc2, at2);
            p.x = ex2_approx(p.x);
            p.y = ex2_approx(p.y);
            const float2 d = __ffma2_rn(__ffma2_rn(zd, neg1, zt), invh2, nK0);
            float2 poly = __ffma2_rn(d, c120, c24);
            poly = __ffma2_rn(d, poly, c6);
            poly = __ffma2_rn(d, poly, half2);
            const float2 phi_s = __fmul2_rn(__fmul2_rn(d, d), poly);  // e^-d - 1 + d, small |d|
            float2 ex = __fmul2_rn(d, nlog2e);
            ex.x = ex2_approx(ex.x);
            ex.y = ex2_approx(ex.y);
            const float2 em1 = __fadd2_rn(ex, neg1);  // e^-d - 1
            const float2 phl = __fadd2_rn(em1, d);
            const float2 phi = make_float2(fabsf(d.x) < 0.25f ? phi_s.x : phl.x, fabsf(d.y) < 0.25f ? phi_s.y : phl.y);
            float2 tkl = __fmul2_rn(p, phi), tg = __fmul2_rn(p, em1);
            if (!(p.x > 0.f) || !(p.y > 0.f)) {  // z_t = -inf: the limits of both terms are q
              if (!(p.x > 0.f)) tkl.x = tg.x = ex2_approx(fmaf(zd.x, c, ad));
              if (!(p.y > 0.f)) tkl.y = tg.y = ex2_approx(fmaf(zd.y, c, ad));
            }
            acc2 = __fadd2_rn(acc2, tkl);
            const float2 gg = __fmul2_rn(wg2, tg);
            g[e] = gg.x;
            g[e + 1] = gg.y;
          }
          if (grow) {
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
        }
      __syncthreads();  // chunk ch is no longer read
      if (tid == 0 && !*abort_flag) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(it + 1, ch);
      }
    }
    const float acc = warp_sum(acc2.x + acc2.y);
    if (lane == 0) C.wk[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      float sum = 0.f;
      for (int i = 0; i < kTtsWarps; ++i) sum += C.wk[i];
      C.klpart[it & 1] = make_float4(sum, ok ? 0.f : 1.f, 0.f, 0.f);
    }
    prev_b = b;
    prev_k = k;
    prev_w = w;
  }
  cluster_sync();  // the last pair's KL partials are published
  if (rank == 0 && tid == 0 && prev_b >= 0) {
    float sum = 0.f, bad = 0.f;
    for (int r = 0; r < cs; ++r) {
      const float4 v = ld_shared_cluster_f4(mapa_shared(&C.klpart[(it - 1) & 1], (uint32_t)r));
      sum += v.x;
      bad += v.y;
    }
    P.out_kl[(size_t)prev_b * K + prev_k] = bad > 0.f ? __int_as_float(0x7fc00000) : prev_w * sum;
  }
  cluster_sync();  // no CTA leaves while rank 0 may still read its shared memory
  if (tid == 0 && *abort_flag) {  // copies still in flight: wait for them (bounded)
    const uint64_t t0 = global_ns();
    for (int ch = 0; ch < kTtsChunks; ++ch)
      while (!mbar_try_wait(&C.full[ch], (uint32_t)(it & 1)) && global_ns() - t0 < 2000000000ull) {
      }
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

namespace {
// Cluster configuration for one (V, element size): the cluster size with the
// most SMs resident, slices of S elements, one or two buffers.
struct TtsCfg {
  int cs, S, nbuf, clusters;
  size_t smem;
};

bool tts_cluster_cfg_uncached(int V, int esz, int dtype, TtsCfg *out) {
  const size_t kSmemMax = 220 * 1024;
  const size_t head = ((sizeof(ClusterSmem) + 127) / 128) * 128;
  TtsCfg best{0, 0, 0, 0, 0};
  for (int cs : {8, 4, 2}) {
    const int unit = 16 / esz;
    const int S = ((V + cs - 1) / cs + unit - 1) / unit * unit;
    const size_t smem = head + 2 * (size_t)S * esz;
    if (smem > kSmemMax) continue;
    const void *fn = dtype == SV_BF16 ? (const void *)tts_cluster_kernel<SV_BF16> : (const void *)tts_cluster_kernel<SV_FP32>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(kTtsThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cs;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (ncl * cs > best.clusters * best.cs) best = TtsCfg{cs, S, 1, ncl, smem};
  }
  if (!best.cs) return false;
  *out = best;
  return true;
}

// small per-process cache keyed by (device, V, dtype)
std::mutex g_tts_mu;
struct TtsCacheEnt {
  int dev, V, dtype, ok;
  TtsCfg cfg;
};
TtsCacheEnt g_tts_cache[16];
int g_tts_n = 0;

bool tts_cluster_cfg(int V, int esz, int dtype, TtsCfg *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(g_tts_mu);
  for (int i = 0; i < g_tts_n; ++i)
    if (g_tts_cache[i].dev == dev && g_tts_cache[i].V == V && g_tts_cache[i].dtype == dtype) {
      *out = g_tts_cache[i].cfg;
      return g_tts_cache[i].ok != 0;
    }
  TtsCfg cfg{};
  const bool ok = tts_cluster_cfg_uncached(V, esz, dtype, &cfg);
  TtsCacheEnt &e = g_tts_cache[g_tts_n < 16 ? g_tts_n++ : 15];
  e = TtsCacheEnt{dev, V, dtype, ok ? 1 : 0, cfg};
  *out = cfg;
  return ok;
}
}  // namespace

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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the cluster path wants 16-byte aligned rows and slices
  const bool aligned16 = ((size_t)V * esz) % 16 == 0 && host_aligned(target_logits, 16) &&
                         host_aligned(draft_logits, 16) && (!out_grad || (host_aligned(out_grad, 16) && V % 8 == 0));
  TtsCfg cfg;
  if (aligned16 && tts_cluster_cfg(V, esz, (int)dtype, &cfg)) {
    long long ncl = (pairs < cfg.clusters) ? pairs : cfg.clusters;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(ncl * cfg.cs), 1, 1);
    lc.blockDim = dim3(kTtsThreads, 1, 1);
    lc.dynamicSmemBytes = cfg.smem;
    lc.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cfg.cs;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    lc.attrs = &attr;
    lc.numAttrs = 1;
    cudaError_t e = dtype == SV_BF16 ? cudaLaunchKernelEx(&lc, tts_cluster_kernel<SV_BF16>, P, cfg.S)
                                     : cudaLaunchKernelEx(&lc, tts_cluster_kernel<SV_FP32>, P, cfg.S);
    return host_cuda_status(e);
  }
  const int grid = (int)(pairs < sms ? pairs : sms);
  if (dtype == SV_BF16) tts_kernel<SV_BF16><<<grid, kTtsThreads, 0, st>>>(P);
  else tts_kernel<SV_FP32><<<grid, kTtsThreads, 0, st>>>(P);
  return host_cuda_status(cudaGetLastError());
}
