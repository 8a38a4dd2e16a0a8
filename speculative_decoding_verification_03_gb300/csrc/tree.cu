// Acceptance walk over a token tree ("Accelerating Sonar through
// Speculation", section "EAGLE": several draft branches verified in one
// target pass, the best-fitting branch kept plus one target token; the rule
// at each node is the cheatsheet's "one speculative step": accept with
// probability min(1, p/q), resample the normalised positive residual).
//
// One CTA per request.  At the current node c the CTA takes the online
// statistics of target row c and draft row c (one pass), then tries c's
// children in ascending order: child j with token x is accepted iff
// u_j < p_j(x) / q(x), where p_0 = p and, after each rejected child,
// p_{j+1} = max(p_j - q, 0) / R_{j+1} (one pass to get R_{j+1}).  An accepted
// child becomes the current node.  When no child is accepted (or c is a
// leaf) one token is drawn from the last p_j by inverting its CDF in
// ascending token order: per-warp segment sums, then one warp walks the
// crossing segment in 256-token chunks.  Greedy rows (tau <= 0) follow the
// target argmax.
#include <cfloat>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreeChunk = 256;  // tokens per lane-pass of the final draw (8 per lane)
constexpr int kTreeMaxChildren = SV_TREE_MAX_NODES - 1;

struct TreeParams {
  int B, N, V, dtype;
  const void *target, *draft;  // [B][N][V]
  const int32_t *tokens, *parents, *n_nodes;
  const float *temperature;
  uint64_t seed;
  int32_t *out_tokens, *out_accept_len, *out_path;
  uint32_t *out_flags;
};

__device__ __forceinline__ float logit(const void *row, int dtype, int v) {
  if (dtype == SV_BF16) return __uint_as_float(((uint32_t)__ldcg(reinterpret_cast<const unsigned short *>(row) + v)) << 16);
  return __ldcg(reinterpret_cast<const float *>(row) + v);
}

// Eight consecutive logits v .. v+7 (v a multiple of 8) of a row: one or two
// 16-byte loads when the row is 16-byte aligned, else plain loads; tokens at
// or beyond V read as -inf.
__device__ __forceinline__ void load8(const void *row, int dtype, int V, int v, bool vec, float (&z)[8]) {
  if (vec && v + 8 <= V) {
    if (dtype == SV_BF16) {
      const uint4 w = __ldcg(reinterpret_cast<const uint4 *>(row) + (v >> 3));
      z[0] = bf16lo(w.x); z[1] = bf16hi(w.x); z[2] = bf16lo(w.y); z[3] = bf16hi(w.y);
      z[4] = bf16lo(w.z); z[5] = bf16hi(w.z); z[6] = bf16lo(w.w); z[7] = bf16hi(w.w);
    } else {
      const uint4 a = __ldcg(reinterpret_cast<const uint4 *>(row) + (v >> 2));
      const uint4 b = __ldcg(reinterpret_cast<const uint4 *>(row) + (v >> 2) + 1);
      z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y); z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
      z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y); z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = v + e < V ? logit(row, dtype, v + e) : -INFINITY;
  }
}

struct Online {
  float m, s;
};
__device__ __forceinline__ void online_add(Online &o, float z, float c) {
  if (z > o.m) {
    o.s = o.s * ex2_approx((o.m - z) * c) + 1.f;
    o.m = z;
  } else if (z > -INFINITY) {
    o.s += ex2_approx((z - o.m) * c);
  }
}
__device__ __forceinline__ Online online_merge(Online a, Online b, float c) {
  if (b.m > a.m) {
    const Online t = a;
    a = b;
    b = t;
  }
  if (b.m == -INFINITY) return a;
  a.s += b.s * ex2_approx((b.m - a.m) * c);
  return a;
}

struct NodeDist {
  float c, Mt, Md, inv_St, inv_Sd;
  const void *trow, *drow;
  int dtype;
  // residual chain: p_0 = p; p_{j+1} = max(p_j - q, 0) * invR[j]
  int nrej;
  float invR[kTreeMaxChildren];
  __device__ __forceinline__ float p0z(float zt) const { return ex2_approx((zt - Mt) * c) * inv_St; }
  __device__ __forceinline__ float qz(float zd) const { return ex2_approx((zd - Md) * c) * inv_Sd; }
  __device__ __forceinline__ float p0(int v) const { return p0z(logit(trow, dtype, v)); }
  __device__ __forceinline__ float q(int v) const { return qz(logit(drow, dtype, v)); }
  // p_j(v) for j = nrej (the current residual) and the un-normalised
  // max(p_j - q, 0) for the next step
  __device__ __forceinline__ float pj(int v, float qv) const { return pjz(logit(trow, dtype, v), qv); }
  __device__ __forceinline__ float pjz(float zt, float qv) const {
    float r = p0z(zt);
    for (int i = 0; i < nrej; ++i) r = fmaxf(r - qv, 0.f) * invR[i];
    return r;
  }
};

__device__ __forceinline__ float block_sum(float v, float *scratch) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < kTreeWarps; ++i) s += scratch[i];
  return s;
}

__global__ void __launch_bounds__(kTreeThreads, 1) tree_kernel(const TreeParams P) {
  __shared__ int s_kids[kTreeMaxChildren + 1];
  __shared__ int s_nkids;
  __shared__ float s_red[kTreeWarps];
  __shared__ Online s_on_t[kTreeWarps], s_on_d[kTreeWarps];
  __shared__ double s_seg[kTreeWarps];
  __shared__ int s_bad, s_tok;
  __shared__ float s_bv[kTreeWarps];
  __shared__ int s_bi[kTreeWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = P.N, V = P.V;
  const int esz = P.dtype == SV_BF16 ? 2 : 4;
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    const int32_t *par = P.parents + (size_t)b * N;
    const int32_t *tok = P.tokens + (size_t)b * N;
    int32_t *out = P.out_tokens + (size_t)b * N;
    int32_t *path = P.out_path ? P.out_path + (size_t)b * (N > 1 ? N - 1 : 1) : nullptr;
    int nb = P.n_nodes ? __ldg(P.n_nodes + b) : N;
    if (tid == 0) s_bad = (nb < 1 || nb > N) ? 1 : 0;
    __syncthreads();
    if (!s_bad)
      for (int n = 1 + tid; n < nb; n += kTreeThreads) {
        const int pn = __ldg(par + n);
        if (pn < 0 || pn >= n) s_bad = 1;
      }
    for (int j = tid; j < N; j += kTreeThreads) out[j] = -1;
    if (path)
      for (int j = tid; j < (N > 1 ? N - 1 : 1); j += kTreeThreads) path[j] = -1;
    __syncthreads();
    uint32_t flags = 0;
    if (s_bad) {
      if (tid == 0) {
        P.out_accept_len[b] = 0;
        if (P.out_flags) P.out_flags[b] = SV_TREE_BAD;
      }
      __syncthreads();
      continue;
    }
    const float tau_in = __ldg(P.temperature + b);
    const bool greedy = !(tau_in > 0.f);
    const float c = greedy ? kLog2e : kLog2e / tau_in;
    int cur = 0, depth = 0;
    for (;;) {
      // children of cur, ascending
      if (warp == 0) {
        int cnt = 0;
        for (int base = 1; base < nb; base += 32) {
          const int n = base + lane;
          const bool is_kid = n < nb && __ldg(par + n) == cur;
          const unsigned m = __ballot_sync(0xffffffffu, is_kid);
          if (is_kid) {
            const int slot = cnt + __popc(m & ((1u << lane) - 1u));
            if (slot < kTreeMaxChildren) s_kids[slot] = n;
          }
          cnt += __popc(m);
        }
        if (lane == 0) s_nkids = min(cnt, kTreeMaxChildren);
      }
      __syncthreads();
      const int nk = s_nkids;
      const void *trow = reinterpret_cast<const char *>(P.target) + ((size_t)b * N + cur) * (size_t)V * esz;
      const void *drow = reinterpret_cast<const char *>(P.draft) + ((size_t)b * N + cur) * (size_t)V * esz;
      const bool vec = ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(drow)) & 15) == 0;
      const int noct = (V + 7) >> 3;  // groups of 8 consecutive tokens
      int next = -1;
      if (greedy) {
        // argmax of target row cur (lowest index on ties)
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int o = tid; o < noct; o += kTreeThreads) {
          float z[8];
          load8(trow, P.dtype, V, o << 3, vec, z);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (z[e] > bv) {
              bv = z[e];
              bi = (o << 3) + e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (lane == 0) {
          s_bv[warp] = bv;
          s_bi[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
          float v = s_bv[0];
          int i = s_bi[0];
          for (int w = 1; w < kTreeWarps; ++w)
            if (s_bv[w] > v || (s_bv[w] == v && s_bi[w] < i)) {
              v = s_bv[w];
              i = s_bi[w];
            }
          s_tok = i == INT_MAX ? 0 : i;
        }
        __syncthreads();
        const int best = s_tok;
        for (int j = 0; j < nk; ++j)
          if (__ldg(tok + s_kids[j]) == best) {
            next = s_kids[j];
            break;
          }
        if (next < 0) {
          if (tid == 0) out[depth] = best;
          break;
        }
      } else {
        // statistics of both rows
        Online ot = {-INFINITY, 0.f}, od = {-INFINITY, 0.f};
        for (int o = tid; o < noct; o += kTreeThreads) {
          float zt[8], zd[8];
          load8(trow, P.dtype, V, o << 3, vec, zt);
          load8(drow, P.dtype, V, o << 3, vec, zd);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            online_add(ot, zt[e], c);
            online_add(od, zd[e], c);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const Online a = {__shfl_xor_sync(0xffffffffu, ot.m, o), __shfl_xor_sync(0xffffffffu, ot.s, o)};
          const Online d = {__shfl_xor_sync(0xffffffffu, od.m, o), __shfl_xor_sync(0xffffffffu, od.s, o)};
          ot = online_merge(ot, a, c);
          od = online_merge(od, d, c);
        }
        if (lane == 0) {
          s_on_t[warp] = ot;
          s_on_d[warp] = od;
        }
        __syncthreads();
        ot = s_on_t[0];
        od = s_on_d[0];
        for (int i = 1; i < kTreeWarps; ++i) {
          ot = online_merge(ot, s_on_t[i], c);
          od = online_merge(od, s_on_d[i], c);
        }
        NodeDist D;
        D.c = c;
        D.Mt = ot.m;
        D.Md = od.m;
        D.inv_St = 1.f / ot.s;
        D.inv_Sd = 1.f / od.s;
        D.trow = trow;
        D.drow = drow;
        D.dtype = P.dtype;
        D.nrej = 0;
        for (int j = 0; j < nk; ++j) {
          const int child = s_kids[j];
          const int x = __ldg(tok + child);
          // acceptance test of child j (every thread computes it identically)
          float ratio = 0.f;
          if (x >= 0 && x < V) {
            const float qx = D.q(x);
            const float px = D.pj(x, qx);
            ratio = qx > 0.f ? px / qx : INFINITY;
          }
          const U32x4 r = philox4x32_10((uint32_t)b, (uint32_t)depth, (uint32_t)j, 0u, (uint32_t)(P.seed & 0xffffffffu),
                                        (uint32_t)(P.seed >> 32));
          const float u = (float)(r.w[0] >> 8) * (1.0f / 16777216.0f);
          if (u < ratio) {
            next = child;
            break;
          }
          // rejected: the residual's mass R_{j+1}
          float part = 0.f;
          for (int o = tid; o < noct; o += kTreeThreads) {
            float zt[8], zd[8];
            load8(trow, P.dtype, V, o << 3, vec, zt);
            load8(drow, P.dtype, V, o << 3, vec, zd);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float qv = D.qz(zd[e]);
              part += fmaxf(D.pjz(zt[e], qv) - qv, 0.f);
            }
          }
          const float R = block_sum(part, s_red);
          if (R > 0.f && D.nrej < kTreeMaxChildren) {
            D.invR[D.nrej] = 1.f / R;
            ++D.nrej;
          } else {
            flags |= SV_TREE_ZERO_RESIDUAL;
          }
        }
        if (next < 0) {
          // draw from the current p_j: per-warp segment sums, then the
          // crossing segment walked in 256-token chunks by one warp
          const U32x4 r = philox4x32_10((uint32_t)b, (uint32_t)depth, 0u, 0u, (uint32_t)(P.seed & 0xffffffffu),
                                        (uint32_t)(P.seed >> 32));
          const float u = (float)(r.w[1] >> 8) * (1.0f / 16777216.0f);
          const int seg = (V + kTreeWarps * kTreeChunk - 1) / (kTreeWarps * kTreeChunk) * kTreeChunk;
          const int s0 = min(V, warp * seg), s1 = min(V, s0 + seg);
          float ws = 0.f;
          for (int v = s0 + lane * 8; v < s1; v += 256) {
            float zt[8], zd[8];
            load8(trow, P.dtype, s1, v, vec, zt);
            load8(drow, P.dtype, s1, v, vec, zd);
#pragma unroll
            for (int e = 0; e < 8; ++e) ws += D.pjz(zt[e], D.qz(zd[e]));
          }
          ws = warp_sum(ws);
          __syncthreads();
          if (lane == 0) s_seg[warp] = (double)ws;
          __syncthreads();
          if (warp == 0) {
            double tot = 0.0;
            for (int w = 0; w < kTreeWarps; ++w) tot += s_seg[w];
            const double T = (double)u * tot;
            double run = 0.0;
            int wseg = -1, last = -1;
            for (int w = 0; w < kTreeWarps; ++w) {
              if (s_seg[w] > 0.0) last = w;
              if (wseg < 0 && run + s_seg[w] > T) wseg = w;
              if (wseg < 0) run += s_seg[w];
            }
            if (wseg < 0) {  // u * R at the total by rounding: the last segment with mass
              wseg = last < 0 ? 0 : last;
              run = tot - (last < 0 ? 0.0 : s_seg[wseg]);
            }
            const int a0 = min(V, wseg * seg), a1 = min(V, a0 + seg);
            int found = -1, lastv = -1;
            for (int cb = a0; cb < a1 && found < 0; cb += kTreeChunk) {
              float pr[8], zt[8], zd[8];
              float lsum = 0.f;
              load8(trow, P.dtype, a1, cb + lane * 8, vec, zt);
              load8(drow, P.dtype, a1, cb + lane * 8, vec, zd);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int v = cb + lane * 8 + e;
                pr[e] = v < a1 ? D.pjz(zt[e], D.qz(zd[e])) : 0.f;
                lsum += pr[e];
                if (pr[e] > 0.f) lastv = max(lastv, v);
              }
              // inclusive prefix of the lane sums across the warp (fp64)
              double incl = (double)lsum;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const double n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
              }
              double pre = run + incl - (double)lsum;
              int cand = INT_MAX;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                pre += (double)pr[e];
                if (cand == INT_MAX && pr[e] > 0.f && pre > T) cand = cb + lane * 8 + e;
              }
              cand = warp_min_i(cand);
              if (cand != INT_MAX) found = cand;
              run += __shfl_sync(0xffffffffu, incl, 31);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lastv = max(lastv, __shfl_xor_sync(0xffffffffu, lastv, o));
            if (lane == 0) s_tok = found >= 0 ? found : (lastv >= 0 ? lastv : 0);
          }
          __syncthreads();
          if (tid == 0) out[depth] = s_tok;
          break;
        }
      }
      if (tid == 0) {
        out[depth] = __ldg(tok + next);
        if (path) path[depth] = next;
      }
      cur = next;
      ++depth;
      __syncthreads();
    }
    if (tid == 0) {
      P.out_accept_len[b] = depth;
      if (P.out_flags) P.out_flags[b] = flags;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status_t sv_verify_tree(int B, int N, int V, sv_dtype_t dtype, const void *target_logits,
                                      const void *draft_logits, const int32_t *tokens, const int32_t *parents,
                                      const int32_t *n_nodes, const float *temperature, uint64_t seed,
                                      int32_t *out_tokens, int32_t *out_accept_len, int32_t *out_path,
                                      uint32_t *out_flags, void *stream) {
  if (B < 0 || B > (1 << 20) || N < 1 || N > SV_TREE_MAX_NODES || V < 1 || V > SV_MAX_V) return SV_ERR_INVALID;
  if (dtype != SV_BF16 && dtype != SV_FP32) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !tokens || !parents || !temperature || !out_tokens || !out_accept_len)
    return SV_ERR_INVALID;
  const int esz = dtype == SV_BF16 ? 2 : 4;
  if (!host_aligned(target_logits, esz) || !host_aligned(draft_logits, esz)) return SV_ERR_INVALID;
  const void *ptrs[] = {tokens, parents, n_nodes, temperature, out_tokens, out_accept_len, out_path, out_flags};
  for (const void *p : ptrs)
    if (!host_aligned(p, 4)) return SV_ERR_INVALID;
  int sms = 0;
  const sv_status_t ds = host_device_info(&sms);
  if (ds != SV_OK) return ds;
  TreeParams P{B, N, V, (int)dtype, target_logits, draft_logits, tokens, parents, n_nodes, temperature, seed,
               out_tokens, out_accept_len, out_path, out_flags};
  const int grid = B < 2 * sms ? B : 2 * sms;
  tree_kernel<<<grid, kTreeThreads, 0, static_cast<cudaStream_t>(stream)>>>(P);
  return host_cuda_status(cudaGetLastError());
}
