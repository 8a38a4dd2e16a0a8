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

#include "sample_common.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreeChunk = 256;  // tokens per lane-pass of the final draw (8 per lane)
constexpr int kTreeMaxChildren = SV_TREE_MAX_NODES - 1;
constexpr int kTreeMaxChunkSums = 32;  // 256-token chunk sums a warp keeps for the staged draw

struct TreeParams {
  int B, N, V, dtype;
  const void *target, *draft;  // [B][N][V]
  const int32_t *tokens, *parents, *n_nodes;
  const float *temperature;
  uint64_t seed;
  int32_t *out_tokens, *out_accept_len, *out_path;
  uint32_t *out_flags;
};

// Row reads: from global memory (L2, .cg) or, when the node's rows were
// staged (kS), from shared memory through generic addresses.
template <bool kS>
__device__ __forceinline__ uint4 ld16(const uint4 *p) {
  if (kS) return *p;
  return __ldcg(p);
}
template <bool kS>
__device__ __forceinline__ float logit(const void *row, int dtype, int v) {
  if (dtype == SV_BF16) {
    const unsigned short *r = reinterpret_cast<const unsigned short *>(row) + v;
    return __uint_as_float(((uint32_t)(kS ? *r : __ldcg(r))) << 16);
  }
  const float *r = reinterpret_cast<const float *>(row) + v;
  return kS ? *r : __ldcg(r);
}

// Eight consecutive logits v .. v+7 (v a multiple of 8) of a row: one or two
// 16-byte loads when the row is 16-byte aligned, else plain loads; tokens at
// or beyond V read as -inf.
template <bool kS>
__device__ __forceinline__ void load8(const void *row, int dtype, int V, int v, bool vec, float (&z)[8]) {
  if (vec && v + 8 <= V) {
    if (dtype == SV_BF16) {
      const uint4 w = ld16<kS>(reinterpret_cast<const uint4 *>(row) + (v >> 3));
      z[0] = bf16lo(w.x); z[1] = bf16hi(w.x); z[2] = bf16lo(w.y); z[3] = bf16hi(w.y);
      z[4] = bf16lo(w.z); z[5] = bf16hi(w.z); z[6] = bf16lo(w.w); z[7] = bf16hi(w.w);
    } else {
      const uint4 a = ld16<kS>(reinterpret_cast<const uint4 *>(row) + (v >> 2));
      const uint4 b = ld16<kS>(reinterpret_cast<const uint4 *>(row) + (v >> 2) + 1);
      z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y); z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
      z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y); z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = v + e < V ? logit<kS>(row, dtype, v + e) : -INFINITY;
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

template <bool kS>
struct NodeDist {
  float c, Mt, Md, inv_St, inv_Sd;
  const void *trow, *drow;
  int dtype;
  // residual chain p_0 = p, p_{j+1} = max(p_j - q, 0) / R_{j+1}, in closed
  // form: p_j = max(p_0 - a_j q, 0) / Z_j with a_0 = 0, Z_0 = 1,
  // a_{j+1} = a_j + Z_j, Z_{j+1} = Z_j R_{j+1} (by induction: where
  // p_0 <= a_j q both sides are 0; elsewhere p_j - q = (p_0 - (a_j + Z_j) q) / Z_j)
  float a, invZ;
  __device__ __forceinline__ float p0z(float zt) const { return ex2_approx((zt - Mt) * c) * inv_St; }
  __device__ __forceinline__ float qz(float zd) const { return ex2_approx((zd - Md) * c) * inv_Sd; }
  __device__ __forceinline__ float q(int v) const { return qz(logit<kS>(drow, dtype, v)); }
  // p_j(v) for j = nrej (the current residual) and the un-normalised
  // max(p_j - q, 0) for the next step
  __device__ __forceinline__ float pj(int v, float qv) const { return pjz(logit<kS>(trow, dtype, v), qv); }
  __device__ __forceinline__ float pjz(float zt, float qv) const { return fmaxf(fmaf(-a, qv, p0z(zt)), 0.f) * invZ; }
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

template <bool kS>
__global__ void __launch_bounds__(kTreeThreads, 1) tree_kernel(const TreeParams P) {
  extern __shared__ __align__(128) uint8_t tree_smem[];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_abort;
  __shared__ uint32_t s_status;
  uint32_t bar_phase = 0;
  __shared__ int s_kids[kTreeMaxChildren + 1];
  __shared__ int s_par[SV_TREE_MAX_NODES], s_tokn[SV_TREE_MAX_NODES];
  __shared__ float s_csum[kS ? kTreeWarps * kTreeMaxChunkSums : 1];
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
  const uint32_t row_bytes = (uint32_t)P.V * (uint32_t)esz;
  uint8_t *s_trow = tree_smem;
  uint8_t *s_drow = tree_smem + ((row_bytes + 127u) & ~127u);
  if (kS) {
    if (tid == 0) {
      mbar_init(&s_bar, 1);
      s_abort = 0;
      s_status = 0u;
      fence_barrier_init();
    }
    __syncthreads();
  }
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    const int32_t *par = P.parents + (size_t)b * N;
    const int32_t *tok = P.tokens + (size_t)b * N;
    int32_t *out = P.out_tokens + (size_t)b * N;
    int32_t *path = P.out_path ? P.out_path + (size_t)b * (N > 1 ? N - 1 : 1) : nullptr;
    int nb = P.n_nodes ? __ldg(P.n_nodes + b) : N;
    if (tid == 0) s_bad = (nb < 1 || nb > N) ? 1 : 0;
    __syncthreads();
    if (!s_bad)
      for (int n = tid; n < nb; n += kTreeThreads) {
        const int pn = __ldg(par + n);
        s_par[n] = pn;
        s_tokn[n] = __ldg(tok + n);
        if (n >= 1 && (pn < 0 || pn >= n)) s_bad = 1;
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
          const bool is_kid = n < nb && s_par[n] == cur;
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
      bool vec = ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(drow)) & 15) == 0;
      if (kS) {
        // node cur's rows into shared memory (one bulk copy each; the draft
        // row only for sampled rows), then every pass reads them there
        if (tid == 0) {
          // the previous node's reads (generic proxy) before the copies overwrite them
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          const uint32_t bytes = greedy ? row_bytes : 2u * row_bytes;
          mbar_arrive_expect_tx(&s_bar, bytes);
          bulk_g2s(s_trow, trow, row_bytes, &s_bar);
          if (!greedy) bulk_g2s(s_drow, drow, row_bytes, &s_bar);
        }
        // bounded (2 s): a copy that never lands flags the request and stops
        // the CTA (nothing else in flight)
        const bool got = mbar_wait_bounded(&s_bar, bar_phase, &s_abort, &s_status, 2000000000ull);
        if (!__syncthreads_and(got)) {
          if (tid == 0) {
            P.out_accept_len[b] = 0;
            if (P.out_flags) P.out_flags[b] = SV_TREE_BAD;
          }
          return;
        }
        bar_phase ^= 1u;
        trow = s_trow;
        drow = s_drow;
        vec = true;
      }
      const int noct = (V + 7) >> 3;  // groups of 8 consecutive tokens
      int next = -1;
      if (greedy) {
        // argmax of target row cur (lowest index on ties)
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int o = tid; o < noct; o += kTreeThreads) {
          float z[8];
          load8<kS>(trow, P.dtype, V, o << 3, vec, z);
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
          if (s_tokn[s_kids[j]] == best) {
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
        if (kS) {
          // rows in shared memory: the maxima first, then the sums
          float mt = -INFINITY, md = -INFINITY;
          for (int o = tid; o < noct; o += kTreeThreads) {
            float zt[8], zd[8];
            load8<kS>(trow, P.dtype, V, o << 3, vec, zt);
            load8<kS>(drow, P.dtype, V, o << 3, vec, zd);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              mt = fmaxf(mt, zt[e]);
              md = fmaxf(md, zd[e]);
            }
          }
          mt = warp_max(mt);
          md = warp_max(md);
          if (lane == 0) {
            s_on_t[warp].m = mt;
            s_on_d[warp].m = md;
          }
          __syncthreads();
          mt = s_on_t[0].m;
          md = s_on_d[0].m;
          for (int i = 1; i < kTreeWarps; ++i) {
            mt = fmaxf(mt, s_on_t[i].m);
            md = fmaxf(md, s_on_d[i].m);
          }
          // a thread's eight terms summed, then added with compensation (long rows)
          float st = 0.f, sd = 0.f, st_c = 0.f, sd_c = 0.f;
          for (int o = tid; o < noct; o += kTreeThreads) {
            float zt[8], zd[8];
            load8<kS>(trow, P.dtype, V, o << 3, vec, zt);
            load8<kS>(drow, P.dtype, V, o << 3, vec, zd);
            float vt = 0.f, vd = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (mt > -INFINITY) vt += ex2_approx((zt[e] - mt) * c);
              if (md > -INFINITY) vd += ex2_approx((zd[e] - md) * c);
            }
            kahan_add(st, st_c, vt);
            kahan_add(sd, sd_c, vd);
          }
          st = warp_sum(__fsub_rn(st, st_c));
          sd = warp_sum(__fsub_rn(sd, sd_c));
          __syncthreads();  // the maxima are read
          if (lane == 0) {
            s_on_t[warp].s = st;
            s_on_d[warp].s = sd;
          }
          __syncthreads();
          st = 0.f;
          sd = 0.f;
          for (int i = 0; i < kTreeWarps; ++i) {
            st += s_on_t[i].s;
            sd += s_on_d[i].s;
          }
          ot = {mt, st};
          od = {md, sd};
        } else {
        for (int o = tid; o < noct; o += kTreeThreads) {
          float zt[8], zd[8];
          load8<kS>(trow, P.dtype, V, o << 3, vec, zt);
          load8<kS>(drow, P.dtype, V, o << 3, vec, zd);
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
        }
        NodeDist<kS> D;
        D.c = c;
        D.Mt = ot.m;
        D.Md = od.m;
        D.inv_St = 1.f / ot.s;
        D.inv_Sd = 1.f / od.s;
        D.trow = trow;
        D.drow = drow;
        D.dtype = P.dtype;
        D.a = 0.f;
        D.invZ = 1.f;
        for (int j = 0; j < nk; ++j) {
          const int child = s_kids[j];
          const int x = s_tokn[child];
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
          float part = 0.f, part_c = 0.f;
          for (int o = tid; o < noct; o += kTreeThreads) {
            float zt[8], zd[8];
            load8<kS>(trow, P.dtype, V, o << 3, vec, zt);
            load8<kS>(drow, P.dtype, V, o << 3, vec, zd);
            float v8 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float qv = D.qz(zd[e]);
              v8 += fmaxf(D.pjz(zt[e], qv) - qv, 0.f);
            }
            kahan_add(part, part_c, v8);
          }
          const float R = block_sum(__fsub_rn(part, part_c), s_red);
          if (R > 0.f) {
            D.a += 1.f / D.invZ;
            D.invZ /= R;
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
          if (kS && seg / kTreeChunk <= kTreeMaxChunkSums) {
            // rows in shared memory: every 256-token chunk's sum, then one
            // warp finds the crossing chunk (double-float prefix) and walks it
            const int ncw = seg / kTreeChunk;
            for (int ci = 0; ci < ncw; ++ci) {
              const int v = s0 + ci * kTreeChunk + lane * 8;
              float cs = 0.f;
              if (v < s1) {
                float zt[8], zd[8];
                load8<kS>(trow, P.dtype, s1, v, vec, zt);
                load8<kS>(drow, P.dtype, s1, v, vec, zd);
#pragma unroll
                for (int e = 0; e < 8; ++e) cs += v + e < s1 ? D.pjz(zt[e], D.qz(zd[e])) : 0.f;
              }
              cs = warp_sum(cs);
              if (lane == 0) s_csum[warp * ncw + ci] = cs;
            }
            __syncthreads();
            if (warp == 0) {
              const int nc = kTreeWarps * ncw;
              const int q = (nc + 31) / 32;
              const int ja = min(nc, lane * q), jb = min(nc, ja + q);
              DF mine = {0.f, 0.f};
              for (int j = ja; j < jb; ++j) mine = df_add_f(mine, s_csum[j]);
              const DF incl = warp_incl_scan_df(mine, lane);
              DF tot;
              tot.hi = __shfl_sync(0xffffffffu, incl.hi, 31);
              tot.lo = __shfl_sync(0xffffffffu, incl.lo, 31);
              const DF T = df_scale(u, tot);
              DF run = df_add(incl, {-mine.hi, -mine.lo});
              int cand = INT_MAX, lastc = -1;
              DF pe = {0.f, 0.f};
              for (int j = ja; j < jb; ++j) {
                const float sj = s_csum[j];
                if (sj > 0.f) lastc = j;
                const DF nxt = df_add_f(run, sj);
                if (cand == INT_MAX && df_gt(nxt, T)) {
                  cand = j;
                  pe = run;
                }
                run = nxt;
              }
              int jstar = warp_min_i(cand);
              DF pexcl;
              if (jstar != INT_MAX) {
                const int owner = __ffs(__ballot_sync(0xffffffffu, cand == jstar)) - 1;
                pexcl.hi = __shfl_sync(0xffffffffu, pe.hi, owner);
                pexcl.lo = __shfl_sync(0xffffffffu, pe.lo, owner);
              } else {  // u * R at the total by rounding: the last chunk with mass
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lastc = max(lastc, __shfl_xor_sync(0xffffffffu, lastc, o));
                jstar = lastc < 0 ? 0 : lastc;
                pexcl = df_add_f(tot, -s_csum[jstar]);
              }
              // chunk jstar = warp (jstar / ncw)'s chunk (jstar % ncw)
              const int cw = jstar / ncw, cc = jstar - cw * ncw;
              const int c0 = min(V, cw * seg), c1 = min(V, c0 + seg);
              const int v0 = c0 + cc * kTreeChunk + lane * 8;
              float pr[8];
              {
                float zt[8], zd[8];
                load8<kS>(trow, P.dtype, c1, v0, vec, zt);
                load8<kS>(drow, P.dtype, c1, v0, vec, zd);
#pragma unroll
                for (int e = 0; e < 8; ++e) pr[e] = v0 + e < c1 ? D.pjz(zt[e], D.qz(zd[e])) : 0.f;
              }
              float pre[8];
              pre[0] = pr[0];
#pragma unroll
              for (int e = 1; e < 8; ++e) pre[e] = pre[e - 1] + pr[e];
              const DF incl2 = warp_incl_scan_df({pre[7], 0.f}, lane);
              const DF base = df_add(pexcl, df_add_f(incl2, -pre[7]));
              int c2 = INT_MAX, back = -1;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                if (c2 == INT_MAX && pr[e] > 0.f && df_gt(df_add_f(base, pre[e]), T)) c2 = v0 + e;
                if (pr[e] > 0.f) back = v0 + e;
              }
              c2 = warp_min_i(c2);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) back = max(back, __shfl_xor_sync(0xffffffffu, back, o));
              if (lane == 0) s_tok = c2 != INT_MAX ? c2 : (back >= 0 ? back : 0);
            }
          } else {
            float ws = 0.f, ws_c = 0.f;
            for (int v = s0 + lane * 8; v < s1; v += 256) {
              float zt[8], zd[8];
              load8<kS>(trow, P.dtype, s1, v, vec, zt);
              load8<kS>(drow, P.dtype, s1, v, vec, zd);
              float v8 = 0.f;
#pragma unroll
              for (int e = 0; e < 8; ++e) v8 += D.pjz(zt[e], D.qz(zd[e]));
              kahan_add(ws, ws_c, v8);
            }
            ws = warp_sum(__fsub_rn(ws, ws_c));
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
                load8<kS>(trow, P.dtype, a1, cb + lane * 8, vec, zt);
                load8<kS>(drow, P.dtype, a1, cb + lane * 8, vec, zd);
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
          }
          __syncthreads();
          if (tid == 0) out[depth] = s_tok;
          break;
        }
      }
      if (tid == 0) {
        out[depth] = s_tokn[next];
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // both rows of a node staged in shared memory when they fit (one CTA per
  // SM then); else the passes read them from L2
  const size_t row_bytes = (size_t)V * esz;
  const size_t smem = 2 * ((row_bytes + 127) / 128 * 128);
  int dev = 0, optin = 0;
  const bool aligned16 = row_bytes % 16 == 0 && host_aligned(target_logits, 16) && host_aligned(draft_logits, 16);
  if (aligned16 && cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
      smem + 1024 <= (size_t)optin &&
      cudaFuncSetAttribute(tree_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
    // one CTA per request (one resident per SM): the requests beyond the
    // first wave start on whichever SM frees up first, which balances walks of
    // different lengths (256 requests at V = 32000: 83 -> 75 us against 152
    // CTAs that each take every 152nd request)
    const int grid = B < 65535 ? B : 65535;
    tree_kernel<true><<<grid, kTreeThreads, smem, st>>>(P);
    return host_cuda_status(cudaGetLastError());
  }
  cudaGetLastError();
  const int grid = B < 2 * sms ? B : 2 * sms;
  tree_kernel<false><<<grid, kTreeThreads, 0, st>>>(P);
  return host_cuda_status(cudaGetLastError());
}
