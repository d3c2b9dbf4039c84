// router.cu - router GEMV, top-k, weights and expert bucketing (one launch).
//
// "WISP - streaming what can't run", section "Insight (Credit: JustVugg / Colibri)":
// the model's own router picks which experts a token activates; "Lesson 2": the router
// is the scheduler.  The score functions are the two the layer supports: softmax with
// the weights renormalised over the k selected, or sigmoid with the selected scores
// divided by their sum.  Both are monotone in the logit, so the top-k is taken on the
// fp32 logits; equal logits rank the lower expert id first.
//
// Optional fused stack step (x, y_prev given): every block computes the token's inverse
// RMS of x + y_prev with the same fixed-order reduction as the residual_rmsnorm kernel,
// uses xn = bf16((x + y_prev) * inv) as the router input and writes its slice of xn for
// the expert kernels; the residual x += y_prev is written later by the combine kernel,
// which reads y_prev just before it overwrites y.
// Phase 1 (all blocks): block (s, g) owns the 1024-wide slice s of H and the group g of
// 8 experts, one per warp.  A warp loads its expert's slice of W into registers before
// it waits on the kernel before (the weights do not depend on it), the block stages the
// slice of the bf16 router input in shared memory, and the warp computes the partial dot
// products of all T tokens.  The group's logits are its partials added in slice order:
// with at most 8 slices the slice blocks of a group are one cluster and add them in
// distributed shared memory (router_cluster_kernel), otherwise the last block of the
// group (an atomic ticket per group) adds them from global memory (router_kernel).  The
// last group to finish (a second ticket) runs phase 2: the top-k per token (one warp per
// token, straight from the logits) and the bucketing of the (token, rank) pairs by
// expert into "passes" of up to pmax tokens: routed experts in ascending id, tokens
// ascending, then the shared expert.  Problems that fit one block use
// router_small_kernel, with no global partials at all.  Deferred (one token): the
// kernels stop once the logits [E] are in global memory (after the slice partials) and
// the expert kernels take the top-k themselves (route.cuh).
#include <cfloat>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "route.cuh"

namespace moe {

constexpr int RSW = 1024;   // inputs per slice: 8 float4 of W per lane
constexpr int REPB = 8;     // experts per block (one per warp)
constexpr int RTG = 32;     // tokens staged per pass over the slice
int router_nch(int H) { return cdiv(H, RSW) + 1; }     // slices of partials + the logits
int router_tickets(int E) { return cdiv(E, REPB) + 1; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Pieces shared by the three router kernels, so that each gives the same bits:
// the W slice of a warp's expert (RSW inputs from h0, 8 float4 per lane, loaded before the
// dependency wait), the bf16 rounding of four normalised inputs, and a warp's dot product
// of its W slice with a staged bf16 slice of x (per-lane fma chain in input order, then
// the warp tree).
__device__ __forceinline__ void router_w_slice(const RouterArgs& a, int e, bool live, int h0, int lane,
                                               float4 (&wv)[RSW / 128]) {
  const float* wr = a.W + (size_t)(live ? e : 0) * a.H;
#pragma unroll
  for (int i = 0; i < RSW / 128; ++i) {
    const int h = h0 + 4 * (lane + 32 * i);
    wv[i] = (live && h < a.H) ? __ldg(reinterpret_cast<const float4*>(wr + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ uint2 bf16x4_scaled(const float4 v, float inv) {
  uint2 o;
  o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x * inv)) |
        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y * inv)) << 16);
  o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z * inv)) |
        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w * inv)) << 16);
  return o;
}

// xs: the slice's bf16 inputs (element j of the slice at xs[j]); with CHECK, elements at
// or past lim are zero (not read)
template <bool CHECK>
__device__ __forceinline__ float slice_dot(const float4 (&wv)[RSW / 128], const uint16_t* xs, int lane, int lim) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < RSW / 128; ++i) {
    const int j = 4 * (lane + 32 * i);
    uint2 xb = make_uint2(0u, 0u);
    if (!CHECK || j < lim) xb = *reinterpret_cast<const uint2*>(xs + j);
    acc = fmaf(wv[i].x, __uint_as_float(xb.x << 16), acc);
    acc = fmaf(wv[i].y, __uint_as_float(xb.x & 0xffff0000u), acc);
    acc = fmaf(wv[i].z, __uint_as_float(xb.y << 16), acc);
    acc = fmaf(wv[i].w, __uint_as_float(xb.y & 0xffff0000u), acc);
  }
  return warp_sum(acc);
}

// dense-group split of an expert's c tokens (pmax == 1): chunks of <= GEMM_MAX_TOKENS
__device__ __forceinline__ int big_chunks(int c, int big_min) {
  return (big_min > 0 && c >= big_min) ? cdiv(c, GEMM_MAX_TOKENS) : 0;
}

// Top-k of token t's E logits by one warp (route.cuh), then the k weights; writes the
// plan's and the per-layer copy of the routing and the token's experts in s_idx.  SMALL:
// E <= 128.
template <bool SMALL>
__device__ __forceinline__ void topk_token(const RouterArgs& a, const float* src, bool global_src, int t, int lane,
                                           int* s_idx) {
  const int k = a.k;
  int my_e;
  float my_l;
  if (SMALL) warp_topk<4>(src, global_src, a.E, k, lane, my_e, my_l);
  else warp_topk_any(src, global_src, a.E, k, lane, my_e, my_l);
  const float w = route_weight(a.kind, k, lane, my_l);
  if (lane < k) {
    a.plan.idx[t * k + lane] = my_e;
    a.plan.w[t * k + lane] = w;
    a.store_idx[t * k + lane] = my_e;
    a.store_w[t * k + lane] = w;
    s_idx[t * k + lane] = my_e;
  }
}

__device__ __forceinline__ OneTokenPlan one_token_plan_args(const RouterArgs& a) {
  return OneTokenPlan{a.E, a.k, a.pmax, a.has_shared, a.big_min, a.store_idx, a.store_w, a.counters,
                      a.record_bytes, (unsigned long long)a.E * a.H * 4ull};
}

// Phase 2 of the router, in one block: top-k per token from the logits lsrc [T][E]
// (global memory when global_src), the weights, and the bucketing of the (token, rank)
// pairs into passes.  s_cnt must be zero and the logits complete (after a barrier);
// SMALL: E <= 128 (one top-k variant).
template <bool SMALL>
__device__ __forceinline__ void router_finish(const RouterArgs& a, const float* lsrc, bool global_src, int* s_cnt,
                                              int* s_off, int* s_idx, int* s_pos, int* s_routed) {
  __shared__ int s_wsum[64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int E = a.E, T = a.T, k = a.k, pmax = a.pmax;
  if (T == 1 && a.big_min != 1) {
    // one token, in warp 0 alone (route.cuh's one-token plan)
    if (warp != 0) return;
    int my_e;
    float my_l;
    if (SMALL) warp_topk<4>(lsrc, global_src, E, k, lane, my_e, my_l);
    else warp_topk_any(lsrc, global_src, E, k, lane, my_e, my_l);
    const float w = route_weight(a.kind, k, lane, my_l);
    write_one_token_plan(a.plan, one_token_plan_args(a), lane, my_e, w, one_token_pass(k, lane, my_e));
    if (lane == 0) *a.ticket = 0u;  // ready for the next launch (stream-ordered)
    return;
  }
  // ---------------- phase 2a: top-k per token (one warp per token)
  for (int t = warp; t < T; t += nwarps) {
    const float* src = lsrc + (size_t)t * E;
    topk_token<SMALL>(a, src, global_src, t, lane, s_idx);
  }
  __syncthreads();

  // ---------------- phase 2b: position of each pair within its expert (tokens ascending)
  if (warp == 0) {
    for (int t = 0; t < T; ++t) {
      if (lane < k) {
        const int ee = s_idx[t * k + lane];   // the k experts of a token are distinct
        const int pos = s_cnt[ee];
        s_cnt[ee] = pos + 1;
        s_pos[t * k + lane] = pos;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  {
    // exclusive scan over experts of (passes, unique flag): a thread owns a contiguous run
    // of experts, warps scan with shuffles, the warp totals go through shared memory
    const int run = cdiv(E, (int)blockDim.x);
    const int e0 = min(E, (int)threadIdx.x * run), e1 = min(E, e0 + run);
    int np = 0, nu = 0;
    for (int ee = e0; ee < e1; ++ee) {
      const int c = s_cnt[ee];
      np += pmax == 1 ? c : cdiv(c, pmax);
      nu += c > 0;
    }
    int inp = np, inu = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, inp, o);
      const int a2 = __shfl_up_sync(0xffffffffu, inu, o);
      if (lane >= o) { inp += a1; inu += a2; }
    }
    if (lane == 31) { s_wsum[warp] = inp; s_wsum[32 + warp] = inu; }
    __syncthreads();
    int bp = 0, bu = 0;
    for (int w = 0; w < warp; ++w) { bp += s_wsum[w]; bu += s_wsum[32 + w]; }
    int off = bp + inp - np, uoff = bu + inu - nu;
    for (int ee = e0; ee < e1; ++ee) {
      s_off[ee] = off;
      const int c = s_cnt[ee];
      if (c > 0) a.plan.uniq[uoff++] = ee;
      off += pmax == 1 ? c : cdiv(c, pmax);
    }
    if (threadIdx.x == blockDim.x - 1) {
      const int tot_p = bp + inp, tot_u = bu + inu;
      const int nsh = a.has_shared ? cdiv(T, pmax) : 0;
      a.plan.hdr->n_pass = tot_p + nsh;
      a.plan.hdr->n_routed_pass = tot_p;
      a.plan.hdr->n_uniq = tot_u;
      a.plan.hdr->T = T;
      *s_routed = tot_p;
      DevCounters* dc = a.counters;
      atomicAdd(&dc->forwards, 1ull);
      atomicAdd(&dc->tokens, (unsigned long long)T);
      atomicAdd(&dc->lookups, (unsigned long long)tot_u);
      atomicAdd(&dc->bytes_touched, (unsigned long long)(tot_u + (a.has_shared ? 1 : 0)) * a.record_bytes);
      atomicAdd(&dc->bytes_router, (unsigned long long)E * a.H * 4ull);
    }
  }
  __syncthreads();

  // ---------------- phase 2c: pass tables
  const int routed_passes = *s_routed;
  for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
    const int c = s_cnt[ee];
    for (int i = 0; i * pmax < c; ++i) {
      a.plan.pass_expert[s_off[ee] + i] = ee;
      a.plan.pass_ntok[s_off[ee] + i] = min(pmax, c - i * pmax);
    }
  }
  for (int q = threadIdx.x; q < T * k; q += blockDim.x) {
    const int ee = s_idx[q], pos = s_pos[q];
    const int pass = s_off[ee] + pos / pmax, slot = pos % pmax;
    a.plan.pass_tok[pass * pmax + slot] = q / k;
    a.plan.pair_pass[q] = pass;
    a.plan.pair_slot[q] = slot;
  }
  if (a.has_shared) {
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
      const int pass = routed_passes + t / pmax, slot = t % pmax;
      a.plan.pass_tok[pass * pmax + slot] = t;
      a.plan.shared_pass[t] = pass;
      a.plan.shared_slot[t] = slot;
      if (slot == 0) {
        a.plan.pass_expert[pass] = E;
        a.plan.pass_ntok[pass] = min(pmax, T - t);
      }
    }
  }
  // dense groups (pmax == 1: one pass per token): experts with >= big_min tokens go to the
  // tcgen05 path in balanced chunks of <= GEMM_MAX_TOKENS, every other pass to the
  // per-token path, both lists in ascending expert id (the shared expert last) then token
  // order.  Warp 0: lane owns a contiguous run of experts, an exclusive scan places it.
  if (warp == 0) {
    if (a.big_min > 0) {
      const int E1 = E + (a.has_shared ? 1 : 0);
      const int run = cdiv(E1, 32);
      const int e0 = min(E1, lane * run), e1 = min(E1, e0 + run);
      auto cnt_of = [&](int ee) { return ee < E ? s_cnt[ee] : T; };
      auto first_of = [&](int ee) { return ee < E ? s_off[ee] : routed_passes; };
      int nb = 0, ns = 0;
      for (int ee = e0; ee < e1; ++ee) {
        const int c = cnt_of(ee), nc = big_chunks(c, a.big_min);
        nb += nc;
        ns += nc ? 0 : c;
      }
      int ib = nb, is = ns;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a1 = __shfl_up_sync(0xffffffffu, ib, o);
        const int a2 = __shfl_up_sync(0xffffffffu, is, o);
        if (lane >= o) { ib += a1; is += a2; }
      }
      int ob = ib - nb, os = is - ns;
      for (int ee = e0; ee < e1; ++ee) {
        const int c = cnt_of(ee), first = first_of(ee), nc = big_chunks(c, a.big_min);
        if (nc) {
          const int base = c / nc, rem = c % nc;
          int start = 0;
          for (int q = 0; q < nc; ++q) {
            const int sz = base + (q < rem ? 1 : 0);
            a.plan.big[3 * ob + 0] = ee;
            a.plan.big[3 * ob + 1] = first + start;
            a.plan.big[3 * ob + 2] = sz;
            ++ob;
            start += sz;
          }
        } else {
          for (int i = 0; i < c; ++i) a.plan.small_order[os++] = first + i;
        }
      }
      if (lane == 31) {
        a.plan.hdr->n_big = ib;
        a.plan.hdr->n_small = is;
      }
    } else if (lane == 0) {
      a.plan.hdr->n_big = 0;
      a.plan.hdr->n_small = routed_passes + (a.has_shared ? cdiv(T, pmax) : 0);
    }
    if (lane == 0) *a.ticket = 0u;  // ready for the next launch (stream-ordered)
  }
}

// bytes of phase 2's shared arrays (s_cnt, s_off, s_idx, s_pos)
__host__ __device__ __forceinline__ size_t router_phase2_bytes(int E, int T, int k) {
  return ((size_t)2 * E + (size_t)2 * T * k) * 4;
}

// H > 8 slices.  MINB = blocks per SM the registers must allow: 3 where the grid is
// larger than two blocks per SM (so it still runs in one wave), else 1 (no register cap).
// No block of this kernel waits on another.
template <int MINB>
__global__ void __launch_bounds__(256, MINB) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) int sm[];
  __shared__ float s_inv[ROUTER_FUSED_MAXT];
  __shared__ float s_red[32];
  __shared__ int s_flag, s_routed;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = cdiv(a.H, RSW), NG = cdiv(a.E, REPB);
  const int sl = blockIdx.x % NS, g = blockIdx.x / NS;
  const int h0 = sl * RSW;
  const int e = g * REPB + warp;
  const bool live = e < a.E;
  const bool fused = a.xres != nullptr;

  // ---------------- W slice of this warp's expert (independent of the kernel before)
  float4 wv[RSW / 128];
  router_w_slice(a, e, live, h0, lane, wv);

  pdl_wait();  // x (and the residual) come from the kernels before
  pdl_launch_dependents();
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);   // [RTG][RSW] bf16 router input
  if (fused) {
    // fused stack step (T <= ROUTER_FUSED_MAXT): this thread's float4 of the slice for
    // every token is loaded together with the norm's loads, then normalised and staged;
    // the blocks of group 0 also write their slice of xn for the expert kernels
    const int hq = 4 * threadIdx.x, h = h0 + hq;
    const bool in = threadIdx.x < RSW / 4 && h < a.H;
    float4 xv[ROUTER_FUSED_MAXT];
#pragma unroll
    for (int t = 0; t < ROUTER_FUSED_MAXT; ++t) {
      xv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < a.T && in) {
        const size_t o = (size_t)t * a.H + h;
        xv[t] = __ldcg(reinterpret_cast<const float4*>(a.xres + o));
        if (a.yprev) {
          const float4 y4 = __ldcg(reinterpret_cast<const float4*>(a.yprev + o));
          xv[t].x += y4.x; xv[t].y += y4.y; xv[t].z += y4.z; xv[t].w += y4.w;
        }
      }
    }
    for (int t = 0; t < a.T; ++t) {
      const float inv = block_inv_rms(a.xres + (size_t)t * a.H, a.yprev ? a.yprev + (size_t)t * a.H : nullptr,
                                      a.H, a.eps, s_red);
      if (threadIdx.x == 0) s_inv[t] = inv;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < ROUTER_FUSED_MAXT; ++t) {
      if (t < a.T && threadIdx.x < RSW / 4) {
        uint2 v = bf16x4_scaled(xv[t], s_inv[t]);
        if (!in) v = make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(xs + t * RSW + hq) = v;
        if (g == 0 && in) *reinterpret_cast<uint2*>(a.xn_out + (size_t)t * a.H + h) = v;
      }
    }
  }

  // ---------------- phase 1: partial logits of slice sl, partial[sl][t][e]
  for (int tg = 0; tg < a.T; tg += RTG) {
    const int nt = min(RTG, a.T - tg);
    __syncthreads();  // the previous group's reads of xs are done (fused: xs is staged)
    if (!fused) {
      for (int q = threadIdx.x; q < nt * (RSW / 4); q += blockDim.x) {
        const int tl = q / (RSW / 4), hq = 4 * (q % (RSW / 4)), h = h0 + hq;
        uint2 v = make_uint2(0u, 0u);
        if (h < a.H) v = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)(tg + tl) * a.H + h));
        *reinterpret_cast<uint2*>(xs + tl * RSW + hq) = v;
      }
      __syncthreads();
    }
    if (live) {
      float keep = 0.f;
      for (int tl = 0; tl < nt; ++tl) {
        const float acc = slice_dot<false>(wv, xs + tl * RSW, lane, RSW);
        if (lane == tl) keep = acc;
      }
      if (lane < nt) a.partial[((size_t)sl * a.T + tg + lane) * a.E + e] = keep;
    }
  }

  // ---------------- tickets: the last block of each expert group adds its group's slices
  // into the logits in ascending slice order, and the last group continues
  float* logits = a.partial + (size_t)NS * a.T * a.E;   // [T][E]
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_flag = (atomicAdd(a.ticket + 1 + g, 1u) == (unsigned)NS - 1);
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  const int ne = min(REPB, a.E - g * REPB);
  for (int q = threadIdx.x; q < a.T * ne; q += blockDim.x) {
    const int t = q / ne, ee = g * REPB + q % ne;
    const float* pp = a.partial + (size_t)t * a.E + ee;
    float v = 0.f;
#pragma unroll 8
    for (int ss = 0; ss < NS; ++ss) v += __ldcg(pp + (size_t)ss * a.T * a.E);
    logits[(size_t)t * a.E + ee] = v;
  }
  if (threadIdx.x == 0) a.ticket[1 + g] = 0u;  // ready for the next launch (stream-ordered)
  if (a.defer) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_flag = (atomicAdd(a.ticket, 1u) == (unsigned)NG - 1);
  __syncthreads();
  if (!s_flag) return;
  __threadfence();

  const int E = a.E, T = a.T, k = a.k;
  int* s_cnt = sm;                  // [E]
  int* s_off = s_cnt + E;           // [E]
  int* s_idx = s_off + E;           // [T*k]
  int* s_pos = s_idx + T * k;       // [T*k]
  for (int q = threadIdx.x; q < E; q += blockDim.x) s_cnt[q] = 0;
  __syncthreads();

  router_finish<false>(a, logits, true, s_cnt, s_off, s_idx, s_pos, &s_routed);
}


// ---------------------------------------------------------------- clusters of slices
// H <= RCLUSTER_MAX * RSW: the NS slice blocks of an expert group are one thread-block
// cluster (block (s, g) is rank s) and meet in distributed shared memory instead of
// global partials.  Values are pushed: a rank stores into the others' shared memory and
// one cluster barrier later every reader finds them in its own.  Fused stack step: the
// inverse RMS is block_inv_rms's fixed tree spread over the cluster: rank s computes the
// tree's logical warps s, s + NS, ... (the same elements in the same order) and stores
// the warp sums in every rank; each block then adds the 8 warp sums in the tree's order,
// so the bits are those of block_inv_rms.  The partial dot products go to rank 0, which
// adds the NS partials of each (token, expert) in ascending slice order (as router_kernel
// does), writes the group's logits and takes the group's ticket; the other ranks are done
// after the barrier, and the last group runs phase 2.  A first barrier phase, arrived at
// on entry and waited for before the first remote store, makes sure that every block of
// the cluster has started.
constexpr int RCLUSTER_MAX = 8;
namespace cg = cooperative_groups;

template <int MINB>
__global__ void __launch_bounds__(256, MINB) router_cluster_kernel(RouterArgs a) {
  extern __shared__ __align__(16) int sm[];
  constexpr int NLW = RMS_NTHR / 32;   // logical warps of the norm tree
  __shared__ float s_inv[ROUTER_FUSED_MAXT];
  __shared__ float s_nrm[ROUTER_FUSED_MAXT][NLW];
  __shared__ int s_flag, s_routed;
  cg::cluster_group cl = cg::this_cluster();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");   // this block has started
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = cdiv(a.H, RSW), NG = cdiv(a.E, REPB);
  const int sl = blockIdx.x % NS, g = blockIdx.x / NS;
  const int h0 = sl * RSW;
  const int e = g * REPB + warp;
  const bool live = e < a.E;
  const bool fused = a.xres != nullptr;
  const int T = a.T, H = a.H;

  float4 wv[RSW / 128];
  router_w_slice(a, e, live, h0, lane, wv);

  pdl_wait();  // x (and the residual) come from the kernels before
  pdl_launch_dependents();
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);                                  // [min(T, RTG)][RSW]
  float* s_part = reinterpret_cast<float*>(sm) + (size_t)min(T, RTG) * RSW / 2;     // [NS][T][REPB] (rank 0)
  bool started = false;   // the entry barrier phase has been waited for
  if (fused) {
    const int hq = 4 * threadIdx.x, h = h0 + hq;
    const bool in = threadIdx.x < RSW / 4 && h < H;
    float4 xv[ROUTER_FUSED_MAXT];
#pragma unroll
    for (int t = 0; t < ROUTER_FUSED_MAXT; ++t) {
      xv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < T && in) {
        const size_t o = (size_t)t * H + h;
        xv[t] = __ldcg(reinterpret_cast<const float4*>(a.xres + o));
        if (a.yprev) {
          const float4 y4 = __ldcg(reinterpret_cast<const float4*>(a.yprev + o));
          xv[t].x += y4.x; xv[t].y += y4.y; xv[t].z += y4.z; xv[t].w += y4.w;
        }
      }
    }
    // this rank's logical warps of every token's tree: lane = logical lane
    const int n4 = H >> 2;
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every block has started
    started = true;
    for (int p = warp; p < T * NLW; p += 8) {
      const int t = p / NLW, lw = p - t * NLW;
      if (lw % NS != sl) continue;
      const float4* x4 = reinterpret_cast<const float4*>(a.xres + (size_t)t * H);
      const float4* y4 = a.yprev ? reinterpret_cast<const float4*>(a.yprev + (size_t)t * H) : nullptr;
      float ss = 0.f;
      for (int i0 = lw * 32 + lane; i0 < n4; i0 += 8 * RMS_NTHR) {
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = i0 + q * RMS_NTHR;
          v[q] = i < n4 ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          if (y4 && i < n4) {
            const float4 b = __ldcg(y4 + i);
            v[q].x += b.x; v[q].y += b.y; v[q].z += b.z; v[q].w += b.w;
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          ss = fmaf(v[q].x, v[q].x, ss);
          ss = fmaf(v[q].y, v[q].y, ss);
          ss = fmaf(v[q].z, v[q].z, ss);
          ss = fmaf(v[q].w, v[q].w, ss);
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane < NS) *cl.map_shared_rank(&s_nrm[t][lw], (unsigned)lane) = ss;   // (every lane holds the sum)
    }
    cl.sync();   // every rank's warp sums are in every rank
    if (warp < T) {
      float v = 0.f;
      if (lane < NLW) v = s_nrm[warp][lane];
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_inv[warp] = rsqrtf(v / (float)H + a.eps);
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < ROUTER_FUSED_MAXT; ++t) {
      if (t < T && threadIdx.x < RSW / 4) {
        uint2 v = bf16x4_scaled(xv[t], s_inv[t]);
        if (!in) v = make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(xs + t * RSW + hq) = v;
        if (g == 0 && in) *reinterpret_cast<uint2*>(a.xn_out + (size_t)t * H + h) = v;
      }
    }
  }

  // ---------------- phase 1: partial logits of slice sl into rank 0's s_part [sl][T][REPB]
  if (!started) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every block has started
  float* part0 = cl.map_shared_rank(s_part, 0u) + (size_t)sl * T * REPB;
  for (int tg = 0; tg < T; tg += RTG) {
    const int nt = min(RTG, T - tg);
    __syncthreads();  // the previous group's reads of xs are done (fused: xs is staged)
    if (!fused) {
      for (int q = threadIdx.x; q < nt * (RSW / 4); q += blockDim.x) {
        const int tl = q / (RSW / 4), hq = 4 * (q % (RSW / 4)), h = h0 + hq;
        uint2 v = make_uint2(0u, 0u);
        if (h < H) v = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)(tg + tl) * H + h));
        *reinterpret_cast<uint2*>(xs + tl * RSW + hq) = v;
      }
      __syncthreads();
    }
    if (live) {
      float keep = 0.f;
      for (int tl = 0; tl < nt; ++tl) {
        const float acc = slice_dot<false>(wv, xs + tl * RSW, lane, RSW);
        if (lane == tl) keep = acc;
      }
      if (lane < nt) part0[(tg + lane) * REPB + warp] = keep;
    }
  }

  // ---------------- the group's logits, in rank 0
  cl.sync();   // every rank's partials are in rank 0
  if (sl != 0) return;
  float* logits = a.partial + (size_t)NS * T * a.E;   // [T][E]
  const int ne = min(REPB, a.E - g * REPB);
  for (int q = threadIdx.x; q < T * REPB; q += blockDim.x) {
    const int t = q / REPB, w = q - t * REPB;
    if (w < ne) {
      float v = 0.f;
      for (int r = 0; r < NS; ++r) v += s_part[((size_t)r * T + t) * REPB + w];
      logits[(size_t)t * a.E + g * REPB + w] = v;
    }
  }
  if (a.defer) return;
  // the group's ticket: its release publishes the logits (written before the barrier),
  // and the last group's acquire makes every group's logits visible to this block
  __syncthreads();
  if (threadIdx.x == 0) s_flag = (atom_add_acq_rel_gpu(a.ticket, 1u) == (unsigned)NG - 1);
  __syncthreads();
  if (!s_flag) return;

  const int E = a.E, k = a.k;
  int* s_cnt = sm;                  // [E]
  int* s_off = s_cnt + E;           // [E]
  int* s_idx = s_off + E;           // [T*k]
  int* s_pos = s_idx + T * k;       // [T*k]
  if (T != 1 || a.big_min == 1) {   // the per-expert counts (not used by the one-token plan)
    for (int q = threadIdx.x; q < E; q += blockDim.x) s_cnt[q] = 0;
    __syncthreads();
  }
  router_finish<false>(a, logits, true, s_cnt, s_off, s_idx, s_pos, &s_routed);
}

size_t router_cluster_smem(int H, int T, int E, int k) {
  const size_t p1 = (size_t)std::min(T, RTG) * RSW * 2 + (size_t)cdiv(H, RSW) * T * REPB * sizeof(float);
  return std::max(p1, router_phase2_bytes(E, T, k));
}

// ---------------------------------------------------------------- small problems, one block
// When every (expert, slice) item fits one warp of a single 1024-thread block and the
// bf16 input fits shared memory, one block does the whole router: no partials in global
// memory, no fences, no tickets.  Warp w owns expert w / NS on slice w % NS and loads its
// W slice before the wait; logits are the slices added in ascending order, as in
// router_kernel, so both give the same bits.
constexpr int RSMALL_THREADS = 1024;
constexpr int ROUTER_SMEM_MAX = 160 * 1024;
__host__ __device__ __forceinline__ bool router_small_fits(int H, int T, int E) {
  return E * cdiv(H, RSW) <= RSMALL_THREADS / 32 && T * H <= 32768 && T <= 32;
}
bool router_one_block(int H, int T, int E) { return router_small_fits(H, T, E); }

// bf16 inputs, slice partials, logits and phase 2's arrays
size_t router_small_smem(int H, int T, int E, int k) {
  return ((size_t)T * H / 2 + (size_t)T * E * cdiv(H, RSW) + (size_t)T * E + (size_t)2 * E + (size_t)2 * T * k) * 4;
}

// V4: float4s of a row each norm thread holds in registers (H <= 4 * RMS_NTHR * V4)
template <int V4>
__global__ void __launch_bounds__(RSMALL_THREADS) router_small_kernel(RouterArgs a) {
  extern __shared__ __align__(16) int sm[];
  __shared__ float s_inv[ROUTER_FUSED_MAXT];
  __shared__ float s_red[32];
  __shared__ int s_routed;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, T = a.T, E = a.E, k = a.k;
  const int NS = cdiv(H, RSW), items = E * NS;
  const int e = warp / NS, sl = warp - e * NS, h0 = sl * RSW;
  const bool live = warp < items;
  const bool fused = a.xres != nullptr;
  uint16_t* xs = reinterpret_cast<uint16_t*>(sm);                        // [T][H] bf16
  float* spart = reinterpret_cast<float*>(xs + (size_t)T * H);           // [T][E][NS]
  float* slog = spart + (size_t)T * E * NS;                              // [T][E]
  int* s_cnt = reinterpret_cast<int*>(slog + (size_t)T * E);            // [E]
  int* s_off = s_cnt + E;                                                // [E]
  int* s_idx = s_off + E;                                                // [T*k]
  int* s_pos = s_idx + T * k;                                            // [T*k]

  float4 wv[RSW / 128];
  router_w_slice(a, e, live, h0, lane, wv);
  pdl_wait();  // x (and the residual) come from the kernels before
  pdl_launch_dependents();
  if (fused && H <= RMS_NTHR * V4 * 4) {
    // one pass over x + y_prev: the first RMS_NTHR threads keep their float4s of a row in
    // registers for both the norm (block_inv_rms_regs: the order of block_inv_rms) and the
    // staging
    for (int t = 0; t < T; ++t) {
      const size_t ro = (size_t)t * H;
      float4 v[V4];
#pragma unroll
      for (int q = 0; q < V4; ++q) {
        const int i = threadIdx.x + q * RMS_NTHR;
        v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if ((int)threadIdx.x < RMS_NTHR && i < H / 4) {
          v[q] = __ldcg(reinterpret_cast<const float4*>(a.xres + ro) + i);
          if (a.yprev) {
            const float4 y4 = __ldcg(reinterpret_cast<const float4*>(a.yprev + ro) + i);
            v[q].x += y4.x; v[q].y += y4.y; v[q].z += y4.z; v[q].w += y4.w;
          }
        }
      }
      const float inv = block_inv_rms_regs<V4>(v, H, a.eps, s_red);
#pragma unroll
      for (int q = 0; q < V4; ++q) {
        const int i = threadIdx.x + q * RMS_NTHR;
        if ((int)threadIdx.x < RMS_NTHR && i < H / 4) {
          const uint2 o = bf16x4_scaled(v[q], inv);
          *reinterpret_cast<uint2*>(a.xn_out + ro + 4 * i) = o;
          *reinterpret_cast<uint2*>(xs + ro + 4 * i) = o;
        }
      }
    }
  } else {
    if (fused) {
      for (int t = 0; t < T; ++t) {
        const float inv = block_inv_rms(a.xres + (size_t)t * H, a.yprev ? a.yprev + (size_t)t * H : nullptr, H,
                                        a.eps, s_red);
        if (threadIdx.x == 0) s_inv[t] = inv;
      }
      __syncthreads();
    }
    for (int q = threadIdx.x; q < T * (H / 4); q += blockDim.x) {
      const int t = q / (H / 4), h = 4 * (q - t * (H / 4));
      const size_t o = (size_t)t * H + h;
      uint2 v;
      if (fused) {
        float4 x4 = __ldcg(reinterpret_cast<const float4*>(a.xres + o));
        if (a.yprev) {
          const float4 y4 = __ldcg(reinterpret_cast<const float4*>(a.yprev + o));
          x4.x += y4.x; x4.y += y4.y; x4.z += y4.z; x4.w += y4.w;
        }
        v = bf16x4_scaled(x4, s_inv[t]);
        *reinterpret_cast<uint2*>(a.xn_out + o) = v;
      } else {
        v = __ldg(reinterpret_cast<const uint2*>(a.x + o));
      }
      *reinterpret_cast<uint2*>(xs + o) = v;
    }
  }
  for (int q = threadIdx.x; q < E; q += blockDim.x) s_cnt[q] = 0;
  __syncthreads();
  if (live) {
    float keep = 0.f;
    for (int t = 0; t < T; ++t) {
      const float acc = slice_dot<true>(wv, xs + (size_t)t * H + h0, lane, H - h0);
      if (lane == t) keep = acc;
    }
    if (lane < T) spart[((size_t)lane * E + e) * NS + sl] = keep;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < T * E; q += blockDim.x) {
    float v = 0.f;
    for (int ss = 0; ss < NS; ++ss) v += spart[(size_t)q * NS + ss];
    slog[q] = v;
    if (a.defer) a.partial[(size_t)NS * T * E + q] = v;   // where the other kernels keep the logits
  }
  if (a.defer) return;
  __syncthreads();
  router_finish<true>(a, slog, false, s_cnt, s_off, s_idx, s_pos, &s_routed);
}

cudaError_t router_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(router_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, ROUTER_SMEM_MAX);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_small_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, ROUTER_SMEM_MAX);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_small_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, ROUTER_SMEM_MAX);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_cluster_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, ROUTER_SMEM_MAX);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_cluster_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, ROUTER_SMEM_MAX);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, ROUTER_SMEM_MAX);
}

// staging of min(T, RTG) bf16 rows of a slice, then (last block) the phase-2 arrays
size_t router_smem_bytes(int H, int T, int E, int k) {
  (void)H;
  return std::max((size_t)std::min(T, RTG) * RSW * 2, router_phase2_bytes(E, T, k));
}

cudaError_t launch_router(const RouterArgs& a, int num_sms, cudaStream_t s) {
  if (router_small_fits(a.H, a.T, a.E)) {
    const size_t smem = router_small_smem(a.H, a.T, a.E, a.k);
    if (smem > ROUTER_SMEM_MAX) return cudaErrorInvalidValue;
    if (a.H <= 4 * RMS_NTHR * 4) return launch_pdl(router_small_kernel<4>, 1, RSMALL_THREADS, smem, s, a);
    return launch_pdl(router_small_kernel<8>, 1, RSMALL_THREADS, smem, s, a);
  }
  const int NS = cdiv(a.H, RSW);
  const int grid = NS * cdiv(a.E, REPB);
  if (NS <= RCLUSTER_MAX) {
    const size_t smem = router_cluster_smem(a.H, a.T, a.E, a.k);
    if (smem > ROUTER_SMEM_MAX) return cudaErrorInvalidValue;
    if (grid > 2 * num_sms) return launch_pdl_cluster(router_cluster_kernel<3>, grid, 256, NS, smem, s, a);
    return launch_pdl_cluster(router_cluster_kernel<1>, grid, 256, NS, smem, s, a);
  }
  const size_t smem = router_smem_bytes(a.H, a.T, a.E, a.k);
  if (smem > ROUTER_SMEM_MAX) return cudaErrorInvalidValue;
  if (grid > 2 * num_sms) return launch_pdl(router_kernel<3>, grid, 256, smem, s, a);
  return launch_pdl(router_kernel<1>, grid, 256, smem, s, a);
}

}  // namespace moe
