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
// slice of the bf16 router input in shared memory, and the warp writes the partial dot
// products of all T tokens.  The last block of a group to finish (an atomic ticket per
// group) adds the group's partials in slice order into the logits; the last group to
// finish (a second ticket) runs phase 2: the top-k per token (one warp per token,
// straight from the logits) and the bucketing of the (token, rank) pairs by expert into
// "passes" of up to pmax tokens: routed experts in ascending id, tokens ascending, then
// the shared expert.  No block ever waits on another.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int RSW = 1024;   // inputs per slice: 8 float4 of W per lane
constexpr int REPB = 8;     // experts per block (one per warp)
constexpr int RTG = 32;     // tokens staged per pass over the slice
constexpr int RXS_BYTES = RTG * RSW * 2;
constexpr int RNS_ONE = 8;                 // the last block adds the slices itself when
constexpr size_t RSUM_ONE_BLOCK = 16384;   // NS <= RNS_ONE and NS * T * E <= RSUM_ONE_BLOCK
__host__ __device__ __forceinline__ bool router_two_level(int NS, int T, int E) {
  return NS > RNS_ONE || (size_t)NS * T * E > RSUM_ONE_BLOCK;
}
int router_nch(int H) { return cdiv(H, RSW) + 1; }     // slices of partials + the logits
int router_tickets(int E) { return cdiv(E, REPB) + 1; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// dense-group split of an expert's c tokens (pmax == 1): chunks of <= GEMM_MAX_TOKENS
__device__ __forceinline__ int big_chunks(int c, int big_min) {
  return (big_min > 0 && c >= big_min) ? cdiv(c, GEMM_MAX_TOKENS) : 0;
}

// Top-k of one token's E logits (one warp; NV * 32 >= E values, lane l holds experts
// l + 32 i), then the k weights; writes the plan's and the per-layer copy of the routing.
// Each lane keeps the maximum of its own experts not yet taken; the warp takes the best k
// times, and only the lane that gave its maximum away looks for its next one.  NaN ranks
// as -inf; equal values rank the lower id first.
template <int NV>
__device__ __forceinline__ void topk_token(const RouterArgs& a, const float* src, bool global_src, int t, int lane,
                                           int* s_idx) {
  const int E = a.E, k = a.k;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int ee = lane + 32 * i;
    v[i] = ee < E ? (global_src ? __ldcg(src + ee) : src[ee]) : -INFINITY;
  }
  uint32_t taken = 0u;
  auto lane_best = [&](float& bv, int& be) {
    bv = -INFINITY;
    be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int ee = lane + 32 * i;
      const float x = v[i] != v[i] ? -INFINITY : v[i];
      if (ee < E && !((taken >> i) & 1u) && (x > bv || (x == bv && ee < be))) { bv = x; be = ee; }
    }
  };
  float lv;
  int le;
  lane_best(lv, le);
  int my_e = 0;
  float my_l = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = lv;
    int be = le;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if (lane == j) { my_e = be; my_l = bv; }
    if (be == le) {   // this lane's maximum was taken (ids are distinct across lanes)
      taken |= 1u << ((be - lane) >> 5);
      lane_best(lv, le);
    }
  }
  // weights over the k selected (rank order = lane order)
  const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
  float num = 0.f;
  if (lane < k) {
    if (a.kind == 0) num = expf(my_l - lmax);
    else num = 1.f / (1.f + expf(-my_l));
  }
  float den = num;
#pragma unroll
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (lane < k) {
    const float w = num / den;
    a.plan.idx[t * k + lane] = my_e;
    a.plan.w[t * k + lane] = w;
    a.store_idx[t * k + lane] = my_e;
    a.store_w[t * k + lane] = w;
    s_idx[t * k + lane] = my_e;
  }
}

// Phase 2 of the router, in one block: top-k per token from the logits lsrc [T][E]
// (global memory when global_src), the weights, and the bucketing of the (token, rank)
// pairs into passes.  s_cnt must be zero and the logits complete (after a barrier).
__device__ __forceinline__ void router_finish(const RouterArgs& a, const float* lsrc, bool global_src, int* s_cnt,
                                              int* s_off, int* s_idx, int* s_pos, int* s_routed) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int E = a.E, T = a.T, k = a.k, pmax = a.pmax;
  // ---------------- phase 2a: top-k per token (one warp per token)
  for (int t = warp; t < T; t += nwarps) {
    const float* src = lsrc + (size_t)t * E;
    if (E <= 128) topk_token<4>(a, src, global_src, t, lane, s_idx);
    else if (E <= 256) topk_token<8>(a, src, global_src, t, lane, s_idx);
    else if (E <= 512) topk_token<16>(a, src, global_src, t, lane, s_idx);
    else topk_token<32>(a, src, global_src, t, lane, s_idx);
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
    // exclusive scan over experts of (passes, unique flag); lane owns a contiguous run
    const int run = cdiv(E, 32);
    const int e0 = min(E, lane * run), e1 = min(E, e0 + run);
    int np = 0, nu = 0;
    for (int ee = e0; ee < e1; ++ee) {
      np += cdiv(s_cnt[ee], pmax);
      nu += s_cnt[ee] > 0;
    }
    int inp = np, inu = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, inp, o);
      const int a2 = __shfl_up_sync(0xffffffffu, inu, o);
      if (lane >= o) { inp += a1; inu += a2; }
    }
    int off = inp - np, uoff = inu - nu;
    for (int ee = e0; ee < e1; ++ee) {
      s_off[ee] = off;
      const int c = s_cnt[ee];
      if (c > 0) a.plan.uniq[uoff++] = ee;
      off += cdiv(c, pmax);
    }
    const int tot_p = __shfl_sync(0xffffffffu, inp, 31);
    const int tot_u = __shfl_sync(0xffffffffu, inu, 31);
    if (lane == 0) {
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

// MINB = blocks per SM the registers must allow: 3 where the grid is larger than two
// blocks per SM (so it still runs in one wave), else 1 (no register cap).
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
  {
    const float* wr = a.W + (size_t)(live ? e : 0) * a.H;
#pragma unroll
    for (int i = 0; i < RSW / 128; ++i) {
      const int h = h0 + 4 * (lane + 32 * i);
      wv[i] = (live && h < a.H) ? __ldg(reinterpret_cast<const float4*>(wr + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

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
        const float inv = s_inv[t];
        uint2 v;
        v.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(xv[t].x * inv)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(xv[t].y * inv)) << 16);
        v.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(xv[t].z * inv)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(xv[t].w * inv)) << 16);
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
        const uint16_t* xr = xs + tl * RSW;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < RSW / 128; ++i) {
          const uint2 xb = *reinterpret_cast<const uint2*>(xr + 4 * (lane + 32 * i));
          acc = fmaf(wv[i].x, __uint_as_float(xb.x << 16), acc);
          acc = fmaf(wv[i].y, __uint_as_float(xb.x & 0xffff0000u), acc);
          acc = fmaf(wv[i].z, __uint_as_float(xb.y << 16), acc);
          acc = fmaf(wv[i].w, __uint_as_float(xb.y & 0xffff0000u), acc);
        }
        acc = warp_sum(acc);
        if (lane == tl) keep = acc;
      }
      if (lane < nt) a.partial[((size_t)sl * a.T + tg + lane) * a.E + e] = keep;
    }
  }

  // ---------------- tickets.  Small problems: the last block overall adds the slices
  // itself.  Otherwise the last block of each expert group adds its group's slices into
  // the logits, and the last group continues.  Both add the slices in ascending order.
  const bool two_level = router_two_level(NS, a.T, a.E);
  float* logits = a.partial + (size_t)NS * a.T * a.E;   // [T][E] (two-level only)
  __threadfence();
  __syncthreads();
  if (two_level) {
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
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_flag = (atomicAdd(a.ticket, 1u) == (unsigned)NG - 1);
  } else {
    if (threadIdx.x == 0) s_flag = (atomicAdd(a.ticket, 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();

  const int E = a.E, T = a.T, k = a.k;
  int* s_cnt = sm;                  // [E]
  int* s_off = s_cnt + E;           // [E]
  int* s_idx = s_off + E;           // [T*k]
  int* s_pos = s_idx + T * k;       // [T*k]
  float* slog = reinterpret_cast<float*>(s_pos + T * k);   // [T][E] (single-level only)
  for (int q = threadIdx.x; q < E; q += blockDim.x) s_cnt[q] = 0;
  if (!two_level) {
    // logits = slice partials added in ascending slice order, all (t, e) in parallel
    const size_t TE = (size_t)T * E;
    for (int q0 = threadIdx.x; q0 < (int)TE; q0 += 2 * blockDim.x) {
      float p[2][RNS_ONE];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = q0 + u * blockDim.x;
#pragma unroll
        for (int ss = 0; ss < RNS_ONE; ++ss) p[u][ss] = (ss < NS && q < (int)TE) ? __ldcg(a.partial + ss * TE + q) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = q0 + u * blockDim.x;
        float v = 0.f;
#pragma unroll
        for (int ss = 0; ss < RNS_ONE; ++ss)
          if (ss < NS) v += p[u][ss];
        if (q < (int)TE) slog[q] = v;
      }
    }
  }
  __syncthreads();

  router_finish(a, two_level ? logits : slog, two_level, s_cnt, s_off, s_idx, s_pos, &s_routed);
}


// ---------------------------------------------------------------- small problems, one block
// When every (expert, slice) item fits one warp of a single 1024-thread block and the
// bf16 input fits shared memory, one block does the whole router: no partials in global
// memory, no fences, no tickets.  Warp w owns expert w / NS on slice w % NS and loads its
// W slice before the wait; logits are the slices added in ascending order, as in
// router_kernel, so both give the same bits.
constexpr int RSMALL_THREADS = 1024;
__host__ __device__ __forceinline__ bool router_small_fits(int H, int T, int E) {
  return E * cdiv(H, RSW) <= RSMALL_THREADS / 32 && T * H <= 32768 && T <= 32;
}
size_t router_small_smem(int H, int T, int E, int k) {
  return (size_t)T * H * 2 + (size_t)T * E * cdiv(H, RSW) * 4 + (size_t)T * E * 4 +
         (size_t)(2 * E + 2 * T * k) * sizeof(int);
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
  {
    const float* wr = a.W + (size_t)(live ? e : 0) * H;
#pragma unroll
    for (int i = 0; i < RSW / 128; ++i) {
      const int h = h0 + 4 * (lane + 32 * i);
      wv[i] = (live && h < H) ? __ldg(reinterpret_cast<const float4*>(wr + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
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
          uint2 o;
          o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[q].x * inv)) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[q].y * inv)) << 16);
          o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[q].z * inv)) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[q].w * inv)) << 16);
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
        const float inv = s_inv[t];
        v.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x4.x * inv)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x4.y * inv)) << 16);
        v.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x4.z * inv)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x4.w * inv)) << 16);
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
      const uint16_t* xr = xs + (size_t)t * H;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < RSW / 128; ++i) {
        const int h = h0 + 4 * (lane + 32 * i);
        uint2 xb = make_uint2(0u, 0u);
        if (h < H) xb = *reinterpret_cast<const uint2*>(xr + h);
        acc = fmaf(wv[i].x, __uint_as_float(xb.x << 16), acc);
        acc = fmaf(wv[i].y, __uint_as_float(xb.x & 0xffff0000u), acc);
        acc = fmaf(wv[i].z, __uint_as_float(xb.y << 16), acc);
        acc = fmaf(wv[i].w, __uint_as_float(xb.y & 0xffff0000u), acc);
      }
      acc = warp_sum(acc);
      if (lane == t) keep = acc;
    }
    if (lane < T) spart[((size_t)lane * E + e) * NS + sl] = keep;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < T * E; q += blockDim.x) {
    float v = 0.f;
    for (int ss = 0; ss < NS; ++ss) v += spart[(size_t)q * NS + ss];
    slog[q] = v;
  }
  __syncthreads();
  router_finish(a, slog, false, s_cnt, s_off, s_idx, s_pos, &s_routed);
}

cudaError_t router_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(router_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_small_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_small_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
}

size_t router_smem_bytes(int H, int T, int E, int k) {
  const size_t p2 = (size_t)(2 * E + 2 * T * k) * sizeof(int) +
                    (router_two_level(cdiv(H, RSW), T, E) ? 0 : (size_t)T * E * sizeof(float));
  return std::max((size_t)RXS_BYTES, p2);
}

cudaError_t launch_router(const RouterArgs& a, int num_sms, cudaStream_t s) {
  if (router_small_fits(a.H, a.T, a.E)) {
    const size_t smem = router_small_smem(a.H, a.T, a.E, a.k);
    if (a.H <= 4 * RMS_NTHR * 4) return launch_pdl(router_small_kernel<4>, 1, RSMALL_THREADS, smem, s, a);
    return launch_pdl(router_small_kernel<8>, 1, RSMALL_THREADS, smem, s, a);
  }
  const int grid = cdiv(a.H, RSW) * cdiv(a.E, REPB);
  const size_t smem = router_smem_bytes(a.H, a.T, a.E, a.k);
  if (grid > 2 * num_sms) return launch_pdl(router_kernel<3>, grid, 256, smem, s, a);
  return launch_pdl(router_kernel<1>, grid, 256, smem, s, a);
}

}  // namespace moe
