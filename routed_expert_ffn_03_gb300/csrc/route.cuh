// route.cuh - the routing decision of one token by one warp: top-k of the logits, the k
// weights, and the one-token pass plan.  Used by the router's last block and, when the
// router only writes logits (one token), by the expert kernels themselves, so both give
// the same bits.
//
// "WISP - streaming what can't run", section "Insight (Credit: JustVugg / Colibri)": the
// model's own router picks the experts.  The score functions are softmax with the weights
// renormalised over the k selected, or sigmoid with the selected scores divided by their
// sum; both are monotone in the logit, so the top-k is taken on the fp32 logits, equal
// logits ranking the lower expert id first and NaN ranking as -inf.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace moe {

// order-preserving 32-bit key of a logit (-0 taken as +0, so that it equals +0)
__device__ __forceinline__ uint32_t logit_key(float x) {
  const uint32_t b = __float_as_uint(x + 0.0f);   // -0 + 0 = +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of one token's E logits by one warp (NV * 32 >= E; lane l holds experts l + 32 i):
// lane j < k receives the j-th expert and its logit.  Selection by k warp reductions:
// each lane keeps the best of its experts not yet taken (key, then id); the warp's
// largest key, then the least id holding it, is the next expert, and only the lane that
// owned it looks for its next best.
template <int NV>
__device__ __forceinline__ void warp_topk(const float* src, bool global_src, int E, int k, int lane, int& my_e,
                                          float& my_l) {
  uint32_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int ee = lane + 32 * i;
    const float x = ee < E ? (global_src ? __ldcg(src + ee) : src[ee]) : -INFINITY;
    key[i] = ee < E ? logit_key(x != x ? -INFINITY : x) : 0u;   // 0: below every expert's key
  }
  uint32_t taken = 0u;
  uint32_t lk = 0u;
  int le = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (key[i] > lk) {   // ascending ids: the first of equal keys stays
      lk = key[i];
      le = lane + 32 * i;
    }
  my_e = 0;
  my_l = 0.f;
  for (int j = 0; j < k; ++j) {
    const uint32_t bk = __reduce_max_sync(0xffffffffu, lk);
    const int be = (int)__reduce_min_sync(0xffffffffu, lk == bk ? (uint32_t)le : 0xffffffffu);
    if (lane == j) {
      my_e = be;
      my_l = key_logit(bk);
    }
    if (le == be) {   // this lane's best was taken (ids are distinct across lanes)
      taken |= 1u << ((be - lane) >> 5);
      lk = 0u;
      le = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (!((taken >> i) & 1u) && key[i] > lk) {
          lk = key[i];
          le = lane + 32 * i;
        }
    }
  }
}

// warp_topk for any E <= 1024 (the register count follows E)
__device__ __forceinline__ void warp_topk_any(const float* src, bool global_src, int E, int k, int lane, int& my_e,
                                              float& my_l) {
  if (E <= 128) warp_topk<4>(src, global_src, E, k, lane, my_e, my_l);
  else if (E <= 256) warp_topk<8>(src, global_src, E, k, lane, my_e, my_l);
  else if (E <= 512) warp_topk<16>(src, global_src, E, k, lane, my_e, my_l);
  else warp_topk<32>(src, global_src, E, k, lane, my_e, my_l);
}

// weight of lane j's selected expert (j < k; the selection in rank order, lane 0 the
// largest logit): softmax over the k (kind 0) or sigmoid divided by the sum (kind 1);
// every lane of the warp must call it
__device__ __forceinline__ float route_weight(int kind, int k, int lane, float my_l) {
  const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
  float num = 0.f;
  if (lane < k) {
    if (kind == 0) num = expf(my_l - lmax);
    else num = 1.f / (1.f + expf(-my_l));
  }
  float den = num;
#pragma unroll
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  return num / den;
}

// position of lane j's expert (j < k) among the k selected by ascending id (the k ids are
// distinct): its pass in the one-token plan
__device__ __forceinline__ int one_token_pass(int k, int lane, int my_e) {
  const int ee = lane < k ? my_e : 0x7fffffff;
  int p = 0;
  for (int j = 0; j < k; ++j) p += __shfl_sync(0xffffffffu, ee, j) < ee ? 1 : 0;
  return p;
}

// The plan of one token, written by one warp from its top-k (lane j < k holds the j-th
// expert, its weight w and its pass p): every selected expert has one pass, the passes in
// ascending expert id, the shared expert's last; no expert reaches a dense group.  Also
// the routing (plan copy and per-layer copy) and the device counters.
__device__ __forceinline__ void write_one_token_plan(const PlanPtrs& plan, const OneTokenPlan& o, int lane, int my_e,
                                                     float w, int p) {
  const int k = o.k;
  if (lane < k) {
    plan.idx[lane] = my_e;
    plan.w[lane] = w;
    o.store_idx[lane] = my_e;
    o.store_w[lane] = w;
    plan.uniq[p] = my_e;
    plan.pass_expert[p] = my_e;
    plan.pass_ntok[p] = 1;
    plan.pass_tok[p * o.pmax] = 0;
    plan.pair_pass[lane] = p;
    plan.pair_slot[lane] = 0;
  }
  const int n_pass = k + (o.has_shared ? 1 : 0);
  if (o.big_min > 0)
    for (int q = lane; q < n_pass; q += 32) plan.small_order[q] = q;
  if (lane == 0) {
    if (o.has_shared) {
      plan.pass_tok[k * o.pmax] = 0;
      plan.shared_pass[0] = k;
      plan.shared_slot[0] = 0;
      plan.pass_expert[k] = o.E;
      plan.pass_ntok[k] = 1;
    }
    plan.hdr->n_pass = n_pass;
    plan.hdr->n_routed_pass = k;
    plan.hdr->n_uniq = k;
    plan.hdr->T = 1;
    plan.hdr->n_big = 0;
    plan.hdr->n_small = n_pass;
    DevCounters* dc = o.counters;
    atomicAdd(&dc->forwards, 1ull);
    atomicAdd(&dc->tokens, 1ull);
    atomicAdd(&dc->lookups, (unsigned long long)k);
    atomicAdd(&dc->bytes_touched, (unsigned long long)n_pass * o.record_bytes);
    atomicAdd(&dc->bytes_router, o.router_bytes);
  }
}

// Routing of one token inside an expert kernel (the router deferred, ExpertArgs
// route_logits set), by warp 0 of a block: the top-k of the logits (E <= 512), each pass's
// expert into s_pe (pass p = the p-th selected expert by id, the shared expert's pass k
// last), and with write_plan the plan for the kernels after (one block of the first
// expert kernel).
__device__ __forceinline__ void route_one_token(const ExpertArgs& a, int lane, int* s_pe, bool write_plan) {
  const int k = a.route.k;
  int my_e;
  float my_l;
  if (a.E <= 256) warp_topk<8>(a.route_logits, true, a.E, k, lane, my_e, my_l);
  else warp_topk<16>(a.route_logits, true, a.E, k, lane, my_e, my_l);
  const int pp = one_token_pass(k, lane, my_e);
  if (lane < k) s_pe[pp] = my_e;
  if (lane == 0) s_pe[k] = a.E;
  if (write_plan) write_one_token_plan(a.plan, a.route, lane, my_e, route_weight(a.route_kind, k, lane, my_l), pp);
}

}  // namespace moe
