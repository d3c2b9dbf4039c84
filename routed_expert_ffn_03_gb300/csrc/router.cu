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
// Phase 1 (all blocks): each warp owns (expert e, 512-wide chunk c of H) and writes the
// partial dot products of all T tokens.  Phase 2 (the block that arrives last, found
// with an atomic ticket; no block waits on another): sums the partials in chunk order
// (all (token, expert) pairs in parallel),
// selects the top-k per token (one warp per token), and buckets the (token, rank) pairs
// by expert into "passes" of up to pmax tokens: routed experts in ascending id, tokens
// ascending, then the shared expert.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int RCH = 512;
int router_nch(int H) { return cdiv(H, RCH); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int LOGIT_SMEM = 8192;  // floats of logits staged per chunk of tokens

__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  extern __shared__ int sm[];
  __shared__ float s_inv[ROUTER_FUSED_MAXT];
  __shared__ float s_red[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int nch = cdiv(a.H, RCH);
  const int nitems = a.E * nch;
  const bool fused = a.xres != nullptr;

  pdl_wait();  // x (and the residual) come from the kernels before
  pdl_launch_dependents();
  if (fused) {
    for (int t = 0; t < a.T; ++t) {
      const float inv = block_inv_rms(a.xres + (size_t)t * a.H, a.yprev ? a.yprev + (size_t)t * a.H : nullptr,
                                      a.H, a.eps, s_red);
      if (threadIdx.x == 0) s_inv[t] = inv;
    }
    __syncthreads();
  }

  if (fused) {
    // xn is not read by this kernel: each block writes a disjoint slice of it
    const int per = cdiv(a.H, gridDim.x);
    for (int t = 0; t < a.T; ++t) {
      const float inv = s_inv[t];
      for (int h = blockIdx.x * per + threadIdx.x; h < min(a.H, (blockIdx.x + 1) * per); h += blockDim.x) {
        const size_t o = (size_t)t * a.H + h;
        float v = __ldcg(a.xres + o);
        if (a.yprev) v += __ldcg(a.yprev + o);
        a.xn_out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(v * inv));
      }
    }
  }

  // ---------------- phase 1: partial logits
  for (int item = blockIdx.x * nwarps + warp; item < nitems; item += gridDim.x * nwarps) {
    const int e = item / nch, c = item % nch;
    const int h0 = c * RCH, h1 = min(a.H, h0 + RCH);
    const float* wr = a.W + (size_t)e * a.H;
    for (int t0 = 0; t0 < a.T; t0 += 8) {
      const int nt = min(8, a.T - t0);
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int h = h0 + lane * 4; h < h1; h += 128) {
        const float4 wv = __ldg(reinterpret_cast<const float4*>(wr + h));
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
          if (tt < nt) {
            float x0, x1, x2, x3;
            if (fused) {
              const size_t o = (size_t)(t0 + tt) * a.H + h;
              float4 v = __ldcg(reinterpret_cast<const float4*>(a.xres + o));
              if (a.yprev) {
                const float4 y = __ldcg(reinterpret_cast<const float4*>(a.yprev + o));
                v.x += y.x; v.y += y.y; v.z += y.z; v.w += y.w;
              }
              const float inv = s_inv[t0 + tt];
              x0 = __bfloat162float(__float2bfloat16_rn(v.x * inv));
              x1 = __bfloat162float(__float2bfloat16_rn(v.y * inv));
              x2 = __bfloat162float(__float2bfloat16_rn(v.z * inv));
              x3 = __bfloat162float(__float2bfloat16_rn(v.w * inv));
            } else {
              const uint2 xb = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)(t0 + tt) * a.H + h));
              x0 = __uint_as_float(xb.x << 16);
              x1 = __uint_as_float(xb.x & 0xffff0000u);
              x2 = __uint_as_float(xb.y << 16);
              x3 = __uint_as_float(xb.y & 0xffff0000u);
            }
            acc[tt] = fmaf(wv.x, x0, acc[tt]);
            acc[tt] = fmaf(wv.y, x1, acc[tt]);
            acc[tt] = fmaf(wv.z, x2, acc[tt]);
            acc[tt] = fmaf(wv.w, x3, acc[tt]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        const float v = warp_sum(acc[tt]);
        if (lane == 0 && tt < nt) a.partial[((size_t)e * nch + c) * a.T + t0 + tt] = v;
      }
    }
  }

  // ---------------- ticket: the last block continues
  __shared__ int s_last, s_routed;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int tk = atomicAdd(a.ticket, 1u);
    s_last = (tk == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int E = a.E, T = a.T, k = a.k, pmax = a.pmax;
  float* slog = reinterpret_cast<float*>(sm);   // [tc][E]
  int* s_cnt = sm + LOGIT_SMEM;                 // [E]
  int* s_off = s_cnt + E;                       // [E]
  int* s_idx = s_off + E;                       // [T*k]
  int* s_pos = s_idx + T * k;                   // [T*k]


  // ---------------- phase 2a: logits (all (t, e) in parallel), then top-k per token
  const int tc = max(1, min(T, LOGIT_SMEM / E));
  for (int tb = 0; tb < T; tb += tc) {
    const int nt = min(tc, T - tb);
    for (int q = threadIdx.x; q < nt * E; q += blockDim.x) {
      const int tl = q / E, e = q % E;
      const float* pp = a.partial + (size_t)e * nch * T + tb + tl;
      float s = 0.f;
#pragma unroll 8
      for (int c = 0; c < nch; ++c) s += __ldcg(pp + (size_t)c * T);
      slog[tl * E + e] = s;
    }
    __syncthreads();
    for (int tl = warp; tl < nt; tl += nwarps) {
      const int t = tb + tl;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? slog[tl * E + e] : -INFINITY;
      }
      int my_e = 0;
      float my_l = 0.f;
      for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = lane + 32 * i;
          if (e < E && (v[i] > bv || (v[i] == bv && e < be))) { bv = v[i]; be = e; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (lane + 32 * i == be) v[i] = -INFINITY;
        if (lane == j) { my_e = be; my_l = bv; }
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
    __syncthreads();
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();

  // ---------------- phase 2b: position of each pair within its expert (tokens ascending)
  if (warp == 0) {
    for (int t = 0; t < T; ++t) {
      if (lane < k) {
        const int e = s_idx[t * k + lane];   // the k experts of a token are distinct
        const int pos = s_cnt[e];
        s_cnt[e] = pos + 1;
        s_pos[t * k + lane] = pos;
      }
      __syncwarp();
    }
    // exclusive scan over experts of (passes, unique flag); lane owns a contiguous run
    const int run = cdiv(E, 32);
    const int e0 = min(E, lane * run), e1 = min(E, e0 + run);
    int np = 0, nu = 0;
    for (int e = e0; e < e1; ++e) {
      np += cdiv(s_cnt[e], pmax);
      nu += s_cnt[e] > 0;
    }
    int inp = np, inu = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, inp, o);
      const int a2 = __shfl_up_sync(0xffffffffu, inu, o);
      if (lane >= o) { inp += a1; inu += a2; }
    }
    int off = inp - np, uoff = inu - nu;
    for (int e = e0; e < e1; ++e) {
      s_off[e] = off;
      const int c = s_cnt[e];
      if (c > 0) a.plan.uniq[uoff++] = e;
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
      s_routed = tot_p;
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
  const int routed_passes = s_routed;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = s_cnt[e];
    for (int i = 0; i * pmax < c; ++i) {
      a.plan.pass_expert[s_off[e] + i] = e;
      a.plan.pass_ntok[s_off[e] + i] = min(pmax, c - i * pmax);
    }
  }
  for (int q = threadIdx.x; q < T * k; q += blockDim.x) {
    const int e = s_idx[q], pos = s_pos[q];
    const int pass = s_off[e] + pos / pmax, slot = pos % pmax;
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
  // per-token path, both lists in ascending expert id then token order
  __syncthreads();
  if (threadIdx.x == 0) {
    int nb = 0, ns = 0;
    auto emit = [&](int expert, int first, int c) {
      if (a.big_min > 0 && c >= a.big_min) {
        const int nch = cdiv(c, GEMM_MAX_TOKENS), base = c / nch, rem = c % nch;
        int start = 0;
        for (int q = 0; q < nch; ++q) {
          const int sz = base + (q < rem ? 1 : 0);
          a.plan.big[3 * nb + 0] = expert;
          a.plan.big[3 * nb + 1] = first + start;
          a.plan.big[3 * nb + 2] = sz;
          ++nb;
          start += sz;
        }
      } else if (a.big_min > 0) {
        for (int i = 0; i < c; ++i) a.plan.small_order[ns++] = first + i;
      }
    };
    if (a.big_min > 0) {
      for (int e = 0; e < E; ++e)
        if (s_cnt[e] > 0) emit(e, s_off[e], s_cnt[e]);
      if (a.has_shared) emit(E, routed_passes, T);
    }
    a.plan.hdr->n_big = nb;
    a.plan.hdr->n_small = a.big_min > 0 ? ns : routed_passes + (a.has_shared ? cdiv(T, pmax) : 0);
    *a.ticket = 0u;  // ready for the next launch (stream-ordered)
  }
}

cudaError_t router_set_attributes() {
  return cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              160 * 1024);
}

cudaError_t launch_router(const RouterArgs& a, int num_sms, cudaStream_t s) {
  const int nch = router_nch(a.H);
  const int nitems = a.E * nch;
  int grid = cdiv(nitems, 8);
  grid = std::max(1, std::min(grid, num_sms));
  const size_t smem = (size_t)(LOGIT_SMEM + 2 * a.E + 2 * a.T * a.k) * sizeof(int);
  return launch_pdl(router_kernel, grid, 256, smem, s, a);
}

}  // namespace moe
