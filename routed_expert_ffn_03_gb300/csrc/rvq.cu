// rvq.cu - residual-VQ (3 stages x 256 x 8 fp16 codebooks, 3 bits/weight) expert GEMV.
//
// "2.78T-parameter model on a laptop: the NVMe streaming inference engine WASTE",
// section "Idle weights only need to arrive on time": experts are stored residual-vector
// quantised at 3.00 bits per weight and the matrices are never expanded.  Here they are
// not expanded either: for a token x and one k-slice of 64 groups, the block first
// builds the table
//     LUT[s][c][q] = sum_i C_s[c][i] * x[8q + i]     (s < 3, c < 256, q < 64)
// in fp32 (192 KB of shared memory), and then every output row is
//     y[r] = sum_q LUT[0][c0(r,q)][q] + LUT[1][c1(r,q)][q] + LUT[2][c2(r,q)][q]
// which equals sum_k W[r][k] x[k] for W[r][8q+i] = C0[c0][i] + C1[c1][i] + C2[c2][i].
//
// Table build: D[q][e] = X[q][.] . Cb[e][.] is a [64 x 8] x [8 x 768] product done with
// m16n8k8 tensor-core mma into fp32 accumulators.  gate/up: the bf16 input and the fp16
// codebook entries are exact in tf32, one tf32 mma per product.  down: the fp32 SwiGLU
// input is split into fp16 hi + lo, two fp16 mma into one accumulator.  Each lane then writes
// its accumulators in a rotated order so that one store instruction touches 32 banks.
//
// Lookups: lane l owns row 32*block + l and visits the 64 groups in the order
// q = l XOR i (i = 0..63); the table is laid out [s][c][q] with 64 words per (s, c), so
// the bank of a lookup is q mod 32 and the 32 lanes hit 32 different banks whatever
// their codes.  The codes are read with 16-byte streaming loads straight into registers
// (one task = 32 rows x 64 groups = 6144 contiguous bytes), taken in two halves of 32
// groups so that the next half is always in flight while the current one is summed;
// 16 warps per block.
#include "common.cuh"
#include "kernels.h"
#include "route.cuh"

namespace moe {

constexpr int RV_NW = 16;                              // warps per block (divides 96)
constexpr int RV_LUT_BYTES = 3 * 256 * RVQ_KS * 4;     // 196608
constexpr int RV_VIN_BYTES = RVQ_KS * RVQ_GROUP * 4;   // 2048
constexpr int RV_PE_BYTES = 33 * 4;                      // pass -> expert of a token routed here (k <= 32)
constexpr int RV_SMEM = RV_LUT_BYTES + RV_VIN_BYTES + RV_PE_BYTES;
constexpr int RV_HQ = RVQ_TASK_BYTES / 512 / 2;        // 6 uint4 per lane per half task (32 groups)

// The table starts the block's dynamic shared memory.  Where that memory starts at
// shared address RV_DYN_BASE (1024 on this part: the reserved 1 KB comes first, and the
// kernel declares no static shared memory, which would come before it) a lookup is a
// single shared load [prmt result + constant]; elsewhere the base is added.
constexpr uint32_t RV_DYN_BASE = 1024;

// Table entry at shared address addr + delta + OFF (delta = 0 on the fast path).  The
// asm is volatile with a memory clobber, so it stays after the barrier that ends the
// table build and before the one that starts the next build.
template <uint32_t OFF, bool FAST>
__device__ __forceinline__ float lds_f32(uint32_t addr, uint32_t delta) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(FAST ? addr : addr + delta), "n"(OFF) : "memory");
  return v;
}

// Half HALF (groups 32 HALF .. 32 HALF + 31 of the lane stream) of a task's codes.
template <int HALF>
__device__ __forceinline__ void load_half(uint4 (&v)[RV_HQ], const uint8_t* task, int lane) {
#pragma unroll
  for (int j = 0; j < RV_HQ; ++j) v[j] = ldg_stream(task + ((HALF * RV_HQ + j) * 32 + lane) * 16);
}

__device__ __forceinline__ uint32_t word_of(const uint4 (&v)[RV_HQ], int w) {
  const uint4& q = v[w >> 2];
  return (w & 3) == 0 ? q.x : (w & 3) == 1 ? q.y : (w & 3) == 2 ? q.z : q.w;
}

// Adds the three lookups of each of the half's 32 groups (positions i = 32 HALF + 0..31,
// group q = lane XOR i) to the stage accumulators.
template <int HALF, bool FAST>
__device__ __forceinline__ void rvq_half_sum(const uint4 (&v)[RV_HQ], uint32_t delta, uint32_t l4, float& acc0,
                                             float& acc1, float& acc2) {
  constexpr uint32_t S0 = RV_DYN_BASE, S1 = RV_DYN_BASE + 65536, S2 = RV_DYN_BASE + 131072;
#pragma unroll
  for (int c4 = 0; c4 < 8; ++c4) {
    const uint32_t w0 = word_of(v, 3 * c4), w1 = word_of(v, 3 * c4 + 1), w2 = word_of(v, 3 * c4 + 2);
    const int i0 = 32 * HALF + 4 * c4;
    const uint32_t q0 = l4 ^ (uint32_t)((i0 + 0) << 2);
    const uint32_t q1 = l4 ^ (uint32_t)((i0 + 1) << 2);
    const uint32_t q2 = l4 ^ (uint32_t)((i0 + 2) << 2);
    const uint32_t q3 = l4 ^ (uint32_t)((i0 + 3) << 2);
    // prmt: byte 1 <- code byte, byte 0 <- 4q, bytes 2,3 <- 0  => (c << 8) | 4q
    acc0 += lds_f32<S0, FAST>(prmt(w0, q0, 0x5504), delta);
    acc1 += lds_f32<S1, FAST>(prmt(w0, q0, 0x5514), delta);
    acc2 += lds_f32<S2, FAST>(prmt(w0, q0, 0x5524), delta);
    acc0 += lds_f32<S0, FAST>(prmt(w0, q1, 0x5534), delta);
    acc1 += lds_f32<S1, FAST>(prmt(w1, q1, 0x5504), delta);
    acc2 += lds_f32<S2, FAST>(prmt(w1, q1, 0x5514), delta);
    acc0 += lds_f32<S0, FAST>(prmt(w1, q2, 0x5524), delta);
    acc1 += lds_f32<S1, FAST>(prmt(w1, q2, 0x5534), delta);
    acc2 += lds_f32<S2, FAST>(prmt(w2, q2, 0x5504), delta);
    acc0 += lds_f32<S0, FAST>(prmt(w2, q3, 0x5514), delta);
    acc1 += lds_f32<S1, FAST>(prmt(w2, q3, 0x5524), delta);
    acc2 += lds_f32<S2, FAST>(prmt(w2, q3, 0x5534), delta);
  }
}

// D += A B on tf32 operands (m16n8k8): a = (row g, col p), (g+8, p), (g, p+4), (g+8, p+4);
// b = (row p, col g), (p+4, g).  bf16 inputs and fp16 codebook entries are exact in tf32.
__device__ __forceinline__ void mma_1688_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct RvUnit {
  int pass, m, ks, expert, tok;   // tok: the pass's token (gate/up; one token per pass)
  const uint8_t* base;            // matrix base (codebooks first)
};

template <bool DOWN>
// s_pe: pass -> expert when the kernel routed the token itself (one token), else null
__device__ __forceinline__ RvUnit rv_unit(const ExpertArgs& a, int u, int nks, int p_begin, const RecGeom& rg,
                                          const int* s_pe) {
  constexpr int mats = DOWN ? 1 : 2;
  RvUnit U;
  U.ks = u % nks;
  const int pm = u / nks;
  U.m = pm % mats;
  const int pi = pm / mats;
  U.pass = a.range.order ? __ldcg(a.range.order + p_begin + pi) : p_begin + pi;
  U.expert = s_pe ? s_pe[U.pass] : __ldcg(a.plan.pass_expert + U.pass);
  U.tok = (DOWN || s_pe) ? 0 : __ldcg(a.plan.pass_tok + U.pass);
  U.base = expert_record(a, U.expert) + (DOWN ? rg.off[2] : (U.m == 0 ? rg.off[0] : rg.off[1]));
  return U;
}

// Block split cost model, fitted to per-warp timestamps of the gate/up kernel: warps take
// the tasks of a unit in rounds of RV_NW (one task each, ~2.3 us with some blocks idle,
// ~2.9 us with every block streaming), so a block pays one round (RV_RND_COST) per
// started round of each unit it touches, plus a table build and the unit's start per unit
// (RV_SEG_COST, ~2.0 to ~2.9 us).  Costs 6 to 9 per 8 of a round give the same split on
// the layer shapes measured.
constexpr int RV_RND_COST = 8;
constexpr int RV_SEG_COST = 7;

// The split itself (BlockSplit): groups of g blocks, every full group holding kk whole
// units and spending at most m_full per block; the G mod g blocks left over form the last
// group, which holds the rest of the units at most m_rem per block.

__host__ __device__ __forceinline__ int imin_hd(int x, int y) { return x < y ? x : y; }
__host__ __device__ __forceinline__ int imax_hd(int x, int y) { return x > y ? x : y; }

// Greedy advance: from task u * n + r (r a multiple of RV_NW), take whole rounds of unit
// u, then of the next units, while the budget B pays a segment and a round; stops at
// unit u_end.  nr = rounds per unit.  Returns the budget spent.
__host__ __device__ __forceinline__ int rv_advance(int& u, int& r, int B, int u_end, int nr) {
  const int B0 = B;
  while (u < u_end && B >= RV_SEG_COST + RV_RND_COST) {
    const int left = nr - r / RV_NW;
    const int take = imin_hd((B - RV_SEG_COST) / RV_RND_COST, left);
    B -= RV_SEG_COST + RV_RND_COST * take;
    if (take == left) {
      ++u;
      r = 0;
    } else {
      r += RV_NW * take;
    }
  }
  return B0 - B;
}

// cost of the tasks from u * n + r to the end of unit u_end - 1
__host__ __device__ __forceinline__ int rv_tail_cost(int u, int r, int u_end, int nr) {
  if (u >= u_end) return 0;
  int c = 0;
  if (r > 0) {
    c = RV_SEG_COST + RV_RND_COST * (nr - r / RV_NW);
    ++u;
  }
  return c + (u_end - u) * (RV_SEG_COST + RV_RND_COST * nr);
}

// `units` whole units over gg blocks: the budget per block (x) and the largest block cost
// (y) of the greedy split, whose last block takes what is left
__host__ __device__ __forceinline__ int2 rv_group(int units, int gg, int nr) {
  const int W = RV_SEG_COST + RV_RND_COST * nr;
  const int M0 = (units * W + RV_SEG_COST * (gg - 1) + gg - 1) / gg;
  int u = 0, r = 0, mx = 0;
  for (int i = 0; i < gg - 1; ++i) mx = imax_hd(mx, rv_advance(u, r, M0, units, nr));
  return make_int2(M0, imax_hd(mx, rv_tail_cost(u, r, units, nr)));
}

// Candidate c < 24 of the split of u_n units of n tasks over G blocks (G < u_n < 2 G):
// groups of g = c / 3 + 1 blocks holding kk = ceil(u_n g / G) - 1 + c mod 3 units each.
// Returns its largest block cost (RV_NO_SPLIT when it cannot hold the units) and the split.
constexpr int RV_NO_SPLIT = (1 << 26) - 1;
__host__ __device__ __forceinline__ int rv_candidate(int u_n, int n, int G, int c, BlockSplit& sp) {
  const int nr = (n + RV_NW - 1) / RV_NW;
  const int g = c / 3 + 1, ng = G / g, rem = G - ng * g;
  const int kk = (u_n * g + G - 1) / G - 1 + c % 3;
  const int ur = imax_hd(0, u_n - ng * kk);
  if (ng == 0 || kk < 1 || (ur > 0 && rem == 0)) return RV_NO_SPLIT;
  const int2 f = rv_group(imin_hd(kk, u_n), g, nr);
  const int2 rr = ur > 0 ? rv_group(ur, rem, nr) : make_int2(0, 0);
  sp = BlockSplit{g, kk, f.x, rr.x};
  return imin_hd(imax_hd(f.y, rr.y), RV_NO_SPLIT);
}

// The split with the least largest block cost among the 24 candidates (ties to the lower
// candidate; g = 1, kk = ceil(u_n / G) always holds the units).  On the device lane c of a
// warp evaluates candidate c and the warp takes the cheapest, so every warp of every block
// computes the same split; the host version (rv_plan_host) takes the same candidates in
// the same order and also weighs equal task ranges.
__device__ __forceinline__ BlockSplit rv_plan(int u_n, int n, int G, int lane) {
  BlockSplit sp{1, 0, 0, 0};
  const int cost = lane < 24 ? rv_candidate(u_n, n, G, lane, sp) : RV_NO_SPLIT;
  const unsigned best = __reduce_min_sync(0xffffffffu, (unsigned)cost << 5 | (unsigned)lane);
  const int wl = best & 31;
  return BlockSplit{__shfl_sync(0xffffffffu, sp.g, wl), __shfl_sync(0xffffffffu, sp.kk, wl),
                    __shfl_sync(0xffffffffu, sp.m_full, wl), __shfl_sync(0xffffffffu, sp.m_rem, wl)};
}

// block b's task range [t0, t1) under the split sp
__host__ __device__ __forceinline__ void rv_range(const BlockSplit& sp, int u_n, int n, int G, int b, int& t0,
                                                  int& t1) {
  if (sp.g < 0) {   // equal task ranges
    t0 = (int)((long long)u_n * n * b / G);
    t1 = (int)((long long)u_n * n * (b + 1) / G);
    return;
  }
  const int nr = (n + RV_NW - 1) / RV_NW;
  const int ng = G / sp.g, j = b / sp.g, i = b - j * sp.g;
  int u0, u1, B, gj;
  if (j < ng) {
    u0 = imin_hd(u_n, j * sp.kk);
    u1 = imin_hd(u_n, u0 + sp.kk);
    B = sp.m_full;
    gj = sp.g;
  } else {
    u0 = imin_hd(u_n, ng * sp.kk);
    u1 = u_n;
    B = sp.m_rem;
    gj = G - ng * sp.g;
  }
  int u = u0, r = 0;
  for (int ii = 0; ii < i; ++ii) rv_advance(u, r, B, u1, nr);
  t0 = u * n + r;
  if (i == gj - 1) {
    t1 = u1 * n;
  } else {
    rv_advance(u, r, B, u1, nr);
    t1 = u * n + r;
  }
}

// The host also weighs equal task ranges (g = -1), which a few unit counts favour; the
// device leaves them out (their exact cost needs every block's range).
static BlockSplit rv_plan_host(int u_n, int n, int G) {
  BlockSplit best{1, 0, 0, 0};
  int best_cost = RV_NO_SPLIT + 1;
  for (int c = 0; c < 24; ++c) {
    BlockSplit sp{};
    const int cost = rv_candidate(u_n, n, G, c, sp);
    if (cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  int eq_cost = 0;
  for (int b = 0; b < G; ++b) {
    int t0, t1, c = 0;
    rv_range(BlockSplit{-1, 0, 0, 0}, u_n, n, G, b, t0, t1);
    for (int i = t0; i < t1;) {   // segments: a table build and the started rounds of each unit
      const int e = imin_hd(t1, (i / n + 1) * n);
      c += RV_SEG_COST + RV_RND_COST * ((e - i + RV_NW - 1) / RV_NW);
      i = e;
    }
    eq_cost = imax_hd(eq_cost, c);
  }
  return eq_cost < best_cost ? BlockSplit{-1, 0, 0, 0} : best;
}

template <bool DOWN>
__global__ void __launch_bounds__(RV_NW * 32, 1) rvq_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* lutf = reinterpret_cast<float*>(smem);
  float* vin = reinterpret_cast<float*>(smem + RV_LUT_BYTES);
  constexpr int nthr = RV_NW * 32;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, p = lane & 3;
  constexpr int mats = DOWN ? 1 : 2;
  const RecGeom rg = rec_geom(WFMT_RVQ, a.H, a.F);
  const MatGeom g = rg.m[DOWN ? 2 : 0];
  const MatGeom gg = rg.m[0];
  const int nks = g.nks, ntask = g.ntask;
  const int rows32 = ntask * 32, rows32_gu = gg.ntask * 32;
  // gate/up waits for the router (plan, x) at once.  down reads only the plan, which is
  // older than the gate/up kernel (that kernel waited for it before letting this one
  // start), and the weights before it waits, so its first codes and codebooks are in
  // flight while gate/up finishes; the gate/up partials are read after the wait.
  const int G = gridDim.x;
  const int p_begin = a.range.p_begin;
  // Work split.  Every unit (pass, matrix, k-slice) costs a table build, so with no more
  // units than blocks each unit goes to its own group of blocks, which split its tasks:
  // every block builds one table; with at least two units per block, blocks take whole
  // units (contiguous unit ranges); in between, rv_plan balances the blocks' costs.  A
  // pass count fixed at launch (one token) comes with that split made on the host.
  int t0 = 0, t1 = -1;   // t1 < 0: not split yet
  if (a.split.g != 0) {
    const int u_n = max(0, a.range.p_end - p_begin) * mats * nks;
    rv_range(a.split, u_n, ntask, G, blockIdx.x, t0, t1);
  }
  if (!DOWN) {
    pdl_wait();
    pdl_launch_dependents();
  }
  bool waited = !DOWN;
  if (t1 < 0) {
    const int p_end = a.range.p_end >= 0 ? a.range.p_end : __ldcg(a.range.count ? a.range.count : &a.plan.hdr->n_pass);
    const int n_units = max(0, p_end - p_begin) * mats * nks;
    if (n_units >= 2 * G) {
      t0 = (int)((long long)n_units * blockIdx.x / G) * ntask;
      t1 = (int)((long long)n_units * (blockIdx.x + 1) / G) * ntask;
    } else if (n_units > 0 && n_units <= G) {
      const int u = (int)((long long)blockIdx.x * n_units / G);
      const int b_lo = (int)(((long long)u * G + n_units - 1) / n_units);
      const int b_hi = (int)(((long long)(u + 1) * G + n_units - 1) / n_units);
      const int i = blockIdx.x - b_lo, n = b_hi - b_lo;
      t0 = u * ntask + (int)((long long)ntask * i / n);
      t1 = u * ntask + (int)((long long)ntask * (i + 1) / n);
    } else if (n_units > 0) {
      rv_range(rv_plan(n_units, ntask, G, lane), n_units, ntask, G, blockIdx.x, t0, t1);
    } else {
      t1 = 0;
    }
  }
  // One token routed here (the router deferred, writing the logits only): warp 0 takes
  // the top-k (gate/up after its wait; down before it, since the logits are older than
  // the gate/up kernel, which waited for them before letting this one start), gate/up's
  // block 0 writes the plan for the kernels after, and each block keeps pass -> expert.
  int* s_pe = reinterpret_cast<int*>(smem + RV_LUT_BYTES + RV_VIN_BYTES);
  if (a.route_logits) {
    if (warp == 0) route_one_token(a, lane, s_pe, !DOWN && blockIdx.x == 0);
    __syncthreads();
  }
  const uint32_t l4 = (uint32_t)lane << 2;
  const uint32_t delta = smem_u32(smem) - RV_DYN_BASE;   // 0 on the fast path

  if (t0 >= t1 && !waited) {
    pdl_wait();
    pdl_launch_dependents();
  }
  static_assert(RVQ_KS * RVQ_GROUP == RV_NW * 32, "one input element of a k-slice per thread");
  for (int i = t0; i < t1;) {
    const int u = i / ntask;
    const int seg_end = min(t1, (u + 1) * ntask);
    const RvUnit U = rv_unit<DOWN>(a, u, nks, p_begin, rg, a.route_logits ? s_pe : nullptr);
    const uint8_t* codes = U.base + RVQ_CB_BYTES + (size_t)U.ks * ntask * RVQ_TASK_BYTES;
    const int useg = u * ntask;

    // first half of this warp's first task goes in flight before the table is built
    int ti = i + warp;
    uint4 ha[RV_HQ], hb[RV_HQ];
    if (ti < seg_end) load_half<0>(ha, codes + (size_t)(ti - useg) * RVQ_TASK_BYTES, lane);

    // this warp's codebook fragments (6 n-tiles of 8 entries) go in flight now as well:
    // gate/up as tf32 (elements p and p + 4 of the entry), down as fp16 pairs (2p, 2p + 1)
    constexpr int RV_NT = 96 / RV_NW;
    uint32_t bfr[RV_NT], bfr1[RV_NT];
    {
      const uint32_t* cb = reinterpret_cast<const uint32_t*>(U.base);  // fp16 [768][8]
      const __half* cbh = reinterpret_cast<const __half*>(U.base);
#pragma unroll
      for (int n = 0; n < RV_NT; ++n) {
        const int e = (warp + n * RV_NW) * 8 + gq;
        if (DOWN) {
          bfr[n] = __ldg(cb + e * 4 + p);
          bfr1[n] = 0u;
        } else {
          bfr[n] = __float_as_uint(__half2float(__ldg(cbh + e * 8 + p)));
          bfr1[n] = __float_as_uint(__half2float(__ldg(cbh + e * 8 + p + 4)));
        }
      }
    }

    if (!waited) {
      pdl_wait();
      pdl_launch_dependents();
      waited = true;
    }
    // gate/up: this thread's input element of the k-slice goes in flight with the rest
    float xv = 0.f;
    if (!DOWN) {
      const int k = U.ks * RVQ_KS * RVQ_GROUP + (int)threadIdx.x;   // one element per thread
      if (k < g.K) xv = bf16_bits_to_float(a.x[(size_t)U.tok * a.H + k]);
    }
    __syncthreads();  // the previous unit's table is no longer read
    {
      const int kbase = U.ks * RVQ_KS * RVQ_GROUP;
      for (int e = threadIdx.x; e < RVQ_KS * RVQ_GROUP; e += nthr) {
        const int k = kbase + e;
        float v = 0.f;
        if (k < g.K) {
          if (!DOWN) {
            v = xv;
          } else {
            const float* pg = a.part_gu + ((size_t)(U.pass * 2 + 0) * gg.nks) * rows32_gu + k;
            const float* pu = a.part_gu + ((size_t)(U.pass * 2 + 1) * gg.nks) * rows32_gu + k;
            float gs = 0.f, us = 0.f;
            for (int s0 = 0; s0 < gg.nks; s0 += 16) {  // 32 loads in flight, added in slice order
              float gv[16], uv[16];
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                const bool in = s0 + q < gg.nks;
                gv[q] = in ? __ldcg(pg + (size_t)(s0 + q) * rows32_gu) : 0.f;
                uv[q] = in ? __ldcg(pu + (size_t)(s0 + q) * rows32_gu) : 0.f;
              }
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                gs += gv[q];
                us += uv[q];
              }
            }
            v = gs / (1.f + expf(-gs)) * us;
          }
        }
        vin[e] = v;
      }
    }
    __syncthreads();
    {
      int jofs[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) jofs[r] = 8 * ((p + r) & 3);
      // A fragments: rows = groups q, k = element i.  gate/up: the bf16 input is exact in
      // tf32, one tf32 mma per product; down: the fp32 input as fp16 hi + lo, two mma.
      uint32_t at[4][4];
      uint32_t ahi[4][2], alo[4][2];
      if (!DOWN) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            at[mt][r] = __float_as_uint(vin[(16 * mt + gq + 8 * (r & 1)) * 8 + p + 4 * (r >> 1)]);
      } else {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int q = 16 * mt + gq + 8 * h;
            __half h0, l0, h1, l1;
            split_half(vin[q * 8 + 2 * p], h0, l0);
            split_half(vin[q * 8 + 2 * p + 1], h1, l1);
            ahi[mt][h] = pack_half2(h0, h1);
            alo[mt][h] = pack_half2(l0, l1);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < RV_NT; ++n) {
        const int e0 = (warp + n * RV_NW) * 8;
        const uint32_t b = bfr[n];
#pragma unroll
        for (int P = 0; P < 2; ++P) {
          float dA[4] = {0.f, 0.f, 0.f, 0.f}, dB[4] = {0.f, 0.f, 0.f, 0.f};
          if (!DOWN) {
            mma_1688_tf32(dA, at[2 * P], b, bfr1[n]);
            mma_1688_tf32(dB, at[2 * P + 1], b, bfr1[n]);
          } else {
            mma_1688(dA, ahi[2 * P][0], ahi[2 * P][1], b);
            mma_1688(dA, alo[2 * P][0], alo[2 * P][1], b);
            mma_1688(dB, ahi[2 * P + 1][0], ahi[2 * P + 1][1], b);
            mma_1688(dB, alo[2 * P + 1][0], alo[2 * P + 1][1], b);
          }
          // value j of entry e: q = 32P + g + 8j  (j: A row g, A row g+8, B row g, B row g+8).
          // Store r writes value j = (p + r) & 3, so one store touches 32 banks: the values
          // are rotated left by p with two conditional swaps instead of indexed selects.
          float v0[4] = {dA[0], dA[2], dB[0], dB[2]}, v1[4] = {dA[1], dA[3], dB[1], dB[3]};
          if (p & 1) {
            const float t0 = v0[0], t1 = v1[0];
            v0[0] = v0[1]; v0[1] = v0[2]; v0[2] = v0[3]; v0[3] = t0;
            v1[0] = v1[1]; v1[1] = v1[2]; v1[2] = v1[3]; v1[3] = t1;
          }
          if (p & 2) {
            float t = v0[0]; v0[0] = v0[2]; v0[2] = t;
            t = v0[1]; v0[1] = v0[3]; v0[3] = t;
            t = v1[0]; v1[0] = v1[2]; v1[2] = t;
            t = v1[1]; v1[1] = v1[3]; v1[3] = t;
          }
          float* row0 = lutf + (size_t)(e0 + 2 * p) * RVQ_KS + 32 * P + gq;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            row0[jofs[r]] = v0[r];
            row0[jofs[r] + RVQ_KS] = v1[r];
          }
        }
      }
    }
    __syncthreads();

    // tasks of this unit: warp-strided; half tasks double-buffered in registers
    float* outp = (DOWN ? a.part_d + ((size_t)U.pass * nks + U.ks) * rows32
                        : a.part_gu + ((size_t)(U.pass * 2 + U.m) * nks + U.ks) * rows32);
    if (delta == 0u) {
      while (ti < seg_end) {
        const uint8_t* task = codes + (size_t)(ti - useg) * RVQ_TASK_BYTES;
        load_half<1>(hb, task, lane);
        float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f;
        rvq_half_sum<0, true>(ha, 0u, l4, acc0, acc1, acc2);
        const int tn = ti + RV_NW;
        if (tn < seg_end) load_half<0>(ha, codes + (size_t)(tn - useg) * RVQ_TASK_BYTES, lane);
        rvq_half_sum<1, true>(hb, 0u, l4, acc0, acc1, acc2);
        outp[(size_t)(ti - useg) * 32 + lane] = (acc0 + acc1) + acc2;
        ti = tn;
      }
    } else {
      while (ti < seg_end) {
        const uint8_t* task = codes + (size_t)(ti - useg) * RVQ_TASK_BYTES;
        load_half<1>(hb, task, lane);
        float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f;
        rvq_half_sum<0, false>(ha, delta, l4, acc0, acc1, acc2);
        const int tn = ti + RV_NW;
        if (tn < seg_end) load_half<0>(ha, codes + (size_t)(tn - useg) * RVQ_TASK_BYTES, lane);
        rvq_half_sum<1, false>(hb, delta, l4, acc0, acc1, acc2);
        outp[(size_t)(ti - useg) * 32 + lane] = (acc0 + acc1) + acc2;
        ti = tn;
      }
    }
    i = seg_end;
  }
}

cudaError_t rvq_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(rvq_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, RV_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rvq_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, RV_SMEM);
}

// the host-made split of a pass count fixed at launch, when units are between one and two
// per block (g = 0: none, the kernel splits)
static BlockSplit host_split(const ExpertArgs& a, bool down, int grid) {
  if (a.range.p_end < 0) return BlockSplit{0, 0, 0, 0};
  const MatGeom g = rec_geom(WFMT_RVQ, a.H, a.F).m[down ? 2 : 0];
  const int u_n = std::max(0, a.range.p_end - a.range.p_begin) * (down ? 1 : 2) * g.nks;
  if (u_n <= grid || u_n >= 2 * grid) return BlockSplit{0, 0, 0, 0};
  return rv_plan_host(u_n, g.ntask, grid);
}
}  // namespace moe

// Diagnostic (include/moe.h): the task ranges of the lookup kernel's blocks for u_n units
// of ntask tasks over a grid of `grid` blocks when units are between one and two per
// block, made by the same functions as the kernel's split.
extern "C" int moe_rvq_block_split(int u_n, int ntask, int grid, int* t0, int* t1) {
  if (u_n <= grid || u_n >= 2 * grid || ntask <= 0 || grid <= 0 || !t0 || !t1 ||
      (long long)u_n * ntask > 0x7fffffffLL)
    return 1;
  const moe::BlockSplit sp = moe::rv_plan_host(u_n, ntask, grid);
  for (int b = 0; b < grid; ++b) moe::rv_range(sp, u_n, ntask, grid, b, t0[b], t1[b]);
  return 0;
}

namespace moe {

cudaError_t launch_rvq_gateup(const ExpertArgs& a0, int grid, cudaStream_t s) {
  ExpertArgs a = a0;
  a.split = host_split(a0, false, grid);
  return launch_pdl(rvq_kernel<false>, grid, RV_NW * 32, RV_SMEM, s, a);
}
cudaError_t launch_rvq_down(const ExpertArgs& a0, int grid, cudaStream_t s) {
  ExpertArgs a = a0;
  a.split = host_split(a0, true, grid);
  return launch_pdl(rvq_kernel<true>, grid, RV_NW * 32, RV_SMEM, s, a);
}

}  // namespace moe
