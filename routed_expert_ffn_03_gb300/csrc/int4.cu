// int4.cu - int4 (symmetric, group 128, fp16 scales) expert kernels.
//
// gate/up:  part_gu[pass][m][ks][slot][row] = sum over k in slice ks of W_m[row][k] x[k]
// down:     part_d[pass][ks][slot][row] = sum over k in slice ks of W_d[row][k] h[k],
//           h = silu(g) * u with g, u the gate / up partials added in k-slice order
//           (computed by the down kernel for the slice it works on).
// A "pass" is one expert with up to 4 tokens (slots).
//
// Data movement: each of the 16 warps of a block streams its own tasks (32 rows x 2
// groups of 128 inputs = 4224 B, contiguous in the kernel layout) with 1-D bulk TMA
// copies into its own ring of shared-memory slots, D tasks ahead of the one it computes,
// and reads a slot with conflict-free 16-byte loads.
//
// Arithmetic: a lane dequantises its own m16n8k16 A fragment from 8 nibbles (q + 1032
// is built as an fp16 bit pattern with one LOP3 per pair and the offset removed exactly),
// and the warp-level tensor-core mma multiplies it by the activations, split into fp16
// hi + lo parts so that hi + lo reproduces fp32 inputs to 2^-22; products of q and an
// fp16 part are exact and accumulate in fp32.  The fp16 group scale multiplies each
// 128-wide group's fp32 sum.  (Feeding q + 1032 itself and removing 1032 * sum(x) after
// the mma saves the fp16 subtractions but loses three orders of magnitude of accuracy
// to the fp32 accumulation of the large offsets, so it is not done.)  The 8 mma columns
// carry (token, hi/lo) pairs, so one pass serves up to 4 tokens at the cost of one.
//
// Work split (both kernels): tasks in a fixed order, blocks take equal contiguous ranges,
// and a block deals its range to its warps round-robin (task i -> warp (i - t0) mod NW);
// each warp walks its tasks with incremental counters.  gate/up tasks run in (pass,
// row block, matrix, k-slice) order; down tasks in (pass, k-slice, row block) order and
// leave k-slice partials for the combine kernel.  The B fragments are kept only for the
// mma columns that carry tokens (2 per token), which leaves room for 3 ring slots per
// warp when a pass has one token.  They are stored per column, k-steps contiguous (two
// k-steps per 16-byte load, columns padded so the lanes of a load hit distinct banks);
// a lane whose column carries no token reads a live column instead, and its results
// land in mma columns nobody reads.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int I4_STAGE = I4_KS * I4_PAIR_BLOCK;          // 4224 B
constexpr int I4_SLICE_KSTEPS = I4_KS * I4_GROUP / 16;   // 16 mma k-steps per slice
constexpr int I4_MAX_RECS = 512;                         // passes one block may touch
constexpr int I4_STATIC_SMEM = I4_MAX_RECS * 8 + 128;

// B fragments: [column][k-step] uint2, column stride kstride(n k-steps) = n + 2 (16 B of
// padding: consecutive columns start 4 or 20 banks apart, so the 8 columns of a 16-byte
// load phase are conflict-free).
__host__ __device__ constexpr int i4_kstride(int nks16) { return nks16 + 2; }

constexpr int DN_UMAX = 2;   // units (pass, k-slice) a down block prepares up front

// nb = mma columns that carry data (2 per token of the widest pass).
template <int NW, int D>
struct I4Smem {
  static constexpr int ring = NW * D * I4_STAGE;
  static constexpr int bars = NW * D * 8;
  static constexpr int gateup(int H, int nb) { return ring + bars + nb * 4 * i4_kstride(H / 16) * 8; }
  // down keeps, for each of up to DN_UMAX units, B fragments for all 8 columns (one slice
  // is small) and the slice inputs
  static constexpr int dn_frag = 8 * 4 * i4_kstride(I4_SLICE_KSTEPS) * 8;
  static constexpr int dn_vin = I4_PMAX * I4_KS * I4_GROUP * 4;
  static constexpr int down() { return ring + bars + DN_UMAX * (dn_frag + dn_vin); }
};

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;  // (a & b) ^ c
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 8 nibbles -> the four half2 registers of an m16n8k16 A fragment (exact integers q):
// (u & 0xF) ^ 8 = q + 8 under the fp16 exponent of 1024 gives 1032 + q; the high nibble
// of a byte gives 1152 + 16 q, rescaled by 1/16.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  const uint32_t LO = 0x000F000Fu, HI = 0x00F000F0u;
  const uint32_t XLO = 0x64086408u, XHI = 0x64806480u;
  const __half2 off_lo = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
  const __half2 sixteenth = __halves2half2(__float2half_rn(0.0625f), __float2half_rn(0.0625f));
  const __half2 off_hi = __halves2half2(__float2half_rn(-72.f), __float2half_rn(-72.f));
  const uint32_t w2 = w >> 8;
  uint32_t t0 = lop3_and_xor(w, LO, XLO);    // rows g,   k 2p / 2p+1
  uint32_t t1 = lop3_and_xor(w, HI, XHI);    // rows g+8, k 2p / 2p+1
  uint32_t t2 = lop3_and_xor(w2, LO, XLO);   // rows g,   k 2p+8 / 2p+9
  uint32_t t3 = lop3_and_xor(w2, HI, XHI);   // rows g+8, k 2p+8 / 2p+9
  __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&t0), off_lo);
  __half2 h1 = __hfma2(*reinterpret_cast<__half2*>(&t1), sixteenth, off_hi);
  __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&t2), off_lo);
  __half2 h3 = __hfma2(*reinterpret_cast<__half2*>(&t3), sixteenth, off_hi);
  a0 = *reinterpret_cast<uint32_t*>(&h0);
  a1 = *reinterpret_cast<uint32_t*>(&h1);
  a2 = *reinterpret_cast<uint32_t*>(&h2);
  a3 = *reinterpret_cast<uint32_t*>(&h3);
}

__device__ __forceinline__ uint32_t pick4(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// One task: 32 rows x NGRP (<= 2) groups from a stage; adds W . x into acc[tile][4].
// stl = stage + 16 * lane, sts = stage + 1024 + 4 * (lane / 4) (the lane's scale word),
// xl = the lane's B-fragment column at the task's first k-step.
template <int NGRP>
__device__ __forceinline__ void i4_task(const uint8_t* stl, const uint8_t* sts, const uint2* xl, float (&acc)[2][4]) {
#pragma unroll
  for (int gi = 0; gi < NGRP; ++gi) {
    const uint8_t* blk = stl + gi * I4_PAIR_BLOCK;
    const uint4 wa0 = *reinterpret_cast<const uint4*>(blk);
    const uint4 wb0 = *reinterpret_cast<const uint4*>(blk + 512);
    const uint4 wa1 = *reinterpret_cast<const uint4*>(blk + I4_BLOCK);
    const uint4 wb1 = *reinterpret_cast<const uint4*>(blk + I4_BLOCK + 512);
    const uint32_t sc0 = *reinterpret_cast<const uint32_t*>(sts + gi * I4_PAIR_BLOCK);
    const uint32_t sc1 = *reinterpret_cast<const uint32_t*>(sts + gi * I4_PAIR_BLOCK + I4_BLOCK);
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint4 bb = *reinterpret_cast<const uint4*>(xl + gi * 8 + 2 * jj);   // k-steps 2jj, 2jj+1
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * jj + h;
        const uint32_t b0 = h ? bb.z : bb.x, b1 = h ? bb.w : bb.y;
        uint32_t x0, x1, x2, x3;
        dequant8(pick4(j < 4 ? wa0 : wb0, j & 3), x0, x1, x2, x3);
        mma_16816(c0, x0, x1, x2, x3, b0, b1);
        dequant8(pick4(j < 4 ? wa1 : wb1, j & 3), x0, x1, x2, x3);
        mma_16816(c1, x0, x1, x2, x3, b0, b1);
      }
    }
    const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(&sc0));
    const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(&sc1));
    acc[0][0] = fmaf(s0.x, c0[0], acc[0][0]);
    acc[0][1] = fmaf(s0.x, c0[1], acc[0][1]);
    acc[0][2] = fmaf(s0.y, c0[2], acc[0][2]);
    acc[0][3] = fmaf(s0.y, c0[3], acc[0][3]);
    acc[1][0] = fmaf(s1.x, c1[0], acc[1][0]);
    acc[1][1] = fmaf(s1.x, c1[1], acc[1][1]);
    acc[1][2] = fmaf(s1.y, c1[2], acc[1][2]);
    acc[1][3] = fmaf(s1.y, c1[3], acc[1][3]);
  }
}

// The B-fragment column a lane reads: its own (token slot g/2, part g%2, pair p) when
// g < nb, else the same pair of a live column.
__device__ __forceinline__ int i4_lane_col(int lane, int nb) {
  const int gq = lane >> 2;
  return (gq < nb ? gq : gq % nb) * 4 + (lane & 3);
}

// B fragment of mma column n = g (token slot n/2, part n%2) for one k-step: elements
// v[0], v[1], v[8], v[9] (inputs k0 + 2p, +1, +8, +9), fp16 hi or lo part.
__device__ __forceinline__ uint2 bfrag(const float* v, int part) {
  __half hi[4], lo[4];
  split_half(v[0], hi[0], lo[0]);
  split_half(v[1], hi[1], lo[1]);
  split_half(v[8], hi[2], lo[2]);
  split_half(v[9], hi[3], lo[3]);
  uint2 r;
  r.x = part ? pack_half2(lo[0], lo[1]) : pack_half2(hi[0], hi[1]);
  r.y = part ? pack_half2(lo[2], lo[3]) : pack_half2(hi[2], hi[3]);
  return r;
}

// B fragments of one pass's tokens for nks16 k-steps from fp32 values val(ts, k)
// (k relative to the first k-step), into xf[column n*4 + p][k-step] (stride kstride).
template <class Val>
__device__ __forceinline__ void build_bfrags(uint2* xf, int nks16, int nb, int tid, int nthr, Val val) {
  const int per = nb * 4, ks = i4_kstride(nks16);
  for (int e = tid; e < nks16 * per; e += nthr) {
    const int kk = e / per, col = e - kk * per, n = col >> 2, pp = col & 3;
    float f[10];
    const int kb = kk * 16 + 2 * pp;
    f[0] = val(n >> 1, kb);
    f[1] = val(n >> 1, kb + 1);
    f[8] = val(n >> 1, kb + 8);
    f[9] = val(n >> 1, kb + 9);
    xf[col * ks + kk] = bfrag(f, n & 1);
  }
}

// The 8 fragment words of k-step kk of token slot ts (4 pairs x hi/lo) from its 16 bf16
// inputs (u0, u1: inputs 2i, 2i+1 in word i), into xf[column n*4 + p][k-step].
__device__ __forceinline__ void bfrag_kstep(uint2* xf, int kstride, int ts, int kk, const uint4& u0, const uint4& u1) {
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    float f[10];
    f[0] = __uint_as_float(w[pp] << 16);
    f[1] = __uint_as_float(w[pp] & 0xffff0000u);
    f[8] = __uint_as_float(w[pp + 4] << 16);
    f[9] = __uint_as_float(w[pp + 4] & 0xffff0000u);
    xf[((2 * ts) * 4 + pp) * kstride + kk] = bfrag(f, 0);
    xf[((2 * ts + 1) * 4 + pp) * kstride + kk] = bfrag(f, 1);
  }
}

// B fragments of all K for the tokens tok[0..ntok) of a pass straight from the bf16 input:
// one thread per (token, k-step) reads its 16 inputs with two 16-byte loads.
__device__ __forceinline__ void build_bfrags_x(uint2* xf, const uint16_t* x, int H, const int (&tok)[I4_PMAX],
                                               int ntok, int tid, int nthr) {
  const int nks16 = H / 16, ks = i4_kstride(nks16);
  for (int e = tid; e < ntok * nks16; e += nthr) {
    const int ts = e / nks16, kk = e - ts * nks16;
    int t = tok[0];
#pragma unroll
    for (int q = 1; q < I4_PMAX; ++q)
      if (ts == q) t = tok[q];
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H + kk * 16);
    bfrag_kstep(xf, ks, ts, kk, __ldg(src), __ldg(src + 1));
  }
}

// ------------------------------------------------------------------ warp-local staging
// Every warp streams its own tasks: lane 0 starts the bulk copy of task j + D into the
// ring slot task j has just released, so the block's warps issue copies in parallel and
// each keeps D tasks in flight.  full[w][d] completes when slot d of warp w has landed.
// No proxy fence is needed before the copy: the warp's shared-memory reads of the slot
// returned their data into registers that the task's mma instructions consumed, which
// the warp issued before this point, so the copy cannot overwrite data still being read.
__device__ __forceinline__ void stage_issue(int lane, uint32_t full, uint32_t dst, const void* src, uint32_t bytes) {
  if (lane == 0) {
    mbar_arrive_expect_tx(full, bytes);
    bulk_g2s(dst, src, bytes, full);
  }
}

__device__ __forceinline__ int pass_of(const ExpertArgs& a, int p_begin, int pi) {
  return a.range.order ? __ldcg(a.range.order + p_begin + pi) : p_begin + pi;
}

// Wait for a full slot (all lanes agree); on a time-out the block is marked aborted.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, volatile int* abort, const ExpertArgs& a,
                                           int lane) {
  bool ok = !*abort && mbar_wait_bounded(bar, parity, a.budget);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && !*abort && lane == 0) {
    *abort = 1;
    atomicOr(a.status, ST_TIMEOUT);
  }
  return ok;
}

// After a time-out: let every copy this warp started land before the block exits.
template <int D>
__device__ __forceinline__ void stage_drain(uint32_t full0, int issued, int consumed, const ExpertArgs& a) {
  for (int j = consumed; j < issued; ++j)
    if (!mbar_wait_bounded(full0 + 8 * (j % D), (j / D) & 1, a.budget)) atomicOr(a.status, ST_TIMEOUT);
}

// Record pointers of the passes [pi0, pi1) of this block's range -> smem.
__device__ __forceinline__ void load_recs(const uint8_t** recs, const ExpertArgs& a, int p_begin, int pi0, int pi1,
                                          int tid, int nthr) {
  for (int q = tid; q < pi1 - pi0; q += nthr)
    recs[q] = expert_record(a, __ldcg(a.plan.pass_expert + pass_of(a, p_begin, pi0 + q)));
}

// ------------------------------------------------------------------ gate/up
template <int NW, int D>
__global__ void __launch_bounds__(NW * 32, 1) int4_gateup_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ const uint8_t* s_rec[I4_MAX_RECS];
  using SM = I4Smem<NW, D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nthr = NW * 32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::ring);
  uint2* xfrag = reinterpret_cast<uint2*>(smem + SM::ring + SM::bars);
  const uint32_t full0 = smem_u32(bars + warp * D);
  const uint32_t ring0 = smem_u32(smem + warp * D * I4_STAGE);

  const RecGeom rg = rec_geom(WFMT_INT4, a.H, a.F);
  const MatGeom g = rg.m[0];                       // gate and up share the geometry
  const int NG = g.ngroup, nks = cdiv(NG, I4_KS), ntask = g.ntask;
  const int per_rb = 2 * nks;                      // tasks of one (pass, row block)
  const int per_pass = per_rb * ntask;
  const int rows32 = ntask * 32;

  pdl_wait();  // the plan and x come from the kernels before
  const int p_begin = a.range.p_begin;
  const int p_end = a.range.p_end >= 0 ? a.range.p_end : __ldcg(a.range.count ? a.range.count : &a.plan.hdr->n_pass);
  const int total = max(0, p_end - p_begin) * per_pass;
  const int t0 = (int)((long long)total * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  const int pi0 = t0 / per_pass, pi1 = t1 > t0 ? (t1 - 1) / per_pass + 1 : pi0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * D; ++i) mbar_init(smem_u32(bars + i), 1);
    s_abort = 0;
    mbar_fence_init();
  }
  // one token: every pass multiplies the same x, so its fragments are built once, from
  // loads issued before this block's weight stream starts (they would queue behind it)
  const bool one = a.T == 1 && a.H / 16 <= nthr;
  uint4 xu0 = make_uint4(0u, 0u, 0u, 0u), xu1 = xu0;
  if (one && t0 < t1 && (int)threadIdx.x < a.H / 16) {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + threadIdx.x * 16);
    xu0 = __ldg(src);
    xu1 = __ldg(src + 1);
  }
  load_recs(s_rec, a, p_begin, pi0, pi1, threadIdx.x, nthr);
  __syncthreads();
  pdl_launch_dependents();
  if (t0 >= t1) return;

  // this warp's tasks: t0 + warp + NW j, j < nw
  const int first = t0 + warp;
  const int nw = first < t1 ? (t1 - first + NW - 1) / NW : 0;
  int ipi = first / per_pass, irb = (first - ipi * per_pass) / per_rb;   // issue cursor
  int it = first - ipi * per_pass - irb * per_rb;
  int j_issue = 0, islot = 0;
  auto issue_next = [&]() {
    const int m = it >= nks ? 1 : 0, ks = it - m * nks;
    const int ng = min(I4_KS, NG - ks * I4_KS);
    const uint8_t* src = s_rec[ipi - pi0] + (m ? rg.off[1] : rg.off[0]) +
                         ((size_t)irb * NG + (size_t)ks * I4_KS) * I4_PAIR_BLOCK;
    stage_issue(lane, full0 + 8 * islot, ring0 + islot * I4_STAGE, src, (uint32_t)ng * I4_PAIR_BLOCK);
    ++j_issue;
    if (++islot == D) islot = 0;
    it += NW;
    while (it >= per_rb) {
      it -= per_rb;
      if (++irb == ntask) { irb = 0; ++ipi; }
    }
  };
  // one copy per warp now, the rest of the ring after the fragments are built: a full
  // ring's worth of copies queued at once makes each issue wait behind the others
  if (j_issue < min(1, nw)) issue_next();

  const int gq = lane >> 2, p = lane & 3;
  const uint8_t* myring = smem + warp * D * I4_STAGE;
  int j = 0;                                 // tasks consumed by this warp
  int cslot = 0;                             // its ring slot and that slot's phase parity
  uint32_t cphase = 0u;
  int ti = first;
  for (int seg = t0; seg < t1;) {            // segments = one pass each
    const int pi = seg / per_pass;
    const int seg_end = min(t1, (pi + 1) * per_pass);
    const int pass = pass_of(a, p_begin, pi);
    // one token per forward: the pass has that token alone, no plan read needed
    const int ntok = a.T == 1 ? 1 : __ldcg(a.plan.pass_ntok + pass);
    const int nb = 2 * ntok;
    int tok[I4_PMAX];
#pragma unroll
    for (int q = 0; q < I4_PMAX; ++q) tok[q] = (q < ntok && a.T > 1) ? __ldcg(a.plan.pass_tok + pass * I4_PMAX + q) : 0;
    if (!(one && seg > t0)) {
      named_sync(1, nthr);
      if (one) {
        if ((int)threadIdx.x < a.H / 16) bfrag_kstep(xfrag, i4_kstride(a.H / 16), 0, threadIdx.x, xu0, xu1);
      } else {
        build_bfrags_x(xfrag, a.x, a.H, tok, ntok, threadIdx.x, nthr);
      }
      named_sync(1, nthr);
    }
    while (j_issue < min(D, nw)) issue_next();
    float* part = a.part_gu + (size_t)pass * 2 * nks * I4_PMAX * rows32;
    const uint2* xcol = xfrag + i4_lane_col(lane, nb) * i4_kstride(a.H / 16);
    int local = ti - pi * per_pass;          // compute cursor within the pass
    int rb = local / per_rb, t = local - rb * per_rb;
    for (; ti < seg_end; ti += NW) {
      const int m = t >= nks ? 1 : 0, ks = t - m * nks;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const bool ok = stage_wait(full0 + 8 * cslot, cphase, &s_abort, a, lane);
      if (ok) {
        const uint8_t* st = myring + cslot * I4_STAGE;
        const uint2* xl = xcol + ks * I4_SLICE_KSTEPS;
        if (ks * I4_KS + 2 <= NG) i4_task<2>(st + lane * 16, st + 1024 + gq * 4, xl, acc);
        else i4_task<1>(st + lane * 16, st + 1024 + gq * 4, xl, acc);
      }
      __syncwarp();
      ++j;
      if (++cslot == D) {
        cslot = 0;
        cphase ^= 1u;
      }
      if (ok && j_issue < nw) issue_next();   // refill the slot just read
      if (ok && p < ntok) {
        float* dst = part + ((size_t)(m * nks + ks) * I4_PMAX + p) * rows32 + rb * 32;
        dst[gq] = acc[0][0] + acc[0][1];
        dst[gq + 8] = acc[0][2] + acc[0][3];
        dst[gq + 16] = acc[1][0] + acc[1][1];
        dst[gq + 24] = acc[1][2] + acc[1][3];
      }
      t += NW;                               // advance the compute cursor by NW tasks
      while (t >= per_rb) {
        t -= per_rb;
        ++rb;
      }
    }
    seg = seg_end;
  }
  if (s_abort && lane == 0) stage_drain<D>(full0, j_issue, j, a);
}

// ------------------------------------------------------------------ down
template <int NW, int D>
__global__ void __launch_bounds__(NW * 32, 1) int4_down_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ const uint8_t* s_rec[I4_MAX_RECS];
  using SM = I4Smem<NW, D>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::ring);
  // unit slot ui: B fragments at xfrag + ui * DFRAG, inputs at vin + ui * DVIN
  constexpr int DFRAG = SM::dn_frag / 8, DVIN = SM::dn_vin / 4;
  uint2* xfrag = reinterpret_cast<uint2*>(smem + SM::ring + SM::bars);
  float* vin = reinterpret_cast<float*>(smem + SM::ring + SM::bars + DN_UMAX * SM::dn_frag);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars + warp * D);
  const uint32_t ring0 = smem_u32(smem + warp * D * I4_STAGE);
  constexpr int nthr = NW * 32;

  const RecGeom rg = rec_geom(WFMT_INT4, a.H, a.F);
  const MatGeom g = rg.m[2];
  const int NG = g.ngroup, nks = cdiv(NG, I4_KS), ntask = g.ntask;
  const int rows32 = ntask * 32;
  const int nks_gu = cdiv(rg.m[0].ngroup, I4_KS), rows32_f = rg.m[0].ntask * 32;
  const int per_pass = nks * ntask;

  // The plan is older than the gate/up kernel, which waited for it before it let this
  // kernel start, so the weights stream before the gate/up partials are ready.
  const int p_begin = a.range.p_begin;
  const int p_end = a.range.p_end >= 0 ? a.range.p_end : __ldcg(a.range.count ? a.range.count : &a.plan.hdr->n_pass);
  const int total = max(0, p_end - p_begin) * per_pass;
  const int t0 = (int)((long long)total * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  const int pi0 = t0 / per_pass, pi1 = t1 > t0 ? (t1 - 1) / per_pass + 1 : pi0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * D; ++i) mbar_init(smem_u32(bars + i), 1);
    s_abort = 0;
    mbar_fence_init();
  }
  load_recs(s_rec, a, p_begin, pi0, pi1, threadIdx.x, nthr);
  __syncthreads();
  if (t0 >= t1) {
    pdl_wait();
    pdl_launch_dependents();
    return;
  }

  const int first = t0 + warp;
  const int nw = first < t1 ? (t1 - first + NW - 1) / NW : 0;
  // issue cursor: pass ipi, k-slice iks, row block irb (no divisions per task)
  int ipi = first / per_pass, iks = (first - ipi * per_pass) / ntask;
  int irb = first - ipi * per_pass - iks * ntask;
  int j_issue = 0, islot = 0;
  auto issue_next = [&]() {
    const int ng = min(I4_KS, NG - iks * I4_KS);
    const uint8_t* src = s_rec[ipi - pi0] + rg.off[2] + ((size_t)irb * NG + (size_t)iks * I4_KS) * I4_PAIR_BLOCK;
    stage_issue(lane, full0 + 8 * islot, ring0 + islot * I4_STAGE, src, (uint32_t)ng * I4_PAIR_BLOCK);
    ++j_issue;
    if (++islot == D) islot = 0;
    irb += NW;
    while (irb >= ntask) {
      irb -= ntask;
      if (++iks == nks) {
        iks = 0;
        ++ipi;
      }
    }
  };
  // one task per warp streams before the wait; the rest of the ring fills after this
  // block's gate/up partials have been read (those reads would queue behind a full ring)
  if (j_issue < min(1, nw)) issue_next();

  pdl_wait();  // the gate/up partials come from the kernel before
  pdl_launch_dependents();
  const int gq = lane >> 2, p = lane & 3;
  const uint8_t* myring = smem + warp * D * I4_STAGE;
  int j = 0;
  int cslot = 0;
  uint32_t cphase = 0u;
  int ti = first;
  // h of a unit's slice: silu(g) * u, the gate / up partials added in k-slice order
  auto unit_h = [&](int pass, int ts, int kbase, int kk, int kvalid) {
    float v = 0.f;
    if (kk < kvalid) {
      const size_t stride = (size_t)I4_PMAX * rows32_f;
      const float* pg = a.part_gu + ((size_t)pass * 2 * nks_gu * I4_PMAX + ts) * rows32_f + kbase + kk;
      const float* pu = pg + (size_t)nks_gu * stride;
      float gs = 0.f, us = 0.f;
      for (int s0 = 0; s0 < nks_gu; s0 += 16) {   // 32 loads in flight, added in slice order
        float gv[16], uv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const bool in = s0 + q < nks_gu;
          gv[q] = in ? __ldcg(pg + (size_t)(s0 + q) * stride) : 0.f;
          uv[q] = in ? __ldcg(pu + (size_t)(s0 + q) * stride) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (s0 + q < nks_gu) {
            gs += gv[q];
            us += uv[q];
          }
        }
      }
      v = gs / (1.f + expf(-gs)) * us;
    }
    return v;
  };
  struct DnUnit {
    int pass, ks, ntok, ng;
  };
  auto unit_at = [&](int u) {
    DnUnit U;
    const int pi = u / nks;
    U.ks = u - pi * nks;
    U.pass = pass_of(a, p_begin, pi);
    U.ntok = a.T == 1 ? 1 : __ldcg(a.plan.pass_ntok + U.pass);
    U.ng = min(I4_KS, NG - U.ks * I4_KS);
    return U;
  };
  // A block's range covers one or two units: both are prepared up front, their inputs
  // read in one round trip, so the warps then run through their tasks without a barrier.
  // A block with more units prepares each when it reaches it.
  const int u_first = t0 / ntask, n_units = (t1 - 1) / ntask - u_first + 1;
  const bool pre = n_units <= DN_UMAX;
  if (pre) {
    DnUnit U0 = unit_at(u_first), U1 = U0;
    if (n_units > 1) U1 = unit_at(u_first + 1);
    const int e0 = U0.ntok * I4_KS * I4_GROUP, e1 = n_units > 1 ? U1.ntok * I4_KS * I4_GROUP : 0;
    for (int q = threadIdx.x; q < e0 + e1; q += nthr) {
      const bool second = q >= e0;
      const DnUnit& U = second ? U1 : U0;
      const int e = second ? q - e0 : q;
      const int ts = e / (I4_KS * I4_GROUP), kk = e - ts * (I4_KS * I4_GROUP);
      vin[(second ? DVIN : 0) + e] = unit_h(U.pass, ts, U.ks * I4_KS * I4_GROUP, kk, U.ng * I4_GROUP);
    }
    named_sync(1, nthr);
    build_bfrags(xfrag, I4_SLICE_KSTEPS, 2 * U0.ntok, threadIdx.x, nthr,
                 [&](int ts, int k) { return vin[ts * (I4_KS * I4_GROUP) + k]; });
    if (n_units > 1)
      build_bfrags(xfrag + DFRAG, I4_SLICE_KSTEPS, 2 * U1.ntok, threadIdx.x, nthr,
                   [&](int ts, int k) { return vin[DVIN + ts * (I4_KS * I4_GROUP) + k]; });
    named_sync(1, nthr);
    while (j_issue < min(D, nw)) issue_next();
  }
  for (int seg = t0; seg < t1;) {  // segments = one unit (pass, k-slice) each
    const int u = seg / ntask;
    const int seg_end = min(t1, (u + 1) * ntask);
    const DnUnit U = unit_at(u);
    const int nb = 2 * U.ntok;
    int slot_u = 0;
    if (pre) {
      slot_u = u - u_first;
    } else {
      named_sync(1, nthr);
      for (int e = threadIdx.x; e < U.ntok * I4_KS * I4_GROUP; e += nthr) {
        const int ts = e / (I4_KS * I4_GROUP), kk = e - ts * (I4_KS * I4_GROUP);
        vin[e] = unit_h(U.pass, ts, U.ks * I4_KS * I4_GROUP, kk, U.ng * I4_GROUP);
      }
      named_sync(1, nthr);
      build_bfrags(xfrag, I4_SLICE_KSTEPS, nb, threadIdx.x, nthr,
                   [&](int ts, int k) { return vin[ts * (I4_KS * I4_GROUP) + k]; });
      named_sync(1, nthr);
      while (j_issue < min(D, nw)) issue_next();
    }
    float* dst0 = a.part_d + ((size_t)U.pass * nks + U.ks) * I4_PMAX * rows32;
    const uint2* xcol = xfrag + slot_u * DFRAG + i4_lane_col(lane, nb) * i4_kstride(I4_SLICE_KSTEPS);
    for (; ti < seg_end; ti += NW) {
      const int rb = ti - u * ntask;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const bool ok = stage_wait(full0 + 8 * cslot, cphase, &s_abort, a, lane);
      if (ok) {
        const uint8_t* st = myring + cslot * I4_STAGE;
        if (U.ng == 2) i4_task<2>(st + lane * 16, st + 1024 + gq * 4, xcol, acc);
        else i4_task<1>(st + lane * 16, st + 1024 + gq * 4, xcol, acc);
      }
      __syncwarp();
      ++j;
      if (++cslot == D) {
        cslot = 0;
        cphase ^= 1u;
      }
      if (ok && j_issue < nw) issue_next();
      if (ok && p < U.ntok) {
        float* dst = dst0 + (size_t)p * rows32 + rb * 32;
        dst[gq] = acc[0][0] + acc[0][1];
        dst[gq + 8] = acc[0][2] + acc[0][3];
        dst[gq + 16] = acc[1][0] + acc[1][1];
        dst[gq + 24] = acc[1][2] + acc[1][3];
      }
    }
    seg = seg_end;
  }
  if (s_abort && lane == 0) stage_drain<D>(full0, j_issue, j, a);
}

// ------------------------------------------------------------------ launch configuration
// 16 warps; ring depth 3 when the B fragments of the widest pass (nb columns, all of K)
// leave room for it, else 2; wide inputs with 4-token passes drop to 8 warps.
struct I4Launch {
  int nw, d;
  size_t smem_gu, smem_down;
};

// every configuration's down kernel fits whatever the shapes (its shared memory does not
// depend on them)
static_assert(I4Smem<24, 2>::down() <= 227 * 1024 - I4_STATIC_SMEM, "down smem");
static_assert(I4Smem<16, 3>::down() <= 227 * 1024 - I4_STATIC_SMEM, "down smem");

static I4Launch i4_config(int H, int max_tokens) {
  const int nb = 2 * std::min(max_tokens, I4_PMAX);
  const size_t cap = 227 * 1024 - I4_STATIC_SMEM;
  if ((size_t)I4Smem<24, 2>::gateup(H, nb) <= cap)
    return {24, 2, (size_t)I4Smem<24, 2>::gateup(H, nb), (size_t)I4Smem<24, 2>::down()};
  if ((size_t)I4Smem<16, 3>::gateup(H, nb) <= cap)
    return {16, 3, (size_t)I4Smem<16, 3>::gateup(H, nb), (size_t)I4Smem<16, 3>::down()};
  if ((size_t)I4Smem<16, 2>::gateup(H, nb) <= cap)
    return {16, 2, (size_t)I4Smem<16, 2>::gateup(H, nb), (size_t)I4Smem<16, 2>::down()};
  return {8, 2, (size_t)I4Smem<8, 2>::gateup(H, nb), (size_t)I4Smem<8, 2>::down()};
}

template <int NW, int D>
static cudaError_t i4_attrs(const I4Launch& c) {
  cudaError_t e = cudaFuncSetAttribute(int4_gateup_kernel<NW, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)c.smem_gu);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(int4_down_kernel<NW, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem_down);
  return e;
}

cudaError_t int4_set_attributes(int H, int max_tokens) {
  const I4Launch c = i4_config(H, max_tokens);
  if (c.nw == 24) return i4_attrs<24, 2>(c);
  if (c.nw == 16 && c.d == 3) return i4_attrs<16, 3>(c);
  if (c.nw == 16) return i4_attrs<16, 2>(c);
  return i4_attrs<8, 2>(c);
}

cudaError_t launch_int4_gateup(const ExpertArgs& a, int grid, cudaStream_t s) {
  const I4Launch c = i4_config(a.H, a.max_tokens);
  if (c.nw == 24) return launch_pdl(int4_gateup_kernel<24, 2>, grid, 24 * 32, c.smem_gu, s, a);
  if (c.nw == 16 && c.d == 3) return launch_pdl(int4_gateup_kernel<16, 3>, grid, 16 * 32, c.smem_gu, s, a);
  if (c.nw == 16) return launch_pdl(int4_gateup_kernel<16, 2>, grid, 16 * 32, c.smem_gu, s, a);
  return launch_pdl(int4_gateup_kernel<8, 2>, grid, 8 * 32, c.smem_gu, s, a);
}

cudaError_t launch_int4_down(const ExpertArgs& a, int grid, cudaStream_t s) {
  const I4Launch c = i4_config(a.H, a.max_tokens);
  if (c.nw == 24) return launch_pdl(int4_down_kernel<24, 2>, grid, 24 * 32, c.smem_down, s, a);
  if (c.nw == 16 && c.d == 3) return launch_pdl(int4_down_kernel<16, 3>, grid, 16 * 32, c.smem_down, s, a);
  if (c.nw == 16) return launch_pdl(int4_down_kernel<16, 2>, grid, 16 * 32, c.smem_down, s, a);
  return launch_pdl(int4_down_kernel<8, 2>, grid, 8 * 32, c.smem_down, s, a);
}

}  // namespace moe
