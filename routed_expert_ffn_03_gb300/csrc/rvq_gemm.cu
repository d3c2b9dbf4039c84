// rvq_gemm.cu - tcgen05 grouped GEMM for RVQ experts that serve many tokens at once.
//
// When one expert is selected by >= GEMM_MIN tokens of a forward (the always-on shared
// expert at T = 32, a draft-verify batch, prefill-like T), its weights are worth
// streaming once and multiplying against all of those tokens as a dense contraction:
//     Y[r][n] = sum_k W[r][k] X[k][n],   W = W0 + W1 + W2,  W_s[r][8q+i] = C_s[c_s(r,q)][i]
// Each stage W_s is a gather of stored fp16 codebook rows, so it is exact in fp16; the
// activations enter as fp16 hi + lo columns (n = 2 token + part), so all products are
// exact and the three stages and all k accumulate in fp32 in tensor memory.
//
// Work item = (group of <= 32 tokens of one expert, 512-input k-slice, matrix, 128-row
// tile), in that order; a block (8 warps) takes an equal contiguous range of items, so
// its consecutive items share the group and k-slice and the B operand (X hi/lo, K-major
// canonical layout, no swizzle, built from 16-byte loads) is built once for them.  Per
// item: the tile's codes (4 row blocks x 6 KB) arrive by a bulk TMA copy issued while the
// item before was computing (two code buffers), the matrix's codebooks (12 KB) by a copy
// only when the matrix changes; then for each of
// the 8 k-blocks of 64 inputs the block gathers the three A stage tiles (128 x 64 fp16
// each, K-major canonical layout; a thread reads its row's 12 code bytes of 4 groups as 3
// words) into one of two buffers and one thread issues
// 3 x 4 tcgen05.mma (M = 128, N = 16..64, K = 16) into the TMEM accumulator, committing
// to that buffer's mbarrier so the gather of the next k-block overlaps them.  The
// epilogue reads TMEM with tcgen05.ld (warps 0-3, one TMEM lane quarter each) and writes
// the k-slice partial of every token in the same layout the lookup-table path uses
// (part_gu[pass][m][ks][row], part_d[pass][ks][row]), so the SwiGLU and combine steps
// are shared.  Every wait is bounded; the tensor memory is always released.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int GM_TILE_M = 128;
constexpr int GM_KB = 64;                                   // inputs per k-block
constexpr int GM_NKB = RVQ_KS * RVQ_GROUP / GM_KB;          // 8 k-blocks per 512-input slice
constexpr int GM_MAXN = 64;                                 // 32 tokens x hi/lo
constexpr int GM_CB = RVQ_CB_BYTES;                         // 12288
constexpr int GM_CODES = 4 * RVQ_TASK_BYTES;                // 24576 (4 row blocks of 32)
constexpr int GM_B = GM_MAXN * RVQ_KS * RVQ_GROUP * 2;      // 65536: N x 512 fp16
constexpr int GM_ASTAGE = GM_TILE_M * GM_KB * 2;            // 16384: 128 x 64 fp16
constexpr int GM_A = 2 * 3 * GM_ASTAGE;                     // two buffers x three stages
constexpr int GM_OFF_CODES = GM_CB;                         // two buffers: item i's codes, item i + 1's
constexpr int GM_OFF_B = GM_OFF_CODES + 2 * GM_CODES;
constexpr int GM_OFF_A = GM_OFF_B + GM_B;
constexpr int GM_OFF_BAR = GM_OFF_A + GM_A;                 // 5 mbarriers + tmem address
constexpr int GM_SMEM = GM_OFF_BAR + 64;
constexpr int GM_THREADS = 256;
constexpr int GM_TMEM_COLS = 64;

// ---------------------------------------------------------------- tcgen05 helpers
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // K-major, no swizzle: start >> 4 [0,14), leading (K-direction core matrix) byte offset
  // >> 4 [16,30), stride (M/N-direction 8-row group) byte offset >> 4 [32,46), descriptor
  // version 1 [46,48), layout type 0 (no swizzle) [61,64).
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// kind::f16 instruction descriptor: D fp32, A and B fp16, both K-major, M, N.
__host__ __device__ __forceinline__ uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (0u << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of element (row, k) in a K-major, no-swizzle canonical tile whose rows are
// kcores * 8 elements long: core matrix (row / 8, k / 8) of 8 x 8 fp16 (128 B), rows of a
// core 16 B apart, cores along K 128 B apart, 8-row groups kcores * 128 B apart.
__device__ __forceinline__ uint32_t canon_off(int row, int k, int kcores) {
  return (uint32_t)(((row >> 3) * kcores + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

struct GmItem {
  int grp, m, ks, tile;
};

template <bool DOWN>
__global__ void __launch_bounds__(GM_THREADS, 1) rvq_gemm_kernel(ExpertArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const RecGeom rg = rec_geom(WFMT_RVQ, a.H, a.F);
  const MatGeom g = rg.m[DOWN ? 2 : 0];
  const MatGeom gg = rg.m[0];
  constexpr int mats = DOWN ? 1 : 2;
  const int nks = g.nks, ntile = cdiv(g.rows, GM_TILE_M);
  const int rows32 = g.ntask * 32, rows32_gu = gg.ntask * 32;

  uint8_t* cb = smem;
  uint8_t* bsm = smem + GM_OFF_B;
  uint8_t* asm_ = smem + GM_OFF_A;
  // [0] codebooks, [1..2] mma buffers, [3..4] code buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GM_OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + GM_OFF_BAR + 48);
  __shared__ volatile int s_abort;
  const uint32_t bar_cb = smem_u32(bars), bar_mma0 = smem_u32(bars + 1), bar_code0 = smem_u32(bars + 3);

  const int n_big = __ldcg(&a.plan.hdr->n_big);
  const int total = n_big * mats * nks * ntile;
  const int it0 = (int)((long long)total * blockIdx.x / gridDim.x);
  const int it1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  if (it0 >= it1) return;  // no item for this block (uniform): no tensor memory taken

  if (tid == 0) {
    mbar_init(bar_cb, 1);
    mbar_init(bar_mma0, 1);
    mbar_init(bar_mma0 + 8, 1);
    mbar_init(bar_code0, 1);
    mbar_init(bar_code0 + 8, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(GM_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int cb_phase = 0, mma_phase[2] = {0, 0}, mma_pending[2] = {0, 0};
  int code_phase[2] = {0, 0}, code_pending[2] = {0, 0};   // thread 0's view of the code copies
  bool cb_pending = false;
  __shared__ int s_tok[GEMM_MAX_TOKENS];
  int b_grp = -1, b_ks = -1;    // the group and k-slice the B operand holds
  int cb_grp = -1, cb_m = -1;   // the matrix whose codebooks are in shared memory
  auto decode = [&](int it) {
    GmItem I;
    I.tile = it % ntile;
    int rest = it / ntile;
    I.m = rest % mats;
    rest /= mats;
    I.ks = rest % nks;
    I.grp = rest / nks;
    return I;
  };
  auto matrix_of = [&](const GmItem& I) {
    const int expert = __ldcg(a.plan.big + 3 * I.grp + 0);
    return expert_record(a, expert) + (DOWN ? rg.off[2] : (I.m == 0 ? rg.off[0] : rg.off[1]));
  };
  // thread 0: the codes of item `it` (4 row blocks of its tile, one k-slice) into buffer b
  auto issue_codes = [&](int it, int b) {
    const GmItem I = decode(it);
    const int rb0 = I.tile * 4, nrb = min(4, g.ntask - rb0);
    const uint8_t* mat = matrix_of(I);
    fence_async_smem();  // an earlier item read this buffer through the generic proxy
    mbar_arrive_expect_tx(bar_code0 + 8 * b, nrb * RVQ_TASK_BYTES);
    bulk_g2s(smem_u32(smem + GM_OFF_CODES + b * GM_CODES), mat + GM_CB + ((size_t)I.ks * g.ntask + rb0) * RVQ_TASK_BYTES,
             nrb * RVQ_TASK_BYTES, bar_code0 + 8 * b);
    code_pending[b] = 1;
  };
  if (tid == 0) issue_codes(it0, 0);
  for (int it = it0; it < it1 && !s_abort; ++it) {
    const int cur = (it - it0) & 1;
    const GmItem I = decode(it);
    const int pass0 = __ldcg(a.plan.big + 3 * I.grp + 1);
    const int ntok = __ldcg(a.plan.big + 3 * I.grp + 2);
    const int N = max(16, (2 * ntok + 15) & ~15);
    const uint8_t* mat = matrix_of(I);
    const int rb0 = I.tile * 4, nrb = min(4, g.ntask - rb0);
    const uint8_t* codes = smem + GM_OFF_CODES + cur * GM_CODES;

    if (tid == 0) {
      // the next item's codes go in flight now (its buffer was last read by the item before)
      if (it + 1 < it1) issue_codes(it + 1, cur ^ 1);
      // codebooks only when the matrix changes (the previous item's gathers are done)
      if (I.grp != cb_grp || I.m != cb_m) {
        fence_async_smem();
        mbar_arrive_expect_tx(bar_cb, GM_CB);
        bulk_g2s(smem_u32(cb), mat, GM_CB, bar_cb);
        cb_pending = true;
      }
    }
    const bool new_cb = I.grp != cb_grp || I.m != cb_m;
    cb_grp = I.grp;
    cb_m = I.m;
    // B operand: column n = 2 t + part of token t of the group, K-major canonical layout;
    // one thread step = 8 consecutive inputs of one token (hi and lo columns)
    if (I.grp != b_grp || I.ks != b_ks) {
      if (!DOWN && tid < ntok) s_tok[tid] = __ldcg(a.plan.pass_tok + pass0 + tid);
      __syncthreads();
      const int kbase = I.ks * RVQ_KS * RVQ_GROUP;
      constexpr int C8 = RVQ_KS * RVQ_GROUP / 8;   // 64 chunks of 8 inputs per slice
      for (int e = tid; e < (N / 2) * C8; e += GM_THREADS) {
        const int t = e / C8, c8 = e - t * C8;
        const int k = c8 * 8, kk0 = kbase + k;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        if (t < ntok) {
          if (!DOWN) {
            const uint16_t* xr = a.x + (size_t)s_tok[t] * a.H + kk0;
            if (kk0 + 8 <= g.K) {
              const uint4 u = __ldg(reinterpret_cast<const uint4*>(xr));
              const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w4[i] << 16);
                v[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
              }
            } else {
              for (int i = 0; i < 8; ++i)
                if (kk0 + i < g.K) v[i] = bf16_bits_to_float(xr[i]);
            }
          } else {
            const float* hp = a.h + (size_t)(pass0 + t) * rows32_gu + kk0;   // SwiGLU (rvq_swiglu_big)
            if (kk0 + 8 <= g.K) {
              const float4 f0 = __ldcg(reinterpret_cast<const float4*>(hp));
              const float4 f1 = __ldcg(reinterpret_cast<const float4*>(hp) + 1);
              v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
              v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
            } else {
              for (int i = 0; i < 8; ++i)
                if (kk0 + i < g.K) v[i] = __ldcg(hp + i);
            }
          }
        }
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __half h0, l0, h1, l1;
          split_half(v[2 * i], h0, l0);
          split_half(v[2 * i + 1], h1, l1);
          hw[i] = pack_half2(h0, h1);
          lw[i] = pack_half2(l0, l1);
        }
        *reinterpret_cast<uint4*>(bsm + canon_off(2 * t, k, C8)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(bsm + canon_off(2 * t + 1, k, C8)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      b_grp = I.grp;
      b_ks = I.ks;
    }
    // the tile's codes (and new codebooks) must have landed before the gather
    bool ok = mbar_wait_bounded(bar_code0 + 8 * cur, code_phase[cur] & 1, a.budget);
    code_phase[cur] ^= 1;
    if (tid == 0 && ok) code_pending[cur] = 0;
    if (ok && new_cb) {
      ok = mbar_wait_bounded(bar_cb, cb_phase & 1, a.budget);
      cb_phase ^= 1;
      if (tid == 0 && ok) cb_pending = false;
    }
    if (!ok) {
      s_abort = 1;
      atomicOr(a.status, ST_TIMEOUT);
    }
    __syncthreads();
    if (s_abort) break;

    const uint32_t idesc = umma_idesc_f16(GM_TILE_M, N);
    for (int kb = 0; kb < GM_NKB; ++kb) {
      const int buf = kb & 1;
      uint8_t* abuf = asm_ + buf * 3 * GM_ASTAGE;
      if (mma_pending[buf]) {  // the mma that read this buffer two k-blocks ago is done
        ok = mbar_wait_bounded(bar_mma0 + 8 * buf, mma_phase[buf] & 1, a.budget);
        mma_phase[buf] ^= 1;
        mma_pending[buf] = 0;
        if (!ok) {
          s_abort = 1;
          atomicOr(a.status, ST_TIMEOUT);
        }
        tc_fence_after();
      }
      // gather: thread = (tile row r, 4 groups of the k-block); the 4 groups' 12 code bytes
      // are 12 contiguous bytes of the row's lane stream (positions P .. P + 3, P = (l ^ q) & ~3
      // for its first group q), read as 3 words; each (position, stage) gives one 16-byte
      // codebook row, stored into the stage tile at the row's group q = l ^ position
      {
        const int r = tid & (GM_TILE_M - 1), hh = tid >> 7;   // GM_THREADS == 2 * GM_TILE_M
        const int rbl = r >> 5, l = r & 31;
        const int q0 = kb * 8 + 4 * hh;                        // first group (within the slice)
        const int P = (l ^ q0) & ~3;                           // first position of the 4
        uint32_t w[3] = {0u, 0u, 0u};
        if (rbl < nrb) {
          const uint8_t* lb = codes + rbl * RVQ_TASK_BYTES + l * 16;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int bp = 3 * P + 4 * j;                      // stream byte, 4-aligned
            w[j] = *reinterpret_cast<const uint32_t*>(lb + (bp >> 4) * 512 + (bp & 15));
          }
        }
#pragma unroll
        for (int d = 0; d < 4; ++d) {
          const int gi = ((P + d) ^ l) - kb * 8;               // group within the k-block
#pragma unroll
          for (int s = 0; s < 3; ++s) {
            const int b = 3 * d + s;                           // byte of the 12
            const uint32_t code = (w[b >> 2] >> (8 * (b & 3))) & 0xffu;
            const uint4 v = *reinterpret_cast<const uint4*>(cb + ((s * 256 + code) * 8) * 2);
            *reinterpret_cast<uint4*>(abuf + s * GM_ASTAGE + canon_off(r, gi * 8, GM_KB / 8)) = v;
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (s_abort) break;
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 3; ++s) {
#pragma unroll
          for (int kk = 0; kk < GM_KB / 16; ++kk) {
            const uint64_t ad = umma_smem_desc(smem_u32(abuf + s * GM_ASTAGE) + kk * 2 * 128, 128, (GM_KB / 8) * 128);
            const uint64_t bd = umma_smem_desc(smem_u32(bsm) + (kb * (GM_KB / 8) + kk * 2) * 128, 128,
                                               (RVQ_KS * RVQ_GROUP / 8) * 128);
            tc_mma(tmem, ad, bd, idesc, kb > 0 || s > 0 || kk > 0);
          }
        }
        tc_commit(bar_mma0 + 8 * buf);
      }
      mma_pending[buf] = 1;
    }
    if (s_abort) break;
    // all mma of this item done (the last commit covers every earlier one)
    const int lastbuf = (GM_NKB - 1) & 1;
    ok = mbar_wait_bounded(bar_mma0 + 8 * lastbuf, mma_phase[lastbuf] & 1, a.budget);
    mma_phase[lastbuf] ^= 1;
    mma_pending[lastbuf] = 0;
    if (mma_pending[lastbuf ^ 1]) {  // its phase also completed (earlier commit)
      ok = ok && mbar_wait_bounded(bar_mma0 + 8 * (lastbuf ^ 1), mma_phase[lastbuf ^ 1] & 1, a.budget);
      mma_phase[lastbuf ^ 1] ^= 1;
      mma_pending[lastbuf ^ 1] = 0;
    }
    if (!ok) {
      s_abort = 1;
      atomicOr(a.status, ST_TIMEOUT);
    }
    __syncthreads();  // the abort flag is the same for every thread from here
    tc_fence_after();
    if (warp < 4 && !s_abort) {
      const int r = warp * 32 + lane;                 // TMEM lane = tile row
      const int row = I.tile * GM_TILE_M + r;
      const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tc_ld16(taddr + c0, v);
        if (row < g.rows) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int t = (c0 >> 1) + q;
            if (t < ntok) {
              const int pass = pass0 + t;
              float* dst = DOWN ? a.part_d + ((size_t)pass * nks + I.ks) * rows32
                                : a.part_gu + ((size_t)(pass * 2 + I.m) * nks + I.ks) * rows32;
              dst[row] = v[2 * q] + v[2 * q + 1];
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM read and smem reused by the next item
  }
  // release: every issued mma has completed (bounded), then the tensor memory
  if (tid == 0) {
    for (int b = 0; b < 2; ++b)
      if (mma_pending[b] && !mbar_wait_bounded(bar_mma0 + 8 * b, mma_phase[b] & 1, a.budget))
        atomicOr(a.status, ST_TIMEOUT);
    // bulk copies this block started and nobody waited for (a time-out, or the last prefetch)
    for (int b = 0; b < 2; ++b)
      if (code_pending[b] && !mbar_wait_bounded(bar_code0 + 8 * b, code_phase[b] & 1, a.budget))
        atomicOr(a.status, ST_TIMEOUT);
    if (cb_pending && !mbar_wait_bounded(bar_cb, cb_phase & 1, a.budget)) atomicOr(a.status, ST_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(GM_TMEM_COLS) : "memory");
}

// h[pass][row] = silu(g) * u for the passes of the GEMM groups, g and u the gate / up
// k-slice partials added in slice order (the same order the lookup-table down kernel uses).
// One thread per (token of the group, row), its partial loads all in flight.
__global__ void __launch_bounds__(256) rvq_swiglu_big_kernel(ExpertArgs a) {
  const RecGeom rg = rec_geom(WFMT_RVQ, a.H, a.F);
  const MatGeom gg = rg.m[0];
  const int rows32 = gg.ntask * 32;
  const int grp = blockIdx.y;
  if (grp >= __ldcg(&a.plan.hdr->n_big)) return;
  const int pass0 = __ldcg(a.plan.big + 3 * grp + 1), ntok = __ldcg(a.plan.big + 3 * grp + 2);
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= ntok * a.F) return;
  const int t = i / a.F, r = i - t * a.F;
  const int pass = pass0 + t;
  const float* pg = a.part_gu + ((size_t)(pass * 2 + 0) * gg.nks) * rows32 + r;
  const float* pu = a.part_gu + ((size_t)(pass * 2 + 1) * gg.nks) * rows32 + r;
  float gs = 0.f, us = 0.f;
  for (int s0 = 0; s0 < gg.nks; s0 += 16) {
    float gv[16], uv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const bool in = s0 + q < gg.nks;
      gv[q] = in ? __ldcg(pg + (size_t)(s0 + q) * rows32) : 0.f;
      uv[q] = in ? __ldcg(pu + (size_t)(s0 + q) * rows32) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (s0 + q < gg.nks) {
        gs += gv[q];
        us += uv[q];
      }
    }
  }
  a.h[(size_t)pass * rows32 + r] = gs / (1.f + expf(-gs)) * us;
}

cudaError_t rvq_gemm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(rvq_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, GM_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rvq_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, GM_SMEM);
}

cudaError_t launch_rvq_gemm_gateup(const ExpertArgs& a, int grid, cudaStream_t s) {
  rvq_gemm_kernel<false><<<grid, GM_THREADS, GM_SMEM, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_rvq_gemm_down(const ExpertArgs& a, int grid, cudaStream_t s, int max_big) {
  dim3 sg(cdiv(GEMM_MAX_TOKENS * a.F, 256), max_big);
  rvq_swiglu_big_kernel<<<sg, 256, 0, s>>>(a);
  rvq_gemm_kernel<true><<<grid, GM_THREADS, GM_SMEM, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
