// int4.cu - int4 (symmetric, group 128, fp16 scales) expert GEMV kernels.
//
// gate/up:  part_gu[pass][m][ks][row][slot] = sum over k in slice ks of W_m[row][k] x[k]
// down:     part_d [pass][ks][row][slot]    = sum over k in slice ks of W_d[row][k] h[k],
//           h = silu(g) * u with g, u the slice sums of part_gu added in slice order.
// A "pass" is one expert with up to 4 tokens; every pass of every selected expert is
// spread over all SMs as equal contiguous ranges of 32-row x 512-input tasks.
//
// Data movement: one producer warp per block streams each task (32 rows x 4 groups =
// 8448 B, contiguous in the kernel layout) with a 1-D bulk TMA copy into a per-warp
// ring of shared-memory stages; consumer warps read their stage with conflict-free
// 16-byte loads.  Arithmetic: a lane dequantises its own m16n8k16 A fragment from 8
// nibbles (q + 1032 is built as an fp16 bit pattern and the offset removed exactly),
// and the warp-level tensor-core mma multiplies it by the activations, split into fp16
// hi + lo parts so that hi + lo reproduces fp32 inputs to 2^-22; products of q and an
// fp16 part are exact and accumulate in fp32.  The fp16 group scale multiplies each
// 128-wide group's fp32 sum.  The 8 mma columns carry (token, hi/lo) pairs, so one
// pass serves up to 4 tokens at the cost of one.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int I4_NW = 8;                                // consumer warps
constexpr int I4_D = 2;                                 // ring stages per consumer warp
constexpr int I4_STAGE = I4_KS * I4_PAIR_BLOCK;         // 8448 B
constexpr int I4_KSTEPS = I4_KS * I4_GROUP / 16;        // 32 mma k-steps per slice
constexpr int I4_XFRAG = I4_KSTEPS * 32 * 8;            // 8192 B of B fragments
constexpr int I4_VIN = I4_PMAX * I4_KS * I4_GROUP * 4;  // 8192 B of slice inputs
constexpr int I4_BAR_OFF = I4_NW * I4_D * I4_STAGE + I4_XFRAG + I4_VIN;
constexpr int I4_SMEM = I4_BAR_OFF + 2 * I4_NW * I4_D * 8;

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;  // (a & b) ^ c
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 8 nibbles -> the four half2 registers of an m16n8k16 A fragment (exact integers q).
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                         uint32_t& a3) {
  const uint32_t LO = 0x000F000Fu, HI = 0x00F000F0u;
  const uint32_t XLO = 0x64086408u, XHI = 0x64806480u;  // fp16 1024 exponent, nibble ^ 8
  const __half2 off_lo = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 sixteenth = __halves2half2(__float2half_rn(0.0625f), __float2half_rn(0.0625f));
  const __half2 off_hi = __halves2half2(__float2half_rn(-72.f), __float2half_rn(-72.f));
  const uint32_t w2 = w >> 8;
  uint32_t t0 = lop3_and_xor(w, LO, XLO);    // 1032 + q  (rows g,   k 2p / 2p+1)
  uint32_t t1 = lop3_and_xor(w, HI, XHI);    // 1152 + 16 q (rows g+8)
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

struct I4Unit {
  int pass, m, ks, ntok, ng;
  const uint8_t* base;  // first byte of the unit's matrix
};

template <bool DOWN>
__device__ __forceinline__ I4Unit i4_unit(const ExpertArgs& a, long long u, int nks, int p_begin,
                                          const RecGeom& rg, const MatGeom& g) {
  constexpr int mats = DOWN ? 1 : 2;
  I4Unit U;
  U.ks = (int)(u % nks);
  const long long pm = u / nks;
  U.m = (int)(pm % mats);
  const int pi = (int)(pm / mats);
  U.pass = a.range.order ? a.range.order[p_begin + pi] : p_begin + pi;
  const int e = a.plan.pass_expert[U.pass];
  U.ntok = a.plan.pass_ntok[U.pass];
  U.ng = min(I4_KS, g.ngroup - U.ks * I4_KS);
  U.base = a.rec_table[e] + (DOWN ? rg.off[2] : (U.m == 0 ? rg.off[0] : rg.off[1]));
  return U;
}

template <bool DOWN>
__global__ void __launch_bounds__((I4_NW + 1) * 32, 1) int4_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  uint2* xfrag = reinterpret_cast<uint2*>(smem + I4_NW * I4_D * I4_STAGE);
  float* vin = reinterpret_cast<float*>(smem + I4_NW * I4_D * I4_STAGE + I4_XFRAG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + I4_BAR_OFF);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + I4_NW * I4_D);
  const uint32_t stage0 = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int mats = DOWN ? 1 : 2;
  const RecGeom rg = rec_geom(WFMT_INT4, a.H, a.F);
  const MatGeom g = rg.m[DOWN ? 2 : 0];
  const int nks = g.nks, ntask = g.ntask;
  const int p_begin = a.range.p_begin;
  const int p_end = a.range.p_end < 0 ? a.plan.hdr->n_pass : a.range.p_end;
  const long long total = (long long)max(0, p_end - p_begin) * mats * nks * ntask;
  const long long t0 = total * blockIdx.x / gridDim.x;
  const long long t1 = total * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * I4_NW * I4_D; ++i) mbar_init(full0 + 8 * i, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (t0 >= t1) return;

  if (warp == I4_NW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int seq[I4_NW], iss[I4_NW];
#pragma unroll
    for (int w = 0; w < I4_NW; ++w) seq[w] = iss[w] = 0;
    for (long long i = t0; i < t1;) {
      const long long u = i / ntask;
      const long long seg_end = min(t1, (u + 1) * ntask);
      const I4Unit U = i4_unit<DOWN>(a, u, nks, p_begin, rg, g);
      const uint32_t bytes = (uint32_t)U.ng * I4_PAIR_BLOCK;
      for (long long r = i; r < seg_end; r += I4_NW) {
#pragma unroll
        for (int w = 0; w < I4_NW; ++w) {
          const long long ti = r + w;
          if (ti < seg_end) {
            const int s = seq[w];
            const int slot = w * I4_D + s % I4_D;
            if (!s_abort) {
              bool ok = true;
              if (s >= I4_D) ok = mbar_wait_bounded(empty0 + 8 * slot, ((s / I4_D) - 1) & 1, a.budget);
              if (!ok) {
                s_abort = 1;
                atomicOr(a.status, ST_TIMEOUT);
              } else {
                const int row_task = (int)(ti % ntask);
                const uint8_t* src =
                    U.base + ((size_t)row_task * g.ngroup + (size_t)U.ks * I4_KS) * I4_PAIR_BLOCK;
                mbar_arrive_expect_tx(full0 + 8 * slot, bytes);
                bulk_g2s(stage0 + slot * I4_STAGE, src, bytes, full0 + 8 * slot);
                iss[w] = s + 1;
              }
            }
            seq[w] = s + 1;
          }
        }
      }
      i = seg_end;
    }
    // drain: every issued copy has landed before the block may exit
#pragma unroll
    for (int w = 0; w < I4_NW; ++w) {
      for (int d = 0; d < I4_D; ++d) {
        if (iss[w] > d) {
          const int last = ((iss[w] - 1 - d) / I4_D) * I4_D + d;  // last fill of this slot
          if (!mbar_wait_bounded(full0 + 8 * (w * I4_D + d), (last / I4_D) & 1, a.budget))
            atomicOr(a.status, ST_TIMEOUT);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gq = lane >> 2, p = lane & 3;
  int seq = 0;
  // gate/up partial geometry (down reads it)
  const MatGeom gg = rg.m[0];
  const int rows32_gu = gg.ntask * 32;
  for (long long i = t0; i < t1;) {
    const long long u = i / ntask;
    const long long seg_end = min(t1, (u + 1) * ntask);
    const I4Unit U = i4_unit<DOWN>(a, u, nks, p_begin, rg, g);
    const int* toks = a.plan.pass_tok + U.pass * I4_PMAX;

    named_sync(1, I4_NW * 32);
    // slice input, fp32 [slot][512]: x (gate/up) or h = silu(g) * u (down)
    const int kbase = U.ks * (I4_KS * I4_GROUP);
    const int kvalid = U.ng * I4_GROUP;
    for (int e = threadIdx.x; e < U.ntok * I4_KS * I4_GROUP; e += I4_NW * 32) {
      const int ts = e / (I4_KS * I4_GROUP), kk = e % (I4_KS * I4_GROUP);
      float v = 0.f;
      if (kk < kvalid) {
        const int k = kbase + kk;
        if (!DOWN) {
          v = bf16_bits_to_float(a.x[(size_t)toks[ts] * a.H + k]);
        } else {
          const float* pg = a.part_gu + (((size_t)(U.pass * 2 + 0) * gg.nks) * rows32_gu + k) * I4_PMAX + ts;
          const float* pu = a.part_gu + (((size_t)(U.pass * 2 + 1) * gg.nks) * rows32_gu + k) * I4_PMAX + ts;
          const size_t stride = (size_t)rows32_gu * I4_PMAX;
          float gs = 0.f, us = 0.f;
#pragma unroll 4
          for (int s2 = 0; s2 < gg.nks; ++s2) {
            gs += __ldcg(pg + s2 * stride);
            us += __ldcg(pu + s2 * stride);
          }
          v = gs / (1.f + expf(-gs)) * us;
        }
      }
      vin[e] = v;
    }
    named_sync(1, I4_NW * 32);
    for (int e = threadIdx.x; e < I4_KSTEPS * 32; e += I4_NW * 32) {
      const int kk = e >> 5, ln = e & 31;
      const int n = ln >> 2, pp = ln & 3;
      const int ts = n >> 1, part = n & 1;
      uint2 v = make_uint2(0u, 0u);
      if (ts < U.ntok) {
        const float* src = vin + ts * (I4_KS * I4_GROUP) + kk * 16 + 2 * pp;
        __half hi[4], lo[4];
        split_half(src[0], hi[0], lo[0]);
        split_half(src[1], hi[1], lo[1]);
        split_half(src[8], hi[2], lo[2]);
        split_half(src[9], hi[3], lo[3]);
        v.x = part ? pack_half2(lo[0], lo[1]) : pack_half2(hi[0], hi[1]);
        v.y = part ? pack_half2(lo[2], lo[3]) : pack_half2(hi[2], hi[3]);
      }
      xfrag[e] = v;
    }
    named_sync(1, I4_NW * 32);

    const int nb = 2 * U.ntok;  // mma columns that carry data
    for (long long ti = i + warp; ti < seg_end; ti += I4_NW) {
      const int slot = warp * I4_D + seq % I4_D;
      bool ok = !s_abort && mbar_wait_bounded(full0 + 8 * slot, (seq / I4_D) & 1, a.budget);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        const uint8_t* st = smem + slot * I4_STAGE;
        float acc[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[t][c] = 0.f;
        for (int gi = 0; gi < U.ng; ++gi) {
          const uint8_t* blk = st + gi * I4_PAIR_BLOCK;
          const uint4 wa0 = *reinterpret_cast<const uint4*>(blk + lane * 16);
          const uint4 wb0 = *reinterpret_cast<const uint4*>(blk + 512 + lane * 16);
          const uint4 wa1 = *reinterpret_cast<const uint4*>(blk + I4_BLOCK + lane * 16);
          const uint4 wb1 = *reinterpret_cast<const uint4*>(blk + I4_BLOCK + 512 + lane * 16);
          const uint32_t sc0 = *reinterpret_cast<const uint32_t*>(blk + 1024 + gq * 4);
          const uint32_t sc1 = *reinterpret_cast<const uint32_t*>(blk + I4_BLOCK + 1024 + gq * 4);
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint2 b = make_uint2(0u, 0u);
            if (gq < nb) b = xfrag[(gi * 8 + j) * 32 + lane];
            uint32_t x0, x1, x2, x3;
            dequant8(pick4(j < 4 ? wa0 : wb0, j & 3), x0, x1, x2, x3);
            mma_16816(c0, x0, x1, x2, x3, b.x, b.y);
            dequant8(pick4(j < 4 ? wa1 : wb1, j & 3), x0, x1, x2, x3);
            mma_16816(c1, x0, x1, x2, x3, b.x, b.y);
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
        if (p < U.ntok) {
          const int row_task = (int)(ti % ntask);
          const int rows32 = ntask * 32;
          float* dst;
          if (!DOWN)
            dst = a.part_gu + ((size_t)(U.pass * 2 + U.m) * nks + U.ks) * rows32 * I4_PMAX;
          else
            dst = a.part_d + ((size_t)U.pass * nks + U.ks) * rows32 * I4_PMAX;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int r = row_task * 32 + t * 16 + gq;
            dst[(size_t)r * I4_PMAX + p] = acc[t][0] + acc[t][1];
            dst[(size_t)(r + 8) * I4_PMAX + p] = acc[t][2] + acc[t][3];
          }
        }
      } else if (!s_abort) {
        if (lane == 0) { s_abort = 1; atomicOr(a.status, ST_TIMEOUT); }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      ++seq;
    }
    i = seg_end;
  }
}

cudaError_t int4_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(int4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, I4_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(int4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, I4_SMEM);
}

cudaError_t launch_int4_gateup(const ExpertArgs& a, int grid, cudaStream_t s) {
  int4_kernel<false><<<grid, (I4_NW + 1) * 32, I4_SMEM, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_int4_down(const ExpertArgs& a, int grid, cudaStream_t s) {
  int4_kernel<true><<<grid, (I4_NW + 1) * 32, I4_SMEM, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
