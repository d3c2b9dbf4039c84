// combine.cu - weighted combine of the selected experts, the residual + RMS-norm step of
// the layer stack, and the bounded-wait check used by the failure tests.
//
// Combine: out[t][r] = sum_{j = 0..k-1} w[t][j] * y_{t,j}[r]  (+ y_shared[t][r]),
// in rank order j, the shared expert (weight 1) added last; y of one pass is the sum of
// its down-projection k-slice partials (part_d[pass][ks][slot][row]) in a fixed order.
// The order never depends on timing, so the result is the same bits whatever the cache
// did.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Block = 32 output rows x 8 k-slice lanes.  Lane kl sums slices kl, kl+8, ... of each
// selected expert in slice order; the 8 lane sums are then added in lane order, the
// experts in rank order, the shared expert last.  The (expert, slice) loads of a thread
// are independent and issued CB_BATCH at a time, so a token's k experts cost one round
// trip to memory, not k.
constexpr int CB_ROWS = 32, CB_KL = 8, CB_MAXJ = 33, CB_BATCH = 16;
__global__ void __launch_bounds__(CB_ROWS * CB_KL) combine_kernel(CombineArgs a) {
  __shared__ float red[CB_KL][CB_MAXJ][CB_ROWS];
  __shared__ long long s_base[CB_MAXJ];
  __shared__ float s_w[CB_MAXJ];
  const int t = blockIdx.y;
  const int rl = threadIdx.x & (CB_ROWS - 1), kl = threadIdx.x / CB_ROWS;
  const int r = blockIdx.x * CB_ROWS + rl;
  const int rows32 = cdiv(a.H, 32) * 32;
  const size_t slot_stride = rows32, ks_stride = (size_t)a.pmax * rows32;
  const int nj = a.k + (a.has_shared ? 1 : 0);
  // The plan entries come from the router, which finished before the expert kernels ran
  // (each of them waited for its predecessor), so they are read before the wait; the
  // down partials are read after it.
  if (threadIdx.x < nj) {
    const int j = threadIdx.x;
    int pass, slot;
    if (j < a.k) {
      pass = a.plan.pair_pass[t * a.k + j];
      slot = a.plan.pair_slot[t * a.k + j];
      s_w[j] = a.plan.w[t * a.k + j];
    } else {
      pass = a.plan.shared_pass[t];
      slot = a.plan.shared_slot[t];
      s_w[j] = 1.f;
    }
    s_base[j] = (long long)pass * a.nks_d * ks_stride + (long long)slot * slot_stride;
  }
  for (int j = 0; j < nj; ++j) red[kl][j][rl] = 0.f;
  pdl_wait();  // part_d comes from the kernels before
  pdl_launch_dependents();
  __syncthreads();
  const int nper = kl < a.nks_d ? cdiv(a.nks_d - kl, CB_KL) : 0;   // slices of this lane per expert
  const int U = r < a.H ? nj * nper : 0;
  int lj = 0, lm = 0;     // (expert, slice) of the next load
  int sj = 0, sm = 0;     // (expert, slice) of the next add
  float run = 0.f;        // running sum of expert sj, in ascending slice order
  for (int u0 = 0; u0 < U; u0 += CB_BATCH) {
    float v[CB_BATCH];
#pragma unroll
    for (int q = 0; q < CB_BATCH; ++q) {
      v[q] = 0.f;
      if (u0 + q < U) {
        v[q] = __ldcg(a.part_d + s_base[lj] + r + (size_t)(kl + CB_KL * lm) * ks_stride);
        if (++lm == nper) { lm = 0; ++lj; }
      }
    }
#pragma unroll
    for (int q = 0; q < CB_BATCH; ++q) {
      if (u0 + q < U) {
        run += v[q];
        if (++sm == nper) {
          red[kl][sj][rl] = run;
          run = 0.f;
          sm = 0;
          ++sj;
        }
      }
    }
  }
  __syncthreads();
  if (kl == 0 && r < a.H) {
    float acc = 0.f;
    for (int j = 0; j < nj; ++j) {
      float y = 0.f;
#pragma unroll
      for (int q = 0; q < CB_KL; ++q) y += red[q][j][rl];
      if (j < a.k) acc = fmaf(s_w[j], y, acc);
      else acc += y;
    }
    const size_t o = (size_t)t * a.H + r;
    if (a.xres) a.xres[o] += a.yprev[o];  // stack step: the residual takes y_prev before y is overwritten
    a.out[o] = acc;
  }
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cdiv(a.H, CB_ROWS), a.T);
  cfg.blockDim = dim3(CB_ROWS * CB_KL);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

// x += y (y may be null); xn = bf16(x / sqrt(mean(x^2) + eps)).  One block of 256
// threads per row; the sum of squares is reduced in the fixed order of block_inv_rms, the
// same one the router's fused stack step uses.
__global__ void __launch_bounds__(256) residual_rmsnorm_kernel(float* __restrict__ x, const float* __restrict__ y,
                                                               uint16_t* __restrict__ xn, int H, float eps) {
  __shared__ float red[32];
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  float* xr = x + (size_t)t * H;
  const float* yr = y ? y + (size_t)t * H : nullptr;
  const float inv = block_inv_rms(xr, yr, H, eps, red);
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float v = xr[h];
    if (yr) {
      v += yr[h];
      xr[h] = v;
    }
    xn[(size_t)t * H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(v * inv));
  }
}

cudaError_t launch_residual_rmsnorm(float* x, const float* y, uint16_t* xn, int T, int H, float eps,
                                    cudaStream_t s) {
  return launch_pdl(residual_rmsnorm_kernel, T, 256, 0, s, x, y, xn, H, eps);
}

// One bounded wait on an mbarrier phase that nothing completes.  On expiry it records
// ST_TIMEOUT in the status word and returns; it never traps and never hangs.
__global__ void wait_timeout_kernel(uint32_t* status, unsigned long long budget) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_fence_init();
    if (!mbar_wait_bounded(b, 0, budget)) atomicOr(status, ST_TIMEOUT);
  }
}

cudaError_t launch_wait_timeout(uint32_t* status, unsigned long long budget, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(status, budget);
  return cudaGetLastError();
}

}  // namespace moe
