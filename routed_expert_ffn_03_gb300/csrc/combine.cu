// combine.cu - weighted combine of the selected experts, the residual + RMS-norm step of
// the layer stack, and the bounded-wait check used by the failure tests.
//
// Combine: out[t][r] = sum_{j = 0..k-1} w[t][j] * y_{t,j}[r]  (+ y_shared[t][r]),
// in rank order j, the shared expert (weight 1) added last; y of one pass is the sum of
// its down-projection k-slice partials in slice order.  The order never depends on
// timing, so the result is the same bits whatever the cache did.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void combine_kernel(CombineArgs a) {
  const int t = blockIdx.y;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= a.H) return;
  const int rows32 = cdiv(a.H, 32) * 32;
  const size_t ks_stride = (size_t)rows32 * a.pmax;
  float acc = 0.f;
  for (int j = 0; j < a.k; ++j) {
    const int pass = a.plan.pair_pass[t * a.k + j];
    const int slot = a.plan.pair_slot[t * a.k + j];
    const float* src = a.part_d + (size_t)pass * a.nks_d * ks_stride + (size_t)r * a.pmax + slot;
    float y = 0.f;
    for (int ks = 0; ks < a.nks_d; ++ks) y += __ldcg(src + ks * ks_stride);
    acc = fmaf(a.plan.w[t * a.k + j], y, acc);
  }
  if (a.has_shared) {
    const int pass = a.plan.shared_pass[t];
    const int slot = a.plan.shared_slot[t];
    const float* src = a.part_d + (size_t)pass * a.nks_d * ks_stride + (size_t)r * a.pmax + slot;
    float y = 0.f;
    for (int ks = 0; ks < a.nks_d; ++ks) y += __ldcg(src + ks * ks_stride);
    acc += y;
  }
  a.out[(size_t)t * a.H + r] = acc;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  dim3 grid(cdiv(a.H, 256), a.T);
  combine_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// x += y (y may be null); xn = bf16(x / sqrt(mean(x^2) + eps)).  One block per row; the
// sum of squares is reduced in a fixed order.
__global__ void residual_rmsnorm_kernel(float* __restrict__ x, const float* __restrict__ y,
                                        uint16_t* __restrict__ xn, int H, float eps) {
  __shared__ float red[32];
  const int t = blockIdx.x;
  float* xr = x + (size_t)t * H;
  float ss = 0.f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float v = xr[h];
    if (y) {
      v += y[(size_t)t * H + h];
      xr[h] = v;
    }
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)H + eps);
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(xr[h] * inv);
    xn[(size_t)t * H + h] = __bfloat16_as_ushort(b);
  }
}

cudaError_t launch_residual_rmsnorm(float* x, const float* y, uint16_t* xn, int T, int H, float eps,
                                    cudaStream_t s) {
  residual_rmsnorm_kernel<<<T, 256, 0, s>>>(x, y, xn, H, eps);
  return cudaGetLastError();
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
