// common.cuh - device helpers shared by the kernels of the routed expert FFN.
//
// Status word: every kernel that can fail reports through one device word owned by
// the context.  Bits are OR-ed in; the host maps them to moe_status.  Every device
// wait is bounded by a budget of SM clock cycles, so no kernel can spin forever: on
// expiry it sets ST_TIMEOUT, drains its own bulk copies (again bounded) and returns.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace moe {

enum : uint32_t {
  ST_TIMEOUT = 1u,   // a bounded wait ran out
  ST_BADPLAN = 2u,   // routing produced an out-of-range expert (never expected)
};

struct DevStatus {
  uint32_t* word;          // OR-ed status bits
  unsigned long long budget;  // cycles a single wait may take
};

__device__ __forceinline__ void report(const DevStatus& st, uint32_t bits) {
  atomicOr(st.word, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete, for at most `budget` cycles.
// Returns false on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((unsigned long long)(clock64() - t0) > budget) return false;
  }
}

// ---------------------------------------------------------------- bulk copy (TMA, 1-D)
// global -> shared, completion counted on `bar` in bytes.  dst, src 16-B aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Start moving `bytes` (a multiple of 16, 16-B aligned) from global memory into L2 so a
// later load hits there; no completion to wait for.
// atomic add with acquire-release semantics at GPU scope: the writes this thread has
// seen (its block's, after a barrier) are visible to whoever reads the new value, and
// what that thread wrote before is visible here
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- named barrier
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- tensor-core mma (legacy
// warp-level path; used where a warp dequantises its own operand in registers)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// ---------------------------------------------------------------- small conversions
__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}
// Split an fp32 value into fp16 hi + lo with hi + lo == v to within 2^-22 |v|
// (hi = round(v), lo = round(v - hi); v - hi is exact in fp32).
__device__ __forceinline__ void split_half(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace moe

namespace moe {
// ---------------------------------------------------------------- programmatic dependent launch
// wait: block until the preceding kernel in the stream has completed and its memory is
// visible (a no-op when the launch did not ask for programmatic serialisation).
// launch_dependents: let the next kernel's blocks be scheduled now; they still run their
// own wait before reading what this kernel writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
}  // namespace moe

namespace moe {
// 1 / sqrt(mean((x + y)^2) + eps) over one row of H values (y may be null; H % 4 == 0,
// rows 16-byte aligned), reduced in a fixed order that depends only on NTHR, the logical
// thread count (the first NTHR threads hold data): thread i sums float4s i, i + NTHR, ...
// in batches of 8, then warp trees, then a tree over the NTHR / 32 warps.  Every caller
// uses the same NTHR, so every kernel that takes this norm of a row gets the same bits.
// All threads of the block call it; red needs 32 floats.
constexpr int RMS_NTHR = 256;
__device__ __forceinline__ float block_inv_rms(const float* x, const float* y, int H, float eps, float* red) {
  float ss = 0.f;
  const int n4 = H >> 2;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const float4* y4 = reinterpret_cast<const float4*>(y);
  if ((int)threadIdx.x < RMS_NTHR) {
    for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * RMS_NTHR) {  // 8 (x, y) float4 loads in flight, summed in order
      float4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * RMS_NTHR;
        v[q] = i < n4 ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (y && i < n4) {
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
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0 && warp < RMS_NTHR / 32) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < RMS_NTHR / 32 ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)H + eps);
  __syncthreads();
  return inv;
}

// block_inv_rms on values already in registers: for a thread i < RMS_NTHR, v[q] is float4
// i + q * RMS_NTHR of the row (zero past the row; NV <= 8, so H <= 32 * RMS_NTHR), the same
// elements and order as block_inv_rms, so the same bits.
template <int NV>
__device__ __forceinline__ float block_inv_rms_regs(const float4 (&v)[NV], int H, float eps, float* red) {
  static_assert(NV <= 8, "one batch");
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    ss = fmaf(v[q].x, v[q].x, ss);
    ss = fmaf(v[q].y, v[q].y, ss);
    ss = fmaf(v[q].z, v[q].z, ss);
    ss = fmaf(v[q].w, v[q].w, ss);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0 && warp < RMS_NTHR / 32) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float w = lane < RMS_NTHR / 32 ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 0) red[0] = w;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)H + eps);
  __syncthreads();
  return inv;
}
}  // namespace moe
