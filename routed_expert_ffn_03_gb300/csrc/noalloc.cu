// noalloc.cu - routing without any allocation (moe_route_noalloc).
//
// Some callers cannot allocate device memory at the moment they need the routing: a
// caller recording a CUDA graph (cudaMalloc is not allowed while a stream is being
// captured), an engine whose own pool already holds all free device memory, or a host
// application whose plugin rules forbid allocating.  This entry point runs the same
// router kernel as moe_forward, but its scratch (partial logits, the expert plan, the
// block tickets) lives in one file-scope device array of fixed size instead of memory the
// context allocates.  The array exists once per device for the life of the process.
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = 1u << 20;  // 1 MiB per device
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_ready[kMaxDevices];
unsigned char* g_ptr[kMaxDevices];

// Per device, once, with that device current: the array's device address (the host-side
// name is only a stand-in) and the router kernel's shared-memory attribute.
moe_status setup_device(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ready[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    if (moe::router_set_attributes() != cudaSuccess) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    g_ptr[dev] = static_cast<unsigned char*>(p);
    g_ready[dev] = true;
  }
  *out = g_ptr[dev];
  return MOE_OK;
}

size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

extern "C" moe_status moe_route_noalloc(const uint16_t* x, const float* W, int T, int H, int E, int k, int router,
                                        int* idx, float* w, void* stream) {
  if (!x || !W || !idx || !w) return MOE_EINVAL;
  if (((uintptr_t)x & 7) || ((uintptr_t)W & 15)) return MOE_EINVAL;
  if (T < 1 || T > 256 || H < 8 || H % 8 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) return MOE_EINVAL;
  if (router != MOE_ROUTER_SOFTMAX_TOPK_RENORM && router != MOE_ROUTER_SIGMOID_TOPK_NORM) return MOE_EINVAL;
  // scratch layout: tickets | counters | partial logits [nch][T][E] | plan ints
  const size_t nch = (size_t)moe::router_nch(H);
  const size_t max_pass = (size_t)T * k;  // one token per pass, no shared expert
  const size_t off_cnt = align_up((size_t)moe::router_tickets(E) * sizeof(unsigned int));
  const size_t off_part = align_up(off_cnt + sizeof(moe::DevCounters));
  const size_t off_plan = align_up(off_part + (size_t)E * nch * T * sizeof(float));
  const size_t plan_ints = 16 + 3 * max_pass + 4 * (size_t)T * k + 2 * (size_t)T + E;
  if (off_plan + plan_ints * sizeof(int) > kScratchBytes) return MOE_EINVAL;  // beyond the fixed maximum

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  unsigned char* base = nullptr;
  moe_status st = setup_device(dev, &base);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the tickets must start at zero
  if (cudaMemsetAsync(base, 0, off_part, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  int* p = reinterpret_cast<int*>(base + off_plan);
  moe::RouterArgs a;
  memset(&a, 0, sizeof(a));
  a.x = x;
  a.W = W;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.kind = router;
  a.pmax = 1;
  a.has_shared = 0;
  a.partial = reinterpret_cast<float*>(base + off_part);
  a.ticket = reinterpret_cast<unsigned int*>(base);
  a.plan.hdr = reinterpret_cast<moe::Plan*>(p);
  p += 16;
  a.plan.pass_expert = p; p += max_pass;
  a.plan.pass_ntok = p; p += max_pass;
  a.plan.pass_tok = p; p += max_pass;
  a.plan.pair_pass = p; p += (size_t)T * k;
  a.plan.pair_slot = p; p += (size_t)T * k;
  a.plan.idx = p; p += (size_t)T * k;
  a.plan.w = reinterpret_cast<float*>(p); p += (size_t)T * k;
  a.plan.shared_pass = p; p += T;
  a.plan.shared_slot = p; p += T;
  a.plan.uniq = p;
  a.store_idx = idx;  // the routing lands in the caller's buffers
  a.store_w = w;
  a.counters = reinterpret_cast<moe::DevCounters*>(base + off_cnt);
  a.record_bytes = 0;
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (moe::launch_router(a, nsm > 0 ? nsm : 1, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  return MOE_OK;
}
