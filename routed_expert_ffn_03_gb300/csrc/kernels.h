// kernels.h - host-side launchers of the routed expert FFN kernels (internal).
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <utility>
#include <cstdint>

#include "layout.h"

namespace moe {

struct DevStatusHost {
  uint32_t* word;
  unsigned long long budget;
};

struct DevCounters {           // updated on the device by the router's last block
  unsigned long long forwards, tokens, lookups, bytes_touched, bytes_router;
};

constexpr int ROUTER_FUSED_MAXT = 4;   // tokens of a fused stack step (norm inside the router)

struct RouterArgs {
  const uint16_t* x;     // bf16 [T][H] router input (when xres is null)
  const float* xres;     // fused stack step: fp32 residual [T][H] (null: not fused)
  const float* yprev;    //   previous layer's output [T][H] or null
  uint16_t* xn_out;      //   bf16(rmsnorm(x + yprev)) written here by the last block
  float eps;
  const float* W;        // [E][H]
  int T, H, E, k, kind, pmax, has_shared;
  float* partial;        // [router_nch(H)][T][E]: slice partials, then the logits
  unsigned int* ticket;  // [router_tickets(E)], zero between launches
  PlanPtrs plan;
  int* store_idx;        // per-layer copy of the routing [T][k]
  float* store_w;
  DevCounters* counters;
  unsigned long long record_bytes;
  int big_min;           // > 0: experts with >= big_min tokens form dense groups (pmax must be 1)
  int defer;             // one token: write the logits only, the expert kernels route (see ExpertArgs)
};
cudaError_t launch_router(const RouterArgs& a, int num_sms, cudaStream_t s);
bool router_one_block(int H, int T, int E);   // the router runs as a single block
cudaError_t router_set_attributes();
int router_nch(int H);
int router_tickets(int E);

// Work over passes: [p_begin, p_end) of the order array (identity when order == null);
// p_end < 0 means "to the plan's n_pass".
struct PassRange {
  const int* order;
  int p_begin, p_end;
  const int* count;   // with p_end < 0: the pass count lives here (null: the plan's n_pass)
};

// What the one-token plan needs besides the plan's own arrays.
struct OneTokenPlan {
  int E, k, pmax, has_shared, big_min;
  int* store_idx;               // per-layer copy of the routing [k]
  float* store_w;
  DevCounters* counters;
  unsigned long long record_bytes, router_bytes;
};

// Work split of the RVQ lookup kernel for a pass count fixed at launch, made on the host
// (g = 0: none, the kernel splits; g = -1: equal task ranges).  Groups of g blocks, full
// groups holding kk units at most m_full per block, the left-over blocks the rest at most
// m_rem per block.
struct BlockSplit {
  int g, kk, m_full, m_rem;
};

struct ExpertArgs {
  const uint8_t* const* rec_table;  // [E + 1] record pointers (E = shared expert)
  const uint8_t* slab_layer;        // resident: this layer's records, expert e at e * rec_bytes
  size_t rec_bytes;                 //   (null when streamed: records are found through rec_table)
  PlanPtrs plan;
  int H, F, E, T, max_tokens;
  const uint16_t* x;                // bf16 [T][H] (gate/up input)
  float* part_gu;                   // [max_pass][2][nks_gu][pmax][rows32(F)] gate/up partials
  float* h;                         // [max_pass][pmax][rows32(F)] SwiGLU outputs (int4; RVQ dense path)
  float* part_d;                    // [max_pass][nks_d][pmax][rows32(H)]
  PassRange range;
  uint32_t* status;
  unsigned long long budget;
  // One token routed inside the RVQ kernels (the router deferred, writing the logits
  // only): every block takes the top-k of route_logits itself, and gate/up block 0 writes
  // the plan.  Null: the router wrote the plan.
  const float* route_logits;
  int route_kind;
  OneTokenPlan route;
  BlockSplit split;                 // set by the RVQ launchers
};
#ifdef __CUDACC__
// Record of expert e (E = the shared expert): resident records sit at a fixed stride, so
// no table read is needed; streamed records are wherever the cache put them.
__device__ __forceinline__ const uint8_t* expert_record(const ExpertArgs& a, int e) {
  return a.slab_layer ? a.slab_layer + (size_t)e * a.rec_bytes : a.rec_table[e];
}
#endif

cudaError_t int4_set_attributes(int H, int max_tokens);
cudaError_t rvq_set_attributes();
cudaError_t launch_int4_gateup(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_int4_down(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_rvq_gateup(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_rvq_down(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t rvq_gemm_set_attributes();
cudaError_t launch_rvq_gemm_gateup(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_rvq_gemm_down(const ExpertArgs& a, int grid, cudaStream_t s, int max_big);

struct CombineArgs {
  PlanPtrs plan;
  const float* part_d;
  int T, H, k, pmax, nks_d, has_shared;
  float* out;
  float* xres;           // fused stack step: x += yprev here (null: plain forward)
  const float* yprev;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

cudaError_t launch_residual_rmsnorm(float* x, const float* y, uint16_t* xn, int T, int H, float eps,
                                    cudaStream_t s);
cudaError_t launch_wait_timeout(uint32_t* status, unsigned long long budget, cudaStream_t s);

cudaError_t launch_repack(int wfmt, const uint8_t* blob, int H, int F, uint8_t* rec,
                          cudaStream_t stream);

// Launch with programmatic stream serialisation (the kernel calls pdl_wait before it reads
// what the previous kernel wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// launch_pdl with thread-block clusters of `cluster` consecutive blocks (grid % cluster == 0)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), int grid, int block, int cluster, size_t smem,
                               cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace moe
