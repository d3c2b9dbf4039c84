// kernels.h - host-side launchers of the routed expert FFN kernels (internal).
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
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

struct RouterArgs {
  const uint16_t* x;     // bf16 [T][H]
  const float* W;        // [E][H]
  int T, H, E, k, kind, pmax, has_shared;
  float* partial;        // [E][nch][T]
  unsigned int* ticket;  // zero between launches
  PlanPtrs plan;
  int* store_idx;        // per-layer copy of the routing [T][k]
  float* store_w;
  DevCounters* counters;
  unsigned long long record_bytes;
};
cudaError_t launch_router(const RouterArgs& a, int num_sms, cudaStream_t s);
cudaError_t router_set_attributes();
int router_nch(int H);

// Work over passes: [p_begin, p_end) of the order array (identity when order == null);
// p_end < 0 means "to the plan's n_pass".
struct PassRange {
  const int* order;
  int p_begin, p_end;
};

struct ExpertArgs {
  const uint8_t* const* rec_table;  // [E + 1] record pointers (E = shared expert)
  PlanPtrs plan;
  int H, F, E, T;
  const uint16_t* x;                // bf16 [T][H] (gate/up input)
  float* part_gu;                   // [max_pass][2][nks_gu][rows32(F)][pmax]
  float* part_d;                    // [max_pass][nks_d][rows32(H)][pmax]
  PassRange range;
  uint32_t* status;
  unsigned long long budget;
};
cudaError_t launch_int4_gateup(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_int4_down(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_rvq_gateup(const ExpertArgs& a, int grid, cudaStream_t s);
cudaError_t launch_rvq_down(const ExpertArgs& a, int grid, cudaStream_t s);

struct CombineArgs {
  PlanPtrs plan;
  const float* part_d;
  int T, H, k, pmax, nks_d, has_shared;
  float* out;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

cudaError_t launch_residual_rmsnorm(float* x, const float* y, uint16_t* xn, int T, int H, float eps,
                                    cudaStream_t s);
cudaError_t launch_wait_timeout(uint32_t* status, unsigned long long budget, cudaStream_t s);

cudaError_t launch_repack(int wfmt, const uint8_t* blob, int H, int F, uint8_t* rec,
                          cudaStream_t stream);

}  // namespace moe
