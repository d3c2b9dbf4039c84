// layout.h - kernel layout of an expert record and the per-forward plan.
//
// The boundary blob (documented in include/moe.h) is repacked at registration into the
// layout below, which the kernels stream with coalesced 16-byte loads.  One expert is
// one contiguous record (gate | up | down, each 256-byte aligned), so a cache miss is a
// single host-to-device copy ("2.78T-parameter model on a laptop: the NVMe streaming
// inference engine WASTE", section "Idle weights only need to arrive on time": one read
// per expert).
//
// int4 (symmetric, 128-element groups along K), per matrix [R rows][K]:
//   rows are taken 32 at a time ("row pair" = two 16-row mma tiles); for each row pair
//   and each 128-wide group there is a 2112-byte block:
//     [tile 0: k-chunk 0 (32 lanes x 16 B) | k-chunk 1 (32 lanes x 16 B) | 8 x u32 scales]
//     [tile 1: same]
//   Lane (g = lane/4, p = lane%4) of k-chunk c holds, in word j (mma k-step 4c + j, 16
//   input elements starting at kb = 128 * group + 16 * (4c + j)), the eight nibbles of
//   its m16n8k16 A fragment:
//     bits  0-3  W[r][kb+2p]     bits 16-19 W[r][kb+2p+1]      (r = 16 * tile + g)
//     bits  4-7  W[r+8][kb+2p]   bits 20-23 W[r+8][kb+2p+1]
//     bits  8-11 W[r][kb+2p+8]   bits 24-27 W[r][kb+2p+9]
//     bits 12-15 W[r+8][kb+2p+8] bits 28-31 W[r+8][kb+2p+9]
//   Scale word g = fp16 pair (s[r][group] low, s[r+8][group] high).  Padding rows are
//   zero (q = 0, s = 0).
//
// RVQ (3 stages, 8-wide groups along K), per matrix [R rows][K], G = K / 8:
//   fp16 codebooks [3][256][8] as in the blob (12288 B), then the codes in k-slices of
//   64 groups and row blocks of 32 rows; per (k-slice, row block) 6144 bytes laid out as
//   [12 word quads][32 lanes][16 B].  Lane l owns row 32 * block + l; its 48 words hold
//   the 64 groups' codes (3 bytes each, stage order 0,1,2) in the order i = 0..63 where
//   position i carries group q = 64 * slice + (l XOR i).  Codes of padding rows and of
//   groups >= G are zero (their input elements are zero, so they add nothing).
#pragma once
#include <cstddef>
#include <cstdint>

#ifdef __CUDACC__
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

enum { WFMT_RVQ = 1, WFMT_INT4 = 2 };

constexpr int ROWS_PER_TASK = 32;   // both formats: one warp task covers 32 rows

// int4
constexpr int I4_GROUP = 128;
constexpr int I4_BLOCK = 1056;           // one 16-row tile x one group
constexpr int I4_PAIR_BLOCK = 2 * I4_BLOCK;
constexpr int I4_KS = 2;                 // groups per k-slice / task (256 inputs)
constexpr int I4_PMAX = 4;               // tokens per pass (hi/lo fill the 8 mma columns)

// RVQ
constexpr int RVQ_GROUP = 8;
constexpr int RVQ_CB_BYTES = 3 * 256 * 8 * 2;
constexpr int RVQ_KS = 64;               // groups per k-slice
constexpr int RVQ_TASK_BYTES = 32 * RVQ_KS * 3;  // 6144
constexpr int RVQ_PMAX = 1;

MOE_HD size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
MOE_HD int cdiv(int a, int b) { return (a + b - 1) / b; }

struct MatGeom {
  int rows, K;      // logical shape (rows x K, K = input dim)
  int ntask;        // row tasks (32 rows each)
  int ngroup;       // groups along K
  int nks;          // k-slices
  int ks_groups;    // groups per k-slice
  size_t bytes;     // bytes of this matrix in the kernel layout
};

MOE_HD MatGeom mat_geom(int wfmt, int rows, int K) {
  MatGeom g;
  g.rows = rows;
  g.K = K;
  g.ntask = cdiv(rows, ROWS_PER_TASK);
  if (wfmt == WFMT_INT4) {
    g.ngroup = K / I4_GROUP;
    g.ks_groups = I4_KS;
    g.nks = cdiv(g.ngroup, I4_KS);
    g.bytes = (size_t)g.ntask * g.ngroup * I4_PAIR_BLOCK;
  } else {
    g.ngroup = K / RVQ_GROUP;
    g.ks_groups = RVQ_KS;
    g.nks = cdiv(g.ngroup, RVQ_KS);
    g.bytes = (size_t)RVQ_CB_BYTES + (size_t)g.nks * g.ntask * RVQ_TASK_BYTES;
  }
  return g;
}

struct RecGeom {
  MatGeom m[3];     // gate, up, down
  size_t off[3];    // byte offset of each matrix in the record
  size_t bytes;     // record bytes (256-aligned)
};

MOE_HD RecGeom rec_geom(int wfmt, int H, int F) {
  RecGeom r;
  r.m[0] = mat_geom(wfmt, F, H);
  r.m[1] = mat_geom(wfmt, F, H);
  r.m[2] = mat_geom(wfmt, H, F);
  r.off[0] = 0;
  r.off[1] = align256(r.m[0].bytes);
  r.off[2] = r.off[1] + align256(r.m[1].bytes);
  r.bytes = r.off[2] + align256(r.m[2].bytes);
  return r;
}

// Boundary blob offsets (the documented input format).
MOE_HD size_t blob_matrix_bytes(int wfmt, int rows, int K) {
  if (wfmt == WFMT_INT4) return (size_t)rows * K / 2 + (size_t)rows * (K / I4_GROUP) * 2;
  return (size_t)RVQ_CB_BYTES + (size_t)rows * (K / RVQ_GROUP) * 3;
}

// ---------------------------------------------------------------- per-forward plan
// Built on the device by the router kernel.  A "pass" is (expert, up to PMAX tokens);
// routed experts come in ascending id, each expert's tokens in ascending order, then
// the shared expert's passes.  Every later kernel iterates over passes.
struct Plan {
  int n_pass;          // passes this forward
  int n_uniq;          // unique routed experts
  int n_routed_pass;   // passes of routed experts (shared passes follow)
  int T;
  int n_big;           // expert token groups for the dense (tcgen05) path
  int n_small;         // passes left for the per-token path (listed in small_order)
};

constexpr int GEMM_MIN_TOKENS = 8;   // an expert with this many tokens takes the dense path
constexpr int GEMM_MAX_TOKENS = 32;  // tokens per dense group (64 mma columns, hi/lo)

struct PlanPtrs {
  Plan* hdr;
  int* pass_expert;    // [max_pass]   expert id, E = shared
  int* pass_ntok;      // [max_pass]
  int* pass_tok;       // [max_pass][PMAX]
  int* pair_pass;      // [maxT][k]
  int* pair_slot;      // [maxT][k]
  int* shared_pass;    // [maxT]
  int* shared_slot;    // [maxT]
  int* uniq;           // [E]
  int* idx;            // [maxT][k]   routing of this forward
  float* w;            // [maxT][k]
  int* big;            // [max_big][3] (expert, first pass, tokens) of the dense groups
  int* small_order;    // [max_pass]   the other passes, ascending
};

}  // namespace moe
