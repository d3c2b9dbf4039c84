// engine.cu - the C ABI of include/moe.h: context, expert registry, HBM expert cache,
// forward orchestration.  Host code; every step of the layer runs in this library's
// kernels (router.cu, int4.cu, rvq.cu, combine.cu, repack.cu).
//
// Expert storage ("WISP - streaming what can't run", section "Insight (Credit: JustVugg
// / Colibri)": VRAM is checked first, then RAM, with LRU promotion; "2.78T-parameter
// model on a laptop: the NVMe streaming inference engine WASTE", section "Idle weights
// only need to arrive on time": the rest of memory is a bounded expert cache, one
// contiguous record per expert):
//   resident  - every expert's record lives in HBM for the life of the context;
//   streamed  - records live in a pinned host pool; an HBM cache of fixed-size slots
//               holds the recently used ones, least recently used evicted first.  The
//               current layer's experts are pinned while it runs.  Misses are copied
//               host-to-device on a side stream; the hits' kernels run first and each
//               missed expert's kernels wait only for its own copy, so a copy overlaps
//               the compute of the experts before it ("WISP", section "Double-Buffer
//               Async Pipeline").  The shared expert and the routers stay resident.
//               With a pool file the host pool is itself a cache: every record lives
//               in the file, and a bounded pinned RAM cache in front of it holds the
//               recently used ones (filetier.h): VRAM, then RAM, then the file.
// Caching changes only timing: the kernels compute each expert pass the same way and
// the combine sums in a fixed order ("Introducing WARP", section "How WARP keeps the
// model out of RAM": prediction changes timing, never results).
#include <sys/sysinfo.h>
#include <unistd.h>

#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <list>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/moe.h"
#include "common.cuh"
#include "filetier.h"
#include "kernels.h"

using namespace moe;

namespace {

constexpr unsigned long long kDefaultBudget = 2000000000ull;  // ~1 s of SM clock

struct DeviceGuard {
  int old = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&old);
    if (old != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (old >= 0 && cur != old) cudaSetDevice(old);
  }
};

size_t host_available_bytes() {
  FILE* f = fopen("/proc/meminfo", "r");
  if (f) {
    char key[64];
    unsigned long long v;
    char unit[16];
    while (fscanf(f, "%63s %llu %15s", key, &v, unit) == 3) {
      if (strcmp(key, "MemAvailable:") == 0) {
        fclose(f);
        return (size_t)v * 1024ull;
      }
    }
    fclose(f);
  }
  struct sysinfo si;
  if (sysinfo(&si) == 0) return (size_t)si.freeram * si.mem_unit;
  return 0;
}

}  // namespace

struct moe_ctx {
  moe_config cfg{};
  int device = 0, num_sms = 0, pmax = 1;
  RecGeom rg{};
  size_t rec_bytes = 0, blob_bytes = 0;
  bool streamed = false;
  int has_shared = 0;
  int E1 = 0;  // records per layer in the resident slab (E + shared)

  uint8_t* d_slab = nullptr;     // resident: [L][E1] records; streamed: slots
  size_t n_slots = 0;
  uint8_t* d_shared = nullptr;   // streamed: [L] shared records
  uint8_t* h_pool = nullptr;     // streamed: pinned [L][E] records (no pool file)
  // pool file: the records in a file behind a pinned RAM cache of ft->slots() records
  FileTier* ft = nullptr;
  std::string pool_path;
  uint8_t* h_ram = nullptr;                  // pinned RAM slots
  uint8_t* h_wstage = nullptr;               // pinned staging of a registered record
  std::vector<cudaEvent_t> ram_ev;           // [RAM slot] after the last copy that read it
  std::vector<char> ram_used;                // that event was recorded
  float* d_router = nullptr;     // [L][E][H]
  std::vector<char> router_ok, expert_ok;

  uint8_t** d_rec_table = nullptr;  // resident: [L][E+1]; streamed: [E+1]
  uint8_t** h_table = nullptr;      // streamed: pinned [E+1]
  int* d_order = nullptr;           // streamed: [max_pass]
  int* h_order = nullptr;           // pinned

  // LRU cache (streamed)
  std::vector<long long> slot_key;
  std::unordered_map<long long, int> where;
  std::list<int> lru;  // front = most recent
  std::vector<std::list<int>::iterator> lru_it;
  std::vector<char> slot_in_lru, slot_pinned;

  // scratch
  float* d_rpart = nullptr;
  unsigned int* d_ticket = nullptr;
  PlanPtrs plan{};
  void* d_plan_mem = nullptr;
  int* d_store_idx = nullptr;
  float* d_store_w = nullptr;
  std::vector<int> last_T;
  float* d_part_gu = nullptr;  // RVQ gate/up k-slice partials
  float* d_h = nullptr;        // int4 SwiGLU outputs
  float* d_part_d = nullptr;
  int max_pass = 0;
  int big_min = 0, max_big = 0;      // dense (tcgen05) groups: RVQ, resident, max_tokens >= 8
  uint32_t* d_status = nullptr;
  uint32_t* d_dbg_status = nullptr;
  DevCounters* d_counters = nullptr;
  int* h_rb = nullptr;  // pinned readback: hdr(4) | uniq[E] | pass_expert[max_pass]

  static constexpr int kCopyStreams = 4;
  cudaStream_t side[kCopyStreams] = {}, reg = nullptr;
  std::vector<cudaEvent_t> copy_ev;
  // link accounting: each batch of copies (one forward's misses, or one read-ahead) is the
  // interval from its first copy's start to its last copy's end, timed against ref_ev; the
  // busy time is the union of the intervals, merged in issue order
  static constexpr int kBatches = 8;
  struct CopyBatch {
    cudaEvent_t t0 = nullptr, t1[kCopyStreams] = {};
    int ns = 0;
  } batch[kBatches];
  int batch_head = 0, batch_count = 0;  // ring of batches not yet accounted
  cudaEvent_t ref_ev = nullptr;
  double busy_end_ms = -1.0;

  // read-ahead (streamed): the next layer's experts predicted from this layer's router input
  int readahead = 0;
  cudaStream_t pred = nullptr;
  float* d_rpart2 = nullptr;
  unsigned int* d_ticket2 = nullptr;
  void* d_plan_mem2 = nullptr;
  PlanPtrs plan2{};
  DevCounters* d_counters2 = nullptr;
  int* d_pstore_idx = nullptr;
  float* d_pstore_w = nullptr;
  int* h_rb2 = nullptr;                 // pinned readback: hdr(4) | pad | uniq[E]
  std::vector<cudaEvent_t> slot_ev;     // [slot] end of the last read-ahead copy into it
  std::vector<char> slot_inflight;      // that copy may still be running
  std::vector<char> slot_prefetched;    // filled by read-ahead and not looked up since
  unsigned long long prefetches = 0, prefetch_hits = 0;
  uint8_t* d_blob_stage = nullptr;
  uint8_t* d_rec_stage = nullptr;

  unsigned long long hits = 0, misses = 0, bytes_h2d = 0;
  unsigned long long launches = 0;  // kernels this context launched for forwards (host-side count)
  double h2d_ms = 0.0;
  int fail_copies = 0;
  moe_status sticky = MOE_OK;
  unsigned long long budget = kDefaultBudget;

  bool prof = false;
  std::vector<cudaEvent_t> prof_ev;  // [L][5]
  std::vector<char> prof_seen;       // [L]
};

namespace {

moe_status cuda_fail(moe_ctx* c) {
  if (c->sticky == MOE_OK) c->sticky = MOE_ECUDA;
  return c->sticky;
}

#define CK(call)                          \
  do {                                    \
    cudaError_t e_ = (call);              \
    if (e_ != cudaSuccess) return cuda_fail(c); \
  } while (0)

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Map the device status word to a sticky status (synchronises the device).
moe_status check_device(moe_ctx* c) {
  if (c->sticky != MOE_OK) return c->sticky;
  if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail(c);
  uint32_t st = 0;
  if (cudaMemcpy(&st, c->d_status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_fail(c);
  if (st & ST_TIMEOUT) c->sticky = MOE_ETIMEOUT;
  else if (st) c->sticky = MOE_ECUDA;
  return c->sticky;
}

uint8_t* record_ptr_resident(moe_ctx* c, int layer, int expert) {
  const int e = expert < 0 ? c->cfg.num_experts : expert;
  return c->d_slab + ((size_t)layer * c->E1 + e) * c->rec_bytes;
}

void free_all(moe_ctx* c) {
  cudaFree(c->d_slab);
  cudaFree(c->d_shared);
  if (c->h_pool) cudaFreeHost(c->h_pool);
  if (c->ft) {
    delete c->ft;
    c->ft = nullptr;
    if (!c->pool_path.empty()) unlink(c->pool_path.c_str());
  }
  if (c->h_ram) cudaFreeHost(c->h_ram);
  if (c->h_wstage) cudaFreeHost(c->h_wstage);
  for (auto& ev : c->ram_ev) cudaEventDestroy(ev);
  c->ram_ev.clear();
  cudaFree(c->d_router);
  cudaFree(c->d_rec_table);
  if (c->h_table) cudaFreeHost(c->h_table);
  cudaFree(c->d_order);
  if (c->h_order) cudaFreeHost(c->h_order);
  cudaFree(c->d_rpart);
  cudaFree(c->d_ticket);
  cudaFree(c->d_plan_mem);
  cudaFree(c->d_store_idx);
  cudaFree(c->d_store_w);
  cudaFree(c->d_part_gu);
  cudaFree(c->d_h);
  cudaFree(c->d_part_d);
  cudaFree(c->d_status);
  cudaFree(c->d_dbg_status);
  cudaFree(c->d_counters);
  if (c->h_rb) cudaFreeHost(c->h_rb);
  for (auto ev : c->copy_ev) cudaEventDestroy(ev);
  for (auto& b : c->batch) {
    if (b.t0) cudaEventDestroy(b.t0);
    for (auto ev : b.t1)
      if (ev) cudaEventDestroy(ev);
  }
  if (c->ref_ev) cudaEventDestroy(c->ref_ev);
  for (auto ev : c->slot_ev) cudaEventDestroy(ev);
  if (c->pred) cudaStreamDestroy(c->pred);
  cudaFree(c->d_rpart2);
  cudaFree(c->d_ticket2);
  cudaFree(c->d_plan_mem2);
  cudaFree(c->d_counters2);
  cudaFree(c->d_pstore_idx);
  cudaFree(c->d_pstore_w);
  if (c->h_rb2) cudaFreeHost(c->h_rb2);
  for (auto ev : c->prof_ev) cudaEventDestroy(ev);
  for (auto st : c->side)
    if (st) cudaStreamDestroy(st);
  if (c->reg) cudaStreamDestroy(c->reg);
  cudaFree(c->d_blob_stage);
  cudaFree(c->d_rec_stage);
}

moe_status validate(const moe_config* g) {
  if (!g) return MOE_EINVAL;
  if (g->num_layers < 1 || g->hidden < 8 || g->ffn < 8) return MOE_EINVAL;
  if (g->num_experts < 1 || g->num_experts > 1024) return MOE_EINVAL;
  if (g->top_k < 1 || g->top_k > g->num_experts || g->top_k > 32) return MOE_EINVAL;
  if (g->shared_ffn != 0 && g->shared_ffn != g->ffn) return MOE_EINVAL;
  if (g->router != MOE_ROUTER_SOFTMAX_TOPK_RENORM && g->router != MOE_ROUTER_SIGMOID_TOPK_NORM)
    return MOE_EINVAL;
  if (g->max_tokens < 1 || g->max_tokens > 256) return MOE_EINVAL;
  if (g->pool_file && (!g->pool_file[0] || g->hbm_cache_bytes == 0)) return MOE_EINVAL;
  if (g->wfmt == MOE_W_RVQ3_G8) {
    if (g->hidden % 8 || g->ffn % 8) return MOE_EINVAL;
  } else if (g->wfmt == MOE_W_INT4_G128) {
    if (g->hidden % 128 || g->ffn % 128) return MOE_EINVAL;
    if (g->hidden > 8192) return MOE_EINVAL;  // the gate/up kernel stages all of x
  } else {
    return MOE_EINVAL;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_strerror(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_ENOMEM: return "out of memory (HBM or pinned host)";
    case MOE_EBUDGET: return "expert cache below one layer's working set";
    case MOE_ECUDA: return "CUDA error";
    case MOE_ESTATE: return "layer not fully registered";
    case MOE_ETIMEOUT: return "device wait timed out";
    case MOE_ENOTFOUND: return "nothing recorded yet";
    case MOE_EIO: return "expert file I/O failed";
  }
  return "unknown status";
}

size_t moe_expert_blob_bytes(int wfmt, int hidden, int ffn) {
  if (wfmt == MOE_W_RVQ3_G8) {
    if (hidden <= 0 || ffn <= 0 || hidden % 8 || ffn % 8) return 0;
  } else if (wfmt == MOE_W_INT4_G128) {
    if (hidden <= 0 || ffn <= 0 || hidden % 128 || ffn % 128) return 0;
  } else {
    return 0;
  }
  return 2 * blob_matrix_bytes(wfmt, ffn, hidden) + blob_matrix_bytes(wfmt, hidden, ffn);
}

moe_status moe_create(const moe_config* cfg, int device, moe_ctx** out) {
  if (!out) return MOE_EINVAL;
  *out = nullptr;
  moe_status v = validate(cfg);
  if (v != MOE_OK) return v;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return ndev == 0 ? MOE_ECUDA : MOE_EINVAL;
  }
  DeviceGuard dg(device);
  moe_ctx* c = new (std::nothrow) moe_ctx();
  if (!c) return MOE_ENOMEM;
  c->cfg = *cfg;
  c->device = device;
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
  const int L = cfg->num_layers, E = cfg->num_experts, H = cfg->hidden, F = cfg->ffn;
  const int k = cfg->top_k, maxT = cfg->max_tokens;
  c->has_shared = cfg->shared_ffn ? 1 : 0;
  c->E1 = E + c->has_shared;
  c->pmax = cfg->wfmt == MOE_W_INT4_G128 ? I4_PMAX : RVQ_PMAX;
  c->rg = rec_geom(cfg->wfmt, H, F);
  c->rec_bytes = c->rg.bytes;
  c->blob_bytes = moe_expert_blob_bytes(cfg->wfmt, H, F);
  c->streamed = cfg->hbm_cache_bytes != 0;
  c->router_ok.assign(L, 0);
  c->expert_ok.assign((size_t)L * c->E1, 0);
  c->last_T.assign(L, -1);

  // scratch geometry
  c->max_pass = maxT * k + (c->has_shared ? maxT : 0);
  if (cdiv(c->max_pass, c->num_sms) + 2 > 512) {  // passes one expert-kernel block may touch
    delete c;
    return MOE_EINVAL;
  }
  const MatGeom& gg = c->rg.m[0];
  const MatGeom& gd = c->rg.m[2];
  const bool int4 = cfg->wfmt == MOE_W_INT4_G128;
  if (!int4 && !c->streamed && maxT >= GEMM_MIN_TOKENS) {
    c->big_min = GEMM_MIN_TOKENS;
    c->max_big = c->max_pass / GEMM_MIN_TOKENS + 2;
  }
  const size_t part_gu = (size_t)c->max_pass * 2 * gg.nks * gg.ntask * 32 * c->pmax;
  const size_t hbuf = (int4 || c->big_min) ? (size_t)c->max_pass * c->pmax * gg.ntask * 32 : 0;
  const size_t part_d = (size_t)c->max_pass * gd.nks * gd.ntask * 32 * c->pmax;
  const size_t rpart = (size_t)E * router_nch(H) * maxT;
  const size_t router_bytes = (size_t)L * E * H * sizeof(float);

  size_t expert_bytes;
  if (!c->streamed) {
    expert_bytes = (size_t)L * c->E1 * c->rec_bytes;
  } else {
    // a forward pins all its unique experts, at most min(E, max_tokens k) of them, and
    // the next layer's must find room beside the current one's: 2 k at T = 1
    size_t slots = cfg->hbm_cache_bytes / c->rec_bytes;
    if (slots < std::max((size_t)2 * k, std::min((size_t)E, (size_t)maxT * k))) {
      delete c;
      return MOE_EBUDGET;
    }
    slots = std::min(slots, (size_t)L * E);
    c->n_slots = slots;
    expert_bytes = slots * c->rec_bytes + (size_t)L * c->has_shared * c->rec_bytes;
    size_t pool = (size_t)L * E * c->rec_bytes;
    if (cfg->pool_file) {
      const size_t stride = (c->rec_bytes + FT_ALIGN - 1) / FT_ALIGN * FT_ALIGN;
      const size_t ram = std::min<size_t>(cfg->host_cache_bytes / stride, (size_t)L * E);
      if (ram < (size_t)2 * k) {
        delete c;
        return MOE_EBUDGET;
      }
      pool = ram * stride;
    }
    const size_t avail = host_available_bytes();
    if (pool + (8ull << 30) > avail) {
      delete c;
      return MOE_ENOMEM;
    }
  }
  size_t free_b = 0, total_b = 0;
  if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
    delete c;
    return MOE_ECUDA;
  }
  const size_t need = expert_bytes + router_bytes + (part_gu + hbuf + part_d + rpart) * 4 +
                      2 * c->blob_bytes + (64ull << 20);
  if (need + (1ull << 30) > free_b) {
    delete c;
    return MOE_ENOMEM;
  }

#define AL(ptr, bytes)                                              \
  do {                                                              \
    if (cudaMalloc((void**)&(ptr), (bytes)) != cudaSuccess) {       \
      cudaGetLastError();                                           \
      free_all(c);                                                  \
      delete c;                                                     \
      return MOE_ENOMEM;                                            \
    }                                                               \
  } while (0)

  if (!c->streamed) {
    AL(c->d_slab, expert_bytes);
    AL(c->d_rec_table, (size_t)L * (E + 1) * sizeof(uint8_t*));
    std::vector<uint8_t*> tab((size_t)L * (E + 1));
    for (int l = 0; l < L; ++l) {
      for (int e = 0; e < E; ++e) tab[(size_t)l * (E + 1) + e] = record_ptr_resident(c, l, e);
      tab[(size_t)l * (E + 1) + E] = c->has_shared ? record_ptr_resident(c, l, -1) : nullptr;
    }
    cudaMemcpy(c->d_rec_table, tab.data(), tab.size() * sizeof(uint8_t*), cudaMemcpyHostToDevice);
  } else {
    AL(c->d_slab, c->n_slots * c->rec_bytes);
    if (c->has_shared) AL(c->d_shared, (size_t)L * c->rec_bytes);
    AL(c->d_rec_table, (size_t)(E + 1) * sizeof(uint8_t*));
    AL(c->d_order, (size_t)c->max_pass * sizeof(int));
    if (cfg->pool_file) {
      const size_t stride = (c->rec_bytes + FT_ALIGN - 1) / FT_ALIGN * FT_ALIGN;
      const size_t ram = std::min<size_t>(cfg->host_cache_bytes / stride, (size_t)L * E);
      if (cudaHostAlloc((void**)&c->h_ram, ram * stride, cudaHostAllocDefault) != cudaSuccess ||
          cudaHostAlloc((void**)&c->h_wstage, stride, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        free_all(c);
        delete c;
        return MOE_ENOMEM;
      }
      c->ft = new (std::nothrow) FileTier();
      c->pool_path = cfg->pool_file;   // removed by free_all, also if open fails half way
      // reader threads: MOE_FILE_READERS (1..64) where set, else 8
      int readers = 8;
      if (const char* env = getenv("MOE_FILE_READERS")) readers = std::min(64, std::max(1, atoi(env)));
      const int fe = c->ft ? c->ft->open(cfg->pool_file, c->rec_bytes, (long long)L * E, c->h_ram, ram * stride,
                                         readers)
                           : ENOMEM;
      if (fe != 0) {
        free_all(c);
        delete c;
        return fe == ENOMEM ? MOE_ENOMEM : MOE_EIO;
      }
      c->cfg.pool_file = nullptr;   // the caller's string need not outlive the call
      c->ram_ev.resize(c->ft->slots());
      for (auto& ev : c->ram_ev) cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      c->ram_used.assign(c->ft->slots(), 0);
    } else if (cudaHostAlloc((void**)&c->h_pool, (size_t)L * E * c->rec_bytes, cudaHostAllocDefault) !=
               cudaSuccess) {
      cudaGetLastError();
      free_all(c);
      delete c;
      return MOE_ENOMEM;
    }
    if (cudaHostAlloc((void**)&c->h_table, (size_t)(E + 1) * sizeof(uint8_t*), cudaHostAllocDefault) !=
            cudaSuccess ||
        cudaHostAlloc((void**)&c->h_order, (size_t)c->max_pass * sizeof(int), cudaHostAllocDefault) !=
            cudaSuccess) {
      cudaGetLastError();
      free_all(c);
      delete c;
      return MOE_ENOMEM;
    }
    c->slot_key.assign(c->n_slots, -1);
    c->lru_it.resize(c->n_slots);
    c->slot_in_lru.assign(c->n_slots, 0);
    c->slot_pinned.assign(c->n_slots, 0);
    c->copy_ev.resize(E);
    for (auto& ev : c->copy_ev) cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    for (auto& b : c->batch) {
      cudaEventCreate(&b.t0);
      for (auto& ev : b.t1) cudaEventCreate(&ev);
    }
    cudaEventCreate(&c->ref_ev);
    c->slot_ev.resize(c->n_slots);
    for (auto& ev : c->slot_ev) cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    c->slot_inflight.assign(c->n_slots, 0);
    c->slot_prefetched.assign(c->n_slots, 0);
  }
  if (cudaHostAlloc((void**)&c->h_rb, (size_t)(8 + E + c->max_pass) * sizeof(int),
                    cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return MOE_ENOMEM;
  }
  AL(c->d_router, router_bytes);
  AL(c->d_rpart, rpart * sizeof(float));
  AL(c->d_ticket, router_tickets(E) * sizeof(unsigned int));
  if (part_gu) AL(c->d_part_gu, part_gu * sizeof(float));
  if (hbuf) AL(c->d_h, hbuf * sizeof(float));
  AL(c->d_part_d, part_d * sizeof(float));
  AL(c->d_status, 4);
  AL(c->d_dbg_status, 4);
  AL(c->d_counters, sizeof(DevCounters));
  AL(c->d_store_idx, (size_t)L * maxT * k * sizeof(int));
  AL(c->d_store_w, (size_t)L * maxT * k * sizeof(float));
  AL(c->d_blob_stage, c->blob_bytes);
  AL(c->d_rec_stage, c->rec_bytes);
  {
    // plan arrays, one allocation
    const size_t n_int = 16 + (size_t)c->max_pass * (2 + c->pmax) + (size_t)maxT * k * 4 +
                         (size_t)maxT * 2 + E + (size_t)c->max_big * 3 + c->max_pass;
    AL(c->d_plan_mem, n_int * sizeof(int));
    int* p = (int*)c->d_plan_mem;
    c->plan.hdr = (Plan*)p;
    p += 16;
    c->plan.pass_expert = p; p += c->max_pass;
    c->plan.pass_ntok = p; p += c->max_pass;
    c->plan.pass_tok = p; p += (size_t)c->max_pass * c->pmax;
    c->plan.pair_pass = p; p += (size_t)maxT * k;
    c->plan.pair_slot = p; p += (size_t)maxT * k;
    c->plan.idx = p; p += (size_t)maxT * k;
    c->plan.w = (float*)p; p += (size_t)maxT * k;
    c->plan.shared_pass = p; p += maxT;
    c->plan.shared_slot = p; p += maxT;
    c->plan.uniq = p; p += E;
    c->plan.big = p; p += (size_t)c->max_big * 3;
    c->plan.small_order = p; p += c->max_pass;
  }
  if (c->streamed) {
    // read-ahead: a second router scratch and plan, so a prediction never touches the real plan
    AL(c->d_rpart2, rpart * sizeof(float));
    AL(c->d_ticket2, router_tickets(E) * sizeof(unsigned int));
    AL(c->d_counters2, sizeof(DevCounters));
    AL(c->d_pstore_idx, (size_t)maxT * k * sizeof(int));
    AL(c->d_pstore_w, (size_t)maxT * k * sizeof(float));
    const size_t n_int = 16 + (size_t)c->max_pass * (2 + c->pmax) + (size_t)maxT * k * 4 + (size_t)maxT * 2 + E;
    AL(c->d_plan_mem2, n_int * sizeof(int));
    int* p = (int*)c->d_plan_mem2;
    c->plan2.hdr = (Plan*)p;
    p += 16;
    c->plan2.pass_expert = p; p += c->max_pass;
    c->plan2.pass_ntok = p; p += c->max_pass;
    c->plan2.pass_tok = p; p += (size_t)c->max_pass * c->pmax;
    c->plan2.pair_pass = p; p += (size_t)maxT * k;
    c->plan2.pair_slot = p; p += (size_t)maxT * k;
    c->plan2.idx = p; p += (size_t)maxT * k;
    c->plan2.w = (float*)p; p += (size_t)maxT * k;
    c->plan2.shared_pass = p; p += maxT;
    c->plan2.shared_slot = p; p += maxT;
    c->plan2.uniq = p;
    if (cudaHostAlloc((void**)&c->h_rb2, (size_t)(8 + E) * sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      free_all(c);
      delete c;
      return MOE_ENOMEM;
    }
    cudaMemset(c->d_ticket2, 0, router_tickets(E) * sizeof(unsigned int));
  }
#undef AL
  cudaMemset(c->d_ticket, 0, router_tickets(E) * sizeof(unsigned int));
  cudaMemset(c->d_status, 0, 4);
  cudaMemset(c->d_counters, 0, sizeof(DevCounters));
  cudaMemset(c->d_plan_mem, 0, 16 * sizeof(int));
  bool streams_ok = cudaStreamCreateWithFlags(&c->reg, cudaStreamNonBlocking) == cudaSuccess;
  for (auto& st : c->side) streams_ok = streams_ok && cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess;
  if (c->streamed) {
    streams_ok = streams_ok && cudaStreamCreateWithFlags(&c->pred, cudaStreamNonBlocking) == cudaSuccess;
    streams_ok = streams_ok && cudaEventRecord(c->ref_ev, c->side[0]) == cudaSuccess;
  }
  if (!streams_ok ||
      router_set_attributes() != cudaSuccess || int4_set_attributes(H, maxT) != cudaSuccess ||
      rvq_set_attributes() != cudaSuccess || rvq_gemm_set_attributes() != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return MOE_ECUDA;
  }
  *out = c;
  return MOE_OK;
}

moe_status moe_destroy(moe_ctx* c) {
  if (!c) return MOE_OK;
  {
    DeviceGuard dg(c->device);
    cudaDeviceSynchronize();
    free_all(c);
  }
  delete c;
  return MOE_OK;
}

moe_status moe_register_router(moe_ctx* c, int layer, const float* w) {
  if (!c || !w || layer < 0 || layer >= c->cfg.num_layers) return MOE_EINVAL;
  if (c->sticky != MOE_OK) return c->sticky;
  DeviceGuard dg(c->device);
  const size_t n = (size_t)c->cfg.num_experts * c->cfg.hidden;
  float* dst = c->d_router + (size_t)layer * n;
  CK(cudaMemcpy(dst, w, n * sizeof(float), is_device_ptr(w) ? cudaMemcpyDeviceToDevice
                                                              : cudaMemcpyHostToDevice));
  c->router_ok[layer] = 1;
  return MOE_OK;
}

moe_status moe_register_expert(moe_ctx* c, int layer, int expert, const void* blob, size_t bytes) {
  if (!c || !blob || layer < 0 || layer >= c->cfg.num_layers) return MOE_EINVAL;
  if (expert < -1 || expert >= c->cfg.num_experts) return MOE_EINVAL;
  if (expert == -1 && !c->has_shared) return MOE_EINVAL;
  if (bytes != c->blob_bytes) return MOE_EINVAL;
  if (c->sticky != MOE_OK) return c->sticky;
  DeviceGuard dg(c->device);
  const uint8_t* src = (const uint8_t*)blob;
  if (!is_device_ptr(blob)) {
    CK(cudaMemcpyAsync(c->d_blob_stage, blob, bytes, cudaMemcpyHostToDevice, c->reg));
    src = c->d_blob_stage;
  }
  const int E = c->cfg.num_experts;
  uint8_t* dst;
  if (!c->streamed) dst = record_ptr_resident(c, layer, expert);
  else if (expert < 0) dst = c->d_shared + (size_t)layer * c->rec_bytes;
  else dst = c->d_rec_stage;
  CK(launch_repack(c->cfg.wfmt, src, c->cfg.hidden, c->cfg.ffn, dst, c->reg));
  if (c->streamed && expert >= 0) {
    const long long fkey = (long long)layer * E + expert;
    if (c->ft) {
      CK(cudaMemcpyAsync(c->h_wstage, dst, c->rec_bytes, cudaMemcpyDeviceToHost, c->reg));
      CK(cudaStreamSynchronize(c->reg));
      if (c->ft->write(fkey, c->h_wstage) != 0) return MOE_EIO;
    } else {
      uint8_t* pool = c->h_pool + ((size_t)layer * E + expert) * c->rec_bytes;
      CK(cudaMemcpyAsync(pool, dst, c->rec_bytes, cudaMemcpyDeviceToHost, c->reg));
    }
    // a stale cached copy of this expert must not survive re-registration
    const long long key = (long long)layer * E + expert;
    auto it = c->where.find(key);
    if (it != c->where.end()) {
      const int s = it->second;
      if (c->slot_in_lru[s]) { c->lru.erase(c->lru_it[s]); c->slot_in_lru[s] = 0; }
      c->slot_key[s] = -1;
      c->where.erase(it);
    }
  }
  CK(cudaStreamSynchronize(c->reg));
  c->expert_ok[(size_t)layer * c->E1 + (expert < 0 ? E : expert)] = 1;
  return MOE_OK;
}

static moe_status layer_ready(moe_ctx* c, int layer) {
  if (!c->router_ok[layer]) return MOE_ESTATE;
  for (int e = 0; e < c->E1; ++e)
    if (!c->expert_ok[(size_t)layer * c->E1 + e]) return MOE_ESTATE;
  return MOE_OK;
}

static ExpertArgs expert_args(moe_ctx* c, uint8_t* const* table, const void* x, int T) {
  ExpertArgs a{};
  a.rec_table = table;
  a.plan = c->plan;
  a.H = c->cfg.hidden;
  a.F = c->cfg.ffn;
  a.E = c->cfg.num_experts;
  a.T = T;
  a.x = (const uint16_t*)x;
  a.part_gu = c->d_part_gu;
  a.h = c->d_h;
  a.max_tokens = c->cfg.max_tokens;
  a.part_d = c->d_part_d;
  a.range.order = nullptr;
  a.range.p_begin = 0;
  a.range.p_end = -1;
  a.range.count = nullptr;
  a.status = c->d_status;
  a.budget = c->budget;
  return a;
}

static cudaError_t launch_experts(moe_ctx* c, const ExpertArgs& a, cudaStream_t s) {
  cudaError_t e;
  if (c->cfg.wfmt == MOE_W_INT4_G128) {
    e = launch_int4_gateup(a, c->num_sms, s);
    if (e == cudaSuccess) e = launch_int4_down(a, c->num_sms, s);
  } else {
    e = launch_rvq_gateup(a, c->num_sms, s);
    if (e == cudaSuccess) e = launch_rvq_down(a, c->num_sms, s);
  }
  return e;
}

// LRU: find or make a slot for `key`; returns slot and whether it was a hit.
static int cache_get(moe_ctx* c, long long key, bool* hit) {
  auto it = c->where.find(key);
  if (it != c->where.end()) {
    const int s = it->second;
    if (c->slot_in_lru[s]) c->lru.erase(c->lru_it[s]);
    c->lru.push_front(s);
    c->lru_it[s] = c->lru.begin();
    c->slot_in_lru[s] = 1;
    *hit = true;
    return s;
  }
  *hit = false;
  int s = -1;
  // an empty slot first, else the least recently used unpinned one
  if (c->where.size() < c->n_slots) {
    for (size_t i = 0; i < c->n_slots; ++i)
      if (c->slot_key[i] < 0) { s = (int)i; break; }
  }
  if (s < 0) {
    for (auto r = c->lru.rbegin(); r != c->lru.rend(); ++r)
      if (!c->slot_pinned[*r]) { s = *r; break; }
    if (s < 0) return -1;
    c->where.erase(c->slot_key[s]);
    c->lru.erase(c->lru_it[s]);
    c->slot_in_lru[s] = 0;
  }
  c->slot_key[s] = key;
  c->where[key] = s;
  c->lru.push_front(s);
  c->lru_it[s] = c->lru.begin();
  c->slot_in_lru[s] = 1;
  return s;
}

// Forget what a slot holds (its content is unknown after a failed copy).
static void forget_slot(moe_ctx* c, int slot) {
  if (c->slot_key[slot] >= 0) c->where.erase(c->slot_key[slot]);
  c->slot_key[slot] = -1;
  if (c->slot_in_lru[slot]) {
    c->lru.erase(c->lru_it[slot]);
    c->slot_in_lru[slot] = 0;
  }
  c->slot_prefetched[slot] = 0;
}

// Host addresses of the records (layer, experts[i]) for i in [i0, i1): the pinned pool, or
// (pool file) the RAM cache, after reading the absent ones from the file.  A RAM slot is
// reused only after the last copy that read it has finished.  ram_slot[i] is -1 for the
// pinned pool.  The batch holds at most ft->slots() records.
static moe_status host_sources(moe_ctx* c, int layer, const int* experts, int n, const uint8_t** src, int* ram_slot) {
  const int E = c->cfg.num_experts;
  if (!c->ft) {
    for (int i = 0; i < n; ++i) {
      src[i] = c->h_pool + ((size_t)layer * E + experts[i]) * c->rec_bytes;
      ram_slot[i] = -1;
    }
    return MOE_OK;
  }
  std::vector<long long> keys(n);
  for (int i = 0; i < n; ++i) keys[i] = (long long)layer * E + experts[i];
  std::vector<uint8_t*> p(n);
  bool cuda_ok = true;
  const int fe = c->ft->fetch(keys.data(), n, p.data(), ram_slot, [c, &cuda_ok](int slot) {
    if (c->ram_used[slot] && cudaEventSynchronize(c->ram_ev[slot]) != cudaSuccess) cuda_ok = false;
    c->ram_used[slot] = 0;
  });
  if (!cuda_ok) return cuda_fail(c);
  if (fe != 0) return MOE_EIO;
  for (int i = 0; i < n; ++i) src[i] = p[i];
  return MOE_OK;
}

// The copy just queued on cs read RAM slot `slot` (pool file): mark it.
static moe_status ram_slot_read(moe_ctx* c, int slot, cudaStream_t cs) {
  if (slot < 0) return MOE_OK;
  CK(cudaEventRecord(c->ram_ev[slot], cs));
  c->ram_used[slot] = 1;
  return MOE_OK;
}

// ---------------------------------------------------------------- link accounting
static void batch_drain(moe_ctx* c, bool wait);

// A batch of copies runs on the first ns side streams: t0 on side[0], the others wait for it.
static moe_status batch_begin(moe_ctx* c, int ns, int* idx) {
  if (c->batch_count == moe_ctx::kBatches) batch_drain(c, true);
  const int i = (c->batch_head + c->batch_count) % moe_ctx::kBatches;
  moe_ctx::CopyBatch& b = c->batch[i];
  CK(cudaEventRecord(b.t0, c->side[0]));
  for (int q = 1; q < ns; ++q) CK(cudaStreamWaitEvent(c->side[q], b.t0, 0));
  b.ns = ns;
  *idx = i;
  return MOE_OK;
}

static moe_status batch_end(moe_ctx* c, int i) {
  moe_ctx::CopyBatch& b = c->batch[i];
  for (int q = 0; q < b.ns; ++q) CK(cudaEventRecord(b.t1[q], c->side[q]));
  ++c->batch_count;
  return MOE_OK;
}

// Add the finished batches, oldest first, to the link's busy time: each is the interval
// [t0, max t1] against ref_ev, merged with the intervals before it.  wait: wait for all.
// When none is left pending the reference moves to now, which keeps the times short.
static void batch_drain(moe_ctx* c, bool wait) {
  while (c->batch_count > 0) {
    moe_ctx::CopyBatch& b = c->batch[c->batch_head];
    bool done = true;
    for (int q = 0; q < b.ns && done; ++q) {
      const cudaError_t e = wait ? cudaEventSynchronize(b.t1[q]) : cudaEventQuery(b.t1[q]);
      if (e != cudaSuccess) done = false;
    }
    cudaGetLastError();
    if (!done) return;
    float t0 = 0.f, t1 = 0.f;
    if (cudaEventElapsedTime(&t0, c->ref_ev, b.t0) == cudaSuccess) {
      t1 = t0;
      for (int q = 0; q < b.ns; ++q) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, c->ref_ev, b.t1[q]) == cudaSuccess && ms > t1) t1 = ms;
      }
      const double start = std::max((double)t0, c->busy_end_ms);
      if (t1 > start) c->h2d_ms += t1 - start;
      c->busy_end_ms = std::max(c->busy_end_ms, (double)t1);
    }
    cudaGetLastError();
    c->batch_head = (c->batch_head + 1) % moe_ctx::kBatches;
    --c->batch_count;
  }
  if (cudaEventRecord(c->ref_ev, c->side[0]) == cudaSuccess) c->busy_end_ms = 0.0;
  cudaGetLastError();
}

// Read-ahead: route layer nl on this forward's router input x (bf16 on the device, written
// before the plan read-back this forward waited for) with the prediction scratch, and
// start copying the predicted experts that are not cached into unpinned slots, behind
// this forward's miss copies.  Only timing depends on it: a slot's kernels always wait
// for the copy that filled it.
static moe_status readahead(moe_ctx* c, int nl, const void* x, int T) {
  const int E = c->cfg.num_experts, H = c->cfg.hidden;
  RouterArgs ra{};
  ra.x = (const uint16_t*)x;
  ra.W = c->d_router + (size_t)nl * E * H;
  ra.T = T;
  ra.H = H;
  ra.E = E;
  ra.k = c->cfg.top_k;
  ra.kind = c->cfg.router;
  ra.pmax = c->pmax;
  ra.has_shared = 0;
  ra.partial = c->d_rpart2;
  ra.ticket = c->d_ticket2;
  ra.plan = c->plan2;
  ra.store_idx = c->d_pstore_idx;
  ra.store_w = c->d_pstore_w;
  ra.counters = c->d_counters2;
  ra.record_bytes = 0;
  ra.big_min = 0;
  CK(launch_router(ra, c->num_sms, c->pred));
  ++c->launches;
  CK(cudaMemcpyAsync(c->h_rb2, c->plan2.hdr, 4 * sizeof(int), cudaMemcpyDeviceToHost, c->pred));
  CK(cudaMemcpyAsync(c->h_rb2 + 8, c->plan2.uniq, (size_t)E * sizeof(int), cudaMemcpyDeviceToHost, c->pred));
  CK(cudaStreamSynchronize(c->pred));
  std::vector<int> todo;
  const int n_uniq = c->h_rb2[1];
  for (int i = 0; i < n_uniq && i < E; ++i) {
    const int e = c->h_rb2[8 + i];
    if (e >= 0 && e < E && !c->where.count((long long)nl * E + e)) todo.push_back(e);
  }
  if (todo.empty()) return MOE_OK;
  if (c->ft && (int)todo.size() > c->ft->slots()) todo.resize(c->ft->slots());
  std::vector<const uint8_t*> srcs(todo.size());
  std::vector<int> rslot(todo.size());
  moe_status hs = host_sources(c, nl, todo.data(), (int)todo.size(), srcs.data(), rslot.data());
  if (hs != MOE_OK) return hs;
  const int ns = (int)std::min<size_t>(moe_ctx::kCopyStreams, todo.size());
  int bi = -1;
  moe_status bs = batch_begin(c, ns, &bi);
  if (bs != MOE_OK) return bs;
  for (size_t m = 0; m < todo.size(); ++m) {
    const int e = todo[m];
    bool hit = false;
    const int slot = cache_get(c, (long long)nl * E + e, &hit);  // evicts an unpinned slot
    if (slot < 0) break;
    cudaStream_t cs = c->side[m % ns];
    if (c->slot_inflight[slot]) CK(cudaStreamWaitEvent(cs, c->slot_ev[slot], 0));
    if (cudaMemcpyAsync(c->d_slab + (size_t)slot * c->rec_bytes, srcs[m], c->rec_bytes, cudaMemcpyHostToDevice,
                        cs) != cudaSuccess) {
      forget_slot(c, slot);
      return cuda_fail(c);
    }
    moe_status rs = ram_slot_read(c, rslot[m], cs);
    if (rs != MOE_OK) return rs;
    CK(cudaEventRecord(c->slot_ev[slot], cs));
    c->slot_inflight[slot] = 1;
    c->slot_prefetched[slot] = 1;
    ++c->prefetches;
    c->bytes_h2d += c->rec_bytes;
  }
  return batch_end(c, bi);
}

// Router input: xn (bf16) when xres is null; else the fused stack step on the residual
// xres (+ yprev), which writes xres and xn_out.
static moe_status forward_impl(moe_ctx* c, int layer, const void* x, float* xres, const float* yprev,
                               uint16_t* xn_out, float eps, float* out, int T, cudaStream_t s) {
  const int L = c->cfg.num_layers, E = c->cfg.num_experts, H = c->cfg.hidden, k = c->cfg.top_k;
  (void)L;

  RouterArgs ra{};
  ra.x = (const uint16_t*)x;
  ra.xres = xres;
  ra.yprev = yprev;
  ra.xn_out = xn_out;
  ra.eps = eps;
  if (xres) x = xn_out;  // the expert kernels read the normalised input
  ra.W = c->d_router + (size_t)layer * E * H;
  ra.T = T;
  ra.H = H;
  ra.E = E;
  ra.k = k;
  ra.kind = c->cfg.router;
  ra.pmax = c->pmax;
  ra.has_shared = c->has_shared;
  ra.partial = c->d_rpart;
  ra.ticket = c->d_ticket;
  ra.plan = c->plan;
  ra.store_idx = c->d_store_idx + (size_t)layer * c->cfg.max_tokens * k;
  ra.store_w = c->d_store_w + (size_t)layer * c->cfg.max_tokens * k;
  ra.counters = c->d_counters;
  ra.record_bytes = c->rec_bytes;
  ra.big_min = c->big_min;
  // One resident RVQ token with a router of many blocks: the router writes the logits
  // only and the two RVQ kernels take the top-k themselves (the router's last-block step
  // and a dependent plan read fewer on the way to the first expert lookup).  A one-block
  // router leaves the other SMs free, so the expert kernel starts early anyway and
  // routing in it would only add to its path.
  ra.defer = (!c->streamed && c->cfg.wfmt == MOE_W_RVQ3_G8 && T == 1 && c->big_min == 0 && k <= 32 && E <= 512 &&
              !router_one_block(H, T, E)) ? 1 : 0;
  if (c->prof && !c->streamed) CK(cudaEventRecordWithFlags(c->prof_ev[(size_t)layer * 5], s, cudaEventRecordExternal));
  CK(launch_router(ra, c->num_sms, s));
  ++c->launches;

  CombineArgs ca{};
  ca.plan = c->plan;
  ca.part_d = c->d_part_d;
  ca.T = T;
  ca.H = H;
  ca.k = k;
  ca.pmax = c->pmax;
  ca.nks_d = c->rg.m[2].nks;
  ca.has_shared = c->has_shared;
  ca.out = out;
  ca.xres = (xres && yprev) ? xres : nullptr;
  ca.yprev = yprev;

  if (!c->streamed) {
    ExpertArgs a = expert_args(c, c->d_rec_table + (size_t)layer * (E + 1), x, T);
    a.slab_layer = c->d_slab + (size_t)layer * c->E1 * c->rec_bytes;
    a.rec_bytes = c->rec_bytes;
    // one token: exactly one pass per selected expert (+ the shared one), known here, so
    // the expert kernels need not read the count from the plan
    if (T == 1 && c->big_min == 0) a.range.p_end = k + c->has_shared;
    if (ra.defer) {
      a.route_logits = c->d_rpart + (size_t)(router_nch(H) - 1) * E;   // after the slice partials (T = 1)
      a.route_kind = c->cfg.router;
      a.route = OneTokenPlan{E, k, c->pmax, c->has_shared, c->big_min, ra.store_idx, ra.store_w, c->d_counters,
                             (unsigned long long)c->rec_bytes, (unsigned long long)E * H * 4ull};
    }
    cudaEvent_t* ev = c->prof ? &c->prof_ev[(size_t)layer * 5] : nullptr;
    if (ev) CK(cudaEventRecordWithFlags(ev[1], s, cudaEventRecordExternal));
    if (c->cfg.wfmt == MOE_W_INT4_G128) {
      CK(launch_int4_gateup(a, c->num_sms, s));
      if (ev) CK(cudaEventRecordWithFlags(ev[2], s, cudaEventRecordExternal));
      CK(launch_int4_down(a, c->num_sms, s));
      c->launches += 2;
    } else if (c->big_min > 0) {
      // per-token path over the small passes, tcgen05 path over the dense groups
      ExpertArgs as = a;
      as.range.order = c->plan.small_order;
      as.range.count = &c->plan.hdr->n_small;
      CK(launch_rvq_gateup(as, c->num_sms, s));
      CK(launch_rvq_gemm_gateup(a, c->num_sms, s));
      if (ev) CK(cudaEventRecordWithFlags(ev[2], s, cudaEventRecordExternal));
      CK(launch_rvq_down(as, c->num_sms, s));
      CK(launch_rvq_gemm_down(a, c->num_sms, s, c->max_big));   // SwiGLU of the dense groups, then their down
      c->launches += 5;
    } else {
      CK(launch_rvq_gateup(a, c->num_sms, s));
      if (ev) CK(cudaEventRecordWithFlags(ev[2], s, cudaEventRecordExternal));
      CK(launch_rvq_down(a, c->num_sms, s));
      c->launches += 2;
    }
    if (ev) CK(cudaEventRecordWithFlags(ev[3], s, cudaEventRecordExternal));
    CK(launch_combine(ca, s));
    ++c->launches;
    if (ev) {
      CK(cudaEventRecordWithFlags(ev[4], s, cudaEventRecordExternal));
      c->prof_seen[layer] = 1;
    }
    c->last_T[layer] = T;
    return MOE_OK;
  }

  // ---------------- streamed: read the plan back (the one host round trip per layer)
  int* rb = c->h_rb;
  CK(cudaMemcpyAsync(rb, c->plan.hdr, 4 * sizeof(int), cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(rb + 8, c->plan.uniq, (size_t)E * sizeof(int), cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(rb + 8 + E, c->plan.pass_expert, (size_t)c->max_pass * sizeof(int),
                     cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  {
    uint32_t st = 0;
    CK(cudaMemcpy(&st, c->d_status, 4, cudaMemcpyDeviceToHost));
    if (st) {
      c->sticky = (st & ST_TIMEOUT) ? MOE_ETIMEOUT : MOE_ECUDA;
      return c->sticky;
    }
  }
  batch_drain(c, false);
  const int n_pass = rb[0], n_uniq = rb[1], n_routed = rb[2];
  const int* uniq = rb + 8;
  const int* pexp = rb + 8 + E;

  // lookups: hits, hits whose read-ahead copy may still be running, misses
  if (n_uniq < 0 || (size_t)n_uniq > c->n_slots) return MOE_EBUDGET;  // create sized the slots for this
  for (size_t i = 0; i < c->n_slots; ++i) c->slot_pinned[i] = 0;
  std::vector<int> miss_experts, miss_slot, wait_experts, wait_slot;
  std::vector<char> grouped(E, 0);
  for (int i = 0; i < n_uniq; ++i) {
    const int e = uniq[i];
    bool hit = false;
    const int slot = cache_get(c, (long long)layer * E + e, &hit);
    if (slot < 0) return MOE_EBUDGET;  // cannot happen: the pinned ones are fewer than the slots
    c->slot_pinned[slot] = 1;
    c->h_table[e] = c->d_slab + (size_t)slot * c->rec_bytes;
    if (hit) {
      ++c->hits;
      if (c->slot_prefetched[slot]) {
        ++c->prefetch_hits;
        c->slot_prefetched[slot] = 0;
      }
      if (c->slot_inflight[slot]) {
        grouped[e] = 1;
        wait_experts.push_back(e);
        wait_slot.push_back(slot);
      }
    } else {
      ++c->misses;
      c->slot_prefetched[slot] = 0;
      grouped[e] = 1;
      miss_experts.push_back(e);
      miss_slot.push_back(slot);
    }
  }
  c->h_table[E] = c->has_shared ? c->d_shared + (size_t)layer * c->rec_bytes : nullptr;

  // pass order: ready experts (and the shared expert) first, then each waiting expert's
  // passes (read-ahead copies in flight, then misses)
  std::vector<int> group_experts(wait_experts);
  group_experts.insert(group_experts.end(), miss_experts.begin(), miss_experts.end());
  int n_first = 0;
  for (int p = 0; p < n_pass; ++p) {
    const bool shared_pass = p >= n_routed;
    if (shared_pass || !grouped[pexp[p]]) c->h_order[n_first++] = p;
  }
  std::vector<int> group_begin(group_experts.size() + 1);
  int pos = n_first;
  for (size_t m = 0; m < group_experts.size(); ++m) {
    group_begin[m] = pos;
    for (int p = 0; p < n_routed; ++p)
      if (pexp[p] == group_experts[m]) c->h_order[pos++] = p;
  }
  group_begin[group_experts.size()] = pos;
  // the record table and pass order go to the device before the miss copies are queued, so
  // the ready experts' kernels do not wait behind the misses' transfers
  CK(cudaMemcpyAsync(c->d_rec_table, c->h_table, (size_t)(E + 1) * sizeof(uint8_t*),
                     cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(c->d_order, c->h_order, (size_t)n_pass * sizeof(int), cudaMemcpyHostToDevice, s));
  // the ready experts' kernels go first, so they run while the host reads missed records
  // from the file (file tier) and queues their copies
  ExpertArgs a = expert_args(c, c->d_rec_table, x, T);
  a.range.order = c->d_order;
  if (n_first > 0) {
    a.range.p_begin = 0;
    a.range.p_end = n_first;
    CK(launch_experts(c, a, s));
    c->launches += 2;
  }

  // miss copies on the side streams (round-robin), in ascending expert id, one event each
  const int ns = (int)std::min<size_t>(moe_ctx::kCopyStreams, std::max<size_t>(1, miss_experts.size()));
  int bi = -1;
  if (!miss_experts.empty()) {
    moe_status bs = batch_begin(c, ns, &bi);
    if (bs != MOE_OK) return bs;
  }
  // sources: the pinned pool, or the RAM cache in chunks of at most its size (a later
  // chunk's reads wait for the copies of an earlier one only where they reuse its slots)
  const size_t chunk = c->ft ? (size_t)c->ft->slots() : std::max<size_t>(1, miss_experts.size());
  std::vector<const uint8_t*> srcs(miss_experts.size());
  std::vector<int> rslot(miss_experts.size(), -1);
  for (size_t m = 0; m < miss_experts.size(); ++m) {
    cudaStream_t cs = c->side[m % ns];
    const int e = miss_experts[m], slot = miss_slot[m];
    if (m % chunk == 0) {
      const int n = (int)std::min(chunk, miss_experts.size() - m);
      moe_status hs = host_sources(c, layer, miss_experts.data() + m, n, srcs.data() + m, rslot.data() + m);
      if (hs != MOE_OK) {
        for (size_t q = m; q < miss_experts.size(); ++q) forget_slot(c, miss_slot[q]);   // never filled
        return hs;
      }
    }
    const uint8_t* src = srcs[m];
    // a read-ahead copy into the victim slot may still be running: this one goes after it
    if (c->slot_inflight[slot]) CK(cudaStreamWaitEvent(cs, c->slot_ev[slot], 0));
    c->slot_inflight[slot] = 0;
    cudaError_t ce;
    if (c->fail_copies > 0) {
      --c->fail_copies;
      ce = cudaErrorInvalidValue;  // injected failure of the copy call
    } else {
      ce = cudaMemcpyAsync(c->h_table[e], src, c->rec_bytes, cudaMemcpyHostToDevice, cs);
    }
    if (ce != cudaSuccess) {
      forget_slot(c, slot);  // the slot's content is unknown now
      return cuda_fail(c);
    }
    moe_status rs = ram_slot_read(c, rslot[m], cs);
    if (rs != MOE_OK) return rs;
    CK(cudaEventRecord(c->copy_ev[m], cs));
    c->bytes_h2d += c->rec_bytes;
  }
  if (bi >= 0) {
    moe_status be = batch_end(c, bi);
    if (be != MOE_OK) return be;
  }

  for (size_t m = 0; m < group_experts.size(); ++m) {
    if (m < wait_experts.size()) {
      const int slot = wait_slot[m];
      CK(cudaStreamWaitEvent(s, c->slot_ev[slot], 0));
      c->slot_inflight[slot] = 0;  // later copies into the slot follow a host sync past these kernels
    } else {
      CK(cudaStreamWaitEvent(s, c->copy_ev[m - wait_experts.size()], 0));
    }
    a.range.p_begin = group_begin[m];
    a.range.p_end = group_begin[m + 1];
    CK(launch_experts(c, a, s));
    c->launches += 2;
  }
  CK(launch_combine(ca, s));
  ++c->launches;
  c->last_T[layer] = T;
  if (c->readahead && layer + 1 < c->cfg.num_layers && layer_ready(c, layer + 1) == MOE_OK)
    return readahead(c, layer + 1, x, T);
  return MOE_OK;
}

moe_status moe_forward(moe_ctx* c, int layer, const void* x, float* out, int T, void* stream) {
  if (!c || !x || !out || layer < 0 || layer >= c->cfg.num_layers) return MOE_EINVAL;
  if ((uintptr_t)x & 15) return MOE_EINVAL;
  if (T < 1 || T > c->cfg.max_tokens) return MOE_EINVAL;
  if (c->sticky != MOE_OK) return c->sticky;
  moe_status rs = layer_ready(c, layer);
  if (rs != MOE_OK) return rs;
  DeviceGuard dg(c->device);
  return forward_impl(c, layer, x, nullptr, nullptr, nullptr, 0.f, out, T, (cudaStream_t)stream);
}

moe_status moe_forward_residual(moe_ctx* c, int layer, float* x, const float* y_prev, uint16_t* xn, float* y,
                                int T, float eps, void* stream) {
  if (!c || !x || !xn || !y || layer < 0 || layer >= c->cfg.num_layers) return MOE_EINVAL;
  if (T < 1 || T > c->cfg.max_tokens) return MOE_EINVAL;
  if (((uintptr_t)x & 15) || ((uintptr_t)y_prev & 15) || ((uintptr_t)xn & 15)) return MOE_EINVAL;
  if (c->sticky != MOE_OK) return c->sticky;
  moe_status rs = layer_ready(c, layer);
  if (rs != MOE_OK) return rs;
  DeviceGuard dg(c->device);
  cudaStream_t s = (cudaStream_t)stream;
  // every router block re-reads the T rows to take their norms: fuse only small steps
  if ((size_t)T * c->cfg.hidden <= 32768 && T <= ROUTER_FUSED_MAXT)
    return forward_impl(c, layer, nullptr, x, y_prev, xn, eps, y, T, s);
  CK(launch_residual_rmsnorm(x, y_prev, xn, T, c->cfg.hidden, eps, s));
  ++c->launches;
  return forward_impl(c, layer, xn, nullptr, nullptr, nullptr, 0.f, y, T, s);
}

moe_status moe_get_routing(moe_ctx* c, int layer, int* idx, float* w, int* T_out) {
  if (!c || layer < 0 || layer >= c->cfg.num_layers) return MOE_EINVAL;
  DeviceGuard dg(c->device);
  moe_status st = check_device(c);
  if (st != MOE_OK) return st;
  const int T = c->last_T[layer];
  if (T_out) *T_out = T < 0 ? 0 : T;
  if (T < 0) return MOE_ENOTFOUND;
  const size_t n = (size_t)T * c->cfg.top_k;
  const size_t off = (size_t)layer * c->cfg.max_tokens * c->cfg.top_k;
  if (idx) CK(cudaMemcpy(idx, c->d_store_idx + off, n * sizeof(int), cudaMemcpyDeviceToHost));
  if (w) CK(cudaMemcpy(w, c->d_store_w + off, n * sizeof(float), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_residual_rmsnorm(moe_ctx* c, float* x, const float* y, uint16_t* xn, int T, float eps,
                                void* stream) {
  if (!c || !x || !xn || T < 1) return MOE_EINVAL;
  if (((uintptr_t)x & 15) || ((uintptr_t)y & 15)) return MOE_EINVAL;
  if (c->sticky != MOE_OK) return c->sticky;
  DeviceGuard dg(c->device);
  CK(launch_residual_rmsnorm(x, y, xn, T, c->cfg.hidden, eps, (cudaStream_t)stream));
  ++c->launches;
  return MOE_OK;
}

moe_status moe_stats(moe_ctx* c, moe_stats_t* out) {
  if (!c || !out) return MOE_EINVAL;
  DeviceGuard dg(c->device);
  moe_status st = check_device(c);
  DevCounters dc{};
  if (cudaMemcpy(&dc, c->d_counters, sizeof(dc), cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_fail(c);
  if (st == MOE_OK && c->streamed) batch_drain(c, true);
  memset(out, 0, sizeof(*out));
  out->forwards = dc.forwards;
  out->tokens = dc.tokens;
  out->lookups = dc.lookups;
  out->hits = c->streamed ? c->hits : dc.lookups;
  out->misses = c->streamed ? c->misses : 0;
  out->bytes_expert_touched = dc.bytes_touched;
  out->bytes_router = dc.bytes_router;
  out->bytes_h2d = c->bytes_h2d;
  out->record_bytes = c->rec_bytes;
  out->cache_slots = c->n_slots;
  out->h2d_ms = c->h2d_ms;
  out->prefetches = c->prefetches;
  out->prefetch_hits = c->prefetch_hits;
  if (c->ft) {
    out->file_reads = c->ft->reads;
    out->file_read_bytes = c->ft->read_bytes;
    out->ram_hits = c->ft->ram_hits;
    out->ram_misses = c->ft->ram_misses;
    out->file_read_ms = c->ft->read_ms;
    out->file_direct = c->ft->direct() ? 1 : 0;
  }
  out->launches = c->launches;
  return st;
}

moe_status moe_reset_stats(moe_ctx* c) {
  if (!c) return MOE_EINVAL;
  DeviceGuard dg(c->device);
  moe_status st = check_device(c);
  if (st != MOE_OK) return st;
  CK(cudaMemset(c->d_counters, 0, sizeof(DevCounters)));
  if (c->streamed) batch_drain(c, true);
  c->hits = c->misses = c->bytes_h2d = 0;
  c->prefetches = c->prefetch_hits = 0;
  c->launches = 0;
  c->h2d_ms = 0.0;
  if (c->ft) {
    c->ft->reads = c->ft->read_bytes = c->ft->ram_hits = c->ft->ram_misses = 0;
    c->ft->read_ms = 0.0;
  }
  return MOE_OK;
}

moe_status moe_set_readahead(moe_ctx* c, int enable) {
  if (!c || enable < 0 || enable > 1) return MOE_EINVAL;
  if (!c->streamed) return enable ? MOE_EINVAL : MOE_OK;
  c->readahead = enable;
  return MOE_OK;
}

moe_status moe_profile(moe_ctx* c, int enable) {
  if (!c) return MOE_EINVAL;
  if (c->streamed && enable) return MOE_EINVAL;
  DeviceGuard dg(c->device);
  if (enable && c->prof_ev.empty()) {
    c->prof_ev.resize((size_t)c->cfg.num_layers * 5);
    for (auto& ev : c->prof_ev) CK(cudaEventCreate(&ev));
  }
  c->prof_seen.assign(c->cfg.num_layers, 0);
  c->prof = enable != 0;
  return MOE_OK;
}

moe_status moe_profile_read(moe_ctx* c, double* ms, int* n_layers) {
  if (!c || !ms || !n_layers) return MOE_EINVAL;
  DeviceGuard dg(c->device);
  moe_status st = check_device(c);
  if (st != MOE_OK) return st;
  for (int i = 0; i < 4; ++i) ms[i] = 0.0;
  int n = 0;
  for (int l = 0; l < c->cfg.num_layers && !c->prof_ev.empty(); ++l) {
    if (!c->prof_seen[l]) continue;
    for (int i = 0; i < 4; ++i) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, c->prof_ev[(size_t)l * 5 + i], c->prof_ev[(size_t)l * 5 + i + 1]) !=
          cudaSuccess) {
        cudaGetLastError();
        return MOE_ENOTFOUND;
      }
      ms[i] += t;
    }
    ++n;
  }
  *n_layers = n;
  return MOE_OK;
}

moe_status moe_debug_fail_copies(moe_ctx* c, int n) {
  if (!c || n < 0) return MOE_EINVAL;
  c->fail_copies = n;
  return MOE_OK;
}

moe_status moe_debug_wait_timeout(moe_ctx* c, unsigned long long cycles, void* stream, int* status) {
  if (!c || !status) return MOE_EINVAL;
  DeviceGuard dg(c->device);
  CK(cudaMemsetAsync(c->d_dbg_status, 0, 4, (cudaStream_t)stream));
  CK(launch_wait_timeout(c->d_dbg_status, cycles, (cudaStream_t)stream));
  uint32_t st = 0;
  CK(cudaMemcpyAsync(&st, c->d_dbg_status, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream));
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  *status = (st & ST_TIMEOUT) ? MOE_ETIMEOUT : (st ? MOE_ECUDA : MOE_OK);
  return MOE_OK;
}

}  // extern "C"
