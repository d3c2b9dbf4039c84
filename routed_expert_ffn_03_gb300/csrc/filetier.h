// filetier.h - the file tier of the streamed expert store (host code, no CUDA).
//
// "WISP - streaming what can't run", section "Insight (Credit: JustVugg / Colibri)":
// an expert is looked up in VRAM, then in RAM, then read from the SSD, with LRU
// promotion.  This is the RAM and SSD part: every expert record lives in one file, at a
// 4096-byte aligned offset (its key times the record stride), and a bounded RAM cache of
// record-sized slots holds the recently used ones, least recently used evicted first.
// Reads of one batch run in parallel on a small pool of reader threads, with O_DIRECT
// where the filesystem takes it (so the page cache neither serves nor holds them), else
// buffered.  The RAM slots are memory the caller owns (pinned host memory in the engine,
// so the HBM copies start from them directly).
#pragma once

#include <condition_variable>
#include <cstddef>
#include <cstdint>
#include <functional>
#include <list>
#include <mutex>
#include <thread>
#include <unordered_map>
#include <vector>

namespace moe {

constexpr size_t FT_ALIGN = 4096;

class FileTier {
 public:
  ~FileTier();
  // Create (truncate) the file at `path` for n_keys records of rec_bytes and use the
  // caller's `ram` (ram_bytes, FT_ALIGN-aligned) as the RAM slots.  Returns 0 or an errno.
  int open(const char* path, size_t rec_bytes, long long n_keys, uint8_t* ram, size_t ram_bytes, int threads);
  // Write record `key` (rec_bytes at `rec`); a RAM copy of the key is dropped.  Returns 0
  // or an errno.
  int write(long long key, const uint8_t* rec);
  // Make the n keys (distinct) resident in RAM slots and return their addresses; the keys
  // are the most recently used afterwards.  n must not exceed slots().  Before a slot is
  // reused, before_reuse(slot) is called (the engine waits there for the last copy that
  // read the slot).  Returns 0 or an errno (a failed read leaves its slot empty).
  int fetch(const long long* keys, int n, uint8_t** out, int* slot_out, const std::function<void(int)>& before_reuse);
  // The slot holding key, or -1 (no LRU update).
  int slot_of(long long key) const;
  int slots() const { return n_ram_; }
  size_t stride() const { return stride_; }
  bool direct() const { return direct_; }

  unsigned long long reads = 0, read_bytes = 0, ram_hits = 0, ram_misses = 0;
  double read_ms = 0.0;   // wall time of the read batches

 private:
  int pread_full(int slot, long long key);
  void worker();
  void touch(int s);
  void drop(int s);

  int fd_ = -1;
  bool direct_ = false;
  size_t rec_bytes_ = 0, stride_ = 0;
  long long n_keys_ = 0;
  uint8_t* ram_ = nullptr;
  int n_ram_ = 0;
  std::vector<long long> key_;
  std::unordered_map<long long, int> where_;
  std::list<int> lru_;   // front = most recent
  std::vector<std::list<int>::iterator> it_;
  std::vector<char> in_lru_;
  std::vector<int> free_;    // slots holding no key
  void* wstage_ = nullptr;   // FT_ALIGN-aligned staging for writes

  // reader pool: jobs (slot, key) of one batch
  std::vector<std::thread> pool_;
  std::mutex mu_;
  std::condition_variable cv_job_, cv_done_;
  std::vector<std::pair<int, long long>> jobs_;
  size_t next_job_ = 0, jobs_done_ = 0;
  int first_err_ = 0;
  bool stop_ = false;
};

}  // namespace moe
