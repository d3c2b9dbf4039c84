// filetier.cpp - the file tier of the streamed expert store; see filetier.h.
#include "filetier.h"

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <cerrno>
#include <chrono>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/moe.h"

namespace moe {

FileTier::~FileTier() {
  {
    std::lock_guard<std::mutex> lk(mu_);
    stop_ = true;
  }
  cv_job_.notify_all();
  for (auto& t : pool_) t.join();
  if (fd_ >= 0) ::close(fd_);
  free(wstage_);
}

int FileTier::open(const char* path, size_t rec_bytes, long long n_keys, uint8_t* ram, size_t ram_bytes,
                   int threads) {
  if (!path || rec_bytes == 0 || n_keys <= 0 || !ram || ((uintptr_t)ram % FT_ALIGN) != 0 || threads < 1)
    return EINVAL;
  rec_bytes_ = rec_bytes;
  stride_ = (rec_bytes + FT_ALIGN - 1) / FT_ALIGN * FT_ALIGN;
  n_keys_ = n_keys;
  ram_ = ram;
  n_ram_ = (int)std::min<size_t>(ram_bytes / stride_, (size_t)n_keys);
  if (n_ram_ < 1) return EINVAL;
  int flags = O_RDWR | O_CREAT | O_TRUNC;
#ifdef O_DIRECT
  fd_ = ::open(path, flags | O_DIRECT, 0600);
  direct_ = fd_ >= 0;
#endif
  if (fd_ < 0) fd_ = ::open(path, flags, 0600);
  if (fd_ < 0) return errno;
  if (ftruncate(fd_, (off_t)(stride_ * (size_t)n_keys)) != 0) return errno;
  if (posix_memalign(&wstage_, FT_ALIGN, stride_) != 0) return ENOMEM;
  memset(wstage_, 0, stride_);
  key_.assign(n_ram_, -1);
  it_.resize(n_ram_);
  in_lru_.assign(n_ram_, 0);
  for (int i = n_ram_ - 1; i >= 0; --i) free_.push_back(i);
  for (int i = 0; i < threads; ++i) pool_.emplace_back([this] { worker(); });
  return 0;
}

int FileTier::write(long long key, const uint8_t* rec) {
  if (fd_ < 0 || key < 0 || key >= n_keys_ || !rec) return EINVAL;
  auto w = where_.find(key);
  if (w != where_.end()) drop(w->second);
  memcpy(wstage_, rec, rec_bytes_);
  const off_t off = (off_t)(stride_ * (size_t)key);
  size_t done = 0;
  while (done < stride_) {
    const ssize_t r = pwrite(fd_, (const uint8_t*)wstage_ + done, stride_ - done, off + (off_t)done);
    if (r < 0) {
      if (errno == EINTR) continue;
      return errno;
    }
    if (r == 0) return EIO;
    done += (size_t)r;
  }
  return 0;
}

int FileTier::slot_of(long long key) const {
  auto w = where_.find(key);
  return w == where_.end() ? -1 : w->second;
}

void FileTier::touch(int s) {
  if (in_lru_[s]) lru_.erase(it_[s]);
  lru_.push_front(s);
  it_[s] = lru_.begin();
  in_lru_[s] = 1;
}

void FileTier::drop(int s) {
  if (key_[s] < 0) return;
  where_.erase(key_[s]);
  key_[s] = -1;
  if (in_lru_[s]) {
    lru_.erase(it_[s]);
    in_lru_[s] = 0;
  }
  free_.push_back(s);
}

int FileTier::pread_full(int slot, long long key) {
  uint8_t* dst = ram_ + (size_t)slot * stride_;
  const off_t off = (off_t)(stride_ * (size_t)key);
  size_t done = 0;
  while (done < stride_) {
    const ssize_t r = pread(fd_, dst + done, stride_ - done, off + (off_t)done);
    if (r < 0) {
      if (errno == EINTR) continue;
      return errno;
    }
    if (r == 0) return EIO;   // the file is sized for every key: a short file is an error
    done += (size_t)r;
  }
  return 0;
}

void FileTier::worker() {
  for (;;) {
    std::pair<int, long long> job;
    {
      std::unique_lock<std::mutex> lk(mu_);
      cv_job_.wait(lk, [this] { return stop_ || next_job_ < jobs_.size(); });
      if (stop_) return;
      job = jobs_[next_job_++];
    }
    const int err = pread_full(job.first, job.second);
    {
      std::lock_guard<std::mutex> lk(mu_);
      if (err && !first_err_) first_err_ = err;
      ++jobs_done_;
    }
    cv_done_.notify_one();
  }
}

int FileTier::fetch(const long long* keys, int n, uint8_t** out, int* slot_out,
                    const std::function<void(int)>& before_reuse) {
  if (fd_ < 0 || n < 0 || n > n_ram_) return EINVAL;
  for (int i = 0; i < n; ++i)
    if (keys[i] < 0 || keys[i] >= n_keys_) return EINVAL;
  // hits first: they become the most recent, so the misses below cannot evict them
  std::vector<char> missing(n, 0);
  for (int i = 0; i < n; ++i) {
    auto w = where_.find(keys[i]);
    if (w != where_.end()) {
      touch(w->second);
      slot_out[i] = w->second;
      ++ram_hits;
    } else {
      missing[i] = 1;
    }
  }
  std::vector<std::pair<int, long long>> jobs;
  for (int i = 0; i < n; ++i) {
    if (!missing[i]) continue;
    ++ram_misses;
    // an empty slot, else the least recently used one: the keys of this batch placed so
    // far are the most recent, and n <= slots, so the victim is never one of them
    if (free_.empty()) drop(lru_.back());
    const int s = free_.back();
    free_.pop_back();
    before_reuse(s);
    key_[s] = keys[i];
    where_[keys[i]] = s;
    touch(s);
    slot_out[i] = s;
    jobs.emplace_back(s, keys[i]);
  }
  int err = 0;
  if (!jobs.empty()) {
    const auto t0 = std::chrono::steady_clock::now();
    {
      std::lock_guard<std::mutex> lk(mu_);
      jobs_ = jobs;
      next_job_ = 0;
      jobs_done_ = 0;
      first_err_ = 0;
    }
    cv_job_.notify_all();
    {
      std::unique_lock<std::mutex> lk(mu_);
      cv_done_.wait(lk, [this] { return jobs_done_ == jobs_.size(); });
      err = first_err_;
      jobs_.clear();
      next_job_ = 0;
    }
    read_ms += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    reads += jobs.size();
    read_bytes += (unsigned long long)jobs.size() * stride_;
    if (err)
      for (auto& j : jobs) drop(j.first);   // contents unknown
  }
  for (int i = 0; i < n; ++i) out[i] = err ? nullptr : ram_ + (size_t)slot_out[i] * stride_;
  return err;
}

}  // namespace moe

// ---------------------------------------------------------------- C entry points
struct moe_filetier {
  moe::FileTier ft;
  uint8_t* ram = nullptr;
};

extern "C" moe_status moe_filetier_create(const char* path, size_t rec_bytes, long long n_keys,
                                          unsigned long long ram_bytes, moe_filetier** out) {
  if (!out) return MOE_EINVAL;
  *out = nullptr;
  if (!path || rec_bytes == 0 || n_keys <= 0) return MOE_EINVAL;
  moe_filetier* h = new (std::nothrow) moe_filetier();
  if (!h) return MOE_ENOMEM;
  const size_t stride = (rec_bytes + moe::FT_ALIGN - 1) / moe::FT_ALIGN * moe::FT_ALIGN;
  if (ram_bytes < stride) {
    delete h;
    return MOE_EBUDGET;
  }
  void* ram = nullptr;
  if (posix_memalign(&ram, moe::FT_ALIGN, (size_t)(ram_bytes / stride) * stride) != 0) {
    delete h;
    return MOE_ENOMEM;
  }
  h->ram = (uint8_t*)ram;
  const int e = h->ft.open(path, rec_bytes, n_keys, h->ram, (size_t)ram_bytes, 4);
  if (e) {
    delete h;
    free(ram);
    return e == ENOMEM ? MOE_ENOMEM : (e == EINVAL ? MOE_EINVAL : MOE_EIO);
  }
  *out = h;
  return MOE_OK;
}

extern "C" moe_status moe_filetier_write(moe_filetier* h, long long key, const void* rec) {
  if (!h || !rec) return MOE_EINVAL;
  const int e = h->ft.write(key, (const uint8_t*)rec);
  return e == 0 ? MOE_OK : (e == EINVAL ? MOE_EINVAL : MOE_EIO);
}

extern "C" moe_status moe_filetier_fetch(moe_filetier* h, const long long* keys, int n, const void** out,
                                         int* slots) {
  if (!h || !keys || !out || !slots || n < 0) return MOE_EINVAL;
  const int e = h->ft.fetch(keys, n, (uint8_t**)out, slots, [](int) {});
  return e == 0 ? MOE_OK : (e == EINVAL ? MOE_EINVAL : MOE_EIO);
}

extern "C" moe_status moe_filetier_info(const moe_filetier* h, moe_filetier_stats_t* out) {
  if (!h || !out) return MOE_EINVAL;
  out->slots = (unsigned long long)h->ft.slots();
  out->stride = (unsigned long long)h->ft.stride();
  out->direct = h->ft.direct() ? 1 : 0;
  out->reads = h->ft.reads;
  out->read_bytes = h->ft.read_bytes;
  out->ram_hits = h->ft.ram_hits;
  out->ram_misses = h->ft.ram_misses;
  out->read_ms = h->ft.read_ms;
  return MOE_OK;
}

extern "C" void moe_filetier_destroy(moe_filetier* h) {
  if (!h) return;
  uint8_t* ram = h->ram;
  delete h;
  free(ram);
}
