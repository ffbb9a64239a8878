// Expert store file writer and bounded-parallel reader (see store.h).
#ifndef _GNU_SOURCE
#define _GNU_SOURCE  // O_DIRECT
#endif
#include "store.h"

#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cerrno>
#include <cstring>

namespace moe {

namespace {

// pwrite/pread of exactly `bytes` (retrying short transfers); false on error.
bool write_all(int fd, const uint8_t* src, int64_t bytes, int64_t off) {
  while (bytes > 0) {
    const ssize_t n = pwrite(fd, src, static_cast<size_t>(bytes), off);
    if (n < 0 && errno == EINTR) continue;
    if (n <= 0) return false;
    src += n;
    off += n;
    bytes -= n;
  }
  return true;
}

bool read_all(int fd, uint8_t* dst, int64_t bytes, int64_t off) {
  while (bytes > 0) {
    const ssize_t n = pread(fd, dst, static_cast<size_t>(bytes), off);
    if (n < 0 && errno == EINTR) continue;
    if (n <= 0) return false;
    dst += n;
    off += n;
    bytes -= n;
  }
  return true;
}

StoreHeader make_header(const Dims& d, int L, int64_t blob) {
  StoreHeader h{};
  std::memcpy(h.magic, kStoreMagic, sizeof h.magic);
  h.version = 1;
  h.D = static_cast<int32_t>(d.D);
  h.E = static_cast<int32_t>(d.E);
  h.I = static_cast<int32_t>(d.I);
  h.K = static_cast<int32_t>(d.K);
  h.S = static_cast<int32_t>(d.S);
  h.group = kGroup;
  h.L = L;
  h.blob_bytes = blob;
  h.stride = store_stride(blob);
  h.data_offset = kStorePage;
  return h;
}

}  // namespace

int store_write(const Dims& d, int L, const moe_layer_weights* layers, const char* path,
                std::string* err) {
  const int64_t blob = expert_blob_bytes(d);
  const StoreHeader hd = make_header(d, L, blob);
  const int fd = ::open(path, O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
  if (fd < 0) {
    *err = std::string("cannot create the expert store: ") + std::strerror(errno);
    return -1;
  }
  std::vector<uint8_t> page(static_cast<size_t>(kStorePage), 0);
  std::memcpy(page.data(), &hd, sizeof hd);
  bool ok = write_all(fd, page.data(), kStorePage, 0);
  std::vector<uint8_t> buf(static_cast<size_t>(d.E * hd.stride));
  for (int l = 0; l < L && ok; ++l) {
    const moe_layer_weights& w = layers[l];
    std::memset(buf.data(), 0, buf.size());
    parallel_for(d.E, [&](int64_t e) {
      repack_expert(d, w.exp_gate[e], w.exp_up[e], w.exp_down[e], buf.data() + e * hd.stride);
    });
    ok = write_all(fd, buf.data(), static_cast<int64_t>(buf.size()),
                   hd.data_offset + int64_t(l) * d.E * hd.stride);
  }
  if (!ok) *err = std::string("writing the expert store failed: ") + std::strerror(errno);
  if (::close(fd) != 0 && ok) {
    ok = false;
    *err = std::string("closing the expert store failed: ") + std::strerror(errno);
  }
  return ok ? 0 : -1;
}

ExpertStore::~ExpertStore() {
  {
    std::lock_guard<std::mutex> lock(mu_);
    stop_ = true;
  }
  cv_work_.notify_all();
  for (auto& t : workers_) t.join();
  if (fd_ >= 0) ::close(fd_);
}

int ExpertStore::open(const char* path, const Dims& d, int L, int64_t blob, int io_threads,
                      bool direct_ok, std::string* err) {
  const StoreHeader want = make_header(d, L, blob);
  int fd = -1;
  if (direct_ok) fd = ::open(path, O_RDONLY | O_DIRECT | O_CLOEXEC);
  direct_ = fd >= 0;
  if (fd < 0) fd = ::open(path, O_RDONLY | O_CLOEXEC);
  if (fd < 0) {
    *err = std::string("cannot open the expert store: ") + std::strerror(errno);
    return -1;
  }
  fd_ = fd;
  // the header through an aligned page (direct I/O needs one)
  void* page = nullptr;
  if (posix_memalign(&page, kStorePage, kStorePage) != 0) {
    *err = "out of host memory";
    return -1;
  }
  bool got = read_all(fd_, static_cast<uint8_t*>(page), kStorePage, 0);
  if (!got && direct_) {  // the file system refused direct I/O: read through the page cache
    ::close(fd_);
    fd_ = ::open(path, O_RDONLY | O_CLOEXEC);
    direct_ = false;
    got = fd_ >= 0 && read_all(fd_, static_cast<uint8_t*>(page), kStorePage, 0);
  }
  StoreHeader have{};
  if (got) std::memcpy(&have, page, sizeof have);
  std::free(page);
  if (!got) {
    *err = "cannot read the expert store header";
    return -1;
  }
  if (std::memcmp(have.magic, want.magic, sizeof want.magic) != 0 || have.version != want.version ||
      have.D != want.D || have.E != want.E || have.I != want.I || have.K != want.K ||
      have.S != want.S || have.group != want.group || have.L != want.L ||
      have.blob_bytes != want.blob_bytes || have.stride != want.stride ||
      have.data_offset != want.data_offset) {
    *err = "the expert store does not match this configuration";
    return -1;
  }
  struct stat sb;
  if (fstat(fd_, &sb) != 0 ||
      sb.st_size < want.data_offset + int64_t(L) * want.E * want.stride) {
    *err = "the expert store is truncated";
    return -1;
  }
  E_ = want.E;
  stride_ = want.stride;
  data_offset_ = want.data_offset;
  const int n = io_threads < 1 ? 1 : io_threads;
  for (int i = 0; i < n; ++i) workers_.emplace_back([this] { worker(); });
  return 0;
}

void ExpertStore::worker() {
  for (;;) {
    Job job;
    {
      std::unique_lock<std::mutex> lock(mu_);
      cv_work_.wait(lock, [this] { return stop_ || next_ < queue_.size(); });
      if (stop_) return;
      job = queue_[next_++];
    }
    const bool ok = !job.fail && read_all(fd_, job.dst, job.bytes, job.offset);
    {
      std::lock_guard<std::mutex> lock(mu_);
      if (!ok) (*failed_)[job.req] = 1;
      if (--pending_ == 0) cv_done_.notify_all();
    }
  }
}

int ExpertStore::read(const std::vector<int>& layer, const std::vector<int>& expert,
                      const std::vector<uint8_t*>& dst, std::vector<int>* failed, int fail_chunk) {
  failed->assign(layer.size(), 0);
  if (layer.empty()) return 0;
  {
    std::lock_guard<std::mutex> lock(mu_);
    queue_.clear();
    next_ = 0;
    failed_ = failed;
    int chunk = 0;
    for (size_t i = 0; i < layer.size(); ++i) {
      const int64_t base = data_offset_ + (int64_t(layer[i]) * E_ + expert[i]) * stride_;
      for (int64_t o = 0; o < stride_; o += kReadChunk) {
        const int64_t n = stride_ - o < kReadChunk ? stride_ - o : kReadChunk;
        queue_.push_back(Job{base + o, dst[i] + o, n, static_cast<int>(i), ++chunk == fail_chunk});
      }
    }
    pending_ = static_cast<int>(queue_.size());
  }
  cv_work_.notify_all();
  std::unique_lock<std::mutex> lock(mu_);
  cv_done_.wait(lock, [this] { return pending_ == 0; });
  queue_.clear();
  next_ = 0;
  int bad = 0;
  for (int f : *failed) bad += f;
  return bad;
}

}  // namespace moe
