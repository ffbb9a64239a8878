// Expert store: the storage tier under the per-layer HBM slot cache.
//
// The pages' runtime keeps the routed experts of every layer in a file on the
// SSD and reads the cold ones with bounded parallel pread() calls into
// buffers the GPU can see, rather than mapping the file and taking page
// faults (blog.hypho.cn "TurboFieldfare gemma4 out-of-core inference",
// section "为什么不用 mmap？": one cold expert in 2.79 ms by pread against
// 9.88 ms by demand paging; shilu.ai "drumih/turbo-fieldfare", section
// 推理引擎的工作原理: misses of the layer's LFU slot cache are read into
// GPU-visible buffers while the GPU computes the shared expert).
//
// File layout: a 4096-byte header (StoreHeader, zero padded), then for layer
// l and expert e the repacked routed-expert blob (the layout of internal.h)
// at data_offset + (l * E + e) * stride, where stride is the blob size
// rounded up to 4096 so that every blob starts on a page and can be read
// with direct I/O.
#pragma once
#include <condition_variable>
#include <cstdint>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "repack.h"

namespace moe {

constexpr char kStoreMagic[8] = {'M', 'O', 'E', 'S', 'T', 'O', 'R', '1'};
constexpr int64_t kStorePage = 4096;
constexpr int64_t kReadChunk = int64_t(1) << 20;  // bytes per pread call

struct StoreHeader {
  char magic[8];
  int32_t version;  // 1
  int32_t D, E, I, K, S, group, L;
  int32_t reserved[2];  // zero; keeps the 64-bit fields at byte 48 without implicit padding
  int64_t blob_bytes, stride, data_offset;
};

inline int64_t store_stride(int64_t blob) { return (blob + kStorePage - 1) / kStorePage * kStorePage; }

// Writes the store for `layers` (host memory, canonical form) to `path`.
// Returns 0, or -1 with *err set.
int store_write(const Dims& d, int L, const moe_layer_weights* layers, const char* path,
                std::string* err);

// An open store and its reader threads.  read() is called by one thread at a
// time (the handle's owner).
class ExpertStore {
 public:
  ExpertStore() = default;
  ExpertStore(const ExpertStore&) = delete;
  ExpertStore& operator=(const ExpertStore&) = delete;
  ~ExpertStore();

  // Opens `path`, checks its header against (d, L, blob) and starts
  // io_threads reader threads.  Direct I/O is used when the file system
  // accepts it and `direct_ok` (the staging buffers are page aligned).
  int open(const char* path, const Dims& d, int L, int64_t blob, int io_threads, bool direct_ok,
           std::string* err);

  // Reads blob (layer[i], expert[i]) into dst[i] (stride() bytes each) for
  // every request, split into kReadChunk preads that up to io_threads threads
  // run at once; returns when all have finished.  failed[i] is set to 1 if
  // any read of request i failed or came up short.  fail_chunk > 0 makes
  // the fail_chunk-th chunk of this call fail without reading (host-side
  // fault injection).  Returns the number of failed requests.
  int read(const std::vector<int>& layer, const std::vector<int>& expert,
           const std::vector<uint8_t*>& dst, std::vector<int>* failed, int fail_chunk);

  int64_t stride() const { return stride_; }
  bool direct() const { return direct_; }
  int threads() const { return static_cast<int>(workers_.size()); }

 private:
  struct Job {
    int64_t offset;
    uint8_t* dst;
    int64_t bytes;
    int req;
    bool fail;
  };
  void worker();

  int fd_ = -1;
  bool direct_ = false;
  int E_ = 0;
  int64_t stride_ = 0, data_offset_ = 0;
  std::vector<std::thread> workers_;
  std::mutex mu_;
  std::condition_variable cv_work_, cv_done_;
  std::vector<Job> queue_;
  size_t next_ = 0;
  int pending_ = 0;
  std::vector<int>* failed_ = nullptr;
  bool stop_ = false;
};

}  // namespace moe
