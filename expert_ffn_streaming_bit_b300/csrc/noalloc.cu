// moe_forward_stack_noalloc: the one-token decode stack with its per-call
// scratch in a fixed, statically sized device array instead of memory the
// handle allocated.
//
// Who needs this: callers that may not allocate device memory once they are
// running.  Examples are code inside a memory-pool or allocator hook,
// real-time loops that forbid cudaMalloc (it can synchronise the device and
// take unbounded time), and hosts whose allocator is owned by another
// framework.  This call makes no allocation of any kind: no cudaMalloc,
// cudaFree, pinned or pooled allocation, and no library routine that
// allocates.
//
// The array lives in this file and exists once per GPU that loads the
// library.  It holds kNoAllocScratchBytes (1 MiB) on every such GPU until the
// process exits.  The decode kernel takes the same pointers it would take into
// the handle's scratch, so the arithmetic is identical.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

}  // namespace

// In host code this name is only a stand-in for the device array, not its
// address; host code must use the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `device`, looked up once per device
// (with that device current) and cached.
int scratch_address(moe_handle* h, int device, unsigned char** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (device < 0 || device >= kMaxDevices)
    return moe::handle_error(h, MOE_ERR_INVALID_ARG, "device index out of range");
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the fixed scratch array: %s",
                    cudaGetErrorString(e));
      return moe::handle_error(h, MOE_ERR_CUDA, msg);
    }
    g_scratch_addr[device] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[device]);
  return MOE_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

#pragma GCC visibility push(default)
extern "C" moe_status moe_forward_stack_noalloc(moe_handle* h, const void* x, void* y,
                                                int n_layers, void* stream,
                                                int32_t* device_status) {
  moe::DecodeParams p;
  int grid = 0, device = -1;
  int st = moe::stack_launch_params(h, x, y, n_layers, &p, &grid, &device);
  if (st != MOE_OK) return static_cast<moe_status>(st);
  int current = -1;
  if (cudaGetDevice(&current) != cudaSuccess || current != device)
    return static_cast<moe_status>(moe::handle_error(
        h, MOE_ERR_STATE, "moe_forward_stack_noalloc: the handle's device must be current"));
  // Carve-up of the fixed array: barrier words, x double buffer, h, router
  // logit accumulators, ids, weights (the same pieces as the handle's own scratch).
  const size_t bar = 256;
  const size_t xbuf = align256(size_t(2) * p.D * 2);
  const size_t hb = align256(size_t(p.K * p.I + p.S) * 2);
  const size_t part = align256(size_t(2) * p.E * 8);
  const size_t ids = align256(size_t(n_layers) * p.K * 4);
  const size_t need = bar + xbuf + hb + part + 2 * ids;
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "moe_forward_stack_noalloc: this shape needs %zu bytes of scratch; the fixed "
                  "array holds %zu",
                  need, kNoAllocScratchBytes);
    return static_cast<moe_status>(moe::handle_error(h, MOE_ERR_INVALID_ARG, msg));
  }
  unsigned char* base = nullptr;
  st = scratch_address(h, device, &base);
  if (st != MOE_OK) return static_cast<moe_status>(st);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p.bar = reinterpret_cast<uint32_t*>(base);
  p.xbuf = reinterpret_cast<uint16_t*>(base + bar);
  p.h = reinterpret_cast<uint16_t*>(base + bar + xbuf);
  p.lacc = reinterpret_cast<unsigned long long*>(base + bar + xbuf + hb);
  p.ids = reinterpret_cast<int32_t*>(base + bar + xbuf + hb + part);
  p.wts = reinterpret_cast<float*>(base + bar + xbuf + hb + part + ids);
  p.trace = nullptr;  // the trace buffer belongs to the handle's own scratch
  // The array keeps the previous call's contents; the grid-barrier counters,
  // the status word and the router logit accumulators must start at zero.
  // Everything else is written before it is read.
  cudaError_t e = cudaMemsetAsync(base, 0, bar, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.lacc, 0, part, s);
  if (e == cudaSuccess) {
    const int le = moe::decode_launch(p, grid, s, true);
    e = static_cast<cudaError_t>(le);
  }
  // The kernel's status word (timeout, bad id) lives in the fixed array, and
  // the next call clears it: hand it to the caller if asked.  A copy into
  // caller-owned host memory allocates nothing.
  if (e == cudaSuccess && device_status)
    e = cudaMemcpyAsync(device_status, p.bar + 2, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "moe_forward_stack_noalloc: %s", cudaGetErrorString(e));
    return static_cast<moe_status>(moe::handle_error(h, MOE_ERR_CUDA, msg));
  }
  return MOE_OK;
}
#pragma GCC visibility pop
