// C ABI of libmoe_b300 (declared in include/moe.h): handle lifetime, weight
// repack and upload, the resident and streaming forward paths, and the
// per-layer expert-slot cache.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "internal.h"
#include "repack.h"
#include "store.h"

using namespace moe;

namespace {

thread_local std::string g_create_error;
int g_inject_pinned_fail = 0;

struct Inject {
  int h2d_fail_in = 0;  // fail the n-th next miss copy (1 = next)
  int slow_copy_ms = 0;
  int stall_ms = 0;     // next decode launch: first grid barrier cannot complete, this wait limit
  int read_fail_in = 0; // fail the first read of the n-th next expert-store batch (1 = next)
  int gemm_stall_ms = 0;// next grouped-GEMM launch: the MMA role stalls, this wait limit
};

}  // namespace

struct moe_handle {
  moe_config cfg{};
  Dims d{};
  int device = 0;
  int num_sms = 0;
  int64_t blob = 0;
  int64_t fixed = 0;
  // device memory
  uint8_t* dev_weights = nullptr;  // fixed parts of all layers + resident experts or slots
  int64_t dev_weight_bytes = 0;
  LayerDev* dev_layers = nullptr;
  std::vector<LayerDev> layers;
  uint8_t* scratch = nullptr;
  int64_t scratch_bytes = 0;
  uint16_t* xbuf = nullptr;
  float* h = nullptr;
  unsigned long long* lacc = nullptr;
  int32_t* ids = nullptr;
  float* wts = nullptr;
  uint32_t* bar = nullptr;
  uint16_t* io_x = nullptr;  // device copies for host-io calls
  uint16_t* io_y = nullptr;
  // host memory
  uint8_t* pool = nullptr;  // pinned expert pool (streaming)
  int64_t pool_bytes = 0;
  std::unique_ptr<ExpertStore> store;  // expert store file (streaming from the SSD tier)
  uint8_t* staging = nullptr;          // pinned: top_k blobs read from the store
  cudaEvent_t staging_free = nullptr;  // the staging buffers' last copies are done
  uint16_t* pin_x = nullptr;
  uint16_t* pin_y = nullptr;
  int32_t* pin_ids = nullptr;
  uint32_t* pin_status = nullptr;
  // streams/events
  cudaStream_t side = nullptr;
  std::vector<cudaEvent_t> layer_done, copy_done;
  cudaEvent_t ev_ids = nullptr;
  cudaEvent_t ev_sync = nullptr;  // host waits on the caller's stream (sync_stream)
  std::vector<SlotTable> tables;
  DecodeParams base{};
  int grid = 0;
  int last_T = 0, last_layers = 0;
  bool last_prefill = false;
  uint64_t* trace = nullptr;  // [grid][kTraceMaxLayers][kTraceEvents], inside scratch
  bool trace_on = false;
  // prefill (T >= 2, resident mode)
  struct LayerMaps {
    CUtensorMap gu_code[2], gu_sb[2], dn_code[2], dn_sb[2];  // [0] routed, [1] shared
    CUtensorMap rt;  // router weight as two fp16 parts, [2 Epad][D]
  };
  std::vector<LayerMaps> maps;
  CUtensorMap bmap_gu[2][kNBox], bmap_dn[2][kNBox];  // activation operands: [0] routed,
                                                    // [1] shared; one per tile height
  uint16_t* pf_xperm = nullptr;        // x16 rows in bucket order (routed gate/up operand)
  uint16_t* pf_rw = nullptr;           // router weights as fp16 parts, [L][2 Epad][D]
  int32_t* pf_hist = nullptr;          // bucketing counts / write bases
  CUtensorMap bmap_rt;                 // x16 in 64 x 128 boxes (router operand)
  bool prefill_ok = false;
  int mt_gu_r = 0, mt_dn = 0, mt_gu_s = 0;
  uint8_t* pf = nullptr;  // prefill scratch (one allocation)
  int64_t pf_bytes = 0;
  uint16_t* pf_x16 = nullptr;
  float* pf_sigma = nullptr;
  float* pf_rscale = nullptr;
  float* pf_hscale = nullptr;
  float* pf_partials = nullptr;
  int32_t* pf_ids = nullptr;     // [L][Tmax][K]
  float* pf_wts = nullptr;       // [L][Tmax][K]
  int32_t* pf_forced = nullptr;  // [Tmax][K]
  int32_t* pf_counts = nullptr;
  int32_t* pf_offsets = nullptr;
  int32_t* pf_perm = nullptr;
  int32_t* pf_inv = nullptr;
  GemmUnit* pf_units_gu = nullptr;
  GemmUnit* pf_units_dn = nullptr;
  int32_t* pf_nunits = nullptr;
  uint16_t* pf_hr = nullptr;
  uint16_t* pf_hs = nullptr;
  uint16_t* pf_e = nullptr;
  float* pf_s = nullptr;
  uint16_t* pf_xs[2] = {nullptr, nullptr};  // stack double buffer
  // phase timing of multi-token calls while tracing is on: 6 events per call
  std::vector<cudaEvent_t> pf_ev;
  int pf_ev_calls = 0;
  Inject inj;
  int timeout_ms = 10000;
  std::string err;
};

struct moe_slot_plan {
  SlotTable t;
};

namespace {

moe_status fail(moe_handle* h, moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h)
    h->err = buf;
  else
    g_create_error = buf;
  return s;
}

#define CUDA_TRY(h, call)                                                                       \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess)                                                                      \
      return fail((h), e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s", \
                  #call, cudaGetErrorString(e_));                                               \
  } while (0)

bool valid_qt(const moe_qtensor& t) { return t.q && t.scale && t.bias; }

void free_all(moe_handle* h) {
  if (!h) return;
  if (h->side) cudaStreamSynchronize(h->side);
  if (h->dev_weights || h->scratch) cudaDeviceSynchronize();
  for (auto e : h->layer_done) cudaEventDestroy(e);
  for (auto e : h->copy_done) cudaEventDestroy(e);
  for (auto e : h->pf_ev) cudaEventDestroy(e);
  if (h->ev_ids) cudaEventDestroy(h->ev_ids);
  if (h->ev_sync) cudaEventDestroy(h->ev_sync);
  if (h->staging_free) cudaEventDestroy(h->staging_free);
  if (h->side) cudaStreamDestroy(h->side);
  cudaFree(h->dev_weights);
  cudaFree(h->dev_layers);
  cudaFree(h->scratch);
  cudaFree(h->pf);
  cudaFree(h->pf_rw);
  cudaFreeHost(h->pool);
  cudaFreeHost(h->staging);
  h->store.reset();
  cudaFreeHost(h->pin_x);
  cudaFreeHost(h->pin_y);
  cudaFreeHost(h->pin_ids);
  cudaFreeHost(h->pin_status);
}

// Host wait on an event with the handle's deadline.  The first kSpinUs are
// spent polling without sleeping: a decode token takes well under that, and
// a sleep of a few microseconds costs tens of them in scheduler latency on
// the host.  Longer waits poll every 20 us so that they do not hold a core.
constexpr int64_t kSpinUs = 5000;

moe_status wait_event(moe_handle* h, cudaEvent_t ev) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorNotReady) return fail(h, MOE_ERR_CUDA, "event wait: %s", cudaGetErrorString(e));
    const int64_t us = std::chrono::duration_cast<std::chrono::microseconds>(
                           std::chrono::steady_clock::now() - t0)
                           .count();
    if (us > int64_t(h->timeout_ms) * 1000)
      return fail(h, MOE_ERR_TIMEOUT, "device work did not finish in %d ms", h->timeout_ms);
    if (us < kSpinUs) std::this_thread::yield();
    else std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

moe_status sync_stream(moe_handle* h, cudaStream_t s) {
  if (!h->ev_sync) CUDA_TRY(h, cudaEventCreateWithFlags(&h->ev_sync, cudaEventDisableTiming));
  CUDA_TRY(h, cudaEventRecord(h->ev_sync, s));
  return wait_event(h, h->ev_sync);
}

// Reads the device status word (synchronising) and maps it to a status.
moe_status check_device_status(moe_handle* h, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(h->pin_status, h->bar + 2, 4, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return fail(h, MOE_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  moe_status st = sync_stream(h, s);
  if (st != MOE_OK) return st;
  const uint32_t v = *h->pin_status;
  if (v == DEV_OK) return MOE_OK;
  cudaMemsetAsync(h->bar, 0, kBarWords * 4, s);
  cudaMemsetAsync(h->lacc, 0, 2 * h->d.E * 8, s);  // an aborted launch may leave partial sums
  cudaStreamSynchronize(s);
  if (v == DEV_TIMEOUT) return fail(h, MOE_ERR_TIMEOUT, "a device-side wait timed out");
  return fail(h, MOE_ERR_DEVICE, "a kernel reported an out-of-range expert id");
}

int gcd(int a, int b) { return b ? gcd(b, a % b) : a; }

constexpr int kPhaseTimedCalls = 256;  // multi-token calls timed per moe_prefill_phase_ms read

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status launch(moe_handle* h, const DecodeParams& p, cudaStream_t s) {
  int e;
  if (h->inj.stall_ms > 0) {  // injected: a barrier that nothing completes, a short wait limit
    DecodeParams q = p;
    q.stall_first_barrier = 1;
    q.timeout_ns = uint64_t(h->inj.stall_ms) * 1000000ull;
    h->inj.stall_ms = 0;
    e = decode_launch(q, h->grid, s, true);
  } else {
    e = decode_launch(p, h->grid, s, true);
  }
  if (e != 0)
    return fail(h, MOE_ERR_CUDA, "decode kernel launch: %s",
                cudaGetErrorString(static_cast<cudaError_t>(e)));
  return MOE_OK;
}

// The misses of one cache step from the expert store: the blobs are read
// into the pinned staging buffers by the store's reader threads (bounded
// parallel pread), then each is copied into its slot on the side stream.
// A blob that could not be read leaves its slot empty.
moe_status cache_fill_from_store(moe_handle* h, int layer, const int32_t* ids, int k,
                                 moe_cache_result* out, uint8_t* slots) {
  // the staging buffers may still feed the previous step's copies
  if (h->staging_free) {
    const cudaError_t e = cudaEventSynchronize(h->staging_free);
    if (e != cudaSuccess) return fail(h, MOE_ERR_CUDA, "staging wait: %s", cudaGetErrorString(e));
  }
  std::vector<int> lay, exp, miss_i;
  std::vector<uint8_t*> dst;
  for (int i = 0; i < k; ++i) {
    if (out->hit[i]) continue;
    miss_i.push_back(i);
    lay.push_back(layer);
    exp.push_back(ids[i]);
    dst.push_back(h->staging + int64_t(dst.size()) * h->store->stride());
  }
  int fail_chunk = 0;
  if (!miss_i.empty() && h->inj.read_fail_in > 0 && --h->inj.read_fail_in == 0) fail_chunk = 1;
  std::vector<int> failed;
  h->store->read(lay, exp, dst, &failed, fail_chunk);
  moe_status result = MOE_OK;
  SlotTable& t = h->tables[layer];
  for (size_t j = 0; j < miss_i.size(); ++j) {
    const int i = miss_i[j];
    if (failed[j]) {
      t.clear_slot(out->slot[i]);
      result = fail(h, MOE_ERR_IO, "reading expert %d of layer %d from the store failed", ids[i],
                    layer);
      continue;
    }
    const cudaError_t e = cudaMemcpyAsync(slots + int64_t(out->slot[i]) * h->blob, dst[j], h->blob,
                                          cudaMemcpyHostToDevice, h->side);
    if (e != cudaSuccess) {
      t.clear_slot(out->slot[i]);
      result = fail(h, MOE_ERR_CUDA, "expert copy: %s", cudaGetErrorString(e));
    }
  }
  CUDA_TRY(h, cudaEventRecord(h->copy_done[layer], h->side));
  CUDA_TRY(h, cudaEventRecord(h->staging_free, h->side));
  return result;
}

// cuTensorMapEncodeTiled, fetched from the driver at run time (the library
// does not link against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// A byte tensor of `rank` 2 or 3: rows of `row_bytes` (pitch `row_bytes`),
// `rows` rows, and for rank 3 `planes` planes `plane_bytes` apart.
// fp16 rows [rows][cols] (pitch `pitch` columns, default cols): box 64
// columns x box_rows rows, 128-byte swizzle (the UMMA K-major operand layout).
bool make_act_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                  uint32_t box_rows = kUnitTokens, uint64_t pitch = 0) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {(pitch ? pitch : cols) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_qrow_map(CUtensorMap* m, const void* base, int rank, uint64_t row_bytes, uint64_t rows,
                   uint64_t planes, uint64_t plane_bytes, uint32_t box_x, bool swizzle) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[3] = {row_bytes, rows, planes};
  const cuuint64_t strides[2] = {row_bytes, plane_bytes};
  const cuuint32_t box[3] = {box_x, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

DecodeParams params_for(moe_handle* h, int layer0, int n_layers, const void* x, void* y, int phases,
                        int flags) {
  DecodeParams p = h->base;
  p.layer0 = layer0;
  p.n_layers = n_layers;
  p.phases = phases;
  p.residual = (flags & MOE_FWD_RESIDUAL) ? 1 : 0;
  p.prenorm = (flags & MOE_FWD_PRENORM) ? 1 : 0;
  p.x_in = static_cast<const uint16_t*>(x);
  p.y_out = static_cast<uint16_t*>(y);
  p.trace = h->trace_on ? h->trace : nullptr;
  return p;
}

}  // namespace

namespace moe {

int stack_launch_params(moe_handle* h, const void* x, void* y, int n_layers, DecodeParams* p,
                        int* grid, int* device) {
  if (!h || !x || !y || x == y || !p || !grid || !device) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return fail(h, MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (h->cfg.n_slots > 0) return fail(h, MOE_ERR_STATE, "the decode stack needs resident mode");
  if (n_layers < 1 || n_layers > h->cfg.n_layers) return fail(h, MOE_ERR_INVALID_ARG, "bad n_layers");
  *p = params_for(h, 0, n_layers, x, y, PH_ALL, MOE_FWD_RESIDUAL | MOE_FWD_PRENORM);
  if (h->inj.stall_ms > 0) {  // a pending injected stall applies to this launch
    p->stall_first_barrier = 1;
    p->timeout_ns = uint64_t(h->inj.stall_ms) * 1000000ull;
    h->inj.stall_ms = 0;
  }
  *grid = h->grid;
  *device = h->device;
  return MOE_OK;
}

int handle_error(moe_handle* h, int status, const char* msg) {
  return fail(h, static_cast<moe_status>(status), "%s", msg);
}

int set_smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> bytes set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[std::make_pair(kernel, dev)];
  if (bytes <= have) return 0;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return static_cast<int>(e);
  have = bytes;
  return 0;
}

}  // namespace moe

#pragma GCC visibility push(default)
extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_OOM: return "out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "timeout";
    case MOE_ERR_INJECTED: return "injected fault";
    case MOE_ERR_STATE: return "invalid state";
    case MOE_ERR_DEVICE: return "device-reported error";
    case MOE_ERR_IO: return "expert store I/O error";
  }
  return "unknown status";
}

const char* moe_last_error(const moe_handle* h) { return h ? h->err.c_str() : g_create_error.c_str(); }

static bool config_ok(const moe_config& c) {
  return c.group == kGroup && c.d_model > 0 && c.d_model % 256 == 0 && c.d_expert > 0 &&
         c.d_expert % 64 == 0 && c.d_shared > 0 && c.d_shared % 64 == 0 && c.top_k >= 1 &&
         c.top_k <= kMaxTopK && c.n_experts >= c.top_k && c.n_experts <= 1024 &&
         c.n_experts % 16 == 0 && c.n_layers >= 1 && c.max_tokens >= 1 &&
         (c.n_slots == 0 || (c.n_slots >= c.top_k && c.n_slots <= c.n_experts)) &&
         (!c.expert_store || (c.n_slots > 0 && c.io_threads >= 1 && c.io_threads <= 256));
}

static bool experts_ok(const moe_config& c, const moe_layer_weights& w) {
  if (!w.exp_gate || !w.exp_up || !w.exp_down) return false;
  for (int e = 0; e < c.n_experts; ++e)
    if (!valid_qt(w.exp_gate[e]) || !valid_qt(w.exp_up[e]) || !valid_qt(w.exp_down[e]))
      return false;
  return true;
}

moe_status moe_store_write(const moe_config* cfg, const moe_layer_weights* layers, const char* path) {
  if (!cfg || !layers || !path) return fail(nullptr, MOE_ERR_INVALID_ARG, "cfg, layers or path is NULL");
  moe_config c = *cfg;
  c.expert_store = nullptr;  // the file is being written, not read
  if (!config_ok(c)) return fail(nullptr, MOE_ERR_INVALID_ARG, "unsupported configuration");
  for (int l = 0; l < c.n_layers; ++l)
    if (!experts_ok(c, layers[l]))
      return fail(nullptr, MOE_ERR_INVALID_ARG, "layer %d: missing expert weights", l);
  const Dims d{c.d_model, c.n_experts, c.d_expert, c.top_k, c.d_shared};
  std::string err;
  if (store_write(d, c.n_layers, layers, path, &err) != 0)
    return fail(nullptr, MOE_ERR_IO, "%s", err.c_str());
  return MOE_OK;
}

moe_status moe_create(const moe_config* cfg, const moe_layer_weights* layers, moe_handle** out) {
  if (!out) return fail(nullptr, MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg || !layers) return fail(nullptr, MOE_ERR_INVALID_ARG, "cfg or layers is NULL");
  const moe_config& c = *cfg;
  if (!config_ok(c)) return fail(nullptr, MOE_ERR_INVALID_ARG, "unsupported configuration");
  const bool from_store = c.expert_store != nullptr;
  for (int l = 0; l < c.n_layers; ++l) {
    const moe_layer_weights& w = layers[l];
    if (!valid_qt(w.router) || !valid_qt(w.shared_gate) || !valid_qt(w.shared_up) ||
        !valid_qt(w.shared_down))
      return fail(nullptr, MOE_ERR_INVALID_ARG, "layer %d: missing weights", l);
    if (!from_store && !experts_ok(c, w))
      return fail(nullptr, MOE_ERR_INVALID_ARG, "layer %d: missing expert weights", l);
  }
  std::unique_ptr<moe_handle> h(new moe_handle());
  h->cfg = c;
  h->d = Dims{c.d_model, c.n_experts, c.d_expert, c.top_k, c.d_shared};
  const Dims& d = h->d;
  moe_status st;
#define CREATE_TRY(call)                                                                 \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess) {                                                            \
      st = fail(nullptr, e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA,  \
                "%s: %s", #call, cudaGetErrorString(e_));                               \
      free_all(h.get());                                                                \
      return st;                                                                        \
    }                                                                                   \
  } while (0)
#define CREATE_FAIL(code, msg)             \
  do {                                     \
    st = fail(nullptr, (code), "%s", msg); \
    free_all(h.get());                     \
    return st;                             \
  } while (0)
  CREATE_TRY(cudaGetDevice(&h->device));
  CREATE_TRY(cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
  int max_smem = 0;
  CREATE_TRY(cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device));
  int coop = 0;
  CREATE_TRY(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device));
  if (!coop) CREATE_FAIL(MOE_ERR_STATE, "device does not support cooperative launches");
  h->blob = expert_blob_bytes(d);
  h->fixed = (layer_fixed_bytes(d) + 255) / 256 * 256;
  const int L = c.n_layers;
  const bool streaming = c.n_slots > 0;
  const int64_t per_layer_experts = (streaming ? c.n_slots : c.n_experts) * h->blob;
  h->dev_weight_bytes = L * (h->fixed + per_layer_experts);
  CREATE_TRY(cudaMalloc(&h->dev_weights, h->dev_weight_bytes));
  if (streaming && from_store) {
    // the SSD tier: staging buffers for the misses of one step, page aligned
    // for direct I/O, and the file with its reader threads
    const int64_t stride = store_stride(h->blob);
    CREATE_TRY(cudaHostAlloc(&h->staging, int64_t(c.top_k) * stride, cudaHostAllocDefault));
    CREATE_TRY(cudaEventCreateWithFlags(&h->staging_free, cudaEventDisableTiming));
    const bool aligned = (reinterpret_cast<uintptr_t>(h->staging) % kStorePage) == 0;
    h->store.reset(new ExpertStore());
    std::string err;
    if (h->store->open(c.expert_store, d, L, h->blob, c.io_threads, aligned, &err) != 0) {
      st = fail(nullptr, err.find("match") != std::string::npos ? MOE_ERR_INVALID_ARG : MOE_ERR_IO,
                "%s", err.c_str());
      free_all(h.get());
      return st;
    }
  } else if (streaming) {
    h->pool_bytes = static_cast<int64_t>(L) * c.n_experts * h->blob;
    if (g_inject_pinned_fail) {
      g_inject_pinned_fail = 0;
      CREATE_FAIL(MOE_ERR_INJECTED, "injected pinned-pool allocation failure");
    }
    CREATE_TRY(cudaHostAlloc(&h->pool, h->pool_bytes, cudaHostAllocDefault));
  }
  // repack + upload, one layer at a time through a host staging buffer
  {
    std::vector<uint8_t> stage(h->fixed + (streaming ? 0 : per_layer_experts));
    for (int l = 0; l < L; ++l) {
      const moe_layer_weights& w = layers[l];
      repack_layer_fixed(d, w, stage.data());
      if (!from_store) {
        uint8_t* exp_dst = streaming ? h->pool + static_cast<int64_t>(l) * c.n_experts * h->blob
                                     : stage.data() + h->fixed;
        parallel_for(c.n_experts, [&](int64_t e) {
          repack_expert(d, w.exp_gate[e], w.exp_up[e], w.exp_down[e], exp_dst + e * h->blob);
        });
      }
      CREATE_TRY(cudaMemcpy(h->dev_weights + l * (h->fixed + per_layer_experts), stage.data(),
                            stage.size(), cudaMemcpyHostToDevice));
    }
  }
  h->layers.resize(L);
  for (int l = 0; l < L; ++l) {
    uint8_t* base = h->dev_weights + l * (h->fixed + per_layer_experts);
    LayerDev& ld = h->layers[l];
    ld.router_t = base;
    ld.router_sb = reinterpret_cast<const uint32_t*>(base + router_t_bytes(d));
    ld.logit_bias = layers[l].router_logit_bias
                        ? reinterpret_cast<const float*>(base + router_t_bytes(d) + router_sb_bytes(d))
                        : nullptr;
    ld.shared_gu = base + router_t_bytes(d) + router_sb_bytes(d) + bias_bytes(d);
    ld.shared_dn = ld.shared_gu + shared_gu_bytes(d);
    ld.experts = base + h->fixed;
    ld.slot_of = nullptr;
  }
  CREATE_TRY(cudaMalloc(&h->dev_layers, sizeof(LayerDev) * L));
  CREATE_TRY(cudaMemcpy(h->dev_layers, h->layers.data(), sizeof(LayerDev) * L, cudaMemcpyHostToDevice));
  // scratch
  const int G = h->num_sms;
  const int64_t T = c.max_tokens;
  auto al = [](int64_t b) { return (b + 255) / 256 * 256; };
  const int64_t sz_xbuf = al(2 * T * d.D * 2), sz_h = al(T * (d.K * d.I + d.S) * 4),
                sz_part = al(2 * d.E * 8), sz_ids = al(int64_t(L) * T * d.K * 4), sz_bar = 256,
                sz_io = al(T * d.D * 2), sz_trace = al(int64_t(G) * kTraceMaxLayers * kTraceEvents * 8);
  h->scratch_bytes = sz_xbuf + sz_h + sz_part + 2 * sz_ids + sz_bar + 2 * sz_io + sz_trace;
  CREATE_TRY(cudaMalloc(&h->scratch, h->scratch_bytes));
  CREATE_TRY(cudaMemset(h->scratch, 0, h->scratch_bytes));
  uint8_t* sp = h->scratch;
  h->xbuf = reinterpret_cast<uint16_t*>(sp);
  sp += sz_xbuf;
  h->h = reinterpret_cast<float*>(sp);
  sp += sz_h;
  h->lacc = reinterpret_cast<unsigned long long*>(sp);
  sp += sz_part;
  h->ids = reinterpret_cast<int32_t*>(sp);
  sp += sz_ids;
  h->wts = reinterpret_cast<float*>(sp);
  sp += sz_ids;
  h->bar = reinterpret_cast<uint32_t*>(sp);
  sp += sz_bar;
  h->io_x = reinterpret_cast<uint16_t*>(sp);
  sp += sz_io;
  h->io_y = reinterpret_cast<uint16_t*>(sp);
  sp += sz_io;
  h->trace = reinterpret_cast<uint64_t*>(sp);
  CREATE_TRY(cudaHostAlloc(&h->pin_x, T * d.D * 2, cudaHostAllocDefault));
  CREATE_TRY(cudaHostAlloc(&h->pin_y, T * d.D * 2, cudaHostAllocDefault));
  CREATE_TRY(cudaHostAlloc(&h->pin_ids, T * d.K * 4 + 64, cudaHostAllocDefault));
  CREATE_TRY(cudaHostAlloc(&h->pin_status, 64, cudaHostAllocDefault));
  CREATE_TRY(cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking));
  CREATE_TRY(cudaEventCreateWithFlags(&h->ev_ids, cudaEventDisableTiming));
  if (streaming) {
    h->tables.resize(L);
    h->layer_done.resize(L);
    h->copy_done.resize(L);
    for (int l = 0; l < L; ++l) {
      h->tables[l].init(c.n_slots, c.n_experts);
      CREATE_TRY(cudaEventCreateWithFlags(&h->layer_done[l], cudaEventDisableTiming));
      CREATE_TRY(cudaEventCreateWithFlags(&h->copy_done[l], cudaEventDisableTiming));
    }
  }
  // decode kernel parameters shared by every launch
  DecodeParams& p = h->base;
  p.layers = h->dev_layers;
  p.D = d.D;
  p.E = d.E;
  p.I = d.I;
  p.S = d.S;
  p.K = d.K;
  p.rbD = static_cast<int>(qrow_bytes(d.D));
  p.rbI = static_cast<int>(qrow_bytes(d.I));
  p.rbS = static_cast<int>(qrow_bytes(d.S));
  p.blob_bytes = h->blob;
  p.dn_off = d.I * 2 * qrow_bytes(d.D);
  p.xbuf = h->xbuf;
  p.h = reinterpret_cast<uint16_t*>(h->h);
  p.lacc = h->lacc;
  p.ids = h->ids;
  p.wts = h->wts;
  p.bar = h->bar;
  p.rms_eps = 1e-6f;
  // C phase: one (branch, 32-column chunk) task per consumer thread; rows per
  // C stage limited by the slot size (a C stage fits the B stage's slot).
  p.ntask = static_cast<int>(d.K * (d.I / 32) + d.S / 32);
  p.rc_max = static_cast<int>(std::max<int64_t>(
      1, (kPairsPerStage * 2 * qrow_bytes(d.D) - 2 * d.E * 4) /
             (d.K * qrow_bytes(d.I) + qrow_bytes(d.S) + d.E)));
  const int best_busy = p.ntask <= kConsumers ? 1 : -1;
  if (best_busy < 0)
    CREATE_FAIL(MOE_ERR_INVALID_ARG, "top_k * d_expert too large for the decode kernel");
  if (d.D > 32 * 32 * 3 || d.K * d.I + d.S > 4 * kConsumers * 8 || d.E > 4 * kConsumers)
    CREATE_FAIL(MOE_ERR_INVALID_ARG, "d_model or top_k * d_expert + d_shared too large for the decode kernel");
  if ((d.D + std::min<int64_t>(G, d.D) - 1) / std::min<int64_t>(G, d.D) > 256)
    CREATE_FAIL(MOE_ERR_INVALID_ARG, "too few SMs for d_model in the decode kernel");
  p.timeout_ns = 2000000000ull;
  if (decode_smem_plan(&p, max_smem) != 0)
    CREATE_FAIL(MOE_ERR_INVALID_ARG, "decode kernel does not fit in shared memory");
  // the first-layer router stage holds a whole CTA row slice
  const int64_t r_stage = int64_t((d.D + G - 1) / G) * d.E + 2 * d.E * 4;
  if (r_stage > p.slot_bytes) CREATE_FAIL(MOE_ERR_INVALID_ARG, "router stage too large for the SM count");
  h->grid = G < d.D ? G : static_cast<int>(d.D);  // every CTA owns at least one output row
  // ---- prefill (T >= 2): tensor maps over the resident weights and scratch
  if (!streaming && c.max_tokens >= 2 && d.E <= kMaxPrefillExperts) {
    h->mt_gu_r = static_cast<int>(2 * d.I / 128);
    h->mt_dn = static_cast<int>(d.D / 128);
    h->mt_gu_s = static_cast<int>(2 * d.S / 128);
    h->maps.resize(L);
    const int64_t rbD = qrow_bytes(d.D), rbI = qrow_bytes(d.I), rbS = qrow_bytes(d.S);
    bool ok = (2 * d.I) % 128 == 0 && d.D % 128 == 0 && (2 * d.S) % 128 == 0;
    for (int l = 0; l < L && ok; ++l) {
      const LayerDev& ld = h->layers[l];
      auto& mp = h->maps[l];
      const uint8_t* dn = ld.experts + d.I * 2 * rbD;
      ok = ok && make_qrow_map(&mp.gu_code[0], ld.experts, 3, rbD, 2 * d.I, d.E, h->blob, 128, true);
      ok = ok && make_qrow_map(&mp.gu_sb[0], ld.experts, 3, rbD, 2 * d.I, d.E, h->blob, 16, false);
      ok = ok && make_qrow_map(&mp.dn_code[0], dn, 3, rbI, d.D, d.E, h->blob, 128, true);
      ok = ok && make_qrow_map(&mp.dn_sb[0], dn, 3, rbI, d.D, d.E, h->blob, 16, false);
      ok = ok && make_qrow_map(&mp.gu_code[1], ld.shared_gu, 2, rbD, 2 * d.S, 1, 0, 128, true);
      ok = ok && make_qrow_map(&mp.gu_sb[1], ld.shared_gu, 2, rbD, 2 * d.S, 1, 0, 16, false);
      ok = ok && make_qrow_map(&mp.dn_code[1], ld.shared_dn, 2, rbS, d.D, 1, 0, 128, true);
      ok = ok && make_qrow_map(&mp.dn_sb[1], ld.shared_dn, 2, rbS, d.D, 1, 0, 16, false);
    }
    if (!ok) CREATE_FAIL(MOE_ERR_CUDA, "could not encode the prefill tensor maps");
    const int64_t Tm = c.max_tokens, K = d.K, E = d.E;
    int64_t part = 0;
    for (int64_t t = 2; t <= Tm; ++t) {
      const int64_t v = int64_t(router_tc_splits(int(t), int(E), int(d.D), G)) * t * E;
      if (v > part) part = v;
    }
    const int64_t nt = Tm * K / kUnitTokens + E + 1, stl = (Tm + kUnitTokens - 1) / kUnitTokens;
    auto groups = [](int64_t tiles) { return (tiles + kTilesPerUnit - 1) / kTilesPerUnit; };
    const int64_t ngu = nt * groups(h->mt_gu_r) + stl * groups(h->mt_gu_s),
                  ndn = (nt + stl) * groups(h->mt_dn);
    const int64_t Dx = d.D + kGsumCols;  // x16 pitch: D columns, then the group sums
    int64_t sizes[] = {Tm * Dx * 2,        Tm * 4,          Tm * 4,        Tm * 4,        part * 4,
                       L * Tm * K * 4,    L * Tm * K * 4,  Tm * K * 4,    E * 4,
                       (E + 1) * 4,       Tm * K * 4,      Tm * K * 4,    ngu * int64_t(sizeof(GemmUnit)),
                       ndn * int64_t(sizeof(GemmUnit)), 16, Tm * K * d.I * 2, Tm * d.S * 2,
                       Tm * K * d.D * 2,  Tm * d.D * 4,    Tm * d.D * 2,  Tm * d.D * 2,
                       Tm * K * Dx * 2,   int64_t(bucket_blocks(int(Tm * K))) * 8 * E * 4};
    const int ns = sizeof(sizes) / sizeof(sizes[0]);
    int64_t offs[32];
    int64_t tot = 0;
    for (int i = 0; i < ns; ++i) {
      offs[i] = tot;
      tot += al(sizes[i]);
    }
    CREATE_TRY(cudaMalloc(&h->pf, tot));
    CREATE_TRY(cudaMemset(h->pf, 0, tot));
    h->pf_bytes = tot;
    int i = 0;
    h->pf_x16 = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_sigma = reinterpret_cast<float*>(h->pf + offs[i++]);
    h->pf_rscale = reinterpret_cast<float*>(h->pf + offs[i++]);
    h->pf_hscale = reinterpret_cast<float*>(h->pf + offs[i++]);
    h->pf_partials = reinterpret_cast<float*>(h->pf + offs[i++]);
    h->pf_ids = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_wts = reinterpret_cast<float*>(h->pf + offs[i++]);
    h->pf_forced = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_counts = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_offsets = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_perm = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_inv = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_units_gu = reinterpret_cast<GemmUnit*>(h->pf + offs[i++]);
    h->pf_units_dn = reinterpret_cast<GemmUnit*>(h->pf + offs[i++]);
    h->pf_nunits = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    h->pf_hr = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_hs = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_e = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_s = reinterpret_cast<float*>(h->pf + offs[i++]);
    h->pf_xs[0] = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_xs[1] = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_xperm = reinterpret_cast<uint16_t*>(h->pf + offs[i++]);
    h->pf_hist = reinterpret_cast<int32_t*>(h->pf + offs[i++]);
    bool mok = make_act_map(&h->bmap_rt, h->pf_x16, d.D, Tm, 128, Dx);
    for (int b = 0; b < kNBox && mok; ++b) {
      const uint32_t r = box_rows(b);
      mok = make_act_map(&h->bmap_gu[0][b], h->pf_xperm, Dx, Tm * K, r) &&
            make_act_map(&h->bmap_gu[1][b], h->pf_x16, Dx, Tm, r) &&
            make_act_map(&h->bmap_dn[0][b], h->pf_hr, d.I, Tm * K, r) &&
            make_act_map(&h->bmap_dn[1][b], h->pf_hs, d.S, Tm, r);
    }
    if (!mok) CREATE_FAIL(MOE_ERR_CUDA, "could not encode the prefill activation tensor maps");
    // Router weights for the tensor-core router GEMM: w = s q + b (fp32, one
    // rounding) split into fp16(w) and fp16(w - fp16(w)); rows E..Epad-1 zero.
    {
      const int64_t Epad = (E + 127) / 128 * 128, ng = d.D / 64;
      const int64_t per = 2 * Epad * d.D;
      std::vector<__half> rw(static_cast<size_t>(per));
      CREATE_TRY(cudaMalloc(&h->pf_rw, per * 2 * L));
      for (int l = 0; l < L; ++l) {
        const moe_qtensor& r = layers[l].router;
        std::fill(rw.begin(), rw.end(), __float2half_rn(0.f));
        parallel_for(E, [&](int64_t e) {
          for (int64_t c = 0; c < d.D; ++c) {
            __half_raw sr, br;
            sr.x = r.scale[e * ng + c / 64];
            br.x = r.bias[e * ng + c / 64];
            const float w = std::fma(__half2float(__half(sr)), static_cast<float>(r.q[e * d.D + c]),
                                     __half2float(__half(br)));
            const __half hi = __float2half_rn(w);
            rw[static_cast<size_t>(e * d.D + c)] = hi;
            rw[static_cast<size_t>((Epad + e) * d.D + c)] = __float2half_rn(w - __half2float(hi));
          }
        });
        uint16_t* dst = h->pf_rw + int64_t(l) * per;
        CREATE_TRY(cudaMemcpy(dst, rw.data(), per * 2, cudaMemcpyHostToDevice));
        if (!make_act_map(&h->maps[l].rt, dst, d.D, 2 * Epad, 128))
          CREATE_FAIL(MOE_ERR_CUDA, "could not encode the router tensor map");
      }
    }
    h->prefill_ok = true;
    h->pf_ev.resize(6 * kPhaseTimedCalls);
    for (auto& ev : h->pf_ev) CREATE_TRY(cudaEventCreate(&ev));
  }
  *out = h.release();
  return MOE_OK;
#undef CREATE_TRY
#undef CREATE_FAIL
}

void moe_destroy(moe_handle* h) {
  if (!h) return;
  free_all(h);
  delete h;
}

moe_status moe_get_info(const moe_handle* h, moe_info* out) {
  if (!h || !out) return MOE_ERR_INVALID_ARG;
  out->device_weight_bytes = h->dev_weight_bytes;
  out->pinned_pool_bytes = h->pool_bytes;
  out->device_scratch_bytes = h->scratch_bytes + h->pf_bytes;
  out->expert_blob_bytes = h->blob;
  out->num_sms = h->grid;
  out->store_direct_io = h->store && h->store->direct() ? 1 : 0;
  out->io_threads = h->store ? h->store->threads() : 0;
  return MOE_OK;
}

moe_status moe_set_timeout_ms(moe_handle* h, int ms) {
  if (!h || ms <= 0) return MOE_ERR_INVALID_ARG;
  h->timeout_ms = ms;
  return MOE_OK;
}

moe_status moe_debug_inject(moe_handle* h, int what, int arg) {
  switch (what) {
    case MOE_INJECT_NONE:
      g_inject_pinned_fail = 0;
      if (h) h->inj = Inject{};
      return MOE_OK;
    case MOE_INJECT_PINNED_ALLOC_FAIL:
      g_inject_pinned_fail = 1;
      return MOE_OK;
    case MOE_INJECT_H2D_FAIL:
      if (!h || arg < 1) return MOE_ERR_INVALID_ARG;
      h->inj.h2d_fail_in = arg;
      return MOE_OK;
    case MOE_INJECT_SLOW_COPY:
      if (!h || arg < 0) return MOE_ERR_INVALID_ARG;
      h->inj.slow_copy_ms = arg;
      return MOE_OK;
    case MOE_INJECT_DEVICE_STALL:
      if (!h || arg < 1 || arg > 2000) return MOE_ERR_INVALID_ARG;
      h->inj.stall_ms = arg;
      return MOE_OK;
    case MOE_INJECT_READ_FAIL:
      if (!h || arg < 1) return MOE_ERR_INVALID_ARG;
      h->inj.read_fail_in = arg;
      return MOE_OK;
    case MOE_INJECT_GEMM_STALL:
      if (!h || arg < 1 || arg > 2000) return MOE_ERR_INVALID_ARG;
      h->inj.gemm_stall_ms = arg;
      return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_slot_plan_create(int n_slots, int n_experts, moe_slot_plan** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_slots < 1 || n_experts < 1 || n_slots > n_experts) return MOE_ERR_INVALID_ARG;
  moe_slot_plan* p = new moe_slot_plan();
  p->t.init(n_slots, n_experts);
  *out = p;
  return MOE_OK;
}

moe_status moe_slot_plan_step(moe_slot_plan* p, const int32_t* ids, int k, moe_cache_result* out) {
  if (!p || !ids || !out || k < 1 || k > 64) return MOE_ERR_INVALID_ARG;
  const int m = p->t.plan(ids, k, out->hit, out->slot, out->evicted);
  if (m < 0) return MOE_ERR_INVALID_ARG;
  out->misses = m;
  return MOE_OK;
}

void moe_slot_plan_destroy(moe_slot_plan* p) { delete p; }

moe_status moe_cache_step(moe_handle* h, int layer, const int32_t* ids, int k, int flags,
                          moe_cache_result* out) {
  if (!h || !ids || !out || k < 1 || k > 64) return MOE_ERR_INVALID_ARG;
  if (h->cfg.n_slots == 0) return fail(h, MOE_ERR_STATE, "moe_cache_step needs streaming mode");
  if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, MOE_ERR_INVALID_ARG, "bad layer");
  SlotTable& t = h->tables[layer];
  const int m = t.plan(ids, k, out->hit, out->slot, out->evicted);
  if (m < 0)
    return fail(h, MOE_ERR_INVALID_ARG, "ids must be %d distinct values in [0, %d)", k,
                h->cfg.n_experts);
  out->misses = m;
  if (flags & MOE_PLAN_ONLY) return MOE_OK;
  // the slots being refilled may still be read by this layer's previous kernels
  CUDA_TRY(h, cudaStreamWaitEvent(h->side, h->layer_done[layer], 0));
  uint8_t* slots =
      h->dev_weights + layer * (h->fixed + int64_t(h->cfg.n_slots) * h->blob) + h->fixed;
  if (h->store) return cache_fill_from_store(h, layer, ids, k, out, slots);
  const uint8_t* pool = h->pool + int64_t(layer) * h->cfg.n_experts * h->blob;
  moe_status result = MOE_OK;
  for (int i = 0; i < k; ++i) {
    if (out->hit[i]) continue;
    if (h->inj.slow_copy_ms)
      std::this_thread::sleep_for(std::chrono::milliseconds(h->inj.slow_copy_ms));
    if (h->inj.h2d_fail_in > 0 && --h->inj.h2d_fail_in == 0) {
      t.clear_slot(out->slot[i]);
      result = fail(h, MOE_ERR_INJECTED, "injected failure of the host->HBM copy of expert %d", ids[i]);
      continue;
    }
    cudaError_t e = cudaMemcpyAsync(slots + int64_t(out->slot[i]) * h->blob,
                                    pool + int64_t(ids[i]) * h->blob, h->blob,
                                    cudaMemcpyHostToDevice, h->side);
    if (e != cudaSuccess) {
      t.clear_slot(out->slot[i]);
      result = fail(h, MOE_ERR_CUDA, "expert copy: %s", cudaGetErrorString(e));
    }
  }
  CUDA_TRY(h, cudaEventRecord(h->copy_done[layer], h->side));
  return result;
}

moe_status moe_last_buckets(moe_handle* h, int32_t* counts, int32_t* offsets, int32_t* perm) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (!h->last_prefill || h->last_T < 2)
    return fail(h, MOE_ERR_STATE, "moe_last_buckets: the last call was not a multi-token call");
  moe_status st = check_device_status(h, nullptr);
  if (st != MOE_OK) return st;
  const int64_t E = h->d.E, n = int64_t(h->last_T) * h->d.K;
  if (counts) CUDA_TRY(h, cudaMemcpy(counts, h->pf_counts, E * 4, cudaMemcpyDeviceToHost));
  if (offsets) CUDA_TRY(h, cudaMemcpy(offsets, h->pf_offsets, (E + 1) * 4, cudaMemcpyDeviceToHost));
  if (perm) CUDA_TRY(h, cudaMemcpy(perm, h->pf_perm, n * 4, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_trace_enable(moe_handle* h, int on) {
  if (!h) return MOE_ERR_INVALID_ARG;
  h->trace_on = on != 0;
  return MOE_OK;
}

moe_status moe_trace_read(moe_handle* h, int64_t* out, int n_layers) {
  if (!h || !out || n_layers < 1 || n_layers > kTraceMaxLayers) return MOE_ERR_INVALID_ARG;
  CUDA_TRY(h, cudaDeviceSynchronize());
  CUDA_TRY(h, cudaMemcpy(out, h->trace, size_t(h->grid) * n_layers * kTraceEvents * 8,
                         cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_prefill_phase_ms(moe_handle* h, float* ms, int* calls) {
  if (!h || !ms) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i) ms[i] = 0.f;
  if (calls) *calls = h->pf_ev_calls;
  if (h->pf_ev_calls == 0) return MOE_OK;
  CUDA_TRY(h, cudaEventSynchronize(h->pf_ev[6 * h->pf_ev_calls - 1]));
  for (int c = 0; c < h->pf_ev_calls; ++c)
    for (int i = 0; i < 5; ++i) {
      float t = 0.f;
      CUDA_TRY(h, cudaEventElapsedTime(&t, h->pf_ev[6 * c + i], h->pf_ev[6 * c + i + 1]));
      ms[i] += t;
    }
  h->pf_ev_calls = 0;
  return MOE_OK;
}

moe_status moe_cache_reset(moe_handle* h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (h->cfg.n_slots == 0) return fail(h, MOE_ERR_STATE, "moe_cache_reset needs streaming mode");
  for (auto& t : h->tables) t.reset();
  return MOE_OK;
}

}  // extern "C"

// One layer for T >= 2 tokens, resident mode: route, bucket, grouped GEMMs on
// the tensor cores, combine.  Everything is enqueued on s; ids and weights of
// the layer land in pf_ids / pf_wts block `slot` ([T][K]).
static moe_status prefill_layer(moe_handle* h, int layer, const void* x, int T, void* y, int flags,
                                const int32_t* forced, cudaStream_t s, int slot) {
  const Dims& d = h->d;
  const int K = static_cast<int>(d.K);
  const int64_t Tm = h->cfg.max_tokens;
  int32_t* ids = h->pf_ids + int64_t(slot) * Tm * K;
  float* wts = h->pf_wts + int64_t(slot) * Tm * K;
  if (forced)
    CUDA_TRY(h, cudaMemcpyAsync(h->pf_forced, forced, sizeof(int32_t) * T * K,
                                cudaMemcpyHostToDevice, s));
  cudaEvent_t* ev = nullptr;  // phase events of this call (tracing only)
  if (h->trace_on && h->pf_ev_calls < kPhaseTimedCalls) ev = &h->pf_ev[6 * h->pf_ev_calls++];
  if (ev) CUDA_TRY(h, cudaEventRecord(ev[0], s));
  const LayerDev& ld = h->layers[layer];
  RouteArgs ra{};
  ra.x = static_cast<const uint16_t*>(x);
  ra.T = T;
  ra.D = static_cast<int>(d.D);
  ra.E = static_cast<int>(d.E);
  ra.K = K;
  ra.prenorm = (flags & MOE_FWD_PRENORM) ? 1 : 0;
  ra.rms_eps = h->base.rms_eps;
  ra.wmap = &h->maps[layer].rt;
  ra.xmap = &h->bmap_rt;
  ra.logit_bias = ld.logit_bias;
  ra.forced = forced ? h->pf_forced : nullptr;
  ra.x16 = h->pf_x16;
  ra.sigma = h->pf_sigma;
  ra.rscale = h->pf_rscale;
  ra.hscale = h->pf_hscale;
  ra.partials = h->pf_partials;
  ra.nsplit = router_tc_splits(T, ra.E, ra.D, h->num_sms);
  ra.status = h->bar + 2;
  ra.timeout_ns = h->base.timeout_ns;
  ra.ids = ids;
  ra.wts = wts;
  int e = prefill_route(ra, s);
  if (e) return fail(h, MOE_ERR_CUDA, "prefill router: %s", cudaGetErrorString(cudaError_t(e)));
  if (ev) CUDA_TRY(h, cudaEventRecord(ev[1], s));
  BucketArgs ba{};
  ba.ids = ids;
  ba.T = T;
  ba.K = K;
  ba.E = ra.E;
  ba.mt_gu_r = h->mt_gu_r;
  ba.mt_dn = h->mt_dn;
  ba.mt_gu_s = h->mt_gu_s;
  ba.counts = h->pf_counts;
  ba.offsets = h->pf_offsets;
  ba.perm = h->pf_perm;
  ba.inv = h->pf_inv;
  ba.units_gu = h->pf_units_gu;
  ba.units_dn = h->pf_units_dn;
  ba.n_units = h->pf_nunits;
  ba.hist = h->pf_hist;
  ba.status = h->bar + 2;
  e = prefill_bucket(ba, s);
  if (e) return fail(h, MOE_ERR_CUDA, "prefill bucketing: %s", cudaGetErrorString(cudaError_t(e)));
  if (ev) CUDA_TRY(h, cudaEventRecord(ev[2], s));
  const auto& mp = h->maps[layer];
  GemmParams gp{};
  gp.perm = h->pf_perm;
  gp.topk = K;
  gp.sigma = h->pf_sigma;
  gp.hscale = h->pf_hscale;
  gp.wts = wts;
  gp.D = static_cast<int>(d.D);
  gp.status = h->bar + 2;
  gp.timeout_ns = h->base.timeout_ns;
  // gate/up (+ GELU): routed rows in bucket order, shared rows by token
  gp.tm_code[0] = mp.gu_code[0];
  gp.tm_code[1] = mp.gu_code[1];
  gp.tm_sb[0] = mp.gu_sb[0];
  gp.tm_sb[1] = mp.gu_sb[1];
  e = gather_rows_launch(h->pf_x16, static_cast<int>(d.D) + kGsumCols, h->pf_perm, K, T * K,
                         h->pf_xperm, s);
  if (e) return fail(h, MOE_ERR_CUDA, "row gather: %s", cudaGetErrorString(cudaError_t(e)));
  gp.units = h->pf_units_gu;
  gp.n_units = h->pf_nunits;
  gp.mode = 0;
  gp.gsum = 1;
  gp.K[0] = gp.K[1] = static_cast<int>(d.D);
  std::memcpy(gp.tm_b, h->bmap_gu, sizeof gp.tm_b);
  gp.hout[0] = h->pf_hr;
  gp.hout[1] = h->pf_hs;
  gp.hld[0] = static_cast<int>(d.I);
  gp.hld[1] = static_cast<int>(d.S);
  if (h->inj.gemm_stall_ms > 0) {  // injected: a wait that nothing completes, a short limit
    gp.stall = 1;
    gp.timeout_ns = uint64_t(h->inj.gemm_stall_ms) * 1000000ull;
    h->inj.gemm_stall_ms = 0;
  }
  e = gemm_tc_launch(gp, h->num_sms, T, s);
  gp.stall = 0;
  gp.timeout_ns = h->base.timeout_ns;
  if (e) return fail(h, MOE_ERR_CUDA, "gate/up GEMM launch: %s", cudaGetErrorString(cudaError_t(e)));
  if (ev) CUDA_TRY(h, cudaEventRecord(ev[3], s));
  // down: routed output weighted by the routing weight (bf16), shared (fp32)
  gp.tm_code[0] = mp.dn_code[0];
  gp.tm_code[1] = mp.dn_code[1];
  gp.tm_sb[0] = mp.dn_sb[0];
  gp.tm_sb[1] = mp.dn_sb[1];
  gp.units = h->pf_units_dn;
  gp.n_units = h->pf_nunits + 1;
  gp.mode = 1;
  gp.gsum = 0;
  gp.K[0] = static_cast<int>(d.I);
  gp.K[1] = static_cast<int>(d.S);
  std::memcpy(gp.tm_b, h->bmap_dn, sizeof gp.tm_b);
  gp.eout = h->pf_e;
  gp.sout = h->pf_s;
  e = gemm_tc_launch(gp, h->num_sms, T, s);
  if (e) return fail(h, MOE_ERR_CUDA, "down GEMM launch: %s", cudaGetErrorString(cudaError_t(e)));
  if (ev) CUDA_TRY(h, cudaEventRecord(ev[4], s));
  CombineArgs ca{};
  ca.x = static_cast<const uint16_t*>(x);
  ca.e = h->pf_e;
  ca.s = h->pf_s;
  ca.inv = h->pf_inv;
  ca.y = static_cast<uint16_t*>(y);
  ca.T = T;
  ca.D = static_cast<int>(d.D);
  ca.K = K;
  ca.residual = (flags & MOE_FWD_RESIDUAL) ? 1 : 0;
  e = prefill_combine(ca, s);
  if (e) return fail(h, MOE_ERR_CUDA, "combine: %s", cudaGetErrorString(cudaError_t(e)));
  if (ev) CUDA_TRY(h, cudaEventRecord(ev[5], s));
  return MOE_OK;
}

static moe_status decode_layer_streaming(moe_handle* h, int layer, const void* x, void* y,
                                         int flags, const int32_t* forced, cudaStream_t s,
                                         moe_layer_stats* stats) {
  const int K = h->cfg.top_k;
  DecodeParams p1 = params_for(h, layer, 1, x, y, 0, flags);
  int32_t ids[kMaxTopK];
  moe_cache_result cr;
  moe_status st;
  // The first launch adds the layer's router logits into the accumulators,
  // and only the second one (the owner of the output rows) clears them.  If
  // the step stops in between, clear them here so the next step starts from
  // zero.
  auto abandon = [&](moe_status why) {
    cudaMemsetAsync(h->lacc, 0, 2 * h->d.E * 8, s);
    return why;
  };
  if (forced) {
    // ids known up front: the router and the shared expert go to the GPU
    // first, then the misses are fetched (read from the store on the host,
    // copied on the side stream) while they run
    std::memcpy(ids, forced, sizeof(int32_t) * K);
    p1.phases = PH_ROUTER | PH_BSHARED;
    p1.forced = 1;
    std::memcpy(p1.forced_ids, ids, sizeof(int32_t) * K);
    st = launch(h, p1, s);
    if (st != MOE_OK) return abandon(st);
    st = moe_cache_step(h, layer, ids, K, 0, &cr);
    if (st != MOE_OK) return abandon(st);
  } else {
    p1.phases = PH_ROUTER;
    st = launch(h, p1, s);
    if (st != MOE_OK) return abandon(st);
    CUDA_TRY(h, cudaMemcpyAsync(h->pin_ids, h->ids, sizeof(int32_t) * K, cudaMemcpyDeviceToHost, s));
    CUDA_TRY(h, cudaEventRecord(h->ev_ids, s));
    p1.phases = PH_BSHARED;  // shared expert runs while the host plans and copies
    st = launch(h, p1, s);
    if (st != MOE_OK) return abandon(st);
    st = wait_event(h, h->ev_ids);
    if (st != MOE_OK) return abandon(st);
    std::memcpy(ids, h->pin_ids, sizeof(int32_t) * K);
    st = moe_cache_step(h, layer, ids, K, 0, &cr);
    if (st != MOE_OK) return abandon(st);
  }
  CUDA_TRY(h, cudaStreamWaitEvent(s, h->copy_done[layer], 0));
  DecodeParams p2 = params_for(h, layer, 1, x, y, PH_BROUTED | PH_C, flags);
  p2.use_slots = 1;
  for (int i = 0; i < K; ++i) p2.slots[i] = cr.slot[i];
  st = launch(h, p2, s);
  if (st != MOE_OK) return abandon(st);
  CUDA_TRY(h, cudaEventRecord(h->layer_done[layer], s));
  if (stats) {
    stats->hits = K - cr.misses;
    stats->misses = cr.misses;
    stats->bytes_h2d = int64_t(cr.misses) * h->blob;
    if (stats->cache) *stats->cache = cr;
  }
  return MOE_OK;
}

extern "C" {

moe_status moe_layer_forward(moe_handle* h, int layer, const void* x, int T, void* y, int flags,
                             const int32_t* forced_ids, void* stream, moe_layer_stats* stats) {
  if (!h || !x || !y || x == y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return fail(h, MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, MOE_ERR_INVALID_ARG, "bad layer %d", layer);
  if (T < 1 || T > h->cfg.max_tokens) return fail(h, MOE_ERR_INVALID_ARG, "T=%d out of range", T);
  const int K = h->cfg.top_k, D = h->cfg.d_model;
  if (forced_ids) {
    for (int t = 0; t < T; ++t)
      for (int i = 0; i < K; ++i) {
        const int v = forced_ids[t * K + i];
        if (v < 0 || v >= h->cfg.n_experts) return fail(h, MOE_ERR_INVALID_ARG, "forced id out of range");
        for (int j = 0; j < i; ++j)
          if (forced_ids[t * K + j] == v) return fail(h, MOE_ERR_INVALID_ARG, "forced ids repeat");
      }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (stats) {
    stats->hits = stats->misses = 0;
    stats->bytes_h2d = 0;
  }
  if (h->cfg.n_slots > 0) {
    if (T != 1) return fail(h, MOE_ERR_STATE, "streaming mode runs one token per call");
    moe_status st = decode_layer_streaming(h, layer, x, y, flags, forced_ids, s, stats);
    if (st != MOE_OK) return st;
  } else if (T >= 2 && h->prefill_ok) {
    moe_status st = prefill_layer(h, layer, x, T, y, flags, forced_ids, s, 0);
    if (st != MOE_OK) return st;
    h->last_T = T;
    h->last_layers = 1;
    h->last_prefill = true;
    if (stats && (stats->ids || stats->weights)) {
      st = check_device_status(h, s);
      if (st != MOE_OK) return st;
      if (stats->ids)
        CUDA_TRY(h, cudaMemcpy(stats->ids, h->pf_ids, sizeof(int32_t) * T * K, cudaMemcpyDeviceToHost));
      if (stats->weights)
        CUDA_TRY(h, cudaMemcpy(stats->weights, h->pf_wts, sizeof(float) * T * K, cudaMemcpyDeviceToHost));
    }
    return MOE_OK;
  } else {
    // resident: one persistent launch per token
    for (int t = 0; t < T; ++t) {
      DecodeParams p = params_for(h, layer, 1, static_cast<const uint16_t*>(x) + int64_t(t) * D,
                                  static_cast<uint16_t*>(y) + int64_t(t) * D, PH_ALL, flags);
      p.ids = h->ids + int64_t(t) * K;
      p.wts = h->wts + int64_t(t) * K;
      if (forced_ids) {
        p.forced = 1;
        std::memcpy(p.forced_ids, forced_ids + t * K, sizeof(int32_t) * K);
      }
      moe_status st = launch(h, p, s);
      if (st != MOE_OK) return st;
    }
  }
  h->last_T = T;
  h->last_layers = 1;
  h->last_prefill = false;
  if (stats && (stats->ids || stats->weights)) {
    moe_status st = check_device_status(h, s);
    if (st != MOE_OK) return st;
    if (stats->ids)
      CUDA_TRY(h, cudaMemcpy(stats->ids, h->ids, sizeof(int32_t) * T * K, cudaMemcpyDeviceToHost));
    if (stats->weights)
      CUDA_TRY(h, cudaMemcpy(stats->weights, h->wts, sizeof(float) * T * K, cudaMemcpyDeviceToHost));
  }
  return MOE_OK;
}

// Fewer tokens than this run the stack as one single-token decode launch per
// token.  Measured on the 30-layer Gemma-shape stack (single-token launches
// at 0.60 ms a token against the multi-token path): 4 tokens 2.40 against
// 2.60 ms, 5 tokens 3.00 against 2.78 ms, 8 tokens 4.81 against 3.57 ms.
// Below 5 tokens the multi-token path's per-layer fixed cost (eight
// launches) outweighs reading each chosen expert once for all its rows.
constexpr int kStackBatchMin = 5;

moe_status moe_forward_stack(moe_handle* h, const void* x, int T, void* y, int n_layers,
                             void* stream) {
  if (!h || !x || !y || x == y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return fail(h, MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (h->cfg.n_slots > 0) return fail(h, MOE_ERR_STATE, "moe_forward_stack needs resident mode");
  if (n_layers < 1 || n_layers > h->cfg.n_layers) return fail(h, MOE_ERR_INVALID_ARG, "bad n_layers");
  if (T < 1 || T > h->cfg.max_tokens) return fail(h, MOE_ERR_INVALID_ARG, "T=%d out of range", T);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = h->cfg.d_model, K = h->cfg.top_k;
  if (T >= kStackBatchMin && h->prefill_ok) {
    // layer by layer over all T tokens through the tensor-core path
    for (int l = 0; l < n_layers; ++l) {
      const void* xin = l == 0 ? x : h->pf_xs[(l - 1) & 1];
      void* yout = l + 1 == n_layers ? y : h->pf_xs[l & 1];
      moe_status st = prefill_layer(h, l, xin, T, yout, MOE_FWD_RESIDUAL | MOE_FWD_PRENORM, nullptr,
                                    s, l);
      if (st != MOE_OK) return st;
    }
    h->last_T = T;
    h->last_layers = n_layers;
    h->last_prefill = true;
    return MOE_OK;
  }
  for (int t = 0; t < T; ++t) {
    DecodeParams p = params_for(h, 0, n_layers, static_cast<const uint16_t*>(x) + int64_t(t) * D,
                                static_cast<uint16_t*>(y) + int64_t(t) * D, PH_ALL,
                                MOE_FWD_RESIDUAL | MOE_FWD_PRENORM);
    // token t's ids: its own layer-major block [n_layers][K]
    p.ids = h->ids + int64_t(t) * n_layers * K;
    p.wts = h->wts + int64_t(t) * n_layers * K;
    moe_status st = launch(h, p, s);
    if (st != MOE_OK) return st;
  }
  h->last_T = T;
  h->last_layers = n_layers;
  h->last_prefill = false;
  return MOE_OK;
}

moe_status moe_forward_stack_host(moe_handle* h, const void* x, int T, void* y, int n_layers,
                                  void* stream) {
  if (!h || !x || !y) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return fail(h, MOE_ERR_INVALID_ARG, "T=%d out of range", T);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = size_t(T) * h->cfg.d_model * 2;
  std::memcpy(h->pin_x, x, bytes);
  CUDA_TRY(h, cudaMemcpyAsync(h->io_x, h->pin_x, bytes, cudaMemcpyHostToDevice, s));
  moe_status st = moe_forward_stack(h, h->io_x, T, h->io_y, n_layers, stream);
  if (st != MOE_OK) return st;
  CUDA_TRY(h, cudaMemcpyAsync(h->pin_y, h->io_y, bytes, cudaMemcpyDeviceToHost, s));
  st = sync_stream(h, s);
  if (st != MOE_OK) return st;
  std::memcpy(y, h->pin_y, bytes);
  return MOE_OK;
}

moe_status moe_stack_ids(moe_handle* h, int n_layers, int T, int32_t* ids, float* weights) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (n_layers != h->last_layers || T != h->last_T)
    return fail(h, MOE_ERR_INVALID_ARG, "moe_stack_ids: the last call ran %d layers x %d tokens",
                h->last_layers, h->last_T);
  moe_status st = check_device_status(h, nullptr);
  if (st != MOE_OK) return st;
  const int K = h->cfg.top_k;
  const size_t n = size_t(n_layers) * T * K;
  if (h->last_prefill) {
    // layer l's block starts at l * max_tokens * K
    const size_t blk = size_t(h->cfg.max_tokens) * K;
    for (int l = 0; l < n_layers; ++l) {
      if (ids)
        CUDA_TRY(h, cudaMemcpy(ids + size_t(l) * T * K, h->pf_ids + l * blk, size_t(T) * K * 4,
                               cudaMemcpyDeviceToHost));
      if (weights)
        CUDA_TRY(h, cudaMemcpy(weights + size_t(l) * T * K, h->pf_wts + l * blk, size_t(T) * K * 4,
                               cudaMemcpyDeviceToHost));
    }
    return MOE_OK;
  }
  std::vector<int32_t> ti(n);
  std::vector<float> tw(n);
  CUDA_TRY(h, cudaMemcpy(ti.data(), h->ids, n * 4, cudaMemcpyDeviceToHost));
  CUDA_TRY(h, cudaMemcpy(tw.data(), h->wts, n * 4, cudaMemcpyDeviceToHost));
  // device order: token-major blocks [t][layer][k]
  for (int l = 0; l < n_layers; ++l)
    for (int t = 0; t < T; ++t)
      for (int i = 0; i < K; ++i) {
        const size_t src = (size_t(t) * n_layers + l) * K + i;
        const size_t dst = (size_t(l) * T + t) * K + i;
        if (ids) ids[dst] = ti[src];
        if (weights) weights[dst] = tw[src];
      }
  return MOE_OK;
}

}  // extern "C"
#pragma GCC visibility pop
