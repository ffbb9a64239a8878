/*
 * moe.h — C ABI of the B300 Mixture-of-Experts layer-step library
 * (libmoe_b300.so, built for sm_103a).
 *
 * The library runs the data-parallel hot path of an out-of-core MoE runtime on
 * one GPU: per layer and token, an 8-bit router scores the experts and keeps
 * the top k, the chosen 4-bit routed experts and an always-on shared expert
 * run as gated FFNs, and their outputs are combined.  Optionally the routed
 * experts live in a pinned host pool and only a per-layer set of HBM slots is
 * resident, filled on demand under an LFU policy.
 *
 * Passages the operations follow (page title, section):
 *   sh.edu-sjtu.cn "TurboFieldfare：8GB Mac 本地跑 Gemma 4 26B-A4B 的 Swift +
 *     Metal 运行时", section "TurboFieldfare 把内存压到约 2GB 的三件事": per
 *     layer the router picks the top-8 expert ids, they are planned against the
 *     layer's 16-slot LFU cache, misses are read into GPU-visible buffers while
 *     the GPU computes the resident shared expert, and the two outputs are
 *     combined; prompts are prefilled in chunks of at most 128 tokens.
 *   shilu.ai "drumih/turbo-fieldfare", overview table (row 权重): MLX affine
 *     4-bit weights with group 64, 8-bit router; section 推理引擎的工作原理:
 *     the same per-layer plan/fill/overlap/combine sequence; section 状态和范围:
 *     bounded expert cache, chunked single-prompt prefill, token-at-a-time
 *     generation.
 * The pages give no formulas.  The readings used: y = sum_i w_i FFN_i(x) +
 * FFN_shared(x), FFN(x) = W_down (gelu_tanh(W_gate x) * (W_up x)), w = softmax
 * of the chosen router logits, ties in the logits go to the lower expert index.
 *
 * Conventions for every call:
 *   - Return value: MOE_OK or a negative moe_status.  No call aborts or throws
 *     across the ABI.  On error the handle stays usable unless the status is
 *     MOE_ERR_CUDA (the CUDA context may be lost) and moe_last_error() holds a
 *     one-line description.
 *   - "device" pointers are CUDA global memory on the handle's device;
 *     "host" pointers are ordinary (pageable or pinned) host memory.
 *   - Activations are bf16 bit patterns, row-major [T][d_model].
 *   - A handle is used by one host thread at a time.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Kernels run asynchronously; an error a kernel reports on the device
 *     (a bounded wait that ran out, an expert id out of range) is returned by
 *     the next call that synchronises (moe_stack_ids, the host-I/O call, or a
 *     forward call that asks for ids).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* bad pointer, size or configuration */
  MOE_ERR_OOM = -2,         /* device or pinned host allocation failed */
  MOE_ERR_CUDA = -3,        /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = -4,     /* a bounded wait (host or device) ran out */
  MOE_ERR_INJECTED = -5,    /* a fault injected with moe_debug_inject() */
  MOE_ERR_STATE = -6,       /* call not valid in this handle's mode or state */
  MOE_ERR_DEVICE = -7,      /* a kernel reported an inconsistent input (e.g. id out of range) */
  MOE_ERR_IO = -8           /* reading or writing the expert store file failed */
} moe_status;

typedef struct moe_handle moe_handle;

/* Shape of the layer stack.  Requirements: group == 64; d_model % 256 == 0;
 * d_expert % 64 == 0; d_shared % 64 == 0; 1 <= top_k <= 32; top_k <= n_experts
 * <= 1024; n_experts % 16 == 0; n_layers >= 1; max_tokens >= 1. */
typedef struct {
  int d_model;    /* D: hidden size */
  int n_experts;  /* E: routed experts per layer */
  int d_expert;   /* I: routed expert inner size */
  int top_k;      /* k: experts chosen per token */
  int d_shared;   /* S: shared expert inner size */
  int group;      /* quantisation group along the input dimension (64) */
  int n_layers;   /* L */
  int n_slots;    /* 0: every expert resident in HBM.  Else per-layer HBM slot
                     count (top_k <= n_slots <= n_experts); the full expert
                     set then lives in a pinned host pool owned by the handle. */
  int max_tokens; /* largest T passed to any forward call */
  const char* expert_store; /* NULL, or (n_slots > 0) the path of an expert store file
                               written by moe_store_write: the routed experts are then
                               read from it on each cache miss instead of being held in
                               a pinned host pool */
  int io_threads; /* expert store only: concurrent pread() calls per miss batch (>= 1) */
} moe_config;

/* One affine-quantised matrix in canonical form, HOST memory, row-major
 * [rows][cols] with groups of `group` along cols:
 *   value(r, c) = fp16(scale[r][c/group]) * code(r, c) + fp16(bias[r][c/group])
 * 4-bit: q is [rows][cols/2]; column 2i is the low nibble of byte i.
 * 8-bit: q is [rows][cols].  scale and bias hold IEEE binary16 bit patterns. */
typedef struct {
  const uint8_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
} moe_qtensor;

/* Weights of one layer, HOST memory, canonical form.  Shapes:
 *   router       8-bit [E][D]
 *   router_logit_bias  fp32 [E], added to the logits before ranking; may be NULL
 *   shared_gate, shared_up   4-bit [S][D];   shared_down  4-bit [D][S]
 *   exp_gate, exp_up         arrays of E tensors, each 4-bit [I][D]
 *   exp_down                 array of E tensors, each 4-bit [D][I]          */
typedef struct {
  moe_qtensor router;
  const float* router_logit_bias;
  moe_qtensor shared_gate, shared_up, shared_down;
  const moe_qtensor* exp_gate;
  const moe_qtensor* exp_up;
  const moe_qtensor* exp_down;
} moe_layer_weights;

/*
 * moe_store_write — write the expert store file for `cfg` at `path`: the
 * storage tier of the slot cache (blog.hypho.cn "TurboFieldfare gemma4
 * out-of-core inference", section "为什么不用 mmap？", and shilu.ai
 * "drumih/turbo-fieldfare", section 推理引擎的工作原理: cold experts live on
 * the SSD and are read with bounded parallel pread() calls, not mapped).
 * Host only (no GPU is touched).  Every routed expert of every layer
 * (`layers`: cfg->n_layers entries, host memory, canonical form; only the
 * exp_* tensors are read) is repacked into the GPU blob layout and written
 * at a page-aligned offset after a 4096-byte header that records the
 * shape.  An existing file is replaced.  Fails with MOE_ERR_INVALID_ARG on
 * a bad configuration or missing tensors, MOE_ERR_IO if the file cannot be
 * written (then the file may be left partial).
 */
moe_status moe_store_write(const moe_config* cfg, const moe_layer_weights* layers, const char* path);

/*
 * moe_create — build a handle for `cfg` on the current CUDA device.
 * Follows shilu.ai "drumih/turbo-fieldfare", overview table (row 权重: the
 * affine 4-bit g64 experts and 8-bit router this call repacks) and section
 * 推理引擎的工作原理 (weights are prepared once into the runtime's own layout,
 * and the expert set sits in a backing store while a per-layer slot cache is
 * resident); one owner per model.
 * Copies and repacks all weights (`layers`: n_layers entries, host memory) into
 * the GPU layout: into HBM when cfg->n_slots == 0, else into a pinned host
 * pool plus n_slots HBM slots per layer.  With cfg->expert_store set (and
 * n_slots > 0) the routed experts come from that file instead: `layers`
 * then only needs the router and shared tensors (exp_* may be NULL), the
 * store's header must match cfg (else MOE_ERR_INVALID_ARG), and the handle
 * holds top_k pinned staging buffers and cfg->io_threads reader threads in
 * place of the pool.  The caller may free `layers` when the call returns.  Allocates the handle's device scratch (sized by
 * max_tokens), a side copy stream and events.  On failure *out is NULL and
 * nothing is leaked.
 */
moe_status moe_create(const moe_config* cfg, const moe_layer_weights* layers, moe_handle** out);

/* moe_destroy — synchronise the handle's own streams and free everything.
 * NULL is accepted.  The counterpart of moe_create: it releases the resident
 * weights, the slot cache and the backing pool that shilu.ai
 * "drumih/turbo-fieldfare", section 推理引擎的工作原理, has one owner hold. */
void moe_destroy(moe_handle* h);

/* Flags for the forward calls. */
#define MOE_FWD_RESIDUAL 1 /* y = bf16(x + moe(u)) instead of bf16(moe(u)) */
#define MOE_FWD_PRENORM 2  /* u = x / sqrt(mean(x^2) + 1e-6) (unit-gain RMS norm per token);
                              without it u = x.  shilu.ai page, section 状态和范围, lists
                              normalisation kernels beside the MoE kernels; the pages'
                              model normalises each FFN block's input. */

/* Outcome of one cache step for k ids (k <= 64). */
typedef struct {
  int32_t hit[64];     /* 1 if ids[i] was resident */
  int32_t slot[64];    /* HBM slot holding ids[i] after the step */
  int32_t evicted[64]; /* expert evicted to make room for ids[i], or -1 */
  int misses;
} moe_cache_result;

/* Per-call statistics (all fields written by the call when non-NULL). */
typedef struct {
  int32_t* ids;     /* host [T][k] or NULL: chosen expert ids (a copy, synchronising) */
  float* weights;   /* host [T][k] or NULL: routing weights (synchronising) */
  int hits;         /* streaming mode: cache hits of this call */
  int misses;       /* streaming mode: cache misses (experts copied host->HBM) */
  int64_t bytes_h2d;/* streaming mode: weight bytes copied host->HBM */
  moe_cache_result* cache; /* host or NULL; streaming mode: the layer's cache step for
                              this call's ids, in slot order i = 0..k-1 of `ids` (the
                              forced ids, or the router's choice in rank order) */
} moe_layer_stats;

/*
 * moe_layer_forward — one MoE layer step for T tokens (1 <= T <= max_tokens).
 * Follows sh.edu-sjtu.cn article, section 三件事 (route to the top-8 experts,
 * compute the resident shared expert while the routed ones are fetched,
 * combine; prefill runs in chunks so each fetched expert serves many rows)
 * and shilu.ai "drumih/turbo-fieldfare", section 推理引擎的工作原理 (the
 * per-layer route / plan / fill / overlap / combine sequence).
 * Resident mode: T == 1 runs the persistent decode kernel; T >= 2 runs the
 *   prefill path: router GEMM + top-k, token-to-expert bucketing, grouped
 *   GEMMs on the tensor cores (fp16 operands: weights dequantised to fp16 in
 *   tensor memory, activations scaled by a per-token power of two; fp32
 *   accumulation; in the gate/up GEMM the weights' per-group biases enter
 *   through the tokens' 64-column group sums), and a gather combine.  The prefill path holds the gated
 *   intermediate h in fp16 scaled per token by a power of two chosen from
 *   the token's input range, and the routed expert outputs in bf16 before
 *   the combine.
 * x: device [T][D] bf16 input.  y: device [T][D] bf16 output; y may not alias x.
 * forced_ids: host [T][k] or NULL.  When given, those experts are used (each
 *   row k distinct ids in [0, E)); their weights are still the softmax of the
 *   router logits over the forced set.
 * Streaming mode (n_slots > 0) requires T == 1: the call routes, plans the
 *   chosen ids against the layer's LFU slots (see moe_cache_step), copies the
 *   misses from the pinned pool on the handle's side stream while the shared
 *   expert runs on `stream`, then runs the routed experts and the combine.
 *   Without forced_ids this reads the ids back to the host (synchronising).
 * All kernels are enqueued on `stream`; the call returns without
 * synchronising unless stats->ids / stats->weights are requested or the mode
 * needs a host decision.
 */
moe_status moe_layer_forward(moe_handle* h, int layer, const void* x, int T, void* y, int flags,
                             const int32_t* forced_ids, void* stream, moe_layer_stats* stats);

/*
 * moe_forward_stack — layers [0, n_layers) back to back (T < 5: one
 * persistent kernel per token for the whole stack; T >= 5: the multi-token
 * path layer by layer over all T tokens, which reads each chosen expert once
 * for all its rows), each reading the
 * RMS-normalised residual stream and adding its output to it:
 * x_{l+1} = bf16(x_l + moe_l(x_l / sqrt(mean(x_l^2) + 1e-6))); y = x_{n_layers}
 * (the flags MOE_FWD_RESIDUAL | MOE_FWD_PRENORM on every layer).
 * Resident mode only.  x, y: device [T][D] bf16, y may not alias x.
 * The split at 5 tokens is measured: on the 30-layer Gemma-shape stack, 4
 * tokens take 2.40 ms as 4 single-token launches and 2.60 ms through the
 * multi-token path, 5 tokens 3.00 against 2.78 ms, 8 tokens 4.81 against
 * 3.57 ms and 32 tokens 19 ms against 5.9 ms.
 */
moe_status moe_forward_stack(moe_handle* h, const void* x, int T, void* y, int n_layers,
                             void* stream);

/*
 * moe_forward_stack_host — moe_forward_stack with HOST input and output:
 * copies x (host [T][D] bf16) to the device, runs the stack, copies the result
 * to y (host [T][D] bf16) and synchronises `stream`.  Uses the handle's
 * pinned staging buffers; x and y may be pageable.
 */
moe_status moe_forward_stack_host(moe_handle* h, const void* x, int T, void* y, int n_layers,
                                  void* stream);

/*
 * moe_forward_stack_noalloc — moe_forward_stack for one token (T = 1) that
 * allocates nothing.  The pages have no counterpart to this call: it exists
 * for callers that may not allocate device memory while they run, such as
 * code inside an allocator or memory-pool hook, real-time loops where
 * cudaMalloc's implicit synchronisation is not allowed, or hosts whose
 * allocator belongs to another framework.
 *   x, y: device [1][D] bf16, y may not alias x (caller-owned, as for
 *   moe_forward_stack).  Resident mode only; the handle's device must be
 *   current.
 *   device_status: host int32 or NULL.  When given, the call enqueues on
 *   `stream`, after the kernel, a copy of the kernel's device status word
 *   into *device_status: 0 no error, 1 a device-side bounded wait ran out,
 *   2 an expert id out of range (y is then undefined).  The value is valid
 *   once `stream` has synchronised; with pageable host memory the copy, and
 *   so the kernel, has finished when the call returns.
 * The per-call scratch (grid-barrier words, activation double buffer, h,
 * router partials, ids, weights) lives in one statically sized device array
 * of 1 MiB inside the library.  Every GPU that loads the library holds that
 * array until the process exits.  A shape whose scratch does not fit is
 * rejected with MOE_ERR_INVALID_ARG and a message giving both sizes.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it, so make that first call before any
 * stream capture.  Every call shares the one array and overwrites what the
 * previous call left there: calls that overlap on the GPU (other streams, or
 * other handles on the same device) race and must be serialised by the
 * caller.  Ids and weights of this call are not retrievable (moe_stack_ids
 * reads the handle's own scratch).  A pending MOE_INJECT_DEVICE_STALL of the
 * handle applies to this call's launch.
 */
moe_status moe_forward_stack_noalloc(moe_handle* h, const void* x, void* y, int n_layers,
                                     void* stream, int32_t* device_status);

/*
 * moe_stack_ids — copy the expert ids and weights chosen by the most recent
 * forward call on this handle: ids host [n_layers][T][k] int32, weights host
 * [n_layers][T][k] fp32 (either may be NULL).  Synchronises the device.
 */
moe_status moe_stack_ids(moe_handle* h, int n_layers, int T, int32_t* ids, float* weights);

/*
 * moe_last_buckets — the token-to-expert bucketing of the most recent
 * multi-token (T >= 2, resident mode) forward call's last layer, copied to
 * host memory (synchronises the device).  For a prefill chunk the T*k
 * assignments a = t*k + j are grouped by expert, stably (sh.edu-sjtu.cn
 * article, section 三件事, third bullet; shilu.ai page, section 推理引擎的工作原理:
 * each expert brought in serves every row routed to it):
 *   counts  [E]     assignments per expert
 *   offsets [E+1]   exclusive prefix sum of counts
 *   perm    [T*k]   assignments in (expert, t, j) order
 * Any pointer may be NULL.  MOE_ERR_STATE if the last call was not a
 * multi-token call.
 */
moe_status moe_last_buckets(moe_handle* h, int32_t* counts, int32_t* offsets, int32_t* perm);

/* Flags for moe_cache_step. */
#define MOE_PLAN_ONLY 1 /* update the slot table but copy no weights */

/*
 * moe_cache_step — the per-layer expert-slot cache of shilu.ai
 * "drumih/turbo-fieldfare", section 推理引擎的工作原理 (the CPU plans the
 * chosen ids against the layer's LFU slots and the misses are read into
 * GPU-visible buffers) and sh.edu-sjtu.cn article, section 三件事 (a bounded
 * cache of recently used experts per layer).
 * Plan k distinct expert ids (host, each in [0, E)) against
 * layer `layer`'s slots: hits first (use count + 1, last use = this step), then
 * misses in ascending expert id take the lowest empty slot, or else evict,
 * among slots this step has not used, the least-used slot (then the least
 * recently used, then the lowest slot index); newcomers start at count 1.
 * Unless MOE_PLAN_ONLY, each miss is copied from the pinned pool into its
 * slot with one cudaMemcpyAsync on the handle's side stream; the copies are
 * ordered before the next forward call on this layer.  With an expert store
 * the misses are first read from the file into the pinned staging buffers,
 * each blob in 1 MiB pread() calls of which up to io_threads run at once
 * (page-aligned direct I/O where the file system allows it); the call
 * returns once the reads are done and the copies enqueued.  Streaming mode
 * only.  If a read fails (MOE_ERR_IO) or a copy cannot be enqueued, the slot
 * is left empty and the call fails; the next step refetches that expert.
 */
moe_status moe_cache_step(moe_handle* h, int layer, const int32_t* ids, int k, int flags,
                          moe_cache_result* out);

/* moe_cache_reset — empty every slot of every layer (no copies). */
moe_status moe_cache_reset(moe_handle* h);

/*
 * Host-only slot planner: the same LFU policy as moe_cache_step, without a
 * handle, a GPU or any copy.  For callers that plan ahead (e.g. to prefetch)
 * and for tests.  moe_slot_plan_step fails with MOE_ERR_INVALID_ARG (state
 * unchanged) if the ids repeat, fall outside [0, n_experts) or k > n_slots.
 */
typedef struct moe_slot_plan moe_slot_plan;
moe_status moe_slot_plan_create(int n_slots, int n_experts, moe_slot_plan** out);
moe_status moe_slot_plan_step(moe_slot_plan* p, const int32_t* ids, int k, moe_cache_result* out);
void moe_slot_plan_destroy(moe_slot_plan* p);

/* Sizes of what the handle holds. */
typedef struct {
  int64_t device_weight_bytes;  /* HBM bytes of repacked weights (incl. slots) */
  int64_t pinned_pool_bytes;    /* pinned host pool (streaming mode) */
  int64_t device_scratch_bytes; /* HBM scratch */
  int64_t expert_blob_bytes;    /* bytes of one repacked routed expert */
  int num_sms;                  /* SMs used by the persistent kernels */
  int store_direct_io;          /* expert store: 1 if reads bypass the page cache */
  int io_threads;               /* expert store: reader threads (0 without a store) */
} moe_info;
moe_status moe_get_info(const moe_handle* h, moe_info* out);

/* Host-side fault injection for tests (never touches the GPU):
 *   MOE_INJECT_H2D_FAIL: the n-th next miss copy is not enqueued and reported
 *     as MOE_ERR_INJECTED; the slot it was meant for is left empty.
 *   MOE_INJECT_SLOW_COPY: sleep `arg` milliseconds on the host before each
 *     miss copy is enqueued (results must not change).
 *   MOE_INJECT_PINNED_ALLOC_FAIL: the next moe_create in this process fails
 *     its pinned-pool allocation (h may be NULL).
 *   MOE_INJECT_DEVICE_STALL: the next decode-kernel launch of h waits at its
 *     first grid barrier for a round of arrivals that never comes, with a
 *     device-side wait limit of `arg` ms (1..2000) instead of 2 s.  The wait
 *     runs out, every CTA leaves after its copies in flight have landed, and
 *     the next status check (a synchronising call) returns MOE_ERR_TIMEOUT
 *     and resets the barrier counter and logit accumulators, so the handle
 *     and the CUDA context stay usable.  No memory is touched out of bounds.
 *   MOE_INJECT_READ_FAIL: in the `arg`-th next expert-store read batch the
 *     first 1 MiB read fails (as if the device returned an error): that
 *     expert's slot is left empty and moe_cache_step returns MOE_ERR_IO.
 *   MOE_INJECT_GEMM_STALL: in the next multi-token (prefill) call of h, the
 *     gate/up grouped GEMM's MMA issuer waits for an accumulator phase that
 *     never completes, with a device-side wait limit of `arg` ms (1..2000).
 *     The wait runs out, the status word records it and every role of the
 *     kernel (loaders, dequantisers, epilogue) leaves through the CTA's abort
 *     flag after its copies in flight have landed; the tensor memory is
 *     freed.  The next synchronising call returns MOE_ERR_TIMEOUT and the
 *     handle stays usable.
 *   MOE_INJECT_NONE: clear everything. */
#define MOE_INJECT_NONE 0
#define MOE_INJECT_H2D_FAIL 1
#define MOE_INJECT_SLOW_COPY 2
#define MOE_INJECT_PINNED_ALLOC_FAIL 3
#define MOE_INJECT_DEVICE_STALL 4
#define MOE_INJECT_READ_FAIL 5
#define MOE_INJECT_GEMM_STALL 6
moe_status moe_debug_inject(moe_handle* h, int what, int arg);

/* Host waits on device work poll with this deadline (default 10000 ms) and
 * return MOE_ERR_TIMEOUT when it passes. */
moe_status moe_set_timeout_ms(moe_handle* h, int ms);

/*
 * Decode tracing (for profiling the persistent decode kernel).
 * moe_trace_enable(h, 1): later decode launches of this handle record, per
 * CTA and layer, MOE_TRACE_EVENTS %globaltimer stamps (ns) taken by the CTA's
 * first consumer thread: (0) layer start, (1) input and router logits loaded
 * and reduced, (2) routing done, (3) first shared gate/up stage in shared
 * memory, (4) shared gate/up done, (5) first and (6) last routed gate/up
 * stage in shared memory, (7) routed gate/up done, (8) h complete (grid
 * barrier), (9) h loaded and converted, (10) first down stage in shared
 * memory, (11) down done, (12) next grid barrier passed.  A stamp that does
 * not occur in a layer is left as it was.  moe_trace_enable(h, 0) stops
 * recording.
 * moe_trace_read(h, out, n_layers): copies the last launch's stamps to host
 * out [num_sms][n_layers][MOE_TRACE_EVENTS] int64 (n_layers of that launch,
 * at most 64; synchronises).
 */
#define MOE_TRACE_EVENTS 13
moe_status moe_trace_enable(moe_handle* h, int on);
moe_status moe_trace_read(moe_handle* h, int64_t* out, int n_layers);

/*
 * While tracing is on, multi-token (prefill) layer calls also record CUDA
 * events between their phases on the call's stream (up to 256 calls).
 * moe_prefill_phase_ms(h, ms, calls) synchronises, writes the summed times
 * of the recorded calls to ms[5] (router prep + GEMM + top-k, bucketing,
 * gate/up GEMM, down GEMM, combine), the number of calls to *calls (may be
 * NULL), and starts a new recording.
 */
moe_status moe_prefill_phase_ms(moe_handle* h, float* ms, int* calls);

/* ------------------------------------------------------------------------
 * Decode attention: the step before the router (shilu.ai
 * "drumih/turbo-fieldfare", section 推理引擎的工作原理: in every layer the GPU
 * computes attention and then the router from resident weights; section
 * 状态和范围: 4-bit MLX affine attention weights, an FP16 KV store that is a
 * bounded ring for sliding-window layers and linear for full-attention
 * layers, and exact split-K/V decode attention with distinct normalised K
 * and V paths).  The pages give no formulas or shapes; the reading used:
 *   u = x / sqrt(mean(x^2) + 1e-6); q = Wq u, k = Wk u, v = Wv u;
 *   each head of q, k and v divided by its RMS (eps 1e-6); RoPE on q and k
 *   (pairs (i, i + d/2) rotated by pos * theta^(-2i/d));
 *   k, v stored in fp16 in slot pos % capacity; scores q . k / sqrt(d) over
 *   the visible positions (a sliding layer: the last `window`; a full layer:
 *   all of 0 .. pos); softmax; o = sum w v; y = Wo o (+ x), bf16.
 *   Query head h reads key/value head h / (n_heads / n_kv_heads).
 */
typedef struct moe_attn moe_attn;

/* Shape of the attention blocks.  Requirements: group == 64; d_model % 256
 * == 0 and <= 4096; n_heads % n_kv_heads == 0; head_dim in {64, 128, 256};
 * n_heads * head_dim % 256 == 0 and <= 4096; window >= 1; max_seq >= 1. */
typedef struct {
  int d_model, n_heads, n_kv_heads, head_dim, group, n_layers;
  int window;               /* sliding layers: attended positions (the ring's capacity) */
  int max_seq;              /* full layers: positions 0 .. max_seq - 1 (linear capacity) */
  const int32_t* sliding;   /* host [n_layers]: 1 sliding window, 0 full; NULL: all full */
  const float* rope_theta;  /* host [n_layers] RoPE base; NULL: 10000 for every layer */
} moe_attn_config;

/* Weights of one attention block, HOST memory, canonical 4-bit form:
 *   wq [n_heads * head_dim][d_model], wk and wv [n_kv_heads * head_dim][d_model],
 *   wo [d_model][n_heads * head_dim]. */
typedef struct {
  moe_qtensor wq, wk, wv, wo;
} moe_attn_weights;

/* moe_attn_create — repack the weights into HBM and allocate the FP16 KV
 * caches (per layer n_kv_heads x capacity x head_dim for keys and for values)
 * on the current device.  The caller may free `layers` afterwards.  On
 * failure *out is NULL (message: moe_attn_last_error(NULL)). */
moe_status moe_attn_create(const moe_attn_config* cfg, const moe_attn_weights* layers,
                           moe_attn** out);
void moe_attn_destroy(moe_attn* a); /* NULL-safe; synchronises the device */
const char* moe_attn_last_error(const moe_attn* a);

/* moe_attn_forward — one token's attention step of layer `layer`.
 * x: device bf16 [d_model] (the layer input), y: device bf16 [d_model],
 * y may not alias x; both 16-byte aligned.  pos: the token's position; a
 * layer takes positions 0, 1, 2, ... in order (pos 0 restarts it, anything
 * else out of order is MOE_ERR_STATE); a full layer refuses pos >= max_seq.
 * The token's key and value are appended to the layer's cache, then
 * y = bf16(attention(x)), or bf16(x + attention(x)) with MOE_FWD_RESIDUAL.
 * Five kernels on `stream`; nothing synchronises. */
moe_status moe_attn_forward(moe_attn* a, int layer, const void* x, long long pos, void* y,
                            int flags, void* stream);

/* moe_attn_reset — forget every layer's positions (the next call of each
 * layer must use pos 0). */
moe_status moe_attn_reset(moe_attn* a);

/* moe_decode_step — one decode token through n_layers full layer steps: for
 * each layer l, x = bf16(x + attention_l(x)) (moe_attn_forward with the
 * residual), then that bf16 x goes straight to layer l's router and experts
 * (moe_layer_forward with MOE_FWD_PRENORM | MOE_FWD_RESIDUAL): the router
 * hand-off stays on the device.  x, y: device bf16 [d_model], y may not
 * alias x.  `h` must have the same d_model and at least n_layers layers. */
moe_status moe_decode_step(moe_attn* a, moe_handle* h, const void* x, long long pos, void* y,
                           int n_layers, void* stream);

const char* moe_status_string(moe_status s);
/* Last error text of this handle ("" if none); with h == NULL, of the last
 * failed moe_create in this process. */
const char* moe_last_error(const moe_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
