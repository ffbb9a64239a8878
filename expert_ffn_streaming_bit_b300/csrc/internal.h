// Internal GPU data layout and kernel parameter blocks of libmoe_b300.
//
// Repacked quantised row ("qrow") of K inputs, used for every 4-bit matrix on
// the GPU: K/2 bytes of codes, then K/64 32-bit words (fp16 scale in the low
// half, fp16 bias in the high half), padded to a multiple of 16 bytes so that
// any run of rows is a legal bulk-copy source.  Inside each 32-bit word of
// codes (columns 8w..8w+7), byte i holds column 8w+i in its low nibble and
// column 8w+4+i in its high nibble (i = 0..3).  So word & 0x0F0F0F0F gives
// the codes of columns 0..3 as bytes and (word >> 4) & 0x0F0F0F0F those of
// columns 4..7, which pair with int16 activation pairs in a 2-way integer dot
// product (decode), or with one byte permute become fp16 1024+q pairs
// (prefill dequantisation).
//
// Per layer (device):
//   router_t   [D][E] uint8 codes, transposed so a run of input rows is contiguous
//   router_sb  [D/64][E] uint32 (scale | bias << 16)
//   shared_gu  [S][2] qrows of K=D: gate row j then up row j
//   shared_dn  [D] qrows of K=S
//   expert blob (one per routed expert, contiguous, `blob_bytes`):
//              [I][2] qrows of K=D (gate/up interleaved), then [D] qrows of K=I
#pragma once
#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)

#include <cstdint>

namespace moe {

constexpr int kGroup = 64;
constexpr int kMaxTopK = 32;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;   // threads that compute
constexpr int kThreads = kConsumers + 32;         // + one producer warp
constexpr int kChunkStride = 80;  // smem bytes per 32-element int16 chunk (64 data + 16 pad)
constexpr int kPairsPerStage = 16;  // gate/up row pairs per B stage (two per consumer warp)
constexpr int kMaxSlots = 6;

inline int64_t qrow_bytes(int64_t K) { return (K * 9 / 16 + 15) / 16 * 16; }

struct LayerDev {
  const uint8_t* router_t;
  const uint32_t* router_sb;
  const float* logit_bias;   // [E] or nullptr
  const uint8_t* shared_gu;
  const uint8_t* shared_dn;
  const uint8_t* experts;    // blob array (all experts, or the layer's HBM slots)
  const int32_t* slot_of;    // [E] blob index of each expert (resident mode), or nullptr
};

enum : int { PH_ROUTER = 1, PH_BSHARED = 2, PH_BROUTED = 4, PH_C = 8, PH_ALL = 15 };

// Device status word codes (bar[2]).
enum : uint32_t { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_ID = 2 };
// Grid synchronisation words (bar[], 256 bytes): [0..1] 64-bit arrival
// counter, [2] status, [32] release flag (its own 128-byte line).
constexpr int kBarWords = 64;
constexpr int kBarFlag = 32;
// Decode trace events per layer (thread 0 of each CTA, %globaltimer ns):
// layer start, x (and router logits) converted, routing done, shared gate/up
// done, routed gate/up done, h complete (barrier), h converted, down done,
// next-layer barrier passed.
constexpr int kTraceEvents = 13;
constexpr int kTraceMaxLayers = 64;

struct DecodeParams {
  const LayerDev* layers;  // device array, indexed by absolute layer
  int layer0, n_layers;
  int D, E, I, S, K;
  int rbD, rbI, rbS;       // qrow bytes for K = D, I, S
  int64_t blob_bytes, dn_off;
  int phases;
  int residual;
  int prenorm;                // layer input is x / sqrt(mean(x^2) + rms_eps)
  float rms_eps;
  int forced;                 // ids of layer0 given below (single-layer launches)
  int forced_ids[kMaxTopK];
  int use_slots;              // blob index of routed slot i = slots[i] (single-layer launches)
  int slots[kMaxTopK];
  const uint16_t* x_in;    // bf16 [D], input of layer0
  uint16_t* y_out;         // bf16 [D], output of the last layer
  uint16_t* xbuf;          // bf16 [2][D] scratch
  uint16_t* h;             // [K*I + S] fp16 bits of h * hscale (hscale: a power of two
                           // from the layer input's range, the same in every CTA)
  unsigned long long* lacc;  // [2][E] router logit accumulators, fixed point (units of
                             // 2^-32, two's complement), one per layer parity
  int32_t* ids;            // [n_layers][K], relative to layer0
  float* wts;              // [n_layers][K]
  uint32_t* bar;           // kBarWords grid synchronisation words
  // C phase: ntask = K * (I/32) + S/32 (branch, chunk) tasks, one per consumer
  // thread; rc_max rows per C stage (limited by the slot size)
  int ntask, rc_max;
  // shared memory carve-up (bytes)
  int slot_bytes, nslots;
  int off_vec, off_rpart, off_xnext, off_xres, off_logits, off_misc, off_bars, smem_total;
  uint64_t timeout_ns;     // bound on every device-side wait
  uint64_t* trace;         // optional: [grid][n_layers][kTraceEvents] %globaltimer stamps
  int stall_first_barrier; // test injection: the launch's first grid barrier waits for
                           // one more round of arrivals, which never comes
};

// ------------------------------------------------------------------ prefill
//
// Multi-token layer step (T >= 2): token prep, SIMT router GEMM + top-k,
// bucketing of the T*k assignments by expert (which also emits the grouped
// GEMM's work units), two grouped GEMMs on the tensor cores (gate/up with the
// GELU epilogue, then down), and a gather combine.

constexpr int kUnitTokens = 160;   // max B rows (tokens) of one GEMM work unit
// Heights of the activation tiles the GEMM loads (one tensor map each): a unit
// of n rows loads the smallest that holds its MMA width (n rounded up to 16),
// so a unit of a few tokens does not fill shared memory with 160 rows.
constexpr int kNBox = 6;
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int box_rows(int i) { return i == 0 ? 16 : 32 * i; }  // 16, 32 .. 160
static_assert(box_rows(kNBox - 1) == kUnitTokens, "the highest tile holds a whole unit");
constexpr int kTilesPerUnit = 1;   // 128-row weight tiles per GEMM work unit
constexpr int kMaxPrefillExperts = 256;

// One work unit of the grouped GEMM: a 128-row tile of one weight matrix
// against up to kUnitTokens activation rows.  16-byte aligned so that a unit
// is written and read as two vector accesses.
struct alignas(16) GemmUnit {
  int kind;    // 0 routed expert, 1 shared expert
  int mt;      // first weight row tile (rows mt*128 ..)
  int expert;  // routed: blob index of the expert
  int row0;    // routed: first bucket position; shared: first token
  int n;       // activation rows in the unit (1 .. kUnitTokens)
  int nmt;     // weight row tiles in the unit (1 .. kTilesPerUnit)
  int pad[2];
};

struct PrefillDims {
  int T, D, E, I, K, S;
  int mt_gu_r, mt_dn, mt_gu_s;  // 128-row tiles: routed gate/up, down, shared gate/up
};

// Router GEMM on the tensor cores: logits partials [nsplit][T][E].
int router_tc_splits(int T, int E, int D, int num_sms);
int router_tc_launch(const CUtensorMap& wmap, const CUtensorMap& xmap, int T, int E, int D,
                     int nsplit, float* partials, uint32_t* status, uint64_t timeout_ns, void* stream);

// x16, the fp16 token rows of the multi-token path, has a row pitch of
// D + kGsumCols: D columns of f_t x, then the token's 64-column group sums
// X_g = sum of the group's fp16 values, held as fp16(X_g / 64) (exact
// scaling; the sum of 64 values of up to 2^15 stays in range), for
// g < D / 64, and zeros after them.  The gate/up GEMM applies the weights'
// per-group biases b_g through these sums: sum_g (64 b_g) (X_g / 64).
constexpr int kGsumCols = 64;

struct RouteArgs {
  const uint16_t* x;  // bf16 [T][D]
  int T, D, E, K;
  int prenorm;
  float rms_eps;
  const CUtensorMap* wmap;    // router weight as fp16 parts: rows [0, Epad) = fp16(w),
                              // rows [Epad, 2 Epad) = fp16(w - fp16(w)), [2 Epad][D]
  const CUtensorMap* xmap;    // x16 [T][D] (pitch D + kGsumCols), 64 x 128 boxes
  const float* logit_bias;    // [E] or nullptr
  const int32_t* forced;      // device [T][K] or nullptr
  uint16_t* x16;              // fp16 [T][D + kGsumCols] out: x * f_t, then the group sums
  float* sigma;               // [T] out: (r_t / f_t), the scale of dot products with x16
  float* rscale;              // [T] out: r_t (pre-norm factor, 1 without)
  float* hscale;              // [T] out: power-of-two scale of the fp16 intermediate h
  float* partials;            // [nsplit][T][E]: sums of w . x16
  int nsplit;
  uint32_t* status;           // device status word
  uint64_t timeout_ns;
  int32_t* ids;               // [T][K] out
  float* wts;                 // [T][K] out
};
int prefill_route(const RouteArgs& a, void* stream);

struct BucketArgs {
  const int32_t* ids;  // [T][K]
  int T, K, E;
  int mt_gu_r, mt_dn, mt_gu_s;
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1]
  int32_t* perm;       // [T*K] bucket position -> assignment t*K + j
  int32_t* inv;        // [T*K] assignment -> bucket position
  GemmUnit* units_gu;  // gate/up units
  GemmUnit* units_dn;  // down units
  int32_t* n_units;    // [2] gate/up, down
  int32_t* hist;       // [bucket_blocks(T*K)][8][E] scratch: counts, then write bases
  uint32_t* status;
};
int bucket_blocks(int n);  // blocks of the bucketing launches for n assignments
int prefill_bucket(const BucketArgs& a, void* stream);

struct CombineArgs {
  const uint16_t* x;   // bf16 [T][D] (residual input)
  const uint16_t* e;   // bf16 [T*K][D] weighted routed outputs, bucket order
  const float* s;      // fp32 [T][D] shared expert output
  const int32_t* inv;  // [T*K]
  uint16_t* y;         // bf16 [T][D]
  int T, D, K, residual;
};
int prefill_combine(const CombineArgs& a, void* stream);

// Grouped GEMM on the tensor cores (gemm_tc.cu).  Index [kind]: 0 routed, 1 shared.
struct GemmParams {
  CUtensorMap tm_code[2];  // 4-bit codes: box 128 B x 128 rows, 128-byte swizzle
  CUtensorMap tm_sb[2];    // scale/bias words: box 16 B x 128 rows
  CUtensorMap tm_b[2][kNBox];  // activation rows (fp16): box 64 x box_rows(i), 128-byte swizzle
  const GemmUnit* units;
  const int32_t* n_units;  // device: number of units
  int mode;                // 0: gate/up (+ GELU epilogue), 1: down
  int K[2];                // reduction length (D for gate/up; I or S for down)
  int gsum;                // 1: the weights' biases enter through the activations' group
                           // sums, one more K block after the K columns (gate/up; the A
                           // operand is then fp16(s q)), 0: A = fp16(s q + b)
  const int32_t* perm;     // bucket position -> assignment
  int topk;
  const float* sigma;      // per-token scale of dot products with x16 (gate/up)
  const float* hscale;     // per-token scale of the fp16 h (gate/up multiplies, down divides)
  void* hout[2];           // gate/up: fp16 h rows (routed: bucket order; shared: tokens)
  int hld[2];
  void* eout;              // down, routed: bf16 [T*K][D], weighted by the routing weight
  float* sout;             // down, shared: fp32 [T][D]
  const float* wts;        // [T*K] routing weights by assignment
  int D;
  uint32_t* status;
  unsigned long long timeout_ns;
  int stall;               // test injection: the MMA role waits for an accumulator phase
                           // that never completes (every role then leaves through abort)
};
int gemm_tc_smem_bytes();
// max_rows: an upper bound on the activation rows of any unit (the batch's
// token count); it picks the kernel's plan: narrow up to 32, medium up to 128,
// wide above.
int gemm_tc_launch(const GemmParams& p, int grid, int max_rows, void* stream);
// out[pos] = x16[perm[pos] / topk] for pos < rows (fp16 rows of `D` columns).
int gather_rows_launch(const void* x16, int D, const int32_t* perm, int topk, int rows, void* out,
                       void* stream);

// Host entry points implemented in decode.cu.
int decode_smem_plan(DecodeParams* p, int max_smem);   // fills the carve-up; 0 if it fits
int decode_launch(const DecodeParams& p, int grid, void* stream, bool cooperative);

}  // namespace moe

// Implemented in api.cu for the library's other translation units.
struct moe_handle;
namespace moe {
// Launch parameters of a one-token resident decode stack over layers
// [0, n_layers) with pre-norm and residual (the moe_forward_stack recipe),
// without scratch pointers.  Fails like moe_forward_stack on bad arguments.
// A pending injected device stall of the handle is applied to (and consumed
// by) the returned parameters.
int stack_launch_params(moe_handle* h, const void* x, void* y, int n_layers, DecodeParams* p,
                        int* grid, int* device);
// Records an error message on the handle and returns `status`.
int handle_error(moe_handle* h, int status, const char* msg);
// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute belongs to the device context, so it is
// set once per (kernel, device); thread-safe.  Returns a cudaError_t.
int set_smem_limit(const void* kernel, int bytes);
}  // namespace moe
