// Internal GPU data layout and kernel parameter blocks of libmoe_b300.
//
// Repacked quantised row ("qrow") of K inputs, used for every 4-bit matrix on
// the GPU: K/2 bytes of codes, then K/64 32-bit words (fp16 scale in the low
// half, fp16 bias in the high half), padded to a multiple of 16 bytes so that
// any run of rows is a legal bulk-copy source.  Inside each 32-bit word of
// codes (columns 8w..8w+7) the nibble at bit 4s holds column 8w+2s and the
// nibble at bit 16+4s holds column 8w+2s+1 (s = 0..3), so one and-or with a
// mask yields two fp16 values 1024+q (or 1024+16q) that pair with one fp16x2
// word of activations.
//
// Per layer (device):
//   router_t   [D][E] uint8 codes, transposed so a run of input rows is contiguous
//   router_sb  [D/64][E] uint32 (scale | bias << 16)
//   shared_gu  [S][2] qrows of K=D: gate row j then up row j
//   shared_dn  [D] qrows of K=S
//   expert blob (one per routed expert, contiguous, `blob_bytes`):
//              [I][2] qrows of K=D (gate/up interleaved), then [D] qrows of K=I
#pragma once
#include <cstdint>

namespace moe {

constexpr int kGroup = 64;
constexpr int kMaxTopK = 32;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;   // threads that compute
constexpr int kThreads = kConsumers + 32;         // + one producer warp
constexpr int kChunkStride = 80;  // smem bytes per 32-element fp16 chunk (64 data + 16 pad)
constexpr int kPairsPerStage = 16;  // gate/up row pairs per B stage (8 warps x 2)
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
  float* h;                // [K*I + S] fp32 scratch
  float* partials;         // [E + 1][G_pad] router partial logits (transposed);
                           // row E holds partial sums of x^2 for the pre-norm
  int32_t* ids;            // [n_layers][K], relative to layer0
  float* wts;              // [n_layers][K]
  uint32_t* bar;           // [0] arrivals, [1] generation, [2] status
  int G_pad;               // partial stride (grid size rounded up to 8)
  // C-phase task mapping
  int cpt_c, nsub_i, nsub_s, tasks_row, rc_max;
  // shared memory carve-up (bytes)
  int slot_bytes, nslots;
  int off_vec, off_contrib, off_rpart, off_xnext, off_xres, off_logits, off_misc, off_bars,
      smem_total;
  uint64_t timeout_ns;     // bound on every device-side wait
};

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
int stack_launch_params(moe_handle* h, const void* x, void* y, int n_layers, DecodeParams* p,
                        int* grid, int* device);
// Records an error message on the handle and returns `status`.
int handle_error(moe_handle* h, int status, const char* msg);
}  // namespace moe
