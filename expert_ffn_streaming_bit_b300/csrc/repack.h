// Host-side repack of canonical weights into the GPU layout (see internal.h)
// and the per-layer LFU slot planner.
#pragma once
#include <cstdint>
#include <functional>
#include <vector>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

struct Dims {
  int64_t D, E, I, K, S;
};

inline int64_t router_t_bytes(const Dims& d) { return d.D * d.E; }
inline int64_t router_sb_bytes(const Dims& d) { return d.D / kGroup * d.E * 4; }
inline int64_t bias_bytes(const Dims& d) { return (d.E * 4 + 15) / 16 * 16; }
inline int64_t shared_gu_bytes(const Dims& d) { return d.S * 2 * qrow_bytes(d.D); }
inline int64_t shared_dn_bytes(const Dims& d) { return d.D * qrow_bytes(d.S); }

int64_t expert_blob_bytes(const Dims& d);
int64_t layer_fixed_bytes(const Dims& d);
// router_t | router_sb | logit bias (fp32, zeros if none) | shared_gu | shared_dn
void repack_layer_fixed(const Dims& d, const moe_layer_weights& w, uint8_t* dst);
// gate/up interleaved qrows of K=D, then down qrows of K=I
void repack_expert(const Dims& d, const moe_qtensor& gate, const moe_qtensor& up,
                   const moe_qtensor& down, uint8_t* blob);
// A whole 4-bit [rows][K] matrix as consecutive qrows of K inputs.
void repack_matrix(const moe_qtensor& t, int64_t rows, int64_t K, uint8_t* dst);
void parallel_for(int64_t n, const std::function<void(int64_t)>& fn);

// LFU slot table of one layer (policy stated in moe.h at moe_cache_step).
class SlotTable {
 public:
  void init(int n_slots, int n_experts);
  void reset();
  // Plans k distinct ids; fills hit/slot/evicted per id.  Returns the number
  // of misses, or -1 if the ids are invalid (then nothing changes).
  int plan(const int32_t* ids, int k, int32_t* hit, int32_t* slot, int32_t* evicted);
  // Marks slot s empty (used when its fill could not be enqueued).
  void clear_slot(int s);
  int expert_in(int s) const { return expert_[s]; }
  int slot_of(int e) const { return where_[e]; }

 private:
  std::vector<int32_t> expert_;  // per slot, -1 = empty
  std::vector<int64_t> count_;   // per slot use count
  std::vector<int64_t> last_;    // per slot last step used
  std::vector<int32_t> where_;   // per expert, slot or -1
  int64_t step_ = 0;
  int n_experts_ = 0;
};

}  // namespace moe
