// Per-layer LFU expert-slot planner (host).
//
// Mirrors the pages' CPU-side plan of the router's top-8 ids against a
// layer's 16-slot LFU expert cache (shilu.ai "drumih/turbo-fieldfare",
// section 推理引擎的工作原理).  Tie-breaks are not on the pages; the ones used
// are stated in moe.h at moe_cache_step.
#include <algorithm>

#include "repack.h"

namespace moe {

void SlotTable::init(int n_slots, int n_experts) {
  expert_.assign(n_slots, -1);
  count_.assign(n_slots, 0);
  last_.assign(n_slots, 0);
  where_.assign(n_experts, -1);
  n_experts_ = n_experts;
  step_ = 0;
}

void SlotTable::reset() { init(static_cast<int>(expert_.size()), n_experts_); }

void SlotTable::clear_slot(int s) {
  if (expert_[s] >= 0) where_[expert_[s]] = -1;
  expert_[s] = -1;
  count_[s] = 0;
  last_[s] = 0;
}

int SlotTable::plan(const int32_t* ids, int k, int32_t* hit, int32_t* slot, int32_t* evicted) {
  const int ns = static_cast<int>(expert_.size());
  if (k < 0 || k > ns) return -1;
  for (int i = 0; i < k; ++i) {
    if (ids[i] < 0 || ids[i] >= n_experts_) return -1;
    for (int j = 0; j < i; ++j)
      if (ids[j] == ids[i]) return -1;
  }
  std::vector<char> used(ns, 0);
  // hits
  for (int i = 0; i < k; ++i) {
    evicted[i] = -1;
    const int s = where_[ids[i]];
    hit[i] = s >= 0 ? 1 : 0;
    slot[i] = s;
    if (s >= 0) {
      count_[s] += 1;
      last_[s] = step_;
      used[s] = 1;
    }
  }
  // misses in ascending expert id
  std::vector<int> miss;
  for (int i = 0; i < k; ++i)
    if (!hit[i]) miss.push_back(i);
  std::sort(miss.begin(), miss.end(), [&](int a, int b) { return ids[a] < ids[b]; });
  for (int i : miss) {
    int best = -1;
    for (int s = 0; s < ns; ++s)
      if (expert_[s] < 0) {
        best = s;
        break;
      }
    if (best < 0) {
      for (int s = 0; s < ns; ++s) {
        if (used[s]) continue;
        if (best < 0 || count_[s] < count_[best] ||
            (count_[s] == count_[best] && last_[s] < last_[best]))
          best = s;
      }
    }
    evicted[i] = expert_[best];
    if (expert_[best] >= 0) where_[expert_[best]] = -1;
    expert_[best] = ids[i];
    where_[ids[i]] = best;
    count_[best] = 1;
    last_[best] = step_;
    used[best] = 1;
    slot[i] = best;
  }
  ++step_;
  return static_cast<int>(miss.size());
}

}  // namespace moe
