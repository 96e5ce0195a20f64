// Host side of offload mode: which (layer, expert) record occupies each HBM
// slot, least-recently-used replacement, and the per-layer hit/miss counts.
//
// PR #385 "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
// (offload backend)", "What this adds": a fraction of the NVFP4 experts stays
// resident in GPU memory and the rest are streamed from host memory every
// step.  Here a forward's touched experts -- those already resident first --
// are placed in slots in batches of at most the slot count; within a batch,
// hits are refreshed first, then every miss takes an empty slot or else the
// least recently used slot that the batch does not use.
#pragma once

#include <stdint.h>

#include <vector>

namespace ftmoe {

class SlotCache {
 public:
  struct Placement {
    int slot;   // slot holding the expert for this batch
    bool miss;  // its record must be copied in before the batch runs
  };

  void reset(int n_slots, int n_layers, int n_experts) {
    n_slots_ = n_slots;
    layer_.assign(n_slots, -1);
    expert_.assign(n_slots, -1);
    stamp_.assign(n_slots, 0);
    slot_of_.assign((size_t)n_layers * n_experts, -1);
    hits_.assign(n_layers, 0);
    misses_.assign(n_layers, 0);
    n_experts_ = n_experts;
    clock_ = 0;
  }

  int slots() const { return n_slots_; }
  int64_t hits(int layer) const { return hits_[layer]; }
  int64_t misses(int layer) const { return misses_[layer]; }
  int slot_of(int layer, int e) const { return slot_of_[(size_t)layer * n_experts_ + e]; }

  // Places one batch (distinct experts of `layer`, at most slots() of them).
  std::vector<Placement> place(int layer, const int* experts, int n) {
    std::vector<Placement> out(n);
    const uint64_t batch_start = clock_ + 1;
    for (int i = 0; i < n; ++i) {  // hits first: refresh them
      const int s = slot_of(layer, experts[i]);
      out[i] = {s, s < 0};
      if (s >= 0) {
        stamp_[s] = ++clock_;
        ++hits_[layer];
      }
    }
    for (int i = 0; i < n; ++i) {
      if (!out[i].miss) continue;
      int victim = -1;
      for (int s = 0; s < n_slots_; ++s) {
        if (layer_[s] < 0) { victim = s; break; }  // an empty slot
        if (stamp_[s] >= batch_start) continue;   // used by this batch
        if (victim < 0 || stamp_[s] < stamp_[victim]) victim = s;
      }
      if (layer_[victim] >= 0) slot_of_[(size_t)layer_[victim] * n_experts_ + expert_[victim]] = -1;
      layer_[victim] = layer;
      expert_[victim] = experts[i];
      slot_of_[(size_t)layer * n_experts_ + experts[i]] = victim;
      stamp_[victim] = ++clock_;
      out[i].slot = victim;
      ++misses_[layer];
    }
    return out;
  }

 private:
  int n_slots_ = 0, n_experts_ = 0;
  std::vector<int> layer_, expert_;
  std::vector<uint64_t> stamp_;
  std::vector<int> slot_of_;
  std::vector<int64_t> hits_, misses_;
  uint64_t clock_ = 0;
};

}  // namespace ftmoe
