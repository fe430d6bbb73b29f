// Slot planner of the partially resident expert pool (host-only C++).
#pragma once

#include <cstdint>
#include <utility>
#include <vector>

namespace moe {

class SlotPlanner {
 public:
  struct Wave {
    std::vector<int> experts;                // experts computed in this wave (ascending id)
    std::vector<int> slots;                  // their slots
    std::vector<std::pair<int, int>> loads;  // (expert, slot) copies to issue before the wave
  };

  SlotPlanner(int n_records, int num_slots);

  // Plans the waves for a set of distinct demanded experts (ascending id).
  // Does not change the state; apply with commit() wave by wave.
  std::vector<Wave> plan(const std::vector<int>& demanded) const;
  // Fixed-order LRU baseline: visit demanded experts in ascending id,
  // replacing the least recently used slot on a miss.
  std::vector<Wave> plan_fixed_order(const std::vector<int>& demanded) const;

  void commit(const Wave& w);
  void invalidate(int slot);
  int slot_of(int expert) const { return expert_slot_[expert]; }
  int expert_in(int slot) const { return slot_expert_[slot]; }
  int num_slots() const { return (int)slot_expert_.size(); }
  int n_records() const { return (int)expert_slot_.size(); }

 private:
  std::vector<int> slot_expert_;
  std::vector<int> expert_slot_;
  std::vector<uint64_t> last_use_;
  uint64_t clock_ = 0;
};

}  // namespace moe
