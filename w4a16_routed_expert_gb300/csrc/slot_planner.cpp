// Slot planner of the partially resident expert pool (host-only C++), plus
// the C entry points of include/moe_residency.h.
#include "slot_planner.h"

#include <algorithm>
#include <new>

#include "moe_residency.h"

namespace moe {

SlotPlanner::SlotPlanner(int n_records, int num_slots)
    : slot_expert_(num_slots, -1), expert_slot_(n_records, -1), last_use_(num_slots, 0) {}

namespace {

// Slots ordered as eviction candidates: empty first, then least recently
// used, then lower slot index.
std::vector<int> victim_order(const std::vector<int>& slot_expert, const std::vector<uint64_t>& last_use,
                              const std::vector<char>& protect) {
  std::vector<int> v;
  for (int s = 0; s < (int)slot_expert.size(); ++s)
    if (!protect[s]) v.push_back(s);
  std::stable_sort(v.begin(), v.end(), [&](int a, int b) {
    const bool ea = slot_expert[a] < 0, eb = slot_expert[b] < 0;
    if (ea != eb) return ea;
    if (last_use[a] != last_use[b]) return last_use[a] < last_use[b];
    return a < b;
  });
  return v;
}

}  // namespace

std::vector<SlotPlanner::Wave> SlotPlanner::plan(const std::vector<int>& demanded) const {
  std::vector<Wave> waves;
  std::vector<int> se = slot_expert_;
  std::vector<uint64_t> lu = last_use_;
  uint64_t clk = clock_;
  std::vector<int> misses;
  Wave w0;
  std::vector<char> protect(se.size(), 0);
  for (int e : demanded) {
    const int s = expert_slot_[e];
    if (s >= 0) {
      w0.experts.push_back(e);
      w0.slots.push_back(s);
      protect[s] = 1;
    } else {
      misses.push_back(e);
    }
  }
  size_t mi = 0;
  {
    const std::vector<int> cand = victim_order(se, lu, protect);
    for (size_t c = 0; c < cand.size() && mi < misses.size(); ++c, ++mi) {
      const int s = cand[c];
      w0.experts.push_back(misses[mi]);
      w0.slots.push_back(s);
      w0.loads.emplace_back(misses[mi], s);
      se[s] = misses[mi];
    }
  }
  ++clk;
  for (int s : w0.slots) lu[s] = clk;
  if (!w0.experts.empty()) waves.push_back(w0);
  while (mi < misses.size()) {
    Wave w;
    const std::vector<char> none(se.size(), 0);
    const std::vector<int> cand = victim_order(se, lu, none);
    for (size_t c = 0; c < cand.size() && mi < misses.size(); ++c, ++mi) {
      const int s = cand[c];
      w.experts.push_back(misses[mi]);
      w.slots.push_back(s);
      w.loads.emplace_back(misses[mi], s);
      se[s] = misses[mi];
    }
    ++clk;
    for (int s : w.slots) lu[s] = clk;
    waves.push_back(w);
  }
  return waves;
}

std::vector<SlotPlanner::Wave> SlotPlanner::plan_fixed_order(const std::vector<int>& demanded) const {
  // One expert per step, LRU replacement; consecutive steps are grouped into
  // waves of at most num_slots experts whose slots are all distinct.
  std::vector<Wave> waves;
  std::vector<int> se = slot_expert_, es = expert_slot_;
  std::vector<uint64_t> lu = last_use_;
  uint64_t clk = clock_;
  Wave cur;
  std::vector<char> in_wave(se.size(), 0);
  for (int e : demanded) {
    int s = es[e];
    bool load = false;
    if (s < 0) {
      s = (int)(std::min_element(lu.begin(), lu.end()) - lu.begin());
      for (int t = 0; t < (int)se.size(); ++t)
        if (se[t] < 0) {
          s = t;
          break;
        }
      load = true;
    }
    if (in_wave[s]) {
      waves.push_back(cur);
      cur = Wave();
      std::fill(in_wave.begin(), in_wave.end(), 0);
    }
    if (load) {
      if (se[s] >= 0) es[se[s]] = -1;
      se[s] = e;
      es[e] = s;
      cur.loads.emplace_back(e, s);
    }
    cur.experts.push_back(e);
    cur.slots.push_back(s);
    in_wave[s] = 1;
    lu[s] = ++clk;
  }
  if (!cur.experts.empty()) waves.push_back(cur);
  return waves;
}

void SlotPlanner::commit(const Wave& w) {
  ++clock_;
  for (const auto& ld : w.loads) {
    const int e = ld.first, s = ld.second;
    if (slot_expert_[s] >= 0) expert_slot_[slot_expert_[s]] = -1;
    slot_expert_[s] = e;
    expert_slot_[e] = s;
  }
  for (size_t i = 0; i < w.slots.size(); ++i) last_use_[w.slots[i]] = clock_;
}

void SlotPlanner::invalidate(int slot) {
  if (slot < 0 || slot >= (int)slot_expert_.size()) return;
  if (slot_expert_[slot] >= 0) expert_slot_[slot_expert_[slot]] = -1;
  slot_expert_[slot] = -1;
  last_use_[slot] = 0;
}

}  // namespace moe

struct moe_slot_planner {
  moe::SlotPlanner p;
  moe_slot_planner(int n, int s) : p(n, s) {}
};

extern "C" {

moe_slot_planner_t* moe_slot_planner_create(int32_t n_records, int32_t num_slots) {
  if (n_records < 1 || num_slots < 1) return nullptr;
  return new (std::nothrow) moe_slot_planner(n_records, num_slots);
}

int32_t moe_slot_planner_plan(moe_slot_planner_t* planner, const int32_t* demanded, int32_t n, int32_t policy,
                              int32_t* wave_of, int32_t* slot_of, int32_t* hit, int32_t* n_waves) {
  if (!planner || n < 0 || (n > 0 && (!demanded || !wave_of || !slot_of || !hit)) || !n_waves) return -1;
  if (policy != MOE_PLAN_HITS_FIRST && policy != MOE_PLAN_FIXED_ORDER_LRU) return -1;
  moe::SlotPlanner& P = planner->p;
  std::vector<int> d(demanded, demanded + n);
  std::sort(d.begin(), d.end());
  for (int i = 0; i < n; ++i) {
    if (d[i] < 0 || d[i] >= P.n_records()) return -1;
    if (i && d[i] == d[i - 1]) return -1;
  }
  std::vector<int> was_resident(n);
  for (int i = 0; i < n; ++i) was_resident[i] = P.slot_of(d[i]) >= 0;
  const auto waves = policy == MOE_PLAN_HITS_FIRST ? P.plan(d) : P.plan_fixed_order(d);
  for (size_t wi = 0; wi < waves.size(); ++wi) {
    const auto& w = waves[wi];
    for (size_t j = 0; j < w.experts.size(); ++j) {
      const int idx = (int)(std::lower_bound(d.begin(), d.end(), w.experts[j]) - d.begin());
      wave_of[idx] = (int32_t)wi;
      slot_of[idx] = w.slots[j];
      hit[idx] = 1;
    }
    for (const auto& ld : w.loads) {
      const int idx = (int)(std::lower_bound(d.begin(), d.end(), ld.first) - d.begin());
      hit[idx] = 0;
    }
    P.commit(w);
  }
  for (int i = 0; i < n; ++i)
    if (!was_resident[i]) hit[i] = 0;
  *n_waves = (int32_t)waves.size();
  return 0;
}

int32_t moe_slot_planner_slot_of(const moe_slot_planner_t* planner, int32_t expert) {
  if (!planner || expert < 0 || expert >= planner->p.n_records()) return -1;
  return planner->p.slot_of(expert);
}

void moe_slot_planner_invalidate(moe_slot_planner_t* planner, int32_t slot) {
  if (planner) planner->p.invalidate(slot);
}

void moe_slot_planner_destroy(moe_slot_planner_t* planner) { delete planner; }

}  // extern "C"
