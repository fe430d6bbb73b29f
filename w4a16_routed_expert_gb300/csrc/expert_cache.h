// Host-side model of the partially resident expert cache (pure C++, no CUDA):
// which expert each GPU row holds, which rows are published in the current
// generation, the eviction policy and the counters. The CUDA driver
// (residency.cu) asks it for one forward's transactions, runs the copies and
// the kernels, and reports each transaction as published or aborted.
//
// Horizon RunMap report, "Partial-residency contract": every request works on
// a complete published generation; a miss is loaded into rows that are not
// published (spare rows) and becomes visible only when the whole routed
// group is published as a new generation; a failure before publication
// leaves the old generation authoritative; eviction discards GPU copies.
// F51 Nitro-MoE, "Layer 1 - expert persistence cache": a fixed pool of slots
// with expert_to_slot / slot_to_expert maps, per-slot frequency and
// last-used counters, LRU-FREQ scoring freq * 1000 - age with frequencies
// decayed by 0.75 every 2x capacity misses. moe-stream, "Findings": LRU and
// LFU as the two basic rules.
#pragma once

#include <cstdint>
#include <vector>

namespace moe {

enum CachePolicy { kCacheLRU = 0, kCacheLFU = 1, kCacheLRUFreq = 2 };

class ExpertCache {
 public:
  // One transaction: a routed group computed together (at most `capacity`
  // experts, all resident once it is published).
  struct Txn {
    std::vector<int> experts;               // the group (hits first, then misses in ascending id)
    std::vector<int> rows;                  // the row each expert is read from
    std::vector<std::pair<int, int>> loads; // (expert, row) copies into unpublished rows
    std::vector<std::pair<int, int>> evict; // (expert, row) dropped from the published set
  };

  // rows = capacity + spares; capacity = most experts published at once.
  ExpertCache(int n_records, int capacity, int spares, CachePolicy policy);

  // Transactions of one forward over distinct demanded experts (any order).
  // Plans one transaction at a time against the state the previous ones
  // leave once published (call publish() / abort() in order).
  Txn next(const std::vector<int>& remaining, bool first);

  // Publishes txn as the new generation: its loads become published, its
  // victims leave the published set and their rows become spares.
  void publish(const Txn& t);
  // A transaction that failed before publication: the published set and
  // generation do not change; the rows it was filling become spares again
  // (their contents untrusted).
  void abort(const Txn& t);

  // Accounting of one demanded access (hit or miss) for the policies; a hit
  // on an expert a prefetch loaded counts that guess as used.
  void touch(int expert, bool hit);

  // A prefetch (moe-stream, "Findings": the next layer's router run early on
  // the current state): the guessed experts as one transaction, planned like
  // next() but without counting accesses; publish it with publish(t, true).
  Txn plan_prefetch(const std::vector<int>& guessed) { return next(guessed, false); }
  void publish(const Txn& t, bool prefetch);

  int row_of(int expert) const { return expert_row_[expert]; }        // published row or -1
  int expert_in(int row) const { return row_expert_[row]; }           // -1: spare / empty
  bool published(int row) const { return row_pub_[row] != 0; }
  int rows() const { return (int)row_expert_.size(); }
  int capacity() const { return capacity_; }
  int n_records() const { return (int)expert_row_.size(); }
  uint64_t generation() const { return generation_; }
  CachePolicy policy() const { return policy_; }

  uint64_t hits = 0, misses = 0, evictions = 0, decays = 0;
  uint64_t prefetched = 0, prefetch_used = 0;  // experts loaded by prefetches; of them, demanded while resident

 private:
  double score(int expert) const;  // lower = evicted first
  std::vector<int> row_expert_;    // expert held by a row (published or loaded-and-unpublished), -1 none
  std::vector<char> row_pub_;      // row is published in the current generation
  std::vector<int> expert_row_;    // published row of an expert, -1 none
  std::vector<double> freq_;       // per expert: accesses (LFU) or decayed frequency (LRU-FREQ)
  std::vector<uint64_t> last_use_; // per expert: clock of the last access
  std::vector<char> guessed_;      // per expert: loaded by a prefetch, not demanded since
  uint64_t clock_ = 0;
  uint64_t generation_ = 0;
  uint64_t misses_since_decay_ = 0;
  int capacity_ = 0;
  CachePolicy policy_;
};

}  // namespace moe
