// Host-side model of the partially resident expert cache (see
// expert_cache.h), plus the C entry points of include/moe_residency.h that
// expose it to tests and tools.
#include "expert_cache.h"

#include <algorithm>
#include <new>

#include "moe_residency.h"

namespace moe {

ExpertCache::ExpertCache(int n_records, int capacity, int spares, CachePolicy policy)
    : row_expert_(capacity + spares, -1),
      row_pub_(capacity + spares, 0),
      expert_row_(n_records, -1),
      freq_(n_records, 0.0),
      last_use_(n_records, 0),
      guessed_(n_records, 0),
      capacity_(capacity),
      policy_(policy) {}

double ExpertCache::score(int e) const {
  switch (policy_) {
    case kCacheLFU:
      return freq_[e];
    case kCacheLRUFreq:
      return freq_[e] * 1000.0 - (double)(clock_ - last_use_[e]);
    case kCacheLRU:
    default:
      return (double)last_use_[e];
  }
}

void ExpertCache::touch(int e, bool hit) {
  ++clock_;
  last_use_[e] = clock_;
  freq_[e] += 1.0;
  if (hit) {
    ++hits;
    if (guessed_[e]) {
      ++prefetch_used;
      guessed_[e] = 0;
    }
  } else {
    ++misses;
    if (policy_ == kCacheLRUFreq && ++misses_since_decay_ >= 2u * (uint64_t)capacity_) {
      for (double& f : freq_) f *= 0.75;
      misses_since_decay_ = 0;
      ++decays;
    }
  }
}

ExpertCache::Txn ExpertCache::next(const std::vector<int>& remaining, bool first) {
  (void)first;
  Txn t;
  std::vector<int> miss;
  for (int e : remaining) {
    if (expert_row_[e] >= 0) {
      t.experts.push_back(e);
      t.rows.push_back(expert_row_[e]);
    } else {
      miss.push_back(e);
    }
  }
  std::sort(miss.begin(), miss.end());
  const int published_n = (int)std::count(row_pub_.begin(), row_pub_.end(), 1);
  const int room = capacity_ - (int)t.experts.size();
  const int nm = std::min((int)miss.size(), std::max(0, room));
  // victims: published experts outside the group, lowest score first (then
  // lower row), enough that the published set stays within capacity
  const int nvict = std::max(0, published_n + nm - capacity_);
  std::vector<char> in_group(expert_row_.size(), 0);
  for (int e : t.experts) in_group[e] = 1;
  std::vector<int> cand;
  for (int r = 0; r < rows(); ++r)
    if (row_pub_[r] && !in_group[row_expert_[r]]) cand.push_back(r);
  std::stable_sort(cand.begin(), cand.end(), [&](int a, int b) {
    const double sa = score(row_expert_[a]), sb = score(row_expert_[b]);
    if (sa != sb) return sa < sb;
    return a < b;
  });
  for (int i = 0; i < nvict && i < (int)cand.size(); ++i) t.evict.emplace_back(row_expert_[cand[i]], cand[i]);
  // rows of the loads: unpublished rows first (lowest index), then the
  // victims' rows (reused once the consumers reading them have retired)
  std::vector<int> free_rows;
  for (int r = 0; r < rows(); ++r)
    if (!row_pub_[r]) free_rows.push_back(r);
  for (const auto& v : t.evict) free_rows.push_back(v.second);
  for (int i = 0; i < nm; ++i) {
    t.experts.push_back(miss[i]);
    t.rows.push_back(free_rows[i]);
    t.loads.emplace_back(miss[i], free_rows[i]);
  }
  return t;
}

void ExpertCache::publish(const Txn& t) { publish(t, false); }

void ExpertCache::publish(const Txn& t, bool prefetch) {
  for (const auto& v : t.evict) {
    guessed_[v.first] = 0;
    expert_row_[v.first] = -1;
    row_pub_[v.second] = 0;
    row_expert_[v.second] = -1;
  }
  for (const auto& l : t.loads) {
    row_expert_[l.second] = l.first;
    row_pub_[l.second] = 1;
    expert_row_[l.first] = l.second;
    if (prefetch) guessed_[l.first] = 1;
  }
  if (prefetch) prefetched += t.loads.size();
  evictions += t.evict.size();
  if (!t.loads.empty() || !t.evict.empty()) ++generation_;
}

void ExpertCache::abort(const Txn& t) {
  for (const auto& l : t.loads)
    if (!row_pub_[l.second]) row_expert_[l.second] = -1;
}

}  // namespace moe

// ---------------------------------------------------------------- C API
struct moe_expert_cache {
  moe::ExpertCache c;
  moe_expert_cache(int n, int cap, int sp, moe::CachePolicy p) : c(n, cap, sp, p) {}
};

extern "C" {

moe_expert_cache_t* moe_expert_cache_create(int32_t n_records, int32_t capacity, int32_t spare_rows,
                                            int32_t policy) {
  if (n_records < 1 || capacity < 1 || spare_rows < 0 || policy < MOE_CACHE_LRU || policy > MOE_CACHE_LRU_FREQ)
    return nullptr;
  return new (std::nothrow) moe_expert_cache(n_records, capacity, spare_rows, (moe::CachePolicy)policy);
}

int32_t moe_expert_cache_access(moe_expert_cache_t* cache, const int32_t* demanded, int32_t n, int32_t abort_txn,
                                int32_t* txn_of, int32_t* row_of, int32_t* hit, int32_t* n_txn) {
  if (!cache || (n > 0 && (!demanded || !txn_of || !row_of || !hit)) || !n_txn || n < 0) return -1;
  moe::ExpertCache& c = cache->c;
  std::vector<int> d(demanded, demanded + n);
  std::sort(d.begin(), d.end());
  for (int i = 0; i < n; ++i)
    if (d[i] < 0 || d[i] >= c.n_records() || (i && d[i] == d[i - 1])) return -1;
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::vector<int> h(n);
  for (int i = 0; i < n; ++i) {
    h[i] = c.row_of(d[i]) >= 0 ? 1 : 0;
    c.touch(d[i], h[i] != 0);
  }
  std::vector<int> remaining = d;
  int ti = 0;
  while (!remaining.empty()) {
    const moe::ExpertCache::Txn t = c.next(remaining, ti == 0);
    if (t.experts.empty()) return -1;
    if (ti == abort_txn) {
      c.abort(t);
      *n_txn = ti;
      return 1;
    }
    c.publish(t);
    for (size_t j = 0; j < t.experts.size(); ++j) {
      const int i = (int)(std::lower_bound(d.begin(), d.end(), t.experts[j]) - d.begin());
      txn_of[i] = ti;
      row_of[i] = t.rows[j];
      hit[i] = h[i];
    }
    std::vector<int> rest;
    for (int e : remaining)
      if (std::find(t.experts.begin(), t.experts.end(), e) == t.experts.end()) rest.push_back(e);
    remaining.swap(rest);
    ++ti;
  }
  // report in the caller's order
  std::vector<int32_t> a(txn_of, txn_of + n), b(row_of, row_of + n), cc(hit, hit + n);
  for (int i = 0; i < n; ++i) {
    const int k = (int)(std::lower_bound(d.begin(), d.end(), demanded[i]) - d.begin());
    txn_of[i] = a[k];
    row_of[i] = b[k];
    hit[i] = cc[k];
  }
  *n_txn = ti;
  return 0;
}

int32_t moe_expert_cache_row_of(const moe_expert_cache_t* cache, int32_t expert) {
  if (!cache || expert < 0 || expert >= cache->c.n_records()) return -1;
  return cache->c.row_of(expert);
}

int32_t moe_expert_cache_stats(const moe_expert_cache_t* cache, uint64_t* out5) {
  if (!cache || !out5) return -1;
  out5[0] = cache->c.hits;
  out5[1] = cache->c.misses;
  out5[2] = cache->c.evictions;
  out5[3] = cache->c.generation();
  out5[4] = cache->c.decays;
  return 0;
}

int32_t moe_expert_cache_prefetch(moe_expert_cache_t* cache, const int32_t* guessed, int32_t n) {
  if (!cache || n < 0 || (n > 0 && !guessed)) return -1;
  std::vector<int> g(guessed, guessed + n);
  std::sort(g.begin(), g.end());
  for (int i = 0; i < n; ++i)
    if (g[i] < 0 || g[i] >= cache->c.n_records() || (i && g[i] == g[i - 1])) return -1;
  const moe::ExpertCache::Txn t = cache->c.plan_prefetch(g);
  cache->c.publish(t, true);
  return (int32_t)t.loads.size();
}

int32_t moe_expert_cache_prefetch_stats(const moe_expert_cache_t* cache, uint64_t* out2) {
  if (!cache || !out2) return -1;
  out2[0] = cache->c.prefetched;
  out2[1] = cache->c.prefetch_used;
  return 0;
}

void moe_expert_cache_destroy(moe_expert_cache_t* cache) { delete cache; }

}  // extern "C"
