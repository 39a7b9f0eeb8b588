// Micro-batch / rank balancing of libtpa (tpa_balance, tpa_packing_metrics).
//
// Blog post "AReaL 序列打包算法 FFD 与 KK" (micro-batch load balancing for RL
// training): weighted items (packed trees, or sequences) are split into
// groups (micro-batches or data-parallel ranks) either by First Fit
// Decreasing — heaviest item first, into the lightest group that still has
// room, a new group when none has — or by the Karmarkar-Karp largest
// differencing method for k-way partitions (Korf, "Multi-Way Number
// Partitioning", IJCAI 2009), which falls back to FFD when a group ends up
// over the capacity.  The packing metrics of the post (spread, imbalance
// ratio, standard deviation, coefficient of variation, utilization, wasted
// tokens) describe a result.
//
// Data structures: FFD keeps the groups in an ordered set keyed by (load,
// creation index), so the lightest group is the first element and the only
// candidate (every other group is at least as heavy).  KK keeps partial
// partitions in a binary heap keyed by (spread, creation id); a set is a
// singly linked list of items (head, tail in a shared next[] array), so
// merging two states costs O(k log k) whatever the set sizes.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <new>
#include <queue>
#include <set>
#include <utility>
#include <vector>

#include "tpa.h"
#include "internal.h"

namespace {

int check_args(const int64_t* w, int32_t n, int64_t capacity, int32_t min_groups, int32_t divisor) {
  if (!w || n < 1 || capacity < 1 || min_groups < 1 || divisor < 1) return TPA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    if (w[i] <= 0) return TPA_ERR_INVALID_ARG;
    if (w[i] > capacity) return TPA_ERR_SEQ_TOO_LONG;
  }
  return TPA_OK;
}

// Items heaviest first; equal weights keep input order.
std::vector<int32_t> heaviest_first(const int64_t* w, int32_t n) {
  std::vector<int32_t> order(n);
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return w[a] > w[b]; });
  return order;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// One FFD pass with `need` groups opened first; returns the group count.
int32_t ffd_once(const int64_t* w, const std::vector<int32_t>& order, int64_t capacity, int32_t need,
                 int32_t* group_of) {
  std::set<std::pair<int64_t, int32_t>> by_load;  // (load, group)
  std::vector<int64_t> load;
  for (int32_t i : order) {
    int32_t g = -1;
    if (int32_t(load.size()) >= need && !by_load.empty()) {
      const auto lightest = by_load.begin();
      if (lightest->first + w[i] <= capacity) {
        g = lightest->second;
        by_load.erase(lightest);
      }
    }
    if (g < 0) {
      g = int32_t(load.size());
      load.push_back(0);
    }
    load[g] += w[i];
    by_load.emplace(load[g], g);
    group_of[i] = g;
  }
  return int32_t(load.size());
}

int ffd(const int64_t* w, int32_t n, int64_t capacity, int32_t min_groups, int32_t divisor, int32_t* group_of,
        int32_t* n_groups) {
  const std::vector<int32_t> order = heaviest_first(w, n);
  int64_t need = min_groups;
  for (;;) {
    if (need > n) return TPA_ERR_INVALID_ARG;  // more groups required than items
    const int32_t g = ffd_once(w, order, capacity, int32_t(need), group_of);
    if (g >= min_groups && g % divisor == 0) {
      *n_groups = g;
      return TPA_OK;
    }
    need = round_up(std::max<int64_t>(need, g), divisor);
  }
}

struct KkSet {
  int64_t sum;
  int32_t head, tail;  // item list in next[]; -1 when empty
};

struct KkState {
  int64_t spread;
  int32_t id;  // creation order: items first (input order), then merges
  int32_t slot;
};

struct KkOrder {  // priority_queue top = largest spread, then smallest id
  bool operator()(const KkState& a, const KkState& b) const {
    return a.spread != b.spread ? a.spread < b.spread : a.id > b.id;
  }
};

int kk(const int64_t* w, int32_t n, int64_t capacity, int32_t min_groups, int32_t divisor, int32_t* group_of,
       int32_t* n_groups, bool* over) {
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) total += w[i];
  int64_t k = std::max<int64_t>(min_groups, (total + capacity - 1) / capacity);
  k = round_up(k, divisor);
  if (k > n) return TPA_ERR_INVALID_ARG;
  const int32_t K = int32_t(k);
  std::vector<int32_t> next(n, -1);
  std::vector<std::vector<KkSet>> slots;  // the sets of every live state
  slots.reserve(size_t(2) * n);
  std::priority_queue<KkState, std::vector<KkState>, KkOrder> heap;
  auto spread_of = [](const std::vector<KkSet>& s) {
    int64_t lo = s[0].sum, hi = s[0].sum;
    for (const KkSet& x : s) {
      lo = std::min(lo, x.sum);
      hi = std::max(hi, x.sum);
    }
    return hi - lo;
  };
  for (int32_t i = 0; i < n; ++i) {
    std::vector<KkSet> s(K, KkSet{0, -1, -1});
    s[0] = KkSet{w[i], i, i};
    heap.push(KkState{spread_of(s), i, int32_t(slots.size())});
    slots.push_back(std::move(s));
  }
  int32_t next_id = n;
  std::vector<int32_t> ad(K), bd(K);
  while (heap.size() > 1) {
    const KkState a = heap.top();
    heap.pop();
    const KkState b = heap.top();
    heap.pop();
    std::vector<KkSet>& sa = slots[a.slot];
    std::vector<KkSet>& sb = slots[b.slot];
    for (int32_t j = 0; j < K; ++j) ad[j] = bd[j] = j;
    std::stable_sort(ad.begin(), ad.end(), [&](int32_t x, int32_t y) { return sa[x].sum > sa[y].sum; });
    std::stable_sort(bd.begin(), bd.end(), [&](int32_t x, int32_t y) { return sb[x].sum < sb[y].sum; });
    std::vector<KkSet> m(K);
    for (int32_t j = 0; j < K; ++j) {  // i-th largest of a with i-th smallest of b
      const KkSet& x = sa[ad[j]];
      const KkSet& y = sb[bd[j]];
      KkSet z{x.sum + y.sum, x.head, x.tail};
      if (y.head >= 0) {
        if (z.head < 0) {
          z.head = y.head;
        } else {
          next[z.tail] = y.head;
        }
        z.tail = y.tail;
      }
      m[j] = z;
    }
    std::vector<KkSet>().swap(sa);
    std::vector<KkSet>().swap(sb);
    heap.push(KkState{spread_of(m), next_id++, int32_t(slots.size())});
    slots.push_back(std::move(m));
  }
  const std::vector<KkSet>& fin = slots[heap.top().slot];
  std::vector<int32_t> order(K);
  for (int32_t j = 0; j < K; ++j) order[j] = j;
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return fin[x].sum > fin[y].sum; });
  *over = false;
  for (int32_t g = 0; g < K; ++g) {
    const KkSet& s = fin[order[g]];
    if (s.sum > capacity) *over = true;
    for (int32_t i = s.head; i >= 0; i = (i == s.tail) ? -1 : next[i]) group_of[i] = g;
  }
  *n_groups = K;
  return TPA_OK;
}

}  // namespace

extern "C" int tpa_balance(const int64_t* weights, int32_t n, int64_t capacity, int32_t min_groups,
                           int32_t groups_divisor, int32_t algorithm, int32_t* group_of, int32_t* n_groups,
                           int32_t* algorithm_used) {
  TPA_NVTX_RANGE("tpa_balance");
  if (!group_of || !n_groups) return TPA_ERR_INVALID_ARG;
  if (algorithm != TPA_BALANCE_FFD && algorithm != TPA_BALANCE_KK) return TPA_ERR_INVALID_ARG;
  int rc = check_args(weights, n, capacity, min_groups, groups_divisor);
  if (rc != TPA_OK) return rc;
  try {
    if (algorithm == TPA_BALANCE_KK) {
      bool over = false;
      rc = kk(weights, n, capacity, min_groups, groups_divisor, group_of, n_groups, &over);
      if (rc != TPA_OK || !over) {
        if (algorithm_used) *algorithm_used = TPA_BALANCE_KK;
        return rc;
      }
    }
    if (algorithm_used) *algorithm_used = TPA_BALANCE_FFD;
    return ffd(weights, n, capacity, min_groups, groups_divisor, group_of, n_groups);
  } catch (const std::bad_alloc&) {
    return TPA_ERR_NO_MEMORY;
  }
}

extern "C" int tpa_packing_metrics(const int64_t* weights, int32_t n, const int32_t* group_of, int32_t n_groups,
                                   int64_t capacity, tpa_packing_metrics_t* out) {
  if (!weights || !group_of || !out || n < 1 || n_groups < 1 || capacity < 1) return TPA_ERR_INVALID_ARG;
  try {
    std::vector<int64_t> load(n_groups, 0);
    for (int32_t i = 0; i < n; ++i) {
      if (group_of[i] < 0 || group_of[i] >= n_groups) return TPA_ERR_INVALID_ARG;
      load[group_of[i]] += weights[i];
    }
    int64_t total = 0, lo = load[0], hi = load[0];
    for (int64_t x : load) {
      total += x;
      lo = std::min(lo, x);
      hi = std::max(hi, x);
    }
    const double mean = double(total) / n_groups;
    double var = 0.0;
    for (int64_t x : load) var += (double(x) - mean) * (double(x) - mean);
    const double sd = std::sqrt(var / n_groups);
    out->n_groups = n_groups;
    out->pad_ = 0;
    out->total = total;
    out->max_load = hi;
    out->min_load = lo;
    out->spread = hi - lo;
    out->wasted = int64_t(n_groups) * capacity - total;
    out->mean = mean;
    out->std_dev = sd;
    out->cv = mean > 0 ? sd / mean : 0.0;
    out->imbalance_ratio = mean > 0 ? double(hi) / mean : 0.0;
    out->utilization = double(total) / (double(n_groups) * double(capacity));
    return TPA_OK;
  } catch (const std::bad_alloc&) {
    return TPA_ERR_NO_MEMORY;
  }
}
