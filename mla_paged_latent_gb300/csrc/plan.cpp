// Host split-KV planner.
//
// The pages fix the planner's inputs and outputs — cache_seqlens, query tokens
// per request x heads and topk in; tile-scheduler metadata and per-request
// split counts out ("Implementation:Sgl project Sglang Flash MLA", Signature
// and I/O Contract of get_mla_metadata) — but not the rule. This file's rule:
// requests are cut into KV blocks of 64 rows, each costing 1 plus a fixed 3 per
// split (a unit's Q load, pipeline fill and epilogue; 3 measured best of 1-4); partitions (one per SM, or per SM group when a request needs several
// query-row groups) are filled greedily in request order up to a payload, the
// smallest one from ceil(total cost / partitions) up with which the fill needs
// no more partitions than there are; a request that does not fit is split. The
// include/mla_decode.h comment on mla_decode_plan states the rule in full.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "mla_kernels.h"

namespace mla {

constexpr int kFixedCost = 3;

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

PlanResult make_plan(const int32_t* seqlens, int batch, int sq, int heads, int topk, int min_splits, int num_sms) {
  PlanResult res;
  const int groups = static_cast<int>(cdiv(static_cast<int64_t>(sq) * heads, kGroupRows));
  const int parts = std::max(1, num_sms / groups);
  std::vector<int> nb(batch);
  int64_t total = 0;
  int min_nb = 1 << 30;  // fewest blocks of a request with at least min_splits blocks
  for (int b = 0; b < batch; ++b) {
    const int64_t K = topk > 0 ? topk : std::max<int32_t>(seqlens[b], 0);
    nb[b] = static_cast<int>(std::max<int64_t>(1, cdiv(K, kBlockRows)));
    total += nb[b] + kFixedCost;
    if (nb[b] >= min_splits) min_nb = std::min(min_nb, nb[b]);
  }
  // Greedy fill in request order; returns the number of partitions it opens and,
  // if out != nullptr, their sched rows and per-request split counts.
  std::vector<int> sp(batch);  // per-request split counts of the current fill (reused)
  auto fill = [&](int64_t payload, std::vector<int32_t>* out, std::vector<int>* splits) -> int {
    int count = 0, b = 0, blk = 0;
    std::fill(sp.begin(), sp.end(), 0);
    while (b < batch) {
      int64_t budget = payload;
      const int begin_b = b, begin_blk = blk, first_split = sp[b];
      while (b < batch && budget > kFixedCost) {
        const int64_t remain = nb[b] - blk;
        const int64_t take = std::min<int64_t>(remain, budget - kFixedCost);
        budget -= take + kFixedCost;
        sp[b] += 1;
        blk += static_cast<int>(take);
        if (blk == nb[b]) {
          ++b;
          blk = 0;
        } else {
          break;
        }
      }
      ++count;
      if (out) {
        const int32_t row[8] = {begin_b, begin_blk, b, blk, first_split, 0, 0, 0};
        out->insert(out->end(), row, row + 8);
      }
    }
    if (splits) *splits = sp;
    return count;
  };
  // the smallest payload from ceil(total / parts) up that needs at most `parts`
  // partitions; ceil(total / parts) + 2 * kFixedCost always does (every closed
  // partition is charged at least payload - kFixedCost and each continuation adds
  // kFixedCost), so the search ends within 2 * kFixedCost + 1 fills
  const int64_t p0 = std::max<int64_t>(cdiv(total, parts), kFixedCost + 1);
  int64_t payload = p0;
  while (payload < p0 + 2 * kFixedCost && fill(payload, nullptr, nullptr) > parts) ++payload;
  if (min_splits > 1 && min_nb < (1 << 30)) {
    // segments of at most s blocks cut n >= min_nb blocks into ceil(n / s) >= min_splits
    // pieces when s <= (min_nb - 1) / (min_splits - 1)
    const int64_t cap = std::max(1, (min_nb - 1) / (min_splits - 1)) + kFixedCost;
    if (cap < payload) {
      // several waves of partitions: the payload up to the cap with the fewest
      // waves x payload (ties: the larger payload)
      int64_t best = cap, best_span = -1;
      for (int64_t p = cap; p > kFixedCost && p > cap - 64; --p) {
        const int64_t span = cdiv(fill(p, nullptr, nullptr), parts) * p;
        if (best_span < 0 || span < best_span) {
          best = p;
          best_span = span;
        }
      }
      payload = best;
    }
  }
  std::vector<int> splits;
  fill(payload, &res.sched, &splits);
  res.num_splits.assign(batch + 1, 0);
  for (int i = 0; i < batch; ++i) {
    res.num_splits[i + 1] = res.num_splits[i] + splits[i];
    res.max_splits = std::max(res.max_splits, splits[i]);
  }
  res.partitions = static_cast<int>(res.sched.size() / 8);
  res.groups = groups;
  res.total_splits = res.num_splits[batch];
  return res;
}

}  // namespace mla
