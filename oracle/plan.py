"""Split-KV planner restatement -- TEST INFRASTRUCTURE ONLY (part of the oracle).

The pages fix what the planner returns -- tile-scheduler metadata plus per-request
split information computed from cache_seqlens, the number of query tokens per
request times heads, and topk ("Implementation:Sgl project Sglang Flash MLA",
Signature / I/O Contract of get_mla_metadata) -- but not how it assigns work.
The algorithm below is this project's own choice; the C++ planner in the
library implements the same rule independently and must agree bit for bit.

Rule
----
* A request's query rows (s_q tokens x N heads, token-major) are cut into
  G = ceil(s_q*N / group_rows) groups; each (partition, group) pair is one CTA
  work item, so P = max(1, num_sms // G) partitions share the SMs.
* Request b has nb_b = max(1, ceil(K_b / block_rows)) KV blocks, with
  K_b = topk for sparse decode and cache_seqlens[b] otherwise. An empty request
  keeps one (fully masked) block so that some CTA writes its zero output.
* Cost of a request = nb_b + FIXED (FIXED = 3 block-equivalents of per-split
  overhead). payload = the smallest value p >= p0 = max(ceil(sum cost / P),
  FIXED + 1) for which the greedy fill below opens at most P partitions;
  p0 + 2*FIXED always qualifies (every closed partition is charged at least
  payload - FIXED and each continuation adds FIXED, so (P'-1)(payload - 2*FIXED)
  < sum cost), so only p0 .. p0 + 2*FIXED are tried.
* With min_splits = k > 1: segments of at most s blocks cut a request of n
  blocks into >= ceil(n / s) pieces, which is >= k when s <= (n - 1) // (k - 1).
  So with n_min = the fewest blocks of a request that has >= k blocks, the cap
  is max(1, (n_min - 1) // (k - 1)) + FIXED. If the cap is below the payload
  above (the plan then needs several waves of P partitions), the payload is the
  value p in (cap - 64, cap], p > FIXED, with the smallest ceil(count(p) / P) * p,
  ties going to the larger p (count(p) = partitions the fill opens with p).
* Partitions are filled greedily in request order: each segment taken costs its
  blocks + FIXED; a partition that cannot hold the rest of a request takes
  (budget - FIXED) blocks of it and closes. Partitions are opened until every
  block is covered (their number may differ from P).
* sched[p] = (begin_req, begin_blk, end_req, end_blk, first_split, 0, 0, 0):
  the partition covers the (request, block) pairs from (begin_req, begin_blk)
  up to, not including, (end_req, end_blk) in request-major order;
  first_split is the split index of its first segment within begin_req.
* num_splits is the prefix sum over requests of the number of segments that
  cover each request (length B + 1); total splits = num_splits[B].
"""
from __future__ import annotations

import numpy as np

FIXED_COST = 3


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def plan_split_kv(cache_seqlens, sq: int, nheads: int, topk: int, min_splits: int, num_sms: int,
                  block_rows: int = 64, group_rows: int = 64):
    seqlens = [int(x) for x in np.asarray(cache_seqlens).ravel()]
    B = len(seqlens)
    G = _cdiv(sq * nheads, group_rows)
    P = max(1, num_sms // G)
    nb = [max(1, _cdiv(topk if topk > 0 else L, block_rows)) for L in seqlens]
    total = sum(n + FIXED_COST for n in nb)

    def fill(payload):
        sched, splits = [], [0] * B
        b, blk = 0, 0
        while b < B:
            budget = payload
            begin_b, begin_blk, first_split = b, blk, splits[b]
            while b < B and budget > FIXED_COST:
                remain = nb[b] - blk
                take = min(remain, budget - FIXED_COST)
                budget -= take + FIXED_COST
                splits[b] += 1
                blk += take
                if blk == nb[b]:
                    b, blk = b + 1, 0
                else:
                    break
            sched.append((begin_b, begin_blk, b, blk, first_split, 0, 0, 0))
        return sched, splits

    p0 = max(_cdiv(total, P), FIXED_COST + 1)
    payload = p0
    while payload < p0 + 2 * FIXED_COST and len(fill(payload)[0]) > P:
        payload += 1
    long_enough = [n for n in nb if n >= min_splits]
    if min_splits > 1 and long_enough:
        cap = max(1, (min(long_enough) - 1) // (min_splits - 1)) + FIXED_COST
        if cap < payload:
            best, best_span = cap, None
            p = cap
            while p > FIXED_COST and p > cap - 64:
                span = _cdiv(len(fill(p)[0]), P) * p
                if best_span is None or span < best_span:
                    best, best_span = p, span
                p -= 1
            payload = best
    sched, splits = fill(payload)

    num_splits = np.zeros(B + 1, dtype=np.int32)
    for i in range(B):
        num_splits[i + 1] = num_splits[i] + splits[i]
    return dict(sched=np.array(sched, dtype=np.int32).reshape(-1, 8), num_splits=num_splits,
                num_partitions=len(sched), groups=G, blocks=np.array(nb, dtype=np.int32),
                payload=payload, total_splits=int(num_splits[B]))


def partition_segments(row, nb):
    """Segments (req, blk_begin, blk_end, split_idx) of one sched row."""
    begin_b, begin_blk, end_b, end_blk, first_split = [int(x) for x in row[:5]]
    segs = []
    r = begin_b
    while r < len(nb) and (r < end_b or (r == end_b and end_blk > 0)):
        lo = begin_blk if r == begin_b else 0
        hi = end_blk if r == end_b else int(nb[r])
        if hi > lo:
            segs.append((r, lo, hi, first_split if r == begin_b else 0))
        r += 1
    return segs
