"""Pins of the split-KV planner restatement (oracle/plan.py).

The pages fix only the planner's interface (cache_seqlens, query tokens x
heads, topk -> tile-scheduler metadata and per-request split counts;
"Implementation:Sgl project Sglang Flash MLA", get_mla_metadata); the rule is
this project's own. It is pinned by a hand-worked example and by invariants
any correct plan must satisfy.
"""
import numpy as np
import pytest

from oracle.plan import FIXED_COST, partition_segments, plan_split_kv


def test_hand_worked_example():
    # seqlens (100, 300, 0, 64, 1000), 128 heads x 1 token -> 2 groups of 64 rows; 8 SMs -> 4 partitions
    # blocks (2, 5, 1, 1, 16), FIXED 3: costs (5, 8, 4, 4, 19), total 40, p0 = ceil(40/4) = 10
    # payload 10: [req0 2 | req1 2], [req1 3 | req2 1], [req3 1 | req4 3], [req4 7], [req4 6] -> 5 > 4
    # payload 11: [req0 2 | req1 3], [req1 2 | req2 1], [req3 1 | req4 4], [req4 8], [req4 4] -> 5 > 4
    # payload 12: p0 req0 (2 blocks, budget 12-5=7), req1 takes 7-3=4 blocks -> closes
    #             p1 req1 block 4 (12-4=8), req2 (8-4=4), req3 (4-4=0) -> closes
    #             p2 req4 takes 12-3=9 blocks; p3 req4 blocks 9..16 = 7 -> 4 partitions: payload 12
    p = plan_split_kv([100, 300, 0, 64, 1000], 1, 128, 0, 1, 8)
    assert p["groups"] == 2 and p["payload"] == 12
    assert list(p["blocks"]) == [2, 5, 1, 1, 16]
    assert p["sched"][:, :5].tolist() == [[0, 0, 1, 4, 0], [1, 4, 4, 0, 1], [4, 0, 4, 9, 0], [4, 9, 5, 0, 1]]
    assert list(p["num_splits"]) == [0, 1, 3, 4, 5, 7]
    segs = [partition_segments(r, p["blocks"]) for r in p["sched"]]
    assert segs == [[(0, 0, 2, 0), (1, 0, 4, 0)], [(1, 4, 5, 1), (2, 0, 1, 0), (3, 0, 1, 0)], [(4, 0, 9, 0)],
                    [(4, 9, 16, 1)]]


def _check_invariants(p, seqlens, topk, min_splits):
    nb = p["blocks"]
    B = len(seqlens)
    cover = [np.zeros(int(n), np.int32) for n in nb]
    split_seen = [[] for _ in range(B)]
    for row in p["sched"]:
        segs = partition_segments(row, nb)
        assert segs, "empty partition"
        cost = sum(hi - lo + FIXED_COST for _, lo, hi, _ in segs)
        assert cost <= p["payload"]
        for r, lo, hi, sidx in segs:
            cover[r][lo:hi] += 1
            split_seen[r].append((lo, sidx))
    for b in range(B):
        assert np.all(cover[b] == 1), f"request {b} not covered exactly once"
        seen = sorted(split_seen[b])
        assert [s for _, s in seen] == list(range(len(seen)))       # split ids 0..n-1 in KV order
        assert p["num_splits"][b + 1] - p["num_splits"][b] == len(seen)
        if min_splits > 1 and nb[b] >= min_splits:
            assert len(seen) >= min_splits
    assert p["num_splits"][0] == 0 and np.all(np.diff(p["num_splits"]) >= 1)
    assert p["total_splits"] == p["num_splits"][-1]


@pytest.mark.parametrize("seed", range(20))
def test_invariants_random(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 140))
    seqlens = rng.integers(0, 20000, B)
    seqlens[rng.random(B) < 0.1] = 0
    sq = int(rng.choice([1, 2, 4]))
    heads = int(rng.choice([16, 64, 128]))
    topk = int(rng.choice([0, 0, 512, 2048]))
    ms = int(rng.choice([1, 1, 4]))
    sms = int(rng.choice([8, 148, 152]))
    p = plan_split_kv(seqlens, sq, heads, topk, ms, sms)
    _check_invariants(p, seqlens, topk, ms)


def test_sparse_config_forces_four_splits():
    p = plan_split_kv([65536] * 64, 1, 128, 2048, 4, 152)
    _check_invariants(p, [65536] * 64, 2048, 4)
    assert all(p["num_splits"][b + 1] - p["num_splits"][b] >= 4 for b in range(64))


@pytest.mark.parametrize("seed", range(10))
def test_partitions_never_exceed_sm_groups(seed):
    rng = np.random.default_rng(500 + seed)
    for _ in range(200):
        B = int(rng.integers(1, 200))
        sl = rng.integers(0, 40000, B)
        sq = int(rng.choice([1, 2, 4]))
        h = int(rng.choice([16, 64, 128]))
        sms = int(rng.choice([8, 40, 148, 152]))
        topk = int(rng.choice([0, 0, 2048]))
        p = plan_split_kv(sl, sq, h, topk, 1, sms)
        assert p["num_partitions"] <= max(1, sms // p["groups"])


def test_balanced_for_uniform_lengths():
    p = plan_split_kv([4096] * 152, 1, 64, 0, 1, 152)
    assert p["num_partitions"] <= 152 and p["total_splits"] <= 2 * 152
