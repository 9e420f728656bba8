"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every entry point declared in include/*.h; the C++ planner agrees bit
for bit with the oracle's restatement; argument validation rejects bad input
before any device work."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import mla_paged_latent_gb300 as mla
from mla_paged_latent_gb300 import build as mla_build
from oracle.plan import plan_split_kv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.load()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert {"mla_decode_plan", "mla_decode", "mla_kv_write", "mla_combine", "mla_kv_gather"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    # and the binding wraps each of them under the same name
    for name in declared:
        if name != "mla_last_error":
            assert callable(getattr(mla, name)), name


def test_page_bytes(lib):
    assert mla.mla_page_bytes(0, 64) == 73728
    assert mla.mla_page_bytes(1, 64) == 37440
    assert mla.mla_page_bytes(2, 64) == 41600
    with pytest.raises(mla.MlaError):
        mla.mla_page_bytes(1, 48)


@pytest.mark.parametrize("seed", range(25))
def test_cpp_planner_matches_oracle(lib, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 160))
    seqlens = rng.integers(0, 40000, B).astype(np.int32)
    seqlens[rng.random(B) < 0.1] = 0
    sq = int(rng.choice([1, 2, 4, 8]))
    heads = int(rng.choice([16, 64, 128]))
    topk = int(rng.choice([0, 0, 2048, 100]))
    ms = int(rng.choice([1, 4]))
    sms = int(rng.choice([148, 152, 16]))
    ref = plan_split_kv(seqlens, sq, heads, topk, ms, sms)
    got = mla.mla_decode_plan(seqlens, sq, heads, topk, ms, sms)
    assert got.num_partitions == ref["num_partitions"]
    assert np.array_equal(got.sched, ref["sched"])
    assert np.array_equal(got.num_splits, ref["num_splits"])
    assert got.groups == ref["groups"] and got.total_splits == ref["total_splits"]
    R = sq * heads
    assert got.workspace_bytes >= 256 + got.total_splits * R * 513 * 4


def test_workload_plans_match_oracle(lib):
    import workloads
    for name in ("tiny", "dsv3", "dsv4", "verify"):
        w = workloads.generate(workloads.CONFIGS[name](new_rows=False))
        c = w.cfg
        ref = plan_split_kv(w.seqlens, c.sq, c.heads, c.topk, c.min_splits, 152)
        got = mla.mla_decode_plan(w.seqlens, c.sq, c.heads, c.topk, c.min_splits, 152)
        assert np.array_equal(got.sched, ref["sched"]) and np.array_equal(got.num_splits, ref["num_splits"])


def test_plan_capacity_and_validation(lib):
    info = mla._PlanInfo()
    sl = np.array([100, 200], np.int32)
    sched = np.zeros((1, 8), np.int32)
    ns = np.zeros(3, np.int32)
    rc = lib.mla_decode_plan(sl.ctypes.data_as(ctypes.c_void_p), 2, 1, 128, 0, 1, 152,
                             sched.ctypes.data_as(ctypes.c_void_p), 1, ns.ctypes.data_as(ctypes.c_void_p),
                             ctypes.byref(info))
    assert rc == -6 and info.num_partitions > 1  # MLA_ERR_CAPACITY with info filled
    assert b"capacity" in lib.mla_last_error()
    bad = np.array([-1], np.int32)
    rc = lib.mla_decode_plan(bad.ctypes.data_as(ctypes.c_void_p), 1, 1, 16, 0, 1, 152, None, 0, None,
                             ctypes.byref(info))
    assert rc == -1


def _decode_rc(lib, **over):
    """Call mla_decode with fake (never dereferenced) device pointers; validation
    rejects the arguments before any CUDA call is made."""
    fake = ctypes.c_void_p(0x100000)
    args = dict(q=fake, kv=fake, layout=0, num_pages=4, page_size=64, bt=fake, max_pages=2, sl=fake, batch=2, sq=1,
                heads=16, scale=0.1, sink=None, idx=None, topk=0, causal=0, sched=fake, ns=fake, parts=1, splits=2,
                ws=ctypes.c_void_p(0x100000), wsb=1 << 30, out=fake, lse=fake)
    args.update(over)
    return lib.mla_decode(args["q"], args["kv"], args["layout"], args["num_pages"], args["page_size"], args["bt"],
                          args["max_pages"], args["sl"], args["batch"], args["sq"], args["heads"], args["scale"],
                          args["sink"], args["idx"], args["topk"], args["causal"], args["sched"], args["ns"],
                          args["parts"], args["splits"], args["ws"], args["wsb"], args["out"], args["lse"], 0, None)


def test_decode_argument_validation(lib):
    assert _decode_rc(lib, q=None) == -1
    assert _decode_rc(lib, layout=7) == -1
    assert _decode_rc(lib, page_size=48) == -2
    assert _decode_rc(lib, page_size=4) == -2
    assert _decode_rc(lib, topk=16) == -1                       # topk without indices
    assert _decode_rc(lib, q=ctypes.c_void_p(0x100008)) == -1   # misaligned q
    assert _decode_rc(lib, wsb=100) == -3                       # workspace too small
    assert _decode_rc(lib, sq=64, heads=128) == -2              # too many rows per request
    assert _decode_rc(lib, splits=1) == -1                      # total_splits < batch
    assert _decode_rc(lib, idx=ctypes.c_void_p(0x100000), topk=64, sq=2, heads=16) == -2
    assert _decode_rc(lib, ws=ctypes.c_void_p(0x100010)) == -1   # workspace not 256-B aligned
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        assert _decode_rc(lib, scale=bad) == -1                 # sm_scale must be positive and finite
    assert _decode_rc(lib, wsb=100) == -3
    assert b"workspace" in lib.mla_last_error()                 # the message names the failed check


def test_combine_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    assert lib.mla_combine(None, fake, fake, 2, 16, 16, None, fake, fake, None) == -1      # NULL part_out
    assert lib.mla_combine(fake, fake, fake, 2, 20, 16, None, fake, fake, None) == -1      # rows % heads != 0
    assert lib.mla_combine(fake, fake, fake, 0, 16, 16, None, fake, fake, None) == -1      # batch < 1
    assert lib.mla_combine(ctypes.c_void_p(0x100004), fake, fake, 2, 16, 16, None, fake, fake, None) == -1


def test_kv_write_and_gather_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    assert lib.mla_kv_write(fake, fake, 4, fake, 9, 4, 64, None, None) == -1
    assert lib.mla_kv_write(fake, fake, 4, fake, 1, 4, 12, None, None) == -1
    assert lib.mla_kv_write(fake, fake, 0, None, 1, 4, 64, None, None) == 0   # nothing to do
    assert lib.mla_kv_gather(fake, 0, 4, 64, None, 2, 10, fake, None) == -1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        mla.mla_kv_write(torch.zeros(4, 576, dtype=torch.bfloat16), torch.zeros(4, dtype=torch.int32),
                         torch.zeros(2, 100, dtype=torch.uint8), 0, 16)


def test_next_row_entry_points_validation(lib):
    """The fused write, the combine + projection / inverse RoPE and the window-run entry points
    reject bad arguments before any device work."""
    fake = ctypes.c_void_p(0x100000)
    odd = ctypes.c_void_p(0x100004)
    # mla_kv_write_norm_rope(raw, slots, positions, w, eps, freqs, max_pos, n, kv, layout, num_pages, ps, status,
    #                        stream)
    assert lib.mla_kv_write_norm_rope(fake, fake, fake, fake, 1e-6, fake, 8, 0, None, 0, 4, 64, None, None) == 0
    assert lib.mla_kv_write_norm_rope(fake, fake, None, fake, 1e-6, fake, 8, 4, fake, 0, 4, 64, None, None) == -1
    assert lib.mla_kv_write_norm_rope(fake, fake, fake, fake, -1.0, fake, 8, 4, fake, 0, 4, 64, None, None) == -1
    assert lib.mla_kv_write_norm_rope(fake, fake, fake, fake, 1e-6, fake, 0, 4, fake, 0, 4, 64, None, None) == -1
    assert lib.mla_kv_write_norm_rope(fake, fake, fake, odd, 1e-6, fake, 8, 4, fake, 1, 4, 64, None, None) == -1
    assert lib.mla_kv_write_norm_rope(fake, fake, fake, fake, 1e-6, fake, 8, 4, fake, 5, 4, 64, None, None) == -1
    # mla_combine_v_up(part_out, part_lse, ns, batch, sq, heads, sink, w, out, lse, o_v, status, stream)
    assert lib.mla_combine_v_up(fake, fake, fake, 2, 1, 16, None, None, fake, fake, fake, None, None) == -1
    assert lib.mla_combine_v_up(fake, None, fake, 2, 1, 16, None, fake, fake, fake, fake, None, None) == -1
    assert lib.mla_combine_v_up(None, None, fake, 0, 1, 16, None, fake, fake, fake, fake, None, None) == -1
    assert lib.mla_combine_v_up(None, None, fake, 2, 1, 16, None, odd, fake, fake, fake, None, None) == -1
    # mla_combine_inv_rope(part_out, part_lse, ns, batch, sq, heads, sink, pos, freqs, max_pos, rope0, out, lse, s)
    assert lib.mla_combine_inv_rope(None, None, fake, 2, 1, 64, None, fake, fake, 10, 450, fake, fake, None) == -1
    assert lib.mla_combine_inv_rope(None, None, fake, 2, 1, 64, None, fake, fake, 10, 452, fake, fake, None) == -1
    assert lib.mla_combine_inv_rope(None, None, fake, 2, 1, 64, None, None, fake, 10, 448, fake, fake, None) == -1
    assert lib.mla_combine_inv_rope(None, None, fake, 2, 1, 64, None, fake, fake, 0, 448, fake, fake, None) == -1
    # mla_swa_plan(kv_indices, lengths, T, topk, ps, step, runs, stream)
    assert lib.mla_swa_plan(fake, None, 4, 128, 64, 2, fake, None) == -1
    assert lib.mla_swa_plan(fake, None, 4, 128, 48, 1, fake, None) == -1
    assert lib.mla_swa_plan(fake, None, 4, 128, 64, 1, odd, None) == -1
    assert lib.mla_swa_plan(fake, None, 0, 128, 64, 1, fake, None) == -1
    # mla_decode_runs(q, kv, layout, num_pages, ps, runs, window, batch, sq, heads, scale, sink, sched, ns,
    #                 parts, splits, ws, ws_bytes, out, lse, flags, stream)
    assert lib.mla_decode_runs(fake, fake, 1, 4, 64, None, 128, 2, 1, 64, 0.1, None, fake, fake, 1, 2, fake,
                               1 << 20, fake, fake, 0, None) == -1
    assert lib.mla_decode_runs(fake, fake, 1, 4, 64, odd, 128, 2, 1, 64, 0.1, None, fake, fake, 1, 2, fake,
                               1 << 20, fake, fake, 0, None) == -1
    assert lib.mla_decode_runs(fake, fake, 1, 4, 64, fake, 0, 2, 1, 64, 0.1, None, fake, fake, 1, 2, fake,
                               1 << 20, fake, fake, 0, None) == -1
    assert lib.mla_decode_runs(fake, fake, 1, 4, 64, fake, 128, 2, 2, 16, 0.1, None, fake, fake, 1, 2, fake,
                               1 << 20, fake, fake, 0, None) == -2          # several tokens need heads % 64 == 0


def test_sparse_prefill_rejects_bad_arguments(lib):
    """mla_sparse_prefill validates its arguments on the host before any CUDA call
    (returns MLA_ERR_INVALID_ARG = -1): missing index list or max_logits, the
    SKIP_COMBINE flag (its split maxima need the combine), empty sizes, misaligned
    max_logits."""
    fake = ctypes.c_void_p(0x100000)

    def rc(**kw):
        a = dict(q=fake, kv=fake, s_kv=100, idx=fake, topk=16, T=2, N=16, scale=0.1, sched=fake, ns=fake, parts=1,
                 splits=2, ws=fake, wsb=1 << 20, out=fake, mx=fake, lse=fake, flags=0)
        a.update(kw)
        return lib.mla_sparse_prefill(a["q"], a["kv"], a["s_kv"], a["idx"], a["topk"], a["T"], a["N"], a["scale"],
                                      a["sched"], a["ns"], a["parts"], a["splits"], a["ws"], a["wsb"], a["out"],
                                      a["mx"], a["lse"], a["flags"], None)

    assert rc(idx=None) == -1
    assert rc(mx=None) == -1
    assert rc(flags=1) == -1 and b"SKIP_COMBINE" in lib.mla_last_error()
    assert rc(s_kv=0) == -1
    assert rc(topk=0) == -1
    assert rc(T=0) == -1
    assert rc(mx=ctypes.c_void_p(0x100002)) == -1
