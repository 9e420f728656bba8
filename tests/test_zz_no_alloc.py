"""The no-allocation decode entry point (mla_decode_static_workspace).

Callers that cannot allocate device memory — a host whose memory pool owns the
whole GPU budget and forbids cudaMalloc by extensions, a latency-critical loop
that must not pay for an allocation, a language binding without CUDA allocation —
use this variant, which runs the same decode on a workspace the library keeps
in a static device array. These tests call it through the C ABI and check it
against mla_decode with a caller-allocated workspace, on two calls in a row, and
the second call's result against the oracle.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_paged_latent_gb300 as mla
import workloads
from gpu_helpers import DeviceWorkload, assert_close, bound_for, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from mla_paged_latent_gb300 import build
    build.build()
    return mla.load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_static(lib, d, out, lse, status):
    c = d.w.cfg
    topk = 0 if d.idx is None else int(d.idx.shape[-1])
    return lib.mla_decode_static_workspace(
        _p(d.q), _p(d.kv), c.layout, d.kv.shape[0], c.page_size, _p(d.bt), d.bt.shape[1], _p(d.sl), c.batch, c.sq,
        c.heads, float(c.sm_scale), _p(d.sink), _p(d.idx), topk, int(c.causal), _p(d.sched), _p(d.ns),
        d.plan.num_partitions, d.plan.total_splits, _p(out), _p(lse), _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = {
    # few partitions -> requests split -> the static workspace holds split partials
    "dsv3_split": (lambda: workloads.dsv3(batch=5, seqlens=(1, 65, 700, 2000, 3001), len_dist="fixed"), 8),
    "dsv4_sink": (lambda: workloads.dsv4(batch=4, seqlens=(0, 100, 900, 2500), len_dist="fixed"), 3),
    "verify_causal": (lambda: workloads.verify(batch=2, seqlens=(30, 700), len_dist="fixed"), 16),
}


@pytest.mark.parametrize("name", list(CASES))
def test_static_workspace_matches_mla_decode(lib, name):
    make, sms = CASES[name]
    w = workloads.generate(make())
    d = DeviceWorkload(w)
    d.kv_write()
    plan = d.make_plan(num_sms=sms)
    assert plan.workspace_bytes <= mla.STATIC_WORKSPACE_BYTES
    d.decode()                      # the existing entry point, caller-allocated workspace
    assert mla.mla_read_status(d.ws) == 0
    torch.cuda.synchronize()
    ref_out = d.out.float().cpu().numpy().astype(np.float64)
    ref_lse = d.lse.cpu().numpy().astype(np.float64)
    T, N = w.q.shape[0], w.cfg.heads
    for call in range(2):           # two calls in a row share (and reuse) the static array
        out = torch.full((T, N, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), 0x7FFF, dtype=torch.int32, device="cuda")
        rc = _call_static(lib, d, out, lse, status)
        assert rc == 0, lib.mla_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got_out = out.float().cpu().numpy().astype(np.float64)
        got_lse = lse.cpu().numpy().astype(np.float64)
        assert_close(got_out, got_lse, ref_out, ref_lse, f"{name} call {call}", bound_for(w.cfg.layout))
    # and the oracle agrees with the static-workspace result
    o_out, o_lse = oracle_decode(w)
    assert_close(got_out, got_lse, o_out, o_lse, f"{name} vs the oracle", bound_for(w.cfg.layout))


def test_static_workspace_rejects_oversized_plans(lib):
    # 32 tokens x 128 heads per request and many splits need more than the static array
    seqlens = np.full(4, 4096, np.int32)
    plan = mla.mla_decode_plan(seqlens, 32, 128, 0, 8, 152)
    assert plan.workspace_bytes > mla.STATIC_WORKSPACE_BYTES
    fake = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(fake.data_ptr())
    rc = lib.mla_decode_static_workspace(p, p, 0, 1, 64, p, 1, p, 4, 32, 128, 0.1, None, None, 0, 1, p, p,
                                         plan.num_partitions, plan.total_splits, p, p, None, None)
    assert rc == -3
    assert b"static workspace" in lib.mla_last_error()
