"""GPU parity at the full workload sizes, in the launch configuration bench.py
times (plan over all SMs of the device). The oracle computes a seeded sample of
(token, head) rows one by one; every output is also checked for properties that
hold at any size (finite, zero/-inf exactly for empty rows, status word clear),
and the KV rows written by mla_kv_write are compared byte for byte."""
import numpy as np
import pytest
import torch

import mla_paged_latent_gb300 as mla
import oracle
import workloads
from gpu_helpers import DeviceWorkload, assert_close, bound_for

pytestmark = pytest.mark.gpu

N_SAMPLE = 48


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_paged_latent_gb300 import build
    build.build()
    mla.load()


def _sample(w, rng):
    T, N = w.q.shape[0], w.cfg.heads
    t = rng.integers(0, T, N_SAMPLE).astype(np.int32)
    # always include the longest request's last token and the shortest request's first token
    sq = w.cfg.sq
    t[0] = int(np.argmax(w.seqlens)) * sq + sq - 1
    t[1] = int(np.argmin(w.seqlens)) * sq
    n = rng.integers(0, N, N_SAMPLE).astype(np.int32)
    n[2] = N - 1
    return t, n


@pytest.mark.parametrize("name", ["dsv3", "dsv4", "verify", "sparse"])
def test_full_size_sampled(name):
    w = workloads.generate(workloads.CONFIGS[name]())
    d = DeviceWorkload(w)
    out, lse = d.run()              # kv_write + plan over all SMs + decode (+ combine)
    assert np.all(np.isfinite(out))
    # properties over every row
    if w.indices is None:
        assert np.all(np.isfinite(lse))
    c = w.cfg
    # written rows: byte-exact against the oracle's kv_write, at the written slots
    kv_ref = oracle.kv_write(w.new_rows, w.new_slots, w.kv_cache, c.layout, c.page_size)
    kv_got = d.kv.cpu().numpy()
    rb = {0: 1152, 1: 576, 2: 640}[c.layout]
    for slot in w.new_slots:
        if slot < 0:
            continue
        p, o = divmod(int(slot), c.page_size)
        assert np.array_equal(kv_got[p, o * rb:(o + 1) * rb], kv_ref[p, o * rb:(o + 1) * rb])
        if c.layout != 0:
            so = c.page_size * rb + o * 8
            assert np.array_equal(kv_got[p, so:so + 8], kv_ref[p, so:so + 8])
    rng = np.random.default_rng(1234)
    t, n = _sample(w, rng)
    ref_out, ref_lse = oracle.mla_decode(w.q, kv_ref, c.layout, c.page_size, w.block_table, w.seqlens, c.sq,
                                         c.sm_scale, sink=w.sink, indices=w.indices, causal=c.causal, select=(t, n))
    assert_close(out[t, n], lse[t, n], ref_out, ref_lse, f"{name} full size, sampled rows", bound_for(c.layout))


def test_full_size_combine_v_up_sampled():
    """The DSV3-shaped decode at full size, split by the plan over all SMs, then the combine
    fused with the W_UV up-projection: o_v on sampled (token, head) rows against the oracle's
    decode of those rows, rounded to bf16 and projected by the oracle."""
    w = workloads.generate(workloads.dsv3())
    c = w.cfg
    d = DeviceWorkload(w)
    d.kv_write()
    plan = d.make_plan()
    T, N = w.q.shape[0], c.heads
    mla.mla_decode(d.q, d.kv, c.layout, c.page_size, d.bt, d.sl, c.sq, c.sm_scale, d.sched, d.ns,
                   plan.num_partitions, plan.total_splits, d.ws, d.out, d.lse, skip_combine=True)
    part_out, part_lse = mla.workspace_partials(d.ws, plan.total_splits, c.sq * N)
    rng = np.random.default_rng(77)
    w_uv = torch.from_numpy((rng.standard_normal((N, 512, 128)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    w_bits = w_uv.view(torch.int16).numpy().view(np.uint16)
    o_v = torch.zeros(T, N, 128, dtype=torch.bfloat16, device="cuda")
    split = plan.total_splits > c.batch
    mla.mla_combine_v_up(part_out if split else None, part_lse if split else None, d.ns, c.sq, N, w_uv.cuda(), d.out,
                         d.lse, o_v)
    mla.mla_read_status(d.ws)
    got = o_v.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    kv_ref = oracle.kv_write(w.new_rows, w.new_slots, w.kv_cache, c.layout, c.page_size)
    t, n = _sample(w, rng)
    ref_out, _ = oracle.mla_decode(w.q, kv_ref, c.layout, c.page_size, w.block_table, w.seqlens, c.sq, c.sm_scale,
                                   select=(t, n))
    x_bits = oracle.bf16_encode(ref_out)                     # [S, 512]
    for k in range(len(t)):
        ref = torch.from_numpy(oracle.v_up(x_bits[k][None, None, :], w_bits[n[k]][None])[0, 0].view(np.int16).copy())
        ref = ref.view(torch.bfloat16).double().numpy()
        g = got[t[k], n[k]]
        # the decode's own error carried through W (|o_v| stays well below 2 here): the flat
        # 1e-2 bound of the bf16 decode outputs
        assert_close(g[None], np.zeros(1), ref[None], np.zeros(1), f"o_v row {(int(t[k]), int(n[k]))}")
