"""Failure detection on the GPU, without a GPU fault: a bounded wait that runs out.

With the test flag MLA_DECODE_TEST_WITHHOLD_SIGNAL the decode kernel withholds
the signal that its first score tile is complete. The softmax's wait gives up
after ~2 s, every role leaves its loop (the MMA issuers first wait for their own
MMAs, the producer for its copies), the call completes and the workspace status
word reports MLA_STATUS_WAIT_TIMEOUT. The same CUDA context then runs a normal
decode that matches the oracle."""
import time

import numpy as np
import pytest
import torch

import mla_paged_latent_gb300 as mla
import workloads
from gpu_helpers import DeviceWorkload, assert_close, bound_for, oracle_decode

pytestmark = pytest.mark.gpu

MLA_STATUS_WAIT_TIMEOUT = 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_paged_latent_gb300 import build
    build.build()
    mla.load()


@pytest.mark.parametrize("cfg,single_sm", [
    (lambda: workloads.dsv3(batch=3, seqlens=(64, 700, 1300), len_dist="fixed", new_rows=False), False),
    (lambda: workloads.dsv3(batch=3, seqlens=(64, 700, 1300), len_dist="fixed", new_rows=False), True),
    (lambda: workloads.dsv4(batch=3, seqlens=(64, 700, 1300), len_dist="fixed", new_rows=False), False),
], ids=["bf16_cta_pair", "bf16_tma_single_sm", "fp8_converters"])
def test_wait_timeout_is_reported_and_context_survives(cfg, single_sm):
    w = workloads.generate(cfg())
    c = w.cfg
    d = DeviceWorkload(w)
    p = d.make_plan()
    t0 = time.monotonic()
    mla.mla_decode(d.q, d.kv, c.layout, c.page_size, d.bt, d.sl, c.sq, c.sm_scale, d.sched, d.ns, p.num_partitions,
                   p.total_splits, d.ws, d.out, d.lse, sink=d.sink, single_sm=single_sm, _test_withhold_signal=True)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    status = int(d.ws[:4].cpu().numpy().view(np.uint32)[0])
    assert status & MLA_STATUS_WAIT_TIMEOUT, f"status {status:#x}: the withheld signal must be reported"
    assert elapsed < 60, f"the call took {elapsed:.1f} s"
    with pytest.raises(mla.MlaError):
        mla.mla_read_status(d.ws)  # reports the device check and clears the word
    assert mla.mla_read_status(d.ws) == 0
    # the context is still usable: a normal decode matches the oracle
    mla.mla_workspace_init(d.ws)
    out, lse = d.run(write=False)
    ref_out, ref_lse = oracle_decode(w)
    assert_close(out, lse, ref_out, ref_lse, "after a timed-out call", bound_for(c.layout))
