"""fp8 rows over the whole e4m3 code range and ue8m0 scale bytes far from 2^0.

The seeded workloads draw NoPE codes from quantiles of N(0,1) (|x| below about 2.7)
and scale bytes from 123..131. Here the fp8 cache bytes of a seeded workload are
rewritten so that every row holds every e4m3 code (subnormals and +-448 included;
the two NaN codes only where the test says so) in a per-row shuffled order, and
the group scale bytes are drawn from a wide range. The gather is compared with the
oracle bit for bit; the decode with small NoPE queries (the dequantised keys decide
the scores) within the output bounds, and the decode with the scores carried by the
RoPE part alone (the values pass through the softmax-weighted mean) within 1e-2 of
the weighted mean of |V|, the scale of its fp32 accumulation error.

Layouts: the fp8 row of the "MLA" API page of HALOps (mla_attention, kv_cache: 448
float8_e4m3fn NoPE elements, ue8m0 scale per 64, 64 bf16 RoPE) and the 512-element
variant of the supported-config paragraph of the same page.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mla_paged_latent_gb300 as mla
import oracle
import workloads
from gpu_helpers import DeviceWorkload, assert_close, oracle_decode

pytestmark = pytest.mark.gpu


def _rewrite_fp8(w, rng, scale_lo, scale_hi, with_nan):
    """A copy of w whose fp8 NoPE bytes cycle through all codes and whose scale bytes
    are uniform in [scale_lo, scale_hi]."""
    c = w.cfg
    layout, ps = c.layout, c.page_size
    rb, nope = workloads._ROW_BYTES[layout], workloads._NOPE[layout]
    ng = nope // 64
    codes = np.arange(256, dtype=np.uint8)
    if not with_nan:
        codes = codes[(codes & 0x7F) != 0x7F]
    kv = w.kv_cache.copy()
    pages = kv.shape[0]
    rows = kv[:, :ps * rb].reshape(pages, ps, rb)
    for p in range(pages):
        for j in range(ps):
            rows[p, j, :nope] = np.resize(rng.permutation(codes), nope)
    kv[:, :ps * rb] = rows.reshape(pages, ps * rb)
    slots = kv[:, ps * rb:ps * rb + ps * 8].reshape(pages, ps, 8)
    slots[:, :, :ng] = rng.integers(scale_lo, scale_hi + 1, size=(pages, ps, ng), dtype=np.uint8)
    kv[:, ps * rb:ps * rb + ps * 8] = slots.reshape(pages, ps * 8)
    return dataclasses.replace(w, kv_cache=kv, new_rows=None, new_slots=None)


def _scaled_q(w, nope_scale, rope_scale):
    """q with its NoPE part scaled by nope_scale and its RoPE part by rope_scale (bf16 bits)."""
    q = w.q.astype(np.uint32) << 16
    x = q.view(np.float32).copy()
    nope = workloads._NOPE[w.cfg.layout]
    x[..., :nope] *= np.float32(nope_scale)
    x[..., nope:] *= np.float32(rope_scale)
    bits = (x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16  # round to nearest even
    return bits.astype(np.uint16)


@pytest.mark.parametrize("layout", [1, 2])
def test_kv_gather_all_codes_wide_scales(layout):
    # scale bytes 20..234 (2^-107 .. 2^107): every dequantised value stays a normal fp32
    # number (2^-9 * 2^-107 .. 448 * 2^107); the two NaN codes gather to NaN
    w = workloads.generate(workloads.dsv4(batch=2, seqlens=(130, 77), len_dist="fixed", page_size=64, layout=layout))
    w = _rewrite_fp8(w, np.random.default_rng(71 + layout), 20, 234, with_nan=True)
    kv = torch.from_numpy(w.kv_cache).cuda()
    for b in range(2):
        L = int(w.seqlens[b])
        out = torch.empty(L, workloads._DQK[layout], dtype=torch.float32, device="cuda")
        mla.mla_kv_gather(kv, layout, 64, torch.from_numpy(w.block_table[b]).cuda(), L, out)
        got = out.cpu().numpy().astype(np.float64)
        ref = oracle.kv_gather(w.kv_cache, layout, 64, w.block_table[b], L)
        nan = np.isnan(ref)
        assert nan.any(), "the NaN codes must be present"
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])
        # the scales reach far beyond 2^+-30 in both directions
        fin = np.abs(ref[~nan])
        assert fin.max() > 1e30 and fin[fin > 0].min() < 1e-30


@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("mode", ["rope_scores", "nope_scores"])
def test_decode_all_codes_wide_scales(layout, mode):
    cfg = workloads.dsv4(batch=2, seqlens=(300, 650), len_dist="fixed", page_size=64, layout=layout, heads=16,
                         sink=False)
    w = workloads.generate(cfg)
    rng = np.random.default_rng(90 + 2 * layout + (mode == "nope_scores"))
    if mode == "rope_scores":
        # q_nope = 0: the scores come from the bf16 RoPE part; the values (dequantised with
        # scale bytes 100..154, i.e. up to 448 * 2^27) enter only the weighted mean
        w = _rewrite_fp8(w, rng, 100, 154, with_nan=False)
        w = dataclasses.replace(w, q=_scaled_q(w, 0.0, 1.0))
    else:
        # small NoPE queries against keys with scale bytes 121..133 (up to 448 * 2^6): the
        # dequantised keys decide the scores, which stay a few units wide
        w = _rewrite_fp8(w, rng, 121, 133, with_nan=False)
        w = dataclasses.replace(w, q=_scaled_q(w, 2.0 ** -13, 1.0))
    d = DeviceWorkload(w)
    got_out, got_lse = d.run(write=False)
    ref_out, ref_lse = oracle_decode(w, kv=w.kv_cache)
    if mode == "nope_scores":
        assert_close(got_out, got_lse, ref_out, ref_lse, f"layout {layout} {mode}", "scaled")
        return
    _assert_within_mean_abs_v(w, got_out, got_lse, ref_out, ref_lse, 1e3)


def _assert_within_mean_abs_v(w, got_out, got_lse, ref_out, ref_lse, min_peak):
    """Values of both signs far above the outputs: an output element is a weighted mean whose
    terms are up to ~10^6 times larger than the mean itself, so the error of any fp32
    accumulation scales with the mean of |V| under the same weights, not with |out|. That
    mean is the oracle's decode of the same cache with the NoPE sign bits cleared (q_nope =
    0: the weights depend on the RoPE part only)."""
    layout = w.cfg.layout
    nope = workloads._NOPE[layout]
    kv_abs = w.kv_cache.copy()
    rb, ps = workloads._ROW_BYTES[layout], w.cfg.page_size
    rows = kv_abs[:, :ps * rb].reshape(kv_abs.shape[0], ps, rb)
    rows[:, :, :nope] &= 0x7F
    kv_abs[:, :ps * rb] = rows.reshape(kv_abs.shape[0], ps * rb)
    mag, _ = oracle_decode(w, kv=kv_abs)
    assert np.abs(ref_out).max() > min_peak, "the wide scales must reach the outputs"
    assert np.all(np.isfinite(got_out))
    err = np.abs(got_out - ref_out)
    bound = 1e-2 * np.maximum(1.0, np.abs(mag))
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), f"layout {layout}: err {err[worst]:.3g} against mean |V| {mag[worst]:.3g}"
    assert np.abs(got_lse - ref_lse).max() <= 1e-3


def _row_max_raises(w, threshold_log2):
    """Per query row, how often a 64-row tile's largest score (log2 units) exceeds the running
    maximum by more than threshold_log2, the running maximum starting at the first tile's
    and moving only then (scores from the oracle's dequantised rows)."""
    c = w.cfg
    counts = []
    for b in range(c.batch):
        L = int(w.seqlens[b])
        K = oracle.kv_gather(w.kv_cache, c.layout, c.page_size, w.block_table[b], L)
        q = (w.q[b].reshape(-1, w.q.shape[-1]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        s = (q @ K.T) * c.sm_scale * np.log2(np.e)
        for r in range(s.shape[0]):
            m, n = s[r, :64].max(), 0
            for t0 in range(64, L, 64):
                mt = s[r, t0:t0 + 64].max()
                if mt > m + threshold_log2:
                    m, n = mt, n + 1
            counts.append(n)
    return np.array(counts)


@pytest.mark.parametrize("layout", [1, 2])
def test_decode_wide_scales_with_rescales(layout):
    # values up to 448 * 2^31 (scale bytes 150..158) while the RoPE scores grow along the
    # sequence (RoPE part of row j scaled by 1 + j/8, q's RoPE part 2, q_nope 0): every query
    # row's running maximum rises past the single-SM kernel's lazy-rescale threshold (2^64),
    # so O^T is rescaled in TMEM while holding values near 2^64 x 2^10 rows x 2^40, inside
    # fp32 by the kernel's range rule (rows x max|V| < 2^64)
    from test_gpu_parity import _scale_rope_with_position
    cfg = workloads.dsv4(batch=2, seqlens=(640, 1000), len_dist="fixed", page_size=64, layout=layout, heads=64,
                         sink=False)
    w = workloads.generate(cfg)
    w = _rewrite_fp8(w, np.random.default_rng(300 + layout), 150, 158, with_nan=False)
    _scale_rope_with_position(w, workloads._ROW_BYTES[layout], workloads._NOPE[layout], 8)
    q = _scaled_q(w, 0.0, 1.0)
    q[..., -64:] = np.uint16(0x4000)  # bf16 2.0
    w = dataclasses.replace(w, q=q)
    assert _row_max_raises(w, 64.0).min() >= 1
    d = DeviceWorkload(w)
    got_out, got_lse = d.run(write=False)
    ref_out, ref_lse = oracle_decode(w, kv=w.kv_cache)
    _assert_within_mean_abs_v(w, got_out, got_lse, ref_out, ref_lse, 1e6)
