"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by
element, on seeded workloads shaped like the decode configurations, at sizes
the oracle finishes in seconds that still span several tiles and ragged tails;
plus the edge cases the method has. Bit-exact where the result is integer or
byte work (KV-row write, page gather); within the stated tolerances otherwise."""
import math

import numpy as np
import pytest
import torch

import mla_paged_latent_gb300 as mla
import oracle
import workloads
from gpu_helpers import DeviceWorkload, assert_close, bf16_tensor, bound_for, oracle_cache, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_paged_latent_gb300 import build
    build.build()
    mla.load()


# ----------------------------------------------------------------------------- KV write / gather (bit-exact)
@pytest.mark.parametrize("layout", [0, 1, 2])
def test_kv_write_bit_exact(layout):
    rng = np.random.default_rng(20 + layout)
    ps = 16
    pb = workloads.page_bytes(layout, ps)
    num_pages = 9
    kv0 = rng.integers(0, 256, (num_pages, pb), dtype=np.uint8)
    n = 70
    re = workloads.row_elems(layout)
    x = (rng.standard_normal((n, re)) * 2.0 ** rng.integers(-30, 30, (n, 1))).astype(np.float32)
    x[0, :64] = 0.0
    x[1, 64:128] = -0.0
    x[2, :] = 1e-12
    x[3, :64] = 448.0
    x[4, :64] = np.linspace(-1000, 1000, 64)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(num_pages * ps)[:n].astype(np.int32)
    slots[5] = -1
    ref = oracle.kv_write(bits, slots, kv0, layout, ps)
    kv = torch.from_numpy(kv0).cuda()
    mla.mla_kv_write(bf16_tensor(bits), torch.from_numpy(slots).cuda(), kv, layout, ps)
    got = kv.cpu().numpy()
    diff = np.argwhere(got != ref)
    assert diff.size == 0, f"{len(diff)} bytes differ, first at {diff[:5].tolist()}"


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_kv_write_nan_inf_and_bad_slots(layout):
    """Rows holding NaN (either sign) and infinities, and slots past the cache. NaN takes no
    part in a group's amax and is stored as the code 0x7F; infinity sets the scale byte to
    254 and is stored as +-448; a slot whose page is past the cache is reported
    (MLA_STATUS_BAD_SLOT) and not written. Bit-exact against the oracle, which skips that slot."""
    rng = np.random.default_rng(40 + layout)
    ps, num_pages, n = 16, 6, 24
    pb = workloads.page_bytes(layout, ps)
    re = workloads.row_elems(layout)
    kv0 = rng.integers(0, 256, (num_pages, pb), dtype=np.uint8)
    x = rng.standard_normal((n, re)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    bits[0, 3] = 0x7FC0                    # +NaN in group 0
    bits[1, 70] = 0xFFC0                   # -NaN in group 1
    bits[2, 5], bits[2, 6] = 0x7F80, 0xFF80  # +inf and -inf in group 0
    bits[3, 0:64] = 0x7FC0                 # a group of NaN only
    bits[4, 200] = 0x7FC1                  # a NaN with a payload
    slots = rng.permutation(num_pages * ps)[:n].astype(np.int32)
    slots[5] = num_pages * ps + 3          # page past the cache
    slots[6] = -1                          # skipped without a report
    ok = slots.copy()
    ok[5] = -1
    ref = oracle.kv_write(bits, ok, kv0, layout, ps)
    kv = torch.from_numpy(kv0).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_kv_write(bf16_tensor(bits), torch.from_numpy(slots).cuda(), kv, layout, ps, status=status)
    got = kv.cpu().numpy()
    assert int(status.item()) == 4
    diff = np.argwhere(got != ref)
    assert diff.size == 0, f"{len(diff)} bytes differ, first at {diff[:5].tolist()}"


def _rope_table(max_pos):
    theta = np.outer(np.arange(max_pos), 10000.0 ** (-np.arange(32) / 32.0))
    f = np.zeros((max_pos, 64), np.float32)
    f[:, 0::2] = np.cos(theta)
    f[:, 1::2] = np.sin(theta)
    return f


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_kv_write_norm_rope(layout):
    """RMSNorm + RoPE + write against the oracle. The kernel normalises in fp32 and the
    oracle in fp64, so a value whose exact result lies within ~1e-6 of a bf16 rounding
    boundary may round the other way: bytes must agree almost everywhere, and every
    written value must lie within one step of its output grid of the oracle's."""
    rng = np.random.default_rng(60 + layout)
    ps, num_pages, n, max_pos = 16, 12, 150, 4096
    pb = workloads.page_bytes(layout, ps)
    re = workloads.row_elems(layout)
    kv0 = rng.integers(0, 256, (num_pages, pb), dtype=np.uint8)
    x = (rng.standard_normal((n, re)) * 2.0 ** rng.integers(-20, 20, (n, 1))).astype(np.float32)
    x[0] = 0.0
    x[1] = 1e-30
    x[5, :64] = 0.0
    raw = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w = torch.from_numpy((1 + 0.2 * rng.standard_normal(512)).astype(np.float32)).to(torch.bfloat16)
    wbits = w.view(torch.int16).numpy().view(np.uint16)
    freqs = _rope_table(max_pos)
    pos = rng.integers(0, max_pos, n).astype(np.int32)
    pos[2], pos[3] = -1, max_pos
    slots = rng.permutation(num_pages * ps)[:n].astype(np.int32)
    slots[4] = -1
    eps = 1e-6
    ref = oracle.kv_write_norm_rope(raw, slots, pos, wbits, eps, freqs, kv0, layout, ps)
    kv = torch.from_numpy(kv0).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_kv_write_norm_rope(bf16_tensor(raw), torch.from_numpy(slots).cuda(), torch.from_numpy(pos).cuda(),
                               bf16_tensor(wbits), eps, torch.from_numpy(freqs).cuda(), kv, layout, ps, status=status)
    got = kv.cpu().numpy()
    assert int(status.item()) == 8, "rows 2 and 3 (positions outside the table) must be reported"
    info = oracle.layout_info(layout, ps)
    rb = info["row_bytes"]
    written = [(r, int(s)) for r, s in enumerate(slots) if s >= 0 and 0 <= pos[r] < max_pos]
    mask = np.zeros_like(kv0, dtype=bool)
    for _, s in written:
        p, o = divmod(s, ps)
        mask[p, o * rb:(o + 1) * rb] = True
        if layout != 0:
            mask[p, ps * rb + o * 8:ps * rb + o * 8 + 8] = True
    assert np.array_equal(got[~mask], ref[~mask]), "bytes outside the written rows changed"
    assert np.array_equal(got[~mask], kv0[~mask])
    frac = np.mean(got[mask] != ref[mask])
    assert frac <= 5e-3, f"{frac:.4f} of the written bytes differ from the oracle"
    nope = info["nope"] if layout != 0 else 0
    for r, s in written:
        p, o = divmod(s, ps)
        g = oracle.decode_row(got, layout, ps, p, o)
        e = oracle.decode_row(ref, layout, ps, p, o)
        # bf16 elements: one bf16 step (2^-7 relative); fp8 groups: one e4m3 step (2^-3 relative),
        # with a floor of 2^-8 of the group's largest magnitude for the subnormal codes
        tol = np.abs(e) * 2.0 ** -7
        for gi in range(nope // 64):
            grp = e[gi * 64:(gi + 1) * 64]
            tol[gi * 64:(gi + 1) * 64] = np.abs(grp) * 2.0 ** -3 + np.abs(grp).max() * 2.0 ** -8
        assert np.all(np.abs(g - e) <= tol + 1e-38), f"row {r}: max excess {np.max(np.abs(g - e) - tol):.3g}"


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_kv_gather_bit_exact(layout):
    cfg = workloads.dsv4(batch=2, seqlens=(77, 150), len_dist="fixed", page_size=16, layout=layout)
    w = workloads.generate(cfg)
    kv = torch.from_numpy(w.kv_cache).cuda()
    for b in range(2):
        L = int(w.seqlens[b])
        out = torch.empty(L, workloads._DQK[layout], dtype=torch.float32, device="cuda")
        mla.mla_kv_gather(kv, layout, 16, torch.from_numpy(w.block_table[b]).cuda(), L, out)
        ref = oracle.kv_gather(w.kv_cache, layout, 16, w.block_table[b], L)
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


# ----------------------------------------------------------------------------- combine
def test_combine_matches_oracle():
    rng = np.random.default_rng(30)
    B, N, sq = 3, 16, 2
    R = sq * N
    nsplit = [3, 1, 5]
    ns = np.concatenate([[0], np.cumsum(nsplit)]).astype(np.int32)
    S = int(ns[-1])
    q = rng.standard_normal((B, R, 576))
    part_out = np.zeros((S, R, 512))
    part_lse = np.zeros((S, R))
    ref_out = np.zeros((B, R, 512))
    ref_lse = np.zeros((B, R))
    sink = rng.standard_normal(N).astype(np.float32)
    for b in range(B):
        for r in range(R):
            rows = rng.standard_normal((int(rng.integers(0, 40)) * nsplit[b] + 1, 576))
            cuts = np.sort(rng.integers(0, rows.shape[0] + 1, nsplit[b] - 1))
            cuts = np.concatenate([[0], cuts, [rows.shape[0]]])
            for s in range(nsplit[b]):
                o, l = oracle.attend(q[b, r], rows[cuts[s]:cuts[s + 1]], 512, 0.05)
                part_out[ns[b] + s, r] = o
                part_lse[ns[b] + s, r] = l
            ref_out[b, r], ref_lse[b, r] = oracle.combine(part_out[ns[b]:ns[b + 1], r], part_lse[ns[b]:ns[b + 1], r],
                                                          sink=float(sink[r % N]))
    out = torch.zeros(B, R, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, R, dtype=torch.float32, device="cuda")
    mla.mla_combine(torch.from_numpy(part_out.astype(np.float32)).cuda(),
                    torch.from_numpy(part_lse.astype(np.float32)).cuda(), torch.from_numpy(ns).cuda(), R, N, out, lse,
                    sink=torch.from_numpy(sink).cuda())
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    # the partials are attention over a few N(0,1) rows, so merged values reach beyond 2, where
    # one bf16 output step alone exceeds 1e-2: the scaled reading of the bound
    for b in (0, 2):
        assert_close(o[b], l[b], ref_out[b], ref_lse[b], f"combine request {b}", "scaled")
    assert np.all(o[1] == 0) and np.all(l[1] == 0)  # single-split request untouched


def _bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("B,sq,N,splits", [(3, 2, 16, (3, 1, 5)), (41, 2, 16, None), (2, 1, 128, (1, 1))])
def test_combine_v_up_matches_oracle(B, sq, N, splits):
    """Split combine + value up-projection against the oracle's combine, bf16 rounding
    and V up-projection (inputs drawn on the host and given to both sides). The second
    case spans two 64-token blocks with a ragged tail; the third has no split at all."""
    rng = np.random.default_rng(32 + B)
    R = sq * N
    T = B * sq
    nsplit = np.array(splits if splits is not None else rng.integers(1, 5, B), dtype=np.int32)
    ns = np.concatenate([[0], np.cumsum(nsplit)]).astype(np.int32)
    S = int(ns[-1])
    part_out = (rng.standard_normal((S, R, 512)) * 2).astype(np.float32)
    part_lse = rng.standard_normal((S, R)).astype(np.float32) * 3
    part_lse[rng.random((S, R)) < 0.05] = -np.inf          # some empty partials
    out_bits = torch.from_numpy(rng.standard_normal((T, N, 512)).astype(np.float32)).to(torch.bfloat16)
    out_bits = out_bits.view(torch.int16).numpy().view(np.uint16)
    lse_in = rng.standard_normal((T, N)).astype(np.float32)
    sink = rng.standard_normal(N).astype(np.float32)
    w_bits = torch.from_numpy((rng.standard_normal((N, 512, 128)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    w_bits = w_bits.view(torch.int16).numpy().view(np.uint16)

    # oracle: merged latent rows (fp64) of split requests, rounded once to bf16; others as given
    x_ref = out_bits.copy()
    merged = {}
    for b in range(B):
        if nsplit[b] < 2:
            continue
        for r in range(R):
            o, l = oracle.combine(part_out[ns[b]:ns[b + 1], r].astype(np.float64),
                                  part_lse[ns[b]:ns[b + 1], r].astype(np.float64), sink=float(sink[r % N]))
            t, n = b * sq + r // N, r % N
            merged[(t, n)] = (o, l)
            x_ref[t, n] = oracle.bf16_encode(o)
    o_ref = _bits_to_f64(oracle.v_up(x_ref, w_bits))

    split = S > B
    out = torch.from_numpy(out_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    lse = torch.from_numpy(lse_in.copy()).cuda()
    o_v = torch.zeros(T, N, 128, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_combine_v_up(torch.from_numpy(part_out).cuda() if split else None,
                         torch.from_numpy(part_lse).cuda() if split else None, torch.from_numpy(ns).cuda(), sq, N,
                         bf16_tensor(w_bits), out, lse, o_v, sink=torch.from_numpy(sink).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_out = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    if merged:
        keys = list(merged)
        # merged values of these synthetic partials reach beyond 2 (one bf16 step > 1e-2): scaled bound
        assert_close(np.stack([got_out[t, n] for t, n in keys]), np.array([got_lse[t, n] for t, n in keys]),
                     np.stack([merged[k][0] for k in keys]), np.array([merged[k][1] for k in keys]), "merged rows",
                     "scaled")
    untouched = np.ones((T, N), bool)
    for (t, n) in merged:
        untouched[t, n] = False
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16)[untouched], out_bits[untouched])
    assert np.array_equal(got_lse[untouched], lse_in[untouched].astype(np.float64))
    # o_v: the GPU merges in fp32, the oracle in fp64, so a merged latent value may round to the
    # neighbouring bf16 (2^-8 of its binade); allow a few such flips per dot product, the fp32
    # accumulation over 512 terms, and half a bf16 step of the result
    x_abs = np.abs(_bits_to_f64(x_ref))
    w_abs = np.abs(_bits_to_f64(w_bits))
    sum_abs = np.einsum("tnl,nlv->tnv", x_abs, w_abs)
    max_term = x_abs.max(axis=2)[:, :, None] * w_abs.max(axis=1)[None, :, :]
    tol = np.abs(o_ref) * 2.0 ** -8 + max_term * 2.0 ** -6 + sum_abs * 1e-4
    got = o_v.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    excess = np.abs(got - o_ref) - tol
    assert np.all(excess <= 0), f"o_v: worst excess {excess.max():.3g} at {np.unravel_index(np.argmax(excess), excess.shape)}"


def test_combine_steps_without_partials_take_rows_as_written():
    """With no partials given, the combine + projection and combine + inverse RoPE take every
    row of out as written, even where num_splits counts several splits (nothing is merged)."""
    rng = np.random.default_rng(99)
    B, N = 4, 64
    T = B
    ns = torch.tensor([0, 3, 4, 6, 7], dtype=torch.int32, device="cuda")   # splits, but no partials
    out_bits = torch.from_numpy(rng.standard_normal((T, N, 512)).astype(np.float32)).to(torch.bfloat16)
    out_bits = out_bits.view(torch.int16).numpy().view(np.uint16)
    w_bits = torch.from_numpy((rng.standard_normal((N, 512, 128)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    w_bits = w_bits.view(torch.int16).numpy().view(np.uint16)
    out = torch.from_numpy(out_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    lse = torch.zeros(T, N, dtype=torch.float32, device="cuda")
    o_v = torch.zeros(T, N, 128, dtype=torch.bfloat16, device="cuda")
    mla.mla_combine_v_up(None, None, ns, 1, N, bf16_tensor(w_bits), out, lse, o_v)
    freqs = _rope_table(16)
    mla.mla_combine_inv_rope(None, None, ns, 1, N, torch.zeros(T, dtype=torch.int32, device="cuda"),
                             torch.from_numpy(freqs).cuda(), out, lse, rope0=448)
    torch.cuda.synchronize()
    # position 0: angle 0, the rotation is the identity
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), out_bits)
    ref = _bits_to_f64(oracle.v_up(out_bits, w_bits))
    got = o_v.float().cpu().numpy().astype(np.float64)
    x_abs = np.abs(_bits_to_f64(out_bits))
    w_abs = np.abs(_bits_to_f64(w_bits))
    tol = np.abs(ref) * 2.0 ** -8 + np.einsum("tnl,nlv->tnv", x_abs, w_abs) * 1e-4
    assert np.all(np.abs(got - ref) <= tol)


@pytest.mark.parametrize("B,sq,N,splits", [(3, 2, 64, (3, 1, 5)), (8, 1, 64, None)])
def test_combine_inv_rope_matches_oracle(B, sq, N, splits):
    """Split combine + inverse RoPE of elements 448..511 (the DSV4 value row) against the
    oracle's combine, bf16 rounding and inverse rotation. Both sides round the merged row
    and the rotated pairs once to bf16 from fp32 (kernel) or fp64 (oracle), so a value may
    land on the neighbouring bf16: nearly all bits agree and every value is within two bf16
    steps of its pair's magnitude (rotated elements) or one step (the others)."""
    rng = np.random.default_rng(70 + B)
    R, T = sq * N, B * sq
    nsplit = np.array(splits if splits is not None else rng.integers(1, 4, B), dtype=np.int32)
    ns = np.concatenate([[0], np.cumsum(nsplit)]).astype(np.int32)
    S = int(ns[-1])
    part_out = (rng.standard_normal((S, R, 512)) * 2).astype(np.float32)
    part_lse = (rng.standard_normal((S, R)) * 3).astype(np.float32)
    out_bits = torch.from_numpy(rng.standard_normal((T, N, 512)).astype(np.float32)).to(torch.bfloat16)
    out_bits = out_bits.view(torch.int16).numpy().view(np.uint16)
    lse_in = rng.standard_normal((T, N)).astype(np.float32)
    sink = rng.standard_normal(N).astype(np.float32)
    max_pos = 5000
    freqs = _rope_table(max_pos)
    pos = rng.integers(0, max_pos, T).astype(np.int32)
    pos[-1] = max_pos + 3  # outside the table: merged but not rotated

    x_ref = out_bits.copy()
    for b in range(B):
        if nsplit[b] < 2:
            continue
        for r in range(R):
            o, _ = oracle.combine(part_out[ns[b]:ns[b + 1], r].astype(np.float64),
                                  part_lse[ns[b]:ns[b + 1], r].astype(np.float64), sink=float(sink[r % N]))
            x_ref[b * sq + r // N, r % N] = oracle.bf16_encode(o)
    ref = oracle.inv_rope(x_ref.reshape(-1, 512), np.repeat(pos, N), freqs, 448).reshape(T, N, 512)

    split = S > B
    out = torch.from_numpy(out_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    lse = torch.from_numpy(lse_in.copy()).cuda()
    mla.mla_combine_inv_rope(torch.from_numpy(part_out).cuda() if split else None,
                             torch.from_numpy(part_lse).cuda() if split else None, torch.from_numpy(ns).cuda(), sq, N,
                             torch.from_numpy(pos).cuda(), torch.from_numpy(freqs).cuda(), out, lse, rope0=448,
                             sink=torch.from_numpy(sink).cuda())
    torch.cuda.synchronize()
    got_bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.mean(got_bits != ref) <= 1e-2
    g, e = _bits_to_f64(got_bits), _bits_to_f64(ref)
    tol = np.abs(e) * 2.0 ** -7
    pair = np.sqrt(e[..., 448::2] ** 2 + e[..., 449::2] ** 2)
    tol[..., 448::2] = pair * 2.0 ** -6
    tol[..., 449::2] = pair * 2.0 ** -6
    excess = np.abs(g - e) - tol
    assert np.all(excess <= 1e-30), f"worst excess {excess.max():.3g} at {np.unravel_index(np.argmax(excess), excess.shape)}"
    unsplit = np.repeat(nsplit < 2, sq)
    assert np.array_equal(got_bits[unsplit][..., :448], out_bits[unsplit][..., :448])


def _windows(rng, T, window, ps, num_slots):
    """Token windows of cache slots: contiguous ranges (ascending or descending, some crossing
    a page), some cut short by a length, and some made of three runs (cut to one row)."""
    idx = np.full((T, window), -1, np.int32)
    lens = np.zeros(T, np.int32)
    steps = np.zeros(T, np.int32)
    for t in range(T):
        n = int(rng.integers(1, window + 1)) if t % 5 else window
        step = 1 if t % 3 else -1
        start = int(rng.integers(n, num_slots - n))
        sl = start + step * np.arange(n)
        if t % 7 == 3 and n > 4:          # three runs
            sl[n // 3:] += 2 * step * ps
            sl[2 * n // 3:] += 2 * step * ps
            sl = np.clip(sl, 0, num_slots - 1)
        idx[t, :n] = sl
        lens[t] = n
        steps[t] = step
    return idx, lens, steps


@pytest.mark.parametrize("ps,step", [(16, 1), (64, -1), (128, 1)])
def test_swa_plan_bit_exact(ps, step):
    rng = np.random.default_rng(80 + ps)
    T, window = 300, 160
    # windows listed both ways: those against `step` fall apart into many runs and are cut
    idx, lens, _ = _windows(rng, T, window, ps, 40 * ps)
    lens[::11] = 0
    ref = oracle.swa_plan(idx, ps, step, lens)
    runs = torch.zeros(T, 4, dtype=torch.int32, device="cuda")
    mla.mla_swa_plan(torch.from_numpy(idx).cuda(), ps, step, runs, topk_lengths=torch.from_numpy(lens).cuda())
    assert np.array_equal(runs.cpu().numpy(), ref)
    ref_nolen = oracle.swa_plan(idx, ps, step)
    mla.mla_swa_plan(torch.from_numpy(idx).cuda(), ps, step, runs)
    assert np.array_equal(runs.cpu().numpy(), ref_nolen)


@pytest.mark.parametrize("layout,heads", [(1, 64), (0, 128), (2, 64)])
def test_decode_runs_matches_oracle(layout, heads):
    """Sliding-window decode: each token over the rows of its runs (from mla_swa_plan on the
    GPU, checked against the oracle's runs first), split by the planner like a top-k decode."""
    ps, window = 64, 96
    cfg = (workloads.dsv4 if layout == 1 else workloads.dsv3)(
        batch=24, seqlens=tuple([300] * 24), len_dist="fixed", page_size=ps, heads=heads, layout=layout)
    w = workloads.generate(cfg)
    c = w.cfg
    rng = np.random.default_rng(90 + layout)
    T = c.batch
    num_slots = w.kv_cache.shape[0] * ps
    idx, lens, steps = _windows(rng, T, window, ps, num_slots)
    # one step per call: ascending windows here, descending ones reversed into ascending order
    idx = np.array([r if steps[t] > 0 else np.concatenate([r[:lens[t]][::-1], r[lens[t]:]])
                    for t, r in enumerate(idx)], np.int32)
    ref_runs = oracle.swa_plan(idx, ps, 1, lens)
    runs = torch.zeros(T, 4, dtype=torch.int32, device="cuda")
    mla.mla_swa_plan(torch.from_numpy(idx).cuda(), ps, 1, runs, topk_lengths=torch.from_numpy(lens).cuda())
    assert np.array_equal(runs.cpu().numpy(), ref_runs)
    plan = mla.mla_decode_plan(np.full(T, window, np.int32), 1, heads, window, 2, 152)
    ws = mla.alloc_workspace(plan.workspace_bytes)
    out = torch.empty(T, heads, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, heads, dtype=torch.float32, device="cuda")
    sink = None if w.sink is None else torch.from_numpy(w.sink).cuda()
    mla.mla_decode_runs(bf16_tensor(w.q), torch.from_numpy(w.kv_cache).cuda(), layout, ps, runs, window, 1,
                        c.sm_scale, torch.from_numpy(plan.sched).cuda(), torch.from_numpy(plan.num_splits).cuda(),
                        plan.num_partitions, plan.total_splits, ws, out, lse, sink=sink)
    mla.mla_read_status(ws)
    ref_out, ref_lse = oracle.decode_runs(w.q, w.kv_cache, layout, ps, ref_runs, c.sm_scale, sink=w.sink)
    assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, f"runs layout {layout}",
                 bound_for(layout))


# ----------------------------------------------------------------------------- decode parity, small shapes
SMALL = {
    "tiny": lambda: workloads.tiny(),
    "dsv3_small": lambda: workloads.dsv3(batch=6, seqlens=(1, 63, 64, 65, 1000, 3001), len_dist="fixed"),
    "dsv4_small": lambda: workloads.dsv4(batch=5, seqlens=(1, 100, 129, 700, 2500), len_dist="fixed"),
    "verify_small": lambda: workloads.verify(batch=3, seqlens=(9, 204, 1004), len_dist="fixed"),
    "sparse_small": lambda: workloads.sparse(batch=3, seqlens=(5000, 300, 7000), topk=300, len_dist="fixed"),
    "dsv3_ps16": lambda: workloads.dsv3(batch=3, seqlens=(37, 130, 700), len_dist="fixed", page_size=16),
    "dsv4_ps256": lambda: workloads.dsv4(batch=3, seqlens=(300, 513, 1500), len_dist="fixed", page_size=256),
    "bf16_sparse": lambda: workloads.dsv3(batch=2, seqlens=(900, 2000), len_dist="fixed", topk=200, pad_frac=0.1),
    "fp8_448_sparse": lambda: workloads.dsv4(batch=2, seqlens=(900, 2000), len_dist="fixed", topk=130, pad_frac=0.1),
    "fp8_512_dense": lambda: workloads.sparse(batch=3, seqlens=(64, 500, 1200), topk=0, min_splits=1, len_dist="fixed"),
    "verify_heads16": lambda: workloads.verify(batch=3, heads=16, seqlens=(4, 70, 300), len_dist="fixed"),
    "tail_nan_bf16": lambda: workloads.dsv3(batch=3, seqlens=(10, 70, 200), len_dist="fixed", tail_fill="nan"),
    "tail_nan_fp8": lambda: workloads.dsv4(batch=3, seqlens=(10, 70, 200), len_dist="fixed", tail_fill="nan"),
    "empty_requests": lambda: workloads.dsv4(batch=4, seqlens=(0, 65, 0, 3), len_dist="fixed", new_rows=False),
    # the smallest page (8 TMA boxes per 64-row slab), empty requests on the bf16 TMA path,
    # a head count that is not a multiple of 16, and the largest query-row count (32 x 128)
    "dsv3_ps8": lambda: workloads.dsv3(batch=3, seqlens=(5, 64, 333), len_dist="fixed", page_size=8),
    "dsv3_ps256": lambda: workloads.dsv3(batch=3, seqlens=(300, 513, 1500), len_dist="fixed", page_size=256),
    "dsv3_sink": lambda: workloads.dsv3(batch=3, seqlens=(100, 700, 1500), len_dist="fixed", sink=True),
    "empty_bf16": lambda: workloads.dsv3(batch=4, seqlens=(0, 65, 0, 3), len_dist="fixed", new_rows=False),
    "heads20": lambda: workloads.dsv3(batch=2, heads=20, seqlens=(100, 700), len_dist="fixed"),
    "rows4096": lambda: workloads.verify(batch=1, sq=32, seqlens=(200,), len_dist="fixed"),
    # a single head (one query row per token): M = 128 with one row used, Q boxes one row high
    "heads1_bf16": lambda: workloads.dsv3(batch=3, heads=1, seqlens=(1, 77, 1300), len_dist="fixed"),
    "heads1_fp8_sink": lambda: workloads.dsv4(batch=3, heads=1, seqlens=(2, 65, 900), len_dist="fixed"),
    # two draft tokens x 64 heads: 128 rows = two query groups, each one token, causal
    "verify_sq2_h64": lambda: workloads.verify(batch=3, sq=2, heads=64, seqlens=(3, 130, 900), len_dist="fixed"),
    # draft tokens with fp8 rows and a sink
    "verify_fp8_sink": lambda: workloads.dsv4(batch=2, sq=3, seqlens=(40, 500), len_dist="fixed", causal=True),
    # top-k lists mostly padding (-1): 3 of 10 tiles hold rows, so split units start on, or
    # consist only of, tiles with no valid row; and lists that are padding throughout
    "sparse_padded": lambda: workloads.sparse(batch=3, seqlens=(5000, 300, 7000), topk=640, pad_frac=0.7,
                                              len_dist="fixed"),
    "sparse_all_pad": lambda: workloads.sparse(batch=2, seqlens=(900, 4000), topk=256, pad_frac=1.0,
                                               len_dist="fixed"),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_small(name):
    w = workloads.generate(SMALL[name]())
    d = DeviceWorkload(w)
    out, lse = d.run()
    if w.new_rows is not None:
        assert np.array_equal(d.kv.cpu().numpy(), oracle_cache(w)), "kv_write bytes differ"
    ref_out, ref_lse = oracle_decode(w)
    assert_close(out, lse, ref_out, ref_lse, name, bound_for(w.cfg.layout))


@pytest.mark.parametrize("name", ["dsv3_small", "dsv4_small", "verify_small", "sparse_small", "sparse_padded"])
@pytest.mark.parametrize("num_sms", [1, 7, 40])
def test_decode_forced_splits(name, num_sms):
    """Few partitions -> long partitions; many partitions -> many splits merged
    by the combine. Every plan must give the same result."""
    w = workloads.generate(SMALL[name]())
    d = DeviceWorkload(w)
    d.kv_write()
    ref_out, ref_lse = oracle_decode(w)
    groups = -(-w.cfg.sq * w.cfg.heads // 64)
    for ms in (1, 6):
        d.make_plan(num_sms=num_sms * groups, min_splits=ms)
        d.decode()
        assert mla.mla_read_status(d.ws) == 0
        out = d.out.float().cpu().numpy().astype(np.float64)
        lse = d.lse.cpu().numpy().astype(np.float64)
        assert_close(out, lse, ref_out, ref_lse, f"{name} sms={num_sms} min_splits={ms} splits={d.plan.total_splits}",
                     bound_for(w.cfg.layout))


PAIR_CASES = ["dsv3_small", "verify_small", "dsv3_ps16", "dsv3_ps8", "dsv3_ps256", "dsv3_sink", "verify_sq2_h64",
              "tail_nan_bf16", "empty_bf16", "rows4096"]


@pytest.mark.parametrize("name", PAIR_CASES)
@pytest.mark.parametrize("min_splits", [1, 5])
def test_decode_pair_and_single_sm_kernels(name, min_splits):
    """bf16 decodes whose query rows come in groups of 128 run on CTA pairs or, with
    MLA_DECODE_SINGLE_SM, on the single-SM kernel: both must agree with the oracle on the
    same plans."""
    w = workloads.generate(SMALL[name]())
    assert (w.cfg.sq * w.cfg.heads) % 128 == 0 and w.cfg.layout == 0
    d = DeviceWorkload(w)
    d.kv_write()
    ref_out, ref_lse = oracle_decode(w)
    d.make_plan(min_splits=min_splits)
    c = w.cfg
    for single in (False, True):
        d.out.fill_(float("nan"))
        mla.mla_decode(d.q, d.kv, c.layout, c.page_size, d.bt, d.sl, c.sq, c.sm_scale, d.sched, d.ns,
                       d.plan.num_partitions, d.plan.total_splits, d.ws, d.out, d.lse, sink=d.sink, causal=c.causal,
                       single_sm=single)
        assert mla.mla_read_status(d.ws) == 0
        out = d.out.float().cpu().numpy().astype(np.float64)
        lse = d.lse.cpu().numpy().astype(np.float64)
        assert_close(out, lse, ref_out, ref_lse, f"{name} {'single-SM' if single else 'pair'} splits={d.plan.total_splits}")


def test_decode_deterministic():
    w = workloads.generate(SMALL["dsv3_small"]())
    d = DeviceWorkload(w)
    a, la = d.run()
    d.decode()
    torch.cuda.synchronize()
    b = d.out.float().cpu().numpy()
    assert np.array_equal(a, b) and np.array_equal(la, d.lse.cpu().numpy())


@pytest.mark.parametrize("heads", [64, 128])
def test_large_score_growth_triggers_rescale(heads):
    """Scores that grow along the sequence force the lazy O rescale: the RoPE scores grow
    to ~200 in log2 units, so every query row's running max rises past the threshold
    (2^64 on the single-SM kernel: 2 to 5 times per row; 2^32 on CTA pairs) between
    tiles. 64 heads run on the single-SM kernel, 128 on CTA pairs."""
    cfg = workloads.dsv3(batch=2, heads=heads, seqlens=(640, 1000), len_dist="fixed", new_rows=False)
    w = workloads.generate(cfg)
    # scale the RoPE part of KV rows up with position so that later tiles dominate
    ps = cfg.page_size
    kv = w.kv_cache.copy()
    for b in range(2):
        for j in range(int(w.seqlens[b])):
            page = w.block_table[b, j // ps]
            off = (j % ps) * 1152
            row = kv[page, off:off + 1152].view(np.uint16).copy()
            vals = torch.from_numpy(row.view(np.int16).copy()).view(torch.bfloat16).float()
            vals[512:] = vals[512:] * (1 + j / 8.0)
            kv[page, off:off + 1152] = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
    w.kv_cache = kv
    w.q[:, :, 512:] = torch.full((1,), 2.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
    d = DeviceWorkload(w)
    out, lse = d.run()
    ref_out, ref_lse = oracle_decode(w)
    assert_close(out, lse, ref_out, ref_lse, f"rescale, {heads} heads")


def _scale_rope_with_position(w, row_bytes, nope_bytes, growth):
    """Multiply the bf16 RoPE part of every valid KV row j by (1 + j/growth), in place."""
    ps = w.cfg.page_size
    kv = w.kv_cache.copy()
    for b in range(w.seqlens.shape[0]):
        for j in range(int(w.seqlens[b])):
            page = w.block_table[b, j // ps]
            off = (j % ps) * row_bytes + nope_bytes
            rope = kv[page, off:off + 128].view(np.int16).copy()
            vals = torch.from_numpy(rope).view(torch.bfloat16).float() * (1 + j / growth)
            kv[page, off:off + 128] = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
    w.kv_cache = kv


@pytest.mark.parametrize("layout", [1, 2])
def test_fp8_score_growth_triggers_rescale(layout):
    """fp8 layouts: scores that grow along the sequence (RoPE part of row j scaled by
    1 + j/8, q's RoPE part 2; ~120 in log2 units at the end) raise the running max
    past the 2^64 lazy-rescale threshold 1 to 4 times per query row (counted on the
    CPU from the same scores), so O is rescaled in TMEM between tiles. In the 448 layout V includes the RoPE part
    (|V| up to ~450), which the bf16 pair P_hi + P_lo carries within the bound."""
    cfg = workloads.dsv4(batch=2, heads=64, seqlens=(640, 1000), len_dist="fixed", new_rows=False, sink=False,
                         layout=layout)
    w = workloads.generate(cfg)
    _scale_rope_with_position(w, 576 if layout == 1 else 640, 448 if layout == 1 else 512, 8)
    w.q[:, :, -64:] = torch.full((1,), 2.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
    d = DeviceWorkload(w)
    out, lse = d.run()
    ref_out, ref_lse = oracle_decode(w)
    assert_close(out, lse, ref_out, ref_lse, f"fp8 rescale layout {layout}", "scaled")


def test_large_query_value():
    """One q element of 1e5 (bf16 holds it): that head's scores are ~1e4 apart, its
    softmax picks one row and its lse is ~1e4, compared relatively since fp32 carries
    it to a few ulps (~2e-3 each); every other head is unaffected."""
    cfg = workloads.dsv3(batch=2, heads=64, seqlens=(100, 70), len_dist="fixed", new_rows=False)
    w = workloads.generate(cfg)
    w.q[1, 3, 20] = np.uint16(torch.tensor([1.0e5]).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF)
    d = DeviceWorkload(w)
    out, lse = d.run()   # asserts a zero status word
    ref_out, ref_lse = oracle_decode(w)
    keep = np.ones(lse.shape, dtype=bool)
    keep[1, 3] = False
    assert_close(out[keep], lse[keep], ref_out[keep], ref_lse[keep], "bf16 large q, other heads")
    # that head's softmax is one-hot: its output is one V row, whose values can exceed 2, where
    # one bf16 output step alone is above 1e-2
    assert_close(out[1, 3][None], np.zeros(1), ref_out[1, 3][None], np.zeros(1), "bf16 large q, that head's output",
                 "scaled")
    # the score's fp32 sum of terms ~1e4 is good to a few of its ulps (~2e-3 each)
    assert abs(lse[1, 3] - ref_lse[1, 3]) <= 1e-5 * abs(ref_lse[1, 3])


def test_causal_with_short_context():
    """Draft tokens whose visible prefix is empty (L < s_q) give zero output and -inf lse."""
    cfg = workloads.verify(batch=2, heads=64, seqlens=(2, 6), len_dist="fixed")
    w = workloads.generate(cfg)
    d = DeviceWorkload(w)
    out, lse = d.run()
    ref_out, ref_lse = oracle_decode(w)
    assert np.isneginf(ref_lse[0]).all() and np.isneginf(ref_lse[1]).all()
    assert_close(out, lse, ref_out, ref_lse, "short causal")


def test_bad_page_is_reported_not_read():
    cfg = workloads.dsv3(batch=2, heads=64, seqlens=(100, 200), len_dist="fixed", new_rows=False)
    w = workloads.generate(cfg)
    w.block_table[1, 1] = 10_000_000   # out of range for a row < L
    d = DeviceWorkload(w)
    d.make_plan()
    d.decode()
    with pytest.raises(mla.MlaError):
        mla.mla_read_status(d.ws)
    ref_out, ref_lse = oracle_decode(workloads.generate(cfg), kv=w.kv_cache)
    out = d.out.float().cpu().numpy().astype(np.float64)
    # the other request is unaffected
    assert_close(out[:1], d.lse.cpu().numpy()[:1].astype(np.float64), ref_out[:1], ref_lse[:1], "good request")


# ----------------------------------------------------------------------------- sparse prefill
SPARSE_PREFILL = {
    # tokens, heads, kv rows, top-k, padding fraction
    "t5_h64": (5, 64, 300, 128, 0.25),
    "t3_h128": (3, 128, 5000, 300, 0.1),
    "t4_h16_ragged": (4, 16, 65, 65, 0.0),   # kv rows not a multiple of 64, every row listed
    "t2_h64_all_pad": (2, 64, 100, 64, 1.0),
    "t9_h128_long": (9, 128, 20000, 2048, 0.1),
}


def _sparse_prefill_inputs(T, N, s_kv, topk, pad, seed):
    rng = np.random.default_rng(seed)
    q = torch.from_numpy(rng.standard_normal((T, N, 576)).astype(np.float32)).to(torch.bfloat16)
    kv = torch.from_numpy(rng.standard_normal((s_kv, 576)).astype(np.float32)).to(torch.bfloat16)
    idx = np.full((T, topk), -1, np.int32)
    k = min(topk, s_kv)
    npad = int(pad * topk)
    for t in range(T):
        idx[t, :k] = rng.choice(s_kv, k, replace=False)
        if npad:
            idx[t, topk - npad:] = -1
    if topk >= 4 and pad < 1.0:
        idx[0, 1] = s_kv + 7          # out of range: skipped
    return q, kv, idx


@pytest.mark.parametrize("name", list(SPARSE_PREFILL))
@pytest.mark.parametrize("num_sms", [None, 3])
def test_sparse_prefill_matches_oracle(name, num_sms):
    """mla_sparse_prefill against the oracle: out and lse within the decode tolerances,
    max_logits within the lse bound (1e-3), -inf exactly where a token has no valid entry.
    Few partitions (num_sms = 3) split tokens, so the combine merges out, lse and the
    per-split maxima."""
    T, N, s_kv, topk, pad = SPARSE_PREFILL[name]
    q, kv, idx = _sparse_prefill_inputs(T, N, s_kv, topk, pad, seed=90 + T)
    q_bits = q.view(torch.int16).numpy().view(np.uint16)
    kv_bits = kv.view(torch.int16).numpy().view(np.uint16)
    scale = 1 / math.sqrt(192)
    ref_out, ref_mx, ref_lse = oracle.sparse_prefill(q_bits, kv_bits, idx, scale)
    plan = mla.mla_decode_plan(np.full(T, s_kv, np.int32), 1, N, topk, 1, num_sms)
    ws = mla.alloc_workspace(plan.workspace_bytes)
    out = torch.full((T, N, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_sparse_prefill(q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda(), scale,
                           torch.from_numpy(plan.sched).cuda(), torch.from_numpy(plan.num_splits).cuda(),
                           plan.num_partitions, plan.total_splits, ws, out, mx, lse)
    assert mla.mla_read_status(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got, lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, f"{name} splits={plan.total_splits}")
    gm = mx.cpu().numpy().astype(np.float64)
    inf = np.isneginf(ref_mx)
    assert np.array_equal(np.isneginf(gm), inf)
    if (~inf).any():
        assert np.abs(gm[~inf] - ref_mx[~inf]).max() <= 1e-3
