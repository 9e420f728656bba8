"""Pins of the oracle against facts fixed outside itself (no GPU needed).

Each test names the source that fixes the expected value: a format
specification, a library routine (torch's float8 / bf16 conversions, torch's
scaled_dot_product_attention and logsumexp in float64), a closed form, an
algebraic identity stated on the pages, or a hand-built fixture.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- codecs
def test_e4m3_decode_all_codes_match_torch(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.isnan(ours).sum() == 2  # S.1111.111 only (OCP E4M3)


def test_e4m3_spec_values(oracle_lib):
    # OCP 8-bit FP spec, E4M3: bias 7, max normal 448, min normal 2^-6, min subnormal 2^-9
    d = oracle.e4m3_decode
    assert d(0x7E) == 448.0
    assert d(0x08) == 2.0 ** -6
    assert d(0x01) == 2.0 ** -9
    assert d(0x07) == 7 * 2.0 ** -9
    assert d(0x38) == 1.0
    assert d(0xB8) == -1.0
    assert d(0x80) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_e4m3_encode_matches_torch_rne(oracle_lib):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-448, 448, 3000), rng.standard_normal(3000) * 2.0 ** rng.integers(-12, 6, 3000),
                        rng.uniform(-2.0 ** -7, 2.0 ** -7, 1000)]).astype(np.float32)
    ours = oracle.e4m3_encode(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_ties_to_even(oracle_lib):
    # exact midpoints between consecutive finite codes round to the even code
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    enc = oracle.e4m3_encode(mids)
    lo = np.arange(0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(enc, expect.astype(np.uint8))
    # and torch agrees (its fp32 -> e4m3 conversion is round-to-nearest-even)
    ref = torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(enc, ref)


def test_e4m3_encode_saturates(oracle_lib):
    enc = oracle.e4m3_encode(np.array([448.0, 448.5, 463.9, 470.0, 1e6, np.inf, -np.inf, -500.0]))
    assert list(enc) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_e4m3_roundtrip_finite_codes(oracle_lib):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_bf16_decode_matches_torch(oracle_lib):
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 1 << 16, 4000).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite
    ours = oracle.bf16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_ue8m0(oracle_lib):
    # OCP MX spec E8M0: 2^(b-127), 0xFF NaN
    d = oracle.ue8m0_decode(np.array([127, 128, 123, 0, 254], dtype=np.uint8))
    assert list(d) == [1.0, 2.0, 1.0 / 16, 2.0 ** -127, 2.0 ** 127]
    assert math.isnan(oracle.ue8m0_decode(np.array([255], dtype=np.uint8))[0])


# ----------------------------------------------------------------------------- layouts
def _read_fixture(name):
    entries = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            entries.append(line.split())
    return entries


def test_fp8_page_layout_golden(oracle_lib):
    ent = _read_fixture("fp8_448_page_ps2.txt")
    pb = int([e for e in ent if e[0] == "page_bytes"][0][1])
    info = oracle.layout_info(oracle.LAYOUT_FP8_448, 2)
    assert info["page_bytes"] == pb and info["dqk"] == 512 and info["row_bytes"] == 576
    page = np.zeros((1, pb), dtype=np.uint8)
    for e in ent:
        if e[0] == "row1_nope":
            page[0, 576 + int(e[1])] = int(e[2], 0)
        elif e[0] == "row1_scale":
            page[0, 2 * 576 + 8 + int(e[1])] = int(e[2], 0)
        elif e[0] == "row1_rope":
            v = int(e[2], 0)
            o = 576 + 448 + 2 * int(e[1])
            page[0, o], page[0, o + 1] = v & 0xFF, v >> 8
    k = oracle.decode_row(page, oracle.LAYOUT_FP8_448, 2, 0, 1)
    expect = np.zeros(512)
    for e in ent:
        if e[0] == "expect":
            expect[int(e[1])] = float(e[2])
    assert np.array_equal(k, expect)
    # row 0 decodes to zeros (its scale bytes are 0 -> 2^-127, codes 0)
    assert np.array_equal(oracle.decode_row(page, oracle.LAYOUT_FP8_448, 2, 0, 0), np.zeros(512))


def test_fp8_512_page_layout_golden(oracle_lib):
    """The fp8-512 page (640-B rows, 8 ue8m0 bytes per scale slot) from a hand-built
    fixture: row stride, scale-slot offset, the eighth group's scale and the RoPE
    offset 512 are each exercised by one nonzero value."""
    ent = _read_fixture("fp8_512_page_ps2.txt")
    pb = int([e for e in ent if e[0] == "page_bytes"][0][1])
    info = oracle.layout_info(oracle.LAYOUT_FP8_512, 2)
    assert info["page_bytes"] == pb and info["dqk"] == 576 and info["row_bytes"] == 640
    page = np.zeros((1, pb), dtype=np.uint8)
    for e in ent:
        if e[0] in ("row0_nope", "row1_nope"):
            page[0, 640 * int(e[0][3]) + int(e[1])] = int(e[2], 0)
        elif e[0] in ("row0_scale", "row1_scale"):
            page[0, 2 * 640 + 8 * int(e[0][3]) + int(e[1])] = int(e[2], 0)
        elif e[0] == "row1_rope":
            v = int(e[2], 0)
            o = 640 + 512 + 2 * int(e[1])
            page[0, o], page[0, o + 1] = v & 0xFF, v >> 8
    expect0, expect1 = np.zeros(576), np.zeros(576)
    for e in ent:
        if e[0] == "expect0":
            expect0[int(e[1])] = float(e[2])
        elif e[0] == "expect":
            expect1[int(e[1])] = float(e[2])
    assert np.array_equal(oracle.decode_row(page, oracle.LAYOUT_FP8_512, 2, 0, 0), expect0)
    assert np.array_equal(oracle.decode_row(page, oracle.LAYOUT_FP8_512, 2, 0, 1), expect1)


def test_page_sizes(oracle_lib):
    # page_bytes a multiple of the row size ("MLA" API page of HALOps, kv_cache parameter)
    assert oracle.layout_info(0, 64)["page_bytes"] == 64 * 1152
    assert oracle.layout_info(1, 64)["page_bytes"] == 37440 and 37440 % 576 == 0
    assert oracle.layout_info(2, 64)["page_bytes"] == 41600 and 41600 % 640 == 0
    for ps in (1, 2, 16, 64, 128, 256):
        for lay, rb in ((1, 576), (2, 640)):
            pb = oracle.layout_info(lay, ps)["page_bytes"]
            assert pb % rb == 0 and pb >= ps * (rb + 8) and pb - ps * (rb + 8) < rb
            assert workloads.page_bytes(lay, ps) == pb


# ----------------------------------------------------------------------------- attention algebra
def test_mha_equals_mqa_absorbed(oracle_lib):
    """Absorbed MQA form == naive MHA form ("mla_attention.py", module docstring:
    Compute Friendly Approach vs Data-Movement Friendly Approach), fp64, tiny
    random weights. ql_nope = einsum(q_nope, W_UK); o = einsum(sdpa_o, W_UV)."""
    rng = np.random.default_rng(3)
    N, P, R, Lkv, V, S = 4, 16, 8, 32, 12, 9
    W_UK = rng.standard_normal((Lkv, N, P))
    W_UV = rng.standard_normal((Lkv, N, V))
    q_nope = rng.standard_normal((N, P))
    q_pe = rng.standard_normal((N, R))
    kv_c = rng.standard_normal((S, Lkv))
    k_pe = rng.standard_normal((S, R))
    scale = 1.0 / math.sqrt(P + R)
    rows = np.concatenate([kv_c, k_pe], axis=1)
    for n in range(N):
        ql = np.einsum("h,lh->l", q_nope[n], W_UK[:, n, :])
        o_lat, lse_mqa = oracle.attend(np.concatenate([ql, q_pe[n]]), rows, Lkv, scale)
        o_mqa = o_lat @ W_UV[:, n, :]
        # MHA with per-head keys/values, computed with torch's float64 SDPA
        k_nope = kv_c @ W_UK[:, n, :]
        v = kv_c @ W_UV[:, n, :]
        qh = torch.tensor(np.concatenate([q_nope[n], q_pe[n]]))[None, None, None, :]
        kh = torch.tensor(np.concatenate([k_nope, k_pe], axis=1))[None, None]
        vh = torch.tensor(v)[None, None]
        o_mha = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, scale=scale)[0, 0, 0].numpy()
        s = (kh[0, 0] @ qh[0, 0, 0]) * scale
        lse_mha = torch.logsumexp(s, 0).item()
        assert np.allclose(o_mqa, o_mha, rtol=0, atol=1e-10)
        assert abs(lse_mqa - lse_mha) < 1e-10


def test_single_key(oracle_lib):
    rng = np.random.default_rng(4)
    q = rng.standard_normal(576)
    k = rng.standard_normal((1, 576))
    out, lse = oracle.attend(q, k, 512, 0.1)
    assert np.array_equal(out, k[0, :512])
    assert abs(lse - 0.1 * float(q @ k[0])) < 1e-12


def test_identical_keys(oracle_lib):
    rng = np.random.default_rng(5)
    q = rng.standard_normal(576)
    k = rng.standard_normal(576)
    L = 37
    out, lse = oracle.attend(q, np.tile(k, (L, 1)), 512, 0.07)
    assert np.allclose(out, k[:512], atol=1e-13)
    assert abs(lse - (0.07 * float(q @ k) + math.log(L))) < 1e-12


def test_empty_candidate_set(oracle_lib):
    out, lse = oracle.attend(np.ones(576), np.zeros((0, 576)), 512, 0.1, sink=1.0)
    assert np.all(out == 0) and lse == -math.inf


def test_split_merge_equals_unsplit(oracle_lib):
    """merge_attn_states semantics ("mla_attention.py", Chunked Prefill; an empty
    partial is a zero output with -inf lse, neutralize_empty_context_partials)."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal(576)
    rows = rng.standard_normal((200, 576))
    full, lse_full = oracle.attend(q, rows, 512, 0.05)
    for cuts in ([0, 1, 200], [0, 64, 128, 200], [0, 17, 17, 99, 200], [0, 200, 200]):
        parts, lses = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, l = oracle.attend(q, rows[a:b], 512, 0.05)
            parts.append(o)
            lses.append(l)
        out, lse = oracle.combine(np.array(parts), np.array(lses))
        assert np.allclose(out, full, atol=1e-12)
        assert abs(lse - lse_full) < 1e-12
    out, lse = oracle.combine(np.zeros((3, 512)), np.full(3, -np.inf))
    assert np.all(out == 0) and lse == -math.inf


def test_sink_enters_denominator_only(oracle_lib):
    """attn_sink: per-head logit added to the softmax denominator ("MLA" API page
    of HALOps, mla_attention)."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal(576)
    rows = rng.standard_normal((50, 576))
    base, lse0 = oracle.attend(q, rows, 512, 0.05)
    for sink in (-3.0, 0.0, 2.5):
        o, lse = oracle.attend(q, rows, 512, 0.05, sink=sink)
        z = math.exp(lse0)
        assert np.allclose(o, base * z / (z + math.exp(sink)), atol=1e-13)
        assert lse == lse0
        # combine applies the same factor after merging sink-free partials
        o1, l1 = oracle.attend(q, rows[:20], 512, 0.05)
        o2, l2 = oracle.attend(q, rows[20:], 512, 0.05)
        oc, lc = oracle.combine(np.array([o1, o2]), np.array([l1, l2]), sink=sink)
        assert np.allclose(oc, o, atol=1e-12) and abs(lc - lse) < 1e-12
    o, lse = oracle.attend(q, rows, 512, 0.05, sink=-math.inf)
    assert np.array_equal(o, base)


# ----------------------------------------------------------------------------- paged decode
def _torch_reference(w, causal=False):
    """Brute force with torch float64 SDPA over rows gathered by plain indexing."""
    cfg = w.cfg
    ps = cfg.page_size
    kv16 = torch.from_numpy(w.kv_cache.view(np.int16).copy()).view(torch.bfloat16).double()
    kv16 = kv16.reshape(w.kv_cache.shape[0], ps, 576)
    q = torch.from_numpy(w.q.view(np.int16).copy()).view(torch.bfloat16).double()
    T, N, D = q.shape
    out = torch.zeros(T, N, 512, dtype=torch.float64)
    lse = torch.zeros(T, N, dtype=torch.float64)
    for t in range(T):
        b, i = t // cfg.sq, t % cfg.sq
        L = int(w.seqlens[b])
        lim = L - cfg.sq + i + 1 if causal else L
        pos = torch.arange(lim)
        pages = torch.from_numpy(w.block_table[b]).long()[pos // ps]
        K = kv16[pages, pos % ps]
        s = (q[t] @ K.T) * cfg.sm_scale
        lse[t] = torch.logsumexp(s, dim=1)
        out[t] = torch.nn.functional.scaled_dot_product_attention(q[t][:, None], K[None].expand(N, -1, -1),
                                                                  K[None, :, :512].expand(N, -1, -1),
                                                                  scale=cfg.sm_scale)[:, 0]
    return out.numpy(), lse.numpy()


def test_tiny_decode_matches_torch_sdpa(oracle_lib):
    w = workloads.generate(workloads.tiny())
    out, lse = oracle.mla_decode(w.q, w.kv_cache, 0, 16, w.block_table, w.seqlens, 1, w.cfg.sm_scale)
    ro, rl = _torch_reference(w)
    assert np.allclose(out, ro, atol=1e-12)
    assert np.allclose(lse, rl, atol=1e-12)


def test_verify_causal_matches_torch_sdpa(oracle_lib):
    cfg = workloads.verify(batch=3, heads=16, seqlens=(4, 70, 131), page_size=16)
    w = workloads.generate(cfg)
    out, lse = oracle.mla_decode(w.q, w.kv_cache, 0, 16, w.block_table, w.seqlens, 4, cfg.sm_scale, causal=True)
    ro, rl = _torch_reference(w, causal=True)
    assert np.allclose(out, ro, atol=1e-12)
    assert np.allclose(lse, rl, atol=1e-12)


def _torch_fp8_rows(kv_cache, layout, ps, bt_row, pos):
    """KV rows at request positions `pos`, decoded with torch's float8_e4m3fn and bfloat16
    conversions from bytes cut out of the pages by plain slicing: a page holds ps rows of
    (nope e4m3 | 64 bf16) followed by ps 8-byte slots of ue8m0 scale bytes, one per 64
    NoPE elements ("MLA" API page of HALOps, mla_attention, kv_cache parameter and the
    supported-config paragraph)."""
    nope = {1: 448, 2: 512}[layout]
    rb = nope + 128
    pos = np.asarray(pos, dtype=np.int64)
    pg = np.asarray(bt_row, dtype=np.int64)[pos // ps]
    off = pos % ps
    rows = kv_cache[pg[:, None], off[:, None] * rb + np.arange(rb)[None, :]]
    slots = kv_cache[pg[:, None], ps * rb + off[:, None] * 8 + np.arange(8)[None, :]]
    codes = torch.from_numpy(np.ascontiguousarray(rows[:, :nope])).view(torch.float8_e4m3fn).double()
    scale = torch.from_numpy(np.ascontiguousarray(slots[:, :nope // 64])).view(torch.float8_e8m0fnu).double()
    k_nope = codes * scale.repeat_interleave(64, dim=1)
    rope = torch.from_numpy(np.ascontiguousarray(rows[:, nope:]).view(np.int16)).view(torch.bfloat16).double()
    return torch.cat([k_nope, rope], dim=1)


@pytest.mark.parametrize("layout,sparse", [(1, False), (2, False), (2, True)])
def test_fp8_decode_matches_torch_sdpa(oracle_lib, layout, sparse):
    """Both fp8 layouts, dense and top-k: the oracle's paged decode against torch float64
    SDPA over rows decoded by torch's own fp8 / e8m0 / bf16 conversions. V is the first
    512 elements of the decoded row: kv_c for the 576-wide row, the whole row (448 NoPE +
    64 RoPE) for the 512-wide one."""
    if sparse:
        cfg = workloads.sparse(batch=2, heads=8, seqlens=(300, 1000), topk=96, pad_frac=0.25, page_size=16)
    elif layout == 1:
        cfg = workloads.dsv4(batch=2, heads=8, seqlens=(70, 300), len_dist="fixed", page_size=16, sink=False)
    else:
        cfg = workloads.sparse(batch=2, heads=8, seqlens=(70, 300), topk=0, min_splits=1, page_size=16)
    w = workloads.generate(cfg)
    out, lse = oracle.mla_decode(w.q, w.kv_cache, layout, 16, w.block_table, w.seqlens, 1, cfg.sm_scale,
                                 indices=w.indices)
    q = torch.from_numpy(w.q.view(np.int16).copy()).view(torch.bfloat16).double()
    for t in range(cfg.batch):
        L = int(w.seqlens[t])
        if sparse:
            pos = [int(i) for i in w.indices[t] if 0 <= i < L]
        else:
            pos = list(range(L))
        K = _torch_fp8_rows(w.kv_cache, layout, 16, w.block_table[t], pos)
        assert K.shape[1] == q.shape[2]
        N = q.shape[1]
        ro = torch.nn.functional.scaled_dot_product_attention(q[t][:, None], K[None].expand(N, -1, -1),
                                                              K[None, :, :512].expand(N, -1, -1),
                                                              scale=cfg.sm_scale)[:, 0]
        rl = torch.logsumexp((q[t] @ K.T) * cfg.sm_scale, dim=1)
        assert np.allclose(out[t], ro.numpy(), rtol=0, atol=1e-11)
        assert np.allclose(lse[t], rl.numpy(), rtol=0, atol=1e-11)


def test_causal_reductions(oracle_lib):
    """Causal verify (bottom-right, seq_len = context_len + query_len,
    "mla_attention.py", MLACommonMetadata): s_q = 1 equals dense; token i equals
    a dense decode over the first L - s_q + i + 1 rows."""
    cfg = workloads.verify(batch=2, heads=16, seqlens=(40, 97), page_size=16)
    w = workloads.generate(cfg)
    sq = 4
    out, lse = oracle.mla_decode(w.q, w.kv_cache, 0, 16, w.block_table, w.seqlens, sq, cfg.sm_scale, causal=True)
    for b in range(2):
        for i in range(sq):
            t = b * sq + i
            Li = int(w.seqlens[b]) - sq + i + 1
            o1, l1 = oracle.mla_decode(w.q[t:t + 1], w.kv_cache, 0, 16, w.block_table[b:b + 1],
                                       np.array([Li], np.int32), 1, cfg.sm_scale)
            assert np.allclose(out[t], o1[0], atol=1e-13) and np.allclose(lse[t], l1[0], atol=1e-13)
    # s_q = 1 causal == dense
    o2, l2 = oracle.mla_decode(w.q[::sq], w.kv_cache, 0, 16, w.block_table, w.seqlens, 1, cfg.sm_scale, causal=True)
    o3, l3 = oracle.mla_decode(w.q[::sq], w.kv_cache, 0, 16, w.block_table, w.seqlens, 1, cfg.sm_scale)
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)


def test_sparse_reductions(oracle_lib):
    """Sparse indices (request-local positions, "Implementation:Sgl project
    Sglang Flash MLA", I/O Contract): the identity list equals dense; order does
    not matter; -1 and out-of-range entries are skipped; a duplicate counts twice."""
    cfg = workloads.dsv4(batch=2, seqlens=(90, 150), len_dist="fixed", page_size=16)
    w = workloads.generate(cfg)
    L0, L1 = 90, 150
    dense, dl = oracle.mla_decode(w.q, w.kv_cache, 1, 16, w.block_table, w.seqlens, 1, cfg.sm_scale, sink=w.sink)
    topk = 160
    idx = np.full((2, topk), -1, np.int32)
    idx[0, :L0] = np.arange(L0)
    idx[1, :L1] = np.arange(L1)
    sp, sl = oracle.mla_decode(w.q, w.kv_cache, 1, 16, w.block_table, w.seqlens, 1, cfg.sm_scale, sink=w.sink,
                               indices=idx)
    assert np.allclose(sp, dense, atol=1e-13) and np.allclose(sl, dl, atol=1e-13)
    rng = np.random.default_rng(8)
    idx2 = idx.copy()
    idx2[0] = rng.permutation(idx2[0])
    idx2[1] = rng.permutation(idx2[1])
    sp2, sl2 = oracle.mla_decode(w.q, w.kv_cache, 1, 16, w.block_table, w.seqlens, 1, cfg.sm_scale, sink=w.sink,
                                 indices=idx2)
    assert np.allclose(sp2, dense, atol=1e-12) and np.allclose(sl2, dl, atol=1e-12)
    idx3 = idx.copy()
    idx3[0, L0:L0 + 5] = [L0, L0 + 7, 10000, -5, -1]   # all invalid for request 0
    sp3, _ = oracle.mla_decode(w.q, w.kv_cache, 1, 16, w.block_table, w.seqlens, 1, cfg.sm_scale, sink=w.sink,
                               indices=idx3)
    assert np.array_equal(sp3, sp)
    # duplicate: index 3 listed twice == a row list with row 3 repeated
    idx4 = np.full((1, 4), -1, np.int32)
    idx4[0, :3] = [3, 3, 9]
    o4, l4 = oracle.mla_decode(w.q[:1], w.kv_cache, 1, 16, w.block_table[:1], w.seqlens[:1], 1, cfg.sm_scale,
                               indices=idx4)
    rows = np.stack([oracle.decode_row(w.kv_cache, 1, 16, w.block_table[0, j // 16], j % 16) for j in (3, 3, 9)])
    qd = oracle.bf16_decode(w.q[0, 5])
    oa, la = oracle.attend(qd, rows, 512, cfg.sm_scale)
    assert np.allclose(o4[0, 5], oa, atol=1e-13) and abs(l4[0, 5] - la) < 1e-13


def test_selected_rows_match_full(oracle_lib):
    w = workloads.generate(workloads.tiny())
    full, fl = oracle.mla_decode(w.q, w.kv_cache, 0, 16, w.block_table, w.seqlens, 1, w.cfg.sm_scale)
    sel = (np.array([1, 0, 1], np.int32), np.array([3, 15, 0], np.int32))
    o, l = oracle.mla_decode(w.q, w.kv_cache, 0, 16, w.block_table, w.seqlens, 1, w.cfg.sm_scale, select=sel)
    for k in range(3):
        assert np.array_equal(o[k], full[sel[0][k], sel[1][k]]) and l[k] == fl[sel[0][k], sel[1][k]]


def test_empty_request(oracle_lib):
    w = workloads.generate(workloads.dsv4(batch=2, seqlens=(0, 70), len_dist="fixed", page_size=16))
    o, l = oracle.mla_decode(w.q, w.kv_cache, 1, 16, w.block_table, w.seqlens, 1, w.cfg.sm_scale, sink=w.sink)
    assert np.all(o[0] == 0) and np.all(l[0] == -np.inf)
    assert np.all(np.isfinite(l[1]))


# ----------------------------------------------------------------------------- kv write
def test_group_exponent_is_minimal(oracle_lib):
    for a in [1e-10, 1e-3, 0.5, 1.0, 447.9, 448.0, 448.1, 896.0, 1e5, 3.0e38]:
        e = oracle.group_exponent(a)
        assert 448.0 * 2.0 ** e >= a and 448.0 * 2.0 ** (e - 1) < a


def test_kv_write_fp8_matches_torch_quantization(oracle_lib):
    """fp8 row quantization: one ue8m0 (power-of-two) scale per 64 NoPE elements
    ("MLA" API page of HALOps, supported config); codes must equal torch's
    float8_e4m3fn rounding of x * 2^-e."""
    rng = np.random.default_rng(9)
    for layout, nope in ((1, 448), (2, 512)):
        ps = 16
        info = oracle.layout_info(layout, ps)
        kv = np.zeros((3, info["page_bytes"]), np.uint8)
        n = 20
        x = (rng.standard_normal((n, info["dqk"])) * 2.0 ** rng.integers(-20, 20, (n, 1))).astype(np.float32)
        x[3, :64] = 0.0            # all-zero group -> eps
        x[4, 64:128] *= 1e-30      # tiny group
        bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        slots = rng.permutation(3 * ps)[:n].astype(np.int32)
        slots[5] = -1              # skipped
        out = oracle.kv_write(bits, slots, kv, layout, ps)
        for r in range(n):
            if slots[r] < 0:
                continue
            p, o = divmod(int(slots[r]), ps)
            row = out[p, o * info["row_bytes"]:(o + 1) * info["row_bytes"]]
            sc = out[p, ps * info["row_bytes"] + o * 8: ps * info["row_bytes"] + o * 8 + 8]
            for g in range(nope // 64):
                grp = xb[r, g * 64:(g + 1) * 64]
                amax = max(np.abs(grp).max(), float(np.float32(1e-10)))
                e = int(sc[g]) - 127
                assert 448.0 * 2.0 ** e >= amax > 448.0 * 2.0 ** (e - 1)
                ref = torch.from_numpy((grp * 2.0 ** -e).astype(np.float32)).to(torch.float8_e4m3fn)
                assert np.array_equal(row[g * 64:(g + 1) * 64], ref.view(torch.uint8).numpy())
            assert np.all(sc[nope // 64:] == 0)
            assert np.array_equal(row[nope:].view(np.uint16), bits[r, nope:])
        # the skipped slot's bytes are untouched
        touched = {int(s) for s in slots if s >= 0}
        for s in range(3 * ps):
            if s not in touched:
                p, o = divmod(s, ps)
                assert np.all(out[p, o * info["row_bytes"]:(o + 1) * info["row_bytes"]] == 0)


def test_kv_write_nan_and_inf_elements(oracle_lib):
    """The reading for non-finite inputs: a NaN element does not enter its group's amax (the
    maximum over the numbers, as C's fmax) and is stored as the NaN code 0x7F; the group's
    other codes are torch's e4m3 rounding at the exponent of the finite amax. An infinite
    element makes amax infinite: exponent 127 (byte 254), stored saturated as +-448."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 576)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    bits[0, 7] = 0x7FC0     # NaN in group 0
    bits[0, 64] = 0xFFC0    # -NaN in group 1
    bits[1, 9] = 0x7F80     # +inf in group 0
    bits[1, 10] = 0xFF80    # -inf in group 0
    xb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    kv = oracle.kv_write(bits, np.array([0, 1], np.int32), np.zeros((1, oracle.layout_info(2, 2)["page_bytes"]),
                                                                    np.uint8), 2, 2)
    rows = kv[0, :1280].reshape(2, 640)
    sc = kv[0, 1280:1296].reshape(2, 8)
    for g in (0, 1):
        grp = xb[0, g * 64:(g + 1) * 64]
        e = int(sc[0, g]) - 127
        finite_amax = np.nanmax(np.abs(grp))
        assert 448.0 * 2.0 ** e >= finite_amax > 448.0 * 2.0 ** (e - 1)
        ref = torch.from_numpy((grp * 2.0 ** -e).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        nan = np.isnan(grp)
        assert np.array_equal(rows[0, g * 64:(g + 1) * 64][~nan], ref[~nan])
        assert np.all(rows[0, g * 64:(g + 1) * 64][nan] == 0x7F)
    assert sc[1, 0] == 254
    assert rows[1, 9] == 0x7E and rows[1, 10] == 0xFE
    # finite elements times 2^-127 are far below the smallest e4m3 subnormal: +-0
    others = np.setdiff1d(np.arange(64), [9, 10])
    assert np.all((rows[1, others] & 0x7F) == 0)


def test_kv_write_bf16_is_bit_copy(oracle_lib):
    rng = np.random.default_rng(10)
    bits = rng.integers(0, 1 << 16, (5, 576)).astype(np.uint16)
    kv = np.zeros((2, 16 * 1152), np.uint8)
    slots = np.array([0, 17, 31, 5, 16], np.int32)
    out = oracle.kv_write(bits, slots, kv, 0, 16)
    for r, s in enumerate(slots):
        p, o = divmod(int(s), 16)
        assert np.array_equal(out[p, o * 1152:(o + 1) * 1152].view(np.uint16), bits[r])


@pytest.mark.parametrize("layout", [1, 2])
def test_kv_write_then_decode_roundtrip_error(oracle_lib, layout):
    """Write then read back, both fp8 layouts: every NoPE element within half an E4M3
    step of its input (relative 2^-4 for normals, absolute 2^(e-10) below), the RoPE
    elements bit-exact, on rows whose groups span 2^-20 .. 2^20 in magnitude."""
    nope = {1: 448, 2: 512}[layout]
    rng = np.random.default_rng(11 + layout)
    group_scale = np.repeat(2.0 ** rng.integers(-20, 21, (8, (nope + 64) // 64)), 64, axis=1)
    x = (rng.standard_normal((8, nope + 64)) * group_scale).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    kv = oracle.kv_write(bits, np.arange(8, dtype=np.int32),
                         np.zeros((1, oracle.layout_info(layout, 8)["page_bytes"]), np.uint8), layout, 8)
    for r in range(8):
        k = oracle.decode_row(kv, layout, 8, 0, r)
        assert k.shape == (nope + 64,)
        for g in range(nope // 64):
            grp = xb[r, g * 64:(g + 1) * 64]
            e = oracle.group_exponent(max(np.abs(grp).max(), 1e-10))
            # E4M3 relative half-ulp is 2^-4 for normals; absolute floor 2^-10 (half subnormal step) * 2^e
            err = np.abs(k[g * 64:(g + 1) * 64] - grp)
            assert np.all(err <= np.maximum(np.abs(grp) * 2.0 ** -4, 2.0 ** (e - 10)) + 1e-300)
        assert np.array_equal(k[nope:], xb[r, nope:])


def test_kv_gather_matches_decode_row(oracle_lib):
    w = workloads.generate(workloads.dsv4(batch=2, seqlens=(33, 70), len_dist="fixed", page_size=16))
    g = oracle.kv_gather(w.kv_cache, 1, 16, w.block_table[1], 70)
    for j in (0, 15, 16, 69):
        assert np.array_equal(g[j], oracle.decode_row(w.kv_cache, 1, 16, w.block_table[1, j // 16], j % 16))


# ----------------------------------------------------------------------------- RMSNorm + RoPE (kv write input)
def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_val(bits):
    return torch.from_numpy(np.asarray(bits).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def _freqs(max_pos, cos, sin):
    f = np.zeros((max_pos, 64), np.float32)
    f[:, 0::2] = cos
    f[:, 1::2] = sin
    return f


def test_bf16_encode_matches_torch_on_fp32_values(oracle_lib):
    # float32 inputs, so torch's float32 -> bfloat16 rounding (nearest even) is the reference
    rng = np.random.default_rng(40)
    x = (rng.standard_normal(4000) * 2.0 ** rng.integers(-60, 60, 4000)).astype(np.float32)
    assert np.array_equal(oracle.bf16_encode(x.astype(np.float64)), _bf16_bits(x))


def test_bf16_encode_ties_subnormals_overflow(oracle_lib):
    # ties go to the even significand; the subnormal step is 2^-133; overflow is inf
    cases = [(1 + 2.0 ** -8, 0x3F80), (1 + 3 * 2.0 ** -8, 0x3F82), (-(1 + 2.0 ** -8), 0xBF80), (2.0 ** -133, 0x0001),
             (2.0 ** -134, 0x0000), (3 * 2.0 ** -134, 0x0002), (2.0 ** 128, 0x7F80), (-0.0, 0x8000), (0.0, 0x0000),
             (float(np.float32(3.3895314e38)), 0x7F7F)]
    for v, bits in cases:
        assert int(oracle.bf16_encode([v])[0]) == bits, (v, hex(int(oracle.bf16_encode([v])[0])))


def test_rmsnorm_constant_row_is_unit(oracle_lib):
    # constant row c with eps = 0 and gain 1: every element becomes sign(c) exactly
    raw = np.zeros((3, 576), np.float32)
    raw[0, :512] = 3.5
    raw[1, :512] = -0.001
    raw[2, :512] = 1e20
    out = oracle.kv_norm_rope(_bf16_bits(raw), np.zeros(3, np.int32), _bf16_bits(np.ones(512)), 0.0,
                              _freqs(1, 1.0, 0.0), 0)
    assert np.all(_bf16_val(out[0, :512]) == 1.0)
    assert np.all(_bf16_val(out[1, :512]) == -1.0)
    assert np.all(_bf16_val(out[2, :512]) == 1.0)


def test_rmsnorm_single_spike_closed_form(oracle_lib):
    # one nonzero latent element a: it becomes sign(a) * sqrt(512), the others stay 0
    raw = np.zeros((2, 576), np.float32)
    raw[0, 77] = 5.0
    raw[1, 500] = -0.25
    out = oracle.kv_norm_rope(_bf16_bits(raw), np.zeros(2, np.int32), _bf16_bits(np.ones(512)), 0.0,
                              _freqs(1, 1.0, 0.0), 0)
    s512 = float(torch.tensor(math.sqrt(512.0), dtype=torch.float64).to(torch.bfloat16).double())
    assert _bf16_val(out[0, 77]) == s512 and _bf16_val(out[1, 500]) == -s512
    assert np.count_nonzero(_bf16_val(out[:, :512])) == 2


def test_rmsnorm_against_closed_form_and_gain(oracle_lib):
    # y = x / sqrt(mean(x^2) + eps) * w to within half a bf16 step; a gain of 2 doubles every bit pattern
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((6, 576)) * 3).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(512)).astype(np.float32)
    xb, wb = _bf16_val(_bf16_bits(x)), _bf16_val(_bf16_bits(w))
    eps = np.float32(0.5)
    out = oracle.kv_norm_rope(_bf16_bits(x), np.zeros(6, np.int32), _bf16_bits(w), eps, _freqs(1, 1.0, 0.0), 0)
    ref = xb[:, :512] / np.sqrt((xb[:, :512] ** 2).mean(1, keepdims=True) + float(eps)) * wb
    got = _bf16_val(out[:, :512])
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    out2 = oracle.kv_norm_rope(_bf16_bits(x), np.zeros(6, np.int32), _bf16_bits(2 * wb), eps, _freqs(1, 1.0, 0.0), 0)
    assert np.array_equal(_bf16_val(out2[:, :512]), 2 * got)
    # k_pe is not normalised: the identity rotation leaves its bits unchanged
    assert np.array_equal(out[:, 512:], _bf16_bits(x)[:, 512:])


def test_rope_quarter_and_half_turns(oracle_lib):
    # (u, v) -> (-v, u) for (cos, sin) = (0, 1) and -> (-u, -v) for (-1, 0), exactly, on k_pe
    rng = np.random.default_rng(42)
    x = rng.standard_normal((4, 576)).astype(np.float32)
    xb = _bf16_val(_bf16_bits(x))
    f = np.concatenate([_freqs(1, 0.0, 1.0), _freqs(1, -1.0, 0.0)])
    out = oracle.kv_norm_rope(_bf16_bits(x), np.array([0, 0, 1, 1], np.int32), _bf16_bits(np.ones(512)), 1e-6, f, 2)
    pe, got = xb[:, 512:], _bf16_val(out[:, 512:])
    assert np.array_equal(got[:2, 0::2], -pe[:2, 1::2]) and np.array_equal(got[:2, 1::2], pe[:2, 0::2])
    assert np.array_equal(got[2:], -pe[2:])


def test_rope_matches_complex_rotation(oracle_lib):
    # interleaved pairs as complex numbers times e^(i theta) (torch complex128), per position
    rng = np.random.default_rng(43)
    max_pos = 50
    theta = np.outer(np.arange(max_pos), 10000.0 ** (-np.arange(32) / 32.0))
    f = _freqs(max_pos, np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32))
    x = (rng.standard_normal((7, 576)) * 4).astype(np.float32)
    pos = np.array([0, 1, 7, 13, 29, 48, 49], np.int32)
    out = oracle.kv_norm_rope(_bf16_bits(x), pos, _bf16_bits(np.ones(512)), 1e-6, f, 2)
    pe = torch.from_numpy(_bf16_val(_bf16_bits(x))[:, 512:].reshape(7, 32, 2).copy())
    rot = torch.complex(torch.from_numpy(f[pos, 0::2].astype(np.float64)), torch.from_numpy(f[pos, 1::2].astype(np.float64)))
    ref = torch.view_as_real(torch.view_as_complex(pe) * rot).reshape(7, 64).numpy()
    got = _bf16_val(out[:, 512:])
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 2.0 ** -133)


def test_dsv4_row_rotates_after_the_norm(oracle_lib):
    # layout 1: the 512-wide row is normalised as a whole, then elements 448..511 are rotated
    rng = np.random.default_rng(44)
    x = rng.standard_normal((3, 512)).astype(np.float32)
    w = _bf16_bits(np.ones(512))
    plain = oracle.kv_norm_rope(_bf16_bits(x), np.zeros(3, np.int32), w, 1e-6, _freqs(1, 1.0, 0.0), 1)
    quarter = oracle.kv_norm_rope(_bf16_bits(x), np.zeros(3, np.int32), w, 1e-6, _freqs(1, 0.0, 1.0), 1)
    assert np.array_equal(plain[:, :448], quarter[:, :448])
    n = _bf16_val(plain[:, 448:])
    q = _bf16_val(quarter[:, 448:])
    assert np.array_equal(q[:, 0::2], -n[:, 1::2]) and np.array_equal(q[:, 1::2], n[:, 0::2])
    ms = (_bf16_val(plain) ** 2).mean(1)
    assert np.all(np.abs(ms - 1) < 2.0 ** -7)


def test_norm_rope_write_skips_bad_positions(oracle_lib):
    # a row whose position is outside the table is not written
    rng = np.random.default_rng(45)
    x = _bf16_bits(rng.standard_normal((3, 576)))
    kv = rng.integers(0, 256, (1, 16 * 1152), dtype=np.uint8)
    out = oracle.kv_write_norm_rope(x, np.array([0, 1, 2], np.int32), np.array([0, 5, -1], np.int32),
                                    _bf16_bits(np.ones(512)), 1e-6, _freqs(4, 1.0, 0.0), kv, 0, 16)
    assert np.array_equal(out[0, 1152:3 * 1152], kv[0, 1152:3 * 1152])
    assert not np.array_equal(out[0, :1152], kv[0, :1152])


# ----------------------------------------------------------------------------- value up-projection
def test_v_up_identity_weight_selects_latent(oracle_lib):
    # W_UV[n] = [I_128; 0]: o_v is the first 128 latent elements, bit for bit
    rng = np.random.default_rng(50)
    x = _bf16_bits(rng.standard_normal((3, 4, 512)))
    w = np.zeros((4, 512, 128), np.float32)
    w[:, np.arange(128), np.arange(128)] = 1.0
    o = oracle.v_up(x, _bf16_bits(w))
    assert np.array_equal(o, x[:, :, :128])


def test_v_up_matches_torch_bmm_and_is_linear(oracle_lib):
    # (N, T, L) x (N, L, V) with torch.bmm in float64, then rounded once to bf16; 2 W doubles o exactly
    rng = np.random.default_rng(51)
    x = _bf16_bits(rng.standard_normal((5, 3, 512)))
    w = _bf16_bits(rng.standard_normal((3, 512, 128)) * 0.05)
    o = oracle.v_up(x, w)
    ref = torch.bmm(torch.from_numpy(_bf16_val(x)).transpose(0, 1), torch.from_numpy(_bf16_val(w))).transpose(0, 1)
    ref = ref.numpy()
    got = _bf16_val(o)
    # half a bf16 step: 2^-8 of the value's binade
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 * (1 + 1e-12) + 1e-300)
    o2 = oracle.v_up(x, _bf16_bits(2 * _bf16_val(w)))
    assert np.array_equal(_bf16_val(o2), 2 * got)


# ----------------------------------------------------------------------------- inverse RoPE of the output
def test_inv_rope_undoes_the_forward_rotation(oracle_lib):
    # the DSV4 row: kv_norm_rope rotates elements 448..511 forward, inv_rope (written separately)
    # rotates them back; the two bf16 roundings leave at most one bf16 step per element
    rng = np.random.default_rng(52)
    max_pos = 300
    theta = np.outer(np.arange(max_pos), 10000.0 ** (-np.arange(32) / 32.0))
    f = _freqs(max_pos, np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32))
    x = rng.standard_normal((6, 512)).astype(np.float32)
    pos = np.array([0, 1, 2, 99, 250, 299], np.int32)
    w = _bf16_bits(np.ones(512))
    plain = oracle.kv_norm_rope(_bf16_bits(x), pos, w, 1e-6, _freqs(max_pos, 1.0, 0.0), 1)
    fwd = oracle.kv_norm_rope(_bf16_bits(x), pos, w, 1e-6, f, 1)
    back = oracle.inv_rope(fwd, pos, f, 448)
    assert np.array_equal(back[:, :448], plain[:, :448])
    a, b = _bf16_val(back[:, 448:]), _bf16_val(plain[:, 448:])
    assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -6 + 2.0 ** -7)


def test_inv_rope_quarter_turn_and_bad_position(oracle_lib):
    # (c, s) = (0, 1): (u, v) -> (v, -u) exactly; a position outside the table copies the row
    rng = np.random.default_rng(53)
    x = _bf16_bits(rng.standard_normal((2, 512)))
    out = oracle.inv_rope(x, np.array([0, 5], np.int32), _freqs(1, 0.0, 1.0), 448)
    xv, ov = _bf16_val(x), _bf16_val(out)
    assert np.array_equal(ov[0, 448::2], xv[0, 449::2]) and np.array_equal(ov[0, 449::2], -xv[0, 448::2])
    assert np.array_equal(out[1], x[1]) and np.array_equal(out[0, :448], x[0, :448])


# ----------------------------------------------------------------------------- sliding-window runs
def test_swa_plan_hand_built_windows(oracle_lib):
    # page size 16; each case worked by hand from the rule (runs of +step within one page,
    # more than two runs -> the first row only, runs stored from their lowest slot)
    pad = -1
    cases = [
        ([32 + g for g in range(16)], 16, 1, (32, 16, 48, 16)),          # one page, one run
        ([40 + g for g in range(16)], 16, 1, (40, 8, 48, 16)),           # crosses into the next page
        ([40, 41, 42, 60, 61, 100] + [pad] * 10, 6, 1, (40, 1, 40, 1)),  # three runs: cut
        ([55 - g for g in range(16)], 16, -1, (48, 8, 40, 16)),          # descending across a page
        ([5, 6, pad, pad] + [pad] * 12, 2, 1, (5, 2, 7, 2)),             # padding past the length
        ([3, 7, 8] + [pad] * 13, 3, 1, (3, 1, 7, 3)),                    # a gap inside one page
        ([9] * 16, 0, 1, (0, 0, 0, 0)),                                  # empty window
        ([20, 19, 18, 30] + [pad] * 12, 4, -1, (18, 3, 30, 4)),          # descending run, then one row
    ]
    idx = np.array([c[0] for c in cases], np.int32)
    lens = np.array([c[1] for c in cases], np.int32)
    for step in (1, -1):
        sel = [i for i, c in enumerate(cases) if c[2] == step]
        runs = oracle.swa_plan(idx[sel], 16, step, lens[sel])
        for k, i in enumerate(sel):
            assert tuple(runs[k]) == cases[i][3], (i, tuple(runs[k]))


def test_swa_plan_lengths_clamp_and_default(oracle_lib):
    idx = np.tile(np.arange(100, 108, dtype=np.int32), (3, 1))
    assert tuple(oracle.swa_plan(idx[:1], 64, 1)[0]) == (100, 8, 108, 8)          # no lengths: topk rows
    runs = oracle.swa_plan(idx, 64, 1, np.array([-3, 50, 3], np.int32))
    assert tuple(runs[0]) == (0, 0, 0, 0) and tuple(runs[1]) == (100, 8, 108, 8) and tuple(runs[2]) == (100, 3, 103, 3)


def test_decode_over_runs_equals_dense_and_is_order_free(oracle_lib):
    # a request whose positions 0..L-1 sit on consecutive slots of pages 3 and 4: its window of
    # all L rows (listed ascending or descending) gives the dense decode of that request
    w = workloads.generate(workloads.tiny())
    c = w.cfg
    ps = c.page_size
    L = 20
    kv = w.kv_cache
    bt = np.array([[3, 4] + [-1] * (w.block_table.shape[1] - 2)], np.int32)
    q = w.q[:1]
    dense_out, dense_lse = oracle.mla_decode(q, kv, c.layout, ps, bt, np.array([L], np.int32), 1, c.sm_scale)
    slots = np.array([3 * ps + p for p in range(L)], np.int32)
    for step, order in ((1, slots), (-1, slots[::-1].copy())):
        runs = oracle.swa_plan(order[None, :], ps, step)
        out, lse = oracle.decode_runs(q, kv, c.layout, ps, runs, c.sm_scale)
        assert np.allclose(out, dense_out, rtol=1e-12, atol=1e-12) and np.allclose(lse, dense_lse, rtol=1e-12)


# ----------------------------------------------------------------------------- sparse prefill
def _bf16_bits_of(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def test_sparse_prefill_all_rows_is_dense_attention(oracle_lib):
    """flash_mla_sparse_fwd ("Implementation:Sgl project Sglang Flash MLA", Signature, I/O
    Contract): with every kv row listed (in any order) the result is dense attention over kv:
    out and lse against torch float64 SDPA / logsumexp, max_logits against torch's max of the
    scaled scores."""
    rng = np.random.default_rng(80)
    T, N, s_kv = 3, 8, 150
    q = _bf16_bits_of(rng.standard_normal((T, N, 576)))
    kv = _bf16_bits_of(rng.standard_normal((s_kv, 576)))
    idx = np.stack([rng.permutation(s_kv) for _ in range(T)]).astype(np.int32)
    scale = 1 / math.sqrt(192)
    out, mx, lse = oracle.sparse_prefill(q, kv, idx, scale)
    Q, K = _bits_f64(q), _bits_f64(kv)
    for t in range(T):
        s = (Q[t] @ K.T) * scale
        ro = torch.nn.functional.scaled_dot_product_attention(Q[t][:, None], K[None].expand(N, -1, -1),
                                                              K[None, :, :512].expand(N, -1, -1), scale=scale)[:, 0]
        assert np.allclose(out[t], ro.numpy(), rtol=0, atol=1e-11)
        assert np.allclose(lse[t], torch.logsumexp(s, 1).numpy(), rtol=0, atol=1e-11)
        assert np.allclose(mx[t], s.max(1).values.numpy(), rtol=0, atol=1e-12)


def test_sparse_prefill_skips_invalid_and_counts_duplicates(oracle_lib):
    """Entries outside [0, s_kv) are skipped; a token with none gives out = 0, lse = -inf and
    max_logits = -inf; a row listed twice adds its weight twice: lse = ln(e^lse1 + e^s_dup)
    (a closed form of the sum over keys). Invariants: max_logits <= lse <= max_logits + ln(n)."""
    rng = np.random.default_rng(81)
    T, N, s_kv, k = 4, 4, 90, 40
    q = _bf16_bits_of(rng.standard_normal((T, N, 576)))
    kv = _bf16_bits_of(rng.standard_normal((s_kv, 576)))
    base = np.stack([rng.choice(s_kv, k, replace=False) for _ in range(T)]).astype(np.int32)
    scale = 0.05
    o1, m1, l1 = oracle.sparse_prefill(q, kv, base, scale)
    noisy = np.concatenate([base, np.full((T, 7), -1, np.int32), np.full((T, 3), s_kv + 5, np.int32)], axis=1)
    noisy = np.stack([rng.permutation(r) for r in noisy]).astype(np.int32)
    o2, m2, l2 = oracle.sparse_prefill(q, kv, noisy, scale)
    assert np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13) and np.array_equal(m1, m2)
    empty = np.full((T, 5), -1, np.int32)
    o3, m3, l3 = oracle.sparse_prefill(q, kv, empty, scale)
    assert np.all(o3 == 0) and np.all(np.isneginf(l3)) and np.all(np.isneginf(m3))
    dup = np.concatenate([base, base[:, :1]], axis=1)
    _, _, l4 = oracle.sparse_prefill(q, kv, dup, scale)
    Q, K = _bits_f64(q), _bits_f64(kv)
    for t in range(T):
        s_dup = ((Q[t] @ K[int(base[t, 0])]) * scale).numpy()
        assert np.allclose(l4[t], np.logaddexp(l1[t], s_dup), atol=1e-12)
    assert np.all(m1 <= l1 + 1e-12) and np.all(l1 <= m1 + math.log(k) + 1e-12)
