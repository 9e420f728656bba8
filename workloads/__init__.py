"""Seeded synthetic inputs for paged-latent MLA decode.

This module only draws random numbers and lays them out in the paged formats;
it holds none of the decode arithmetic. Both the CUDA path (tests, bench) and
the oracle consume what it produces.

Workloads (shapes of DeepSeek-V3/V4-style decode, speculative verify and sparse top-k batches):
  tiny    2 x 1 token, N=16, bf16 KV, L = (37, 130), page 16, values N(0,1)*0.5
  dsv3    64 x 1 token, N=128, bf16 KV, L ~ U{1024..8192}, page 64
  dsv4    128 x 1 token, N=64, fp8-448 KV (ue8m0/64, exponents U{-4..4}),
          L = floor(exp(U(ln 512, ln 32768))), page 64, per-head sink ~ N(0,1)
  verify  32 x 4 draft tokens, N=128, bf16 KV, context ~ U{2048..16384},
          L = context + 4, causal, the 4 new rows written by mla_kv_write
  sparse  64 x 1 token, N=128, fp8-512 KV, L = 65536, topk 2048 drawn without
          replacement, the last 10% of each index list set to -1, >= 4 splits

Draw order (one numpy Generator per workload, seed 0 unless overridden):
seqlens -> page permutation -> q -> KV -> sink -> indices -> new rows.
bf16 values are float32 normal draws rounded to nearest-even by torch's bf16
conversion. fp8 NoPE codes are drawn from 256 equiprobable quantiles of N(0,1),
each rounded to E4M3 by torch's float8_e4m3fn conversion (a discrete stand-in
for "N(0,1) quantized to e4m3" that generates gigabytes quickly); scale bytes
are 127 + U{-4..4}.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LAYOUT_BF16 = 0
LAYOUT_FP8_448 = 1
LAYOUT_FP8_512 = 2

_ROW_BYTES = {LAYOUT_BF16: 1152, LAYOUT_FP8_448: 576, LAYOUT_FP8_512: 640}
_NOPE = {LAYOUT_BF16: 512, LAYOUT_FP8_448: 448, LAYOUT_FP8_512: 512}
_DQK = {LAYOUT_BF16: 576, LAYOUT_FP8_448: 512, LAYOUT_FP8_512: 576}


def page_bytes(layout: int, page_size: int) -> int:
    """Bytes per page: rows, then (fp8 layouts) one 8-byte scale slot per row,
    rounded up to a multiple of the row size ("MLA" API page of HALOps,
    mla_attention, kv_cache parameter)."""
    rb = _ROW_BYTES[layout]
    if layout == LAYOUT_BF16:
        return page_size * rb
    return -(-(page_size * (rb + 8)) // rb) * rb


def row_elems(layout: int) -> int:
    """bf16 elements of one new KV row handed to mla_kv_write."""
    return _DQK[layout]


@dataclasses.dataclass
class Config:
    name: str
    batch: int
    sq: int
    heads: int
    layout: int
    page_size: int
    sm_scale: float
    seqlens: tuple | None = None          # fixed lengths, else drawn
    len_dist: str = "uniform"             # uniform | loguniform | fixed
    len_lo: int = 1
    len_hi: int = 1
    value_scale: float = 1.0
    sink: bool = False
    causal: bool = False
    topk: int = 0
    pad_frac: float = 0.0
    min_splits: int = 1
    new_rows: bool = True                 # the last s_q rows of each request are (re)written by mla_kv_write
    rmsnorm_new_rows: bool = False
    add_sq_to_len: bool = False           # drawn lengths are contexts; L = context + s_q
    seed: int = 0
    tail_fill: str = "random"             # content of page rows past each request's length: random | nan


def tiny(**kw) -> Config:
    c = Config("tiny", 2, 1, 16, LAYOUT_BF16, 16, 1 / math.sqrt(192), seqlens=(37, 130), len_dist="fixed",
               value_scale=0.5)
    return dataclasses.replace(c, **kw)


def dsv3(**kw) -> Config:
    c = Config("dsv3", 64, 1, 128, LAYOUT_BF16, 64, 1 / math.sqrt(192), len_lo=1024, len_hi=8192)
    return dataclasses.replace(c, **kw)


def dsv4(**kw) -> Config:
    c = Config("dsv4", 128, 1, 64, LAYOUT_FP8_448, 64, 1 / math.sqrt(512), len_dist="loguniform", len_lo=512,
               len_hi=32768, sink=True)
    return dataclasses.replace(c, **kw)


def verify(**kw) -> Config:
    c = Config("verify", 32, 4, 128, LAYOUT_BF16, 64, 1 / math.sqrt(192), len_lo=2048, len_hi=16384, causal=True,
               rmsnorm_new_rows=True, add_sq_to_len=True)
    return dataclasses.replace(c, **kw)


def sparse(**kw) -> Config:
    c = Config("sparse", 64, 1, 128, LAYOUT_FP8_512, 64, 1 / math.sqrt(192), len_dist="fixed",
               seqlens=(65536,) * 64, topk=2048, pad_frac=0.1, min_splits=4)
    return dataclasses.replace(c, **kw)


CONFIGS = {"tiny": tiny, "dsv3": dsv3, "dsv4": dsv4, "verify": verify, "sparse": sparse}


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _fp8_quantile_table() -> np.ndarray:
    import torch
    from scipy.special import ndtri
    u = (np.arange(256, dtype=np.float64) + 0.5) / 256.0
    vals = torch.from_numpy(ndtri(u).astype(np.float32))
    return vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


@dataclasses.dataclass
class Workload:
    cfg: Config
    q: np.ndarray               # uint16 bf16 bits [T, N, dqk]
    kv_cache: np.ndarray        # uint8 [num_pages, page_bytes]
    block_table: np.ndarray     # int32 [B, max_pages] (-1 past a request's pages)
    seqlens: np.ndarray         # int32 [B]
    sink: np.ndarray | None     # float32 [N]
    indices: np.ndarray | None  # int32 [T, topk]
    new_rows: np.ndarray | None  # uint16 bf16 bits [B*s_q, row_elems]
    new_slots: np.ndarray | None  # int32 [B*s_q]

    @property
    def dqk(self) -> int:
        return _DQK[self.cfg.layout]

    @property
    def tokens(self) -> int:
        return self.cfg.batch * self.cfg.sq

    def kv_rows_touched(self) -> int:
        """KV rows the decode reads (dense: sum L; sparse: valid indices)."""
        if self.indices is not None:
            L = np.repeat(self.seqlens, self.cfg.sq)[:, None]
            return int(((self.indices >= 0) & (self.indices < L)).sum())
        return int(self.seqlens.sum())


def generate(cfg: Config) -> Workload:
    rng = np.random.default_rng(cfg.seed)
    B, sq, N, ps, layout = cfg.batch, cfg.sq, cfg.heads, cfg.page_size, cfg.layout
    # 1. sequence lengths
    if cfg.len_dist == "fixed" or cfg.seqlens is not None:
        seqlens = np.asarray(cfg.seqlens, dtype=np.int64)
        assert seqlens.shape[0] == B
    elif cfg.len_dist == "uniform":
        seqlens = rng.integers(cfg.len_lo, cfg.len_hi + 1, size=B)
    elif cfg.len_dist == "loguniform":
        seqlens = np.floor(np.exp(rng.uniform(math.log(cfg.len_lo), math.log(cfg.len_hi), size=B))).astype(np.int64)
    else:
        raise ValueError(cfg.len_dist)
    if cfg.add_sq_to_len and cfg.seqlens is None and cfg.len_dist != "fixed":
        seqlens = seqlens + sq          # context + the s_q freshly written rows
    seqlens = seqlens.astype(np.int32)
    # 2. pages: a random permutation of exactly sum ceil(L/ps) pages
    npages_req = [max(0, -(-int(L) // ps)) for L in seqlens]
    total_pages = max(1, sum(npages_req))
    perm = rng.permutation(total_pages).astype(np.int32)
    max_pages = max(1, max(npages_req) if npages_req else 1)
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        block_table[b, :npages_req[b]] = perm[off:off + npages_req[b]]
        off += npages_req[b]
    # 3. q
    dqk = _DQK[layout]
    T = B * sq
    q = _bf16_bits(rng.standard_normal((T, N, dqk), dtype=np.float32) * np.float32(cfg.value_scale))
    # 4. KV pages
    pb = page_bytes(layout, ps)
    rb = _ROW_BYTES[layout]
    kv = np.zeros((total_pages, pb), dtype=np.uint8)
    nrows = total_pages * ps
    if layout == LAYOUT_BF16:
        vals = rng.standard_normal((nrows, 576), dtype=np.float32) * np.float32(cfg.value_scale)
        bits = _bf16_bits(vals).reshape(total_pages, ps * 576)
        kv[:, :ps * rb] = bits.view(np.uint8).reshape(total_pages, ps * rb)
    else:
        nope = _NOPE[layout]
        table = _fp8_quantile_table()
        rows = kv[:, :ps * rb].reshape(total_pages, ps, rb)
        chunk = max(1, (1 << 24) // (ps * nope))
        for p0 in range(0, total_pages, chunk):
            p1 = min(total_pages, p0 + chunk)
            u = rng.integers(0, 256, size=(p1 - p0, ps, nope), dtype=np.uint8)
            rows[p0:p1, :, :nope] = table[u]
            rope = rng.standard_normal((p1 - p0, ps, 64), dtype=np.float32) * np.float32(cfg.value_scale)
            rows[p0:p1, :, nope:] = _bf16_bits(rope).view(np.uint8).reshape(p1 - p0, ps, 128)
        scales = kv[:, ps * rb:ps * rb + ps * 8].reshape(total_pages, ps, 8)
        ng = nope // 64
        scales[:, :, :ng] = rng.integers(123, 132, size=(total_pages, ps, ng), dtype=np.uint8)
        kv[:, ps * rb:ps * rb + ps * 8] = scales.reshape(total_pages, ps * 8)
    if cfg.tail_fill == "nan":
        # rows past each request's length hold NaN bit patterns (never-written cache memory)
        for b in range(B):
            L = int(seqlens[b])
            for j in range(L, npages_req[b] * ps):
                page = block_table[b, j // ps]
                r0 = (j % ps) * rb
                nan16 = np.frombuffer(np.full(rb // 2, 0x7FC1, dtype=np.uint16).tobytes(), np.uint8)
                if layout == LAYOUT_BF16:
                    kv[page, r0:r0 + rb] = nan16
                else:
                    nope = _NOPE[layout]
                    kv[page, r0:r0 + nope] = 0x7F
                    kv[page, r0 + nope:r0 + rb] = nan16[:rb - nope]
    # 5. sink
    sink = rng.standard_normal(N).astype(np.float32) if cfg.sink else None
    # 6. sparse indices (request-local positions)
    indices = None
    if cfg.topk > 0:
        indices = np.empty((T, cfg.topk), dtype=np.int32)
        npad = int(math.floor(cfg.pad_frac * cfg.topk))
        for t in range(T):
            L = int(seqlens[t // sq])
            k = min(cfg.topk, L)
            row = np.full(cfg.topk, -1, dtype=np.int32)
            if k > 0:
                row[:k] = rng.choice(L, size=k, replace=False).astype(np.int32)
            if npad > 0:
                row[cfg.topk - npad:] = -1
            indices[t] = row
    # 7. new rows for mla_kv_write: the last s_q positions of each request
    new_rows = new_slots = None
    if cfg.new_rows:
        re = _DQK[layout]
        x = rng.standard_normal((T, re), dtype=np.float32) * np.float32(cfg.value_scale)
        if cfg.rmsnorm_new_rows:
            # the rows arrive already RMSNorm'd (gain 1, eps 1e-6) over the latent part;
            # the RoPE part passes through
            nl = _NOPE[layout]
            lat = x[:, :nl].astype(np.float64)
            x[:, :nl] = (lat / np.sqrt(np.mean(lat * lat, axis=1, keepdims=True) + 1e-6)).astype(np.float32)
        new_rows = _bf16_bits(x)
        new_slots = np.full(T, -1, dtype=np.int32)
        for b in range(B):
            L = int(seqlens[b])
            for i in range(sq):
                j = L - sq + i
                if j >= 0:
                    new_slots[b * sq + i] = block_table[b, j // ps] * ps + j % ps
    return Workload(cfg, q, kv, block_table, seqlens, sink, indices, new_rows, new_slots)
