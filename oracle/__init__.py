"""Oracle for paged-latent MLA decode -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct CPU definition the CUDA path
is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
library in ``mla_paged_latent_gb300`` never does, and this package imports
nothing from it.

The arithmetic lives in ``oracle.c`` (IEEE binary64) and the split-KV planner
restatement in ``plan.py``. This module compiles ``oracle.c`` with the system C
compiler on first use (or through ``build()``) and marshals numpy arrays into it.

Sources (page title, section) are listed in the header of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .plan import plan_split_kv, partition_segments  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

LAYOUT_BF16 = 0
LAYOUT_FP8_448 = 1
LAYOUT_FP8_512 = 2


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.mo_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.mo_bf16_decode.restype = f64
        lib.mo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.mo_e4m3_decode.restype = f64
        lib.mo_e4m3_encode.argtypes = [f64]
        lib.mo_e4m3_encode.restype = ctypes.c_uint8
        lib.mo_ue8m0_decode.argtypes = [ctypes.c_uint8]
        lib.mo_ue8m0_decode.restype = f64
        lib.mo_group_exponent.argtypes = [f64]
        lib.mo_group_exponent.restype = i32
        lib.mo_layout_info.argtypes = [i32, i32, P, P, P, P, P]
        lib.mo_layout_info.restype = i32
        lib.mo_decode_row.argtypes = [P, i32, i32, i64, i32, P]
        lib.mo_decode_row.restype = i32
        lib.mo_attend.argtypes = [P, i32, P, i32, i32, f64, i32, f64, P, P]
        lib.mo_attend.restype = None
        lib.mo_mla_decode.argtypes = [P, P, i32, i64, i32, P, i32, P, i32, i32, i32, f64, P, P, i32, i32,
                                      P, P, i32, P, P, i32]
        lib.mo_mla_decode.restype = i32
        lib.mo_combine.argtypes = [P, P, i32, i32, i32, f64, P, P]
        lib.mo_combine.restype = None
        lib.mo_kv_write.argtypes = [P, P, i32, P, i32, i64, i32]
        lib.mo_kv_write.restype = i32
        lib.mo_kv_gather.argtypes = [P, i32, i64, i32, P, i32, i32, P]
        lib.mo_kv_gather.restype = i32
        lib.mo_bf16_encode.argtypes = [f64]
        lib.mo_bf16_encode.restype = ctypes.c_uint16
        lib.mo_kv_norm_rope.argtypes = [P, P, P, f64, P, i32, i32, i32, P]
        lib.mo_kv_norm_rope.restype = i32
        lib.mo_v_up.argtypes = [P, P, i32, i32, i32, P]
        lib.mo_v_up.restype = None
        lib.mo_inv_rope.argtypes = [P, P, P, i32, i32, i32, P]
        lib.mo_inv_rope.restype = None
        lib.mo_swa_plan.argtypes = [P, P, i32, i32, i32, i32, P]
        lib.mo_swa_plan.restype = None
        lib.mo_sparse_prefill.argtypes = [P, P, i32, P, i32, i32, i32, f64, P, P, P, i32]
        lib.mo_sparse_prefill.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------- codecs
def bf16_decode(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.mo_bf16_decode(int(x)) for x in b.ravel()], dtype=np.float64).reshape(b.shape)


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.mo_e4m3_decode(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.mo_e4m3_encode(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def ue8m0_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.mo_ue8m0_decode(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def group_exponent(amax: float) -> int:
    return int(_load().mo_group_exponent(float(amax)))


# ----------------------------------------------------------------------------- layouts
def layout_info(layout: int, page_size: int) -> dict:
    lib = _load()
    rb, pb = ctypes.c_int64(), ctypes.c_int64()
    dqk, nope, ns = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib.mo_layout_info(layout, page_size, ctypes.byref(rb), ctypes.byref(pb), ctypes.byref(dqk),
                            ctypes.byref(nope), ctypes.byref(ns))
    if rc != 0:
        raise ValueError("bad layout / page size")
    return dict(row_bytes=rb.value, page_bytes=pb.value, dqk=dqk.value, nope=nope.value, n_scales=ns.value)


def decode_row(kv_cache: np.ndarray, layout: int, page_size: int, page: int, offset: int) -> np.ndarray:
    lib = _load()
    info = layout_info(layout, page_size)
    kv = np.ascontiguousarray(kv_cache, dtype=np.uint8)
    out = np.zeros(info["dqk"], dtype=np.float64)
    lib.mo_decode_row(_ptr(kv), layout, page_size, page, offset, _ptr(out))
    return out


# ----------------------------------------------------------------------------- attention
def attend(q: np.ndarray, rows: np.ndarray, dv: int, scale: float, sink: float | None = None):
    """Attention of one fp64 query over explicit fp64 rows (V = rows[:, :dv])."""
    lib = _load()
    qd = _c(q, np.float64)
    rd = _c(rows, np.float64).reshape(-1, qd.shape[0]) if np.size(rows) else np.zeros((0, qd.shape[0]))
    rd = np.ascontiguousarray(rd)
    out = np.zeros(dv, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib.mo_attend(_ptr(qd), qd.shape[0], _ptr(rd), rd.shape[0], dv, float(scale), int(sink is not None),
                  float(sink) if sink is not None else 0.0, _ptr(out), _ptr(lse))
    return out, float(lse[0])


def mla_decode(q_bits, kv_cache, layout, page_size, block_table, cache_seqlens, sq, sm_scale, sink=None,
               indices=None, causal=False, select=None, nthreads=0):
    """Paged decode. q_bits: uint16 [T, N, dqk] (bf16 bits). Returns (out [.., 512], lse).

    select: optional (t_idx, n_idx) arrays; only those rows are computed and the
    result has shape [n_sel, 512] / [n_sel]. Otherwise [T, N, 512] / [T, N].
    """
    lib = _load()
    q = _c(q_bits, np.uint16)
    T, N, dqk = q.shape
    kv = np.ascontiguousarray(kv_cache, dtype=np.uint8).reshape(kv_cache.shape[0], -1)
    bt = _c(block_table, np.int32)
    sl = _c(cache_seqlens, np.int32)
    B = sl.shape[0]
    assert T == B * sq
    sk = _c(sink, np.float32)
    idx = _c(indices, np.int32)
    topk = 0 if idx is None else idx.shape[-1]
    if select is not None:
        st = _c(select[0], np.int32)
        sn = _c(select[1], np.int32)
        n_sel = st.shape[0]
        out = np.zeros((n_sel, 512), dtype=np.float64)
        lse = np.zeros(n_sel, dtype=np.float64)
    else:
        st = sn = None
        n_sel = 0
        out = np.zeros((T, N, 512), dtype=np.float64)
        lse = np.zeros((T, N), dtype=np.float64)
    rc = lib.mo_mla_decode(_ptr(q), _ptr(kv), layout, kv.shape[0], page_size, _ptr(bt), bt.shape[1], _ptr(sl), B,
                           sq, N, float(sm_scale), _ptr(sk), _ptr(idx), topk, int(bool(causal)), _ptr(st), _ptr(sn),
                           n_sel, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: out-of-range page reference")
    return out, lse


def combine(part_out: np.ndarray, part_lse: np.ndarray, sink: float | None = None):
    """Merge split partials of one row: part_out [S, dv], part_lse [S]."""
    lib = _load()
    po = _c(part_out, np.float64)
    pl = _c(part_lse, np.float64)
    S, dv = po.shape
    out = np.zeros(dv, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib.mo_combine(_ptr(po), _ptr(pl), S, dv, int(sink is not None), float(sink) if sink is not None else 0.0,
                   _ptr(out), _ptr(lse))
    return out, float(lse[0])


def kv_write(rows_bits, slots, kv_cache: np.ndarray, layout: int, page_size: int) -> np.ndarray:
    """Write rows (uint16 bf16 bits [n, row_elems]) into a copy of kv_cache; returns the copy."""
    lib = _load()
    r = _c(rows_bits, np.uint16)
    s = _c(slots, np.int32)
    kv = np.array(kv_cache, dtype=np.uint8, copy=True, order="C")
    rc = lib.mo_kv_write(_ptr(r), _ptr(s), s.shape[0], _ptr(kv), layout, kv.shape[0], page_size)
    if rc != 0:
        raise ValueError("oracle: slot out of range")
    return kv


def bf16_encode(x) -> np.ndarray:
    """bfloat16 bits (uint16) of float64 values, rounded once to nearest even."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    return np.array([lib.mo_bf16_encode(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def kv_norm_rope(raw_bits, positions, weight_bits, eps, freqs, layout: int) -> np.ndarray:
    """RMSNorm + RoPE of raw KV rows (uint16 bf16 bits [n, row_elems]) -> bf16 bits of the
    rows mla_kv_write would take. eps is taken at float32 precision (the kernel's);
    rows with a position outside [0, len(freqs)) come back as zeros."""
    lib = _load()
    x = _c(raw_bits, np.uint16)
    pos = _c(positions, np.int32)
    w = _c(weight_bits, np.uint16)
    f = _c(freqs, np.float32)
    assert w.shape[0] == 512 and f.shape[1] == 64
    out = np.zeros_like(x)
    lib.mo_kv_norm_rope(_ptr(x), _ptr(pos), _ptr(w), float(np.float32(eps)), _ptr(f), f.shape[0], x.shape[0], layout,
                        _ptr(out))
    return out


def kv_write_norm_rope(raw_bits, slots, positions, weight_bits, eps, freqs, kv_cache, layout: int,
                       page_size: int) -> np.ndarray:
    """kv_write of kv_norm_rope's rows; a row with an out-of-range position is not written."""
    rows = kv_norm_rope(raw_bits, positions, weight_bits, eps, freqs, layout)
    s = np.array(slots, dtype=np.int32, copy=True)
    p = np.asarray(positions)
    s[(p < 0) | (p >= np.asarray(freqs).shape[0])] = -1
    return kv_write(rows, s, kv_cache, layout, page_size)


def v_up(x_bits, w_bits) -> np.ndarray:
    """Value up-projection: x bf16 bits [T, N, 512], w bf16 bits [N, 512, dv] -> bf16 bits [T, N, dv]."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    T, N = x.shape[0], x.shape[1]
    dv = w.shape[2]
    assert x.shape[2] == 512 and w.shape[0] == N and w.shape[1] == 512
    o = np.zeros((T, N, dv), np.uint16)
    lib.mo_v_up(_ptr(x), _ptr(w), T, N, dv, _ptr(o))
    return o


def inv_rope(x_bits, positions, freqs, rope0: int = 448) -> np.ndarray:
    """Inverse RoPE of bf16 rows [rows, 512] (elements rope0 .. rope0 + 63), one position per row."""
    lib = _load()
    x = _c(x_bits, np.uint16).reshape(-1, 512)
    pos = _c(positions, np.int32)
    f = _c(freqs, np.float32)
    assert pos.shape[0] == x.shape[0] and f.shape[1] == 64
    out = np.zeros_like(x)
    lib.mo_inv_rope(_ptr(x), _ptr(pos), _ptr(f), f.shape[0], rope0, x.shape[0], _ptr(out))
    return out


def swa_plan(kv_indices, page_size: int, step: int, topk_lengths=None) -> np.ndarray:
    """Window runs: kv_indices int32 [T, topk] -> int32 [T, 4] (slot0, len0, slot1, rows)."""
    lib = _load()
    idx = _c(kv_indices, np.int32)
    T, topk = idx.shape
    lens = _c(topk_lengths, np.int32)
    runs = np.zeros((T, 4), np.int32)
    lib.mo_swa_plan(_ptr(idx), _ptr(lens), T, topk, page_size, step, _ptr(runs))
    return runs


def run_slots(run) -> np.ndarray:
    """The cache slots of one token's runs (slot0, len0, slot1, rows), in row order."""
    s0, l0, s1, rows = (int(v) for v in run)
    g = np.arange(rows)
    return np.where(g < l0, s0 + g, s1 + g - l0).astype(np.int64)


def decode_runs(q_bits, kv_cache, layout: int, page_size: int, runs, sm_scale: float, sink=None):
    """Attention of every (token, head) over the rows of its token's runs: slots address
    the cache directly; slots outside it are skipped. Returns (out [T, N, 512], lse [T, N])."""
    q = _c(q_bits, np.uint16)
    T, N, dqk = q.shape
    info = layout_info(layout, page_size)
    kv = np.ascontiguousarray(kv_cache, dtype=np.uint8)
    npages = kv.shape[0]
    out = np.zeros((T, N, 512))
    lse = np.zeros((T, N))
    qf = bf16_decode(q.reshape(-1)).reshape(T, N, dqk)
    for t in range(T):
        slots = [s for s in run_slots(runs[t]) if 0 <= s < npages * page_size]
        rows = np.array([decode_row(kv, layout, page_size, s // page_size, s % page_size) for s in slots]
                        ).reshape(-1, info["dqk"])
        for n in range(N):
            o, l = attend(qf[t, n], rows, 512, sm_scale, None if sink is None else float(sink[n]))
            out[t, n], lse[t, n] = o, l
    return out, lse


def sparse_prefill(q_bits, kv_bits, indices, sm_scale: float, nthreads: int = 0):
    """Sparse prefill over an unpaged bf16 latent kv (flash_mla_sparse_fwd's contract).
    q_bits uint16 [T, N, 576], kv_bits uint16 [s_kv, 576], indices int32 [T, topk].
    Returns (out [T, N, 512], max_logits [T, N], lse [T, N]) in float64."""
    lib = _load()
    q = _c(q_bits, np.uint16)
    kv = _c(kv_bits, np.uint16)
    idx = _c(indices, np.int32)
    T, N, D = q.shape
    assert D == 576 and kv.shape[1] == 576 and idx.shape[0] == T
    out = np.zeros((T, N, 512))
    mx = np.zeros((T, N))
    lse = np.zeros((T, N))
    lib.mo_sparse_prefill(_ptr(q), _ptr(kv), kv.shape[0], _ptr(idx), idx.shape[1], T, N, float(sm_scale), _ptr(out),
                          _ptr(mx), _ptr(lse), int(nthreads))
    return out, mx, lse


def kv_gather(kv_cache, layout, page_size, block_table_row, length) -> np.ndarray:
    lib = _load()
    info = layout_info(layout, page_size)
    kv = np.ascontiguousarray(kv_cache, dtype=np.uint8)
    bt = _c(block_table_row, np.int32)
    out = np.zeros((length, info["dqk"]), dtype=np.float64)
    rc = lib.mo_kv_gather(_ptr(kv), layout, kv.shape[0], page_size, _ptr(bt), bt.shape[0], length, _ptr(out))
    if rc != 0:
        raise ValueError("oracle: out-of-range page reference")
    return out
