"""Python binding of the GB300 paged-latent MLA decode library.

Thin argument marshalling over the C ABI in include/mla_decode.h: every step of
the decode path runs in the library's CUDA kernels. PyTorch supplies device
memory and streams only. The functions keep the C names.

If the compiled library is missing, every entry point raises: there is no CPU
fallback. Build it with ``python -m mla_paged_latent_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB

MLA_KV_BF16_576 = 0
MLA_KV_FP8_448_UE8M0 = 1
MLA_KV_FP8_512_UE8M0 = 2
DQK = {0: 576, 1: 512, 2: 576}
ROW_ELEMS = {0: 576, 1: 512, 2: 576}
DV = 512
WORKSPACE_HEADER = 256

MLA_OK = 0
ERRORS = {-1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "WORKSPACE_TOO_SMALL", -4: "CUDA", -5: "DEVICE_CHECK",
          -6: "CAPACITY"}

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class _PlanInfo(ctypes.Structure):
    _fields_ = [("num_partitions", ctypes.c_int32), ("groups", ctypes.c_int32), ("total_splits", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("workspace_bytes", ctypes.c_size_t)]


EXPORTS = ["mla_page_bytes", "mla_decode_plan", "mla_decode", "mla_decode_runs", "mla_sparse_prefill", "mla_swa_plan",
           "mla_decode_static_workspace", "mla_combine",
           "mla_combine_v_up", "mla_combine_inv_rope", "mla_kv_write", "mla_kv_write_norm_rope", "mla_kv_gather", "mla_workspace_init", "mla_read_status",
           "mla_last_error"]
STATIC_WORKSPACE_BYTES = 64 << 20


def load(path: str | None = None):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first (python -m mla_paged_latent_gb300.build)")
        lib = ctypes.CDLL(p)
        V, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.mla_page_bytes.argtypes = [I32, I32, ctypes.POINTER(I64)]
        lib.mla_decode_plan.argtypes = [V, I32, I32, I32, I32, I32, I32, V, I32, V, ctypes.POINTER(_PlanInfo)]
        lib.mla_decode.argtypes = [V, V, I32, I64, I32, V, I32, V, I32, I32, I32, F32, V, V, I32, I32, V, V, I32, I32,
                                   V, SZ, V, V, ctypes.c_uint32, V]
        lib.mla_decode_runs.argtypes = [V, V, I32, I64, I32, V, I32, I32, I32, I32, F32, V, V, V, I32, I32, V, SZ, V,
                                        V, ctypes.c_uint32, V]
        lib.mla_swa_plan.argtypes = [V, V, I32, I32, I32, I32, V, V]
        lib.mla_sparse_prefill.argtypes = [V, V, I32, V, I32, I32, I32, F32, V, V, I32, I32, V, SZ, V, V, V,
                                           ctypes.c_uint32, V]
        lib.mla_decode_static_workspace.argtypes = [V, V, I32, I64, I32, V, I32, V, I32, I32, I32, F32, V, V, I32, I32,
                                                    V, V, I32, I32, V, V, V, V]
        lib.mla_combine.argtypes = [V, V, V, I32, I32, I32, V, V, V, V]
        lib.mla_combine_v_up.argtypes = [V, V, V, I32, I32, I32, V, V, V, V, V, V, V]
        lib.mla_combine_inv_rope.argtypes = [V, V, V, I32, I32, I32, V, V, V, I32, I32, V, V, V]
        lib.mla_kv_write.argtypes = [V, V, I32, V, I32, I64, I32, V, V]
        lib.mla_kv_write_norm_rope.argtypes = [V, V, V, V, F32, V, I32, I32, V, I32, I64, I32, V, V]
        lib.mla_kv_gather.argtypes = [V, I32, I64, I32, V, I32, I32, V, V]
        lib.mla_workspace_init.argtypes = [V, V]
        lib.mla_read_status.argtypes = [V, ctypes.POINTER(ctypes.c_uint32), I32, V]
        lib.mla_last_error.restype = ctypes.c_char_p
        for name in EXPORTS[:-1]:
            getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(rc: int):
    if rc != MLA_OK:
        raise MlaError(rc, load().mla_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _require_cuda(*tensors):
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors passed to the device entry points must live on the GPU")


def mla_page_bytes(layout: int, page_size: int) -> int:
    out = ctypes.c_int64()
    _check(load().mla_page_bytes(layout, page_size, ctypes.byref(out)))
    return out.value


@dataclasses.dataclass
class Plan:
    sched: np.ndarray            # int32 [num_partitions, 8]
    num_splits: np.ndarray       # int32 [batch + 1]
    num_partitions: int
    groups: int
    total_splits: int
    max_splits: int
    workspace_bytes: int


def mla_decode_plan(cache_seqlens, q_tokens_per_req: int, num_heads: int, topk: int = 0, min_splits: int = 1,
                    num_sms: int | None = None) -> Plan:
    """Host planner. cache_seqlens: host int array [batch]."""
    lib = load()
    sl = np.ascontiguousarray(np.asarray(cache_seqlens).astype(np.int32).ravel())
    if num_sms is None:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    info = _PlanInfo()
    ns = np.empty(sl.shape[0] + 1, dtype=np.int32)
    # one call with room for a partition per SM x 4; the rare larger plan reports its size
    # (MLA_ERR_CAPACITY) and is made again into a buffer of that size
    cap = 4 * int(num_sms)
    while True:
        sched = np.empty((cap, 8), dtype=np.int32)
        rc = lib.mla_decode_plan(sl.ctypes.data, sl.shape[0], q_tokens_per_req, num_heads, topk, min_splits, num_sms,
                                 sched.ctypes.data, cap, ns.ctypes.data, ctypes.byref(info))
        if rc == -6 and info.num_partitions > cap:
            cap = info.num_partitions
            continue
        _check(rc)
        break
    return Plan(sched[:info.num_partitions], ns, info.num_partitions, info.groups, info.total_splits, info.max_splits,
                info.workspace_bytes)


def mla_decode(q, kv_cache, layout: int, page_size: int, block_table, cache_seqlens, q_tokens_per_req: int,
               sm_scale: float, sched, num_splits, num_partitions: int, total_splits: int, workspace, out, lse,
               sink=None, indices=None, causal: bool = False, skip_combine: bool = False, stream=None,
               single_sm: bool = False, _test_withhold_signal: bool = False):
    """Enqueue decode (+ split combine) on `stream`. All tensors on the GPU:
    q bf16 [T, N, Dqk]; kv_cache uint8 [num_pages, page_bytes]; block_table int32 [B, max_pages];
    cache_seqlens int32 [B]; sched int32 [P, 8]; num_splits int32 [B+1]; workspace uint8;
    out bf16 [T, N, 512]; lse float32 [T, N]; sink float32 [N] or None; indices int32 [T, topk] or None.
    single_sm: run a dense bf16 decode whose query rows come in groups of 128 on the single-SM
    kernel instead of the CTA-pair kernel."""
    _require_cuda(q, kv_cache, block_table, cache_seqlens, sched, num_splits, workspace, out, lse, sink, indices)
    T, N, D = q.shape
    B = cache_seqlens.shape[0]
    topk = 0 if indices is None else int(indices.shape[-1])
    _check(load().mla_decode(_ptr(q), _ptr(kv_cache), layout, kv_cache.shape[0], page_size, _ptr(block_table),
                             block_table.shape[1], _ptr(cache_seqlens), B, q_tokens_per_req, N, float(sm_scale),
                             _ptr(sink), _ptr(indices), topk, int(bool(causal)), _ptr(sched), _ptr(num_splits),
                             num_partitions, total_splits, _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
                             (1 if skip_combine else 0) | (2 if single_sm else 0) |
                             (0x80000000 if _test_withhold_signal else 0),
                             _stream(stream)))


def mla_sparse_prefill(q, kv, indices, sm_scale: float, sched, num_splits, num_partitions: int, total_splits: int,
                       workspace, out, max_logits, lse, stream=None):
    """Sparse prefill over one unpaged latent run (flash_mla_sparse_fwd's contract): q bf16
    [T, N, 576]; kv bf16 [s_kv, 576]; indices int32 [T, topk] (positions in kv, others skipped);
    the plan from mla_decode_plan(np.full(T, s_kv), 1, N, topk, ...). Writes out bf16
    [T, N, 512], max_logits float32 [T, N] and lse float32 [T, N]."""
    _require_cuda(q, kv, indices, sched, num_splits, workspace, out, max_logits, lse)
    T, N, D = q.shape
    _check(load().mla_sparse_prefill(_ptr(q), _ptr(kv), kv.shape[0], _ptr(indices), int(indices.shape[-1]), T, N,
                                     float(sm_scale), _ptr(sched), _ptr(num_splits), num_partitions, total_splits,
                                     _ptr(workspace), workspace.numel(), _ptr(out), _ptr(max_logits), _ptr(lse), 0,
                                     _stream(stream)))


def mla_swa_plan(kv_indices, page_size: int, kv_run_step: int, runs, topk_lengths=None, stream=None):
    """Window runs: kv_indices int32 [T, topk] cache slots -> runs int32 [T, 4] (slot0, len0, slot1, rows)."""
    _require_cuda(kv_indices, runs, topk_lengths)
    T, topk = kv_indices.shape
    _check(load().mla_swa_plan(_ptr(kv_indices), _ptr(topk_lengths), T, topk, page_size, kv_run_step, _ptr(runs),
                               _stream(stream)))


def mla_decode_runs(q, kv_cache, layout: int, page_size: int, runs, window: int, q_tokens_per_req: int,
                    sm_scale: float, sched, num_splits, num_partitions: int, total_splits: int, workspace, out, lse,
                    sink=None, skip_combine: bool = False, stream=None):
    """Decode where token t attends over the rows of its window runs (runs int32 [T, 4] from
    mla_swa_plan); the plan comes from mla_decode_plan with topk = window."""
    _require_cuda(q, kv_cache, runs, sched, num_splits, workspace, out, lse, sink)
    T, N, D = q.shape
    B = T // q_tokens_per_req
    _check(load().mla_decode_runs(_ptr(q), _ptr(kv_cache), layout, kv_cache.shape[0], page_size, _ptr(runs), window,
                                  B, q_tokens_per_req, N, float(sm_scale), _ptr(sink), _ptr(sched), _ptr(num_splits),
                                  num_partitions, total_splits, _ptr(workspace), workspace.numel(), _ptr(out),
                                  _ptr(lse), 1 if skip_combine else 0, _stream(stream)))


def mla_decode_static_workspace(q, kv_cache, layout: int, page_size: int, block_table, cache_seqlens,
                                q_tokens_per_req: int, sm_scale: float, sched, num_splits, num_partitions: int,
                                total_splits: int, out, lse, sink=None, indices=None, causal: bool = False,
                                status_out=None, stream=None):
    """mla_decode without a caller workspace: for callers that cannot allocate device
    memory, the library's static device workspace (STATIC_WORKSPACE_BYTES) is used.
    status_out: optional device int32/uint32 [1] receiving the call's status bits."""
    _require_cuda(q, kv_cache, block_table, cache_seqlens, sched, num_splits, out, lse, sink, indices, status_out)
    T, N, D = q.shape
    B = cache_seqlens.shape[0]
    topk = 0 if indices is None else int(indices.shape[-1])
    _check(load().mla_decode_static_workspace(
        _ptr(q), _ptr(kv_cache), layout, kv_cache.shape[0], page_size, _ptr(block_table), block_table.shape[1],
        _ptr(cache_seqlens), B, q_tokens_per_req, N, float(sm_scale), _ptr(sink), _ptr(indices), topk,
        int(bool(causal)), _ptr(sched), _ptr(num_splits), num_partitions, total_splits, _ptr(out), _ptr(lse),
        _ptr(status_out), _stream(stream)))


def workspace_partials(workspace, total_splits: int, rows_per_req: int):
    """(part_out [S, R, 512], part_lse [S, R]) float32 views into a decode workspace."""
    import torch
    n = total_splits * rows_per_req
    lse_off = WORKSPACE_HEADER
    out_off = WORKSPACE_HEADER + ((n * 4 + 255) // 256) * 256
    part_lse = workspace[lse_off:lse_off + n * 4].view(torch.float32).view(total_splits, rows_per_req)
    part_out = workspace[out_off:out_off + n * 512 * 4].view(torch.float32).view(total_splits, rows_per_req, 512)
    return part_out, part_lse


def mla_combine(part_out, part_lse, num_splits, rows_per_req: int, num_heads: int, out, lse, sink=None,
                stream=None):
    _require_cuda(part_out, part_lse, num_splits, out, lse, sink)
    B = num_splits.shape[0] - 1
    _check(load().mla_combine(_ptr(part_out), _ptr(part_lse), _ptr(num_splits), B, rows_per_req, num_heads,
                              _ptr(sink), _ptr(out), _ptr(lse), _stream(stream)))


def mla_kv_write(rows, slots, kv_cache, layout: int, page_size: int, status=None, stream=None):
    """Write new rows into their page slots. status: optional device uint32 [1] that
    receives MLA_STATUS_BAD_SLOT (4) for a row whose page is out of range (not written)."""
    _require_cuda(rows, slots, kv_cache, status)
    _check(load().mla_kv_write(_ptr(rows), _ptr(slots), slots.shape[0], _ptr(kv_cache), layout, kv_cache.shape[0],
                               page_size, _ptr(status), _stream(stream)))


def mla_combine_v_up(part_out, part_lse, num_splits, q_tokens_per_req: int, num_heads: int, w_uv, out, lse, o_v,
                     sink=None, status=None, stream=None):
    """Split combine + value up-projection: o_v [T, N, 128] bf16 = bf16 latent out [T, N, 512] x W_UV[n]
    (w_uv bf16 [N, 512, 128]); split requests are merged into out / lse first. part_out / part_lse may be
    None when no request is split. status: optional device uint32 [1] (bit 0: a bounded wait ran out)."""
    _require_cuda(part_out, part_lse, num_splits, w_uv, out, lse, o_v, sink, status)
    B = num_splits.shape[0] - 1
    _check(load().mla_combine_v_up(_ptr(part_out), _ptr(part_lse), _ptr(num_splits), B, q_tokens_per_req, num_heads,
                                   _ptr(sink), _ptr(w_uv), _ptr(out), _ptr(lse), _ptr(o_v), _ptr(status),
                                   _stream(stream)))


def mla_combine_inv_rope(part_out, part_lse, num_splits, q_tokens_per_req: int, num_heads: int, positions, freqs,
                         out, lse, rope0: int = 448, sink=None, stream=None):
    """Split combine + inverse RoPE of out[..., rope0:rope0 + 64] (in place, bf16 [T, N, 512]);
    positions int32 [T]; freqs float32 [max_pos, 64]. part_out / part_lse may be None when no
    request is split."""
    _require_cuda(part_out, part_lse, num_splits, positions, freqs, out, lse, sink)
    B = num_splits.shape[0] - 1
    _check(load().mla_combine_inv_rope(_ptr(part_out), _ptr(part_lse), _ptr(num_splits), B, q_tokens_per_req,
                                       num_heads, _ptr(sink), _ptr(positions), _ptr(freqs), freqs.shape[0], rope0,
                                       _ptr(out), _ptr(lse), _stream(stream)))


def mla_kv_write_norm_rope(raw, slots, positions, norm_weight, eps: float, freqs, kv_cache, layout: int,
                           page_size: int, status=None, stream=None):
    """RMSNorm + RoPE + write of new KV rows: raw bf16 [n, 576] (layouts 0, 2) or [n, 512] (layout 1);
    slots int32 [n]; positions int32 [n]; norm_weight bf16 [512]; freqs float32 [max_pos, 64]
    (32 interleaved (cos, sin) pairs per position). All on the GPU. status: optional device
    uint32 [1] receiving MLA_STATUS_BAD_SLOT (4) / MLA_STATUS_BAD_POSITION (8) for skipped rows."""
    _require_cuda(raw, slots, positions, norm_weight, freqs, kv_cache, status)
    _check(load().mla_kv_write_norm_rope(_ptr(raw), _ptr(slots), _ptr(positions), _ptr(norm_weight), float(eps),
                                         _ptr(freqs), freqs.shape[0], slots.shape[0], _ptr(kv_cache), layout,
                                         kv_cache.shape[0], page_size, _ptr(status), _stream(stream)))


def mla_kv_gather(kv_cache, layout: int, page_size: int, block_table_row, length: int, out, stream=None):
    _require_cuda(kv_cache, block_table_row, out)
    _check(load().mla_kv_gather(_ptr(kv_cache), layout, kv_cache.shape[0], page_size, _ptr(block_table_row),
                                block_table_row.shape[0], length, _ptr(out), _stream(stream)))


def mla_workspace_init(workspace, stream=None):
    _require_cuda(workspace)
    _check(load().mla_workspace_init(_ptr(workspace), _stream(stream)))


def mla_read_status(workspace, reset: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device status word (raises if nonzero)."""
    _require_cuda(workspace)
    st = ctypes.c_uint32()
    _check(load().mla_read_status(_ptr(workspace), ctypes.byref(st), int(reset), _stream(stream)))
    return st.value


def alloc_workspace(nbytes: int, device="cuda"):
    """A 256-byte aligned uint8 workspace with its status header zeroed."""
    import torch
    ws = torch.empty(max(int(nbytes), WORKSPACE_HEADER), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    mla_workspace_init(ws)
    return ws
