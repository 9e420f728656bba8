#!/usr/bin/env python3
"""Benchmark of the paged-latent MLA decode hot path on GB300.

One step = one pass of the whole path over one batch: mla_kv_write of the
batch's new rows, then mla_decode (persistent decode kernel) and, for requests
the plan split, mla_combine. Inputs are resident in HBM when the timed region
starts; L2 is flushed (a 256 MiB buffer is overwritten) between steps, outside
each step's CUDA-event pair, unless a step reads more than twice the L2 size (then
no flush: inputs larger than L2; the line's config says which).

Default workload (N=1): the DeepSeek-V3-shaped bf16 decode batch — 64 requests
x 1 token, 128 heads, bf16 latent KV rows [512 | 64], context lengths
U{1024..8192}, page 64, seed 0. Other workloads: --config dsv4|verify|sparse|tiny.

Under torchrun (N > 1) every rank runs its own replica (the decode shards by
request and needs no collective); timings are max-reduced over ranks.

--impl reference times the oracle (plain fp64 C, OpenMP) on this machine's
host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode query-tokens/s, KV GB/s and % of roofline on 1 GB300"
UNIT = "query-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_cost(w):
    """Bytes and MMA FLOPs one decode launch must move / perform: every candidate
    KV row once (row + its scale slot for fp8), q, out, lse (and the sparse index
    list); 2 x (D_qk + 512) FLOPs per candidate row and query row."""
    c = w.cfg
    T, N = w.q.shape[0], c.heads
    row_b = {0: 1152, 1: 576 + 8, 2: 640 + 8}[c.layout]
    dqk = {0: 576, 1: 512, 2: 576}[c.layout]
    if w.indices is not None:
        L = np.repeat(w.seqlens, c.sq)[:, None]
        rows_per_token = ((w.indices >= 0) & (w.indices < L)).sum(axis=1)
        kv_rows = int(rows_per_token.sum())          # rows gathered per token (tokens do not share rows)
        scored = int(rows_per_token.sum()) * N
        extra = w.indices.nbytes
    else:
        kv_rows = int(w.seqlens.sum())
        if c.causal:
            scored = 0
            for b in range(c.batch):
                L = int(w.seqlens[b])
                for i in range(c.sq):
                    scored += max(0, min(L, L - c.sq + i + 1)) * N
        else:
            scored = kv_rows * N * c.sq
        extra = 0
    kv_bytes = kv_rows * row_b
    q_bytes = T * N * dqk * 2
    out_bytes = T * N * 512 * 2 + T * N * 4
    flops = 2.0 * scored * (dqk + 512)
    return dict(kv_bytes=kv_bytes, bytes=kv_bytes + q_bytes + out_bytes + extra, flops=flops, kv_rows=kv_rows)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for k, name in enumerate(names):
                    if parts[5 + k].lower() == "active":
                        reasons.add(name)
            os.unlink(self.path)
        except Exception:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def _code_tokens(text):
    """C / C++ / CUDA source with its comments removed and every run of whitespace
    made one space (string and character literals kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The sources that make each decode kernel and its launches (tensor maps, grid, plan): the
# recorded ncu counters of a decode launch depend on these and on nothing else.
DECODE_COMMON = ("mla_paged_latent_gb300/csrc/api.cpp", "mla_paged_latent_gb300/csrc/plan.cpp",
                 "mla_paged_latent_gb300/csrc/decode_common.cuh", "mla_paged_latent_gb300/csrc/ptx_sm103.cuh",
                 "mla_paged_latent_gb300/csrc/mla_kernels.h", "include/mla_decode.h")
DECODE_SOURCES = {"mla_decode_pair_kernel": DECODE_COMMON + ("mla_paged_latent_gb300/csrc/decode_pair_sm103.cu",),
                  "mla_decode_kernel": DECODE_COMMON + ("mla_paged_latent_gb300/csrc/decode_sm103.cu",)}


def source_hash(kernel="mla_decode_pair_kernel"):
    """Hash of one decode kernel's code (DECODE_SOURCES[kernel]; comments and layout of
    whitespace aside): the recorded ncu counters of that kernel stay valid while it is
    unchanged."""
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(rel.encode() + _code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(config_name, kernel):
    """Per-launch DRAM bytes of the decode kernel from a committed ncu summary,
    valid only while that kernel's sources are unchanged."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(config_name)
        if e and e.get("kernel") == kernel and e.get("source_hash") == source_hash(kernel):
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def run_reference(args, rank, world):
    import oracle
    import workloads
    if rank != 0:
        return
    w = workloads.generate(workloads.CONFIGS[args.config]())
    c = w.cfg
    oracle.build()
    T, N = w.q.shape[0], c.heads
    # each step: one head for each of `npairs` distinct tokens, (one oracle call)
    cores = os.cpu_count() or 1
    npairs = min(T, cores)
    kv = oracle.kv_write(w.new_rows, w.new_slots, w.kv_cache, c.layout, c.page_size) if w.new_rows is not None \
        else w.kv_cache
    step_times = []
    for s in range(args.warmup + args.steps):
        toks = (np.arange(npairs) + s * npairs) % T
        heads = (s * 7 + np.arange(npairs)) % N
        t0 = time.perf_counter()
        oracle.mla_decode(w.q, kv, c.layout, c.page_size, w.block_table, w.seqlens, c.sq, c.sm_scale, sink=w.sink,
                          indices=w.indices, causal=c.causal, select=(toks.astype(np.int32), heads.astype(np.int32)))
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            step_times.append(dt)
    total = sum(step_times)
    tokens = len(step_times) * npairs / N
    value = tokens / total
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(step_times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": config_dict(w, args.config),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, npairs), "kind": "oracle",
                             "sample": f"per step {npairs} (token, head) pairs of the {args.config} batch "
                                       f"({npairs}/{N} query-tokens), fp64 oracle, OpenMP over tokens"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x, dist, device="cpu"):
    """The maximum of a per-rank scalar over all ranks (the slowest replica's
    time); x itself when there is no process group."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


CONFIG_DESC = {
    "dsv3": "DSV3-shaped bf16 decode: 64 x 1 token, 128 heads, bf16 KV [512|64], L~U{1024..8192}, page 64",
    "dsv4": "DSV4-shaped fp8 decode: 128 x 1 token, 64 heads, fp8-448+ue8m0/64 KV, L log-uniform [512,32768], "
            "page 64, sink",
    "verify": "speculative verify: 32 x 4 draft tokens (causal), 128 heads, bf16 KV, context U{2048..16384}+4, "
              "page 64, mla_kv_write of the 128 new rows",
    "sparse": "sparse top-k decode: 64 x 1 token, 128 heads, fp8-512+ue8m0/64 KV, L=65536, topk 2048 (10% -1), "
              "page 64, >= 4 splits",
    "tiny": "tiny decode: 2 x 1 token, 16 heads, bf16 KV, L=(37,130), page 16",
}
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}


L2_BYTES = 129 << 20  # GB300 L2 (the device property is used when torch reports it)


def l2_policy(w, l2_bytes=L2_BYTES):
    """Between timed steps, L2 is flushed (a 256 MiB buffer overwritten) unless the bytes one
    step must read are more than twice the L2 size: such inputs cannot stay in L2 from one
    step to the next, and a flush would leave 129 MB of dirty lines whose write-back then
    competes with the measured step."""
    nbytes = algorithmic_cost(w)["bytes"]
    flush = nbytes < 2 * l2_bytes
    note = ("flushed between steps (256 MiB write)" if flush else
            f"not flushed: inputs larger than L2 (a step reads {nbytes / 1e6:.0f} MB, more than twice the "
            f"{l2_bytes / 1e6:.0f} MB L2)")
    return flush, note


def config_dict(w, name):
    c = w.cfg
    return {"workload": CONFIG_DESC[name], "batch": c.batch, "q_tokens_per_req": c.sq, "heads": c.heads,
            "kv_layout": ["bf16-576", "fp8-448-ue8m0", "fp8-512-ue8m0"][c.layout], "page_size": c.page_size,
            "kv_rows": int(w.seqlens.sum()), "seed": c.seed, "l2": l2_policy(w)[1]}


class Rig:
    """One workload resident on the device: inputs, plan, workspace and outputs, and the
    step (kv_write of the new rows + decode (+ combine)) that the bench times."""

    def __init__(self, name, dev, num_sms):
        import torch
        import mla_paged_latent_gb300 as mla
        import workloads
        self.mla, self.torch = mla, torch
        self.name = name
        self.w = w = workloads.generate(workloads.CONFIGS[name](seed=0))
        c = self.c = w.cfg
        self.T, self.N = w.q.shape[0], c.heads
        self.dev = dev

        def bf16(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

        self.q = bf16(w.q)
        self.kv = torch.from_numpy(w.kv_cache).to(dev)
        self.bt = torch.from_numpy(w.block_table).to(dev)
        self.sl = torch.from_numpy(w.seqlens).to(dev)
        self.sink = None if w.sink is None else torch.from_numpy(w.sink).to(dev)
        self.idx = None if w.indices is None else torch.from_numpy(w.indices).to(dev)
        self.rows = None if w.new_rows is None else bf16(w.new_rows)
        self.slots = None if w.new_slots is None else torch.from_numpy(w.new_slots).to(dev)
        self.num_sms = num_sms
        self.plan = mla.mla_decode_plan(w.seqlens, c.sq, self.N, c.topk, c.min_splits, num_sms)
        self.sched = torch.from_numpy(self.plan.sched).to(dev)
        self.ns = torch.from_numpy(self.plan.num_splits).to(dev)
        self.ws = mla.alloc_workspace(self.plan.workspace_bytes, dev)
        self.out = torch.empty(self.T, self.N, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(self.T, self.N, dtype=torch.float32, device=dev)
        self.part_out, self.part_lse = mla.workspace_partials(self.ws, self.plan.total_splits, c.sq * self.N)
        self.split = self.plan.total_splits > c.batch
        self.launches_per_step = (1 if self.rows is not None else 0) + 1 + (1 if self.split else 0)

    def step(self, stream, evs=None, breakdown=False):
        # The step's kernels go back to back on one stream (each may launch while the
        # previous one drains). Events between them would serialise the launches, so the
        # timed pass records only the step boundaries and a second pass the breakdown.
        mla, c = self.mla, self.c
        if evs:
            evs[0].record(stream)
        if self.rows is not None:
            mla.mla_kv_write(self.rows, self.slots, self.kv, c.layout, c.page_size, stream=stream)
        if breakdown:
            evs[1].record(stream)
        mla.mla_decode(self.q, self.kv, c.layout, c.page_size, self.bt, self.sl, c.sq, c.sm_scale, self.sched,
                       self.ns, self.plan.num_partitions, self.plan.total_splits, self.ws, self.out, self.lse,
                       sink=self.sink, indices=self.idx, causal=c.causal, skip_combine=True, stream=stream)
        if breakdown:
            evs[2].record(stream)
        if self.split:
            mla.mla_combine(self.part_out, self.part_lse, self.ns, c.sq * self.N, self.N, self.out, self.lse,
                            sink=self.sink, stream=stream)
        if evs:
            evs[3].record(stream)


def time_rig(rig, args, flush, stream, dist, dev, local):
    """W warm-up steps, then K timed steps (CUDA events at the step boundaries, L2 flushed
    between steps outside the event pairs unless the inputs are larger than L2 (l2_policy),
    nvidia-smi clocks sampled meanwhile), then a breakdown pass with events between the
    kernels."""
    torch, mla = rig.torch, rig.mla
    do_flush = l2_policy(rig.w)[0]
    for _ in range(args.warmup):
        if do_flush:
            flush.fill_(1)
        rig.step(stream)
    torch.cuda.synchronize(dev)
    mla.mla_read_status(rig.ws)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.15)
    for k in range(args.steps):
        if do_flush:
            flush.fill_(k & 0xFF)
        rig.step(stream, events[k])
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if dist is not None:
        dist.barrier()
    mla.mla_read_status(rig.ws)
    step_ms = [e[0].elapsed_time(e[3]) for e in events]
    nbd = min(args.steps, 50)
    bd = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nbd)]
    for k in range(nbd):
        if do_flush:
            flush.fill_(k & 0xFF)
        rig.step(stream, bd[k], breakdown=True)
    torch.cuda.synchronize(dev)
    mla.mla_read_status(rig.ws)
    return {"step_ms": step_ms, "dec_ms": [e[1].elapsed_time(e[2]) for e in bd],
            "kvw_ms": [e[0].elapsed_time(e[1]) for e in bd], "cmb_ms": [e[2].elapsed_time(e[3]) for e in bd],
            "clocks": clocks, "nbd": nbd}


def decode_kernel_name(w):
    """The decode kernel mla_decode launches for this workload: dense bf16 rows whose query
    rows per request come in groups of 128 run on CTA pairs, everything else on the
    single-SM kernel."""
    c = w.cfg
    pair = c.layout == 0 and c.topk == 0 and (c.sq * c.heads) % 128 == 0
    return "mla_decode_pair_kernel" if pair else "mla_decode_kernel"


def roofline_of(w, name, dec_ms, peaks, peak_src):
    """The decode kernel against the slower of its algorithmic bytes at the HBM peak and its
    algorithmic FLOPs at the bf16 tensor peak: the measured peaks (MEASURED_PEAKS.json,
    burst) and, beside them, the nominal GB300 figures (7.9 TB/s, 2.25 PFLOP/s dense)."""
    cost = algorithmic_cost(w)
    dec_avg_s = statistics.mean(dec_ms) * 1e-3
    t_hbm = cost["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = cost["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = cost["bytes"] / dec_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "frac_of_nominal": achieved / NOMINAL_PEAKS["hbm_gbs"]}
    else:
        achieved = cost["flops"] / dec_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "frac_of_nominal": achieved / NOMINAL_PEAKS["bf16_tflops"]}
    roof.update({"traffic": recorded_traffic(name, decode_kernel_name(w)),
                 "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback",
                 "nominal_peak": NOMINAL_PEAKS["hbm_gbs"] if roof["bound"] == "hbm" else NOMINAL_PEAKS["bf16_tflops"],
                 "kernel": decode_kernel_name(w), "alg_bytes_per_launch": cost["bytes"],
                 "alg_flops_per_launch": cost["flops"], "kernel_ms": statistics.mean(dec_ms),
                 "roofline_ms": 1e3 * max(t_hbm, t_tc)})
    return roof, cost


def cpu_baseline_of(w, name, budget_s):
    """The oracle as it stands (fp64 C, OpenMP over tokens) on this host's cores: whole
    passes (kv_write + decode of a sample of the batch's tokens) until about budget_s."""
    import oracle
    oracle.build()
    c = w.cfg
    T, N = w.q.shape[0], c.heads
    toks = np.arange(T) if name in ("dsv3", "tiny", "dsv4") else np.arange(min(T, 32))
    sel_t = np.repeat(toks, N).astype(np.int32)
    sel_n = np.tile(np.arange(N), len(toks)).astype(np.int32)
    t0 = time.perf_counter()
    passes, dt = 0, 0.0
    while passes == 0 or (dt < budget_s and passes < 8):
        kv_o = oracle.kv_write(w.new_rows, w.new_slots, w.kv_cache, c.layout, c.page_size) \
            if w.new_rows is not None else w.kv_cache
        oracle.mla_decode(w.q, kv_o, c.layout, c.page_size, w.block_table, w.seqlens, c.sq, c.sm_scale,
                          sink=w.sink, indices=w.indices, causal=c.causal, select=(sel_t, sel_n))
        passes += 1
        dt = time.perf_counter() - t0
    return {"value": passes * len(toks) / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(toks)} query tokens x {N} heads of the {name} batch (+ its kv_write), "
                      f"{passes} pass(es), fp64 C oracle, OpenMP over tokens, {dt:.1f} s"}


def _rope_freqs(max_pos):
    theta = np.outer(np.arange(max_pos), 10000.0 ** (-np.arange(32) / 32.0))
    ftab = np.zeros((max_pos, 64), np.float32)
    ftab[:, 0::2], ftab[:, 1::2] = np.cos(theta), np.sin(theta)
    return ftab


def next_row_extras(rig, flush, stream, dev, nbd):
    """The next-row kernels timed alone on this workload's step outputs (L2 flushed):
    combine + W_UV up-projection (576-wide rows), combine + inverse RoPE and the
    sliding-window plan + decode (the DSV4 row), and the fused RMSNorm + RoPE write."""
    torch, mla, w, c = rig.torch, rig.mla, rig.w, rig.c
    T, N, out, lse, split = rig.T, rig.N, rig.out, rig.lse, rig.split
    part_out, part_lse, ns, plan = rig.part_out, rig.part_lse, rig.ns, rig.plan
    res = {"combine_v_up": None, "combine_inv_rope": None, "swa_decode": None, "kv_write_norm_rope": None}
    if c.layout != 1:
        gen = torch.Generator(device=dev).manual_seed(0)
        w_uv = (torch.randn(N, 512, 128, device=dev, generator=gen) * 0.05).to(torch.bfloat16)
        o_v = torch.empty(T, N, 128, dtype=torch.bfloat16, device=dev)
        out_keep, lse_keep = out.clone(), lse.clone()
        ck = []
        for k in range(nbd):
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mla.mla_combine_v_up(part_out if split else None, part_lse if split else None, ns, c.sq, N, w_uv, out, lse,
                                 o_v, sink=rig.sink, stream=stream)
            e1.record(stream)
            ck.append((e0, e1))
        torch.cuda.synchronize(dev)
        us = statistics.mean(a.elapsed_time(b) for a, b in ck) * 1e3
        nsplit_rows = int((np.diff(plan.num_splits) >= 2).astype(np.int64) @ np.full(c.batch, c.sq * N))
        part_bytes = (plan.total_splits * c.sq * N * (512 * 4 + 4)) if split else 0
        nbytes = N * 512 * 128 * 2 + part_bytes + T * N * 512 * 2 + nsplit_rows * (512 * 2 + 4) + T * N * 128 * 2
        flops = 2.0 * T * N * 512 * 128
        res["combine_v_up"] = {
            "us": us, "alg_bytes": nbytes, "gbps": nbytes / (us * 1e-6) / 1e9, "tflops": flops / (us * 1e-6) / 1e12,
            "note": "merge of split rows + bf16 latent x W_UV[n] (dv 128) as tcgen05 MMAs, one CTA per head; "
                    "W_UV random bf16; L2 flushed"}
        out.copy_(out_keep)   # the merged rows it rewrote; the e2e check compares against the decode's own
        lse.copy_(lse_keep)
    if c.layout == 1:
        tpos = np.concatenate([np.arange(int(L) - c.sq, int(L)) for L in w.seqlens]).astype(np.int32)
        max_pos = int(w.seqlens.max()) + 1
        d_tpos, d_ftab = torch.from_numpy(tpos).to(dev), torch.from_numpy(_rope_freqs(max_pos)).to(dev)
        out_keep, lse_keep = out.clone(), lse.clone()
        ck = []
        for k in range(nbd):
            out.copy_(out_keep)
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mla.mla_combine_inv_rope(part_out if split else None, part_lse if split else None, ns, c.sq, N, d_tpos,
                                     d_ftab, out, lse, rope0=448, sink=rig.sink, stream=stream)
            e1.record(stream)
            ck.append((e0, e1))
        torch.cuda.synchronize(dev)
        out.copy_(out_keep)
        lse.copy_(lse_keep)
        us = statistics.mean(a.elapsed_time(b) for a, b in ck) * 1e3
        nsplit_rows = int((np.diff(plan.num_splits) >= 2).astype(np.int64) @ np.full(c.batch, c.sq * N))
        part_bytes = (plan.total_splits * c.sq * N * (512 * 4 + 4)) if split else 0
        nbytes = part_bytes + (T * N - nsplit_rows) * 1024 + T * N * 1024 + nsplit_rows * 4 + T * 4
        res["combine_inv_rope"] = {
            "us": us, "alg_bytes": nbytes, "gbps": nbytes / (us * 1e-6) / 1e9,
            "note": "merge of split rows + inverse RoPE of elements 448..511 of every row, in place; L2 flushed"}
        # Sliding-window variant on the same cache: every token attends over a window of 96
        # consecutive cache slots straddling two 64-row pages (two runs), made by mla_swa_plan and
        # decoded by mla_decode_runs with the planner's top-k schedule (window 96).
        window, ps, npg = 96, c.page_size, rig.kv.shape[0]
        srng = np.random.default_rng(7)
        first = srng.integers(0, npg - 2, T) * ps + srng.integers(1, 2 * ps - window + 1, T)
        widx = (first[:, None] + np.arange(window)[None, :]).astype(np.int32)
        d_widx = torch.from_numpy(widx).to(dev)
        d_runs = torch.zeros(T, 4, dtype=torch.int32, device=dev)
        splan = mla.mla_decode_plan(np.full(c.batch, window, np.int32), c.sq, N, window, 1, rig.num_sms)
        s_sched, s_ns = torch.from_numpy(splan.sched).to(dev), torch.from_numpy(splan.num_splits).to(dev)
        s_ws = mla.alloc_workspace(splan.workspace_bytes, dev)
        s_out, s_lse = torch.empty_like(out), torch.empty_like(lse)
        tp, td = [], []
        for k in range(nbd):
            flush.fill_(k & 0xFF)
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            mla.mla_swa_plan(d_widx, ps, 1, d_runs, stream=stream)
            e1.record(stream)
            mla.mla_decode_runs(rig.q, rig.kv, c.layout, ps, d_runs, window, c.sq, c.sm_scale, s_sched, s_ns,
                                splan.num_partitions, splan.total_splits, s_ws, s_out, s_lse, sink=rig.sink,
                                stream=stream)
            e2.record(stream)
            tp.append((e0, e1))
            td.append((e1, e2))
        torch.cuda.synchronize(dev)
        mla.mla_read_status(s_ws)
        assert np.all(d_runs.cpu().numpy()[:, 3] == window)
        res["swa_decode"] = {
            "window": window, "tokens": T, "us_plan": statistics.mean(a.elapsed_time(b) for a, b in tp) * 1e3,
            "us_decode": statistics.mean(a.elapsed_time(b) for a, b in td) * 1e3,
            "note": "per token 96 consecutive cache slots over two pages (two runs); plan + decode (+ combine); "
                    "L2 flushed"}
    if rig.rows is not None:
        # the fused RMSNorm + RoPE + write of the same new rows (raw rows in, cache rows out); it
        # rewrites those slots, so the plain write puts the step's rows back afterwards
        nr = int(w.new_rows.shape[0])
        kpos = np.concatenate([np.arange(int(L) - c.sq, int(L)) for L in w.seqlens]).astype(np.int32)
        max_pos = int(w.seqlens.max()) + 1
        d_pos, d_f = torch.from_numpy(kpos).to(dev), torch.from_numpy(_rope_freqs(max_pos)).to(dev)
        d_w = torch.ones(512, dtype=torch.bfloat16, device=dev)
        nk = []
        for k in range(nbd):
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mla.mla_kv_write_norm_rope(rig.rows, rig.slots, d_pos, d_w, 1e-6, d_f, rig.kv, c.layout, c.page_size,
                                       stream=stream)
            e1.record(stream)
            nk.append((e0, e1))
        torch.cuda.synchronize(dev)
        mla.mla_kv_write(rig.rows, rig.slots, rig.kv, c.layout, c.page_size, stream=stream)
        us = statistics.mean(a.elapsed_time(b) for a, b in nk) * 1e3
        row_elems = w.new_rows.shape[1]
        row_out = {0: 1152, 1: 584, 2: 648}[c.layout]
        nbytes = nr * (row_elems * 2 + row_out + 4 + 4 + 64 * 4) + 512 * 2
        res["kv_write_norm_rope"] = {
            "rows": nr, "us": us, "alg_bytes": nbytes, "gbps": nbytes / (us * 1e-6) / 1e9,
            "note": "raw rows -> RMSNorm + RoPE (fp32) -> bf16 -> cache rows; L2 flushed; launch-bound at this size"}
    return res


def sparse_prefill_entry(flush, stream, dev, nbd, num_sms, peaks, peak_src, cpu_budget_s):
    """mla_sparse_prefill (flash_mla_sparse_fwd's contract) on a prefill-shaped batch: 512 query
    tokens x 128 heads over one unpaged bf16 latent run of 32768 rows, 2048 distinct indices
    per token (seeded), sm_scale 1/sqrt(192); the decode + combine timed with CUDA events,
    L2 flushed. Bound by the tensor pipe: the gathered rows are reused across tokens."""
    import torch
    import mla_paged_latent_gb300 as mla
    T, N, s_kv, topk = 512, 128, 32768, 2048
    gen = torch.Generator(device=dev).manual_seed(11)
    q = torch.randn(T, N, 576, device=dev, generator=gen).to(torch.bfloat16)
    kv = torch.randn(s_kv, 576, device=dev, generator=gen).to(torch.bfloat16)
    idx = torch.rand(T, s_kv, device=dev, generator=gen).argsort(dim=1)[:, :topk].to(torch.int32).contiguous()
    scale = 1.0 / math.sqrt(192.0)
    plan = mla.mla_decode_plan(np.full(T, s_kv, np.int32), 1, N, topk, 1, num_sms)
    sched, ns = torch.from_numpy(plan.sched).to(dev), torch.from_numpy(plan.num_splits).to(dev)
    ws = mla.alloc_workspace(plan.workspace_bytes, dev)
    out = torch.empty(T, N, 512, dtype=torch.bfloat16, device=dev)
    mx = torch.empty(T, N, dtype=torch.float32, device=dev)
    lse = torch.empty(T, N, dtype=torch.float32, device=dev)
    evs = []
    for k in range(nbd + 3):
        flush.fill_(k & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mla.mla_sparse_prefill(q, kv, idx, scale, sched, ns, plan.num_partitions, plan.total_splits, ws, out, mx, lse,
                               stream=stream)
        e1.record(stream)
        if k >= 3:
            evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    assert mla.mla_read_status(ws) == 0
    us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    flops = 2.0 * T * N * topk * (576 + 512)
    nbytes = T * N * 576 * 2 + s_kv * 1152 + T * topk * 4 + T * N * (512 * 2 + 4 + 4)
    tflops = flops / (us * 1e-6) / 1e12
    entry = {"config": {"workload": f"sparse prefill: {T} tokens x {N} heads, unpaged bf16 latent run of {s_kv} "
                                    f"rows, {topk} indices per token, sm_scale 1/sqrt(192)"},
             "value": T / (us * 1e-6), "unit": UNIT, "kernel_us": us,
             "plan": {"partitions": plan.num_partitions, "total_splits": plan.total_splits},
             "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                          "frac": tflops / peaks["bf16_tflops"],
                          "frac_of_nominal": tflops / NOMINAL_PEAKS["bf16_tflops"], "traffic": None,
                          "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback",
                          "alg_flops_per_launch": flops, "alg_bytes_per_launch": nbytes,
                          "kernel": "mla_decode_kernel (bf16 gather) + combine_kernel"},
             "cpu_baseline": None}
    if cpu_budget_s > 0:
        import oracle
        oracle.build()
        q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
        kv_bits = kv.view(torch.int16).cpu().numpy().view(np.uint16)
        idx_h = idx.cpu().numpy()
        t0, done = time.perf_counter(), 0
        while done == 0 or (time.perf_counter() - t0 < cpu_budget_s and done < T):
            oracle.sparse_prefill(q_bits[done:done + 4], kv_bits, idx_h[done:done + 4], scale)
            done += 4
        dt = time.perf_counter() - t0
        entry["cpu_baseline"] = {"value": done / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": f"{done} query tokens x {N} heads of the same batch, fp64 C oracle, "
                                           f"OpenMP over tokens, {dt:.1f} s"}
    return entry


def run_e2e(rig, args, dist, dev, world):
    """End to end through the public API with host buffers (pinned), copies inside the
    timed region. A serving loop: every step plans on the host, copies its inputs host ->
    device, runs kv_write + decode (+ combine) and copies out / lse back to the host. Three
    streams overlap the copies of neighbouring steps with the compute of the current one
    (inputs, outputs and host output buffers are double-buffered; events order every reuse),
    compute stays in step order on one stream, and the clock runs from the first copy to the
    last one landing on the host. All of a step's inputs live in one pinned host buffer and
    move in one copy; out and lse come back in one copy too."""
    torch, mla, w, c = rig.torch, rig.mla, rig.w, rig.c
    T, N, kv, ws, sink = rig.T, rig.N, rig.kv, rig.ws, rig.sink
    num_sms = rig.num_sms
    p0 = mla.mla_decode_plan(w.seqlens, c.sq, N, c.topk, c.min_splits, num_sms)
    nb = 2
    in_fields = [("q", w.q.view(np.int16)), ("rows", None if w.new_rows is None else w.new_rows.view(np.int16)),
                 ("slots", w.new_slots), ("bt", w.block_table), ("sl", w.seqlens), ("idx", w.indices),
                 ("sched", p0.sched), ("ns", p0.num_splits)]
    in_off, in_bytes = {}, 0
    for name, arr in in_fields:
        if arr is not None:
            in_off[name] = (in_bytes, arr.nbytes, arr.dtype, arr.shape)
            in_bytes += (arr.nbytes + 255) // 256 * 256
    res_fields = [("out", T * N * 512 * 2, np.int16, (T, N, 512)), ("lse", T * N * 4, np.float32, (T, N))]
    res_off, res_bytes = {}, 0
    for name, n, dt, shp in res_fields:
        res_off[name] = (res_bytes, n, np.dtype(dt), shp)
        res_bytes += (n + 255) // 256 * 256
    tdt = {np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32, np.dtype(np.float32): torch.float32}

    def view(buf, off, name):
        o, n, dt, shp = off[name]
        return buf[o:o + n].view(tdt[np.dtype(dt)]).view(shp)

    hin = [torch.empty(in_bytes, dtype=torch.uint8).pin_memory() for _ in range(nb)]
    din = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(nb)]
    hres = [torch.empty(res_bytes, dtype=torch.uint8).pin_memory() for _ in range(nb)]
    dres = [torch.empty(res_bytes, dtype=torch.uint8, device=dev) for _ in range(nb)]
    for b in range(nb):
        for name, arr in in_fields:
            if arr is not None and name not in ("sched", "ns"):
                view(hin[b], in_off, name).numpy()[...] = arr
    dv = [{name: view(din[b], in_off, name) for name in in_off} for b in range(nb)]
    hsch = [view(hin[b], in_off, "sched").numpy() for b in range(nb)]
    hns = [view(hin[b], in_off, "ns").numpy() for b in range(nb)]
    dout = [view(dres[b], res_off, "out").view(torch.bfloat16) for b in range(nb)]
    dlse = [view(dres[b], res_off, "lse") for b in range(nb)]
    hout = [view(hres[b], res_off, "out") for b in range(nb)]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_done, comp_done, out_done = ([torch.cuda.Event() for _ in range(nb)] for _ in range(3))
    used = [False] * nb

    def e2e_step(i):
        b = i % nb
        p = mla.mla_decode_plan(w.seqlens, c.sq, N, c.topk, c.min_splits, num_sms)
        assert p.sched.shape == p0.sched.shape
        if used[b]:
            in_done[b].synchronize()              # the pinned inputs of step i - 2 have been read
        hsch[b][...] = p.sched
        hns[b][...] = p.num_splits
        d = dv[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])     # step i - 2 no longer reads these inputs
            din[b].copy_(hin[b], non_blocking=True)
            in_done[b].record(s_in)
        s_comp.wait_event(in_done[b])
        if used[b]:
            s_comp.wait_event(out_done[b])        # out / lse of step i - 2 are on the host
        if "rows" in d:
            mla.mla_kv_write(d["rows"].view(torch.bfloat16), d["slots"], kv, c.layout, c.page_size, stream=s_comp)
        mla.mla_decode(d["q"].view(torch.bfloat16), kv, c.layout, c.page_size, d["bt"], d["sl"], c.sq, c.sm_scale,
                       d["sched"], d["ns"], p.num_partitions, p.total_splits, ws, dout[b], dlse[b], sink=sink,
                       indices=d.get("idx"), causal=c.causal, stream=s_comp)
        comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            hres[b].copy_(dres[b], non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for i in range(5):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i)
    for b in range(nb):
        out_done[b].synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    # the last step's results must equal those of the device-timed path
    matches = bool(torch.equal(hout[(args.e2e_steps - 1) % nb], rig.out.view(torch.int16).cpu()))
    return {"value": world * T * args.e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(in_bytes),
            "d2h_bytes_per_step": int(res_bytes), "steps": args.e2e_steps, "matches_device_path": matches,
            "includes": "per step: host plan, one pinned H2D copy of the packed q/new rows/slots/"
                        "block_table/seqlens/indices/plan, kv_write, decode, combine, one D2H copy of "
                        "out+lse; copies of neighbouring steps overlap the current step's compute "
                        "(3 streams, double-buffered, event-ordered)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="dsv3", choices=["dsv3", "dsv4", "verify", "sparse", "tiny"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true", help="time the --config workload alone (no other workloads)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)

    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return

    import torch

    import mla_paged_latent_gb300 as mla
    from mla_paged_latent_gb300 import build as mla_build

    if rank == 0 or world == 1:
        mla_build.build()
    if dist is not None:
        dist.barrier()
    mla.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    # ---- the headline workload: timed steps, breakdown, next-row kernels, e2e
    rig = Rig(args.config, dev, num_sms)
    w, c, T, N = rig.w, rig.c, rig.T, rig.N
    tm = time_rig(rig, args, flush, stream, dist, dev, local)
    extras = next_row_extras(rig, flush, stream, dev, tm["nbd"])
    total_ms = max_over_ranks(sum(tm["step_ms"]), dist, dev)
    ms_per_step = total_ms / args.steps
    value = world * T / (ms_per_step * 1e-3)
    e2e = run_e2e(rig, args, dist, dev, world)
    roof, cost = roofline_of(w, args.config, tm["dec_ms"], peaks, peak_src)
    roof["step_frac_of_roofline"] = roof["roofline_ms"] / ms_per_step
    launches = rig.launches_per_step * args.steps
    headline_plan = {"partitions": rig.plan.num_partitions, "groups": rig.plan.groups,
                     "total_splits": rig.plan.total_splits}
    del rig

    # ---- the other workloads of the same metric, each timed the same way (replicas on every rank)
    others = {}
    if not args.only and args.config == "dsv3":
        for name in ("dsv4", "verify", "sparse"):
            torch.cuda.empty_cache()
            r2 = Rig(name, dev, num_sms)
            t2 = time_rig(r2, args, flush, stream, dist, dev, local)
            ms2 = max_over_ranks(sum(t2["step_ms"]), dist, dev) / args.steps
            roof2, cost2 = roofline_of(r2.w, name, t2["dec_ms"], peaks, peak_src)
            roof2["step_frac_of_roofline"] = roof2["roofline_ms"] / ms2
            ex2 = next_row_extras(r2, flush, stream, dev, t2["nbd"])
            entry = {"config": config_dict(r2.w, name), "value": world * r2.T / (ms2 * 1e-3), "unit": UNIT,
                     "ms_per_step": ms2, "steps": args.steps, "warmup": args.warmup,
                     "kv_gbps": world * cost2["kv_bytes"] / (ms2 * 1e-3) / 1e9,
                     "kernel_ms": {"kv_write": statistics.mean(t2["kvw_ms"]), "decode": statistics.mean(t2["dec_ms"]),
                                   "combine": statistics.mean(t2["cmb_ms"])},
                     "roofline": roof2, "clocks": t2["clocks"],
                     "plan": {"partitions": r2.plan.num_partitions, "groups": r2.plan.groups,
                              "total_splits": r2.plan.total_splits},
                     "cpu_baseline": None}
            entry.update({k: v for k, v in ex2.items() if v is not None})
            if world == 1 and rank == 0 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline_of(r2.w, name, 5.0)
            launches += r2.launches_per_step * args.steps
            others[name] = entry
            del r2
        torch.cuda.empty_cache()
        others["sparse_prefill"] = sparse_prefill_entry(
            flush, stream, dev, max(5, min(tm["nbd"], 20)), num_sms, peaks, peak_src,
            5.0 if (world == 1 and rank == 0 and not args.no_cpu_baseline) else 0.0)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_of(w, args.config, 10.0)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(w, args.config),
            "kv_gbps": world * cost["kv_bytes"] / (ms_per_step * 1e-3) / 1e9,
            "kernel_ms": {"kv_write": statistics.mean(tm["kvw_ms"]), "decode": statistics.mean(tm["dec_ms"]),
                          "combine": statistics.mean(tm["cmb_ms"])},
            "kv_write_norm_rope": extras["kv_write_norm_rope"],
            "combine_v_up": extras["combine_v_up"],
            "combine_inv_rope": extras["combine_inv_rope"],
            "swa_decode": extras["swa_decode"],
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches,
            "plan": headline_plan,
            "clocks": tm["clocks"],
            "workloads": others or None}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
