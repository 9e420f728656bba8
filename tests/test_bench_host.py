"""Host logic of bench.py that needs no GPU: the code hash that keys the recorded
ncu counters (comments and whitespace layout do not change it; code does)."""
import os
import shutil

import bench


def test_code_tokens_drop_comments_keep_literals():
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x//y /* z */";\nchar q = \'"\';\n'
    assert bench._code_tokens(src) == 'int a = 1; const char* s = "x//y /* z */"; char q = \'"\';'


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    for sub in ("mla_paged_latent_gb300/csrc", "include"):
        shutil.copytree(os.path.join(bench.ROOT, sub), tmp_path / sub)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash("mla_decode_kernel")
    hp = bench.source_hash("mla_decode_pair_kernel")
    # a comment and blank lines in a decode source: same hash
    p = tmp_path / "mla_paged_latent_gb300" / "csrc" / "decode_common.cuh"
    text = p.read_text()
    p.write_text("// an added comment line\n" + text.replace("\n", "\n\n", 3))
    assert bench.source_hash("mla_decode_kernel") == h0
    # code of a source both decode kernels use: new hashes for both
    assert "ex2.approx.ftz.f32" in text
    p.write_text(text.replace("ex2.approx.ftz.f32", "ex2.approx.f32", 1))
    assert bench.source_hash("mla_decode_kernel") != h0
    assert bench.source_hash("mla_decode_pair_kernel") != hp
    p.write_text(text)
    # code of the single-SM kernel alone: the pair kernel's counters stay valid
    sk = tmp_path / "mla_paged_latent_gb300" / "csrc" / "decode_sm103.cu"
    st = sk.read_text()
    sk.write_text(st + "\nstatic int unused_probe_value = 1;\n")
    assert bench.source_hash("mla_decode_kernel") != h0
    assert bench.source_hash("mla_decode_pair_kernel") == hp
    sk.write_text(st)
    # code outside the decode kernels (the combine's merge): the decode's counters stay valid
    q = tmp_path / "mla_paged_latent_gb300" / "csrc" / "combine_row.cuh"
    qt = q.read_text()
    assert "acc[i] *= f;" in qt
    q.write_text(qt.replace("acc[i] *= f;", "acc[i] *= 2.f * f;", 1))
    assert bench.source_hash("mla_decode_kernel") == h0
    assert bench.source_hash("mla_decode_pair_kernel") == hp


def test_algorithmic_cost_tiny_closed_form():
    """The roofline numerator on the tiny workload (2 requests of 37 and 130 rows, 16
    heads, bf16 rows of 1152 B): every KV row once, q, out and lse; 2 x (576 + 512)
    FLOPs per (row, query row)."""
    import workloads
    w = workloads.generate(workloads.tiny())
    c = bench.algorithmic_cost(w)
    T, N = 2, 16
    assert c["kv_rows"] == 37 + 130
    assert c["kv_bytes"] == 167 * 1152
    assert c["bytes"] == 167 * 1152 + T * N * 576 * 2 + T * N * 512 * 2 + T * N * 4
    assert c["flops"] == 2.0 * 167 * N * (576 + 512)


def test_algorithmic_cost_causal_and_sparse_by_brute_force():
    """Causal verify counts, per draft token i, the rows j <= L - s_q + i; sparse counts
    the valid listed entries (0 <= idx < L) once per token."""
    import numpy as np
    import workloads
    w = workloads.generate(workloads.verify(batch=3, sq=4, heads=16, seqlens=(2, 9, 70), len_dist="fixed"))
    scored = sum(sum(1 for j in range(L) if j <= L - 4 + i) for L in (2, 9, 70) for i in range(4))
    assert bench.algorithmic_cost(w)["flops"] == 2.0 * scored * 16 * (576 + 512)
    w = workloads.generate(workloads.sparse(batch=2, seqlens=(900, 4000), topk=256, len_dist="fixed"))
    valid = sum(int(((w.indices[t] >= 0) & (w.indices[t] < w.seqlens[t])).sum()) for t in range(2))
    c = bench.algorithmic_cost(w)
    assert c["kv_rows"] == valid
    assert c["kv_bytes"] == valid * (640 + 8)
    assert c["flops"] == 2.0 * valid * 128 * (576 + 512)
    assert c["bytes"] == valid * 648 + 2 * 128 * 576 * 2 + 2 * 128 * 512 * 2 + 2 * 128 * 4 + w.indices.nbytes
