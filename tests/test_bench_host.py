"""Host logic of bench.py that needs no GPU: the code hash that keys the recorded
ncu counters (comments and whitespace layout do not change it; code does)."""
import os
import shutil

import bench


def test_code_tokens_drop_comments_keep_literals():
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x//y /* z */";\nchar q = \'"\';\n'
    assert bench._code_tokens(src) == 'int a = 1; const char* s = "x//y /* z */"; char q = \'"\';'


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "mla_paged_latent_gb300", "csrc")
    dst = tmp_path / "mla_paged_latent_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash()
    p = dst / "combine_row.cuh"
    text = p.read_text()
    p.write_text("// an added comment line\n" + text.replace("\n", "\n\n", 3))
    assert bench.source_hash() == h0
    p.write_text(text.replace("acc[i] *= f;", "acc[i] *= 2.f * f;", 1))
    assert bench.source_hash() != h0
