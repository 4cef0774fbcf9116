"""bench.kernel_sources_sha256: the hash that decides whether a recorded ncu DRAM-traffic
figure still describes the library's kernels covers their code, not their comments."""
import os
import shutil

import bench


def test_code_only_drops_comments_and_blank_space_but_keeps_literals():
    src = 'int a = 1;  // note\nconst char* s = "// kept";  /* block\n comment */ int b = \'/\';\n\n'
    assert bench._code_only(src) == 'int a = 1; const char* s = "// kept"; int b = \'/\';'
    assert bench._code_only('x = "a\\"//b"; // c') == 'x = "a\\"//b";'


def test_hash_ignores_comment_edits_and_sees_code_edits(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "quantized_kv_cache_decode_gb300", "csrc")
    dst = tmp_path / "quantized_kv_cache_decode_gb300" / "csrc"
    shutil.copytree(csrc, dst, ignore=shutil.ignore_patterns("*.o"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_sources_sha256()
    p = dst / "kvq_common.cuh"
    text = p.read_text(encoding="utf-8")
    p.write_text("// an added comment line\n" + text.replace("\n", "\n\n", 3), encoding="utf-8")
    assert bench.kernel_sources_sha256() == h0
    p.write_text(text + "\nconstexpr int kAnotherConstant = 1;\n", encoding="utf-8")
    assert bench.kernel_sources_sha256() != h0
