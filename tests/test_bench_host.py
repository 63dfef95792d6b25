"""Host logic of bench.py that needs no GPU: the source hash that decides
whether the recorded DRAM traffic of the GEMMs still applies."""

import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_whitespace():
    src = "int a = 1;  // one\n/* block\n comment */ int b =\n  2;\n"
    assert bench._code_only(src) == "int a = 1; int b = 2;"


def _copy_sources(tmp_path):
    csrc = os.path.join(ROOT, "nvfp4_token_quantized_gb300", "csrc")
    dst = tmp_path / "nvfp4_token_quantized_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.GEMM_SOURCES:
        shutil.copy(os.path.join(csrc, f), dst / f)
    return dst


def test_source_hash_ignores_comment_edits_but_not_code_edits(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    p = dst / "kernels.h"
    text = p.read_text()
    p.write_text(text + "\n// a comment added at the end\n/* and a block */\n")
    assert bench.kernel_source_hash() == h0
    p.write_text(text + "\nconstexpr int unused_constant = 1;\n")
    assert bench.kernel_source_hash() != h0

