"""Host logic of bench.py: the comment-insensitive kernel digest that ties the
committed ncu summary to the step kernel's sources, and the traffic figure it
gates. No GPU."""
import os
import re
import shutil

import pytest

import bench


def test_code_only_strips_comments_but_keeps_code_and_strings():
    src = '// a line comment\nint x = 1; /* block\n comment */ int y = 2;\nconst char* s = "a // not a comment";\n'
    out = bench._code_only(src)
    assert "comment" not in out.replace("not a comment", "")
    assert 'int x = 1; int y = 2; const char* s = "a // not a comment";' == out
    # whitespace runs collapse, so re-indentation does not change the digest input
    assert bench._code_only("int   a;\n\n\tint b;") == "int a; int b;"


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    csrc = root / "bit_quantized_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.STEP_KERNEL_SOURCES:
        shutil.copy(os.path.join(bench.ROOT, "bit_quantized_moe_gb300", "csrc", f), csrc / f)
    (root / "profiles").mkdir()
    return root, csrc


def test_digest_ignores_comments_and_tracks_code(tmp_path, monkeypatch):
    root, csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    d0 = bench.kernel_source_digest()
    assert d0 == bench.kernel_source_digest()
    f = csrc / "qmv_matvec.cuh"
    text = f.read_text()
    f.write_text("// an added comment line\n" + text.replace("namespace qmv {", "namespace qmv {  /* note */", 1))
    assert bench.kernel_source_digest() == d0
    f.write_text(text.replace("constexpr int kCtasPerSm = 2;", "constexpr int kCtasPerSm = 1;"))
    assert bench.kernel_source_digest() != d0


def test_traffic_only_for_matching_digest(tmp_path, monkeypatch):
    root, csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    prof = root / "profiles" / "mxfp4_gather_2880_top4.md"
    assert bench.traffic_for_current_kernel() is None           # no summary
    prof.write_text(f"dram_bytes_per_launch: 12345\nkernel_source_sha256: {bench.kernel_source_digest()}\n")
    assert bench.traffic_for_current_kernel() == 12345.0
    prof.write_text("dram_bytes_per_launch: 12345\nkernel_source_sha256: " + "0" * 64 + "\n")
    assert bench.traffic_for_current_kernel() is None           # stale summary


def test_committed_profile_names_a_digest_and_traffic():
    txt = open(os.path.join(bench.ROOT, "profiles", "mxfp4_gather_2880_top4.md")).read()
    assert re.search(r"kernel_source_sha256:\s*[0-9a-f]{64}", txt)
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.]+)", txt)
    assert m and float(m.group(1)) > 0
    t = bench.traffic_for_current_kernel()
    assert t is None or t == float(m.group(1))
