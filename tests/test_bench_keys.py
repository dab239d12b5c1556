"""Host-side logic of bench.py that decides whether a committed ncu capture
still describes the attention kernel: the fingerprint of its code ignores
comments and blank lines and changes with any code edit."""
import os
import shutil

import bench

CSRC = os.path.join("medusa_tree_speculative_attn_gb300", "csrc")


def _copy_sources(tmp_path):
    os.makedirs(tmp_path / CSRC)
    for f in ("attn_tc.cu", "tc_ptx.cuh", "common.cuh"):
        shutil.copy(os.path.join(bench.ROOT, CSRC, f), tmp_path / CSRC / f)


def test_fingerprint_ignores_comments_but_not_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_code_fingerprint()
    src = tmp_path / CSRC / "attn_tc.cu"
    text = src.read_text()
    src.write_text("// a new comment line\n\n/* and a\n   block comment */\n" +
                   text.replace("namespace mt {", "namespace mt {  // trailing comment", 1))
    assert bench.kernel_code_fingerprint() == base
    src.write_text(text.replace("constexpr int kSmemLimit = 232448;", "constexpr int kSmemLimit = 232447;", 1))
    assert bench.kernel_code_fingerprint() != base


def test_traffic_only_for_the_captured_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    prof = tmp_path / "profiles" / "attn_tc_w.md"
    prof.write_text(f"traffic_bytes_per_launch: 1234\nkernel_code_sha256_16: {bench.kernel_code_fingerprint()}\n")
    assert bench.ncu_traffic("w", "auto") == 1234
    assert bench.ncu_traffic("w", "simt") is None      # another kernel
    assert bench.ncu_traffic("other", "auto") is None  # no capture for that workload
    assert bench.ncu_traffic("w", "auto", "e4m3") is None  # a 16-bit capture for an FP8 cache
    (tmp_path / "profiles" / "attn_tc_e4m3_w.md").write_text(
        f"traffic_bytes_per_launch: 617\nkernel_code_sha256_16: {bench.kernel_code_fingerprint()}\n")
    assert bench.ncu_traffic("w", "auto", "e4m3") == 617
    prof.write_text("traffic_bytes_per_launch: 1234\nkernel_code_sha256_16: 0000000000000000\n")
    assert bench.ncu_traffic("w", "auto") is None      # captured on other code
