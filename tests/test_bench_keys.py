"""Host-side logic of bench.py: whether a committed ncu capture still
describes the attention kernel (the fingerprint of its code ignores comments
and blank lines and changes with any code edit), the algorithmic bytes the
roofline lines divide by, and the whole-job rate."""
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


def test_algorithmic_bytes_of_the_profiled_workload():
    # the serving workload as bench.py draws it (seed 1, rank 0): the bytes the
    # roofline lines divide by, as the committed profiles state them
    import workloads
    w = workloads.generate("serve_b16_gqa_bf16", seed=bench.rank_seed(1, 0), with_logits=False)
    ab = bench.algorithmic_bytes(w)
    assert ab["attn"] == 314_421_248
    B, T, Hq, Hkv, D = w["B"], w["T"], w["Hq"], w["Hkv"], w["head_dim"]
    assert ab["tree_qo"] == B * T * Hq * D * 2 * 2       # bf16 q in, out written
    assert ab["attn"] == ab["prefix_kv"] + ab["tree_qo"] + ab["tree_kv"]
    # an FP8 cache halves the cached bytes only
    ab8 = bench.algorithmic_bytes(w, 1)
    assert ab8["attn"] == 165_599_232
    assert ab8["prefix_kv"] * 2 == ab["prefix_kv"] and ab8["tree_qo"] == ab["tree_qo"]


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(1024, 1, 0.125) == 1024 / 0.125e-3
    assert bench.whole_job_rate(1024, 4, 0.125) == 4 * 1024 / 0.125e-3
