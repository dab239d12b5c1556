"""GPU parity of the FP8 (E4M3) KV-cache path against the CPU oracle.

The caches hold E4M3 codes of value / scale (one scale for K, one for V).  The
codes the attention call writes for the tree's keys and values, and the bytes
the commit moves, must match the oracle bit for bit; the attention outputs,
taken over the same dequantised cache, keep the act dtype's tolerance (fp32
1e-5, fp16 2e-3, bf16 1e-2), since both sides read identical cache values.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import medusa_tree_speculative_attn_gb300 as mt
import oracle
import workloads
from gpu_helpers import TOL, Step, to_host

pytestmark = pytest.mark.gpu

CASES = [
    ("fanout_gqa", dict(B=3, Hq=8, Hkv=2, head_dim=128, prefix=("list", [0, 63, 200]),
                        tree=("fanout", (4, 3, 2), 17), max_depth=3)),
    ("chain_d64", dict(B=2, Hq=4, Hkv=4, head_dim=64, prefix=("list", [64, 65]),
                       tree=("chain", 9), max_depth=8)),
    ("single_node", dict(B=4, Hq=4, Hkv=2, head_dim=128, prefix=("list", [1, 15, 16, 17]),
                         tree=("fixed", (-1,)), max_depth=0)),
    ("tree64_g8", dict(B=2, Hq=16, Hkv=2, head_dim=128, prefix=("list", [130, 777]),
                       tree=("fanout", (10, 5, 3, 2), 64), max_depth=4)),
    ("long_ragged", dict(B=3, Hq=8, Hkv=1, head_dim=128, prefix=("list", [1000, 2049, 3]),
                         tree=("fanout", (3, 2, 2, 1), 26), max_depth=4)),
]


def _fp8_workload(spec, seed, k_scale, v_scale):
    """A workload whose caches are E4M3 codes of its N(0,1) act-dtype caches / scale."""
    w = workloads.generate(spec, seed=seed)
    kf = oracle.act_to_f64(w["k_cache"], w["dtype"]).astype(np.float32) / np.float32(k_scale)
    vf = oracle.act_to_f64(w["v_cache"], w["dtype"]).astype(np.float32) / np.float32(v_scale)
    return w, oracle.e4m3_encode(kf.astype(np.float64)), oracle.e4m3_encode(vf.astype(np.float64))


def _step(w, kc, vc, k_scale, v_scale, num_splits=0, kernel="auto"):
    step = Step(w, kernel=kernel, num_splits=num_splits)
    step.d["k_cache"] = torch.from_numpy(kc).view(torch.float8_e4m3fn).cuda()
    step.d["v_cache"] = torch.from_numpy(vc).view(torch.float8_e4m3fn).cuda()
    step.k_scale, step.v_scale = float(k_scale), float(v_scale)
    # the workspace for the kernel that runs (its size depends on the kernel)
    desc = mt.make_desc(step.d["q"], step.d["k_cache"], step.d["block_tables"], num_splits, kernel,
                        k_scale=max(float(k_scale), 1.0), v_scale=max(float(v_scale), 1.0))
    if mt.attn_workspace_size(desc) > 0:   # (0 for a descriptor the library refuses)
        step.ws = mt.alloc_attn_workspace(desc)
    return step


def _oracle_scatter(w, kc, vc, k_scale, v_scale):
    q_rot, k_rot = oracle.rotate_inputs(w)
    kc2, vc2 = oracle.tree_scatter_e4m3(w, kc, vc, k_scale, v_scale, k_rot=k_rot)
    return q_rot, kc2, vc2


# (k_scale, v_scale): amax-style scales (N(0,1) values reach about 5, and 5/448 ~ 0.011), and a
# tight key scale under which the larger keys saturate at +-448
SCALES = [(0.0113, 0.0127), (0.004, 0.02)]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", [c[0] for c in CASES])
@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_fp8_attention_and_scatter(dtype, case, splits, kernel):
    if dtype == "f32" and kernel == "tc":
        pytest.skip("the tensor-core kernel takes fp16/bf16 act dtypes")
    spec = workloads.custom(case, dtype=dtype, **dict(CASES)[case])
    for seed, (ks, vs) in enumerate(SCALES):
        w, kc, vc = _fp8_workload(spec, seed, ks, vs)
        step = _step(w, kc, vc, ks, vs, num_splits=splits, kernel=kernel)
        step.attn()
        assert step.status()[0] == 0
        q_rot, kc2, vc2 = _oracle_scatter(w, kc, vc, ks, vs)
        assert np.array_equal(to_host(step.d["k_cache"]), kc2)
        assert np.array_equal(to_host(step.d["v_cache"]), vc2)
        want = oracle.tree_attn_e4m3(w, kc2, vc2, ks, vs, q_rot=q_rot)
        got = step.out.float().cpu().numpy().astype(np.float64)
        err = np.max(np.abs(got - want))
        assert err <= TOL[dtype], f"max abs error {err}"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_fp8_subnormal_and_every_code_read_exactly(dtype, kernel):
    # Prefix keys drawn from the 14 subnormal codes only, under a K scale that
    # makes the scores depend on them entirely (a reading that flushed them to
    # zero would turn the prefix attention uniform); prefix values drawn from
    # every finite code.  Slots that hold NaN codes (outside the sequences)
    # keep them.  The tree's own K/V codes come from the prep kernel as usual.
    spec = workloads.custom("f8codes", dtype=dtype, **dict(CASES)["fanout_gqa"])
    w, kc, vc = _fp8_workload(spec, 3, 0.0113, 0.0127)
    rng = np.random.default_rng(7)
    sub = np.array([s | m for s in (0x00, 0x80) for m in range(1, 8)], dtype=np.uint8)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    kc = np.where((kc & 0x7F) == 0x7F, kc, rng.choice(sub, kc.shape)).astype(np.uint8)
    vc = np.where((vc & 0x7F) == 0x7F, vc, rng.choice(finite, vc.shape)).astype(np.uint8)
    ks, vs = 300.0, 1.0 / 448.0
    step = _step(w, kc, vc, ks, vs, kernel=kernel)
    step.attn()
    assert step.status()[0] == 0
    q_rot, kc2, vc2 = _oracle_scatter(w, kc, vc, ks, vs)
    assert np.array_equal(to_host(step.d["k_cache"]), kc2)
    want = oracle.tree_attn_e4m3(w, kc2, vc2, ks, vs, q_rot=q_rot)
    got = step.out.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - want)) <= TOL[dtype]
    # the prefix scores matter: the same call with the subnormal keys zeroed
    # gives outputs far from these
    kz = np.where(np.isin(kc, sub), np.uint8(0), kc).astype(np.uint8)
    flat = oracle.tree_attn_e4m3(w, *_oracle_scatter(w, kz, vc, ks, vs)[1:], ks, vs, q_rot=q_rot)
    assert np.max(np.abs(flat - want)) > 20 * TOL[dtype]


def test_fp8_tight_scale_saturates_tree_keys():
    spec = workloads.custom("sat", dtype="bf16", **dict(CASES)["fanout_gqa"])
    w, kc, vc = _fp8_workload(spec, 0, 0.004, 0.02)
    step = _step(w, kc, vc, 0.004, 0.02)
    step.attn()
    _, kc2, _ = _oracle_scatter(w, kc, vc, 0.004, 0.02)
    got = to_host(step.d["k_cache"])
    assert np.array_equal(got, kc2)
    P = w["page_size"]
    tree = np.stack([got[w["block_tables"][b, s // P], :, s % P]
                     for b in range(w["B"]) for s in range(int(w["seq_lens"][b]), int(w["seq_lens"][b]) + w["T"])])
    assert np.any((tree & 0x7F) == 0x7E)     # the tree's keys hold +-448 codes
    assert not np.any((tree & 0x7F) == 0x7F)  # and no NaN codes


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_fp8_fused_accept_commit_moves_codes(dtype):
    for seed, tree in enumerate([("chain", 20), ("fanout", (2, 2, 2, 2, 2), 40), ("chain", 64)]):
        md = tree[1] - 1 if tree[0] == "chain" else 5
        spec = workloads.custom("fp8commit", B=5, Hq=8, Hkv=4, head_dim=128, dtype=dtype,
                                prefix=("list", [0, 15, 16, 17, 300]), tree=tree, max_depth=md,
                                vocab=50, logits_dtype="f32", plant=("uniform", 0, md))
        w, kc, vc = _fp8_workload(spec, seed, 0.0113, 0.0127)
        step = _step(w, kc, vc, 0.0113, 0.0127)
        step.attn()
        step.accept_commit()
        assert step.status() == (0, 0)
        _, kc2, vc2 = _oracle_scatter(w, kc, vc, 0.0113, 0.0127)
        o_am, o_len, o_path, _ = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"],
                                                      w["tree_parents"], md)
        ko, vo, bto, slo, relo = oracle.kv_commit(w, o_path, o_len, kc2, vc2, w["block_tables"],
                                                  w["seq_lens"], md, cache_dtype="e4m3")
        assert np.array_equal(step.am.cpu().numpy(), o_am)
        assert np.array_equal(step.path.cpu().numpy(), o_path)
        assert np.array_equal(step.d["seq_lens"].cpu().numpy(), slo)
        assert np.array_equal(step.d["block_tables"].cpu().numpy(), bto)
        assert np.array_equal(step.rel.cpu().numpy(), relo)
        assert np.array_equal(to_host(step.d["k_cache"]), ko)
        assert np.array_equal(to_host(step.d["v_cache"]), vo)


def test_fp8_two_call_commit_moves_codes():
    spec = workloads.custom("fp8commit2", B=4, Hq=4, Hkv=2, head_dim=64, dtype="bf16",
                            prefix=("list", [0, 16, 31, 300]), tree=("fanout", (3, 2, 2), 20),
                            max_depth=3, vocab=40, logits_dtype="f32", plant=("uniform", 0, 3))
    w, kc, vc = _fp8_workload(spec, 5, 0.0113, 0.0127)
    step = _step(w, kc, vc, 0.0113, 0.0127)
    step.attn()
    step.accept()
    step.commit()
    assert step.status() == (0, 0)
    _, kc2, vc2 = _oracle_scatter(w, kc, vc, 0.0113, 0.0127)
    _, o_len, o_path, _ = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"],
                                               w["tree_parents"], 3)
    ko, vo, _, slo, _ = oracle.kv_commit(w, o_path, o_len, kc2, vc2, w["block_tables"], w["seq_lens"], 3,
                                         cache_dtype="e4m3")
    assert np.array_equal(step.d["seq_lens"].cpu().numpy(), slo)
    assert np.array_equal(to_host(step.d["k_cache"]), ko)
    assert np.array_equal(to_host(step.d["v_cache"]), vo)


def test_fp8_refusals():
    # fp32 act values have no tensor-core kernel, FP8 cache or not
    spec = workloads.custom("fp8tc32", dtype="f32", **dict(CASES)["fanout_gqa"])
    w, kc, vc = _fp8_workload(spec, 0, 0.0113, 0.0127)
    step = _step(w, kc, vc, 0.0113, 0.0127)
    step.kernel = "tc"
    with pytest.raises(mt.MedusaTreeError) as e:
        step.attn()
    assert e.value.status == -2
    # a scale that is not positive
    spec = workloads.custom("fp8tc", dtype="bf16", **dict(CASES)["fanout_gqa"])
    w, kc, vc = _fp8_workload(spec, 0, 0.0113, 0.0127)
    step = _step(w, kc, vc, 0.0, 0.0127)
    with pytest.raises(mt.MedusaTreeError) as e:
        step.attn()
    assert e.value.status == -1


@pytest.mark.parametrize("name", ["serve_b16_gqa_bf16", "verify_b64_fp16"])
def test_fp8_tensor_core_full_size(name):
    # the named workloads' caches as E4M3 codes (amax-style scales), every
    # output against the oracle's reading of the same codes
    w = workloads.generate(name, seed=2, backend="torch", device="cuda")
    w_np = workloads.to_numpy(w)
    ks, vs = 0.0113, 0.0127
    # the cache contents are inputs: torch's own E4M3 cast of value / scale,
    # clamped to +-448 (its cast does not saturate); the oracle alone gives
    # the expected codes of the tree slots and the outputs
    codes = lambda c, sc: ((c.float() / sc).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
                           .view(torch.uint8).cpu().numpy())
    kc, vc = codes(w["k_cache"], ks), codes(w["v_cache"], vs)
    step = _step(w, kc, vc, ks, vs, kernel="tc")
    step.attn()
    assert step.status()[0] == 0
    q_rot, kc2, vc2 = _oracle_scatter(w_np, kc, vc, ks, vs)
    assert np.array_equal(to_host(step.d["k_cache"]), kc2)
    assert np.array_equal(to_host(step.d["v_cache"]), vc2)
    want = oracle.tree_attn_e4m3(w_np, kc2, vc2, ks, vs, q_rot=q_rot)
    got = step.out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - want)) <= TOL[w_np["dtype"]]
