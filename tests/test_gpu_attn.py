"""GPU parity of tree attention (through the C ABI) against the CPU oracle.

Tolerances (max abs error on outputs read back from the act dtype, inputs
N(0,1)): fp32 1e-5, fp16 2e-3, bf16 1e-2.  The tree keys the call writes into
the cache's scratch slots must equal the oracle's rotated keys bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads
from gpu_helpers import TOL, Step, to_host

pytestmark = pytest.mark.gpu

KERNELS_16 = ["simt", "tc"]


def _kernels(dtype):
    return ["simt"] if dtype == "f32" else KERNELS_16


def _check_full(w, step):
    want = oracle.tree_attn(w)
    got = step.out.float().cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - want))
    assert err <= TOL[w["dtype"]], f"max abs error {err}"
    return err


def _check_scatter(w, step):
    _, k_rot = oracle.rotate_inputs(w)
    kc, vc = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
    assert np.array_equal(to_host(step.d["k_cache"]).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(to_host(step.d["v_cache"]).view(np.uint8), vc.view(np.uint8))


SMALL = [
    # (name, spec kwargs)
    ("fanout_gqa", dict(B=3, Hq=8, Hkv=2, head_dim=128, prefix=("list", [0, 63, 200]),
                        tree=("fanout", (4, 3, 2), 17), max_depth=3)),
    ("chain", dict(B=2, Hq=4, Hkv=4, head_dim=128, prefix=("list", [64, 65]),
                   tree=("chain", 9), max_depth=8)),
    ("star", dict(B=2, Hq=2, Hkv=1, head_dim=64, prefix=("list", [16, 1]),
                  tree=("star", 12), max_depth=1)),
    ("single_node", dict(B=4, Hq=4, Hkv=2, head_dim=128, prefix=("list", [1, 15, 16, 17]),
                         tree=("fixed", (-1,)), max_depth=0)),
    ("tree64_g8", dict(B=2, Hq=16, Hkv=2, head_dim=128, prefix=("list", [130, 777]),
                       tree=("fanout", (10, 5, 3, 2), 64), max_depth=4)),
    ("long_ragged", dict(B=3, Hq=8, Hkv=1, head_dim=128, prefix=("list", [1000, 2049, 3]),
                         tree=("fanout", (3, 2, 2, 1), 26), max_depth=4)),
]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", [c[0] for c in SMALL])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_small_cases(dtype, case, splits):
    kw = dict(SMALL)[case]
    spec = workloads.custom(case, dtype=dtype, **kw)
    for kernel in _kernels(dtype):
        for seed in range(2):
            w = workloads.generate(spec, seed=seed)
            step = Step(w, kernel=kernel, num_splits=splits)
            step.attn()
            assert step.status()[0] == 0
            _check_full(w, step)
            _check_scatter(w, step)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("splits", [3, 8])
def test_split_chunks_past_short_segments_are_never_read(dtype, splits):
    # with more key chunks than a segment has tiles, the leading chunks are
    # empty and no kernel writes their partial slots: fill the workspace with
    # NaN bytes (past the status word) so that reading one would show
    kw = dict(B=3, Hq=4, Hkv=2, head_dim=128, prefix=("list", [16, 1, 70]),
              tree=("fanout", (3, 2), 9), max_depth=2)
    spec = workloads.custom("short_split", dtype=dtype, **kw)
    for kernel in _kernels(dtype):
        w = workloads.generate(spec, seed=3)
        step = Step(w, kernel=kernel, num_splits=splits)
        step.ws.fill_(0xFF)
        step.ws[:256].zero_()
        step.attn()
        assert step.status()[0] == 0
        assert torch.isfinite(step.out.float()).all()
        _check_full(w, step)


def test_tiny_tree_fp32():
    w = workloads.generate("tiny_tree_fp32", seed=0)
    step = Step(w)
    step.attn()
    assert step.status()[0] == 0
    _check_full(w, step)
    _check_scatter(w, step)


@pytest.mark.parametrize("kernel", KERNELS_16)
def test_llama7b_b1_fp16_full(kernel):
    w = workloads.generate("llama7b_b1_fp16", seed=0)
    step = Step(w, kernel=kernel)
    step.attn()
    assert step.status()[0] == 0
    _check_full(w, step)
    _check_scatter(w, step)


_LARGE = {}


def _large(name):
    """The workload (on the device), its NumPy copy and the oracle's full
    output, computed once per workload and shared by every kernel variant."""
    if name not in _LARGE:
        _LARGE.clear()
        w = workloads.generate(name, seed=1, backend="torch", device="cuda")
        w_np = workloads.to_numpy(w)
        _LARGE[name] = (w, w_np, oracle.tree_attn(w_np))
    return _LARGE[name]


@pytest.mark.parametrize("splits", [0, 64])
@pytest.mark.parametrize("kernel", KERNELS_16)
@pytest.mark.parametrize("name", ["serve_b16_gqa_bf16", "llama70b_32k_b8_bf16", "verify_b64_fp16"])
def test_large_configs_full(name, kernel, splits):
    # every (sequence, node, head, column) output against the oracle, at the
    # workloads' full sizes, on the balanced schedule and with 64 key chunks
    w, w_np, want = _large(name)
    step = Step(w, kernel=kernel, num_splits=splits)
    step.attn()
    assert step.status()[0] == 0
    got = step.out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    err = np.max(np.abs(got - want))
    assert err <= TOL[w_np["dtype"]], f"max abs error {err}"
    # scatter of the tree keys: bit-exact on every sequence's scratch slots
    _, k_rot = oracle.rotate_inputs(w_np)
    kc = to_host(step.d["k_cache"])
    vc = to_host(step.d["v_cache"])
    P = w_np["page_size"]
    for b in range(w_np["B"]):
        L = int(w_np["seq_lens"][b])
        for i in range(w_np["T"]):
            s = L + i
            page = w_np["block_tables"][b, s // P]
            assert np.array_equal(kc[page, :, s % P].view(np.uint8), k_rot[b, i].view(np.uint8))
            assert np.array_equal(vc[page, :, s % P].view(np.uint8), w_np["v_new"][b, i].view(np.uint8))


@pytest.mark.skipif("tc" not in KERNELS_16, reason="tensor-core kernel not built")
def test_kernels_agree_with_each_other():
    # the SIMT and tensor-core kernels are independent implementations
    spec = workloads.custom("agree", B=4, Hq=32, Hkv=8, head_dim=128, dtype="bf16",
                            prefix=("list", [300, 1200, 64, 4000]), tree=("fanout", (10, 5, 3, 2), 64),
                            max_depth=4)
    w = workloads.generate(spec, seed=3)
    a = Step(w, kernel="simt")
    a.attn()
    b = Step(w, kernel="tc")
    b.attn()
    diff = (a.out.float() - b.out.float()).abs().max().item()
    assert diff <= 2 * TOL["bf16"]


def test_page_relabeling_is_invisible():
    spec = workloads.custom("relabel", B=2, Hq=8, Hkv=2, head_dim=128, dtype="f16",
                            prefix=("list", [333, 100]), tree=("fanout", (4, 3), 10), max_depth=2)
    w = workloads.generate(spec, seed=5)
    s1 = Step(w)
    s1.attn()
    perm = np.random.default_rng(1).permutation(w["num_pages"])
    w2 = dict(w)
    w2["k_cache"] = np.empty_like(w["k_cache"])
    w2["v_cache"] = np.empty_like(w["v_cache"])
    w2["k_cache"][perm] = w["k_cache"]
    w2["v_cache"][perm] = w["v_cache"]
    bt = w["block_tables"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    w2["block_tables"] = bt
    s2 = Step(w2)
    s2.attn()
    assert torch.equal(s1.out, s2.out)


def test_repeated_calls_are_deterministic():
    w = workloads.generate("llama7b_b1_fp16", seed=2)
    s = Step(w)
    s.attn()
    first = s.out.clone()
    for _ in range(3):
        s.attn()
        assert torch.equal(first, s.out)
