"""GPU parity of the candidate-tree call (through the C ABI) against the oracle.

Tokens are integers: bit-exact.  Inputs are seeded; the serving shapes use the
workloads' 64-node fanout trees (choice ranks up to 9) over 5 heads and a
32000-entry vocab.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import medusa_tree_speculative_attn_gb300 as mt
import oracle
import workloads
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def _trees(B, fanout, T, max_depth, seed):
    spec = workloads.custom("cand", B=B, Hq=1, Hkv=1, head_dim=64, dtype="f32",
                            prefix=("list", [1] * B), tree=("fanout", fanout, T), max_depth=max_depth)
    return workloads.generate(spec, seed=seed, with_logits=False)["tree_parents"]


def _run(root, heads, par, dtype):
    dev = "cuda"
    r = to_dev(root, dtype, dev)
    h = to_dev(heads, dtype, dev)
    p = torch.from_numpy(np.ascontiguousarray(par, np.int32)).to(dev)
    tok = torch.full(par.shape, -7, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    mt.tree_candidates(r, h, p, tok, status_ws=ws)
    st = mt.read_status(ws)
    return tok.cpu().numpy(), st


def _logits(rng, shape, dtype, ties=False):
    if ties:
        x = rng.integers(-3, 4, size=shape).astype(np.float32) * 0.25
    else:
        x = rng.standard_normal(shape, dtype=np.float32)
    return oracle.round_to_act(x, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_serving_shapes(dtype):
    rng = np.random.default_rng(11)
    B, T, H, V = 16, 64, 5, 32000
    par = _trees(B, (10, 5, 3, 2, 2), T, H, seed=3)
    root = _logits(rng, (B, V), dtype)
    heads = _logits(rng, (B, H, V), dtype)
    got, st = _run(root, heads, par, dtype)
    want, wst = oracle.tree_candidates(root, heads, dtype, par)
    assert st == 0 and wst == 0
    assert np.array_equal(got, want)


@pytest.mark.parametrize("V", [7, 16, 1001, 4096])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_ties_and_ragged_vocab(dtype, V):
    # heavy ties (7 distinct values), vocab sizes below the 16 choices, not a
    # multiple of a 16-byte vector (unaligned rows), and a power of two
    rng = np.random.default_rng(V)
    B, H = 5, 3
    fan = (3, 2, 2) if V < 16 else (10, 4, 2)
    par = _trees(B, fan, 26 if V >= 16 else 12, H, seed=V)
    root = _logits(rng, (B, V), dtype, ties=True)
    heads = _logits(rng, (B, H, V), dtype, ties=True)
    got, st = _run(root, heads, par, dtype)
    want, wst = oracle.tree_candidates(root, heads, dtype, par)
    assert st == 0 and wst == 0
    assert np.array_equal(got, want)


def test_single_node_tree():
    rng = np.random.default_rng(5)
    root = _logits(rng, (3, 300), "bf16")
    heads = _logits(rng, (3, 2, 300), "bf16")
    par = np.full((3, 1), -1, np.int32)
    got, st = _run(root, heads, par, "bf16")
    want, _ = oracle.tree_candidates(root, heads, "bf16", par)
    assert st == 0 and np.array_equal(got, want)


def test_errors_reported():
    rng = np.random.default_rng(9)
    V, H = 64, 2
    root = _logits(rng, (1, V), "f32")
    heads = _logits(rng, (1, H, V), "f32")
    # 20 children of the root: ranks up to 19, more than the 16 choices supported
    par = np.array([[-1] + [0] * 20], np.int32)
    got, st = _run(root, heads, par, "f32")
    assert st == -3
    assert got[0, 0] == oracle.tree_candidates(root, heads, "f32", par)[0][0, 0]
    # malformed (parent not earlier) and too deep for the heads
    _, st = _run(root, heads, np.array([[-1, 2, 0]], np.int32), "f32")
    assert st == -3
    _, st = _run(root, heads, np.array([[-1, 0, 1, 2]], np.int32), "f32")
    assert st == -3


def test_choice_rank_past_the_vocab():
    # 10 children of the root over a 7-entry vocab: ranks 7..9 have no entry (-1)
    rng = np.random.default_rng(2)
    V, H = 7, 1
    par = np.array([[-1] + [0] * 10], np.int32)
    root = _logits(rng, (1, V), "f16")
    heads = _logits(rng, (1, H, V), "f16")
    got, st = _run(root, heads, par, "f16")
    want, wst = oracle.tree_candidates(root, heads, "f16", par)
    assert st == 0 and wst == 0
    assert want[0, 8:].tolist() == [-1, -1, -1]
    assert np.array_equal(got, want)
