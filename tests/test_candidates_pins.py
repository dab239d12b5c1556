"""Pins of the oracle's candidate-tree rule, independent of its C code.

Reading (lmdeploy PR 1231 "[WIP] support Medusa": porting generate_candidates,
Medusa heads at top-k over a 64-choice tree): node 0 takes the argmax of the
base logits; a node at depth d with r earlier siblings takes the rank-r entry of
head d-1, ranked by larger value first and lower index first among equal values.
Each pin would fail for a plausible mistake: counting all siblings instead of the
earlier ones, reversing the tie order, taking head d instead of head d-1, or
comparing in a wider or narrower precision than the logits' own values.
"""
import numpy as np

import oracle
import workloads

PAR7 = np.array([-1, 0, 0, 1, 2, 3, 3], np.int32)  # branch 0->1->3->{5,6}, branch 0->2->4


def _rank_order(x):
    """Indices of x by the stated order, via Python's own sort."""
    return sorted(range(len(x)), key=lambda v: (-float(x[v]), v))


def _depths(par):
    d = [0] * len(par)
    for i in range(1, len(par)):
        d[i] = d[par[i]] + 1
    return d


def _brute(root, heads, par):
    """The rule written with Python sorts (no selection passes)."""
    B, T = par.shape
    out = np.empty((B, T), np.int64)
    for b in range(B):
        d = _depths(par[b])
        out[b, 0] = _rank_order(root[b])[0]
        for i in range(1, T):
            r = sum(1 for j in range(1, i) if par[b, j] == par[b, i])
            out[b, i] = _rank_order(heads[b, d[i] - 1])[r]
    return out


def test_closed_form_ranks():
    # head logits strictly decreasing in the index: rank r is index r, so each
    # node's token is its number of earlier siblings; the root's planted max wins
    V, H = 40, 3
    root = np.zeros((1, V), np.float32)
    root[0, 23] = 4.0
    heads = np.tile(-np.arange(V, dtype=np.float32), (1, H, 1))
    tok, st = oracle.tree_candidates(root, heads, "f32", PAR7[None])
    assert st == 0
    assert tok[0].tolist() == [23, 0, 1, 0, 0, 0, 1]


def test_each_depth_reads_its_own_head():
    # head h ranks index (h + 1) * 5 first: a node at depth d with rank 0 takes
    # token 5 * d, so an off-by-one head index shows
    V, H = 32, 3
    heads = np.zeros((1, H, V), np.float32)
    for h in range(H):
        heads[0, h, (h + 1) * 5] = 1.0
    root = np.zeros((1, V), np.float32)
    tok, st = oracle.tree_candidates(root, heads, "f32", PAR7[None])
    assert st == 0
    d = _depths(PAR7)
    for i in (1, 3, 4, 5):  # the rank-0 nodes
        assert tok[0, i] == 5 * d[i]


def test_ties_lowest_index_first():
    V, H = 12, 3
    heads = np.ones((1, H, V), np.float32)  # all equal: rank r is index r
    root = np.ones((1, V), np.float32)
    tok, st = oracle.tree_candidates(root, heads, "f32", PAR7[None])
    assert st == 0
    assert tok[0].tolist() == [0, 0, 1, 0, 0, 0, 1]
    # +0 and -0 are equal: the lower index wins whichever sign it carries
    root = np.full((1, V), -1.0, np.float32)
    root[0, 7] = 0.0
    root[0, 3] = -0.0
    tok, _ = oracle.tree_candidates(root, heads, "f32", PAR7[None])
    assert tok[0, 0] == 3


def test_bruteforce_with_many_ties():
    rng = np.random.default_rng(7)
    for dtype in ("f32", "f16", "bf16"):
        for trial in range(6):
            B, V, H = 3, int(rng.integers(5, 40)), 4
            spec = workloads.custom("t", B=B, Hq=1, Hkv=1, head_dim=64, dtype="f32",
                                    prefix=("list", [1] * B), tree=("fanout", (4, 3, 2, 2), 30),
                                    max_depth=4)
            par = workloads.generate(spec, seed=trial, with_logits=False)["tree_parents"]
            vals = rng.integers(-2, 3, size=(B, H + 1, V)).astype(np.float32) * 0.5
            root, heads = vals[:, 0], vals[:, 1:]
            root_a = oracle.round_to_act(root, dtype)
            heads_a = oracle.round_to_act(heads, dtype)
            tok, st = oracle.tree_candidates(root_a, heads_a, dtype, par)
            assert st == 0
            want = _brute(oracle.act_to_f64(root_a, dtype), oracle.act_to_f64(heads_a, dtype), par)
            assert np.array_equal(tok, want)


def test_values_compared_at_logit_precision():
    # two bf16 values one ulp apart (1.0 and the next bf16 above it) rank by value,
    # two fp32 values that round to the same bf16 tie and rank by index
    V = 8
    heads = np.zeros((1, 1, V), np.float32)
    heads[0, 0, 5] = 1.0
    heads[0, 0, 2] = np.float32(1.0 + 2.0 ** -7)  # the bf16 right above 1.0
    root = np.zeros((1, V), np.float32)
    par = np.array([[-1, 0, 0]], np.int32)
    hb = oracle.round_to_act(heads, "bf16")
    tok, _ = oracle.tree_candidates(oracle.round_to_act(root, "bf16"), hb, "bf16", par)
    assert tok[0].tolist() == [0, 2, 5]
    heads[0, 0, 2] = np.float32(1.0 + 2.0 ** -12)  # rounds to 1.0 in bf16: a tie
    hb = oracle.round_to_act(heads, "bf16")
    tok, _ = oracle.tree_candidates(oracle.round_to_act(root, "bf16"), hb, "bf16", par)
    assert tok[0].tolist() == [0, 2, 5]
    tok32, _ = oracle.tree_candidates(root, heads, "f32", par)
    assert tok32[0].tolist() == [0, 2, 5]
    heads[0, 0, 5] = np.float32(1.0 + 2.0 ** -11)  # now index 5 is larger in fp32 only
    tok32, _ = oracle.tree_candidates(root, heads, "f32", par)
    assert tok32[0].tolist() == [0, 5, 2]
    hb = oracle.round_to_act(heads, "bf16")
    tok, _ = oracle.tree_candidates(oracle.round_to_act(root, "bf16"), hb, "bf16", par)
    assert tok[0].tolist() == [0, 2, 5]


def test_bad_trees_report():
    V = 10
    root = np.zeros((1, V), np.float32)
    heads = np.zeros((1, 2, V), np.float32)
    _, st = oracle.tree_candidates(root, heads, "f32", np.array([[-1, 0, 2]], np.int32))
    assert st == -3  # parent not earlier
    _, st = oracle.tree_candidates(root, heads, "f32", np.array([[-1, 0, 1, 2]], np.int32))
    assert st == -3  # depth 3 with only 2 heads
