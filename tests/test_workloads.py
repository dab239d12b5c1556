"""The seeded input generator keeps the recipe it states: tree shapes, distinct
sibling tokens, page pools with poison pages, NaN in every slot that is not a
committed prefix token, planted paths, the named workloads' sizes, and
determinism.  (The generator holds no method arithmetic; these are checks of
the inputs both the oracle and the CUDA path are fed.)"""
import numpy as np
import pytest

import workloads as wl


def test_named_workloads_have_the_stated_sizes():
    want = {  # B, Hq, Hkv, D, dtype, T, vocab, logits dtype
        "tiny_tree_fp32": (1, 1, 1, 64, "f32", 7, 1000, "f32"),
        "llama7b_b1_fp16": (1, 32, 32, 128, "f16", 64, 32000, "f32"),
        "serve_b16_gqa_bf16": (16, 32, 8, 128, "bf16", 64, 32000, "bf16"),
        "llama70b_32k_b8_bf16": (8, 64, 8, 128, "bf16", 26, None, None),
        "verify_b64_fp16": (64, 32, 32, 128, "f16", 32, 32000, "f16"),
    }
    for name, (B, Hq, Hkv, D, dt, T, V, ldt) in want.items():
        s = wl.SPECS[name]
        assert (s.B, s.Hq, s.Hkv, s.head_dim, s.dtype, s.vocab, s.logits_dtype) == (B, Hq, Hkv, D, dt, V, ldt)
        par, dep = wl._trees(np.random.default_rng(0), s)
        assert par.shape == (B, T) and dep.max() <= s.max_depth
    assert wl.SPECS["tiny_tree_fp32"].tree[1] == (-1, 0, 0, 1, 2, 3, 3)


@pytest.mark.parametrize("name,lo,hi", [("serve_b16_gqa_bf16", 512, 8192), ("verify_b64_fp16", 256, 4096),
                                        ("llama70b_32k_b8_bf16", 32768, 32768)])
def test_prefix_lengths_stay_in_range(name, lo, hi):
    for seed in range(20):
        L = wl._prefix_lengths(np.random.default_rng(seed), wl.SPECS[name])
        assert L.min() >= lo and L.max() <= hi


@pytest.mark.parametrize("caps,n", [((10, 5, 3, 2), 64), ((10, 5, 3, 2, 2), 64), ((3, 2, 2, 1), 26),
                                    ((10, 5, 3, 2), 32), ((2, 2), 7)])
def test_fanout_trees_are_topological_depth_major_and_within_the_fanouts(caps, n):
    for seed in range(10):
        par, dep, paths = wl.fanout_tree(np.random.default_rng(seed), caps, n)
        assert len(par) == n and par[0] == -1 and dep[0] == 0
        assert all(0 <= par[i] < i for i in range(1, n))
        assert np.array_equal(dep, wl.depths_of(par))
        assert np.all(np.diff(dep) >= 0)                       # depth-major numbering
        kids = np.bincount(par[1:], minlength=n)
        assert all(kids[i] <= caps[dep[i]] if dep[i] < len(caps) else kids[i] == 0 for i in range(n))
        assert len(set(paths)) == n                            # each top-k rank path once


def test_a_tree_larger_than_its_fanouts_allow_is_refused():
    with pytest.raises(ValueError):
        wl.fanout_tree(np.random.default_rng(0), (2, 2), 8)


def test_sibling_tokens_are_distinct():
    rng = np.random.default_rng(3)
    for _ in range(20):
        par, _, _ = wl.fanout_tree(rng, (10, 5, 3, 2), 64)
        tok = wl.tree_tokens(rng, par, 50)
        for p in np.unique(par[1:]):
            sib = tok[np.nonzero(par == p)[0]]
            assert len(np.unique(sib)) == len(sib)


def _small(seed=0, dtype="bf16"):
    spec = wl.custom("rec", B=5, Hq=4, Hkv=2, head_dim=64, dtype=dtype, prefix=("list", [0, 1, 15, 16, 40]),
                     tree=("fanout", (3, 2, 2), 12), max_depth=3, vocab=30, logits_dtype=dtype,
                     plant=("uniform", 0, 3))
    return wl.generate(spec, seed=seed)


def test_page_pool_gives_each_sequence_its_own_pages_plus_poison_pages():
    w = _small()
    bt, P, T = w["block_tables"], w["page_size"], w["T"]
    used = []
    for b in range(w["B"]):
        n = -(-(int(w["seq_lens"][b]) + T) // P)
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, n:] == -1)
        used += list(bt[b, :n])
    assert len(set(used)) == len(used)                          # no page shared
    assert w["num_pages"] - len(used) == w["spec"].poison_pages  # unreferenced poison pages
    assert max(used) < w["num_pages"]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_only_committed_prefix_slots_hold_numbers(dtype):
    w = _small(dtype=dtype)
    P = w["page_size"]
    vals = w["k_cache"]
    if dtype == "bf16":
        vals = (vals.astype(np.uint32) << 16).view(np.float32)
    finite = np.isfinite(vals).all(axis=(1, 3))                 # [pages, P]
    want = np.zeros_like(finite)
    for b in range(w["B"]):
        for s in range(int(w["seq_lens"][b])):
            want[w["block_tables"][b, s // P], s % P] = True
    assert np.array_equal(finite, want)
    assert np.isnan(vals.transpose(0, 2, 1, 3)[~want]).all()


def test_planted_paths_are_root_paths_with_the_planted_logit():
    for seed in range(5):
        w = _small(seed=seed, dtype="f32")
        for b, path in enumerate(w["planted_nodes"]):
            dep = w["tree_depths"][b]
            assert len(path) == min(int(w["planted_len"][b]), int(dep.max()))
            prev = 0
            for node in path:
                assert w["tree_parents"][b, node] == prev
                assert w["logits"][b, prev, w["tree_tokens"][b, node]] == wl.PLANT_LOGIT
                prev = node


def test_geometric_plant_lengths():
    spec = wl.custom("geo", B=20000, max_depth=5, plant=("geometric", 0.4))
    L = wl._planted_lengths(np.random.default_rng(1), spec)
    assert L.min() == 0 and L.max() == 5
    assert abs((L == 0).mean() - 0.4) < 0.02                   # P(G = 1) = p
    assert abs((L == 5).mean() - 0.6 ** 5) < 0.02              # G >= 6 is cut to the maximum depth


def test_bf16_values_are_truncated_float32_draws():
    a = wl._np_normal(np.random.default_rng(7), (1000,), "bf16")
    x = np.random.default_rng(7).standard_normal(size=(1000,), dtype=np.float32)
    assert np.array_equal(a, (x.view(np.uint32) >> 16).astype(np.uint16))


def test_seeds_are_deterministic_and_distinct():
    a, b, c = _small(seed=4), _small(seed=4), _small(seed=5)
    for k in ("q", "k_cache", "logits", "tree_parents", "block_tables", "tree_tokens"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["q"], c["q"])
