"""GPU parity of greedy acceptance and KV commit against the CPU oracle.

Integer outputs (argmax, accept_len, accept_path, next_token, block tables,
seq_lens, released pages) and the committed KV bytes must match bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import medusa_tree_speculative_attn_gb300 as mt
import oracle
import workloads
from gpu_helpers import Step, to_dev, to_host

pytestmark = pytest.mark.gpu


def _accept_dev(tokens, logits, dt, parents, md, ws=None):
    dev = "cuda"
    B, T = tokens.shape
    t_tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).to(dev)
    t_par = torch.from_numpy(np.ascontiguousarray(parents, np.int32)).to(dev)
    t_lg = to_dev(logits, dt, dev)
    am = torch.full((B, T), -7, dtype=torch.int32, device=dev)
    alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
    path = torch.full((B, md + 1), -7, dtype=torch.int32, device=dev)
    nxt = torch.full((B,), -7, dtype=torch.int32, device=dev)
    if ws is None:
        ws = mt.alloc_accept_workspace(B, T, dev)
    mt.tree_accept_greedy(t_tok, t_lg, t_par, alen, path, argmax_out=am, next_token=nxt, workspace=ws)
    st = mt.read_status(ws)
    return st, am.cpu().numpy(), alen.cpu().numpy(), path.cpu().numpy(), nxt.cpu().numpy(), ws


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [2, 3, 5, 37, 1000])
def test_accept_random_small_vocab(dt, V):
    rng = np.random.default_rng(V)
    B = 64
    for T in (1, 2, 7, 33, 64):
        parents = np.zeros((B, T), np.int32)
        for b in range(B):
            parents[b] = [-1] + [int(rng.integers(i)) for i in range(1, T)]
        depth = np.stack([workloads.depths_of(p) for p in parents])
        md = int(depth.max())
        tokens = rng.integers(0, V, (B, T)).astype(np.int32)
        logits = rng.integers(-2, 3, (B, T, V)).astype(np.float32)      # many ties
        logits[logits == 0] *= rng.choice([-1.0, 1.0], size=int((logits == 0).sum()))
        lg = oracle.round_to_act(logits, dt)
        st, am, alen, path, nxt, _ = _accept_dev(tokens, lg, dt, parents, md)
        assert st == 0
        o_am, o_len, o_path, o_next = oracle.accept_greedy(tokens, lg, dt, parents, md)
        assert np.array_equal(am, o_am)
        assert np.array_equal(alen, o_len)
        assert np.array_equal(path, o_path)
        assert np.array_equal(nxt, o_next)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [4096, 6000, 32000])
def test_accept_split_rows_with_ties_across_slices(dt, V):
    # Few rows and long vocabularies: each row is split over several CTAs
    # whose (value, lowest index) results meet in a per-row key.  Values from
    # {-2 .. 2} with signed zeros put equal maxima in many slices; the lowest
    # index must still win, and a second call on the same workspace (keys and
    # counters left at zero) must give the same answer.
    rng = np.random.default_rng(V)
    for B, T in ((1, 1), (1, 9), (3, 5)):
        parents = np.zeros((B, T), np.int32)
        for b in range(B):
            parents[b] = [-1] + [int(rng.integers(i)) for i in range(1, T)]
        md = int(np.stack([workloads.depths_of(p) for p in parents]).max())
        logits = rng.integers(-2, 3, (B, T, V)).astype(np.float32)
        logits[logits == 0] *= rng.choice([-1.0, 1.0], size=int((logits == 0).sum()))
        # some rows whose maximum sits only near the end of the row
        logits[:, 0, :] = np.minimum(logits[:, 0, :], 1.0)
        logits[:, 0, V - 3] = 2.0
        tokens = rng.integers(0, V, (B, T)).astype(np.int32)
        lg = oracle.round_to_act(logits, dt)
        o = oracle.accept_greedy(tokens, lg, dt, parents, md)
        ws = None
        for _ in range(2):
            st, am, alen, path, nxt, ws = _accept_dev(tokens, lg, dt, parents, md, ws)
            assert st == 0
            for got, want in zip((am, alen, path, nxt), o):
                assert np.array_equal(got, want)
        assert (o[0][:, 0] == V - 3).all()


@pytest.mark.parametrize("name", ["tiny_tree_fp32", "llama7b_b1_fp16", "serve_b16_gqa_bf16",
                                  "verify_b64_fp16"])
def test_accept_named_configs(name):
    w = workloads.generate(name, seed=2)
    st, am, alen, path, nxt, ws = _accept_dev(w["tree_tokens"], w["logits"], w["logits_dtype"],
                                              w["tree_parents"], w["max_depth"])
    assert st == 0
    o = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"], w["tree_parents"],
                             w["max_depth"])
    for got, want in zip((am, alen, path, nxt), o):
        assert np.array_equal(got, want)
    # the planted paths are found (or beaten by accidental matches)
    for b in range(w["B"]):
        assert alen[b] >= len(w["planted_nodes"][b])
    # counters are left at zero: a second call gives the same answer
    st2, am2, alen2, path2, nxt2, _ = _accept_dev(w["tree_tokens"], w["logits"], w["logits_dtype"],
                                                  w["tree_parents"], w["max_depth"])
    assert st2 == 0 and np.array_equal(alen2, alen) and np.array_equal(path2, path)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_accept_special_rows(dt):
    # all equal (ties everywhere), all -inf, max only in the last element, max
    # in a later 16-element chunk of a long fp32 row, signed zeros
    V = 40000
    rows = []
    rows.append(np.zeros(V, np.float32))
    rows.append(np.full(V, -np.inf, np.float32))
    r = np.full(V, -1.0, np.float32); r[-1] = 2.0; rows.append(r)
    r = np.full(V, -3.0, np.float32); r[33000] = 1.5; r[39999] = 1.5; rows.append(r)
    r = np.full(V, -0.0, np.float32); r[7] = 0.0; rows.append(r)
    r = np.random.default_rng(0).standard_normal(V).astype(np.float32); rows.append(r)
    T = len(rows)
    logits = oracle.round_to_act(np.stack(rows)[None], dt)
    parents = np.array([[-1] + list(range(T - 1))], np.int32)
    tokens = np.zeros((1, T), np.int32)
    st, am, alen, path, nxt, _ = _accept_dev(tokens, logits, dt, parents, T - 1)
    o = oracle.accept_greedy(tokens, logits, dt, parents, T - 1)
    assert st == 0
    assert np.array_equal(am, o[0]), (am, o[0])
    assert np.array_equal(alen, o[1]) and np.array_equal(path, o[2]) and np.array_equal(nxt, o[3])


def test_accept_rejects_bad_parents_without_fault():
    tokens = np.zeros((2, 4), np.int32)
    parents = np.array([[-1, 0, 1, 2], [-1, 2, 0, 1]], np.int32)   # second: parent after child
    lg = np.zeros((2, 4, 8), np.float32)
    st, am, alen, path, nxt, _ = _accept_dev(tokens, lg, "f32", parents, 3)
    assert st == mt.MedusaTreeError(-3, "").status


def _commit_check(w, step, kc0, vc0):
    o_am, o_len, o_path, o_next = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"],
                                                       w["tree_parents"], w["max_depth"])
    ko, vo, bto, slo, relo = oracle.kv_commit(w, o_path, o_len, kc0, vc0, w["block_tables"],
                                              w["seq_lens"], w["max_depth"])
    assert np.array_equal(step.alen.cpu().numpy(), o_len)
    assert np.array_equal(step.path.cpu().numpy(), o_path)
    assert np.array_equal(step.d["block_tables"].cpu().numpy(), bto)
    assert np.array_equal(step.d["seq_lens"].cpu().numpy(), slo)
    assert np.array_equal(step.rel.cpu().numpy(), relo)
    assert np.array_equal(to_host(step.d["k_cache"]).view(np.uint8), ko.view(np.uint8))
    assert np.array_equal(to_host(step.d["v_cache"]).view(np.uint8), vo.view(np.uint8))


@pytest.mark.parametrize("name", ["tiny_tree_fp32", "llama7b_b1_fp16", "serve_b16_gqa_bf16"])
def test_full_step_commit_bytes(name):
    w = workloads.generate(name, seed=3)
    step = Step(w)
    step.attn()
    step.accept()
    step.commit()
    assert step.status() == (0, 0)
    _, k_rot = oracle.rotate_inputs(w)
    kc0, vc0 = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
    _commit_check(w, step, kc0, vc0)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_commit_random_paths(dtype):
    # long planted paths over deep chains and bushy trees, prefixes straddling pages
    for seed, tree in enumerate([("chain", 20), ("fanout", (2, 2, 2, 2, 2), 40), ("star", 9)]):
        md = {"chain": 19, "fanout": 5, "star": 1}[tree[0]]
        spec = workloads.custom("commit", B=5, Hq=4, Hkv=2, head_dim=64, dtype=dtype,
                                prefix=("list", [0, 15, 16, 17, 300]), tree=tree, max_depth=md,
                                vocab=50, logits_dtype="f32", plant=("uniform", 0, md))
        w = workloads.generate(spec, seed=seed)
        step = Step(w)
        step.attn()
        step.accept()
        step.commit()
        assert step.status() == (0, 0)
        _, k_rot = oracle.rotate_inputs(w)
        kc0, vc0 = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
        _commit_check(w, step, kc0, vc0)


def test_bad_page_id_sets_status_without_fault():
    spec = workloads.custom("badpage", B=2, Hq=4, Hkv=2, head_dim=128, dtype="bf16",
                            prefix=("list", [100, 40]), tree=("fanout", (3, 2), 6), max_depth=2)
    w = workloads.generate(spec, seed=0)
    bt = w["block_tables"].copy()
    bt[0, 2] = w["num_pages"] + 5        # inside sequence 0's prefix
    w["block_tables"] = bt
    # the tensor-core kernel maps an out-of-range page to a row past the end of
    # its TMA tensor (zero fill) and records the error
    for kernel in ("simt", "tc"):
        step = Step(w, kernel=kernel)
        step.attn()
        assert step.status()[0] == mt.MedusaTreeError(-4, "").status


def test_bounded_wait_times_out_and_the_next_call_is_correct():
    # The tensor-core kernel's first pipeline wait is made one that nothing
    # completes, with a 200 us bound: the call must return, report
    # MT_ERR_TIMEOUT in its status word and leave the context usable; the next
    # call, with the default bound, must match the oracle.
    spec = workloads.custom("timeout", B=3, Hq=8, Hkv=2, head_dim=128, dtype="bf16",
                            prefix=("list", [300, 40, 1000]), tree=("fanout", (3, 2), 9), max_depth=2)
    w = workloads.generate(spec, seed=0)
    step = Step(w, kernel="tc")
    try:
        mt.debug_set_wait(200_000, stall=True)
        step.attn()
        assert step.status()[0] == -6
    finally:
        mt.debug_set_wait(0, stall=False)
    step.attn()
    assert step.status()[0] == 0
    want = oracle.tree_attn(w)
    got = step.out.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - want)) <= 1e-2


def test_bad_tree_sets_status_without_fault():
    spec = workloads.custom("badtree", B=2, Hq=4, Hkv=2, head_dim=128, dtype="f16",
                            prefix=("list", [10, 40]), tree=("fanout", (3, 2), 6), max_depth=2)
    w = workloads.generate(spec, seed=0)
    par = w["tree_parents"].copy()
    par[1, 3] = 5
    w["tree_parents"] = par
    step = Step(w)
    step.attn()
    assert step.status()[0] == -3


# ---- acceptance and commit in one launch (mt_tree_accept_commit) ----

def _fused_check(w, step, kc0, vc0):
    o_am = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"], w["tree_parents"],
                                w["max_depth"])[0]
    assert np.array_equal(step.am.cpu().numpy(), o_am)
    _commit_check(w, step, kc0, vc0)


@pytest.mark.parametrize("name", ["tiny_tree_fp32", "llama7b_b1_fp16", "serve_b16_gqa_bf16",
                                  "verify_b64_fp16"])
def test_fused_step_matches_oracle(name):
    w = workloads.generate(name, seed=4)
    step = Step(w)
    step.attn()
    step.accept_commit()
    assert step.status() == (0, 0)
    _, k_rot = oracle.rotate_inputs(w)
    kc0, vc0 = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
    _fused_check(w, step, kc0, vc0)
    o_next = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"], w["tree_parents"],
                                  w["max_depth"])[3]
    assert np.array_equal(step.nxt.cpu().numpy(), o_next)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_fused_random_paths(dtype):
    # long planted paths (many register passes of the commit), prefixes straddling pages
    for seed, tree in enumerate([("chain", 20), ("fanout", (2, 2, 2, 2, 2), 40), ("star", 9),
                                 ("chain", 64)]):
        md = tree[1] - 1 if tree[0] == "chain" else {"fanout": 5, "star": 1}[tree[0]]
        spec = workloads.custom("fused", B=5, Hq=8, Hkv=4, head_dim=128, dtype=dtype,
                                prefix=("list", [0, 15, 16, 17, 300]), tree=tree, max_depth=md,
                                vocab=50, logits_dtype="f32", plant=("uniform", 0, md))
        w = workloads.generate(spec, seed=seed)
        step = Step(w)
        step.attn()
        step.accept_commit()
        assert step.status() == (0, 0)
        _, k_rot = oracle.rotate_inputs(w)
        kc0, vc0 = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
        _fused_check(w, step, kc0, vc0)


def test_fused_equals_the_two_calls_and_leaves_counters_at_zero():
    w = workloads.generate("serve_b16_gqa_bf16", seed=6)
    a, b = Step(w), Step(w)
    a.attn()
    b.attn()
    a.accept()
    a.commit()
    b.accept_commit()
    assert a.status() == (0, 0) and b.status() == (0, 0)
    for x, y in ((a.am, b.am), (a.alen, b.alen), (a.path, b.path), (a.nxt, b.nxt), (a.rel, b.rel)):
        assert torch.equal(x, y)
    for key in ("block_tables", "seq_lens", "k_cache", "v_cache"):  # bytes: the pool may hold NaNs
        assert torch.equal(a.d[key].view(torch.uint8), b.d[key].view(torch.uint8))
    # the arrival counters are back at zero: acceptance alone on the same
    # workspace gives the same path
    path0 = b.path.clone()
    b.accept()
    assert mt.read_status(b.aws) == 0 and torch.equal(b.path, path0)


def test_fused_bad_page_sets_status_without_fault():
    spec = workloads.custom("fusedpage", B=3, Hq=4, Hkv=2, head_dim=128, dtype="bf16",
                            prefix=("list", [100, 40, 7]), tree=("fanout", (3, 2), 6), max_depth=2,
                            vocab=64, logits_dtype="bf16", plant=("uniform", 0, 2))
    w = workloads.generate(spec, seed=1)
    step = Step(w)
    step.attn()
    bt = step.d["block_tables"]
    L1 = int(w["seq_lens"][1])
    bt[1, (L1 + 5) // w["page_size"]] = w["num_pages"] + 5   # a scratch slot of sequence 1
    step.accept_commit()
    assert mt.read_status(step.aws) == mt.MedusaTreeError(-4, "").status
    # sequence 1 is untouched; the others are committed as the oracle says
    sl = step.d["seq_lens"].cpu().numpy()
    assert sl[1] == L1
    o_len = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"], w["tree_parents"],
                                 w["max_depth"])[1]
    for b in (0, 2):
        assert sl[b] == int(w["seq_lens"][b]) + int(o_len[b]) + 1


def test_fused_bad_tree_commits_the_root_only():
    spec = workloads.custom("fusedtree", B=2, Hq=4, Hkv=2, head_dim=64, dtype="f16",
                            prefix=("list", [10, 40]), tree=("fanout", (3, 2), 6), max_depth=2,
                            vocab=64, logits_dtype="f16", plant=("uniform", 0, 2))
    w = workloads.generate(spec, seed=0)
    step = Step(w)
    step.attn()
    step.d["tree_parents"][1, 3] = 5   # parent after child: acceptance rejects the tree
    step.accept_commit()
    assert mt.read_status(step.aws) == -3
    assert step.alen.cpu().numpy()[1] == 0
    assert step.d["seq_lens"].cpu().numpy()[1] == int(w["seq_lens"][1]) + 1
