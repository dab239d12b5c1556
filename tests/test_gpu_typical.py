"""GPU parity of typical acceptance against the CPU oracle.

The device decides each node's test in fp32 with its own summation order, the
oracle in float64.  Where q[token] and the threshold differ by more than a
relative 1e-3 (two orders of magnitude above the fp32 error of a 32000-term
sum) the decisions must agree; closer nodes may go either way.  The path,
accept_len and next_token are integer functions of the device's own node
decisions and must match them exactly, and the oracle's whenever no node on
the way is that close.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import medusa_tree_speculative_attn_gb300 as mt
import oracle
import workloads
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

MARGIN = 1e-3


def _typical_dev(tokens, logits, dt, parents, md, tau, eps, delta):
    dev = "cuda"
    B, T = tokens.shape
    t_tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).to(dev)
    t_par = torch.from_numpy(np.ascontiguousarray(parents, np.int32)).to(dev)
    t_lg = to_dev(logits, dt, dev)
    ok = torch.full((B, T), -7, dtype=torch.int32, device=dev)
    alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
    path = torch.full((B, md + 1), -7, dtype=torch.int32, device=dev)
    nxt = torch.full((B,), -7, dtype=torch.int32, device=dev)
    ws = mt.alloc_accept_workspace(B, T, dev)
    mt.tree_accept_typical(t_tok, t_lg, t_par, alen, path, node_accept=ok, next_token=nxt, workspace=ws,
                           temperature=tau, epsilon=eps, delta=delta)
    return (mt.read_status(ws), ok.cpu().numpy(), alen.cpu().numpy(), path.cpu().numpy(),
            nxt.cpu().numpy(), ws)


def _path_from_flags(flags, parents, md):
    """Deepest node whose whole root path passes (lowest index among equals)."""
    B, T = flags.shape
    alen = np.zeros(B, np.int32)
    path = np.full((B, md + 1), -1, np.int32)
    ends = np.zeros(B, np.int64)
    for b in range(B):
        depth = workloads.depths_of(parents[b])
        end = 0
        for i in range(T):
            n, good = i, True
            while n >= 0:
                good = good and bool(flags[b, n])
                n = int(parents[b, n])
            if good and depth[i] > depth[end]:
                end = i
        ends[b] = end
        alen[b] = depth[end]
        n = end
        while n >= 0:
            path[b, depth[n]] = n
            n = int(parents[b, n])
    return alen, path, ends


def _check(tokens, lg, dt, parents, md, tau, eps, delta):
    st, ok, alen, path, nxt, _ = _typical_dev(tokens, lg, dt, parents, md, tau, eps, delta)
    assert st == 0
    r = oracle.accept_typical(tokens, lg, dt, parents, md, tau, eps, delta)
    assert r["status"] == 0
    clear = np.abs(r["prob"] - r["thr"]) > MARGIN * r["thr"]
    clear[:, 0] = True
    assert np.array_equal(ok[clear], r["node_accept"][clear])
    assert np.all((ok == 0) | (ok == 1)) and np.all(ok[:, 0] == 1)
    want_len, want_path, ends = _path_from_flags(ok, parents, md)
    assert np.array_equal(alen, want_len)
    assert np.array_equal(path, want_path)
    x64 = oracle.act_to_f64(lg, dt)
    assert np.array_equal(nxt, [int(np.argmax(x64[b, e])) for b, e in enumerate(ends)])
    if clear.all():
        assert np.array_equal(alen, r["accept_len"]) and np.array_equal(path, r["accept_path"])
        assert np.array_equal(nxt, r["next_token"])
    return ok, alen


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("V", [2, 3, 37, 1000, 4096])
def test_typical_random_trees(dt, V):
    rng = np.random.default_rng(V + len(dt))
    B = 48
    seen = []
    for T, tau in ((1, 1.0), (2, 0.7), (7, 1.0), (33, 1.3), (64, 0.7)):
        parents = np.zeros((B, T), np.int32)
        for b in range(B):
            parents[b] = [-1] + [int(rng.integers(i)) for i in range(1, T)]
        md = int(max(workloads.depths_of(p).max() for p in parents))
        tokens = rng.integers(-1, V + 1, (B, T)).astype(np.int32)
        lg = oracle.round_to_act(rng.normal(0, 2, (B, T, V)).astype(np.float32), dt)
        ok, _ = _check(tokens, lg, dt, parents, md, tau, 0.09, 0.3)
        seen.append(ok[:, 1:].ravel())
    seen = np.concatenate(seen)
    assert seen.any() and not seen.all()   # both outcomes occur


@pytest.mark.parametrize("name", ["llama7b_b1_fp16", "serve_b16_gqa_bf16", "verify_b64_fp16"])
def test_typical_named_configs(name):
    w = workloads.generate(name, seed=5)
    for tau, eps, delta in ((1.0, 0.09, 0.3), (0.5, 0.3, 0.55)):
        ok, alen = _check(w["tree_tokens"], w["logits"], w["logits_dtype"], w["tree_parents"], w["max_depth"],
                          tau, eps, delta)
    assert alen.max() >= 1


def test_typical_on_peaked_rows_equals_greedy_on_device():
    rng = np.random.default_rng(11)
    B, T, V = 16, 40, 3000
    parents = np.stack([[-1] + [int(rng.integers(i)) for i in range(1, T)] for _ in range(B)]).astype(np.int32)
    md = int(max(workloads.depths_of(p).max() for p in parents))
    lg = rng.normal(0, 1, (B, T, V)).astype(np.float32)
    top = rng.integers(0, V, (B, T))
    np.put_along_axis(lg, top[..., None], 60.0, axis=2)
    tokens = np.where(rng.random((B, T)) < 0.8, np.take_along_axis(top, parents.clip(0), 1),
                      rng.integers(0, V, (B, T))).astype(np.int32)
    st, ok, alen, path, nxt, _ = _typical_dev(tokens, lg, "f32", parents, md, 1.0, 0.09, 0.3)
    assert st == 0
    t_tok = torch.from_numpy(tokens).cuda()
    am = torch.empty((B, T), dtype=torch.int32, device="cuda")
    galen = torch.empty(B, dtype=torch.int32, device="cuda")
    gpath = torch.empty((B, md + 1), dtype=torch.int32, device="cuda")
    gnxt = torch.empty(B, dtype=torch.int32, device="cuda")
    mt.tree_accept_greedy(t_tok, torch.from_numpy(lg).cuda(), torch.from_numpy(parents).cuda(), galen, gpath,
                          argmax_out=am, next_token=gnxt, workspace=mt.alloc_accept_workspace(B, T))
    assert np.array_equal(alen, galen.cpu().numpy())
    assert np.array_equal(path, gpath.cpu().numpy())
    assert np.array_equal(nxt, gnxt.cpu().numpy())
    assert alen.max() >= 2


def test_typical_repeated_calls_reuse_the_workspace():
    rng = np.random.default_rng(2)
    B, T, V = 8, 20, 500
    parents = np.stack([[-1] + [int(rng.integers(i)) for i in range(1, T)] for _ in range(B)]).astype(np.int32)
    md = int(max(workloads.depths_of(p).max() for p in parents))
    tokens = rng.integers(0, V, (B, T)).astype(np.int32)
    lg = rng.normal(0, 2, (B, T, V)).astype(np.float32)
    dev = "cuda"
    args = [torch.from_numpy(x).to(dev) for x in (tokens, lg, parents)]
    ws = mt.alloc_accept_workspace(B, T, dev)
    outs = []
    for _ in range(3):
        ok = torch.empty((B, T), dtype=torch.int32, device=dev)
        alen = torch.empty(B, dtype=torch.int32, device=dev)
        path = torch.empty((B, md + 1), dtype=torch.int32, device=dev)
        nxt = torch.empty(B, dtype=torch.int32, device=dev)
        mt.tree_accept_typical(*args, alen, path, node_accept=ok, next_token=nxt, workspace=ws,
                               temperature=0.8, epsilon=0.09, delta=0.3)
        outs.append([t.cpu().numpy() for t in (ok, alen, path, nxt)])
    assert mt.read_status(ws) == 0
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert np.array_equal(a, b)


def test_typical_bad_tree_sets_status_without_fault():
    tokens = np.zeros((2, 4), np.int32)
    parents = np.array([[-1, 0, 1, 2], [-1, 2, 0, 1]], np.int32)   # second: parent after child
    lg = np.zeros((2, 4, 8), np.float32)
    st, ok, alen, path, nxt, _ = _typical_dev(tokens, lg, "f32", parents, 3, 1.0, 0.09, 0.3)
    assert st == -3
    assert alen[1] == 0 and path[1, 0] == 0


def test_typical_rejects_bad_temperature():
    B, T, V = 1, 2, 8
    dev = "cuda"
    z = lambda *s: torch.zeros(s, dtype=torch.int32, device=dev)
    with pytest.raises(mt.MedusaTreeError) as e:
        mt.tree_accept_typical(z(B, T), torch.zeros((B, T, V), device=dev), z(B, T), z(B), z(B, 2),
                               node_accept=z(B, T), next_token=z(B), workspace=mt.alloc_accept_workspace(B, T),
                               temperature=0.0, epsilon=0.09, delta=0.3)
    assert e.value.status == -1
