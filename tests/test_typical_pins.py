"""Pins of the oracle's typical acceptance, independent of its C code: closed
forms (uniform rows, two-token rows), SciPy's own softmax and entropy with an
exhaustive path search, the reduction to greedy acceptance on peaked rows, the
temperature as a logit scale, and monotonicity in the thresholds.

Reading pinned (the pages name the scheme without defining it): node i > 0
passes when q[token_i] > min(epsilon, delta * exp(-H)), q the softmax of its
parent's logits / temperature and H that distribution's entropy in nats."""
import math

import numpy as np
import pytest

import oracle
import workloads

scipy_special = pytest.importorskip("scipy.special")
scipy_stats = pytest.importorskip("scipy.stats")


def _chain(T):
    return np.array([[-1] + list(range(T - 1))], np.int32)


def _random_parents(rng, B, T):
    return np.stack([[-1] + [int(rng.integers(i)) for i in range(1, T)] for _ in range(B)]).astype(np.int32)


def test_uniform_row_closed_form():
    # equal logits: q = 1/V, H = ln V, so thr = min(epsilon, delta / V)
    V, T = 5, 3
    lg = np.full((1, T, V), 0.75, np.float32)
    tok = np.array([[0, 1, 4]], np.int32)
    for eps, delta, passes in ((0.3, 0.5, True), (0.3, 2.0, False), (0.15, 2.0, True), (0.2, 2.0, False)):
        r = oracle.accept_typical(tok, lg, "f32", _chain(T), T - 1, 1.0, eps, delta)
        assert r["status"] == 0
        assert np.allclose(r["prob"][0, 1:], 1 / V, rtol=1e-14)
        assert np.allclose(r["thr"][0, 1:], min(eps, delta / V), rtol=1e-14)
        assert list(r["node_accept"][0]) == [1] + [int(passes)] * (T - 1)
        assert r["accept_len"][0] == (T - 1 if passes else 0)


@pytest.mark.parametrize("tau", [0.5, 1.0, 3.0])
def test_two_token_row_closed_form(tau):
    a = 1.75
    lg = np.array([[[a, 0.0], [0.0, 0.0]]], np.float32)
    tok = np.array([[0, 1]], np.int32)   # the child asks for token 1 under row [a, 0]
    eps, delta = 0.9, 0.6
    r = oracle.accept_typical(tok, lg, "f32", _chain(2), 1, tau, eps, delta)
    q1 = 1.0 / (1.0 + math.exp(a / tau))
    q0 = 1.0 - q1
    h = -(q0 * math.log(q0) + q1 * math.log(q1))
    thr = min(eps, delta * math.exp(-h))
    assert r["prob"][0, 1] == pytest.approx(q1, rel=1e-13)
    assert r["thr"][0, 1] == pytest.approx(thr, rel=1e-13)
    assert r["node_accept"][0, 1] == int(q1 > thr)


def _brute(tokens, x64, parents, max_depth, tau, eps, delta):
    """SciPy softmax/entropy per parent row, then every node's root path checked."""
    B, T = tokens.shape
    V = x64.shape[-1]
    prob = np.zeros((B, T))
    thr = np.zeros((B, T))
    own = np.zeros((B, T), bool)
    alen = np.zeros(B, np.int32)
    path = np.full((B, max_depth + 1), -1, np.int32)
    nxt = np.zeros(B, np.int32)
    for b in range(B):
        own[b, 0] = True
        prob[b, 0] = 1.0
        for i in range(1, T):
            q = scipy_special.softmax(x64[b, parents[b, i]] / tau)
            h = scipy_stats.entropy(q)
            t = int(tokens[b, i])
            prob[b, i] = q[t] if 0 <= t < V else 0.0
            thr[b, i] = min(eps, delta * math.exp(-h))
            own[b, i] = prob[b, i] > thr[b, i]
        best, best_d = 0, 0
        for i in range(T):
            chain, n = [], i
            while n >= 0:
                chain.append(n)
                n = int(parents[b, n])
            if all(own[b, n] for n in chain) and len(chain) - 1 > best_d:
                best, best_d = i, len(chain) - 1
        alen[b] = best_d
        n = best
        while n >= 0:
            path[b, workloads.depths_of(parents[b])[n]] = n
            n = int(parents[b, n])
        nxt[b] = int(np.argmax(x64[b, best]))   # first index among equal maxima
    return prob, thr, own, alen, path, nxt


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("tau", [0.5, 1.0, 1.7])
def test_matches_scipy_softmax_entropy_and_exhaustive_paths(dtype, tau):
    rng = np.random.default_rng(int(tau * 10) + len(dtype))
    B, T, V = 8, 12, 7
    parents = _random_parents(rng, B, T)
    md = int(max(workloads.depths_of(p).max() for p in parents))
    lg = oracle.round_to_act(rng.normal(0, 2.0, (B, T, V)).astype(np.float32), dtype)
    tokens = rng.integers(-1, V + 1, (B, T)).astype(np.int32)   # includes -1 and V: never accepted
    eps, delta = 0.2, 0.6
    r = oracle.accept_typical(tokens, lg, dtype, parents, md, tau, eps, delta)
    assert r["status"] == 0
    x64 = oracle.act_to_f64(lg, dtype)
    prob, thr, own, alen, path, nxt = _brute(tokens, x64, parents, md, tau, eps, delta)
    assert np.allclose(r["prob"], prob, rtol=1e-12, atol=1e-300)
    assert np.allclose(r["thr"], thr, rtol=1e-12)
    clear = np.abs(prob - thr) > 1e-9 * np.maximum(thr, 1e-300)
    assert np.array_equal(r["node_accept"].astype(bool)[clear], own[clear])
    assert np.array_equal(r["accept_len"], alen)
    assert np.array_equal(r["accept_path"], path)
    assert np.array_equal(r["next_token"], nxt)
    assert own.sum() > T and (~own).sum() > T   # both outcomes occur


def test_peaked_rows_reduce_to_greedy():
    # one logit far above the rest: q[argmax] ~ 1, H ~ 0, thr = min(eps, delta) < 1
    rng = np.random.default_rng(7)
    B, T, V = 6, 16, 50
    parents = _random_parents(rng, B, T)
    md = int(max(workloads.depths_of(p).max() for p in parents))
    lg = rng.normal(0, 1, (B, T, V)).astype(np.float32)
    top = rng.integers(0, V, (B, T))
    np.put_along_axis(lg, top[..., None], 80.0, axis=2)
    tokens = np.where(rng.random((B, T)) < 0.7, np.take_along_axis(top, parents.clip(0), 1),
                      rng.integers(0, V, (B, T))).astype(np.int32)
    r = oracle.accept_typical(tokens, lg, "f32", parents, md, 1.0, 0.09, 0.3)
    am, alen, path, nxt = oracle.accept_greedy(tokens, lg, "f32", parents, md)
    assert np.array_equal(r["accept_len"], alen)
    assert np.array_equal(r["accept_path"], path)
    assert np.array_equal(r["next_token"], nxt)
    assert alen.max() >= 2


def test_temperature_is_a_logit_scale():
    rng = np.random.default_rng(3)
    B, T, V = 4, 10, 33
    parents = _random_parents(rng, B, T)
    md = int(max(workloads.depths_of(p).max() for p in parents))
    lg = rng.normal(0, 3, (B, T, V)).astype(np.float32)
    tokens = rng.integers(0, V, (B, T)).astype(np.int32)
    a = oracle.accept_typical(tokens, lg, "f32", parents, md, 2.0, 0.05, 0.4)
    b = oracle.accept_typical(tokens, lg / np.float32(2), "f32", parents, md, 1.0, 0.05, 0.4)
    assert np.allclose(a["prob"], b["prob"], rtol=1e-13)
    assert np.allclose(a["thr"], b["thr"], rtol=1e-13)
    assert np.array_equal(a["node_accept"], b["node_accept"])


def test_accepted_sets_shrink_as_thresholds_grow():
    rng = np.random.default_rng(5)
    B, T, V = 6, 20, 40
    parents = _random_parents(rng, B, T)
    md = int(max(workloads.depths_of(p).max() for p in parents))
    lg = rng.normal(0, 2, (B, T, V)).astype(np.float32)
    tokens = rng.integers(0, V, (B, T)).astype(np.int32)
    prev = None
    for eps, delta in ((0.01, 0.05), (0.02, 0.1), (0.05, 0.3), (0.1, 0.6), (0.3, 2.0)):
        r = oracle.accept_typical(tokens, lg, "f32", parents, md, 1.0, eps, delta)
        cur = r["node_accept"].astype(bool)
        if prev is not None:
            assert not np.any(cur & ~prev)
            assert np.all(r["accept_len"] <= prev_len)
        prev, prev_len = cur, r["accept_len"]
    assert prev.sum() < B * T


def test_rejects_bad_parameters():
    lg = np.zeros((1, 2, 4), np.float32)
    tok = np.zeros((1, 2), np.int32)
    for tau, eps, delta in ((0.0, 0.1, 0.1), (1.0, 0.0, 0.1), (1.0, 0.1, -1.0), (float("nan"), 0.1, 0.1),
                            (1.0, float("inf"), 0.1)):
        assert oracle.accept_typical(tok, lg, "f32", _chain(2), 1, tau, eps, delta)["status"] == -1
    bad = np.array([[-1, 1]], np.int32)
    assert oracle.accept_typical(tok, lg, "f32", bad, 1, 1.0, 0.1, 0.1)["status"] == -3
