"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties an oracle function to an independent fact: a library routine
for a special case, a closed form, an invariant the mathematics guarantees, an
exhaustive enumeration, or a hand-derived fixture under ``tests/golden/``.
A plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong tie rule) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from oracle import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand():
    with open(os.path.join(GOLDEN, "tiny_tree_hand.json")) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def _edge_floats():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 3,
        rng.standard_normal(5000).astype(np.float32) * 1e-6,      # fp16 subnormals
        rng.standard_normal(5000).astype(np.float32) * 1e4,
        np.array([0.0, -0.0, 65504, 65519.99, 65520, -65520, 1e-8, 5.96e-8, 2.98e-8,
                  1.0 + 2**-11, 1.0 + 3 * 2**-11, 1.0 + 2**-8, 1.0 + 3 * 2**-8,
                  3.3895314e38, 3.4e38, 1e-40, -1e-45], dtype=np.float32),
    ])
    return x


def test_f16_rounding_matches_numpy():
    # NumPy's float32 -> float16 cast rounds to nearest, ties to even.
    x = _edge_floats()
    got = oracle.round_to_act(x, "f16")
    with np.errstate(over="ignore"):
        want = x.astype(np.float16)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_bf16_rounding_is_nearest_even():
    # From the definition: the result is the nearer of the two bf16 values that
    # bracket x (truncation and truncation + 1 ulp), the even one on a tie.
    x = _edge_floats()
    x = x[np.abs(x) < 3.38e38]
    got = oracle.round_to_act(x, "bf16").astype(np.uint32)
    bits = x.view(np.uint32)
    lo = bits >> 16
    hi = lo + 1
    lo_v = (lo << 16).view(np.float32).astype(np.float64)
    hi_v = (hi << 16).view(np.float32).astype(np.float64)
    xd = x.astype(np.float64)
    dlo, dhi = np.abs(xd - lo_v), np.abs(hi_v - xd)
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    assert np.array_equal(got, want)


def _same_f64(got, want):
    # equal values, NaN where NaN, and the sign of every zero
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_f16_widening_matches_numpy_on_every_code():
    # every binary16 bit pattern: zeros, subnormals, normals, infinities, NaNs
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = codes.view(np.float16)
    got = oracle.act_to_f64(x, "f16")
    _same_f64(got, x.astype(np.float64))
    # a few values the format fixes, read off its definition
    assert got[0x0001] == 2.0**-24 and got[0x03FF] == 1023 * 2.0**-24
    assert got[0x0400] == 2.0**-14 and got[0x3C00] == 1.0 and got[0x7BFF] == 65504.0
    assert got[0x7C00] == np.inf and got[0xFC00] == -np.inf and np.isnan(got[0x7E00])
    assert got[0x8000] == 0.0 and np.signbit(got[0x8000])


def test_bf16_widening_matches_torch_on_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.act_to_f64(codes, "bf16")
    want = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    _same_f64(got, want)
    assert got[0x0001] == 2.0**-133 and got[0x0080] == 2.0**-126 and got[0x3F80] == 1.0
    assert got[0x7F7F] == 255 * 2.0**120 and got[0x7F80] == np.inf and np.isnan(got[0x7FC0])
    assert got[0xC000] == -2.0


def test_f32_widening_is_exact():
    x = _edge_floats()
    _same_f64(oracle.act_to_f64(x, "f32"), x.astype(np.float64))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = _edge_floats()
    got = oracle.round_to_act(x, "bf16")
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_table_literals():
    c, s = oracle.rope_table(10000.0, 64, 200)
    assert c[0].tolist() == [1.0] * 32 and s[0].tolist() == [0.0] * 32
    # pos 1, pair 0: angle 1 rad
    assert c[1, 0] == np.float32(0.5403023058681398)
    assert s[1, 0] == np.float32(0.8414709848078965)
    # pair 16 of D=64 has frequency 10000^(-1/2) = 0.01: pos 100 is 1 rad again
    assert abs(float(c[100, 16]) - 0.5403023058681398) < 1e-7
    assert abs(float(s[100, 16]) - 0.8414709848078965) < 1e-7
    # pos 2, pair 0: angle 2 rad
    assert c[2, 0] == np.float32(-0.4161468365471424)
    assert s[2, 0] == np.float32(0.9092974268256817)


def test_rope_rotation_direction_and_pairing():
    # e_0 at position 1 must become cos(1) e_0 + sin(1) e_{D/2}: this fixes the
    # half-split pairing (not interleaved) and the rotation's sign.
    D = 64
    table = oracle.rope_table(10000.0, D, 8)
    x = np.zeros((1, D), np.float32)
    x[0, 0] = 1.0
    y = oracle.rope_rotate(x, "f32", np.array([1]), table)
    want = np.zeros(D, np.float32)
    want[0] = np.float32(0.5403023058681398)
    want[D // 2] = np.float32(0.8414709848078965)
    assert np.array_equal(y[0], want)
    x = np.zeros((1, D), np.float32)
    x[0, D // 2] = 1.0
    y = oracle.rope_rotate(x, "f32", np.array([1]), table)
    want = np.zeros(D, np.float32)
    want[0] = -np.float32(0.8414709848078965)
    want[D // 2] = np.float32(0.5403023058681398)
    assert np.array_equal(y[0], want)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_rope_position_zero_is_identity(dtype):
    rng = np.random.default_rng(1)
    x = workloads._np_normal(rng, (5, 128), dtype)
    table = oracle.rope_table(10000.0, 128, 4)
    y = oracle.rope_rotate(x, dtype, np.zeros(5, np.int32), table)
    assert np.array_equal(y.view(np.uint8), x.view(np.uint8))


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(2)
    D = 128
    x = rng.standard_normal((50, D)).astype(np.float32)
    pos = rng.integers(0, 40000, 50)
    y = oracle.rope_rotate(x, "f32", pos, oracle.rope_table(10000.0, D, 40001))
    n0 = x[:, :D // 2].astype(np.float64) ** 2 + x[:, D // 2:].astype(np.float64) ** 2
    n1 = y[:, :D // 2].astype(np.float64) ** 2 + y[:, D // 2:].astype(np.float64) ** 2
    assert np.allclose(n0, n1, rtol=2e-6, atol=1e-6)


def test_rope_scores_depend_on_relative_position_only():
    # <R(p) q, R(p + d) k> is the same for every p (RoPE's defining property).
    rng = np.random.default_rng(3)
    D = 128
    q = rng.standard_normal((1, D)).astype(np.float32)
    k = rng.standard_normal((1, D)).astype(np.float32)
    table = oracle.rope_table(10000.0, D, 5000)
    ref = None
    for p in (0, 7, 300, 2048, 4000):
        qr = oracle.rope_rotate(q, "f32", np.array([p]), table).astype(np.float64)
        kr = oracle.rope_rotate(k, "f32", np.array([p + 5]), table).astype(np.float64)
        s = float(qr[0] @ kr[0])
        if ref is None:
            ref = s
        assert abs(s - ref) < 2e-3 * (1 + abs(ref))


# --------------------------------------------------------------------------
# tree attention
# --------------------------------------------------------------------------

def _small_cases():
    cases = []
    for dtype in ("f32", "f16", "bf16"):
        cases.append(workloads.custom(B=2, Hq=4, Hkv=2, head_dim=16, dtype=dtype,
                                      prefix=("list", [37, 5]), tree=("fanout", (3, 2, 2), 9),
                                      max_depth=3, page_size=4))
    cases.append(workloads.custom(B=1, Hq=2, Hkv=1, head_dim=8, dtype="f32", prefix=("fixed", 0),
                                  tree=("chain", 6), max_depth=5, page_size=4))
    cases.append(workloads.custom(B=3, Hq=3, Hkv=3, head_dim=8, dtype="f32",
                                  prefix=("list", [1, 16, 17]), tree=("star", 5), max_depth=1,
                                  page_size=16))
    cases.append(workloads.custom(B=2, Hq=2, Hkv=2, head_dim=8, dtype="bf16",
                                  prefix=("list", [3, 64]), tree=("fixed", (-1,)), max_depth=0,
                                  page_size=16))
    cases.append(workloads.custom(B=1, Hq=1, Hkv=1, head_dim=64, dtype="f32",
                                  prefix=("fixed", 128), tree=("fixed", workloads.TINY_TREE_PARENTS),
                                  max_depth=3))
    return cases


@pytest.mark.parametrize("case", range(7))
def test_tree_attn_matches_dense_brute_force(case):
    spec = _small_cases()[case]
    for seed in range(3):
        w = workloads.generate(spec, seed=seed)
        q_rot, k_rot = oracle.rotate_inputs(w)
        got = oracle.tree_attn(w, q_rot=q_rot, k_rot=k_rot)
        want = bf.dense_tree_attn(w, q_rot, k_rot)
        assert np.max(np.abs(got - want)) < 1e-12


def test_tree_attn_uniform_weights_hand_fixture():
    # q = 0: every visible key scores 0, so each output is the mean of the
    # visible values; the golden file lists the ancestor sets and the means.
    hand = _hand()
    parents = hand["tree"]["parents"]
    spec = workloads.custom(B=1, Hq=1, Hkv=1, head_dim=4, dtype="f32", prefix=("fixed", 2),
                            tree=("fixed", tuple(parents)), max_depth=3, page_size=4)
    w = workloads.generate(spec, seed=5)
    pv = hand["uniform_attention"]["prefix_values"]
    tv = hand["uniform_attention"]["tree_values"]
    w["q"][:] = 0.0
    for slot, val in enumerate(pv):
        page = w["block_tables"][0, slot // 4]
        w["v_cache"][page, 0, slot % 4, :] = val
    w["v_new"][0, :, 0, :] = np.asarray(tv, np.float32)[:, None]
    out = oracle.tree_attn(w)
    want = [float(Fraction(f)) for f in hand["uniform_attention"]["expected_fractions"]]
    assert np.allclose(out[0, :, 0, :], np.asarray(want)[:, None], rtol=0, atol=1e-12)
    # and the ancestor sets of the hand fixture are what the brute force derives
    anc = bf.ancestor_matrix(parents)
    for i, lst in enumerate(hand["tree"]["ancestors_inclusive"]):
        assert sorted(np.nonzero(anc[i])[0].tolist()) == lst


def test_tree_attn_path_invariant():
    # node i's output = ordinary causal attention over prefix || (root..i),
    # read at the last position.
    spec = workloads.custom(B=2, Hq=4, Hkv=2, head_dim=16, dtype="f16", prefix=("list", [21, 40]),
                            tree=("fanout", (4, 3, 2), 12), max_depth=3, page_size=8)
    w = workloads.generate(spec, seed=11)
    q_rot, k_rot = oracle.rotate_inputs(w)
    got = oracle.tree_attn(w, q_rot=q_rot, k_rot=k_rot)
    q = oracle.act_to_f64(q_rot, "f16")
    kt = oracle.act_to_f64(k_rot, "f16")
    vt = oracle.act_to_f64(w["v_new"], "f16")
    kc = oracle.act_to_f64(w["k_cache"], "f16")
    vc = oracle.act_to_f64(w["v_cache"], "f16")
    scale = 1 / math.sqrt(16)
    for b in range(2):
        L = int(w["seq_lens"][b])
        kp = bf.gather_prefix(kc, w["block_tables"][b], L, 8)
        vp = bf.gather_prefix(vc, w["block_tables"][b], L, 8)
        for i in range(w["T"]):
            path = [i]
            while path[-1] != 0:
                path.append(int(w["tree_parents"][b][path[-1]]))
            path = path[::-1]
            for h in range(4):
                kvh = h // 2
                n = L + len(path)
                qs = np.zeros((n, 16))
                qs[-1] = q[b, i, h]
                ks = np.concatenate([kp[:, kvh], kt[b, path, kvh]])
                vs = np.concatenate([vp[:, kvh], vt[b, path, kvh]])
                want = bf.causal_attention(qs, ks, vs, scale)[-1]
                assert np.max(np.abs(got[b, i, h] - want)) < 1e-12


def test_tree_attn_chain_is_causal_multi_token_decode():
    # Medusa list decoding: a single chain of T nodes after a prefix is causal
    # attention of the T new tokens over prefix + chain; with prefix 0 it is
    # textbook causal self-attention.
    for L in (0, 13):
        spec = workloads.custom(B=1, Hq=2, Hkv=2, head_dim=16, dtype="f32", prefix=("fixed", L),
                                tree=("chain", 7), max_depth=6, page_size=4)
        w = workloads.generate(spec, seed=3 + L)
        q_rot, k_rot = oracle.rotate_inputs(w)
        got = oracle.tree_attn(w, q_rot=q_rot, k_rot=k_rot)
        kp = bf.gather_prefix(w["k_cache"].astype(np.float64), w["block_tables"][0], L, 4)
        vp = bf.gather_prefix(w["v_cache"].astype(np.float64), w["block_tables"][0], L, 4)
        for h in range(2):
            ks = np.concatenate([kp[:, h], k_rot[0, :, h].astype(np.float64)])
            vs = np.concatenate([vp[:, h], w["v_new"][0, :, h].astype(np.float64)])
            qs = np.concatenate([np.zeros((L, 16)), q_rot[0, :, h].astype(np.float64)])
            want = bf.causal_attention(qs, ks, vs, 0.25)[L:]
            assert np.max(np.abs(got[0, :, h] - want)) < 1e-12


def test_tree_attn_single_node_is_paged_decode():
    # T = 1: one new token against the paged cache, the case single-token
    # paged decode kernels handle.
    spec = workloads.custom(B=3, Hq=8, Hkv=2, head_dim=32, dtype="bf16",
                            prefix=("list", [1, 33, 100]), tree=("fixed", (-1,)), max_depth=0,
                            page_size=16)
    w = workloads.generate(spec, seed=9)
    q_rot, k_rot = oracle.rotate_inputs(w)
    got = oracle.tree_attn(w, q_rot=q_rot, k_rot=k_rot)
    kc = oracle.act_to_f64(w["k_cache"], "bf16")
    vc = oracle.act_to_f64(w["v_cache"], "bf16")
    q = oracle.act_to_f64(q_rot, "bf16")
    kt = oracle.act_to_f64(k_rot, "bf16")
    vt = oracle.act_to_f64(w["v_new"], "bf16")
    for b in range(3):
        L = int(w["seq_lens"][b])
        kp = bf.gather_prefix(kc, w["block_tables"][b], L, 16)
        vp = bf.gather_prefix(vc, w["block_tables"][b], L, 16)
        for h in range(8):
            ks = np.concatenate([kp[:, h // 4], kt[b, :1, h // 4]])
            vs = np.concatenate([vp[:, h // 4], vt[b, :1, h // 4]])
            want = bf.decode_attention(q[b, 0, h], ks, vs, 1 / math.sqrt(32))
            assert np.max(np.abs(got[b, 0, h] - want)) < 1e-12


def test_tree_attn_page_relabeling_invariance():
    spec = workloads.custom(B=2, Hq=2, Hkv=1, head_dim=16, dtype="f16", prefix=("list", [30, 9]),
                            tree=("fanout", (2, 2), 6), max_depth=2, page_size=4)
    w = workloads.generate(spec, seed=4)
    base = oracle.tree_attn(w)
    perm = np.random.default_rng(0).permutation(w["num_pages"])
    w2 = dict(w)
    w2["k_cache"] = np.empty_like(w["k_cache"])
    w2["v_cache"] = np.empty_like(w["v_cache"])
    w2["k_cache"][perm] = w["k_cache"]
    w2["v_cache"][perm] = w["v_cache"]
    bt = w["block_tables"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    w2["block_tables"] = bt
    assert np.array_equal(oracle.tree_attn(w2), base)


def test_tree_attn_sharp_key_selects_its_value():
    # One prefix key aligned with the query, scaled far above the rest: the
    # output is that key's value.
    spec = workloads.custom(B=1, Hq=1, Hkv=1, head_dim=8, dtype="f32", prefix=("fixed", 20),
                            tree=("fixed", (-1, 0)), max_depth=1, page_size=4)
    w = workloads.generate(spec, seed=2)
    q_rot, k_rot = oracle.rotate_inputs(w)
    page = w["block_tables"][0, 13 // 4]
    w["k_cache"][page, 0, 13 % 4, :] = q_rot[0, 1, 0, :] * 400.0
    out = oracle.tree_attn(w, q_rot=q_rot, k_rot=k_rot)
    assert np.allclose(out[0, 1, 0], w["v_cache"][page, 0, 13 % 4].astype(np.float64), atol=1e-9)


def test_tree_attn_rejects_bad_trees_and_pages():
    spec = workloads.custom(B=1, Hq=1, Hkv=1, head_dim=8, dtype="f32", prefix=("fixed", 8),
                            tree=("fanout", (2,), 3), max_depth=1, page_size=4)
    w = workloads.generate(spec, seed=0)
    bad = dict(w)
    bad["tree_parents"] = np.array([[-1, 2, 0]], np.int32)     # parent after child
    with pytest.raises(oracle.OracleError):
        oracle.tree_attn(bad)
    bad = dict(w)
    bt = w["block_tables"].copy()
    bt[0, 0] = w["num_pages"]                                    # page out of range
    bad["block_tables"] = bt
    with pytest.raises(oracle.OracleError):
        oracle.tree_attn(bad)
    assert not oracle.check_tree([-1, 0, 0], [0, 1, 2])
    assert oracle.check_tree([-1, 0, 0], [0, 1, 1])


def test_tree_scatter_places_rotated_keys():
    spec = workloads.custom(B=2, Hq=2, Hkv=2, head_dim=8, dtype="bf16", prefix=("list", [5, 16]),
                            tree=("fanout", (2, 2), 5), max_depth=2, page_size=4)
    w = workloads.generate(spec, seed=1)
    q_rot, k_rot = oracle.rotate_inputs(w)
    kc, vc = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
    for b in range(2):
        L = int(w["seq_lens"][b])
        for i in range(w["T"]):
            s = L + i
            page = w["block_tables"][b, s // 4]
            assert np.array_equal(kc[page, :, s % 4], k_rot[b, i])
            assert np.array_equal(vc[page, :, s % 4], w["v_new"][b, i])
    # nothing below the prefix length changed
    mask = workloads._prefix_slot_mask(spec, w["block_tables"], w["seq_lens"], w["num_pages"])
    assert np.array_equal(kc.transpose(0, 2, 1, 3)[mask], w["k_cache"].transpose(0, 2, 1, 3)[mask])


# --------------------------------------------------------------------------
# greedy acceptance
# --------------------------------------------------------------------------

def test_accept_hand_fixture():
    hand = _hand()["accept"]
    parents = np.array([_hand()["tree"]["parents"]], np.int32)
    logits = np.array([hand["logits"]], np.float32)
    am, alen, path, nxt = oracle.accept_greedy(np.array([hand["tokens"]]), logits, "f32", parents,
                                               hand["max_depth"])
    assert am[0].tolist() == hand["argmax"]
    assert alen[0] == hand["accept_len"]
    assert path[0].tolist() == hand["accept_path"]
    assert nxt[0] == hand["next_token"]


@pytest.mark.parametrize("V", [2, 3, 5])
def test_accept_matches_exhaustive_enumeration(V):
    rng = np.random.default_rng(V)
    for trial in range(300):
        T = int(rng.integers(1, 9))
        parents = np.array([-1] + [int(rng.integers(i)) for i in range(1, T)], np.int32)
        depth = workloads.depths_of(parents)
        tokens = rng.integers(0, V, T).astype(np.int32)
        # small integer logits force ties; sprinkle signed zeros
        logits = rng.integers(-1, 2, (T, V)).astype(np.float32)
        logits[logits == 0] *= rng.choice([-1.0, 1.0], size=int((logits == 0).sum()))
        md = int(depth.max()) + int(rng.integers(0, 2))
        for dt in ("f32", "f16", "bf16"):
            lg = oracle.round_to_act(logits, dt)
            am, alen, path, nxt = oracle.accept_greedy(tokens[None], lg[None], dt, parents[None], md)
            want_len, want_path, want_next, want_am = bf.enumerate_accept(
                tokens.tolist(), logits.astype(np.float64), parents.tolist(), md)
            assert am[0].tolist() == want_am
            assert alen[0] == want_len and path[0].tolist() == want_path and nxt[0] == want_next


def test_accept_argmax_matches_numpy_on_vocab_rows():
    rng = np.random.default_rng(7)
    for dt in ("f32", "f16", "bf16"):
        x = rng.standard_normal((1, 6, 32000)).astype(np.float32)
        lg = oracle.round_to_act(x, dt)
        am, *_ = oracle.accept_greedy(np.zeros((1, 6), np.int32), lg, dt,
                                      np.array([[-1, 0, 1, 2, 3, 4]], np.int32), 5)
        ref = np.argmax(oracle.act_to_f64(lg, dt), axis=-1)
        assert np.array_equal(am, ref)


def test_accept_recovers_planted_paths():
    for name in ("tiny_tree_fp32", "llama7b_b1_fp16"):
        w = workloads.generate(name, seed=1)
        am, alen, path, nxt = oracle.accept_greedy(w["tree_tokens"], w["logits"], w["logits_dtype"],
                                                   w["tree_parents"], w["max_depth"])
        for b in range(w["B"]):
            planted = w["planted_nodes"][b]
            assert alen[b] >= len(planted)
            if alen[b] == len(planted):
                assert path[b, 1:1 + len(planted)].tolist() == planted


# --------------------------------------------------------------------------
# KV commit
# --------------------------------------------------------------------------

def test_commit_hand_fixture():
    hand = _hand()["commit"]
    P = hand["page_size"]
    T = 7
    w = dict(B=1, T=T, Hkv=1, head_dim=2, dtype="f32", page_size=P, max_blocks=4,
             num_pages=hand["num_pages"])
    kc = np.full((hand["num_pages"], 1, P, 2), -7.0, np.float32)
    vc = np.full((hand["num_pages"], 1, P, 2), -9.0, np.float32)
    bt = np.array([hand["block_table"]], np.int32)
    L = hand["seq_len"]
    for i in range(T):
        s = L + i
        kc[bt[0, s // P], 0, s % P] = [100 + i, 200 + i]
        vc[bt[0, s // P], 0, s % P] = [300 + i, 400 + i]
    path = np.array([hand["accept_path"]], np.int32)
    k2, v2, bt2, sl2, rel = oracle.kv_commit(w, path, np.array([hand["accept_len"]]), kc, vc, bt,
                                             np.array([L]), max_depth=3)
    assert sl2.tolist() == [hand["expected_seq_len"]]
    assert bt2[0].tolist() == hand["expected_block_table"]
    assert rel[0].tolist() == hand["expected_released"]
    for slot, node in hand["expected_slot_nodes"].items():
        s = int(slot)
        page = bt[0, s // P]
        assert k2[page, 0, s % P].tolist() == [100 + node, 200 + node]
        assert v2[page, 0, s % P].tolist() == [300 + node, 400 + node]
    assert np.array_equal(k2[4], kc[4]) and np.array_equal(v2[4], vc[4])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_commit_against_gather_scatter_model(dtype):
    spec = workloads.custom(B=4, Hq=4, Hkv=2, head_dim=8, dtype=dtype,
                            prefix=("list", [3, 16, 29, 0]), tree=("fanout", (3, 2, 2, 1), 11),
                            max_depth=4, page_size=4, vocab=7, logits_dtype="f32",
                            plant=("uniform", 0, 4))
    w = workloads.generate(spec, seed=8)
    q_rot, k_rot = oracle.rotate_inputs(w)
    kc, vc = oracle.tree_scatter(w, w["k_cache"], w["v_cache"], k_rot=k_rot)
    _, alen, path, _ = oracle.accept_greedy(w["tree_tokens"], w["logits"], "f32", w["tree_parents"], 4)
    k2, v2, bt2, sl2, rel = oracle.kv_commit(w, path, alen, kc, vc, w["block_tables"], w["seq_lens"], 4)
    P = 4
    touched = np.zeros((w["num_pages"], P), bool)
    for b in range(4):
        L = int(w["seq_lens"][b])
        n = int(alen[b]) + 1
        assert sl2[b] == L + n
        bt = w["block_tables"][b]
        for d in range(n):
            src, dst = L + path[b, d], L + d
            assert np.array_equal(k2[bt[dst // P], :, dst % P].view(np.uint8),
                                  kc[bt[src // P], :, src % P].view(np.uint8))
            assert np.array_equal(v2[bt[dst // P], :, dst % P].view(np.uint8),
                                  vc[bt[src // P], :, src % P].view(np.uint8))
            touched[bt[dst // P], dst % P] = True
        # released: logical blocks starting at or past the new length that hold scratch
        want_rel = [int(bt[p]) for p in range(len(bt)) if bt[p] >= 0 and p * P >= L + n and p * P < L + w["T"]]
        assert rel[b].tolist() == want_rel + [-1] * (rel.shape[1] - len(want_rel))
        for p in range(len(bt)):
            assert bt2[b, p] == (-1 if int(bt[p]) in want_rel else bt[p])
    # every other byte of the cache is unchanged
    keep = ~touched
    assert np.array_equal(k2.transpose(0, 2, 1, 3)[keep].view(np.uint8),
                          kc.transpose(0, 2, 1, 3)[keep].view(np.uint8))
    assert np.array_equal(v2.transpose(0, 2, 1, 3)[keep].view(np.uint8),
                          vc.transpose(0, 2, 1, 3)[keep].view(np.uint8))
