"""Pins of the oracle's FP8-cache reading (tree scatter, tree attention and KV
commit over E4M3 codes with one scale for K and one for V), independent of its
C code: a dense-mask attention over the dequantised cache in NumPy, the
scatter's quantisation redone with NumPy float32 division and the (separately
pinned) codec, and the commit's byte moves restated in Python."""
import numpy as np

import oracle
import workloads
from oracle.bruteforce import ancestor_matrix, gather_prefix

K_SCALE, V_SCALE = np.float32(0.0173), np.float32(0.031)


def _work(seed=0):
    spec = workloads.custom("fp8", B=3, Hq=4, Hkv=2, head_dim=64, dtype="bf16",
                            prefix=("list", [0, 20, 37]), tree=("fanout", (3, 2, 2), 12), max_depth=3)
    w = workloads.generate(spec, seed=seed)
    rng = np.random.default_rng(seed)
    codes = lambda: rng.integers(0, 0x7E, size=w["k_cache"].shape, dtype=np.uint8) | (
        rng.integers(0, 2, size=w["k_cache"].shape, dtype=np.uint8) << 7)  # finite codes, both signs
    return w, codes(), codes()


def test_scatter_quantises_the_act_values_in_float32():
    w, kc, vc = _work(1)
    _, k_rot = oracle.rotate_inputs(w)
    kc2, vc2 = oracle.tree_scatter_e4m3(w, kc, vc, K_SCALE, V_SCALE, k_rot=k_rot)
    kq = oracle.act_to_f64(k_rot, "bf16").astype(np.float32) / K_SCALE
    vq = oracle.act_to_f64(w["v_new"], "bf16").astype(np.float32) / V_SCALE
    touched = np.zeros(kc.shape, bool)
    P = w["page_size"]
    for b in range(w["B"]):
        L = int(w["seq_lens"][b])
        for i in range(w["T"]):
            s = L + i
            page = w["block_tables"][b, s // P]
            assert np.array_equal(kc2[page, :, s % P], oracle.e4m3_encode(kq[b, i].astype(np.float64)))
            assert np.array_equal(vc2[page, :, s % P], oracle.e4m3_encode(vq[b, i].astype(np.float64)))
            touched[page, :, s % P] = True
    assert np.array_equal(kc2[~touched], kc[~touched]) and np.array_equal(vc2[~touched], vc[~touched])


def test_attention_equals_dense_masked_softmax_over_the_dequantised_cache():
    w, kc, vc = _work(2)
    q_rot, k_rot = oracle.rotate_inputs(w)
    kc, vc = oracle.tree_scatter_e4m3(w, kc, vc, K_SCALE, V_SCALE, k_rot=k_rot)
    got = oracle.tree_attn_e4m3(w, kc, vc, K_SCALE, V_SCALE, q_rot=q_rot)
    kd = oracle.e4m3_decode(kc) * float(K_SCALE)
    vd = oracle.e4m3_decode(vc) * float(V_SCALE)
    q = oracle.act_to_f64(q_rot, "bf16")
    B, T, Hq, Hkv, D = w["B"], w["T"], w["Hq"], w["Hkv"], w["head_dim"]
    g = Hq // Hkv
    for b in range(B):
        L = int(w["seq_lens"][b])
        keys = gather_prefix(kd, w["block_tables"][b], L + T, w["page_size"])   # [L+T, Hkv, D]
        vals = gather_prefix(vd, w["block_tables"][b], L + T, w["page_size"])
        visible = np.concatenate([np.ones((T, L), bool), ancestor_matrix(w["tree_parents"][b])], axis=1)
        for h in range(Hq):
            s = q[b, :, h, :] @ keys[:, h // g, :].T / np.sqrt(D)
            s = np.where(visible, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            want = (p / p.sum(axis=1, keepdims=True)) @ vals[:, h // g, :]
            assert np.allclose(got[b, :, h, :], want, rtol=1e-12, atol=1e-12)


def test_commit_moves_fp8_bytes_as_defined():
    w, kc, vc = _work(3)
    B, T, P = w["B"], w["T"], w["page_size"]
    md = w["max_depth"]
    rng = np.random.default_rng(3)
    depth = np.stack([workloads.depths_of(p) for p in w["tree_parents"]])
    alen = np.zeros(B, np.int32)
    path = np.full((B, md + 1), -1, np.int32)
    for b in range(B):   # a random root path of each tree
        node = int(rng.choice(np.nonzero(depth[b] == rng.integers(0, depth[b].max() + 1))[0]))
        chain = []
        while node >= 0:
            chain.append(node)
            node = int(w["tree_parents"][b][node])
        chain = chain[::-1]
        alen[b] = len(chain) - 1
        path[b, :len(chain)] = chain
    ko, vo, bt, sl, rel = oracle.kv_commit(w, path, alen, kc, vc, w["block_tables"], w["seq_lens"], md,
                                           cache_dtype="e4m3")
    kw, vw = kc.copy(), vc.copy()
    for b in range(B):
        L = int(w["seq_lens"][b])
        src = [kc[w["block_tables"][b, (L + int(path[b, d])) // P], :, (L + int(path[b, d])) % P].copy()
               for d in range(alen[b] + 1)]
        srv = [vc[w["block_tables"][b, (L + int(path[b, d])) // P], :, (L + int(path[b, d])) % P].copy()
               for d in range(alen[b] + 1)]
        for d in range(alen[b] + 1):
            s = L + d
            kw[w["block_tables"][b, s // P], :, s % P] = src[d]
            vw[w["block_tables"][b, s // P], :, s % P] = srv[d]
        assert sl[b] == L + alen[b] + 1
    assert np.array_equal(ko, kw) and np.array_equal(vo, vw)
