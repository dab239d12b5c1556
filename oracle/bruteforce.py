"""Dense-mask brute force and textbook attention, NumPy float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  These formulations are
deliberately different from ``medusa_oracle.c`` so that the tests can pin one
against the other:

* ``dense_tree_attn`` gathers each sequence's prefix from the paged cache with
  NumPy fancy indexing, builds the full ``[T, L+T]`` visibility matrix (prefix
  columns all visible; tree columns from the ancestor-or-self relation, found
  as the transitive closure of the parent relation by repeated boolean matrix
  products), and runs one dense masked softmax per head.
* ``causal_attention`` is ordinary causal self-attention over a flat sequence.
* ``decode_attention`` is single-query attention over a key list.

The pages fix what the tree mask means (vLLM issue 1171, void-main: "set
medusa tree mask ... in single_query_cached_kv_attention"; each candidate sees
the existing KV cache plus its own tree ancestors); these are the plain
definitions, vectorised.
"""
from __future__ import annotations

import numpy as np


def act_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen act-dtype values to float64 with NumPy's own conversions, not the
    C oracle's decoder, so that the brute force does not inherit a slip in it:
    fp16 through NumPy's binary16 type; bf16 as the upper half of a float32
    (the bfloat16 layout), read by NumPy as float32."""
    if dtype == "f32":
        return np.asarray(x, np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(x, np.float16).astype(np.float64)
    bits = np.asarray(x, np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def ancestor_matrix(parents) -> np.ndarray:
    """A[i, j] = True iff j is i or an ancestor of i (transitive closure)."""
    parents = np.asarray(parents)
    T = len(parents)
    step = np.zeros((T, T), dtype=np.int64)
    for i in range(1, T):
        step[i, parents[i]] = 1
    reach = np.eye(T, dtype=np.int64)
    while True:
        nxt = ((reach + reach @ step) > 0).astype(np.int64)
        if np.array_equal(nxt, reach):
            return reach.astype(bool)
        reach = nxt


def gather_prefix(cache: np.ndarray, block_table: np.ndarray, L: int, page_size: int) -> np.ndarray:
    """[L, Hkv, D] rows of logical slots 0..L-1 from a [pages, Hkv, P, D] cache."""
    slots = np.arange(L)
    pages = block_table[slots // page_size]
    assert np.all(pages >= 0), "block table does not cover the prefix"
    return cache[pages, :, slots % page_size, :]


def dense_tree_attn(w: dict, q_rot: np.ndarray, k_rot: np.ndarray) -> np.ndarray:
    """[B, T, Hq, D] float64 outputs by dense masked softmax."""
    dt = w["dtype"]
    B, T, Hq, Hkv, D = w["B"], w["T"], w["Hq"], w["Hkv"], w["head_dim"]
    g = Hq // Hkv
    scale = w.get("sm_scale") or 1.0 / np.sqrt(D)
    kc = act_to_f64(w["k_cache"], dt)
    vc = act_to_f64(w["v_cache"], dt)
    q = act_to_f64(q_rot, dt)
    kt = act_to_f64(k_rot, dt)
    vt = act_to_f64(w["v_new"], dt)
    out = np.zeros((B, T, Hq, D))
    for b in range(B):
        L = int(w["seq_lens"][b])
        kp = gather_prefix(kc, w["block_tables"][b], L, w["page_size"])
        vp = gather_prefix(vc, w["block_tables"][b], L, w["page_size"])
        keys = np.concatenate([kp, kt[b]], axis=0)          # [L+T, Hkv, D]
        vals = np.concatenate([vp, vt[b]], axis=0)
        visible = np.concatenate([np.ones((T, L), dtype=bool),
                                  ancestor_matrix(w["tree_parents"][b])], axis=1)
        for h in range(Hq):
            kvh = h // g
            s = q[b, :, h, :] @ keys[:, kvh, :].T * scale    # [T, L+T]
            s = np.where(visible, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            out[b, :, h, :] = p @ vals[:, kvh, :]
    return out


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Textbook causal self-attention over one flat sequence, [n, D] each."""
    n = q.shape[0]
    s = q @ k.T * scale
    s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def decode_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """One query [D] against keys/values [n, D] (the single-token decode case)."""
    s = k @ q * scale
    p = np.exp(s - s.max())
    return (p / p.sum()) @ v


def enumerate_accept(tokens, logits_f64: np.ndarray, parents, max_depth: int):
    """Greedy acceptance by exhaustive enumeration of root paths (one sequence).

    Every root-to-node path is listed; a path is accepted when each of its
    non-root tokens equals the argmax (first index among equal maxima) of its
    parent's logits.  The answer is the longest accepted path, the one ending at
    the lowest node index among equally long ones.  Returns (accept_len,
    path padded to max_depth+1 with -1, next_token)."""
    parents = list(parents)
    T = len(parents)
    am = [int(np.argmax(logits_f64[i])) for i in range(T)]
    best = None
    for end in range(T):
        path = [end]
        while path[-1] != 0:
            path.append(parents[path[-1]])
        path = path[::-1]
        ok = all(tokens[path[k]] == am[path[k - 1]] for k in range(1, len(path)))
        if ok and (best is None or len(path) > len(best)):
            best = path
    padded = best + [-1] * (max_depth + 1 - len(best))
    return len(best) - 1, padded, am[best[-1]], am
