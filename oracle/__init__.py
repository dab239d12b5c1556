"""CPU oracle for the Medusa tree-verification step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``medusa_oracle.c`` (float64, plain loops, compiled
with ``-ffp-contract=off`` so fp32 steps are not fused); this module only
marshals NumPy arrays.  ``bruteforce.py`` holds an independent dense-mask
formulation that the tests use to pin the C code.

Array conventions: act-dtype arrays are NumPy ``float32`` (fp32), ``float16``
(fp16) or ``uint16`` holding bfloat16 bit patterns (bf16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "medusa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}  # e4m3: FP8 cache elements (codes)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.or_round_to_act.argtypes = [i32, i64, P, P]
            lib.or_act_to_double.argtypes = [i32, i64, P, P]
            lib.or_e4m3_encode_array.argtypes = [i64, P, P]
            lib.or_tree_scatter_e4m3.argtypes = [i32] * 8 + [P] * 6 + [ctypes.c_float, ctypes.c_float]
            lib.or_tree_attn_e4m3.argtypes = [i32] * 9 + [P] * 3 + [dbl, dbl] + [P] * 3 + [dbl, i64, P, P]
            lib.or_e4m3_decode_array.argtypes = [i64, P, P]
            lib.or_num_threads.restype = i32
            lib.or_rope_table.argtypes = [dbl, i32, i32, P, P]
            lib.or_rope_rotate.argtypes = [i32, i64, i32, P, P, i32, P, P, P]
            lib.or_check_tree.argtypes = [i32, P, P]
            lib.or_tree_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                         P, P, P, P, P, P, P, P, dbl, i64, P, P]
            lib.or_tree_scatter.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                            P, P, P, P, P, P]
            lib.or_accept_greedy.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
            lib.or_accept_typical.argtypes = [i32, i32, i32, i32, i32, P, P, P, dbl, dbl, dbl,
                                              P, P, P, P, P, P]
            lib.or_tree_candidates.argtypes = [i32, i32, i32, i32, i32, P, P, P, P]
            lib.or_kv_commit.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                         P, P, P, P, P, P, P, i32]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _act(a: np.ndarray, dtype: str) -> np.ndarray:
    want = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    assert a.dtype == want, f"{dtype} arrays must be {want}, got {a.dtype}"
    return np.ascontiguousarray(a)


class OracleError(RuntimeError):
    pass


def _check(st: int, what: str):
    if st != 0:
        raise OracleError(f"{what}: oracle status {st}")


def num_threads() -> int:
    return int(_load().or_num_threads())


def round_to_act(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the act dtype (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype={"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype])
    _load().or_round_to_act(DTYPES[dtype], x.size, _ptr(x), _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """FP8 E4M3 codes (uint8) of float64 values: nearest, ties to the even code,
    finite overflow and infinities saturated to +-448, NaN kept."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().or_e4m3_encode_array(x.size, _ptr(x), _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of FP8 E4M3 codes."""
    codes = np.ascontiguousarray(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().or_e4m3_decode_array(codes.size, _ptr(codes), _ptr(out))
    return out


def act_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    x = _act(x, dtype)
    out = np.empty(x.shape, dtype=np.float64)
    _load().or_act_to_double(DTYPES[dtype], x.size, _ptr(x), _ptr(out))
    return out


def rope_table(base: float, head_dim: int, max_pos: int):
    """fp32 cos/sin tables, each [max_pos, head_dim/2]."""
    c = np.empty((max_pos, head_dim // 2), dtype=np.float32)
    s = np.empty((max_pos, head_dim // 2), dtype=np.float32)
    _load().or_rope_table(float(base), head_dim, max_pos, _ptr(c), _ptr(s))
    return c, s


def rope_rotate(x: np.ndarray, dtype: str, pos: np.ndarray, table) -> np.ndarray:
    """Rotate rows of x ([..., D]); pos broadcasts over the leading dims."""
    x = _act(x, dtype)
    D = x.shape[-1]
    rows = x.size // D
    pos = _i32(np.broadcast_to(np.asarray(pos)[..., None], x.shape[:-1] + (1,))[..., 0]).reshape(-1)
    assert pos.size == rows
    cos_t, sin_t = table
    out = np.empty_like(x)
    st = _load().or_rope_rotate(DTYPES[dtype], rows, D, _ptr(x), _ptr(pos), cos_t.shape[0],
                                _ptr(cos_t), _ptr(sin_t), _ptr(out))
    _check(st, "rope_rotate")
    return out


def check_tree(parents, depths=None) -> bool:
    parents = _i32(parents)
    d = _i32(depths) if depths is not None else None
    st = _load().or_check_tree(parents.size, _ptr(parents), _ptr(d) if d is not None else None)
    return st == 0


def tree_positions(seq_lens, depths) -> np.ndarray:
    """Position of every tree token: prefix length + tree depth, [B, T]."""
    return _i32(np.asarray(seq_lens, dtype=np.int64)[:, None] + np.asarray(depths, dtype=np.int64))


def rotate_inputs(w: dict, table=None):
    """Rotated q [B,T,Hq,D] and rotated tree keys [B,T,Hkv,D] for a workload dict."""
    if table is None:
        table = rope_table(w["rope_base"], w["head_dim"], int(w["seq_lens"].max()) + w["T"] + 1)
    pos = tree_positions(w["seq_lens"], w["tree_depths"])
    q_rot = rope_rotate(w["q"], w["dtype"], pos[:, :, None], table)
    k_rot = rope_rotate(w["k_new"], w["dtype"], pos[:, :, None], table)
    return q_rot, k_rot


def tree_attn(w: dict, sel=None, q_rot=None, k_rot=None) -> np.ndarray:
    """Attention outputs (float64).

    sel: None for every (b, h, i) -> returns [B, T, Hq, D]; or an int array
    [n, 3] of (b, h, i) triples -> returns [n, D].
    """
    lib = _load()
    B, T, Hq, Hkv, D = w["B"], w["T"], w["Hq"], w["Hkv"], w["head_dim"]
    if q_rot is None or k_rot is None:
        q_rot, k_rot = rotate_inputs(w)
    full = sel is None
    if full:
        bb, ii, hh = np.meshgrid(np.arange(B), np.arange(T), np.arange(Hq), indexing="ij")
        sel = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)  # (b, i, h) order
    sel = _i32(sel).reshape(-1, 3)
    out = np.empty((sel.shape[0], D), dtype=np.float64)
    scale = w.get("sm_scale") or 1.0 / np.sqrt(D)
    st = lib.or_tree_attn(DTYPES[w["dtype"]], B, T, Hq, Hkv, D, w["page_size"], w["max_blocks"],
                          w["num_pages"], _ptr(q_rot), _ptr(k_rot), _ptr(_act(w["v_new"], w["dtype"])),
                          _ptr(_act(w["k_cache"], w["dtype"])), _ptr(_act(w["v_cache"], w["dtype"])),
                          _ptr(_i32(w["block_tables"])), _ptr(_i32(w["seq_lens"])),
                          _ptr(_i32(w["tree_parents"])), float(scale), sel.shape[0], _ptr(sel),
                          _ptr(out))
    _check(st, "tree_attn")
    if full:
        return out.reshape(B, T, Hq, D)
    return out


def tree_scatter(w: dict, k_cache: np.ndarray, v_cache: np.ndarray, k_rot=None):
    """The cache after the attention call: tree K (rotated) / V at slots len+i."""
    if k_rot is None:
        _, k_rot = rotate_inputs(w)
    kc = np.ascontiguousarray(k_cache).copy()
    vc = np.ascontiguousarray(v_cache).copy()
    st = _load().or_tree_scatter(DTYPES[w["dtype"]], w["B"], w["T"], w["Hkv"], w["head_dim"],
                                 w["page_size"], w["max_blocks"], w["num_pages"], _ptr(k_rot),
                                 _ptr(_act(w["v_new"], w["dtype"])), _ptr(kc), _ptr(vc),
                                 _ptr(_i32(w["block_tables"])), _ptr(_i32(w["seq_lens"])))
    _check(st, "tree_scatter")
    return kc, vc


def tree_scatter_e4m3(w: dict, k_codes: np.ndarray, v_codes: np.ndarray, k_scale: float,
                      v_scale: float, k_rot=None):
    """An FP8 cache (E4M3 codes, uint8) after the attention call: at slots len+i,
    the codes of the act-dtype rotated key / raw value divided by its scale in
    float32."""
    if k_rot is None:
        _, k_rot = rotate_inputs(w)
    kc = np.ascontiguousarray(k_codes, np.uint8).copy()
    vc = np.ascontiguousarray(v_codes, np.uint8).copy()
    st = _load().or_tree_scatter_e4m3(DTYPES[w["dtype"]], w["B"], w["T"], w["Hkv"], w["head_dim"],
                                      w["page_size"], w["max_blocks"], w["num_pages"], _ptr(k_rot),
                                      _ptr(_act(w["v_new"], w["dtype"])), _ptr(kc), _ptr(vc),
                                      _ptr(_i32(w["block_tables"])), _ptr(_i32(w["seq_lens"])),
                                      float(k_scale), float(v_scale))
    _check(st, "tree_scatter_e4m3")
    return kc, vc


def tree_attn_e4m3(w: dict, k_codes: np.ndarray, v_codes: np.ndarray, k_scale: float, v_scale: float,
                   sel=None, q_rot=None) -> np.ndarray:
    """Attention outputs (float64) over an FP8 cache that already holds the tree's
    K/V (tree_scatter_e4m3): every visible slot, prefix and tree, read as
    decode(code) * scale.  sel as in tree_attn."""
    B, T, Hq, Hkv, D = w["B"], w["T"], w["Hq"], w["Hkv"], w["head_dim"]
    if q_rot is None:
        q_rot, _ = rotate_inputs(w)
    full = sel is None
    if full:
        bb, ii, hh = np.meshgrid(np.arange(B), np.arange(T), np.arange(Hq), indexing="ij")
        sel = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    sel = _i32(sel).reshape(-1, 3)
    out = np.empty((sel.shape[0], D), dtype=np.float64)
    scale = w.get("sm_scale") or 1.0 / np.sqrt(D)
    st = _load().or_tree_attn_e4m3(DTYPES[w["dtype"]], B, T, Hq, Hkv, D, w["page_size"], w["max_blocks"],
                                   w["num_pages"], _ptr(q_rot), _ptr(np.ascontiguousarray(k_codes, np.uint8)),
                                   _ptr(np.ascontiguousarray(v_codes, np.uint8)), float(k_scale),
                                   float(v_scale), _ptr(_i32(w["block_tables"])), _ptr(_i32(w["seq_lens"])),
                                   _ptr(_i32(w["tree_parents"])), float(scale), sel.shape[0], _ptr(sel),
                                   _ptr(out))
    _check(st, "tree_attn_e4m3")
    if full:
        return out.reshape(B, T, Hq, D)
    return out


def accept_greedy(tokens, logits: np.ndarray, logits_dtype: str, parents, max_depth: int):
    """Returns (argmax [B,T], accept_len [B], accept_path [B,max_depth+1], next_token [B])."""
    tokens = _i32(tokens)
    parents = _i32(parents)
    B, T = tokens.shape
    V = logits.shape[-1]
    logits = _act(logits, logits_dtype)
    am = np.empty((B, T), np.int32)
    alen = np.empty(B, np.int32)
    path = np.empty((B, max_depth + 1), np.int32)
    nxt = np.empty(B, np.int32)
    st = _load().or_accept_greedy(DTYPES[logits_dtype], B, T, V, max_depth, _ptr(tokens),
                                  _ptr(logits), _ptr(parents), _ptr(am), _ptr(alen), _ptr(path),
                                  _ptr(nxt))
    _check(st, "accept_greedy")
    return am, alen, path, nxt


def accept_typical(tokens, logits: np.ndarray, logits_dtype: str, parents, max_depth: int,
                   temperature: float, epsilon: float, delta: float):
    """Typical acceptance (see or_accept_typical for the reading).  Returns a dict:
    node_accept [B,T] int32 (each node's own test), prob and thr [B,T] float64
    (q[token] and min(epsilon, delta*exp(-H)) of the parent's row), accept_len [B],
    accept_path [B,max_depth+1], next_token [B], status."""
    tokens = _i32(tokens)
    parents = _i32(parents)
    B, T = tokens.shape
    V = logits.shape[-1]
    logits = _act(logits, logits_dtype)
    r = dict(node_accept=np.zeros((B, T), np.int32), prob=np.zeros((B, T)), thr=np.zeros((B, T)),
             accept_len=np.zeros(B, np.int32), accept_path=np.full((B, max_depth + 1), -1, np.int32),
             next_token=np.zeros(B, np.int32))
    r["status"] = _load().or_accept_typical(
        DTYPES[logits_dtype], B, T, V, max_depth, _ptr(tokens), _ptr(logits), _ptr(parents),
        float(temperature), float(epsilon), float(delta), _ptr(r["node_accept"]), _ptr(r["prob"]),
        _ptr(r["thr"]), _ptr(r["accept_len"]), _ptr(r["accept_path"]), _ptr(r["next_token"]))
    return r


def tree_candidates(root_logits: np.ndarray, head_logits: np.ndarray, logits_dtype: str, parents):
    """Returns (tokens [B,T], status): node 0 the argmax of root_logits[b], node i the
    rank-r entry of head_logits[b][depth_i - 1], r = number of earlier siblings."""
    parents = _i32(parents)
    B, T = parents.shape
    heads, V = head_logits.shape[1], head_logits.shape[2]
    root = _act(root_logits, logits_dtype)
    heads_a = _act(head_logits, logits_dtype)
    tokens = np.full((B, T), -1, np.int32)
    st = _load().or_tree_candidates(DTYPES[logits_dtype], B, T, heads, V, _ptr(root), _ptr(heads_a),
                                    _ptr(parents), _ptr(tokens))
    return tokens, st


def released_width(T: int, page_size: int) -> int:
    return (T + page_size - 1 + page_size - 1) // page_size


def kv_commit(w: dict, accept_path, accept_len, k_cache, v_cache, block_tables, seq_lens,
              max_depth: int, cache_dtype: str = None):
    """Returns the committed (k_cache, v_cache, block_tables, seq_lens, released_pages).
    cache_dtype: the cache's element type when it is not the act dtype ("e4m3")."""
    kc = np.ascontiguousarray(k_cache).copy()
    vc = np.ascontiguousarray(v_cache).copy()
    bt = _i32(block_tables).copy()
    sl = _i32(seq_lens).copy()
    width = released_width(w["T"], w["page_size"])
    rel = np.empty((w["B"], width), np.int32)
    st = _load().or_kv_commit(DTYPES[cache_dtype or w["dtype"]], w["B"], w["T"], w["Hkv"], w["head_dim"],
                              w["page_size"], w["max_blocks"], w["num_pages"], max_depth,
                              _ptr(_i32(accept_path)), _ptr(_i32(accept_len)), _ptr(kc), _ptr(vc),
                              _ptr(bt), _ptr(sl), _ptr(rel), width)
    _check(st, "kv_commit")
    return kc, vc, bt, sl, rel
