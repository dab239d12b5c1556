"""Host-side checks of the Python binding (no GPU): every call validates dtypes,
shapes and buffer sizes against one another, and refuses host tensors, before
anything reaches the library; the descriptor carries the FP8 cache fields.

A complete, consistent set of host tensors must fail only on the device check:
that shows the shape checks accept what the GPU tests and the bench pass."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import medusa_tree_speculative_attn_gb300 as mt
import workloads


def _attn_args(dtype=torch.bfloat16, fp8=False):
    spec = workloads.custom("bind", B=3, Hq=8, Hkv=2, head_dim=128, dtype="bf16",
                            prefix=("list", [0, 20, 37]), tree=("fanout", (3, 2), 7), max_depth=2)
    w = workloads.generate(spec, seed=0)
    B, T, Hq, Hkv, D = w["B"], w["T"], w["Hq"], w["Hkv"], w["head_dim"]
    cache_dt = torch.float8_e4m3fn if fp8 else dtype
    a = dict(q=torch.zeros((B, T, Hq, D), dtype=dtype),
             k_cache=torch.zeros(w["k_cache"].shape, dtype=cache_dt),
             v_cache=torch.zeros(w["v_cache"].shape, dtype=cache_dt),
             block_tables=torch.from_numpy(w["block_tables"]), seq_lens=torch.from_numpy(w["seq_lens"]),
             tree_parents=torch.from_numpy(w["tree_parents"]), tree_depths=torch.from_numpy(w["tree_depths"]),
             out=torch.zeros((B, T, Hq, D), dtype=dtype))
    kw = dict(k_new=torch.zeros((B, T, Hkv, D), dtype=dtype), v_new=torch.zeros((B, T, Hkv, D), dtype=dtype),
              rope=object(), workspace=torch.zeros(1 << 16, dtype=torch.uint8))
    return a, kw


def _call_attn(a, kw, **extra):
    mt.tree_attn_paged(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["seq_lens"],
                       a["tree_parents"], a["tree_depths"], a["out"], **kw, **extra)


@pytest.mark.parametrize("fp8", [False, True])
def test_attention_args_pass_every_check_but_the_device(fp8):
    a, kw = _attn_args(fp8=fp8)
    with pytest.raises(ValueError, match="CUDA device"):
        _call_attn(a, kw, k_scale=0.02, v_scale=0.03)


@pytest.mark.parametrize("key,bad", [
    ("out", lambda t: t[:, :-1]), ("seq_lens", lambda t: t[:-1]), ("tree_depths", lambda t: t[:, :-1]),
    ("tree_parents", lambda t: t[:-1]), ("block_tables", lambda t: t[:-1]),
    ("v_cache", lambda t: t[:-1]), ("k_new", lambda t: t[:, :, :1]), ("v_new", lambda t: t[:-1]),
])
def test_attention_shape_mismatches_are_refused(key, bad):
    a, kw = _attn_args()
    if key in a:
        a[key] = bad(a[key]).contiguous()
    else:
        kw[key] = bad(kw[key]).contiguous()
    with pytest.raises(ValueError, match=key):
        _call_attn(a, kw)


def test_attention_dtype_mismatches_are_refused():
    a, kw = _attn_args()
    a["v_cache"] = a["v_cache"].to(torch.float16)
    with pytest.raises(ValueError, match="v_cache"):
        _call_attn(a, kw)
    a, kw = _attn_args(fp8=True)
    a["v_cache"] = torch.zeros(a["v_cache"].shape, dtype=torch.bfloat16)   # K in FP8, V not
    with pytest.raises(ValueError, match="v_cache"):
        _call_attn(a, kw)


def test_descriptor_carries_the_fp8_cache():
    a, _ = _attn_args(fp8=True)
    d = mt.make_desc(a["q"], a["k_cache"], a["block_tables"], k_scale=0.02, v_scale=0.03)
    assert d.cache_dtype == mt.MT_E4M3 and d.dtype == 2
    assert d.k_scale == pytest.approx(0.02) and d.v_scale == pytest.approx(0.03)
    a, _ = _attn_args()
    assert mt.make_desc(a["q"], a["k_cache"], a["block_tables"]).cache_dtype == 0


def _accept_args(B=4, T=9, V=50, md=3):
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)
    return dict(tree_tokens=i32(B, T), target_logits=torch.zeros((B, T, V)), tree_parents=i32(B, T),
                accept_len=i32(B), accept_path=i32(B, md + 1)), dict(
        argmax_out=i32(B, T), next_token=i32(B), workspace=torch.zeros(4096, dtype=torch.uint8))


def test_acceptance_args_pass_every_check_but_the_device():
    pos, kw = _accept_args()
    with pytest.raises(ValueError, match="CUDA device"):
        mt.tree_accept_greedy(*pos.values(), **kw)
    kw_t = dict(kw)
    kw_t["node_accept"] = kw_t.pop("argmax_out")
    with pytest.raises(ValueError, match="CUDA device"):
        mt.tree_accept_typical(*pos.values(), **kw_t, temperature=1.0, epsilon=0.09, delta=0.3)


@pytest.mark.parametrize("key", ["target_logits", "tree_parents", "accept_len", "accept_path", "argmax_out",
                                 "next_token"])
def test_acceptance_shape_mismatches_are_refused(key):
    pos, kw = _accept_args()
    d = pos if key in pos else kw
    d[key] = d[key][:-1].contiguous()
    with pytest.raises(ValueError, match=key):
        mt.tree_accept_greedy(*pos.values(), **kw)


def test_typical_node_accept_shape_is_checked():
    pos, kw = _accept_args()
    kw["node_accept"] = kw.pop("argmax_out")[:, :-1].contiguous()
    with pytest.raises(ValueError, match="node_accept"):
        mt.tree_accept_typical(*pos.values(), **kw, temperature=1.0, epsilon=0.09, delta=0.3)


def _commit_args(fp8=False):
    a, _ = _attn_args(fp8=fp8)
    B, T = a["tree_parents"].shape
    P = a["k_cache"].shape[2]
    return dict(accept_path=torch.zeros((B, 3), dtype=torch.int32), accept_len=torch.zeros(B, dtype=torch.int32),
                k_cache=a["k_cache"], v_cache=a["v_cache"], block_tables=a["block_tables"],
                seq_lens=a["seq_lens"],
                released_pages=torch.zeros((B, mt.released_width(T, P)), dtype=torch.int32)), T


@pytest.mark.parametrize("fp8", [False, True])
def test_commit_args_pass_every_check_but_the_device(fp8):
    c, T = _commit_args(fp8)
    with pytest.raises(ValueError, match="CUDA device"):
        mt.kv_commit(*c.values(), tree_size=T, status_ws=torch.zeros(256, dtype=torch.uint8))
    B = c["block_tables"].shape[0]
    pos, kw = _accept_args(B=B, T=T, md=2)
    with pytest.raises(ValueError, match="CUDA device"):
        mt.tree_accept_commit(pos["tree_tokens"], pos["target_logits"], pos["tree_parents"], pos["accept_len"],
                              pos["accept_path"], c["k_cache"], c["v_cache"], c["block_tables"], c["seq_lens"],
                              c["released_pages"], **kw)


def test_commit_mismatches_are_refused():
    c, T = _commit_args()
    ws = torch.zeros(256, dtype=torch.uint8)
    for key in ("accept_len", "seq_lens", "accept_path", "released_pages", "v_cache"):
        bad = dict(c)
        bad[key] = c[key][:-1].contiguous()
        with pytest.raises(ValueError, match=key):
            mt.kv_commit(*bad.values(), tree_size=T, status_ws=ws)
    with pytest.raises(ValueError, match="status_ws"):
        mt.kv_commit(*c.values(), tree_size=T, status_ws=torch.zeros(64, dtype=torch.uint8))


def test_candidates_and_status_checks():
    B, heads, V, T = 2, 3, 40, 6
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)
    args = (torch.zeros((B, V)), torch.zeros((B, heads, V)), i32(B, T), i32(B, T))
    with pytest.raises(ValueError, match="CUDA device"):
        mt.tree_candidates(*args, status_ws=torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="status_ws"):
        mt.tree_candidates(*args, status_ws=torch.zeros(8, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA device"):
        mt.read_status(torch.zeros(256, dtype=torch.uint8))
