"""Seeded synthetic inputs for the Medusa tree-verification step.

This module only draws inputs: speculation trees, page pools and block tables,
N(0,1) activations, logits with planted matches.  It holds none of the
method's arithmetic (no RoPE, no attention, no argmax, no commit), so the CUDA
path and the CPU oracle can both be fed from it without sharing any code.

Shapes follow the pages' workloads (Medusa on 7B/13B/70B LLaMA-class models,
64-choice trees; lmdeploy PR 1231 "[WIP] support Medusa" and the TensorRT-LLM /
vLLM threads); there is no dataset or checkpoint here, so the values are seeded
random draws:

  tiny_tree_fp32      batch 1, 1 head, D 64, fp32, prefix 128 in 8 shuffled
                      pages, 7-node tree, vocab 1000 fp32 logits
  llama7b_b1_fp16     batch 1, 32/32 heads, D 128, fp16, prefix 2048, 64-node
                      tree from top-k fanouts (10,5,3,2), fp32 logits vocab
                      32000, planted path length uniform in 0..4
  serve_b16_gqa_bf16  batch 16, 32 q / 8 kv heads, D 128, bf16, prefixes
                      uniform in [512, 8192], 64-node trees (depth <= 5),
                      bf16 logits vocab 32000, planted geometric(0.4) paths
  llama70b_32k_b8_bf16  batch 8, 64 q / 8 kv heads, D 128, bf16, prefix 32768,
                      26-node trees from fanouts (3,2,2,1); attention only
  verify_b64_fp16     batch 64, 32/32 heads, D 128, fp16, prefixes uniform in
                      [256, 4096], 32-node trees (depth <= 4), fp16 logits
                      vocab 32000, planted geometric(0.4) paths

Arrays are NumPy (``backend="numpy"``; bf16 as uint16 bit patterns, obtained
by truncating float32 draws) or torch tensors on a device (``backend="torch"``).
The structural parts (trees, tokens, tables, lengths, planted paths) always
come from the same NumPy generator, so both backends share them exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np

PLANT_LOGIT = 10.0  # far above the largest of 32000 N(0,1) draws


@dataclass(frozen=True)
class Spec:
    name: str
    B: int
    Hq: int
    Hkv: int
    head_dim: int
    dtype: str                      # "f32" | "f16" | "bf16"
    prefix: tuple                   # ("fixed", L) or ("uniform", lo, hi)
    tree: tuple                     # ("fixed", parents) | ("fanout", caps, n_nodes)
    max_depth: int
    page_size: int = 16
    rope_base: float = 10000.0
    vocab: Optional[int] = None     # None: no acceptance inputs
    logits_dtype: Optional[str] = None
    plant: tuple = ("none",)        # ("uniform", lo, hi) | ("geometric", p) | ("none",)
    poison_pages: int = 2
    description: str = ""


TINY_TREE_PARENTS = (-1, 0, 0, 1, 2, 3, 3)

SPECS = {
    "tiny_tree_fp32": Spec(
        "tiny_tree_fp32", B=1, Hq=1, Hkv=1, head_dim=64, dtype="f32", prefix=("fixed", 128),
        tree=("fixed", TINY_TREE_PARENTS), max_depth=3, vocab=1000, logits_dtype="f32",
        plant=("uniform", 0, 3),
        description="batch 1, 1 head, D 64, fp32, prefix 128, 7-node tree, vocab 1000"),
    "llama7b_b1_fp16": Spec(
        "llama7b_b1_fp16", B=1, Hq=32, Hkv=32, head_dim=128, dtype="f16", prefix=("fixed", 2048),
        tree=("fanout", (10, 5, 3, 2), 64), max_depth=4, vocab=32000, logits_dtype="f32",
        plant=("uniform", 0, 4),
        description="7B-class batch-1 verify: 32 heads, D 128, fp16, prefix 2048, 64-node tree"),
    "serve_b16_gqa_bf16": Spec(
        "serve_b16_gqa_bf16", B=16, Hq=32, Hkv=8, head_dim=128, dtype="bf16",
        prefix=("uniform", 512, 8192), tree=("fanout", (10, 5, 3, 2, 2), 64), max_depth=5,
        vocab=32000, logits_dtype="bf16", plant=("geometric", 0.4),
        description="serving batch 16, GQA 32/8, D 128, bf16, prefixes U[512,8192], 64-node trees"),
    "llama70b_32k_b8_bf16": Spec(
        "llama70b_32k_b8_bf16", B=8, Hq=64, Hkv=8, head_dim=128, dtype="bf16",
        prefix=("fixed", 32768), tree=("fanout", (3, 2, 2, 1), 26), max_depth=4,
        description="70B-class long context: batch 8, GQA 64/8, D 128, bf16, prefix 32768, 26-node trees"),
    "verify_b64_fp16": Spec(
        "verify_b64_fp16", B=64, Hq=32, Hkv=32, head_dim=128, dtype="f16",
        prefix=("uniform", 256, 4096), tree=("fanout", (10, 5, 3, 2), 32), max_depth=4,
        vocab=32000, logits_dtype="f16", plant=("geometric", 0.4),
        description="high-batch verify: batch 64, 32 heads, D 128, fp16, prefixes U[256,4096], 32-node trees"),
}


def custom(name="custom", **kw) -> Spec:
    """A spec with arbitrary sizes (randomised parity cases)."""
    base = dict(B=1, Hq=1, Hkv=1, head_dim=64, dtype="f32", prefix=("fixed", 16),
                tree=("fanout", (2, 2), 5), max_depth=2)
    base.update(kw)
    return Spec(name, **base)


# ---------------------------------------------------------------------------
# Trees
# ---------------------------------------------------------------------------

def fanout_tree(rng: np.random.Generator, caps: Sequence[int], n_nodes: int):
    """A Medusa candidate tree: node at depth d has up to caps[d] children (the
    top-k of the depth-(d+1) head); n_nodes of the full tree are kept by seeded
    ancestor-closed frontier sampling.  Returns (parents, depths, rank paths)
    in depth-major order, so every parent precedes its children."""
    full = 1
    width = 1
    for c in caps:
        width *= c
        full += width
    if n_nodes > full:
        raise ValueError(f"a tree with fanouts {tuple(caps)} has only {full} nodes")
    chosen = [()]
    frontier = [(r,) for r in range(caps[0])] if caps else []
    while len(chosen) < n_nodes:
        k = int(rng.integers(len(frontier)))
        node = frontier.pop(k)
        chosen.append(node)
        if len(node) < len(caps):
            frontier.extend(node + (r,) for r in range(caps[len(node)]))
    chosen.sort(key=lambda p: (len(p), p))
    index = {p: i for i, p in enumerate(chosen)}
    parents = np.array([-1] + [index[p[:-1]] for p in chosen[1:]], dtype=np.int32)
    depths = np.array([len(p) for p in chosen], dtype=np.int32)
    return parents, depths, chosen


def depths_of(parents) -> np.ndarray:
    parents = np.asarray(parents)
    d = np.zeros(len(parents), dtype=np.int32)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def chain_tree(n: int):
    parents = np.arange(-1, n - 1, dtype=np.int32)
    return parents, np.arange(n, dtype=np.int32)


def star_tree(n: int):
    parents = np.zeros(n, dtype=np.int32)
    parents[0] = -1
    depths = np.ones(n, dtype=np.int32)
    depths[0] = 0
    return parents, depths


def tree_tokens(rng: np.random.Generator, parents: np.ndarray, vocab: int) -> np.ndarray:
    """Token of every node; siblings get distinct tokens (top-k of one head)."""
    T = len(parents)
    tok = np.zeros(T, dtype=np.int32)
    tok[0] = rng.integers(vocab)
    children = {}
    for i in range(1, T):
        children.setdefault(int(parents[i]), []).append(i)
    for p, kids in children.items():
        draw = rng.choice(vocab, size=len(kids), replace=len(kids) > vocab)
        tok[kids] = draw
    return tok


# ---------------------------------------------------------------------------
# Whole workloads
# ---------------------------------------------------------------------------

def _prefix_lengths(rng, spec: Spec) -> np.ndarray:
    kind = spec.prefix[0]
    if kind == "fixed":
        return np.full(spec.B, spec.prefix[1], dtype=np.int32)
    if kind == "uniform":
        return rng.integers(spec.prefix[1], spec.prefix[2] + 1, size=spec.B).astype(np.int32)
    if kind == "list":
        return np.asarray(spec.prefix[1], dtype=np.int32)
    raise ValueError(kind)


def _trees(rng, spec: Spec):
    kind = spec.tree[0]
    if kind == "fixed":
        p = np.asarray(spec.tree[1], dtype=np.int32)
        par = np.tile(p, (spec.B, 1))
        dep = np.tile(depths_of(p), (spec.B, 1))
        return par, dep
    if kind == "fanout":
        caps, n = spec.tree[1], spec.tree[2]
        pars, deps = [], []
        for _ in range(spec.B):
            p, d, _ = fanout_tree(rng, caps, n)
            pars.append(p)
            deps.append(d)
        return np.stack(pars), np.stack(deps)
    if kind == "chain":
        p, d = chain_tree(spec.tree[1])
        return np.tile(p, (spec.B, 1)), np.tile(d, (spec.B, 1))
    if kind == "star":
        p, d = star_tree(spec.tree[1])
        return np.tile(p, (spec.B, 1)), np.tile(d, (spec.B, 1))
    if kind == "list":
        par = np.asarray(spec.tree[1], dtype=np.int32)
        return par, np.stack([depths_of(p) for p in par])
    raise ValueError(kind)


def _planted_lengths(rng, spec: Spec) -> np.ndarray:
    kind = spec.plant[0]
    if kind == "none":
        return np.zeros(spec.B, dtype=np.int32)
    if kind == "uniform":
        return rng.integers(spec.plant[1], spec.plant[2] + 1, size=spec.B).astype(np.int32)
    if kind == "geometric":
        g = rng.geometric(spec.plant[1], size=spec.B)      # >= 1
        return np.minimum(g - 1, spec.max_depth).astype(np.int32)
    raise ValueError(kind)


def _page_layout(rng, spec: Spec, seq_lens: np.ndarray, T: int):
    P = spec.page_size
    need = (seq_lens.astype(np.int64) + T + P - 1) // P
    num_pages = int(need.sum()) + spec.poison_pages
    max_blocks = int(need.max())
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((spec.B, max_blocks), -1, dtype=np.int32)
    cursor = 0
    for b in range(spec.B):
        n = int(need[b])
        bt[b, :n] = perm[cursor:cursor + n]
        cursor += n
    return bt, num_pages, max_blocks


def _prefix_slot_mask(spec: Spec, bt, seq_lens, num_pages):
    """[num_pages, P] True where a page slot holds a committed prefix token."""
    P = spec.page_size
    mask = np.zeros((num_pages, P), dtype=bool)
    for b in range(spec.B):
        L = int(seq_lens[b])
        full = L // P
        pages = bt[b, :full]
        mask[pages] = True
        if L % P:
            mask[bt[b, full], : L % P] = True
    return mask


_NP_ACT = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
_POISON_BITS = {"f32": 0x7FC00001, "f16": 0x7E01, "bf16": 0x7FC1}   # quiet NaNs


def _np_normal(rng, shape, dtype: str):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    return (x.view(np.uint32) >> 16).astype(np.uint16)     # bf16 by truncation


def _poison_value(dtype: str):
    if dtype == "f32":
        return np.array([_POISON_BITS["f32"]], dtype=np.uint32).view(np.float32)[0]
    if dtype == "f16":
        return np.array([_POISON_BITS["f16"]], dtype=np.uint16).view(np.float16)[0]
    return np.uint16(_POISON_BITS["bf16"])


def generate(spec, seed: int = 0, backend: str = "numpy", device: str = "cuda",
             with_logits: bool = True) -> dict:
    """Draw one workload.  Returns a dict of sizes and arrays (see module doc)."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    rng = np.random.default_rng(seed)
    seq_lens = _prefix_lengths(rng, spec)
    parents, depths = _trees(rng, spec)
    T = parents.shape[1]
    bt, num_pages, max_blocks = _page_layout(rng, spec, seq_lens, T)
    w = dict(name=spec.name, spec=spec, B=spec.B, T=T, Hq=spec.Hq, Hkv=spec.Hkv,
             head_dim=spec.head_dim, dtype=spec.dtype, page_size=spec.page_size,
             rope_base=spec.rope_base, sm_scale=None, max_depth=spec.max_depth,
             seq_lens=seq_lens, tree_parents=parents, tree_depths=depths, block_tables=bt,
             num_pages=num_pages, max_blocks=max_blocks)
    # acceptance inputs: tokens and planted paths are structural (NumPy)
    planted_nodes = []
    if spec.vocab is not None and with_logits:
        V = spec.vocab
        tokens = np.stack([tree_tokens(rng, parents[b], V) for b in range(spec.B)])
        plant_len = _planted_lengths(rng, spec)
        for b in range(spec.B):
            want = int(plant_len[b])
            cand = np.nonzero(depths[b] == min(want, int(depths[b].max())))[0]
            end = int(cand[rng.integers(len(cand))])
            path = []
            a = end
            while a > 0:
                path.append(a)
                a = int(parents[b, a])
            planted_nodes.append(path[::-1])
        w.update(vocab=V, logits_dtype=spec.logits_dtype, tree_tokens=tokens,
                 planted_len=plant_len, planted_nodes=planted_nodes)
    shapes = dict(q=(spec.B, T, spec.Hq, spec.head_dim),
                  k_new=(spec.B, T, spec.Hkv, spec.head_dim),
                  v_new=(spec.B, T, spec.Hkv, spec.head_dim),
                  cache=(num_pages, spec.Hkv, spec.page_size, spec.head_dim))
    mask = _prefix_slot_mask(spec, bt, seq_lens, num_pages)
    bulk_seed = int(rng.integers(2**62))
    if backend == "numpy":
        brng = np.random.default_rng(bulk_seed)
        for key in ("q", "k_new", "v_new"):
            w[key] = _np_normal(brng, shapes[key], spec.dtype)
        for key in ("k_cache", "v_cache"):
            c = _np_normal(brng, shapes["cache"], spec.dtype)
            c.transpose(0, 2, 1, 3)[~mask] = _poison_value(spec.dtype)
            w[key] = c
        if "vocab" in w:
            lg = _np_normal(brng, (spec.B, T, w["vocab"]), w["logits_dtype"])
            _plant_numpy(lg, w)
            w["logits"] = lg
    elif backend == "torch":
        import torch
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
        gen = torch.Generator(device=device)
        gen.manual_seed(bulk_seed)
        for key in ("q", "k_new", "v_new"):
            w[key] = torch.randn(shapes[key], generator=gen, device=device,
                                 dtype=torch.float32).to(tdt[spec.dtype])
        tmask = torch.from_numpy(~mask).to(device)
        for key in ("k_cache", "v_cache"):
            c = torch.empty(shapes["cache"], device=device, dtype=tdt[spec.dtype])
            # draw in page chunks to bound the fp32 temporary
            step = max(1, (1 << 27) // max(1, spec.Hkv * spec.page_size * spec.head_dim))
            for p0 in range(0, num_pages, step):
                p1 = min(num_pages, p0 + step)
                c[p0:p1] = torch.randn((p1 - p0,) + shapes["cache"][1:], generator=gen,
                                       device=device, dtype=torch.float32).to(tdt[spec.dtype])
            c.transpose(1, 2)[tmask] = float("nan")
            w[key] = c
        if "vocab" in w:
            lg = torch.randn((spec.B, T, w["vocab"]), generator=gen, device=device,
                             dtype=torch.float32).to(tdt[w["logits_dtype"]])
            for b, path in enumerate(w["planted_nodes"]):
                for node in path:
                    lg[b, int(parents[b, node]), int(w["tree_tokens"][b, node])] = PLANT_LOGIT
            w["logits"] = lg
        for key in ("seq_lens", "tree_parents", "tree_depths", "block_tables"):
            w[key + "_host"] = w[key]
            w[key] = torch.from_numpy(np.ascontiguousarray(w[key])).to(device)
        if "tree_tokens" in w:
            w["tree_tokens_host"] = w["tree_tokens"]
            w["tree_tokens"] = torch.from_numpy(w["tree_tokens"]).to(device)
    else:
        raise ValueError(backend)
    return w


def _plant_numpy(lg: np.ndarray, w: dict):
    dt = w["logits_dtype"]
    if dt == "bf16":
        val = np.uint16(np.array([PLANT_LOGIT], np.float32).view(np.uint32)[0] >> 16)
    else:
        val = PLANT_LOGIT
    for b, path in enumerate(w["planted_nodes"]):
        for node in path:
            lg[b, int(w["tree_parents"][b, node]), int(w["tree_tokens"][b, node])] = val


def to_numpy(w: dict) -> dict:
    """A NumPy copy of a torch-backend workload (bf16 as uint16 bits)."""
    import torch
    out = {}
    for k, v in w.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu()
            if t.dtype == torch.bfloat16:
                out[k] = t.view(torch.int16).numpy().view(np.uint16)
            else:
                out[k] = t.numpy()
        else:
            out[k] = v
    for k in ("seq_lens", "tree_parents", "tree_depths", "block_tables", "tree_tokens"):
        if k + "_host" in w:
            out[k] = w[k + "_host"]
    return out
