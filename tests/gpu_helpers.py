"""Helpers shared by the GPU tests: upload a workload, run the three calls
through the Python binding (which calls the C ABI), download the results."""
from __future__ import annotations

import numpy as np
import torch

import medusa_tree_speculative_attn_gb300 as mt
import workloads

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 1e-2}
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_dev(x, dtype: str, dev):
    """NumPy act array (bf16 as uint16 bits) -> device tensor of the act dtype."""
    a = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        a = a.view(torch.bfloat16)
    return a.to(dev)


def to_host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> NumPy (bf16 as uint16 bits)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def upload(w: dict, dev="cuda") -> dict:
    """Device copies of a NumPy-backend workload."""
    d = {}
    for k in ("q", "k_new", "v_new", "k_cache", "v_cache"):
        d[k] = to_dev(w[k], w["dtype"], dev)
    for k in ("block_tables", "seq_lens", "tree_parents", "tree_depths", "tree_tokens"):
        if k in w:
            d[k] = torch.from_numpy(np.ascontiguousarray(w[k])).to(dev)
    if "logits" in w:
        d["logits"] = to_dev(w["logits"], w["logits_dtype"], dev)
    return d


def device_inputs(w: dict) -> dict:
    """Device tensors of a workload of either backend."""
    if isinstance(w["q"], torch.Tensor):
        d = {k: w[k] for k in ("q", "k_new", "v_new", "k_cache", "v_cache", "block_tables",
                               "seq_lens", "tree_parents", "tree_depths") if k in w}
        for k in ("tree_tokens", "logits"):
            if k in w:
                d[k] = w[k]
        return d
    return upload(w)


class Step:
    """One verify step's buffers for a workload; run() calls the library."""

    def __init__(self, w: dict, kernel="auto", num_splits=0, dev="cuda"):
        self.w = w
        self.d = device_inputs(w)
        d = self.d
        self.rope = mt.Rope(w["rope_base"], w["head_dim"], int(np.max(_host(w, "seq_lens"))) + w["T"] + 1)
        self.desc = mt.make_desc(d["q"], d["k_cache"], d["block_tables"], num_splits, kernel)
        self.kernel, self.num_splits = kernel, num_splits
        self.k_scale = self.v_scale = 1.0   # FP8 caches only
        self.ws = mt.alloc_attn_workspace(self.desc, dev)
        self.out = torch.empty_like(d["q"])
        B, T = w["B"], w["T"]
        md = w["max_depth"]
        self.am = torch.empty((B, T), dtype=torch.int32, device=dev)
        self.alen = torch.empty(B, dtype=torch.int32, device=dev)
        self.path = torch.empty((B, md + 1), dtype=torch.int32, device=dev)
        self.nxt = torch.empty(B, dtype=torch.int32, device=dev)
        self.aws = mt.alloc_accept_workspace(B, T, dev)
        self.rel = torch.empty((B, mt.released_width(T, w["page_size"])), dtype=torch.int32, device=dev)

    def attn(self):
        d = self.d
        mt.tree_attn_paged(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["seq_lens"],
                           d["tree_parents"], d["tree_depths"], self.out, k_new=d["k_new"],
                           v_new=d["v_new"], rope=self.rope, workspace=self.ws,
                           num_splits=self.num_splits, kernel=self.kernel, k_scale=self.k_scale,
                           v_scale=self.v_scale)

    def accept(self):
        d = self.d
        mt.tree_accept_greedy(d["tree_tokens"], d["logits"], d["tree_parents"], self.alen, self.path,
                              argmax_out=self.am, next_token=self.nxt, workspace=self.aws)

    def commit(self):
        d = self.d
        mt.kv_commit(self.path, self.alen, d["k_cache"], d["v_cache"], d["block_tables"],
                     d["seq_lens"], self.rel, tree_size=self.w["T"], status_ws=self.ws)

    def accept_commit(self):
        d = self.d
        mt.tree_accept_commit(d["tree_tokens"], d["logits"], d["tree_parents"], self.alen, self.path,
                              d["k_cache"], d["v_cache"], d["block_tables"], d["seq_lens"], self.rel,
                              argmax_out=self.am, next_token=self.nxt, workspace=self.aws)

    def status(self):
        return mt.read_status(self.ws), mt.read_status(self.aws)


def _host(w, key):
    v = w.get(key + "_host", w[key])
    return v.cpu().numpy() if isinstance(v, torch.Tensor) else v
