"""Medusa tree-verification step for NVIDIA GB300 (sm_103a).

A thin ctypes binding over ``lib/libmedusa_tree.so`` (C ABI in
``include/medusa_tree.h``).  Python only marshals arguments: every step of the
path (RoPE, tree mask, attention, combine, argmax, acceptance, commit) runs in
the library's CUDA kernels.  PyTorch supplies device memory and the stream.
There is no CPU fallback: if the library is missing this module raises.

Calls (same names as the C ABI without the ``mt_`` prefix):
  tree_attn_paged    tree tokens attend to the paged prefix + their ancestors
  tree_accept_greedy per-node argmax and the longest matching root path
  kv_commit          move accepted K/V into place, grow lengths, release pages
  tree_accept_commit the last two in one launch
  tree_candidates    the tree's tokens from the base and Medusa-head logits
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmedusa_tree.so")

MT_OK = 0
KERNELS = {"auto": 0, "simt": 1, "tc": 2}
_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
MT_E4M3 = 3  # cache element type: OCP FP8 E4M3 codes (torch.float8_e4m3fn)


class MedusaTreeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status} ({status_string(status)})")


class AttnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("tree_size", ctypes.c_int),
                ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("page_size", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("num_splits", ctypes.c_int), ("dtype", ctypes.c_int),
                ("sm_scale", ctypes.c_float), ("kernel", ctypes.c_int),
                ("cache_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                               "(there is no fallback path)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        D = ctypes.POINTER(AttnDesc)
        lib.mt_version.restype = I
        lib.mt_status_string.argtypes = [I]
        lib.mt_status_string.restype = ctypes.c_char_p
        lib.mt_rope_create.argtypes = [ctypes.c_double, I, I, ctypes.POINTER(P)]
        lib.mt_rope_destroy.argtypes = [P]
        lib.mt_tree_attn_workspace_size.argtypes = [D]
        lib.mt_tree_attn_workspace_size.restype = Z
        lib.mt_tree_attn_paged.argtypes = [D] + [P] * 12 + [Z, P]
        lib.mt_tree_accept_workspace_size.argtypes = [I, I]
        lib.mt_tree_accept_workspace_size.restype = Z
        lib.mt_tree_accept_greedy.argtypes = [I, I, I, I, I] + [P] * 8 + [Z, P]
        lib.mt_tree_accept_typical.argtypes = ([I, I, I, I, I] + [P] * 3 + [ctypes.c_float] * 3 +
                                               [P] * 5 + [Z, P])
        lib.mt_kv_commit.argtypes = [D, I] + [P] * 8 + [P]
        lib.mt_tree_accept_commit.argtypes = [D, I, I, I] + [P] * 12 + [P, Z, P]
        lib.mt_tree_candidates.argtypes = [I, I, I, I, I] + [P] * 5 + [P]
        lib.mt_read_status.argtypes = [P, P, ctypes.POINTER(I)]
        lib.mt_profile_enable.argtypes = [I]
        lib.mt_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float), I, ctypes.POINTER(I)]
        lib.mt_debug_set_wait.argtypes = [ctypes.c_ulonglong, I]
        _lib = lib
    return _lib


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def status_string(status: int) -> str:
    return _load().mt_status_string(int(status)).decode()


def _check(st: int, what: str):
    if st != MT_OK:
        raise MedusaTreeError(st, what)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _shape(t: torch.Tensor, name: str, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _min_bytes(t: torch.Tensor, name: str, n: int):
    if t.numel() * t.element_size() < n:
        raise ValueError(f"{name} must hold at least {n} bytes")


def _on_device(**tensors):
    """Every tensor on the first one's CUDA device: the kernels dereference the
    pointers as device memory, so a host tensor must never reach them."""
    dev = None
    for name, t in tensors.items():
        if not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {dev}")


class Rope:
    """Library-owned fp32 cos/sin table on the current device."""

    def __init__(self, base: float, head_dim: int, max_pos: int):
        self._lib = _load()
        self.handle = ctypes.c_void_p()
        _check(self._lib.mt_rope_create(float(base), int(head_dim), int(max_pos),
                                        ctypes.byref(self.handle)), "mt_rope_create")
        self.base, self.head_dim, self.max_pos = base, head_dim, max_pos

    def __del__(self):
        if getattr(self, "handle", None) and self.handle.value:
            self._lib.mt_rope_destroy(self.handle)
            self.handle = ctypes.c_void_p()


def _fp8(cache: torch.Tensor) -> bool:
    return cache.dtype == torch.float8_e4m3fn


def make_desc(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
              num_splits: int = 0, kernel: str = "auto", sm_scale: float = 0.0,
              k_scale: float = 1.0, v_scale: float = 1.0) -> AttnDesc:
    """The call's descriptor; an FP8 E4M3 cache (torch.float8_e4m3fn) holds the
    codes of value / k_scale (keys) and value / v_scale (values)."""
    B, T, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("q and k_cache head_dim differ")
    return AttnDesc(B, T, Hq, Hkv, D, P, block_tables.shape[1], num_pages, int(num_splits),
                    _DTYPES[q.dtype], float(sm_scale), KERNELS[kernel],
                    MT_E4M3 if _fp8(k_cache) else 0, float(k_scale), float(v_scale))


def _commit_desc(B: int, T: int, k_cache: torch.Tensor, max_blocks: int) -> AttnDesc:
    num_pages, Hkv, P, D = k_cache.shape
    if _fp8(k_cache):   # the act dtype does not matter to a commit: bytes move as they are
        return AttnDesc(B, T, Hkv, Hkv, D, P, max_blocks, num_pages, 0, _DTYPES[torch.bfloat16],
                        0.0, 0, MT_E4M3, 1.0, 1.0)
    return AttnDesc(B, T, Hkv, Hkv, D, P, max_blocks, num_pages, 0, _DTYPES[k_cache.dtype], 0.0, 0,
                    0, 1.0, 1.0)


def attn_workspace_size(desc: AttnDesc) -> int:
    return int(_load().mt_tree_attn_workspace_size(ctypes.byref(desc)))


def alloc_attn_workspace(desc: AttnDesc, device="cuda") -> torch.Tensor:
    n = attn_workspace_size(desc)
    if n == 0:
        raise MedusaTreeError(-1, "mt_tree_attn_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def accept_workspace_size(batch: int, tree_size: int) -> int:
    return int(_load().mt_tree_accept_workspace_size(int(batch), int(tree_size)))


def alloc_accept_workspace(batch: int, tree_size: int, device="cuda") -> torch.Tensor:
    return torch.zeros(accept_workspace_size(batch, tree_size), dtype=torch.uint8, device=device)


def tree_attn_paged(q, k_cache, v_cache, block_tables, seq_lens, tree_parents, tree_depths, out, *,
                    k_new, v_new, rope: Rope, workspace: torch.Tensor, num_splits: int = 0,
                    kernel: str = "auto", sm_scale: float = 0.0, k_scale: float = 1.0,
                    v_scale: float = 1.0, stream=None):
    """out[b,i,h] = attention of tree node i (head h) over the prefix + its ancestors.

    The caches hold q's dtype, or FP8 E4M3 codes (torch.float8_e4m3fn) of
    value / k_scale and value / v_scale (read on either kernel; the tensor-core
    kernel converts the codes to q's dtype in shared memory)."""
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("out", out)):
        _need(t, name, q.dtype, 4)
    cache_dtype = torch.float8_e4m3fn if _fp8(k_cache) else q.dtype
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, cache_dtype, 4)
    for name, t in (("block_tables", block_tables), ("tree_parents", tree_parents),
                    ("tree_depths", tree_depths)):
        _need(t, name, torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(workspace, "workspace")
    B, T, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _shape(t, name, (B, T, Hkv, D))
    _shape(out, "out", q.shape)
    _shape(v_cache, "v_cache", k_cache.shape)
    _shape(seq_lens, "seq_lens", (B,))
    if block_tables.shape[0] != B:
        raise ValueError("block_tables must have one row per sequence")
    for name, t in (("tree_parents", tree_parents), ("tree_depths", tree_depths)):
        _shape(t, name, (B, T))
    desc = make_desc(q, k_cache, block_tables, num_splits, kernel, sm_scale, k_scale, v_scale)
    _on_device(q=q, k_new=k_new, v_new=v_new, out=out, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, seq_lens=seq_lens, tree_parents=tree_parents,
               tree_depths=tree_depths, workspace=workspace)
    st = _load().mt_tree_attn_paged(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new),
                                    _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                    _ptr(seq_lens), _ptr(tree_parents), _ptr(tree_depths),
                                    rope.handle, _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "mt_tree_attn_paged")
    return out


def tree_accept_greedy(tree_tokens, target_logits, tree_parents, accept_len, accept_path, *,
                       argmax_out, next_token, workspace: torch.Tensor, max_depth: Optional[int] = None,
                       stream=None):
    """Greedy acceptance; fills argmax_out, accept_len, accept_path, next_token."""
    _need(tree_tokens, "tree_tokens", torch.int32, 2)
    _need(tree_parents, "tree_parents", torch.int32, 2)
    _need(target_logits, "target_logits", None, 3)
    for name, t in (("accept_len", accept_len), ("next_token", next_token)):
        _need(t, name, torch.int32, 1)
    _need(accept_path, "accept_path", torch.int32, 2)
    _need(argmax_out, "argmax_out", torch.int32, 2)
    _need(workspace, "workspace")
    B, T = tree_tokens.shape
    V = target_logits.shape[2]
    if max_depth is None:
        max_depth = accept_path.shape[1] - 1
    if accept_path.shape[1] != max_depth + 1:
        raise ValueError("accept_path must have max_depth + 1 columns")
    _accept_shapes(B, T, V, target_logits, tree_parents, accept_len, accept_path, next_token,
                   argmax_out=argmax_out)
    _on_device(tree_tokens=tree_tokens, target_logits=target_logits, tree_parents=tree_parents,
               argmax_out=argmax_out, accept_len=accept_len, accept_path=accept_path,
               next_token=next_token, workspace=workspace)
    st = _load().mt_tree_accept_greedy(B, T, V, int(max_depth), _DTYPES[target_logits.dtype],
                                       _ptr(tree_tokens), _ptr(target_logits), _ptr(tree_parents),
                                       _ptr(argmax_out), _ptr(accept_len), _ptr(accept_path),
                                       _ptr(next_token), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "mt_tree_accept_greedy")
    return accept_len, accept_path


def _accept_shapes(B, T, V, target_logits, tree_parents, accept_len, accept_path, next_token, **per_node):
    _shape(target_logits, "target_logits", (B, T, V))
    _shape(tree_parents, "tree_parents", (B, T))
    _shape(accept_len, "accept_len", (B,))
    _shape(next_token, "next_token", (B,))
    if accept_path.shape[0] != B:
        raise ValueError("accept_path must have one row per sequence")
    for name, t in per_node.items():
        _shape(t, name, (B, T))


def tree_accept_typical(tree_tokens, target_logits, tree_parents, accept_len, accept_path, *,
                        node_accept, next_token, workspace: torch.Tensor, temperature: float,
                        epsilon: float, delta: float, max_depth: Optional[int] = None, stream=None):
    """Typical acceptance: node i passes when its token's probability under its
    parent's tempered row exceeds min(epsilon, delta * exp(-entropy)); fills
    node_accept, accept_len, accept_path, next_token (the end row's argmax)."""
    _need(tree_tokens, "tree_tokens", torch.int32, 2)
    _need(tree_parents, "tree_parents", torch.int32, 2)
    _need(target_logits, "target_logits", None, 3)
    for name, t in (("accept_len", accept_len), ("next_token", next_token)):
        _need(t, name, torch.int32, 1)
    _need(accept_path, "accept_path", torch.int32, 2)
    _need(node_accept, "node_accept", torch.int32, 2)
    _need(workspace, "workspace")
    B, T = tree_tokens.shape
    V = target_logits.shape[2]
    if max_depth is None:
        max_depth = accept_path.shape[1] - 1
    if accept_path.shape[1] != max_depth + 1:
        raise ValueError("accept_path must have max_depth + 1 columns")
    _accept_shapes(B, T, V, target_logits, tree_parents, accept_len, accept_path, next_token,
                   node_accept=node_accept)
    _on_device(tree_tokens=tree_tokens, target_logits=target_logits, tree_parents=tree_parents,
               node_accept=node_accept, accept_len=accept_len, accept_path=accept_path,
               next_token=next_token, workspace=workspace)
    st = _load().mt_tree_accept_typical(B, T, V, int(max_depth), _DTYPES[target_logits.dtype],
                                        _ptr(tree_tokens), _ptr(target_logits), _ptr(tree_parents),
                                        float(temperature), float(epsilon), float(delta),
                                        _ptr(node_accept), _ptr(accept_len), _ptr(accept_path),
                                        _ptr(next_token), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "mt_tree_accept_typical")
    return accept_len, accept_path


def released_width(tree_size: int, page_size: int) -> int:
    return (tree_size + 2 * page_size - 2) // page_size


def kv_commit(accept_path, accept_len, k_cache, v_cache, block_tables, seq_lens, released_pages, *,
              tree_size: int, status_ws: torch.Tensor, stream=None):
    """Commit accepted K/V, grow seq_lens, release scratch pages (in place)."""
    _need(accept_path, "accept_path", torch.int32, 2)
    _need(accept_len, "accept_len", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(released_pages, "released_pages", torch.int32, 2)
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4)
    _need(status_ws, "status_ws")
    P = k_cache.shape[2]
    B = block_tables.shape[0]
    if released_pages.shape != (B, released_width(tree_size, P)):
        raise ValueError("released_pages must be [B, (T + 2P - 2) // P]")
    _shape(v_cache, "v_cache", k_cache.shape)
    _shape(accept_len, "accept_len", (B,))
    _shape(seq_lens, "seq_lens", (B,))
    if accept_path.shape[0] != B:
        raise ValueError("accept_path must have one row per sequence")
    _min_bytes(status_ws, "status_ws", 256)
    desc = _commit_desc(B, int(tree_size), k_cache, block_tables.shape[1])
    _on_device(accept_path=accept_path, accept_len=accept_len, k_cache=k_cache, v_cache=v_cache,
               block_tables=block_tables, seq_lens=seq_lens, released_pages=released_pages,
               status_ws=status_ws)
    st = _load().mt_kv_commit(ctypes.byref(desc), accept_path.shape[1] - 1, _ptr(accept_path),
                              _ptr(accept_len), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                              _ptr(seq_lens), _ptr(released_pages), _ptr(status_ws), _stream(stream))
    _check(st, "mt_kv_commit")


def tree_accept_commit(tree_tokens, target_logits, tree_parents, accept_len, accept_path, k_cache,
                       v_cache, block_tables, seq_lens, released_pages, *, argmax_out, next_token,
                       workspace: torch.Tensor, max_depth: Optional[int] = None, stream=None):
    """tree_accept_greedy followed by kv_commit, in one launch (same results)."""
    _need(tree_tokens, "tree_tokens", torch.int32, 2)
    _need(tree_parents, "tree_parents", torch.int32, 2)
    _need(target_logits, "target_logits", None, 3)
    for name, t in (("accept_len", accept_len), ("next_token", next_token), ("seq_lens", seq_lens)):
        _need(t, name, torch.int32, 1)
    for name, t in (("accept_path", accept_path), ("argmax_out", argmax_out),
                    ("block_tables", block_tables), ("released_pages", released_pages)):
        _need(t, name, torch.int32, 2)
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4)
    _need(workspace, "workspace")
    B, T = tree_tokens.shape
    V = target_logits.shape[2]
    if max_depth is None:
        max_depth = accept_path.shape[1] - 1
    if accept_path.shape[1] != max_depth + 1:
        raise ValueError("accept_path must have max_depth + 1 columns")
    P = k_cache.shape[2]
    if released_pages.shape != (B, released_width(T, P)):
        raise ValueError("released_pages must be [B, (T + 2P - 2) // P]")
    _accept_shapes(B, T, V, target_logits, tree_parents, accept_len, accept_path, next_token,
                   argmax_out=argmax_out)
    _shape(v_cache, "v_cache", k_cache.shape)
    _shape(seq_lens, "seq_lens", (B,))
    if block_tables.shape[0] != B:
        raise ValueError("block_tables must have one row per sequence")
    desc = _commit_desc(B, int(T), k_cache, block_tables.shape[1])
    _on_device(tree_tokens=tree_tokens, target_logits=target_logits, tree_parents=tree_parents,
               argmax_out=argmax_out, accept_len=accept_len, accept_path=accept_path,
               next_token=next_token, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               seq_lens=seq_lens, released_pages=released_pages, workspace=workspace)
    st = _load().mt_tree_accept_commit(ctypes.byref(desc), V, int(max_depth),
                                       _DTYPES[target_logits.dtype], _ptr(tree_tokens),
                                       _ptr(target_logits), _ptr(tree_parents), _ptr(argmax_out),
                                       _ptr(accept_len), _ptr(accept_path), _ptr(next_token),
                                       _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       _ptr(seq_lens), _ptr(released_pages), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "mt_tree_accept_commit")
    return accept_len, accept_path


def tree_candidates(root_logits, head_logits, tree_parents, tree_tokens, *, status_ws: torch.Tensor,
                    stream=None):
    """Tree tokens from the base logits [B,V] and the Medusa heads' logits [B,heads,V]:
    node 0 takes the argmax of the base logits, the r-th child (r earlier siblings)
    of a depth-(d-1) node the rank-r token of head d-1."""
    _need(root_logits, "root_logits", None, 2)
    _need(head_logits, "head_logits", root_logits.dtype, 3)
    _need(tree_parents, "tree_parents", torch.int32, 2)
    _need(tree_tokens, "tree_tokens", torch.int32, 2)
    B, V = root_logits.shape
    heads = head_logits.shape[1]
    if head_logits.shape != (B, heads, V):
        raise ValueError("head_logits must be [B, heads, V]")
    T = tree_parents.shape[1]
    if tree_parents.shape != (B, T) or tree_tokens.shape != (B, T):
        raise ValueError("tree_parents and tree_tokens must be [B, T]")
    _need(status_ws, "status_ws")
    _min_bytes(status_ws, "status_ws", 256)
    _on_device(root_logits=root_logits, head_logits=head_logits, tree_parents=tree_parents,
               tree_tokens=tree_tokens, status_ws=status_ws)
    st = _load().mt_tree_candidates(B, T, heads, V, _DTYPES[root_logits.dtype], _ptr(root_logits),
                                    _ptr(head_logits), _ptr(tree_parents), _ptr(tree_tokens),
                                    _ptr(status_ws), _stream(stream))
    _check(st, "mt_tree_candidates")
    return tree_tokens


def read_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream, returns and clears the device status word."""
    _need(workspace, "workspace")
    _min_bytes(workspace, "workspace", 4)
    _on_device(workspace=workspace)
    v = ctypes.c_int(0)
    _check(_load().mt_read_status(_ptr(workspace), _stream(stream), ctypes.byref(v)), "mt_read_status")
    return v.value


def profile_enable(max_records: int):
    """Record CUDA events around the main attention kernel of the next calls."""
    _check(_load().mt_profile_enable(int(max_records)), "mt_profile_enable")


def profile_read(max_records: int = 65536):
    """Elapsed milliseconds of the main attention kernel, one per recorded call."""
    buf = (ctypes.c_float * max_records)()
    n = ctypes.c_int(0)
    _check(_load().mt_profile_read(buf, max_records, ctypes.byref(n)), "mt_profile_read")
    return [buf[i] for i in range(n.value)]


def debug_set_wait(limit_ns: int = 0, stall: bool = False):
    """Bound of the tensor-core kernel's pipeline waits for later attention
    calls (0: the default, 2 s); stall=True makes its first wait one that only
    a timeout ends (tests of the timeout path)."""
    _check(_load().mt_debug_set_wait(int(limit_ns), 1 if stall else 0), "mt_debug_set_wait")


def version() -> int:
    return int(_load().mt_version())
