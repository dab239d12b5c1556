"""The C ABI library loads on a machine without a GPU, exports every function
that include/medusa_tree.h declares, and rejects bad host-side arguments
before touching the device."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "medusa_tree.h")


@pytest.fixture(scope="module")
def lib():
    from medusa_tree_speculative_attn_gb300 import build
    build.build()
    import medusa_tree_speculative_attn_gb300 as mt
    return mt.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(mt_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("mt_tree_attn_paged", "mt_tree_accept_greedy", "mt_kv_commit", "mt_tree_candidates",
              "mt_tree_accept_commit",
              "mt_tree_attn_workspace_size", "mt_tree_accept_workspace_size", "mt_rope_create",
              "mt_rope_destroy", "mt_read_status", "mt_status_string", "mt_version",
              "mt_debug_set_wait"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in medusa_tree.h but not exported"


def test_status_strings_and_version(lib):
    import medusa_tree_speculative_attn_gb300 as mt
    assert mt.version() == 10000
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert mt.status_string(code) != "unknown status"


def _desc(**kw):
    import medusa_tree_speculative_attn_gb300 as mt
    base = dict(batch=2, tree_size=8, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                max_blocks_per_seq=8, num_pages=32, num_splits=0, dtype=2, sm_scale=0.0, kernel=0,
                cache_dtype=0, k_scale=1.0, v_scale=1.0)
    base.update(kw)
    return mt.AttnDesc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(tree_size=65), -2), (dict(tree_size=0), -2), (dict(head_dim=96), -2),
    (dict(page_size=32), -2), (dict(num_q_heads=6, num_kv_heads=4), -1), (dict(batch=0), -1),
    (dict(dtype=7), -2), (dict(kernel=9), -1), (dict(kernel=2, dtype=0), -2),
    (dict(num_splits=-1), -1), (dict(sm_scale=float("nan")), -1),
    # FP8 cache: E4M3 only, as a cache type only, positive finite scales, and on
    # tensor cores only with a 16-bit act dtype
    (dict(dtype=3), -2), (dict(cache_dtype=5), -2), (dict(cache_dtype=1), -2),
    (dict(cache_dtype=3, k_scale=0.0), -1), (dict(cache_dtype=3, v_scale=-1.0), -1),
    (dict(cache_dtype=3, k_scale=float("nan")), -1), (dict(cache_dtype=3, v_scale=float("inf")), -1),
    (dict(cache_dtype=3, kernel=2, dtype=0), -2),
])
def test_attn_rejects_bad_descriptors(lib, kw, code):
    d = _desc(**kw)
    P = ctypes.c_void_p
    buf = (ctypes.c_char * 4096)()
    p = ctypes.cast(buf, P)
    st = lib.mt_tree_attn_paged(ctypes.byref(d), p, p, p, p, p, p, p, p, p, p, p, p, 4096, None)
    assert st == code
    assert lib.mt_tree_attn_workspace_size(ctypes.byref(d)) == 0


def test_attn_rejects_null_and_misaligned_pointers(lib):
    d = _desc()
    buf = (ctypes.c_char * 4096)()
    base = ctypes.addressof(buf)
    al = ctypes.c_void_p((base + 255) // 256 * 256)
    mis = ctypes.c_void_p(al.value + 4)
    args = [al] * 12
    args_null = list(args)
    args_null[0] = None
    assert lib.mt_tree_attn_paged(ctypes.byref(d), *args_null, 4096, None) == -1
    args_mis = list(args)
    args_mis[0] = mis
    assert lib.mt_tree_attn_paged(ctypes.byref(d), *args_mis, 4096, None) == -1


def test_accept_and_commit_reject_bad_sizes(lib):
    P = ctypes.c_void_p
    buf = (ctypes.c_char * 4096)()
    p = ctypes.cast(buf, P)
    # tree larger than one 64-bit mask
    assert lib.mt_tree_accept_greedy(1, 65, 10, 3, 0, p, p, p, p, p, p, p, p, 4096, None) == -2
    assert lib.mt_tree_accept_greedy(1, 8, 0, 3, 0, p, p, p, p, p, p, p, p, 4096, None) == -1
    assert lib.mt_tree_accept_greedy(1, 8, 10, 3, 9, p, p, p, p, p, p, p, p, 4096, None) == -2
    assert lib.mt_tree_accept_greedy(1, 8, 10, 3, 0, None, p, p, p, p, p, p, p, 4096, None) == -1
    assert lib.mt_tree_accept_workspace_size(0, 8) == 0
    d = _desc(tree_size=70)
    assert lib.mt_kv_commit(ctypes.byref(d), 3, p, p, p, p, p, p, p, p, None) == -2
    d = _desc()
    assert lib.mt_kv_commit(ctypes.byref(d), 3, None, p, p, p, p, p, p, p, None) == -1


def test_fused_accept_commit_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    buf = (ctypes.c_char * 4096)()
    p = ctypes.cast(buf, P)
    f = lib.mt_tree_accept_commit
    f.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int] + [P] * 12 + [P, ctypes.c_size_t, P]
    d = _desc()
    ok = [p] * 12
    assert f(ctypes.byref(_desc(tree_size=70)), 10, 3, 0, *ok, p, 4096, None) == -2  # tree too large
    assert f(ctypes.byref(d), 0, 3, 0, *ok, p, 4096, None) == -1  # empty vocab
    assert f(ctypes.byref(d), 10, 64, 0, *ok, p, 4096, None) == -1  # max_depth past one mask
    assert f(ctypes.byref(d), 10, 3, 9, *ok, p, 4096, None) == -2  # unknown logits dtype
    assert f(ctypes.byref(d), 10, 3, 0, *ok, p, 0, None) == -1  # workspace too small
    for k in range(12):
        args = list(ok)
        args[k] = None
        assert f(ctypes.byref(d), 10, 3, 0, *args, p, 4096, None) == -1  # null pointer
    assert f(ctypes.byref(d), 10, 3, 0, *ok, None, 4096, None) == -1


def test_typical_acceptance_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    buf = (ctypes.c_char * 16384)()
    p = ctypes.cast(buf, P)
    al = ctypes.c_void_p((ctypes.addressof(buf) + 255) // 256 * 256)
    f = lib.mt_tree_accept_typical
    f.argtypes = [ctypes.c_int] * 5 + [P] * 3 + [ctypes.c_float] * 3 + [P] * 5 + [ctypes.c_size_t, P]
    ok = dict(temperature=1.0, epsilon=0.09, delta=0.3)

    def call(B=1, T=8, V=10, md=3, dt=0, t=ok["temperature"], e=ok["epsilon"], d=ok["delta"], ptrs=None,
             ws=al, nbytes=8192):
        args = ptrs if ptrs is not None else [p] * 7
        return f(B, T, V, md, dt, args[0], args[1], args[2], t, e, d, args[3], args[4], args[5], args[6],
                 ws, nbytes, None)
    assert lib.mt_tree_accept_workspace_size(1, 8) <= 8192
    assert call(T=65) == -2 and call(V=0) == -1 and call(md=64) == -1 and call(dt=9) == -2
    assert call(B=0) == -1
    for bad in (dict(t=0.0), dict(t=-1.0), dict(t=float("nan")), dict(t=float("inf")), dict(t=1e-40),
                dict(e=0.0), dict(e=float("inf")), dict(d=0.0), dict(d=float("nan"))):
        assert call(**bad) == -1, bad
    for k in range(7):
        ptrs = [p] * 7
        ptrs[k] = None
        assert call(ptrs=ptrs) == -1
    assert call(ws=None) == -1
    assert call(ws=ctypes.c_void_p(al.value + 16)) == -1   # workspace not 256-byte aligned
    assert call(nbytes=lib.mt_tree_accept_workspace_size(1, 8) - 1) == -1


def test_accept_workspace_holds_typical_scratch(lib):
    lib.mt_tree_accept_workspace_size.restype = ctypes.c_size_t
    for B, T in ((1, 1), (16, 64), (3, 7)):
        # status, counters, argmax and statistics per row, split-row keys and
        # counters, and 16 split-row statistics entries per row (up to 1024 rows)
        rows = B * T
        assert lib.mt_tree_accept_workspace_size(B, T) >= 256 + 4 * B + 32 * rows + 256 * min(rows, 1024)
        assert lib.mt_tree_accept_workspace_size(B, T) % 256 == 0


def test_candidates_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    buf = (ctypes.c_char * 4096)()
    p = ctypes.cast(buf, P)
    c = lib.mt_tree_candidates
    assert c(1, 65, 2, 10, 0, p, p, p, p, p, None) == -2  # tree larger than 64 nodes
    assert c(1, 0, 2, 10, 0, p, p, p, p, p, None) == -2
    assert c(1, 8, 0, 10, 0, p, p, p, p, p, None) == -1  # no heads
    assert c(1, 8, 64, 10, 0, p, p, p, p, p, None) == -1  # more heads than tree depths
    assert c(1, 8, 2, 0, 0, p, p, p, p, p, None) == -1  # empty vocab
    assert c(0, 8, 2, 10, 0, p, p, p, p, p, None) == -1  # empty batch
    assert c(1, 8, 2, 10, 7, p, p, p, p, p, None) == -2  # unknown dtype
    for k in range(5):
        args = [p] * 5
        args[k] = None
        assert c(1, 8, 2, 10, 0, *args, None) == -1  # null pointer


def test_rope_create_rejects_bad_arguments(lib):
    out = ctypes.c_void_p()
    assert lib.mt_rope_create(10000.0, 96, 100, ctypes.byref(out)) == -1
    assert lib.mt_rope_create(-1.0, 128, 100, ctypes.byref(out)) == -1
    assert lib.mt_rope_create(10000.0, 128, 0, ctypes.byref(out)) == -1
    assert lib.mt_rope_destroy(None) == 0


def test_binding_refuses_to_run_without_library(tmp_path, monkeypatch):
    import medusa_tree_speculative_attn_gb300 as mt
    monkeypatch.setattr(mt, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mt, "_lib", None)
    with pytest.raises(RuntimeError):
        mt.library()


C_PROGRAM = r"""
#include "medusa_tree.h"
#include <stdio.h>
int main(void) {
  mt_attn_desc d = {0};
  d.batch = 2; d.tree_size = 8; d.num_q_heads = 8; d.num_kv_heads = 2; d.head_dim = 96;
  d.page_size = 16; d.max_blocks_per_seq = 4; d.num_pages = 8; d.dtype = MT_BF16;
  printf("%d %d %zu\n", mt_version(), (int)mt_tree_attn_workspace_size(&d),
         mt_tree_accept_workspace_size(0, 8));
  return 0;
}
"""


def test_header_compiles_as_c_and_links(lib, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from medusa_tree_speculative_attn_gb300 import LIB_PATH
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    libdir = os.path.dirname(LIB_PATH)
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-I", cuda_inc, str(src), "-o", str(exe), "-L", libdir, "-lmedusa_tree",
                           "-Wl,-rpath," + libdir])
    out = subprocess.check_output([str(exe)]).decode().split()
    assert out == ["10000", "0", "0"]   # version; head_dim 96 refused (size 0); empty batch


def test_debug_set_wait_refuses_bad_stall(lib):
    assert lib.mt_debug_set_wait(0, 2) == -1
    assert lib.mt_debug_set_wait(0, 0) == 0

