"""The allocation-free tree attention entry point.

Some callers cannot allocate device memory on the calling path (a serving
loop that must not risk cudaMalloc's device synchronisation or out-of-memory
failure between steps, or code that only receives its input and output
buffers from a pool it does not own).  mt_tree_attn_paged_noalloc serves them
from a fixed array the library reserves on each device.  This test calls it
through the C ABI twice in a row, on two different workloads, and checks each
result against mt_tree_attn_paged with an allocated workspace.  Both run the
same kernels on the same schedule, so the outputs must be equal bit for bit.
It also checks that a call, once the library is loaded on the device, leaves
the device's free memory unchanged.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import medusa_tree_speculative_attn_gb300 as mt
import workloads
from gpu_helpers import Step

pytestmark = pytest.mark.gpu


def _noalloc(step, device_status, out):
    lib = mt.library()
    fn = lib.mt_tree_attn_paged_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(mt.AttnDesc)] + [P] * 12 + [P]
    d = step.d
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    st = fn(ctypes.byref(step.desc), ptr(d["q"]), ptr(d["k_new"]), ptr(d["v_new"]), ptr(d["k_cache"]),
            ptr(d["v_cache"]), ptr(d["block_tables"]), ptr(d["seq_lens"]), ptr(d["tree_parents"]),
            ptr(d["tree_depths"]), step.rope.handle, ptr(out), ptr(device_status),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    specs = [
        workloads.custom("noalloc_bf16", B=4, Hq=32, Hkv=8, head_dim=128, dtype="bf16",
                         prefix=("list", [700, 64, 2049, 5]), tree=("fanout", (10, 5, 3, 2), 64),
                         max_depth=4),
        workloads.custom("noalloc_fp16", B=3, Hq=16, Hkv=16, head_dim=128, dtype="f16",
                         prefix=("list", [1000, 17, 333]), tree=("fanout", (4, 3, 2), 20),
                         max_depth=3),
    ]
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    for k, spec in enumerate(specs):
        w = workloads.generate(spec, seed=10 + k)
        ref = Step(w)
        ref.attn()
        assert ref.status()[0] == 0
        out = torch.full_like(ref.out, float("nan"))
        st = _noalloc(ref, status, out)
        assert st == 0, mt.status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref.out)
        # a second call on the same buffers allocates nothing on the device
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = _noalloc(ref, status, out)
        torch.cuda.synchronize()
        assert st == 0 and int(status.item()) == 0
        assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(out, ref.out)


def test_noalloc_reports_bad_descriptors_like_the_workspace_call():
    lib = mt.library()
    fn = lib.mt_tree_attn_paged_noalloc
    fn.argtypes = [ctypes.POINTER(mt.AttnDesc)] + [ctypes.c_void_p] * 13
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    bad = mt.AttnDesc(0, 8, 4, 2, 128, 16, 4, 64, 0, 2, 0.0, 0)   # batch 0
    assert fn(ctypes.byref(bad), p, p, p, p, p, p, p, p, p, p, p, None, None) == -1
    assert fn(None, p, p, p, p, p, p, p, p, p, p, p, None, None) == -1


def test_noalloc_rejects_oversized_workspace():
    # a batch whose workspace is beyond the fixed array is refused, not run
    desc = mt.AttnDesc(8192, 64, 64, 8, 128, 16, 4, 1 << 20, 0, 2, 0.0, 0)
    lib = mt.library()
    fn = lib.mt_tree_attn_paged_noalloc
    fn.argtypes = [ctypes.POINTER(mt.AttnDesc)] + [ctypes.c_void_p] * 13
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    assert mt.attn_workspace_size(desc) > (64 << 20)
    st = fn(ctypes.byref(desc), p, p, p, p, p, p, p, p, p, p, p, None, None)
    assert st == -2
