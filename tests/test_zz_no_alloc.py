"""attn_fwd_splitkv_noalloc: the split-KV decode entry point for callers that
cannot allocate device memory (an allocator or memory-pool callback, a hot
loop under a no-allocation policy, a plain C caller with no device memory to
spare for a workspace).  It keeps its partial results in a fixed scratch
array inside the library instead of a caller-provided workspace.

Checked through the C ABI against attn_fwd_splitkv (the entry point that
takes a workspace) on two calls in a row, within the parity tolerances the
other GPU tests use.  This file is named to be collected last, and passes
both on its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_io_aware_14_gb300 import _native, build as native_build, workloads
from tests._parity import LSE_ABS, O_MAX_ABS, O_MEAN_ABS

pytestmark = pytest.mark.gpu

SCRATCH_MAX = 8 << 20  # ATTN_SPLITKV_NOALLOC_MAX_BYTES


@pytest.fixture(scope="module", autouse=True)
def _lib():
    native_build.build()
    _native.lib()
    torch.cuda.init()


def _noalloc(q, k, v, L, o, lse, scale, chunk):
    """Raw C-ABI call of attn_fwd_splitkv_noalloc (no workspace argument)."""
    B, _, Hq, d = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return _native.lib().attn_fwd_splitkv_noalloc(p(q), p(k), p(v), p(L), S, p(o), p(lse), B, Hq, Hkv, d,
                                                  ctypes.c_float(scale), chunk, stream)


def _close(o_a, lse_a, o_b, lse_b):
    err = (o_a.float() - o_b.float()).abs()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    fin = torch.isfinite(lse_b)
    assert torch.equal(torch.isfinite(lse_a), fin)
    assert (lse_a[fin] - lse_b[fin]).abs().max().item() <= LSE_ABS


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    w = workloads.DECODE
    assert _native.attn_splitkv_workspace_size(w.B, w.Hq, w.max_seqlen, w.d, w.chunk) <= SCRATCH_MAX
    inputs = []
    for seed in (w.seed, w.seed + 1):  # two different problems, one after the other
        q, k, v, L = workloads.decode_inputs(w.B, w.Hq, w.Hkv, w.max_seqlen, w.d, w.len_lo, w.len_hi, seed=seed)
        inputs.append(tuple(x.cuda() for x in (q, k, v, L)))
    for q, k, v, L in inputs:
        o_ref, lse_ref = _native.decode(q, k, v, L, w.scale, w.chunk)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
        assert _noalloc(q, k, v, L, o, lse, w.scale, w.chunk) == 0
        torch.cuda.synchronize()
        assert _native.attn_get_device_status() == 0
        assert torch.isfinite(o.float()).all()
        _close(o, lse, o_ref, lse_ref)


def test_noalloc_smaller_shape_after_larger_one():
    """The scratch keeps the previous call's contents; a smaller call must not
    read any of them."""
    q, k, v, L = workloads.decode_inputs(3, 8, 2, 2048, 64, 0, 0, seed=61, seqlens=[1, 1024, 1999])
    q, k, v, L = (x.cuda() for x in (q, k, v, L))
    for _ in range(2):
        o_ref, lse_ref = _native.decode(q, k, v, L, 0.125, 256)
        o = torch.empty_like(q)
        lse = torch.empty((3, 8, 1), dtype=torch.float32, device="cuda")
        assert _noalloc(q, k, v, L, o, lse, 0.125, 256) == 0
        torch.cuda.synchronize()
        _close(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_sizes_beyond_the_scratch():
    # 64 x 32 heads x 32 splits x (128 + 1) floats is about 33 MB > 8 MiB: refused before any launch
    assert _native.attn_splitkv_workspace_size(64, 32, 32768, 128, 1024) > SCRATCH_MAX
    q = torch.zeros((64, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((64, 16, 8, 128), dtype=torch.bfloat16, device="cuda")  # never read
    L = torch.zeros((64,), dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((64, 32, 1), dtype=torch.float32, device="cuda")
    B, _, Hq, d = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = _native.lib().attn_fwd_splitkv_noalloc(p(q), p(k), p(k), p(L), 32768, p(o), p(lse), B, Hq, 8, d,
                                                ctypes.c_float(0.1), 1024, stream)
    assert rc == 7  # ATTN_ERR_WORKSPACE
