"""attn_fwd_splitkv_noalloc: the split-KV decode entry point for callers that
cannot allocate device memory (an allocator or memory-pool callback, a hot
loop under a no-allocation policy, a plain C caller with no device memory to
spare for a workspace).  It keeps its partial results in a fixed scratch
array inside the library instead of a caller-provided workspace.

Checked through the C ABI against attn_fwd_splitkv (the entry point that
takes a workspace) on two calls in a row.  Both run the same kernels on the
same inputs, so the results must be bitwise equal (which is inside the
parity tolerances the other GPU tests use); one call is also compared with
the fp64 oracle.  The refusal of sizes beyond the scratch needs no GPU and is
checked in tests/test_abi.py.  This file is named to be collected last, and
passes both on its own in a fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

import oracle
from exact_io_aware_14_gb300 import _native, build as native_build, workloads
from tests._parity import compare

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


def _bitwise(o_a, lse_a, o_b, lse_b):
    assert torch.equal(o_a.view(torch.int16), o_b.view(torch.int16))
    assert torch.equal(lse_a.view(torch.int32), lse_b.view(torch.int32))


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    w = workloads.DECODE
    assert _native.attn_splitkv_workspace_size(w.B, w.Hq, w.max_seqlen, w.d, w.chunk) <= SCRATCH_MAX
    cpu_inputs = []
    for seed in (w.seed, w.seed + 1):  # two different problems, one after the other
        cpu_inputs.append(workloads.decode_inputs(w.B, w.Hq, w.Hkv, w.max_seqlen, w.d, w.len_lo, w.len_hi,
                                                  seed=seed))
    for n, (qc, kc, vc, Lc) in enumerate(cpu_inputs):
        q, k, v, L = (x.cuda() for x in (qc, kc, vc, Lc))
        o_ref, lse_ref = _native.decode(q, k, v, L, w.scale, w.chunk)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
        assert _noalloc(q, k, v, L, o, lse, w.scale, w.chunk) == 0
        torch.cuda.synchronize()
        assert _native.attn_get_device_status() == 0
        _bitwise(o, lse, o_ref, lse_ref)
        if n == 0:
            o_or, lse_or = oracle.attn_fwd(qc, kc, vc, False, w.scale, kv_len=Lc.numpy())
            compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_or, lse_or, "noalloc decode workload")


def test_noalloc_smaller_shape_after_larger_one():
    """The scratch keeps the previous call's contents; a smaller call must not
    read any of them.  The second call goes through the Python binding."""
    q, k, v, L = workloads.decode_inputs(3, 8, 2, 2048, 64, 0, 0, seed=61, seqlens=[1, 1024, 1999])
    q, k, v, L = (x.cuda() for x in (q, k, v, L))
    for n in range(2):
        o_ref, lse_ref = _native.decode(q, k, v, L, 0.125, 256)
        o = torch.empty_like(q)
        lse = torch.empty((3, 8, 1), dtype=torch.float32, device="cuda")
        if n == 0:
            assert _noalloc(q, k, v, L, o, lse, 0.125, 256) == 0
        else:
            assert _native.attn_fwd_splitkv_noalloc(q, k, v, L, o, lse, 0.125, 256) == 0
        torch.cuda.synchronize()
        assert _native.attn_get_device_status() == 0
        _bitwise(o, lse, o_ref, lse_ref)
