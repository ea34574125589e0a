"""The software exp2 on the GPU, and the prefill built to use it.

(1) attn_selftest_exp2_poly evaluates the kernel's software exp2
(csrc/exp2_poly.cuh: Cody and Waite's range reduction and a fitted degree-3
polynomial, as FA4 uses to relieve the MUFU unit -- "FlashAttention: Part
2", sections 1.7 and 1.8) on the device; it must stay within 1.02e-4
relative error of float64 exp2 over the softmax's range, agree with CUDA's
own exp2f (torch.exp2 on the device) to the same bound, give exact powers
of two at integers, and clamp as documented.  (2) The library built with
ATTN_EXP2_POLY=4 (every fourth pair of a row's exponentials in software)
matches the fp64 oracle within the usual tolerances.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_14_gb300 import _native, build as native_build, workloads
from tests._parity import compare

pytestmark = pytest.mark.gpu

BOUND = 1.02e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    native_build.build()
    _native.lib()
    torch.cuda.init()


def _poly(x_host):
    x = torch.as_tensor(np.asarray(x_host, dtype=np.float32)).cuda()
    y = torch.empty_like(x)
    assert _native.attn_selftest_exp2_poly(x, y) == 0
    torch.cuda.synchronize()
    return x, y


def test_software_exp2_error_bound():
    # the softmax's inputs: s*c - m*c, at most 16 above the reference before a
    # half's sum moves it, unbounded below; odd length tests the unpaired tail
    x_host = np.concatenate([np.linspace(-125.0, 64.0, 2_000_001), np.linspace(-1.0, 1.0, 100_001)])
    x, y = _poly(x_host)
    ref = np.exp2(x.cpu().numpy().astype(np.float64))
    rel = np.abs(y.cpu().numpy().astype(np.float64) / ref - 1.0)
    assert rel.max() <= BOUND, rel.max()
    # against CUDA's own exp2f on the same device
    cuda = torch.exp2(x).cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y.cpu().numpy() / cuda - 1.0)) <= BOUND + 2e-7


def test_software_exp2_exact_powers_and_clamps():
    ints = np.arange(-125, 65, dtype=np.float32)
    _, y = _poly(ints)
    assert np.array_equal(y.cpu().numpy(), np.exp2(ints.astype(np.float64)).astype(np.float32))
    _, y = _poly([-1000.0, -np.inf, np.nan, 1000.0, np.inf])
    got = y.cpu().numpy()
    assert got[0] == got[1] == got[2] == np.float32(2.0 ** -125)
    assert got[3] == got[4] == np.float32(2.0 ** 64)


def test_selftest_argument_checks():
    x = torch.zeros(4, device="cuda")
    L = _native.lib()
    assert L.attn_selftest_exp2_poly(None, None, 0, None) == 0
    assert L.attn_selftest_exp2_poly(None, None, -1, None) == 1
    assert L.attn_selftest_exp2_poly(None, x.data_ptr(), 4, None) == 1
    assert L.attn_selftest_exp2_poly(x.data_ptr() + 2, x.data_ptr(), 1, None) == 3


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 2, 300, 300, 128, False),
    (1, 2, 2, 300, 300, 128, True),
    (2, 4, 2, 200, 333, 64, True),
    (2, 32, 8, 700, 700, 128, True),
    (3, 40, 40, 300, 300, 128, True),
])
def test_prefill_with_software_exp2_matches_the_oracle(B, Hq, Hkv, Nq, Nk, d, causal):
    L = _native.variant_lib("exp2poly4")
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=300 + Nq + Hq)
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward(q.cuda(), k.cuda(), v.cuda(), causal, scale, library=L)
    assert L.attn_get_device_status(None) == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "exp2poly4 %s" % ((B, Hq, Nq, causal),))


def test_training_workload_with_software_exp2_every_row():
    L = _native.variant_lib("exp2poly4")
    w = workloads.TRAIN_CAUSAL
    q, k, v = workloads.workload_inputs(w)
    o, lse = _native.forward(q.cuda(), k.cuda(), v.cuda(), w.causal, w.scale, library=L)
    assert L.attn_get_device_status(None) == 0
    o_gpu, lse_gpu = o.float().cpu().numpy(), lse.cpu().numpy()
    del o, lse
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    compare(o_gpu, lse_gpu, o_ref, lse_ref, w.name + " with the software exp2")


def test_read_probe_reads_every_word():
    """attn_probe_read_bandwidth folds every 16-byte word of the buffer into
    its sink by XOR: over a buffer whose words XOR to a known value the sink
    must hold it (no load skipped, none read twice), including a ragged tail
    that is not a multiple of the grid's stride."""
    n_words = (64 << 20) // 4 + 12  # 64 MB plus three 16-byte words
    buf = torch.zeros(n_words, dtype=torch.int32, device="cuda")
    buf[5] = 0x12345678
    buf[n_words - 1] = 0x0F0F0F0F      # in the last 16-byte word
    buf[n_words // 2] = 0x00FF00FF
    sink = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert _native.attn_probe_read_bandwidth(buf, sink) == 0
    torch.cuda.synchronize()
    expect = 0x12345678 ^ 0x0F0F0F0F ^ 0x00FF00FF
    assert int(sink.item()) == expect
    assert _native.attn_get_device_status() == 0
