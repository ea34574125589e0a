"""GPU parity: attn_fwd_splitkv (CUDA split-KV decode + combine, through the
C ABI) against the fp64 CPU oracle with per-sequence cache lengths.

The full decode workload (B=16, Hq=32, Hkv=8, d=128, lengths U[1024, 16384],
chunk 1024) is compared on every output.  Cache positions at or beyond a
sequence's length hold NaN, so any read of them into the result would show.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_14_gb300 import _native, build as native_build, workloads
from tests._parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    native_build.build()
    _native.lib()
    torch.cuda.init()


def _check(q, k, v, L, scale, chunk, what):
    o, lse = _native.decode(q.cuda(), k.cuda(), v.cuda(), L.cuda(), scale, chunk)
    assert _native.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, scale, kv_len=L.numpy())
    return compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what)


def test_decode_workload_full():
    w = workloads.DECODE
    q, k, v, L = workloads.workload_decode_inputs(w)
    _check(q, k, v, L, w.scale, w.chunk, w.name)


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 8, 128), (16, 2, 64), (6, 3, 128), (8, 1, 128), (12, 2, 64)])
def test_group_sizes_and_head_dims(Hq, Hkv, d):
    lens = [1, 63, 64, 65, 1023, 1024, 1025, 2048, 3001]
    q, k, v, L = workloads.decode_inputs(len(lens), Hq, Hkv, 3072, d, 0, 0, seed=31 + Hq, seqlens=lens)
    _check(q, k, v, L, d ** -0.5, 1024, "Hq%d Hkv%d d%d" % (Hq, Hkv, d))


def test_lengths_at_the_workload_maximum():
    """Lengths at the workload's top (16384: sixteen full 1024-key splits) and
    right around it and its lowest length, in the workload's configuration."""
    w = workloads.DECODE
    lens = [16384, 16383, 15361, 1024, 1025, 16384]
    q, k, v, L = workloads.decode_inputs(len(lens), w.Hq, w.Hkv, w.max_seqlen, w.d, 0, 0, seed=48, seqlens=lens)
    _check(q, k, v, L, w.scale, w.chunk, "lengths at 16384")


@pytest.mark.parametrize("chunk", [64, 256, 1024, 4096])
def test_chunk_sizes(chunk):
    lens = [5, 700, 4096, 4000]
    q, k, v, L = workloads.decode_inputs(len(lens), 8, 2, 4096, 128, 0, 0, seed=40, seqlens=lens)
    _check(q, k, v, L, 0.0884, chunk, "chunk%d" % chunk)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_rising_scores_move_the_reference(sign):
    """Scores that climb by ~60 (natural-log units) along each sequence move
    the exponent reference many times inside one split; a negative scale
    runs the same path on -s."""
    lens = [3000, 1500, 700]
    B, Hq, Hkv, d, N = len(lens), 8, 2, 128, 3072
    q, k, v, L = workloads.decode_inputs(B, Hq, Hkv, N, d, 0, 0, seed=42, seqlens=lens)
    q = torch.ones_like(q)
    ramp = torch.zeros((B, N), dtype=torch.float32)
    for b, n in enumerate(lens):
        ramp[b, :n] = torch.linspace(-4.0, 4.0, n)
    k = (ramp[:, :, None, None] * torch.ones((1, 1, Hkv, d))).to(torch.bfloat16)
    _check(q, k, v, L, sign * d ** -0.5, 1024, "rising scores sign %+d" % sign)


@pytest.mark.parametrize("B", [33, 64, 70])
def test_many_sequences(B):
    """Work order across the batch: lanes of both halves of the listing warp
    (B > 32), the largest batch it lists (64), and the plain order beyond."""
    g = torch.Generator().manual_seed(43 + B)
    lens = torch.randint(0, 300, (B,), generator=g).tolist()
    lens[0], lens[-1] = 256, 0
    q, k, v, L = workloads.decode_inputs(B, 4, 2, 320, 64, 0, 0, seed=44 + B, seqlens=lens)
    _check(q, k, v, L, 0.125, 64, "B%d" % B)


def _check_paged(q, k, v, L, scale, chunk, page_size, what, seed=0):
    """Paged decode against the oracle on the logical cache the pages stand for."""
    kp, vp, bt = workloads.page_cache(k, v, page_size, seed=seed)
    o, lse = _native.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), bt.cuda(), L.cuda(), scale, chunk)
    assert _native.attn_get_device_status() == 0
    kc = oracle.paged_to_contiguous(kp, bt)
    vc = oracle.paged_to_contiguous(vp, bt)
    o_ref, lse_ref = oracle.attn_fwd(q, kc, vc, False, scale, kv_len=L.numpy())
    return compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what)


@pytest.mark.parametrize("page_size,chunk", [(64, 1024), (256, 1024), (256, 256), (512, 1024), (1024, 256)])
def test_paged_cache(page_size, chunk):
    """Pages in a shuffled order, unused pages full of NaN, lengths that end
    inside a page, on a page boundary, and at zero."""
    lens = [3000, 1536, 1, 0, 700]
    q, k, v, L = workloads.decode_inputs(len(lens), 8, 2, 3072, 128, 0, 0, seed=45, seqlens=lens)
    _check_paged(q, k, v, L, 128 ** -0.5, chunk, page_size, "paged ps%d chunk%d" % (page_size, chunk), seed=page_size)


def test_paged_cache_gqa_d64():
    lens = [640, 1, 1024]
    q, k, v, L = workloads.decode_inputs(len(lens), 12, 3, 1024, 64, 0, 0, seed=46, seqlens=lens)
    _check_paged(q, k, v, L, 0.125, 512, 128, "paged gqa d64")


def test_paged_bad_page_is_reported():
    """A block-table entry outside the page pool reads page 0 instead and is
    reported on the device; nothing faults."""
    lens = [300, 200]
    q, k, v, L = workloads.decode_inputs(2, 4, 2, 512, 128, 0, 0, seed=47, seqlens=lens)
    kp, vp, bt = workloads.page_cache(k, v, 256, seed=3)
    bt = bt.clone()
    bt[1, 0] = kp.shape[0] + 5
    _native.attn_get_device_status()  # clear
    o, lse = _native.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), bt.cuda(), L.cuda(), 0.1, 256)
    assert _native.attn_get_device_status() == _native.ATTN_ERR_DEVICE_ARG


def test_zero_length_sequence():
    lens = [0, 17]
    q, k, v, L = workloads.decode_inputs(2, 4, 2, 128, 128, 0, 0, seed=41, seqlens=lens)
    o, lse = _native.decode(q.cuda(), k.cuda(), v.cuda(), L.cuda(), 0.1, 64)
    assert torch.count_nonzero(o[0]).item() == 0 and torch.isneginf(lse[0]).all()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 0.1, kv_len=L.numpy())
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "zero length")


def test_bad_length_is_reported_on_the_device():
    q, k, v, L = workloads.decode_inputs(2, 4, 2, 128, 128, 0, 0, seed=42, seqlens=[10, 20])
    L = torch.tensor([10, 129], dtype=torch.int32)
    _native.decode(q.cuda(), k.cuda(), v.cuda(), L.cuda(), 0.1, 64)
    assert _native.attn_get_device_status() == 6
    assert _native.attn_get_device_status() == 0  # cleared by the read


def test_workspace_too_small_is_refused():
    q, k, v, L = workloads.decode_inputs(2, 4, 2, 256, 128, 0, 0, seed=43, seqlens=[10, 20])
    need = _native.attn_splitkv_workspace_size(2, 4, 256, 128, 64)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q.cuda())
    lse = torch.empty((2, 4, 1), device="cuda")
    rc = _native.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), L.cuda(), o, lse, 0.1, 64, ws)
    assert rc == 7


def test_repeat_runs_are_bitwise_identical():
    w = workloads.DECODE
    q, k, v, L = workloads.decode_inputs(4, 32, 8, 8192, 128, 1024, 8192, seed=44)
    args = (q.cuda(), k.cuda(), v.cuda(), L.cuda(), w.scale, 1024)
    a, b = _native.decode(*args), _native.decode(*args)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
