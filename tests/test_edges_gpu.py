"""GPU parity at shapes the other suites do not reach: large GQA groups (8
and 16 query heads per KV head, several decode head blocks), odd batch
counts, a query block one row short of a tile, a single query row against a
long key range (many key tiles for one row), the smallest page size with the
largest chunk the paged decode accepts, and d = 64 against a cache with a
window.  Each is compared with the fp64 oracle element by element."""
import math

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


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 64, 8, 600, 600, 128, 1),     # group of 8: four head pairs per KV head
    (7, 6, 2, 140, 140, 64, 0),       # odd batch count, group of 3
    (2, 4, 4, 127, 1, 128, 0),        # one row short of a tile, a single key
    (1, 2, 1, 1, 20000, 128, 2),      # one query row against 157 key tiles
    (3, 16, 1, 257, 515, 64, 2),      # multi-query (one KV head), bottom-right
])
def test_prefill_edges(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=600 + Nq + Hq)
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    assert _native.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
            "edge B%d Hq%d Hkv%d Nq%d Nk%d d%d c%d" % (B, Hq, Hkv, Nq, Nk, d, causal))


def _decode_check(q, k, v, L, scale, o, lse, what):
    B, _, Hq, d = q.shape
    rows = np.array([(b, h, 0) for b in range(B) for h in range(Hq)], dtype=np.int32)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, rows, False, scale, kv_len=L.numpy())
    got_o = o[:, 0].float().cpu().numpy().reshape(B * Hq, d)
    got_l = lse[:, :, 0].cpu().numpy().reshape(B * Hq)
    compare(got_o, got_l, o_ref, lse_ref, what)


def test_decode_group_of_16():
    """Hq / Hkv = 16: four blocks of four query heads per KV head."""
    lens = [4100, 1, 2048, 777]
    q, k, v, L = workloads.decode_inputs(len(lens), 64, 4, 4100, 128, 0, 0, seed=610, seqlens=lens)
    o, lse = _native.decode(q.cuda(), k.cuda(), v.cuda(), L.cuda(), 0.1, 1024)
    assert _native.attn_get_device_status() == 0
    _decode_check(q, k, v, L, 0.1, o, lse, "decode Hq64 Hkv4")


def test_paged_smallest_page_largest_chunk():
    """64-key pages with 4096-key splits: 66 pages listed per split."""
    lens = [8192, 4097, 63, 6000]
    q, k, v, L = workloads.decode_inputs(len(lens), 8, 2, 8192, 128, 0, 0, seed=611, seqlens=lens)
    kp, vp, bt = workloads.page_cache(k, v, 64, seed=9)
    o, lse = _native.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), bt.cuda(), L.cuda(), 0.125, chunk=4096)
    assert _native.attn_get_device_status() == 0
    _decode_check(q, k, v, L, 0.125, o, lse, "paged page64 chunk4096")


@pytest.mark.parametrize("causal,window", [(2, (50, 0)), (0, (31, 31))])
def test_kvcache_window_head_dim_64(causal, window):
    B, Hq, Hkv, Nq, S, d = 3, 6, 2, 90, 600, 64
    lens = [600, 200, 90]
    q = workloads.prefill_inputs(B, Hq, Hkv, Nq, 1, d, seed=612)[0]
    _, k, v, L = workloads.decode_inputs(B, Hq, Hkv, S, d, 0, 0, seed=613, seqlens=lens)
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward_kvcache(q.cuda(), k.cuda(), v.cuda(), L.cuda(), causal, scale, window=window)
    assert _native.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale, kv_len=L.numpy(), window=window)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "kvcache d64 window %s" % (window,))
