"""GPU parity: attn_fwd_kvcache (a block of Nq query rows against a KV cache
with a length per sequence; CUDA through the C ABI) against the fp64 CPU
oracle with the same cache lengths.  Cache positions at or past a
sequence's length hold NaN, so any read of them into the result would
show (the kernel clears them in the last V tile it loads)."""
import math

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


def _inputs(B, Hq, Hkv, Nq, S, d, lens, seed):
    q = workloads.prefill_inputs(B, Hq, Hkv, Nq, 1, d, seed=seed)[0]
    _, k, v, L = workloads.decode_inputs(B, Hq, Hkv, S, d, 0, 0, seed=seed + 1, seqlens=lens)
    return q, k, v, L


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("B,Hq,Hkv,Nq,S,d,lens", [
    (3, 8, 2, 77, 1000, 128, [1000, 333, 128]),       # GQA head pairs, ragged query block
    (2, 6, 2, 300, 700, 64, [700, 301]),             # group of 3: row-tile pairs, d = 64
    (4, 4, 4, 1, 520, 128, [520, 1, 0, 257]),        # several decode-like single rows, an empty cache
    (2, 4, 1, 129, 400, 128, [100, 400]),            # a cache shorter than the query block
])
def test_kvcache_parity(B, Hq, Hkv, Nq, S, d, lens, causal):
    q, k, v, L = _inputs(B, Hq, Hkv, Nq, S, d, lens, seed=60 + Nq)
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward_kvcache(q.cuda(), k.cuda(), v.cuda(), L.cuda(), causal, scale)
    assert _native.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale, kv_len=L.numpy())
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
            "kvcache B%d Hq%d Hkv%d Nq%d S%d d%d causal%d" % (B, Hq, Hkv, Nq, S, d, causal))


def test_kvcache_full_length_equals_attn_fwd():
    """With every cache full, the call is attn_fwd over the whole cache."""
    B, Hq, Hkv, Nq, S, d = 2, 8, 2, 200, 384, 128
    q, k, v, _ = _inputs(B, Hq, Hkv, Nq, S, d, [S, S], seed=70)
    L = torch.full((B,), S, dtype=torch.int32)
    for causal in (0, 1, 2):
        a = _native.forward_kvcache(q.cuda(), k.cuda(), v.cuda(), L.cuda(), causal, 0.09)
        b = _native.forward(q.cuda(), k.cuda(), v.cuda(), causal, 0.09)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_kvcache_bad_length_is_reported():
    q, k, v, _ = _inputs(2, 4, 2, 64, 256, 64, [256, 10], seed=71)
    L = torch.tensor([256, 300], dtype=torch.int32)
    _native.attn_get_device_status()
    _native.forward_kvcache(q.cuda(), k.cuda(), v.cuda(), L.cuda(), 2, 0.125)
    assert _native.attn_get_device_status() == _native.ATTN_ERR_DEVICE_ARG
