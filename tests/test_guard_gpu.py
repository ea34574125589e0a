"""Out-of-bounds writes, caught without a sanitizer: every output (O, LSE)
and the split-KV workspace is placed inside a larger buffer whose bytes
before and after it hold a fixed pattern.  After the call the pattern must
be intact and the result must equal, bit for bit, the same call on plain
tensors.  The shapes have ragged tails (row counts that are not multiples of
the 128-row tile, keys not multiples of the key tiles) so the epilogue's
partial tiles and the decode's short last splits are exercised.
"""
import math

import pytest
import torch

from exact_io_aware_14_gb300 import _native, build as native_build, workloads

pytestmark = pytest.mark.gpu

PAD_BYTES = 8192
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    native_build.build()
    _native.lib()
    torch.cuda.init()


class Guarded:
    """A tensor of `shape` inside a byte buffer with PAD_BYTES of pattern on each side."""

    def __init__(self, shape, dtype):
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((PAD_BYTES + n + PAD_BYTES,), PATTERN, dtype=torch.uint8, device="cuda")
        self.n = n
        self.t = self.buf[PAD_BYTES:PAD_BYTES + n].view(dtype).view(shape)

    def intact(self):
        head = self.buf[:PAD_BYTES]
        tail = self.buf[PAD_BYTES + self.n:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _prefill_outputs(B, Hq, Nq, d):
    return Guarded((B, Nq, Hq, d), torch.bfloat16), Guarded((B, Hq, Nq), torch.float32)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", [(2, 4, 2, 300, 333, 128), (1, 6, 3, 129, 1000, 64),
                                             (3, 40, 40, 77, 77, 128)])
def test_prefill_writes_stay_inside_o_and_lse(B, Hq, Hkv, Nq, Nk, d):
    q, k, v = (x.cuda() for x in workloads.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=500 + Nq))
    scale = 1 / math.sqrt(d)
    for causal in (0, 1, 2):
        o, lse = _prefill_outputs(B, Hq, Nq, d)
        assert _native.attn_fwd(q, k, v, o.t, lse.t, causal, scale) == _native.ATTN_OK
        ref = _native.forward(q, k, v, causal, scale)
        assert _native.attn_get_device_status() == _native.ATTN_OK
        assert o.intact() and lse.intact(), "write outside O or LSE (causal %d)" % causal
        assert torch.equal(o.t, ref[0]) and torch.equal(lse.t, ref[1])
    o, lse = _prefill_outputs(B, Hq, Nq, d)
    assert _native.attn_fwd_window(q, k, v, o.t, lse.t, 0, (60, 5), scale) == _native.ATTN_OK
    ref = _native.forward_window(q, k, v, 0, (60, 5), scale)
    assert _native.attn_get_device_status() == _native.ATTN_OK
    assert o.intact() and lse.intact()
    assert torch.equal(o.t, ref[0]) and torch.equal(lse.t, ref[1])


def test_kvcache_writes_stay_inside_o_and_lse():
    B, Hq, Hkv, Nq, S, d = 3, 8, 2, 77, 700, 128
    q = workloads.prefill_inputs(B, Hq, Hkv, Nq, 1, d, seed=510)[0].cuda()
    _, k, v, L = workloads.decode_inputs(B, Hq, Hkv, S, d, 0, 0, seed=511, seqlens=[700, 333, 5])
    k, v, L = k.cuda(), v.cuda(), L.cuda()
    o, lse = _prefill_outputs(B, Hq, Nq, d)
    assert _native.attn_fwd_kvcache(q, k, v, L, o.t, lse.t, 2, 0.1) == _native.ATTN_OK
    ref = _native.forward_kvcache(q, k, v, L, 2, 0.1)
    assert _native.attn_get_device_status() == _native.ATTN_OK
    assert o.intact() and lse.intact()
    assert torch.equal(o.t, ref[0]) and torch.equal(lse.t, ref[1])


@pytest.mark.parametrize("paged", [False, True])
def test_decode_writes_stay_inside_outputs_and_workspace(paged):
    B, Hq, Hkv, S, d, chunk = 5, 16, 4, 3000, 128, 512
    q, k, v, L = workloads.decode_inputs(B, Hq, Hkv, S, d, 0, 0, seed=520, seqlens=[3000, 1, 0, 2049, 513])
    q, L = q.cuda(), L.cuda()
    need = _native.attn_splitkv_workspace_size(B, Hq, S if not paged else 3072, d, chunk)
    ws = Guarded((need,), torch.uint8)
    o, lse = Guarded((B, 1, Hq, d), torch.bfloat16), Guarded((B, Hq, 1), torch.float32)
    if paged:
        kp, vp, bt = workloads.page_cache(k, v, 256, seed=7)
        kp, vp, bt = kp.cuda(), vp.cuda(), bt.cuda()
        rc = _native.attn_fwd_splitkv_paged(q, kp, vp, bt, L, o.t, lse.t, 0.09, chunk, ws.t)
        ref = _native.decode_paged(q, kp, vp, bt, L, 0.09, chunk)
    else:
        k, v = k.cuda(), v.cuda()
        rc = _native.attn_fwd_splitkv(q, k, v, L, o.t, lse.t, 0.09, chunk, ws.t)
        ref = _native.decode(q, k, v, L, 0.09, chunk)
    assert rc == _native.ATTN_OK
    assert _native.attn_get_device_status() == _native.ATTN_OK
    assert o.intact() and lse.intact() and ws.intact(), "write outside O, LSE or the workspace"
    assert torch.equal(o.t, ref[0]) and torch.equal(lse.t, ref[1])
