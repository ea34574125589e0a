"""GPU parity at the largest sizes the tests reach.

- Prefill whose q and o hold more than 2^31 elements (135,000 rows x 128
  query heads x d 128, GQA onto 8 KV heads, causal): rows whose output
  offsets lie past 2^31 elements are checked against the oracle, so any
  32-bit address arithmetic would show.
- Decode against a single cache of 1,048,909 keys: 1025 splits of 1024 keys
  merged by one combine.

Inputs are drawn on the GPU (seeded CUDA generator, N(0, 1) rounded to bf16,
in slices to bound the fp32 transient); the oracle gets the CPU copies of
K and V and of the sampled query rows.  A sampled causal row i is computed by
the oracle as one unmasked query against the first i + 1 keys (the causal
mask written as a cache length).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_14_gb300 import _native, build as native_build
from tests._parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    native_build.build()
    _native.lib()
    torch.cuda.init()


def _randn_bf16(shape, gen):
    x = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    flat = x.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        n = min(step, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=gen, device="cuda").to(torch.bfloat16)
    return x


def test_prefill_beyond_2_31_elements():
    B, Hq, Hkv, N, d = 1, 128, 8, 135000, 128
    gen = torch.Generator(device="cuda").manual_seed(11)
    q = _randn_bf16((B, N, Hq, d), gen)
    k = _randn_bf16((B, N, Hkv, d), gen)
    v = _randn_bf16((B, N, Hkv, d), gen)
    assert q.numel() > 2 ** 31
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward(q, k, v, True, scale)
    torch.cuda.synchronize()
    assert _native.attn_get_device_status() == 0
    first_past = 2 ** 31 // (Hq * d)  # the first row whose output offset passes 2^31 elements
    pick = np.random.default_rng(5)
    rows = [(Hq - 1, N - 1), (0, first_past), (Hq - 1, first_past - 1), (77, N - 129), (3, 0)]
    rows += [(int(h), int(i)) for h, i in zip(pick.integers(0, Hq, 24), pick.integers(first_past, N, 24))]
    rows += [(int(h), int(i)) for h, i in zip(pick.integers(0, Hq, 8), pick.integers(0, first_past, 8))]
    kc, vc = k.cpu(), v.cpu()
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for h, i in rows:
        qs = q[:, i:i + 1].cpu()
        ro, rl = oracle.attn_rows(qs, kc, vc, [(0, h, 0)], False, scale, kv_len=[i + 1])
        ref_o.append(ro[0])
        ref_l.append(rl[0])
        got_o.append(o[0, i, h].float().cpu().numpy())
        got_l.append(float(lse[0, h, i]))
    compare(np.stack(got_o), np.array(got_l), np.stack(ref_o), np.array(ref_l), "prefill 2.2e9-element q/o")


def test_decode_million_key_cache():
    B, Hq, Hkv, d, S, chunk = 1, 16, 8, 128, 1048909, 1024
    gen = torch.Generator(device="cuda").manual_seed(12)
    q = _randn_bf16((B, 1, Hq, d), gen)
    k = _randn_bf16((B, S, Hkv, d), gen)
    v = _randn_bf16((B, S, Hkv, d), gen)
    seqlens = torch.tensor([S], dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    o, lse = _native.decode(q, k, v, seqlens, scale, chunk)
    torch.cuda.synchronize()
    assert _native.attn_get_device_status() == 0
    rows = np.array([(0, h, 0) for h in range(Hq)], dtype=np.int32)
    ro, rl = oracle.attn_rows(q.cpu(), k.cpu(), v.cpu(), rows, False, scale)
    compare(o[0, 0].float().cpu().numpy(), lse[0, :, 0].cpu().numpy(), ro, rl, "decode 1M keys, 1025 splits")
