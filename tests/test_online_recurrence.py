"""The tiled online-softmax algebra the GPU kernels rely on, checked on the
CPU against the naive fp64 oracle (no GPU).

"FlashAttention: Part 2" (chizkidd.github.io), section 6.2: the running state
(m, l, a) with rescale alpha = exp(m - m') reproduces the full-row softmax;
"Trace FlashAttention's evolution through plain PyTorch code": FA2 defers the
normalisation to the end and FA4 rescales only when needed; pyshine.com
flash-attention tour, "Why You Need This": split-KV decode combines partial
results.  All of these must reach the naive definition up to rounding.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import online


def _rand(Nq, Nk, d, seed):
    gen = torch.Generator().manual_seed(seed)
    f = lambda *s: torch.randn(s, generator=gen).to(torch.bfloat16)
    return f(1, Nq, 1, d), f(1, Nk, 1, d), f(1, Nk, 1, d)


def _head(x):
    return x[0, :, 0].double().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tile", [1, 2, 7, 16, 64, 100])
@pytest.mark.parametrize("variant", ["fa1", "fa2", "fa4"])
def test_online_matches_naive(causal, tile, variant):
    Nq = Nk = 45
    d = 16
    q, k, v = _rand(Nq, Nk, d, seed=40 + tile)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    o, lse = online.online_attention(
        _head(q), _head(k), _head(v), scale, causal=causal, tile=tile,
        conditional_rescale=(variant == "fa4"), normalise_each_tile=(variant == "fa1"))
    np.testing.assert_allclose(o, o_ref[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=0, atol=1e-12)


def test_conditional_rescale_is_bitwise_identical_to_always_rescaling():
    """Skipping the rescale exactly when m' == m multiplies by exp(0) = 1
    in the other form, so the two forms agree bit for bit."""
    q, k, v = _rand(64, 300, 32, seed=50)
    for causal in (False, True):
        a = online.online_attention(_head(q), _head(k), _head(v), 0.2, causal, 32, conditional_rescale=True)
        b = online.online_attention(_head(q), _head(k), _head(v), 0.2, causal, 32, conditional_rescale=False)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("threshold", [0.0, 8 * math.log(2), 40.0])
@pytest.mark.parametrize("amp", [1.0, 12.0])
def test_thresholded_reference_matches_naive(causal, threshold, amp):
    """Keeping a stale exponent reference until the max rises by more than a
    threshold reaches the same O and LSE (large amp forces moves)."""
    q, k, v = _rand(40, 300, 16, seed=54)
    qd = _head(q) * amp
    qb = torch.from_numpy(qd).to(torch.bfloat16)[None, :, None, :]
    o_ref, lse_ref = oracle.attn_fwd(qb, k, v, causal, 0.25)
    o, lse = online.online_attention(qb[0, :, 0].double().numpy(), _head(k), _head(v), 0.25, causal, 32,
                                     rescale_threshold=threshold)
    np.testing.assert_allclose(o, o_ref[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-14, atol=1e-12)


def test_online_with_cache_length_and_empty_row():
    q, k, v = _rand(3, 50, 8, seed=51)
    for L in (0, 1, 17, 50):
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 0.3, kv_len=[L])
        o, lse = online.online_attention(_head(q), _head(k), _head(v), 0.3, tile=16, kv_len=L)
        np.testing.assert_allclose(o, o_ref[0, :, 0], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isinf(lse), np.isinf(lse_ref[0, 0]))
        fin = np.isfinite(lse)
        np.testing.assert_allclose(lse[fin], lse_ref[0, 0][fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 128, 1000])
@pytest.mark.parametrize("L", [1, 63, 64, 65, 200])
def test_splitkv_combine_matches_unsplit(chunk, L):
    q, k, v = _rand(4, 200, 16, seed=52)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 0.25, kv_len=[L])
    o_s, lse_s = online.splitkv_partials(_head(q), _head(k), _head(v), 0.25, chunk, L)
    assert o_s.shape[0] == -(-L // chunk)
    o, lse = online.combine(o_s, lse_s)
    np.testing.assert_allclose(o, o_ref[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=0, atol=1e-12)


def test_combine_ignores_empty_splits():
    q, k, v = _rand(2, 40, 8, seed=53)
    o_s, lse_s = online.splitkv_partials(_head(q), _head(k), _head(v), 0.5, 16, 40)
    o_s2 = np.concatenate([o_s, np.zeros_like(o_s[:2])])
    lse_s2 = np.concatenate([lse_s, np.full_like(lse_s[:2], -np.inf)])
    a, b = online.combine(o_s, lse_s), online.combine(o_s2, lse_s2)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-15)


@pytest.mark.parametrize("order", ["edge_last", "reversed", "shuffled"])
@pytest.mark.parametrize("threshold", [None, 8 * math.log(2)])
def test_any_tile_order_matches_naive(order, threshold):
    """A unit's key tiles may be visited in another order (the prefill kernel
    visits a window's left-edge tile last): the running state only takes
    maxima and rescaled sums, so every order reaches the naive result, also
    for rows that see nothing in the first tiles visited (causal rows of the
    first tile when it comes last) and with a cache length."""
    Nq, Nk, d, tile = 40, 70, 16, 16  # five key tiles, the last one ragged
    q, k, v = _rand(Nq, Nk, d, seed=77)
    n = -(-Nk // tile)
    orders = {"edge_last": list(range(1, n)) + [0], "reversed": list(range(n))[::-1],
              "shuffled": [int(t) for t in np.random.default_rng(3).permutation(n)]}
    for causal in (False, True):
        for L in (Nk, 53):
            o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 0.3, kv_len=[L])
            o, lse = online.online_attention(_head(q), _head(k), _head(v), 0.3, causal, tile, kv_len=L,
                                             rescale_threshold=threshold, tile_order=orders[order])
            np.testing.assert_allclose(o, o_ref[0, :, 0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=0, atol=1e-12)


def test_tile_order_must_be_a_permutation():
    q, k, v = _rand(4, 40, 8, seed=78)
    with pytest.raises(AssertionError):
        online.online_attention(_head(q), _head(k), _head(v), 0.3, tile=16, tile_order=[0, 0, 1])
