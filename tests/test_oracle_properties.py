"""Properties of the fp64 oracle that hold at any shape, checked on randomly
drawn small problems (CPU only).

For every query row, over the keys the row may see:

- softmax weights are positive and sum to one, so each column of O lies
  between the smallest and the largest visible V entry of that column, and
  a constant V comes back unchanged ("FlashAttention: Part 2", section 1.3:
  the softmax of a score row is a probability distribution);
- log-sum-exp bounds: max_j s_j <= LSE <= max_j s_j + ln(count);
- a row that sees no key has O = 0 and LSE = -inf (the reading taken for
  empty rows).

Which keys a row sees follows the mask readings: keys at or past the
sequence's length are never visible; causal 1 aligns top-left (j <= i),
causal 2 bottom-right (j <= i + L - Nq); a window (left, right) is aligned
bottom-right (L - Nq + i - left <= j <= L - Nq + i + right, a negative side
unbounded) and intersects the causal mask.  Shapes, group sizes, masks,
windows, cache lengths, scales and values are drawn by hypothesis.
"""
import math

import numpy as np
import pytest
import torch

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


def visible(Nq, Nk, L, causal, window):
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    pos = i + L - Nq
    vis = (j < L) & (i >= 0)
    if causal == 1:
        vis = vis & (j <= i)
    elif causal == 2:
        vis = vis & (j <= pos)
    if window is not None:
        wl, wr = window
        if wl >= 0:
            vis = vis & (j >= pos - wl)
        if wr >= 0:
            vis = vis & (j <= pos + wr)
    return vis


def bf16(rng, shape, amp):
    return torch.from_numpy(rng.standard_normal(shape) * amp).to(torch.bfloat16)


@settings(max_examples=120, deadline=None, derandomize=True)
@given(B=st.integers(1, 2), G=st.sampled_from([1, 2, 3]), Hkv=st.integers(1, 2), Nq=st.integers(1, 40),
       Nk=st.integers(1, 40), d=st.sampled_from([4, 8, 16]), causal=st.sampled_from([0, 1, 2]),
       window=st.one_of(st.none(), st.tuples(st.integers(-1, 45), st.integers(-1, 45))),
       use_lens=st.booleans(), scale=st.floats(-2.0, 2.0, allow_nan=False), amp=st.sampled_from([0.5, 1.0, 4.0]),
       seed=st.integers(0, 2 ** 31 - 1))
def test_weights_form_a_distribution_over_the_visible_keys(B, G, Hkv, Nq, Nk, d, causal, window, use_lens, scale,
                                                          amp, seed):
    rng = np.random.default_rng(seed)
    Hq = G * Hkv
    q = bf16(rng, (B, Nq, Hq, d), amp)
    k = bf16(rng, (B, Nk, Hkv, d), amp)
    v = bf16(rng, (B, Nk, Hkv, d), 1.0)
    lens = [int(x) for x in rng.integers(0, Nk + 1, B)] if use_lens else [Nk] * B
    o, lse = oracle.attn_fwd(q, k, v, causal, scale, kv_len=lens if use_lens else None, window=window)
    c = torch.full_like(v, 3.25)  # exactly representable in bf16
    oc, _ = oracle.attn_fwd(q, k, c, causal, scale, kv_len=lens if use_lens else None, window=window)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for b in range(B):
        vis = visible(Nq, Nk, lens[b], causal, window)
        for h in range(Hq):
            g = h // G  # contiguous groups of query heads share a KV head
            s = scale * (qd[b, :, h] @ kd[b, :, g].T)
            for i in range(Nq):
                cols = np.flatnonzero(vis[i])
                if cols.size == 0:
                    assert np.all(o[b, i, h] == 0.0) and lse[b, h, i] == -math.inf
                    assert np.all(oc[b, i, h] == 0.0)
                    continue
                m = s[i, cols].max()
                tol = 1e-12 * max(1.0, abs(m))  # the two sides sum the dot products in different orders
                assert m - tol <= lse[b, h, i] <= m + math.log(cols.size) + tol
                lo = vd[b, cols, g].min(axis=0)
                hi = vd[b, cols, g].max(axis=0)
                assert np.all(o[b, i, h] >= lo - 1e-12) and np.all(o[b, i, h] <= hi + 1e-12)
                np.testing.assert_allclose(oc[b, i, h], 3.25, rtol=0, atol=1e-12)
