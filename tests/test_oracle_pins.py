"""Pins for the fp64 CPU oracle (no GPU).

The oracle is the plain definition of exact attention forward
("FlashAttention: Part 2", chizkidd.github.io, section 2.1: softmax(QK^T/sqrt d)V;
section 1.3: one log-sum-exp per query row).  It is pinned here to things
other than itself: hand-derived closed forms (tests/golden), closed-form
special cases, invariants of the mathematics, brute force in pure Python with
exactly rounded sums, and torch's own fp64 CPU scaled_dot_product_attention
(section 2.1 names that API).  Each plausible slip -- a dropped scale, a sign,
swapped K/V, a transposed operand, a causal off-by-one, a modulo GQA map, a
log2 LSE -- fails at least one test below.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_14_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
_MATH = {n: getattr(math, n) for n in ("log", "exp", "tanh", "sqrt")}
_MATH["inf"] = math.inf


def _closed(expr):
    return float(eval(str(expr), {"__builtins__": {}}, _MATH))


def _bf16(nested):
    t = torch.tensor(np.array(nested, dtype=object).astype(float), dtype=torch.float32)
    out = t.to(torch.bfloat16)
    fin = torch.isfinite(t)
    assert torch.equal(out.float()[fin], t[fin]), "fixture value not exact in bf16"
    return out


def _rand(B, Hq, Hkv, Nq, Nk, d, seed, amp=1.0):
    gen = torch.Generator().manual_seed(seed)
    f = lambda *s: (torch.randn(s, generator=gen) * amp).to(torch.bfloat16)
    return f(B, Nq, Hq, d), f(B, Nk, Hkv, d), f(B, Nk, Hkv, d)


def _cases():
    with open(GOLDEN) as fh:
        return json.load(fh)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_derived_cases(case):
    q, k, v = _bf16(case["q"]), _bf16(case["k"]), _bf16(case["v"])
    o, lse = oracle.attn_fwd(q, k, v, case["causal"], _closed(case["scale"]), kv_len=case["kv_len"])
    want_o = np.vectorize(_closed)(np.array(case["o"], dtype=object)).astype(float)
    want_lse = np.vectorize(_closed)(np.array(case["lse"], dtype=object)).astype(float)
    np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 33, 33, 16), (2, 4, 2, 17, 40, 8), (1, 8, 1, 5, 70, 64)])
def test_value_ones_gives_ones(shape, causal):
    """With V = 1 the output is the row sum of P, which softmax makes exactly 1."""
    B, Hq, Hkv, Nq, Nk, d = shape
    q, k, _ = _rand(B, Hq, Hkv, Nq, Nk, d, seed=11)
    v = torch.ones((B, Nk, Hkv, d), dtype=torch.bfloat16)
    o, lse = oracle.attn_fwd(q, k, v, causal, 1 / math.sqrt(d))
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("use_scale_zero", [False, True])
def test_zero_scores_give_mean_of_visible_values(causal, use_scale_zero):
    """Q = 0 (or scale = 0): every score is 0, so O is the plain mean of the
    visible V rows and LSE = ln(number of visible keys)."""
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 9, 9, 8
    q, k, v = _rand(B, Hq, Hkv, Nq, Nk, d, seed=12)
    kv_len = [9, 6]
    if use_scale_zero:
        scale = 0.0
    else:
        q = torch.zeros_like(q)
        scale = 0.125
    o, lse = oracle.attn_fwd(q, k, v, causal, scale, kv_len=kv_len)
    vd = v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(Nq):
                n = min(kv_len[b], i + 1) if causal else kv_len[b]
                np.testing.assert_allclose(o[b, i, h], vd[b, :n, g].mean(axis=0), rtol=0, atol=1e-12)
                assert abs(lse[b, h, i] - math.log(n)) < 1e-13


def test_dominant_key_returns_its_value_row():
    """A key whose score beats all others by > 50 takes all the weight."""
    B, Hq, Hkv, N, d = 1, 2, 1, 50, 64
    q, k, v = _rand(B, Hq, Hkv, N, N, d, seed=13)
    q = torch.zeros_like(q)
    q[0, :, :, 0] = 8.0
    k = k.clone()
    star = {7: 31, 20: 3, 49: 49}
    for j in star.values():
        k[0, j, 0, 0] = 64.0  # score 8*64/8 = 64; the rest are N(0,1)
    o, lse = oracle.attn_fwd(q, k, v, False, 1 / 8)
    # every row sees the same three dominant keys (31, 3, 49) tied at 64
    want = v[0, [31, 3, 49], 0].double().numpy().mean(axis=0)
    for i in range(N):
        for h in range(Hq):
            np.testing.assert_allclose(o[0, i, h], want, rtol=0, atol=1e-12)
            assert abs(lse[0, h, i] - (64 + math.log(3))) < 1e-9


def test_single_dominant_key_per_row():
    d = 16
    N = 16
    q = torch.zeros((1, N, 1, d), dtype=torch.bfloat16)
    k = torch.zeros((1, N, 1, d), dtype=torch.bfloat16)
    gen = torch.Generator().manual_seed(14)
    v = torch.randn((1, N, 1, d), generator=gen).to(torch.bfloat16)
    perm = torch.randperm(N, generator=gen)
    for i in range(N):  # row i points at key perm[i] only, score 60 vs 0
        q[0, i, 0, i % d] = 8.0
        k[0, perm[i], 0, i % d] = 30.0
    o, lse = oracle.attn_fwd(q, k, v, False, 0.25)
    for i in range(N):
        np.testing.assert_allclose(o[0, i, 0], v[0, perm[i], 0].double().numpy(), rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i] - (60 + math.log1p((N - 1) * math.exp(-60)))) < 1e-12


def test_causal_row_zero_is_v0():
    B, Hq, Hkv, N, d = 2, 4, 4, 20, 32
    q, k, v = _rand(B, Hq, Hkv, N, N, d, seed=15)
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attn_fwd(q, k, v, True, scale)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(o[b, 0, h], vd[b, 0, h])
            s00 = scale * math.fsum(qd[b, 0, h] * kd[b, 0, h])
            assert abs(lse[b, h, 0] - s00) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_exactly_rounded_sums(causal):
    """Pure-Python brute force with math.fsum on a small case."""
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 6, 9, 5
    q, k, v = _rand(B, Hq, Hkv, Nq, Nk, d, seed=16)
    scale = 0.7
    o, lse = oracle.attn_fwd(q, k, v, causal, scale)
    qd, kd, vd = q.double().tolist(), k.double().tolist(), v.double().tolist()
    for h in range(Hq):
        for i in range(Nq):
            keys = [j for j in range(Nk) if (not causal or j <= i)]
            s = [scale * math.fsum(qd[0][i][h][t] * kd[0][j][0][t] for t in range(d)) for j in keys]
            L = math.log(math.fsum(math.exp(x) for x in s))
            assert abs(lse[0, h, i] - L) < 1e-13
            for t in range(d):
                ot = math.fsum(math.exp(x - L) * vd[0][j][0][t] for x, j in zip(s, keys))
                assert abs(o[0, i, h, t] - ot) < 1e-13


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 2, 16, 16, 64, False),
    (2, 4, 4, 31, 31, 32, True),
    (1, 8, 2, 20, 20, 16, True),     # GQA
    (2, 4, 1, 7, 29, 16, True),      # Nq < Nk, top-left causal
    (1, 2, 2, 29, 7, 16, True),      # Nq > Nk
    (1, 4, 2, 1, 50, 128, False),    # decode-like row
])
def test_matches_torch_sdpa_fp64(B, Hq, Hkv, Nq, Nk, d, causal):
    """torch.nn.functional.scaled_dot_product_attention on the CPU in fp64
    (math backend, top-left is_causal, enable_gqa) -- an independent library."""
    q, k, v = _rand(B, Hq, Hkv, Nq, Nk, d, seed=17)
    scale = 1 / math.sqrt(d)
    o, _ = oracle.attn_fwd(q, k, v, causal, scale)
    tq, tk, tv = (x.double().permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, is_causal=causal, scale=scale, enable_gqa=(Hq != Hkv))
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_matches_torch_sdpa_with_cache_lengths():
    B, Hq, Hkv, Nk, d = 3, 4, 2, 40, 32
    q, k, v = _rand(B, Hq, Hkv, 1, Nk, d, seed=18)
    kv_len = [40, 1, 23]
    o, _ = oracle.attn_fwd(q, k, v, False, 0.2, kv_len=kv_len)
    mask = torch.arange(Nk)[None, :] < torch.tensor(kv_len)[:, None]
    tq, tk, tv = (x.double().permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=mask[:, None, None, :], scale=0.2, enable_gqa=True)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_key_permutation_invariance():
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 2, 12, 37, 16
    q, k, v = _rand(B, Hq, Hkv, Nq, Nk, d, seed=19)
    perm = torch.randperm(Nk, generator=torch.Generator().manual_seed(5))
    o1, l1 = oracle.attn_fwd(q, k, v, False, 0.3)
    o2, l2 = oracle.attn_fwd(q, k[:, perm], v[:, perm], False, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_affine_in_values():
    """O(Q, K, 2V + 1) = 2 O(Q, K, V) + 1 because rows of P sum to one.
    V holds small integers so 2V + 1 stays exact in bf16."""
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 10, 10, 8
    q, k, _ = _rand(B, Hq, Hkv, Nq, Nk, d, seed=20)
    gen = torch.Generator().manual_seed(21)
    v = torch.randint(-8, 9, (B, Nk, Hkv, d), generator=gen).to(torch.bfloat16)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd(q, k, v, causal, 0.35)
        o2, l2 = oracle.attn_fwd(q, k, (2 * v.float() + 1).to(torch.bfloat16), causal, 0.35)
        np.testing.assert_allclose(o2, 2 * o1 + 1, rtol=0, atol=1e-12)
        assert np.array_equal(l1, l2)


def test_gqa_equals_mha_with_repeated_kv_heads():
    B, Hq, Hkv, N, d = 2, 8, 2, 19, 16
    q, k, v = _rand(B, Hq, Hkv, N, N, d, seed=22)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd(q, k, v, causal, 0.25)
        rep = Hq // Hkv
        o2, l2 = oracle.attn_fwd(q, k.repeat_interleave(rep, dim=2), v.repeat_interleave(rep, dim=2),
                                 causal, 0.25)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_row_subset_and_thread_count_do_not_change_bits():
    B, Hq, Hkv, N, d = 2, 4, 2, 33, 32
    q, k, v = _rand(B, Hq, Hkv, N, N, d, seed=23)
    o_full, l_full = oracle.attn_fwd(q, k, v, True, 0.2, n_threads=1)
    o_mt, l_mt = oracle.attn_fwd(q, k, v, True, 0.2, n_threads=7)
    assert np.array_equal(o_full, o_mt) and np.array_equal(l_full, l_mt)
    rows = workloads.sample_rows(B, Hq, N, 25, seed=3, force=[(0, 0, 0), (1, 3, 32)])
    o_r, l_r = oracle.attn_rows(q, k, v, rows, True, 0.2)
    for r, (b, h, i) in enumerate(rows):
        assert np.array_equal(o_r[r], o_full[b, i, h])
        assert l_r[r] == l_full[b, h, i]


def test_rejects_bad_arguments():
    q, k, v = _rand(1, 3, 2, 4, 4, 8, seed=24)
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, False, 0.1)            # 3 query heads over 2 KV heads
    q, k, v = _rand(1, 2, 2, 4, 4, 8, seed=24)
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, False, 0.1, kv_len=[5])  # longer than the cache


def test_nan_beyond_cache_length_is_never_read():
    w = workloads.decode_inputs(3, 4, 2, 64, 16, 1, 64, seed=25, seqlens=[64, 1, 40])
    q, k, v, L = w
    o, lse = oracle.attn_fwd(q, k, v, False, 0.25, kv_len=L.numpy())
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert torch.isnan(k[1, 1:]).all()


def test_paged_cache_definition_by_hand():
    """Page table semantics on a hand example: key k of sequence b is row
    k % page_size of page block_table[b, k // page_size]."""
    pages = torch.arange(6, dtype=torch.float32).reshape(3, 2, 1, 1)   # page p holds 2p, 2p+1
    bt = torch.tensor([[2, 0], [1, 2]], dtype=torch.int32)
    got = oracle.paged_to_contiguous(pages, bt)[..., 0, 0]
    assert got.tolist() == [[4.0, 5.0, 0.0, 1.0], [2.0, 3.0, 4.0, 5.0]]


def test_paged_cache_round_trip():
    """Scattering a cache into shuffled pages (the input generator) and
    gathering it back (the oracle's definition) returns the cache."""
    from exact_io_aware_14_gb300 import workloads as W
    q, k, v, L = W.decode_inputs(3, 4, 2, 300, 64, 0, 0, seed=1, seqlens=[300, 17, 0])
    for ps in (64, 256):
        kp, vp, bt = W.page_cache(k, v, ps, seed=ps)
        assert sorted(set(bt.reshape(-1).tolist())) == sorted(bt.reshape(-1).tolist())   # pages not shared
        kc = oracle.paged_to_contiguous(kp, bt)[:, :300]
        vc = oracle.paged_to_contiguous(vp, bt)[:, :300]
        assert torch.equal(torch.nan_to_num(kc.float(), nan=7.0), torch.nan_to_num(k.float(), nan=7.0))
        assert torch.equal(torch.nan_to_num(vc.float(), nan=7.0), torch.nan_to_num(v.float(), nan=7.0))


@pytest.mark.parametrize("Nq,Nk", [(7, 29), (29, 7), (16, 16), (1, 50)])
def test_bottom_right_causal_matches_sdpa_with_its_mask(Nq, Nk):
    """causal=2 (aligned bottom-right: row i sees keys j <= i + Nk - Nq)
    against torch's fp64 SDPA with that boolean mask written out; rows that
    see no key are O = 0, LSE = -inf."""
    B, Hq, Hkv, d = 2, 4, 2, 16
    q, k, v = _rand(B, Hq, Hkv, Nq, Nk, d, seed=21)
    o, lse = oracle.attn_fwd(q, k, v, 2, 0.25)
    mask = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    seen = mask.any(dim=1)
    tq, tk, tv = (x.double().permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=mask, scale=0.25, enable_gqa=True).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(o[:, seen.numpy()], ref[:, seen.numpy()], rtol=0, atol=1e-12)
    assert (o[:, ~seen.numpy()] == 0).all()
    assert np.isneginf(lse[:, :, ~seen.numpy()]).all()


def test_bottom_right_causal_special_cases():
    """Nq == Nk: bottom-right is top-left; Nq == 1: the one row sees every key."""
    q, k, v = _rand(1, 2, 2, 24, 24, 16, seed=22)
    a = oracle.attn_fwd(q, k, v, 1, 0.3)
    b = oracle.attn_fwd(q, k, v, 2, 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    q1, k1, v1 = _rand(1, 2, 2, 1, 37, 16, seed=23)
    c = oracle.attn_fwd(q1, k1, v1, 2, 0.3)
    e = oracle.attn_fwd(q1, k1, v1, False, 0.3)
    assert np.array_equal(c[0], e[0]) and np.array_equal(c[1], e[1])
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, 3, 0.3)


def test_bottom_right_with_cache_lengths_is_prefill_against_a_cache():
    """With kv_len, bottom-right puts query row i at cache position
    L_b - Nq + i: the same as the rows of one causal pass over the whole
    cache (top-left, Nq = Nk = L_b) that hold the last Nq positions."""
    B, Hq, Hkv, Nq, S, d = 2, 4, 2, 5, 30, 16
    q, k, v = _rand(B, Hq, Hkv, S, S, d, seed=24)
    kv_len = [30, 12]
    for b, L in enumerate(kv_len):
        o_full, l_full = oracle.attn_fwd(q[b:b + 1, :L], k[b:b + 1, :L], v[b:b + 1, :L], True, 0.2)
        qs = q[b:b + 1, L - Nq:L].contiguous()
        o_tail, l_tail = oracle.attn_fwd(qs, k[b:b + 1], v[b:b + 1], 2, 0.2, kv_len=[L])
        np.testing.assert_allclose(o_tail, o_full[:, L - Nq:L], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_tail, l_full[:, :, L - Nq:L], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- local window
# "FlashAttention: Part 2", section 3.2: local attention keeps i -> j only for
# |i - j| <= w; the window is given as (left, right), positions aligned
# bottom-right (row i at key position i + L - Nq), a negative side unbounded.

def _band(Nq, Nk, wl, wr):
    """Boolean [Nq, Nk] mask of the window, written out with torch."""
    pos = torch.arange(Nq)[:, None] + (Nk - Nq)
    j = torch.arange(Nk)[None, :]
    m = torch.ones(Nq, Nk, dtype=torch.bool)
    if wl >= 0:
        m &= j >= pos - wl
    if wr >= 0:
        m &= j <= pos + wr
    return m


@pytest.mark.parametrize("Nq,Nk,wl,wr", [(16, 16, 3, 3), (16, 16, 2, 5), (9, 31, 4, 0), (31, 9, 6, 2),
                                         (12, 40, -1, 3), (12, 40, 7, -1), (20, 20, 0, -1)])
def test_window_matches_sdpa_with_its_band_mask(Nq, Nk, wl, wr):
    """torch's fp64 CPU SDPA with the band |i - j| <= w (one bound per side)
    as an explicit boolean mask; rows whose band holds no key: O = 0, LSE = -inf."""
    B, Hq, Hkv, d = 2, 4, 2, 16
    q, k, v = _rand(B, Hq, Hkv, Nq, Nk, d, seed=31 + Nq + wl)
    o, lse = oracle.attn_fwd(q, k, v, 0, 0.25, window=(wl, wr))
    mask = _band(Nq, Nk, wl, wr)
    seen = mask.any(dim=1).numpy()
    tq, tk, tv = (x.double().permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=mask, scale=0.25, enable_gqa=True).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(o[:, seen], ref[:, seen], rtol=0, atol=1e-12)
    assert (o[:, ~seen] == 0).all() and np.isneginf(lse[:, :, ~seen]).all()


def test_window_zero_is_the_diagonal():
    """Window (0, 0), Nq == Nk: row i sees key i alone, so O_i = v_i exactly
    and LSE_i is its one score."""
    q, k, v = _rand(1, 2, 2, 20, 20, 16, seed=32)
    o, lse = oracle.attn_fwd(q, k, v, 0, 0.4, window=(0, 0))
    qd, kd = q.double().numpy(), k.double().numpy()
    assert np.array_equal(o, v.double().numpy())
    s = 0.4 * np.einsum("bihd,bihd->bhi", qd, kd)
    np.testing.assert_allclose(lse, s, rtol=0, atol=1e-13)


def test_window_one_left_is_a_two_key_softmax():
    """Window (1, 0): row i >= 1 sees keys i-1 and i, weights
    sigma(s_i - s_{i-1}) on v_i; row 0 sees key 0 alone."""
    q, k, v = _rand(1, 1, 1, 15, 15, 8, seed=33)
    o, lse = oracle.attn_fwd(q, k, v, 0, 0.5, window=(1, 0))
    qd, kd, vd = (x.double().numpy()[0, :, 0] for x in (q, k, v))
    s = 0.5 * np.einsum("id,jd->ij", qd, kd)
    np.testing.assert_array_equal(o[0, 0, 0], vd[0])
    for i in range(1, 15):
        w = 1.0 / (1.0 + math.exp(s[i, i - 1] - s[i, i]))
        np.testing.assert_allclose(o[0, i, 0], w * vd[i] + (1 - w) * vd[i - 1], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, i], np.logaddexp(s[i, i], s[i, i - 1]), rtol=0, atol=1e-13)


def test_window_reductions():
    """A right side of 0 is bottom-right causal; sides at least the sequence
    long are no window; window and causal masks intersect."""
    q, k, v = _rand(1, 2, 1, 13, 29, 16, seed=34)
    a = oracle.attn_fwd(q, k, v, 2, 0.3)
    b = oracle.attn_fwd(q, k, v, 0, 0.3, window=(-1, 0))
    c = oracle.attn_fwd(q, k, v, 0, 0.3, window=(28 + 13, 0))
    assert all(np.array_equal(x, y) for x, y in zip(a, b)) and all(np.array_equal(x, y) for x, y in zip(a, c))
    e = oracle.attn_fwd(q, k, v, 0, 0.3)
    f = oracle.attn_fwd(q, k, v, 0, 0.3, window=(100, 100))
    assert all(np.array_equal(x, y) for x, y in zip(e, f))
    g = oracle.attn_fwd(q, k, v, 2, 0.3, window=(5, 9))
    h = oracle.attn_fwd(q, k, v, 0, 0.3, window=(5, 0))
    assert all(np.array_equal(x, y) for x, y in zip(g, h))


def test_window_query_block_at_the_end_is_the_full_pass():
    """Bottom-right alignment puts a query block of Nq rows at the last Nq
    positions of the cache: its rows equal those rows of one windowed pass
    with Nq = Nk = L (both with and without per-sequence lengths)."""
    B, Hq, Hkv, Nq, S, d = 2, 4, 2, 6, 33, 16
    q, k, v = _rand(B, Hq, Hkv, S, S, d, seed=35)
    for wl, wr in [(4, 0), (7, 2), (3, -1)]:
        for b, L in enumerate([33, 14]):
            o_full, l_full = oracle.attn_fwd(q[b:b + 1, :L], k[b:b + 1, :L], v[b:b + 1, :L], 0, 0.2, window=(wl, wr))
            qs = q[b:b + 1, L - Nq:L].contiguous()
            o_t, l_t = oracle.attn_fwd(qs, k[b:b + 1], v[b:b + 1], 0, 0.2, kv_len=[L], window=(wl, wr))
            np.testing.assert_allclose(o_t, o_full[:, L - Nq:L], rtol=0, atol=1e-13)
            np.testing.assert_allclose(l_t, l_full[:, :, L - Nq:L], rtol=0, atol=1e-13)


def test_window_never_reads_keys_outside_it():
    """Keys and values outside every row's band may hold NaN: nothing changes."""
    Nq = Nk = 24
    q, k, v = _rand(1, 2, 2, Nq, Nk, 16, seed=36)
    wl, wr = 3, 1
    a = oracle.attn_fwd(q, k, v, 0, 0.3, window=(wl, wr))
    # rows 10..13 only: keys 7..14 are in some band, the rest are poisoned
    rows = np.array([(0, h, i) for h in range(2) for i in range(10, 14)], dtype=np.int32)
    k2, v2 = k.clone(), v.clone()
    for x in (k2, v2):
        x[:, :7] = float("nan")
        x[:, 15:] = float("nan")
    o_r, l_r = oracle.attn_rows(q, k2, v2, rows, 0, 0.3, window=(wl, wr))
    exp_o = np.stack([a[0][0, i, h] for _, h, i in rows])
    exp_l = np.array([a[1][0, h, i] for _, h, i in rows])
    assert np.array_equal(o_r, exp_o) and np.array_equal(l_r, exp_l)
