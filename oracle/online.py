"""CPU (numpy, fp64) restatement of the tiled online-softmax recurrence and of
the split-KV partial/combine step -- TEST INFRASTRUCTURE ONLY.

These are not the oracle the GPU is compared against (that is the naive
definition in ``attn_oracle.c``).  They exist so the algebra the GPU kernels
rely on is itself checked against the naive definition on the CPU, in code
that shares nothing with the CUDA sources:

* FA1 tiled online softmax -- "FlashAttention: Part 2" (chizkidd.github.io),
  section 6.2 "FlashAttention Summary": split Q into Q_i and K, V into
  K_j, V_j; per score tile keep the running state (m, l, a) -- running max,
  running sum of exponentials, running un-normalised value sum -- and when a
  tile raises the max to m', rescale l and a by alpha = exp(m - m'); the tile
  is then discarded.
* FA2 deferred normalisation -- "Trace FlashAttention's evolution through
  plain PyTorch code" (beyondmarketintelligence.com): keep ``a`` un-normalised
  and divide by ``l`` once at the end.  The FA1 form (``normalise_each_tile``)
  keeps the output normalised after every tile instead.
* FA4 conditional rescaling -- same post, and "FlashAttention: Part 2"
  sections 1.7/1.8: skip the rescale when the running max did not move.
  Reading taken: skip exactly when m' == m (alpha would be exactly 1).
* Split-KV decode -- pyshine.com flash-attention tour, "Why You Need This":
  with query length one the key range is split across blocks whose partial
  results are then combined.  Each split returns its normalised partial
  output O_s and its log-sum-exp LSE_s; the combine weights split s by
  exp(LSE_s - LSE) with LSE = log sum_s exp(LSE_s).

Arrays: q [Nq, d], k and v [Nk, d], float64; one head.
"""
import numpy as np


def _visible(nq, nk, causal, kv_len):
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    vis = j < (nk if kv_len is None else kv_len)
    if causal:
        vis = vis & (j <= i)
    return vis


def _tile_starts(nk, tile, tile_order):
    starts = list(range(0, nk, tile))
    if tile_order is None:
        return starts
    assert sorted(tile_order) == list(range(len(starts))), "tile_order must be a permutation of the tiles"
    return [starts[t] for t in tile_order]


def online_attention(q, k, v, scale, causal=False, tile=64, kv_len=None,
                     conditional_rescale=True, normalise_each_tile=False, rescale_threshold=None,
                     tile_order=None):
    """Tiled online softmax over key tiles of ``tile`` keys. Returns (O, LSE).

    ``tile_order``: the order in which the key tiles are visited (a
    permutation of their indices; default ascending).  The running state
    (m, l, a) only ever takes a max and rescaled sums, so any order reaches
    the same result up to rounding.

    ``rescale_threshold`` (natural-log units): when given, the exponent
    reference m of a row is moved -- and l, a rescaled -- only when a tile's
    max exceeds it by more than the threshold ("skip the rescale when the
    running max doesn't need it", read as: while the exponentials stay within
    a bounded range); otherwise the stale reference is kept and p may exceed 1.
    """
    if rescale_threshold is not None:
        return _online_thresholded(q, k, v, scale, causal, tile, kv_len, rescale_threshold, tile_order)
    nq, d = q.shape
    nk = k.shape[0]
    vis = _visible(nq, nk, causal, kv_len)
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    a = np.zeros((nq, v.shape[1]))
    for j0 in _tile_starts(nk, tile, tile_order):
        j1 = min(nk, j0 + tile)
        s = scale * (q @ k[j0:j1].T)                      # score tile
        s = np.where(vis[:, j0:j1], s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        # rows that still have seen no visible key keep a zero state
        seen = m_new > -np.inf
        m_safe = np.where(seen, m_new, 0.0)
        p = np.exp(s - m_safe[:, None])                   # exp(-inf) = 0
        if conditional_rescale:
            moved = m_new != m
            alpha = np.ones(nq)
            alpha[moved & seen] = np.exp(m[moved & seen] - m_new[moved & seen])
        else:
            alpha = np.where(seen, np.exp(m - m_safe), 1.0)
        l_new = alpha * l + p.sum(axis=1)
        if normalise_each_tile:
            # FA1 form: a holds the normalised output after every tile
            with np.errstate(invalid="ignore", divide="ignore"):
                a = np.where(seen[:, None],
                             ((alpha * l)[:, None] * a + p @ v[j0:j1]) / l_new[:, None],
                             0.0)
        else:
            a = alpha[:, None] * a + p @ v[j0:j1]
        l = l_new
        m = m_new
    seen = l > 0
    with np.errstate(invalid="ignore", divide="ignore"):
        o = a if normalise_each_tile else np.where(seen[:, None], a / l[:, None], 0.0)
        lse = np.where(seen, m + np.log(l), -np.inf)
    return o, lse


def _online_thresholded(q, k, v, scale, causal, tile, kv_len, threshold, tile_order=None):
    nq = q.shape[0]
    nk = k.shape[0]
    vis = _visible(nq, nk, causal, kv_len)
    m = np.full(nq, -np.inf)          # exponent reference (may lag the true max)
    l = np.zeros(nq)
    a = np.zeros((nq, v.shape[1]))
    for j0 in _tile_starts(nk, tile, tile_order):
        j1 = min(nk, j0 + tile)
        s = scale * (q @ k[j0:j1].T)
        s = np.where(vis[:, j0:j1], s, -np.inf)
        mt = s.max(axis=1)
        with np.errstate(invalid="ignore"):
            move = (m == -np.inf) | (mt - m > threshold)
        m_new = np.where(move, np.maximum(m, mt), m)
        seen = m_new > -np.inf
        m_safe = np.where(seen, m_new, 0.0)
        alpha = np.where(m == -np.inf, 0.0, np.where(move, np.exp(m - m_safe), 1.0))
        p = np.exp(s - m_safe[:, None])
        l = alpha * l + p.sum(axis=1)
        a = alpha[:, None] * a + p @ v[j0:j1]
        m = m_new
    seen = l > 0
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(seen[:, None], a / l[:, None], 0.0)
        lse = np.where(seen, m + np.log(l), -np.inf)
    return o, lse


def splitkv_partials(q, k, v, scale, chunk, kv_len):
    """Partial (O_s, LSE_s) of each split of ``chunk`` keys below ``kv_len``.

    q: [Nq, d].  Returns O_s [S, Nq, d] (normalised inside the split) and
    LSE_s [S, Nq]; a split with no key has O_s = 0 and LSE_s = -inf.
    """
    n_split = max(1, -(-kv_len // chunk))
    outs, lses = [], []
    for s_idx in range(n_split):
        j0, j1 = s_idx * chunk, min(kv_len, (s_idx + 1) * chunk)
        if j1 <= j0:
            outs.append(np.zeros((q.shape[0], v.shape[1])))
            lses.append(np.full(q.shape[0], -np.inf))
            continue
        o_s, lse_s = online_attention(q, k[j0:j1], v[j0:j1], scale, tile=j1 - j0)
        outs.append(o_s)
        lses.append(lse_s)
    return np.stack(outs), np.stack(lses)


def combine(o_s, lse_s):
    """Merges partials: LSE = log sum_s exp(LSE_s); O = sum_s exp(LSE_s - LSE) O_s."""
    m = lse_s.max(axis=0)
    seen = m > -np.inf
    m_safe = np.where(seen, m, 0.0)
    w = np.exp(lse_s - m_safe[None, :])
    tot = w.sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        lse = np.where(seen, m_safe + np.log(tot), -np.inf)
        o = np.where(seen[:, None], (w[:, :, None] * o_s).sum(axis=0) / tot[:, None], 0.0)
    return o, lse
