"""fp64 CPU oracle for exact attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never does,
and this package imports nothing from the product library.

``attn_rows`` / ``attn_fwd`` call the plain C oracle in ``attn_oracle.c``
(full score row in fp64, two-pass softmax, LSE).  See that file's header for
the definition and the passages it follows ("FlashAttention: Part 2",
sections 1.3, 2.1 and 6.2; pyshine.com flash-attention tour, "Why You Need
This", for grouped K/V heads and KV-cache lengths).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
and ``tests/test_online_recurrence.py`` (closed forms, special cases,
invariants, brute force, hand-derived fixtures and torch's fp64 CPU SDPA).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_attn_rows.restype = ctypes.c_int
        lib.oracle_attn_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        _lib = lib
    return _lib


def host_threads() -> int:
    """Threads the oracle uses by default: the cores this process may run on."""
    return len(os.sched_getaffinity(0))


def _bf16_bits(x):
    """Accepts a torch bfloat16 CPU tensor or a numpy uint16 array of bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16 and x.device.type == "cpu"
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))


def _causal_code(causal):
    """False/0: none; True/1: aligned top-left; 2: aligned bottom-right."""
    c = int(causal)
    if c not in (0, 1, 2):
        raise ValueError("causal must be 0, 1 (top-left) or 2 (bottom-right)")
    return c


def _window(window):
    """None, or (left, right): row i (at key position i + L - Nq) sees keys
    from position - left to position + right; a negative side is unbounded."""
    if window is None:
        return -1, -1
    wl, wr = (int(x) for x in window)
    return wl, wr


def attn_rows(q, k, v, rows, causal, scale, kv_len=None, n_threads=None, window=None):
    """O and LSE for the listed query rows.

    q: [B, Nq, Hq, d] bf16; k, v: [B, Nk, Hkv, d] bf16 (Nk = allocated length);
    rows: int array [n, 3] of (b, hq, i); kv_len: optional int32 [B] valid keys;
    window: optional local window (left, right), see ``_window``.
    Returns (o [n, d] float64, lse [n] float64).
    """
    lib = _load()
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    B, Nq, Hq, d = qb.shape
    Bk, Nk, Hkv, dk = kb.shape
    assert Bk == B and dk == d and vb.shape == kb.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = rows.shape[0]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    kl = None
    if kv_len is not None:
        kl = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32).reshape(B))
    nt = host_threads() if n_threads is None else int(n_threads)
    rc = lib.oracle_attn_rows(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
        B, Hq, Hkv, Nq, Nk, d,
        None if kl is None else kl.ctypes.data, _causal_code(causal), *_window(window), float(scale),
        rows.ctypes.data, n, o.ctypes.data, lse.ctypes.data, nt)
    if rc != 0:
        raise ValueError("oracle_attn_rows failed with code %d" % rc)
    return o, lse


def all_rows(B, Hq, Nq):
    """Every (b, hq, i) triple, ordered so the result reshapes to [B, Nq, Hq]."""
    b, i, h = np.meshgrid(np.arange(B), np.arange(Nq), np.arange(Hq), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int32)


def paged_to_contiguous(pages, block_table):
    """The logical cache a paged one stands for: key k of sequence b is row
    k % page_size of page block_table[b, k // page_size] (pyshine.com
    flash-attention tour, "Why You Need This": paged KV cache).
    pages [num_pages, page_size, H, d], block_table int [B, max_blocks] ->
    [B, max_blocks * page_size, H, d]."""
    bt = np.asarray(block_table, dtype=np.int64)
    pages = np.asarray(pages) if not hasattr(pages, "numpy") else pages
    gathered = pages[bt.reshape(-1)]                      # [B*max_blocks, page_size, H, d]
    B, mb = bt.shape
    return gathered.reshape((B, mb * gathered.shape[1]) + tuple(gathered.shape[2:]))


def attn_fwd(q, k, v, causal, scale, kv_len=None, n_threads=None, window=None):
    """Full forward: O [B, Nq, Hq, d] float64 and LSE [B, Hq, Nq] float64."""
    qb = _bf16_bits(q)
    B, Nq, Hq, d = qb.shape
    o, lse = attn_rows(qb, k, v, all_rows(B, Hq, Nq), causal, scale, kv_len, n_threads, window)
    return o.reshape(B, Nq, Hq, d), lse.reshape(B, Nq, Hq).transpose(0, 2, 1).copy()
