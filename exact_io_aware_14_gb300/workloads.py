"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic.  Both the CUDA path (tests, bench) and the CPU
oracle are fed from here.

Recipe: torch CPU ``Generator.manual_seed(seed)``; draw order q, k, v, then
(decode only) the cache lengths; values are fp32 N(0, 1), multiplied by an
amplitude (0.5 for the GQA prefill workload, exact in fp32) and rounded to
bf16 (round-to-nearest-even).  Layout is BSHD, d innermost.  Cache
positions at or beyond a sequence's length are filled with NaN so any read
of them shows up in the output.
"""
from dataclasses import dataclass
import math

import torch


@dataclass(frozen=True)
class Prefill:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    amp: float = 1.0
    seed: int = 0
    window: tuple = None  # local window (left, right), aligned bottom-right; None: no window

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def keys_per_row(self):
        """How many keys each query row sees (int64 [N]); for work accounting."""
        i = torch.arange(self.N, dtype=torch.int64)
        lo = torch.zeros_like(i)
        hi = torch.full_like(i, self.N - 1)
        if self.causal:
            hi = torch.minimum(hi, i)
        if self.window is not None:
            wl, wr = self.window
            if wl >= 0:
                lo = torch.maximum(lo, i - wl)
            if wr >= 0:
                hi = torch.minimum(hi, i + wr)
        return (hi - lo + 1).clamp(min=0)

    def flops(self) -> float:
        """4*B*Hq*Nq*Nk*d, halved for causal (the workload's FLOP convention);
        with a window, 4*B*Hq*d times the pairs the window leaves visible."""
        if self.window is not None:
            return 4.0 * self.B * self.Hq * self.d * float(self.keys_per_row().sum())
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f


@dataclass(frozen=True)
class Decode:
    name: str
    B: int
    Hq: int
    Hkv: int
    max_seqlen: int
    d: int
    chunk: int
    len_lo: int
    len_hi: int
    seed: int = 4
    page_size: int = 0  # > 0: the cache is paged (shuffled pages of this many keys)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The workloads: tiny parity case, training shape (causal and not), GQA
# prefill, long single sequence, sliding window, split-KV decode.
TINY = Prefill("tiny_mha_b1_h2_n256_d64", 1, 2, 2, 256, 64, False, seed=0)
TRAIN_CAUSAL = Prefill("train_b4_h16_n4096_d128_causal", 4, 16, 16, 4096, 128, True, seed=1)
TRAIN = Prefill("train_b4_h16_n4096_d128", 4, 16, 16, 4096, 128, False, seed=1)
GQA = Prefill("gqa_prefill_b2_hq32_hkv8_n8192_d128_causal", 2, 32, 8, 8192, 128, True, amp=0.5, seed=2)
LONG = Prefill("long_b1_h8_n32768_d128_causal", 1, 8, 8, 32768, 128, True, seed=3)
# the pyshine.com tour's usage example (Hq 32, Hkv 8, N 2048, d 128, causal,
# window (1023, 0)) with a batch of 16
WINDOW = Prefill("window_b16_hq32_hkv8_n2048_d128_causal_w1023", 16, 32, 8, 2048, 128, True, seed=5,
                 window=(1023, 0))
DECODE = Decode("decode_b16_hq32_hkv8_len1024to16384_d128_chunk1024", 16, 32, 8, 16384, 128, 1024,
                1024, 16384, seed=4)
DECODE_PAGED = Decode("decode_paged_b16_hq32_hkv8_len1024to16384_d128_chunk1024_page256", 16, 32, 8, 16384, 128,
                      1024, 1024, 16384, seed=4, page_size=256)

PREFILL_WORKLOADS = (TINY, TRAIN_CAUSAL, TRAIN, GQA, LONG, WINDOW)


def _randn_bf16(gen, shape, amp):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if amp != 1.0:
        x.mul_(amp)
    return x.to(torch.bfloat16)


def prefill_inputs(B, Hq, Hkv, Nq, Nk, d, amp=1.0, seed=0):
    """q [B,Nq,Hq,d], k and v [B,Nk,Hkv,d], bf16 on the CPU."""
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (B, Nq, Hq, d), amp)
    k = _randn_bf16(gen, (B, Nk, Hkv, d), amp)
    v = _randn_bf16(gen, (B, Nk, Hkv, d), amp)
    return q, k, v


def workload_inputs(w: Prefill):
    return prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.N, w.d, w.amp, w.seed)


def decode_inputs(B, Hq, Hkv, max_seqlen, d, len_lo, len_hi, seed=4, poison=True, seqlens=None):
    """q [B,1,Hq,d]; k_cache, v_cache [B,max_seqlen,Hkv,d]; seqlens int32 [B].

    Cache lengths are drawn uniformly from the integers [len_lo, len_hi]
    unless given.  Positions >= seqlens[b] hold NaN when ``poison``.
    """
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (B, 1, Hq, d), 1.0)
    k = torch.empty((B, max_seqlen, Hkv, d), dtype=torch.bfloat16)
    v = torch.empty((B, max_seqlen, Hkv, d), dtype=torch.bfloat16)
    for b in range(B):  # one batch row at a time keeps the fp32 draw small
        k[b] = _randn_bf16(gen, (max_seqlen, Hkv, d), 1.0)
    for b in range(B):
        v[b] = _randn_bf16(gen, (max_seqlen, Hkv, d), 1.0)
    if seqlens is None:
        seqlens = torch.randint(len_lo, len_hi + 1, (B,), generator=gen, dtype=torch.int32)
    else:
        seqlens = torch.as_tensor(seqlens, dtype=torch.int32)
    if poison:
        for b in range(B):
            L = int(seqlens[b])
            k[b, L:] = float("nan")
            v[b, L:] = float("nan")
    return q, k, v, seqlens


def page_cache(k, v, page_size, extra_pages=3, seed=0):
    """Scatter a contiguous cache [B, max_seqlen, Hkv, d] into page pools
    [num_pages, page_size, Hkv, d] under a seeded random page order.

    Returns (k_pages, v_pages, block_table int32 [B, max_blocks]); key k of
    sequence b is row k % page_size of page block_table[b, k // page_size].
    Pages that no sequence uses (``extra_pages`` of them) hold NaN.
    """
    B, S, Hkv, d = k.shape
    max_blocks = -(-S // page_size)
    num_pages = B * max_blocks + extra_pages
    gen = torch.Generator().manual_seed(5000 + seed)
    order = torch.randperm(num_pages, generator=gen)[: B * max_blocks].to(torch.int32)
    block_table = order.reshape(B, max_blocks).contiguous()
    k_pages = torch.full((num_pages, page_size, Hkv, d), float("nan"), dtype=k.dtype)
    v_pages = torch.full((num_pages, page_size, Hkv, d), float("nan"), dtype=v.dtype)
    for b in range(B):
        for blk in range(max_blocks):
            lo, hi = blk * page_size, min(S, (blk + 1) * page_size)
            pg = int(block_table[b, blk])
            k_pages[pg, : hi - lo] = k[b, lo:hi]
            v_pages[pg, : hi - lo] = v[b, lo:hi]
    return k_pages, v_pages, block_table


def workload_decode_inputs(w: Decode, poison=True):
    return decode_inputs(w.B, w.Hq, w.Hkv, w.max_seqlen, w.d, w.len_lo, w.len_hi, w.seed, poison)


def sample_rows(B, Hq, Nq, n, seed, force=()):
    """n seeded (b, hq, i) triples, plus the forced ones first (int32 [m, 3])."""
    gen = torch.Generator().manual_seed(1000 + seed)
    b = torch.randint(0, B, (n,), generator=gen)
    h = torch.randint(0, Hq, (n,), generator=gen)
    i = torch.randint(0, Nq, (n,), generator=gen)
    rows = [tuple(t) for t in force] + list(zip(b.tolist(), h.tolist(), i.tolist()))
    return torch.tensor(rows, dtype=torch.int32).numpy()
