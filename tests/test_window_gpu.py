"""GPU parity: local (sliding-window) attention -- attn_fwd_window, and
attn_fwd_kvcache with a window -- against the fp64 CPU oracle.

The window (left, right) is aligned bottom-right: query row i sits at key
position i + L - Nq and sees keys from position - left to position + right
("FlashAttention: Part 2", section 3.2; the pyshine.com tour's usage
example passes causal with window (1023, 0)).  Shapes span several tiles
with ragged tails, both ways of pairing query tiles in a CTA (GQA head
pairs, consecutive row tiles of one head), more units than SMs, windows
narrower than a tile, one-sided windows, rows whose window holds no key, and
head pairs whose left-edge key tile is visited last (also against a cache
whose last V tile runs past the cache length).
"""
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


def _check(B, Hq, Hkv, Nq, Nk, d, causal, window, seed):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed)
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward_window(q.cuda(), k.cuda(), v.cuda(), causal, window, scale)
    assert _native.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale, window=window)
    return compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
                   "window %s B%d Hq%d Hkv%d Nq%d Nk%d d%d causal%d" % (window, B, Hq, Hkv, Nq, Nk, d, causal))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,window", [
    (1, 2, 2, 300, 300, 128, 0, (127, 0)),       # consecutive row tiles, causal-style window
    (1, 2, 2, 300, 300, 128, 0, (64, 64)),       # symmetric, narrower than a tile
    (1, 2, 2, 300, 300, 128, 0, (0, 0)),         # the diagonal alone
    (1, 2, 2, 300, 300, 128, 0, (200, -1)),      # left side only
    (1, 2, 2, 300, 300, 128, 0, (-1, 50)),       # right side only
    (1, 2, 2, 300, 300, 128, 1, (100, 0)),       # with top-left causal
    (1, 2, 2, 300, 300, 128, 2, (33, 7)),        # intersected with bottom-right causal
    (2, 4, 2, 200, 333, 64, 0, (50, 0)),         # Nq < Nk, GQA head pairs, d = 64
    (2, 4, 2, 200, 333, 64, 0, (10, 20)),
    (1, 3, 1, 390, 130, 128, 0, (64, 0)),        # Nq > Nk: the first 260 rows see no key
    (1, 4, 4, 640, 640, 128, 0, (200, 0)),       # row-tile pairs: the second tile starts later
    (1, 4, 4, 640, 640, 128, 0, (129, 300)),
    (3, 40, 40, 300, 300, 128, 0, (129, 3)),     # more units than SMs
    (2, 32, 8, 700, 700, 128, 2, (255, -1)),     # GQA head pairs, several units per CTA
    (2, 96, 32, 130, 390, 128, 0, (17, 5)),      # group size 3
    (2, 2, 2, 1, 517, 128, 0, (100, 0)),         # one query row: the last 101 keys
    (1, 2, 2, 1000, 1000, 64, 0, (500, 500)),
    (2, 8, 2, 600, 600, 64, 1, (383, 0)),        # head pairs whose left-edge key tile is visited last
])
def test_window_parity(B, Hq, Hkv, Nq, Nk, d, causal, window):
    _check(B, Hq, Hkv, Nq, Nk, d, causal, window, seed=300 + Nq + Nk)


def test_window_zero_returns_the_values():
    """Window (0, 0) with Nq == Nk: each row attends to its own key alone, so
    O is V rounded to bf16 exactly and the LSE is the row's one score."""
    q, k, v = workloads.prefill_inputs(1, 4, 4, 260, 260, 128, seed=301)
    o, _ = _native.forward_window(q.cuda(), k.cuda(), v.cuda(), 0, (0, 0), 0.1)
    assert torch.equal(o.cpu(), v)


def test_window_covering_everything_equals_attn_fwd_bitwise():
    """A window wide enough to bound nothing (but not normalised away by the
    host) gives attn_fwd's result bit for bit; so does (w >= Nk, 0) against
    bottom-right causal."""
    q, k, v = workloads.prefill_inputs(2, 8, 2, 300, 400, 128, seed=302)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a = _native.forward_window(qd, kd, vd, 0, (699, 699), 0.09)
    b = _native.forward(qd, kd, vd, 0, 0.09)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c = _native.forward_window(qd, kd, vd, 0, (500, 0), 0.09)
    e = _native.forward(qd, kd, vd, 2, 0.09)
    assert torch.equal(c[0], e[0]) and torch.equal(c[1], e[1])


@pytest.mark.parametrize("causal,window", [(2, (100, 0)), (0, (40, 40)), (1, (300, -1)), (2, (300, 0))])
def test_kvcache_with_window(causal, window):
    """A query block against a cache with per-sequence lengths and a window
    (positions taken with L = the sequence's cache length); cache positions
    past a length hold NaN."""
    B, Hq, Hkv, Nq, S, d = 3, 8, 2, 77, 1000, 128
    lens = [1000, 333, 128]
    q = workloads.prefill_inputs(B, Hq, Hkv, Nq, 1, d, seed=303)[0]
    _, k, v, L = workloads.decode_inputs(B, Hq, Hkv, S, d, 0, 0, seed=304, seqlens=lens)
    scale = 1 / math.sqrt(d)
    o, lse = _native.forward_kvcache(q.cuda(), k.cuda(), v.cuda(), L.cuda(), causal, scale, window=window)
    assert _native.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale, kv_len=L.numpy(), window=window)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "kvcache window %s causal%d" % (window, causal))


def test_window_workload_every_row():
    """The sliding-window workload at full size, in the launch configuration
    the benchmark times, against the oracle on every output row."""
    w = workloads.WINDOW
    q, k, v = workloads.workload_inputs(w)
    o, lse = _native.forward_window(q.cuda(), k.cuda(), v.cuda(), w.causal, w.window, w.scale)
    assert _native.attn_get_device_status() == 0
    o_gpu, lse_gpu = o.float().cpu().numpy(), lse.cpu().numpy()
    del o, lse
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale, window=w.window)
    compare(o_gpu, lse_gpu, o_ref, lse_ref, w.name + " (every row)")


@pytest.mark.parametrize("scale", [-0.11, 0.0])
def test_window_and_cache_with_negative_or_zero_scale(scale):
    """The general kernel instance also has a negative-scale variant (it works
    on -s with |scale|); scale 0 gives uniform weights over each row's window."""
    q, k, v = workloads.prefill_inputs(2, 4, 2, 300, 450, 128, seed=305)
    for causal, window in [(0, (100, 20)), (2, (257, -1))]:
        o, lse = _native.forward_window(q.cuda(), k.cuda(), v.cuda(), causal, window, scale)
        assert _native.attn_get_device_status() == 0
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale, window=window)
        compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "window %s scale %g" % (window, scale))
    lens = [450, 77]
    _, kc, vc, L = workloads.decode_inputs(2, 4, 2, 450, 128, 0, 0, seed=306, seqlens=lens)
    for causal in (0, 2):
        o, lse = _native.forward_kvcache(q.cuda(), kc.cuda(), vc.cuda(), L.cuda(), causal, scale)
        assert _native.attn_get_device_status() == 0
        o_ref, lse_ref = oracle.attn_fwd(q, kc, vc, causal, scale, kv_len=L.numpy())
        compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "kvcache scale %g causal%d" % (scale, causal))


@pytest.mark.parametrize("window", [(63, 0), (1, 1), (300, 64)])
def test_window_head_dim_64(window):
    _check(2, 6, 3, 333, 333, 64, 0, window, seed=307 + window[0])
