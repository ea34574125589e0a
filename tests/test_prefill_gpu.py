"""GPU parity: attn_fwd (CUDA, through the C ABI) against the fp64 CPU oracle.

Small cases are compared element by element on every output.  The full-size
workloads run in the same launch configuration the benchmark times: the
training shape (causal and non-causal) and the GQA prefill are compared on
every output row, the oracle running over all rows on the host cores; the
long-context workload is compared on 256 seeded query rows that the oracle
computes one by one (its full oracle run would take about ten minutes).
Tolerances (tests/_parity.py): O max-abs 2e-2, O mean-abs 2e-3, LSE 1e-3.
"""
import math

import numpy as np
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


def _run(q, k, v, causal, scale):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = _native.forward(qd, kd, vd, causal, scale)
    assert _native.attn_get_device_status() == 0
    return o, lse


def _full_check(q, k, v, causal, scale, what):
    o, lse = _run(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    return compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what)


def test_tiny_workload_full():
    w = workloads.TINY
    q, k, v = workloads.workload_inputs(w)
    _full_check(q, k, v, w.causal, w.scale, w.name)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 2, 300, 300, 128, False),    # several tiles and a ragged tail
    (1, 2, 2, 300, 300, 128, True),
    (2, 4, 2, 200, 333, 64, False),     # GQA, Nq != Nk, ragged both ways
    (2, 4, 2, 200, 333, 64, True),      # top-left causal with Nq < Nk
    (1, 3, 1, 390, 130, 128, True),     # Nq > Nk: rows past Nk see every key
    (1, 8, 2, 257, 257, 128, True),
    (2, 2, 2, 1, 1, 64, False),         # single query, single key
    (1, 2, 1, 1, 517, 128, False),      # one query row against many keys
    (1, 1, 1, 129, 1, 128, True),
    (3, 2, 2, 128, 128, 64, True),      # exactly one tile
    (1, 4, 4, 640, 640, 128, False),
    # more work units than SMs, so each persistent CTA runs several units;
    # odd query-tile counts leave the second tile of some units inactive
    (3, 40, 40, 300, 300, 128, True),
    (3, 40, 40, 300, 300, 64, False),
    (2, 32, 8, 700, 700, 128, True),    # GQA head pairs, 192 units
    (2, 64, 16, 700, 700, 128, False),  # no mask: units head slot by head slot, GQA pairs, 384 units
    (5, 24, 24, 520, 520, 64, False),   # no mask, consecutive row tiles, odd tile count, 240 units
    (2, 96, 32, 130, 390, 128, True),   # group size 3: consecutive row tiles
])
def test_small_shapes(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=100 + Nq + Nk)
    _full_check(q, k, v, causal, 1 / math.sqrt(d), "B%d Hq%d Hkv%d Nq%d Nk%d d%d c%d" % (B, Hq, Hkv, Nq, Nk, d, causal))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", [
    (1, 4, 2, 200, 333, 64),      # Nq < Nk: every row sees the first Nk - Nq keys
    (1, 3, 1, 390, 130, 128),     # Nq > Nk: the first 260 rows see nothing
    (2, 4, 4, 130, 1000, 128),    # a short query block at the end of a long key range
    (2, 32, 8, 300, 700, 128),    # GQA head pairs, several units per CTA
    (1, 2, 2, 257, 257, 128),     # Nq == Nk: the same as top-left
])
def test_bottom_right_causal(B, Hq, Hkv, Nq, Nk, d):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=200 + Nq + Nk)
    _full_check(q, k, v, 2, 1 / math.sqrt(d), "bottom-right B%d Hq%d Hkv%d Nq%d Nk%d d%d" % (B, Hq, Hkv, Nq, Nk, d))


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.5])
def test_negative_zero_and_large_scale(scale):
    """A negative scale runs the sign-flipped kernel variant; scale 0 gives
    uniform weights (masked columns must still get exactly 0)."""
    q, k, v = workloads.prefill_inputs(1, 4, 2, 300, 300, 128, seed=12)
    for causal in (False, True):
        _full_check(q, k, v, causal, scale, "scale %g causal=%d" % (scale, causal))


@pytest.mark.parametrize("B,H,Nq", [(1, 2, 130), (2, 100, 300)])
def test_no_keys_gives_zero_and_minus_inf(B, H, Nq):
    q, k, v = workloads.prefill_inputs(B, H, H, Nq, 0, 64, seed=7)
    o, lse = _run(q, k, v, False, 0.125)
    assert torch.count_nonzero(o).item() == 0
    assert torch.isneginf(lse).all()


def test_large_scores_and_constant_rows():
    """Scores of +-100s (exp2 range edge) and rows whose max never moves."""
    B, H, N, d = 1, 2, 384, 128
    q, k, v = workloads.prefill_inputs(B, H, H, N, N, d, seed=8)
    q = (q.float() * 6).to(torch.bfloat16)
    k = k.clone()
    k[:, 0] = (q[:, 0].float() * 4).to(torch.bfloat16)  # key 0 dominates every row early
    for causal in (False, True):
        _full_check(q, k, v, causal, 1 / math.sqrt(d), "large causal=%d" % causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_rising_scores_move_the_reference(causal, sign):
    """Scores that climb by about 17 (natural-log units) every 64 keys: the
    exponent reference a row set on its first tile must move in both halves
    of later tiles, including half 1 after half 0's P has gone to the tensor
    core (the O accumulator is then rescaled in place).  Without the moves
    the exponentials would overflow fp32 long before the last key; a negative
    scale runs the same path on -s."""
    B, H, N, d = 1, 2, 640, 128
    q, k, v = workloads.prefill_inputs(B, H, H, N, N, d, seed=13)
    q = torch.ones_like(q)
    ramp = torch.arange(N, dtype=torch.float32) * (0.26 / math.sqrt(d))
    k = (sign * ramp[None, :, None, None] * torch.ones((B, 1, H, d))).to(torch.bfloat16)
    _full_check(q, k, v, causal, sign / math.sqrt(d), "rising scores causal=%d sign %+d" % (causal, sign))


def test_repeat_runs_are_bitwise_identical():
    q, k, v = workloads.prefill_inputs(2, 4, 2, 700, 700, 128, seed=9)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a = _native.forward(qd, kd, vd, True, 0.088)
    b = _native.forward(qd, kd, vd, True, 0.088)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_argument_errors_return_codes():
    q = torch.zeros((1, 8, 3, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 3, 8), dtype=torch.float32, device="cuda")
    assert _native.attn_fwd(q, k, k, o, lse, False, 0.1) == 1
    q = torch.zeros((1, 8, 2, 96), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 8, 2, 96), dtype=torch.bfloat16, device="cuda")
    assert _native.attn_fwd(q, k, k, torch.empty_like(q), torch.empty((1, 2, 8), device="cuda"), False, 0.1) == 2
    assert _native.attn_get_device_status() == 0


def _sampled_check(w, n_rows=160):
    q, k, v = workloads.workload_inputs(w)
    o, lse = _run(q, k, v, w.causal, w.scale)
    force = [(0, 0, 0), (w.B - 1, w.Hq - 1, w.N - 1), (0, w.Hq - 1, 127), (w.B - 1, 0, 128)]
    rows = workloads.sample_rows(w.B, w.Hq, w.N, n_rows, seed=w.seed, force=force)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
    o_c, lse_c = o.float().cpu().numpy(), lse.cpu().numpy()
    got_o = np.stack([o_c[b, i, h] for b, h, i in rows])
    got_l = np.array([lse_c[b, h, i] for b, h, i in rows])
    stats = compare(got_o, got_l, o_ref, lse_ref, w.name)
    assert torch.isfinite(o).all()
    return stats


def test_long_context_workload_sampled():
    """The long-context workload on 256 seeded query rows (plus the first and
    last rows and the rows either side of the first tile boundary)."""
    _sampled_check(workloads.LONG, n_rows=256)


@pytest.mark.parametrize("w", [workloads.TRAIN_CAUSAL, workloads.TRAIN, workloads.GQA], ids=lambda w: w.name)
def test_full_size_workloads_every_row(w):
    """Every O element and every LSE of the workload against the oracle: a
    slip confined to some CTAs' later persistent rounds, to the zig-zag unit
    order or to one head slot of a pair cannot hide from a full comparison."""
    q, k, v = workloads.workload_inputs(w)
    o, lse = _run(q, k, v, w.causal, w.scale)
    o_gpu, lse_gpu = o.float().cpu().numpy(), lse.cpu().numpy()
    del o, lse
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    compare(o_gpu, lse_gpu, o_ref, lse_ref, w.name + " (every row)")
