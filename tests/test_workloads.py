"""Host logic of the workload definitions: the visible-pair counts behind the
FLOP accounting of the benchmark (the rate of the sliding-window workload
depends on them), checked against brute force over the mask and the closed
forms, and the seeded inputs' reproducibility."""
import numpy as np
import torch

from exact_io_aware_14_gb300 import workloads as W


def _brute(N, causal, window):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    vis = np.ones((N, N), dtype=bool)
    if causal:
        vis &= j <= i
    if window is not None:
        wl, wr = window
        if wl >= 0:
            vis &= j >= i - wl
        if wr >= 0:
            vis &= j <= i + wr
    return vis.sum(axis=1)


def test_keys_per_row_matches_the_mask():
    for causal, window in [(False, None), (True, None), (True, (5, 0)), (False, (3, 2)), (False, (-1, 4)),
                           (True, (0, 0)), (False, (7, -1))]:
        w = W.Prefill("t", 1, 1, 1, 37, 64, causal, window=window)
        assert np.array_equal(w.keys_per_row().numpy(), _brute(37, causal, window)), (causal, window)


def test_flops_closed_forms():
    w = W.Prefill("t", 2, 3, 3, 100, 64, True)
    assert w.flops() == 4.0 * 2 * 3 * 100 * 100 * 64 / 2          # the halved causal convention
    w = W.Prefill("t", 2, 3, 3, 100, 64, False)
    assert w.flops() == 4.0 * 2 * 3 * 100 * 100 * 64
    # causal window (W, 0): rows below W see i + 1 keys, the rest W + 1
    Wn, N = 9, 100
    w = W.Prefill("t", 1, 1, 1, N, 64, True, window=(Wn, 0))
    pairs = sum(min(i + 1, Wn + 1) for i in range(N))
    assert w.flops() == 4.0 * 64 * pairs
    ww = W.WINDOW
    pairs = 1024 * 1025 // 2 + (ww.N - 1024) * 1024
    assert ww.flops() == 4.0 * ww.B * ww.Hq * ww.d * pairs


def test_seeded_inputs_are_reproducible():
    a = W.prefill_inputs(1, 2, 1, 5, 7, 64, seed=3)
    b = W.prefill_inputs(1, 2, 1, 5, 7, 64, seed=3)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    c = W.prefill_inputs(1, 2, 1, 5, 7, 64, seed=4)
    assert not torch.equal(a[0], c[0])
