"""Shared comparison helpers for the GPU parity tests (no attention arithmetic).

Tolerances for bf16 outputs against the fp64 oracle: O max-abs <= 2e-2,
O mean-abs <= 2e-3, LSE abs <= 1e-3 (the workload's stated bar).
"""
import numpy as np

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_gpu/o_ref: [..., d]; lse_gpu/lse_ref: matching shapes. Returns error stats."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert lse_gpu.shape == lse_ref.shape, (lse_gpu.shape, lse_ref.shape)
    assert np.isfinite(o_gpu).all(), "%s: non-finite O" % what
    inf_ref = np.isinf(lse_ref)
    assert np.array_equal(np.isinf(lse_gpu) & (lse_gpu < 0), inf_ref), "%s: -inf LSE pattern differs" % what
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(lse_gpu[~inf_ref] - lse_ref[~inf_ref])
    stats = dict(o_max=float(err.max()) if err.size else 0.0, o_mean=float(err.mean()) if err.size else 0.0,
                 lse_max=float(lerr.max()) if lerr.size else 0.0)
    assert stats["o_max"] <= O_MAX_ABS, "%s: O max-abs %g > %g" % (what, stats["o_max"], O_MAX_ABS)
    assert stats["o_mean"] <= O_MEAN_ABS, "%s: O mean-abs %g > %g" % (what, stats["o_mean"], O_MEAN_ABS)
    assert stats["lse_max"] <= LSE_ABS, "%s: LSE abs %g > %g" % (what, stats["lse_max"], LSE_ABS)
    return stats
