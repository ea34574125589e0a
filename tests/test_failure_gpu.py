"""Failure detection on the GPU without a fault: the library's bounded wait
gives up, reports ATTN_ERR_TIMEOUT through the device status word, and the
context stays usable.

The self-test kernel waits on barriers that nothing completes (nothing is
faulted, trapped or left spinning): one warp with a 1 ms limit, the other
with the library's full 2 s limit, which must end at once when it sees the
first warp's abort.
"""
import math
import time

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


def test_bounded_wait_reports_timeout_and_the_context_survives():
    assert _native.attn_get_device_status() == _native.ATTN_OK
    t0 = time.perf_counter()
    assert _native.attn_selftest_wait_timeout(1_000_000) == _native.ATTN_OK
    status = _native.attn_get_device_status()
    elapsed = time.perf_counter() - t0
    assert status == _native.ATTN_ERR_TIMEOUT
    assert elapsed < 1.0, "the 2 s wait did not follow the abort (%.3f s)" % elapsed
    assert _native.attn_get_device_status() == _native.ATTN_OK  # reading clears the word
    # the same process and context go on computing correct results
    q, k, v = workloads.prefill_inputs(1, 4, 2, 300, 300, 128, seed=41)
    o, lse = _native.forward(q.cuda(), k.cuda(), v.cuda(), True, 1 / math.sqrt(128))
    assert _native.attn_get_device_status() == _native.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1 / math.sqrt(128))
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "after a timeout")
