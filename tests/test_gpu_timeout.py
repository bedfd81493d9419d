"""The bounded device waits, driven to expiry on purpose.

Every barrier wait inside the library's kernels gives up after a time limit,
records DSA_ERR_DEVICE_TIMEOUT in the library's error word and lets its kernel
return (failure detection without a GPU fault).  dsa_wait_selftest queues a
kernel whose barriers nothing completes: one wait with a short limit, one with
the ordinary 2 s limit that the first wait's abort flag must end early.  The
test checks the reported status, that the word is cleared once read, that the
whole thing took far less than 2 s, and that the context still computes
correctly afterwards.
"""
import time

import pytest
import torch

from sparse_top_attention_gb300 import dsa
from sparse_top_attention_gb300 import workloads as WL
from tests.parity_util import check_bwd, check_fwd
from tests.test_gpu_parity import DEV, _lib, counts_of, oracle_exact, run  # noqa: F401

pytestmark = pytest.mark.gpu

DSA_ERR_DEVICE_TIMEOUT = 6


def test_wait_limit_runs_out_and_is_reported():
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    t0 = time.perf_counter()
    dsa.wait_selftest(20000)  # 20 ms
    st = dsa.device_status()  # synchronises the stream
    dt = time.perf_counter() - t0
    assert st == DSA_ERR_DEVICE_TIMEOUT
    assert dt < 1.0, dt  # the 2 s waiter was released by the abort flag
    assert dsa.device_status() == 0  # read and cleared


def test_context_still_works_after_a_timeout():
    dsa.wait_selftest(1000)
    assert dsa.device_status() == DSA_ERR_DEVICE_TIMEOUT
    w = WL.make("tiny")
    out, lse, dq, dkv, dsink = run(w)
    ref, g = oracle_exact(w)
    counts = counts_of(w)
    check_fwd(out, lse, ref, counts)
    check_bwd(dq, dkv, dsink, g, counts)


def test_selftest_rejects_bad_limits():
    for bad in (0, 1000001):
        with pytest.raises(dsa.DsaError):
            dsa.wait_selftest(bad)
