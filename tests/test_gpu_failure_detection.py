"""Failure detection without a GPU fault: a wait that can never complete
gives up after its limit, the kernel returns normally with a status the host
reads, and the context stays usable (the pipelined kernels' copy waits use
the same bounded wait, with a 100 ms limit)."""
import time

import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def test_wait_on_a_barrier_nothing_completes_gives_up():
    t0 = time.time()
    assert rq.debug_bounded_wait(1_000_000) == 1        # 1 ms limit: every thread gave up
    assert time.time() - t0 < 5.0
    assert rq.take_fault_flags() == 0                   # the library's own flags are untouched
    # the context is still usable: a normal call afterwards is exact
    wl = ri.make_workload("after", 64, 1024, seed=3)
    want = oracle.run_workload(wl, "fp8_per_token")
    got = P.run_gpu(wl, "fp8_per_token", None)
    P.compare(got, want, "fp8_per_token", "after a timed-out wait")


def test_bounded_wait_arguments():
    with pytest.raises(rq.RmsqError):
        rq.debug_bounded_wait(0)
    with pytest.raises(rq.RmsqError):
        rq.debug_bounded_wait(2_000_000_000)
