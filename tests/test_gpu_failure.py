"""Device-side failure detection: the bounded waits of the tensor-core kernels.

Every spin-wait in those kernels (a CTA waiting for the other CTAs of its
M-tile, a warp waiting on an mbarrier) gives up after a wall-clock limit and
reports DSPARK_ERR_TIMEOUT through the error word instead of hanging.  These
tests run the same waits on a condition nothing satisfies (a flag nobody sets,
an mbarrier nobody arrives at) with a short limit, check the reported status
and that the context stays usable afterwards.
"""
import time

import pytest
import torch

from speculative_decoding_drafter_markov_gb300 import _lib as dsp

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms


@pytest.mark.parametrize("mode", [0, 1], ids=["counter", "mbarrier"])
def test_wait_gives_up_and_reports_timeout(mode):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")  # nothing ever sets it
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dsp.wait_selfcheck(flag, 1, mode, LIMIT_NS, err)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == dsp.ERR_TIMEOUT
    assert elapsed < 2.0  # gave up near the limit rather than spinning on


@pytest.mark.parametrize("mode", [0, 1], ids=["counter", "mbarrier"])
def test_satisfied_wait_reports_nothing(mode):
    flag = torch.ones(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    target = 1 if mode == 0 else 0  # mode 1: target <= 0 arrives on the barrier first
    dsp.wait_selfcheck(flag, target, mode, LIMIT_NS, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_context_usable_after_timeout():
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsp.wait_selfcheck(flag, 1, 0, LIMIT_NS, err)
    torch.cuda.synchronize()
    assert int(err.item()) == dsp.ERR_TIMEOUT
    # ordinary work on the same context afterwards
    ctr = torch.arange(16, dtype=torch.int32, device="cuda").view(4, 4)
    out = dsp.philox(ctr, seed=7)
    torch.cuda.synchronize()
    assert out.shape == (4, 4)
