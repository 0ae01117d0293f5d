"""The profiled cost table (DSpark digest, Module E: SPS(B) is profiled once and
only looked up at run time; production section: real capacity curves fall in
steps).

* Host logic with a fake timer: the table holds 1 / (step time) at every timed
  size and interpolates linearly between them, over exactly B_min..B_max.
* On the GPU: a table profiled from a stand-in target forward is positive and
  finite, and the scheduler run on it (both modes) matches the oracle bit for
  bit -- the scheduler's parity on a measured, non-smooth curve.
"""
import numpy as np
import pytest
import torch

from parity import host
from speculative_decoding_drafter_markov_gb300 import sps
from speculative_decoding_drafter_markov_gb300 import workloads as W


def test_table_from_a_fake_timer():
    # a sawtooth: the step time grows by 10 us at every multiple of 64 tokens
    step_s = lambda B: 1e-5 * (1 + (B - 1) // 64)
    timer = lambda fwd, B, reps, warmup: step_s(B)
    t = sps.profile_sps(None, 40, 200, step=16, timer=timer)
    assert t.shape == (161,) and t.dtype == np.float64
    for B in range(40, 201, 16):  # timed sizes: exact
        assert t[B - 40] == pytest.approx(1.0 / step_s(B), rel=1e-15)
    assert t[-1] == pytest.approx(1.0 / step_s(200), rel=1e-15)  # B_max is always timed
    # between two timed sizes the rate is linear
    assert t[120 - 40 + 3] == pytest.approx(t[120 - 40] + 3 / 16 * (t[136 - 40] - t[120 - 40]), rel=1e-14)
    with pytest.raises(ValueError):
        sps.profile_sps(None, 10, 5, timer=timer)
    with pytest.raises(RuntimeError):
        sps.profile_sps(None, 1, 4, timer=lambda *a: 0.0)


@pytest.mark.gpu
def test_profiled_table_drives_the_scheduler(orc):
    from speculative_decoding_drafter_markov_gb300 import _lib as dsp
    R, gamma = 24, 6
    fwd = W.stand_in_target(d=512, layers=1, max_B=R * (gamma + 1), device="cuda")
    table = sps.profile_sps(fwd, R, R * (gamma + 1), step=4, reps=3)
    assert np.all(np.isfinite(table)) and np.all(table > 0)
    c = W.confidences(R, gamma, seed=8)
    c_d = torch.as_tensor(c, device="cuda")
    t_d = torch.as_tensor(table, device="cuda")
    sync = dsp.schedule(c_d, t_d, R, mode=dsp.SCHED_SYNC)
    asyn = dsp.schedule(c_d, t_d, R, mode=dsp.SCHED_ASYNC, K_in=sync["K_out"])
    torch.cuda.synchronize()
    ref_s = orc.schedule(c, table, R, mode=orc.SCHED_SYNC)
    K = int(ref_s["K_out"])
    ref_a = orc.schedule(c, table, R, mode=orc.SCHED_ASYNC, K_in=K)
    assert np.array_equal(host(sync["ell"]), ref_s["ell"])
    assert int(host(sync["K_out"])[0]) == K
    assert host(sync["theta_best"])[0] == ref_s["theta_best"]
    assert np.array_equal(host(asyn["ell"]), ref_a["ell"])
    assert host(asyn["theta_best"])[0] == ref_a["theta_best"]
    # the search without the break never does worse than the break on the same pool
    assert ref_a["theta_best"] >= ref_s["theta_best"]
