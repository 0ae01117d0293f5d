"""GPU parity of the prefix scheduler: verify lengths, capacity, Theta and the
survival products must equal the oracle's bit for bit on the same confidences."""
import numpy as np
import pytest
import torch

from parity import host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(orc, c, sps, B_min, mode, K_in=-1):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    K_dev = torch.tensor([K_in], dtype=torch.int32, device="cuda")
    out = dsp.schedule(torch.as_tensor(c, device="cuda"), torch.as_tensor(sps, device="cuda"), B_min,
                       mode=mode, K_in=K_dev if mode == dsp.SCHED_ASYNC else None, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = orc.schedule(c, sps, B_min, mode=mode, K_in=K_in)
    assert np.array_equal(host(out["ell"]), ref["ell"])
    assert int(out["K_out"].item()) == ref["K_out"]
    assert float(out["theta_best"].item()) == ref["theta_best"]
    assert np.array_equal(host(out["a"]), ref["a"])
    return ref


def _table(R, gamma, kind, seed=0):
    B = np.arange(R, R * (gamma + 1) + 1, dtype=np.float64)
    if kind == "smooth":
        return 1000.0 / (20.0 + 0.01 * B)
    if kind == "steep":
        return 1000.0 / (20.0 + 2.0 * B)
    wl = W.Workload("t", R, gamma, 8, 1, 1, "f32", sps="sawtooth")
    return W.sps_table(wl, seed)


@pytest.mark.parametrize("R,gamma", [(1, 1), (4, 4), (7, 3), (64, 8), (256, 16), (512, 16),
                                     (8192, 1), (3, 5), (2, 700), (3, 1000), (1, 8192)])
@pytest.mark.parametrize("kind", ["smooth", "steep", "saw"])
def test_sync(orc, R, gamma, kind):
    c = W.confidences(R, gamma, seed=R * 31 + gamma)
    _run(orc, c, _table(R, gamma, kind), R, dsp.SCHED_SYNC)


@pytest.mark.parametrize("R,gamma", [(512, 16), (100, 7), (5, 2)])
@pytest.mark.parametrize("K", [-1, 0, 1, 333, 100000])
def test_async(orc, R, gamma, K):
    c = W.confidences(R, gamma, seed=K + 7)
    _run(orc, c, _table(R, gamma, "saw"), R, dsp.SCHED_ASYNC, K_in=K)


def test_ties_and_zeros(orc):
    R, gamma = 40, 6
    rng = np.random.default_rng(0)
    c = np.round(W.confidences(R, gamma, seed=5, low=0.0, high=1.0) * 4) / 4  # many exact ties
    c[rng.random(c.shape) < 0.1] = 1.0
    c[rng.random(c.shape) < 0.05] = 0.0
    c = c.astype(np.float32)
    for mode, K in ((dsp.SCHED_SYNC, -1), (dsp.SCHED_ASYNC, 50), (dsp.SCHED_ASYNC, 10**6)):
        _run(orc, c, _table(R, gamma, "smooth"), R, mode, K)


def test_appendix_a(orc):
    c = np.array([[0.8, 0.9]], np.float32)
    ref = _run(orc, c, np.array([1.0, 0.5, 0.45]), 1, dsp.SCHED_SYNC)
    assert ref["ell"].tolist() == [0]


def test_table_offset(orc):
    # the table may start below R
    R, gamma = 30, 4
    B = np.arange(10, R * (gamma + 1) + 40, dtype=np.float64)
    _run(orc, W.confidences(R, gamma, seed=1), 500.0 / (5.0 + 0.1 * B), 10, dsp.SCHED_SYNC)


def test_bad_confidence_reports_range():
    c = torch.full((3, 2), 0.5, device="cuda")
    c[1, 0] = 1.5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dsp.schedule(c, torch.ones(9, dtype=torch.float64, device="cuda"), 1, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dsp.ERR_RANGE
    assert host(out["ell"]).tolist() == [0, 0, 0]


def test_build_tags():
    for R, gamma in ((1, 1), (37, 5), (512, 16), (3000, 2)):
        ell = np.random.default_rng(R).integers(0, gamma + 1, R).astype(np.int32)
        tags, N = dsp.build_tags(torch.as_tensor(ell, device="cuda"), gamma)
        torch.cuda.synchronize()
        expect = W.tags_from_ell(ell)
        assert int(N.item()) == len(expect)
        assert np.array_equal(host(tags)[:len(expect)], expect)
