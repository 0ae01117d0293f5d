"""Pins of the oracle's hardware-aware prefix scheduler (DSpark digest, Module E,
Algorithm 1, Appendix A and the production asynchronous variant).

* Appendix A's worked numbers: a_1 = 0.8 and SPS(1, 2, 3) = 1.0 / 0.5 / 0.45 stop
  the synchronous scheduler at l = 0 (Theta_0 = 1.0 > Theta_1 = 0.9), while the
  backtracking search admits l = 2 when c_2 = 0.9 (Theta_2 = 1.134) and l = 0 when
  c_2 = 0 (Theta_2 = 0.81).
* Monotone a makes the greedy pool admit prefixes only (Module E): every admitted
  set is exactly {(r, j): j <= l_r} and equals the top of the sorted pool.
* With a log-concave SPS table Theta is unimodal along the greedy path, so the
  early-stop result equals brute force over every l vector for tiny R, gamma.
* The asynchronous variant admits exactly min(K, |E|) entries of the current
  order and K_in < 0 falls back to Algorithm 1.
"""
import itertools

import numpy as np
import pytest

from speculative_decoding_drafter_markov_gb300 import workloads as wlmod


def _theta(ell, a, sps, B_min):
    R = len(ell)
    tau = R + sum(float(np.float64(a[rq, :ell[rq]]).sum()) for rq in range(R))
    B = R + int(sum(ell))
    return tau * sps[B - B_min]


def test_appendix_a_counterexample(orc):
    sps = np.array([1.0, 0.5, 0.45])
    c_hi = np.array([[0.8, 0.9]], np.float32)
    c_lo = np.array([[0.8, 0.0]], np.float32)
    out = orc.schedule(c_hi, sps, 1, mode=orc.SCHED_SYNC)
    assert out["ell"].tolist() == [0]
    assert out["theta_best"] == pytest.approx(1.0, abs=1e-12)
    out = orc.schedule(c_lo, sps, 1, mode=orc.SCHED_SYNC)
    assert out["ell"].tolist() == [0]
    hi = orc.schedule(c_hi, sps, 1, mode=orc.SCHED_NOBREAK)
    assert hi["ell"].tolist() == [2]
    assert hi["theta_best"] == pytest.approx(1.134, abs=1e-6)
    lo = orc.schedule(c_lo, sps, 1, mode=orc.SCHED_NOBREAK)
    assert lo["ell"].tolist() == [0]
    assert lo["theta_best"] == pytest.approx(1.0, abs=1e-12)
    assert hi["K_out"] == 2 and lo["K_out"] == 0


def _check_prefix(out, c):
    a = out["a"]
    R, gamma = c.shape
    ell = out["ell"]
    assert np.all(np.diff(a, axis=1) <= 0)
    # admitted set == top-|admitted| of the pool, ties by (request, position)
    flat = np.arange(R * gamma)
    order = np.lexsort((flat, -a.reshape(-1)))
    order = [e for e in order if a.reshape(-1)[e] > 0]
    n_adm = int(ell.sum())
    top = set(order[:n_adm])
    adm = {rq * gamma + j for rq in range(R) for j in range(ell[rq])}
    assert top == adm


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_prefix_invariant(orc, seed, mode):
    rng = np.random.default_rng(seed)
    R, gamma = int(rng.integers(1, 40)), int(rng.integers(1, 9))
    c = wlmod.confidences(R, gamma, seed=seed, low=0.0, high=1.0)
    c[rng.random(c.shape) < 0.05] = 1.0  # ties inside a request
    c[rng.random(c.shape) < 0.02] = 0.0  # zero survival: excluded from the pool
    B = np.arange(R, R * (gamma + 1) + 1)
    sps = 1000.0 / (20.0 + 0.05 * B)
    K_in = int(rng.integers(-1, R * gamma + 2)) if mode == 1 else -1
    out = orc.schedule(c, sps, R, mode=mode, K_in=K_in)
    _check_prefix(out, c)
    pool = int((out["a"] > 0).sum())
    if mode == 1 and K_in >= 0:
        assert out["ell"].sum() == min(K_in, pool)
    if mode == 2:
        assert out["ell"].sum() == out["K_out"]


@pytest.mark.parametrize("seed", range(25))
def test_sync_equals_brute_force_on_log_concave_table(orc, seed):
    rng = np.random.default_rng(100 + seed)
    R, gamma = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    c = rng.uniform(0.05, 1.0, (R, gamma)).astype(np.float32)
    slope = rng.uniform(0.005, 0.06)
    B = np.arange(1, R * (gamma + 1) + 1)
    sps = 1.0 - slope * B  # linear decrease, positive on the table: log-concave
    out = orc.schedule(c, sps, 1, mode=orc.SCHED_SYNC)
    best, arg = -1.0, None
    for ell in itertools.product(range(gamma + 1), repeat=R):
        th = _theta(ell, out["a"], sps, 1)
        if th > best:
            best, arg = th, ell
    assert out["theta_best"] == pytest.approx(best, rel=1e-9)
    assert tuple(out["ell"]) == arg
    # the backtracking search reaches the same point on a unimodal objective
    nb = orc.schedule(c, sps, 1, mode=orc.SCHED_NOBREAK)
    assert tuple(nb["ell"]) == arg and nb["K_out"] == sum(arg)


def test_async_fallback_and_capacity(orc):
    R, gamma = 16, 6
    c = wlmod.confidences(R, gamma, seed=3)
    B = np.arange(R, R * (gamma + 1) + 1)
    sps = 1000.0 / (20.0 + 0.5 * B)
    sync = orc.schedule(c, sps, R, mode=orc.SCHED_SYNC)
    fall = orc.schedule(c, sps, R, mode=orc.SCHED_ASYNC, K_in=-1)
    assert np.array_equal(sync["ell"], fall["ell"]) and sync["theta_best"] == fall["theta_best"]
    for K in (0, 1, 7, 40, R * gamma, R * gamma + 5):
        o = orc.schedule(c, sps, R, mode=orc.SCHED_ASYNC, K_in=K)
        assert o["ell"].sum() == min(K, R * gamma)
        _check_prefix(o, c)
        assert o["K_out"] == sync["K_out"]  # capacity depends on the current pool only


def test_table_range_and_bad_confidence(orc):
    c = np.full((3, 2), 0.5, np.float32)
    with pytest.raises(ValueError):
        orc.schedule(c, np.ones(8), 1)  # needs B up to 9
    orc.schedule(c, np.ones(9), 1)
    with pytest.raises(ValueError):
        orc.schedule(c, np.ones(9), 4)  # B_min above R
    bad = c.copy()
    bad[1, 1] = np.nan
    with pytest.raises(ValueError):
        orc.schedule(bad, np.ones(9), 1)
    bad[1, 1] = 1.5
    with pytest.raises(ValueError):
        orc.schedule(bad, np.ones(9), 1)


def test_theta_is_fixed_point_of_sorted_survival(orc):
    # Theta_best equals tau * SPS(B) at the admitted point, tau from the fp32 products
    R, gamma = 8, 5
    c = wlmod.confidences(R, gamma, seed=12)
    B = np.arange(R, R * (gamma + 1) + 1)
    sps = 50.0 / (1.0 + 0.1 * B)
    out = orc.schedule(c, sps, R, mode=orc.SCHED_SYNC)
    assert out["theta_best"] == pytest.approx(_theta(out["ell"], out["a"], sps, R), rel=1e-9)
    assert out["theta_best"] >= R * sps[0]
