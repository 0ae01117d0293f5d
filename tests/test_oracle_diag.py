"""Pins of the oracle's acceptance diagnostics (DSpark digest, analysis 1 and the
offline results).

The digest reads the drafter's quality position by position through the
conditional acceptance rate: at position k the denominator counts only the
instances whose positions 1..k-1 were all accepted, which removes the penalty of
an earlier rejection. The acceptance length tau counts the accepted drafted
tokens plus the target's own token.

* A worked example by hand (below), which also separates the reading from two
  plausible mistakes: counting every verified position in the denominator, and
  counting positions that were never verified.
* Counting identities that hold for any outcomes.
* A prefix process with known per-position acceptance probabilities gives them
  back as the conditional rates (a statistical check of the denominator).
"""
import numpy as np
import pytest


def test_worked_example(orc):
    # gamma = 4, three requests: (n, ell) = (2, 4), (4, 4), (0, 2).
    # position 1: tested for all three (ell >= 1, n >= 0); accepted by the first two.
    # position 2: tested for the first two (n >= 1); the third stopped at position 1.
    # position 3: tested for the first two (n >= 2, ell >= 3); accepted by the second.
    # position 4: tested only for the second (n >= 3); accepted.
    st = orc.accept_stats([2, 4, 0], [4, 4, 2], gamma=4)
    assert st["reached"].tolist() == [3, 2, 2, 1]
    assert st["accepted"].tolist() == [2, 2, 1, 1]
    # tau = n + 1 = 3, 5, 1: indexed by n
    assert st["tau_hist"].tolist() == [1, 0, 1, 0, 1]
    assert st["ell_hist"].tolist() == [0, 0, 1, 0, 2]
    cond = st["accepted"] / st["reached"]
    assert cond.tolist() == [2 / 3, 1.0, 0.5, 1.0]
    # a denominator of all verified positions would give 2/3, 2/3, 1/2, 1/2 instead
    verified = [sum(1 for l in (4, 4, 2) if l >= k) for k in range(1, 5)]
    assert (st["accepted"] / np.array(verified)).tolist() != cond.tolist()


def test_unverified_requests_and_accumulation(orc):
    st = orc.accept_stats([1, 0], [-1, 0], gamma=3)  # the first is not in this cycle's batch
    assert st["reached"].tolist() == [0, 0, 0]  # ell = 0: nothing verified, only the target's token
    assert st["tau_hist"].tolist() == [1, 0, 0, 0]
    orc.accept_stats([3], [3], gamma=3, into=st)  # a second cycle adds to the same counters
    assert st["reached"].tolist() == [1, 1, 1]
    assert st["accepted"].tolist() == [1, 1, 1]
    assert st["tau_hist"].tolist() == [1, 0, 0, 1]
    with pytest.raises(ValueError):
        orc.accept_stats([3], [2], gamma=3)  # more accepted than verified


def test_counting_identities(orc):
    rng = np.random.default_rng(5)
    gamma, R = 7, 400
    ell = rng.integers(-1, gamma + 1, R)
    n = np.array([rng.integers(0, l + 1) if l >= 0 else 0 for l in ell])
    st = orc.accept_stats(n, ell, gamma=gamma)
    live = ell >= 0
    assert int(st["tau_hist"].sum()) == int(live.sum())
    assert int(st["ell_hist"].sum()) == int(live.sum())
    assert int(st["accepted"].sum()) == int(n[live].sum())  # n = sum_k 1[n >= k]
    assert np.all(st["accepted"] <= st["reached"])
    assert np.all(st["reached"][1:] <= st["accepted"][:-1])  # reaching k needs k - 1 accepted
    assert int(st["reached"][0]) == int((ell >= 1).sum())


def test_prefix_process_recovers_position_rates(orc):
    # every request verifies all gamma positions; position k passes with
    # probability a_k given that 1..k-1 passed, so the conditional rates are a_k
    rng = np.random.default_rng(11)
    a = np.array([0.9, 0.6, 0.75, 0.5, 0.8])
    R = 200_000
    passed = rng.random((R, len(a))) < a
    n = np.argmin(np.concatenate([passed, np.zeros((R, 1), bool)], axis=1), axis=1)
    st = orc.accept_stats(n, None, gamma=len(a))
    cond = st["accepted"] / st["reached"]
    se = np.sqrt(a * (1 - a) / st["reached"])
    assert np.all(np.abs(cond - a) < 5 * se)
    # the unconditional fraction accepted at position k is prod_{i<=k} a_i instead
    assert abs(st["accepted"][2] / R - a[:3].prod()) < 0.005
