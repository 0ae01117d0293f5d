"""Pins of the oracle's sequential temperature scaling (DSpark digest, Module D).

Module D calibrates, left to right, the probability that the first k drafted
tokens are all accepted, P_k = prod_{i<=k} sigma(s_i / T_i), choosing T_k on a
grid to minimise the expected calibration error (ECE) against the held-out
outcome 1[n >= k], with the earlier temperatures held fixed.

* A worked example small enough to do by hand. Logits are +-ln 9 and 0, so
  sigma(s / T) is rational on the grid {1/2, 1, 2}: sigma(ln 9 / T) = 81/82,
  9/10, 3/4. Each ECE is a fraction derived below. The example also separates
  the reading from two plausible mistakes. Position 2 without the prefix product
  would pick T = 2, not 1/2. Calibrating position 2 only on the blocks that
  survived position 1 gives different values.
* Closed form with one bin and one logit value: ECE(T) = |sigma(s/T) - mean y|.
* Recovery: blocks drawn from a known per-position acceptance temperature
  give back that temperature, and the fit cuts the ECE of the raw (T = 1)
  products by several times, which matches the pages' finding.
* Invariants: sample order, dataset duplication, a common power-of-two scale
  of logits and grid (sigma(a s / (a T)) = sigma(s / T) bit for bit), and
  left-to-right independence from later positions.
"""
import math

import numpy as np
import pytest

from speculative_decoding_drafter_markov_gb300 import workloads as wlmod

GRID3 = np.array([0.5, 1.0, 2.0], np.float32)
# the logits are fp32 roundings of +-ln 9 (relative error <= 2^-24), which moves each
# sigma(s / T) on this grid by at most ln 9 * 2^-24 / (4 * 0.5) < 7e-8
FP32_LN9 = 3e-7


def _worked_example():
    l9 = math.log(9.0)
    s = np.array([[l9, l9], [l9, -l9], [-l9, 0.0], [0.0, l9]], np.float32)
    n = np.array([2, 1, 0, 1], np.int32)
    return s, n


# Position 1, y = (1, 1, 0, 1), four bins of width 1/4:
#   T = 1/2: P = (81/82, 81/82, 1/82, 1/2) -> bins 3, 3, 0, 2; bin sums of P - y:
#            -2/82, 1/82, -1/2 -> ECE = (3/82 + 41/82) / 4 = 11/82
#   T = 1:   P = (9/10, 9/10, 1/10, 1/2)   -> -2/10, 1/10, -1/2 -> 8/10 / 4 = 1/5
#   T = 2:   P = (3/4, 3/4, 1/4, 1/2)      -> bins 3, 3, 1, 2: -1/2, 1/4, -1/2 -> 5/16
# so T_1 = 1/2 and the prefix is (81/82, 81/82, 1/82, 1/2).
# Position 2, y = (1, 0, 0, 0):
#   T = 1/2: P = (6561/6724, 81/6724, 1/164, 81/164) -> bins 3, 0, 0, 1:
#            -163/6724, (81 + 41)/6724, 3321/6724 -> 3606/6724 / 4 = 1803/13448
#   T = 1:   P = (729/820, 81/820, 1/164, 9/20)     -> bins 3, 0, 0, 1:
#            -91/820, 86/820, 369/820 -> 546/820 / 4 = 273/1640
#   T = 2:   P = (243/328, 81/328, 1/164, 3/8)      -> bins 2, 0, 0, 1:
#            -85/328, 83/328, 123/328 -> 291/328 / 4 = 291/1312
WORKED_CURVE = [[11 / 82, 1 / 5, 5 / 16], [1803 / 13448, 273 / 1640, 291 / 1312]]
# without the prefix product, position 2 would score P = sigma(s_2 / T) alone:
#   T = 1/2: (81/82, 1/82, 1/2, 81/82) -> bins 3, 0, 2, 3: 80/82, 1/82, 1/2 -> 122/328
#   T = 1:   0.8, 0.1, 0.5 -> 0.35;  T = 2: 0.5, 0.25, 0.5 -> 0.3125  (argmin T = 2)
NO_PRODUCT_CURVE2 = [122 / 328, 0.35, 0.3125]
# scoring position 2 only on the blocks that passed position 1 (m0, m1, m3, y = 1, 0, 0)
# with sigma(s_2 / T) alone, at T = 1/2: (81/82, 1/82, 81/82) -> bins 3, 0, 3:
#   80/82, 1/82 -> (81/82) / 3 = 27/82
CONDITIONAL_T05 = 27 / 82


def test_worked_example(orc):
    s, n = _worked_example()
    out = orc.sts_fit(s, n, GRID3, n_bins=4)
    np.testing.assert_allclose(out["curve"], WORKED_CURVE, rtol=0, atol=FP32_LN9)
    assert out["T"].tolist() == [0.5, 0.5]
    np.testing.assert_allclose(out["ece"], [11 / 82, 1803 / 13448], rtol=0, atol=FP32_LN9)
    # the reading is distinguishable from dropping the prefix product
    assert not np.allclose(out["curve"][1], NO_PRODUCT_CURVE2, atol=1e-3)
    assert abs(out["curve"][1][0] - CONDITIONAL_T05) > 0.1


def test_worked_example_near_edge(orc):
    """Position 1 has P = 1/2 (logit 0) on the edge between bins 1 and 2 at every
    temperature, and at T = 2 also 3/4, 3/4 and 1/4: four samples on edges.  No
    product of position 2 (1/164, 81/6724, 81/164, 9/20, 3/8, ...) lies within
    1e-4 of a multiple of 1/4."""
    s, n = _worked_example()
    out = orc.sts_fit(s, n, GRID3, n_bins=4, edge_eps=1e-4)
    assert out["near_edge"].tolist() == [[1, 1, 4], [0, 0, 0]]


def test_worked_example_forced_prefix(orc):
    """T_prefix replaces the chosen T_1 in position 2's products: with T_1 = 2
    the prefix is (3/4, 3/4, 1/4, 1/2) and, at T_2 = 2, P = (9/16, 3/16, 1/8, 3/8)
    -> bins 2, 0, 0, 1: sums -7/16, 5/16, 6/16 -> ECE = (18/16) / 4 = 9/32."""
    s, n = _worked_example()
    out = orc.sts_fit(s, n, GRID3, n_bins=4, T_prefix=np.array([2.0, 2.0], np.float32))
    assert out["T"][0] == 0.5  # position 1 is still fitted on its own
    assert out["curve"][1][2] == pytest.approx(9 / 32, abs=FP32_LN9)


def test_single_bin_closed_form(orc):
    """One bin, every block with the same logit s at position 1: the ECE is
    |sigma(s/T) - ybar|, zero at T* = s / logit(ybar)."""
    M, s0 = 40, 2.0
    n = np.zeros(M, np.int32)
    n[:32] = 1  # ybar = 0.8
    s = np.full((M, 1), s0, np.float32)
    grid = np.linspace(0.5, 3.0, 251).astype(np.float32)
    out = orc.sts_fit(s, n, grid, n_bins=1)
    t_star = s0 / math.log(0.8 / 0.2)
    expect = [abs(1.0 / (1.0 + math.exp(-s0 / float(t))) - 0.8) for t in grid]
    np.testing.assert_allclose(out["curve"][0], expect, rtol=0, atol=1e-12)
    assert abs(float(out["T"][0]) - t_star) <= 0.01
    assert out["ece"][0] < 1e-3


def test_recovers_acceptance_temperature(orc):
    T_true = [1.5, 2.0, 0.8, 1.2]
    s, n = wlmod.calibration_set(20000, 4, seed=1, T_true=T_true)
    grid = np.round(np.arange(0.2, 4.0001, 0.05), 4).astype(np.float32)
    out = orc.sts_fit(s, n, grid, n_bins=15)
    np.testing.assert_allclose(out["T"], T_true, rtol=0.15)
    raw = orc.sts_fit(s, n, np.array([1.0], np.float32), n_bins=15)
    # raw sigma(s) is over-confident here; calibration cuts the ECE several-fold
    assert np.all(out["ece"] * 4 < raw["ece"])
    assert out["ece"].mean() < 0.015


def test_invariances(orc):
    s, n = wlmod.calibration_set(3000, 5, seed=3)
    grid = np.round(np.arange(0.25, 3.0001, 0.125), 4).astype(np.float32)
    base = orc.sts_fit(s, n, grid, n_bins=10)
    perm = np.random.default_rng(0).permutation(len(n))
    out = orc.sts_fit(s[perm], n[perm], grid, n_bins=10)
    assert out["T"].tolist() == base["T"].tolist()
    np.testing.assert_allclose(out["curve"], base["curve"], rtol=0, atol=1e-12)
    dup = orc.sts_fit(np.concatenate([s, s]), np.concatenate([n, n]), grid, n_bins=10)
    np.testing.assert_allclose(dup["curve"], base["curve"], rtol=0, atol=1e-12)
    # sigma(4 s / (4 T)) == sigma(s / T) exactly (power-of-two scaling)
    sc = orc.sts_fit(s * 4, n, grid * 4, n_bins=10)
    assert np.array_equal(sc["curve"], base["curve"])
    assert np.array_equal(sc["T"], base["T"] * 4)
    # left to right: positions 1..3 do not see the logits of positions 4..5
    s2 = s.copy()
    s2[:, 3:] = -s2[:, 3:]
    part = orc.sts_fit(s2, n, grid, n_bins=10)
    assert part["T"][:3].tolist() == base["T"][:3].tolist()
    np.testing.assert_array_equal(part["curve"][:3], base["curve"][:3])
    # imposing the fit's own choices changes nothing
    same = orc.sts_fit(s, n, grid, n_bins=10, T_prefix=base["T"])
    np.testing.assert_array_equal(same["curve"], base["curve"])


def test_lowest_index_on_ties(orc):
    """Logit 0 gives P = 1/2 at every temperature: all grid points tie."""
    s = np.zeros((6, 2), np.float32)
    n = np.array([0, 1, 2, 2, 1, 0], np.int32)
    out = orc.sts_fit(s, n, np.array([3.0, 1.0, 2.0], np.float32), n_bins=5)
    assert out["T"].tolist() == [3.0, 3.0]


@pytest.mark.parametrize("bad", ["n_high", "n_neg", "nan", "grid0"])
def test_rejects_bad_arguments(orc, bad):
    s, n = _worked_example()
    grid = GRID3.copy()
    if bad == "n_high":
        n = n.copy(); n[0] = 3
    elif bad == "n_neg":
        n = n.copy(); n[1] = -1
    elif bad == "nan":
        s = s.copy(); s[2, 1] = np.nan
    else:
        grid[1] = 0.0
    with pytest.raises(ValueError):
        orc.sts_fit(s, n, grid, n_bins=4)


def test_confidence_logit_output(orc):
    """The draft's confidence logit does not depend on T_k, and c_k at T_k is
    the logistic of logit / T_k (eq. (7) with Module D's scaling)."""
    wl = wlmod.small("tiny", R=2, gamma=3, V=64)
    inp = wlmod.draft_inputs(wl, seed=5)
    args = [wlmod.bf16_bits(inp[k]) for k in ("U", "h", "W1", "W2t")]
    w = inp["w"].numpy(); anchor = inp["anchor"].numpy()
    T = np.array([0.5, 2.0, 3.0], np.float32)
    a = orc.draft_markov(*args, w, anchor, seed=1)
    b = orc.draft_markov(*args, w, anchor, seed=1, sts_T=T)
    np.testing.assert_array_equal(a["conf_logit"], b["conf_logit"])
    logit_b = np.log(b["c"]) - np.log1p(-b["c"])
    np.testing.assert_allclose(logit_b * T[None, :], a["conf_logit"], rtol=1e-9, atol=1e-9)
