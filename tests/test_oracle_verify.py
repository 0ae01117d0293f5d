"""Pins of the oracle's lossless verification ("DSpark explained" section 06
single-token rule, applied along the scheduled prefix; DSpark digest Appendix A).

* Accept with min(1, p/q), else resample from norm(max(0, p - q)), reproduces the
  target distribution p: 10^6 single-token trials, chi-square.
* First-position acceptance rate equals sum_v min(p_v, q_v) = 1 - TV(p, q)
  (eq. 8 of the digest).
* Appendix A's two-token vocabulary: p_t = (0.7, 0.3), p_d = (0.5, 0.5) gives an
  acceptance rate of 0.8 and Pr(Y = A) = 0.7 with Algorithm 1's break, but 0.85
  when the lossy backtracking search lets x_1 decide its own admission.
* p == q accepts every scheduled token; p(x_1) = 0 rejects at the first position;
  the bonus token after a fully accepted prefix follows p.
* The correction / bonus token is the inverse-CDF draw with one stream-2 uniform
  (recomputed here with numpy's cumulative sums and searchsorted).
"""
import numpy as np
import pytest
from scipy import special, stats

from speculative_decoding_drafter_markov_gb300 import workloads as wlmod


def _zero_bias(V, r=1):
    return np.zeros((V, r), np.float32), np.zeros((V, r), np.float32)


def _draft_then_verify(orc, U_draft, T_rows, ell, seed, cycle, A=None):
    """Draft gamma tokens from softmax(U) (zero bias) and verify them against target
    rows T_rows [R, gamma+1, V] with l_r = ell[r]."""
    R, gamma, V = U_draft.shape
    W1, W2t = _zero_bias(V)
    h = np.zeros((R, gamma, 1), np.float32)
    w = np.zeros(2, np.float32)
    anchor = np.zeros(R, np.int32)
    d = orc.draft_markov(U_draft, h, W1, W2t, w, anchor, seed=seed, cycle=cycle)
    tags = wlmod.tags_from_ell(ell)
    T = np.stack([T_rows[rq, j] for rq, j in tags]).astype(np.float32)
    v = orc.verify(T, tags, anchor, d["x"], d["logq"].astype(np.float32),
                   d["lse"].astype(np.float32), U_draft, W1, W2t, seed=seed, cycle=cycle)
    return d, v


def test_single_token_rule_reproduces_target(orc):
    V, R, cycles = 6, 1000, 1000
    rng = np.random.default_rng(5)
    q_logits = rng.standard_normal(V).astype(np.float32) * 1.5
    p_logits = rng.standard_normal(V).astype(np.float32) * 1.5
    U = np.broadcast_to(q_logits, (R, 1, V)).copy()
    T_rows = np.broadcast_to(p_logits, (R, 2, V)).copy()
    ell = np.ones(R, np.int64)
    counts = np.zeros(V, np.int64)
    for cyc in range(cycles):
        _, v = _draft_then_verify(orc, U, T_rows, ell, seed=77, cycle=cyc)
        counts += np.bincount(v["out_tokens"][:, 0], minlength=V)
    p = special.softmax(p_logits.astype(np.float64))
    assert stats.chisquare(counts, p * counts.sum()).pvalue > 1e-4, (counts, p)


def test_first_position_acceptance_is_one_minus_tv(orc):
    V, R, cycles = 10, 2000, 50
    rng = np.random.default_rng(9)
    q_logits = (rng.standard_normal(V) * 2).astype(np.float32)
    p_logits = (rng.standard_normal(V) * 2).astype(np.float32)
    U = np.broadcast_to(q_logits, (R, 1, V)).copy()
    T_rows = np.broadcast_to(p_logits, (R, 2, V)).copy()
    acc = 0
    for cyc in range(cycles):
        _, v = _draft_then_verify(orc, U, T_rows, np.ones(R, np.int64), seed=3, cycle=cyc)
        acc += int((v["n_accept"] == 1).sum())
    p = special.softmax(p_logits.astype(np.float64))
    q = special.softmax(q_logits.astype(np.float64))
    expect = np.minimum(p, q).sum()
    assert expect == pytest.approx(1 - 0.5 * np.abs(p - q).sum(), abs=1e-12)
    n = R * cycles
    assert abs(acc / n - expect) < 5 * np.sqrt(expect * (1 - expect) / n)


def _two_token_trials(orc, mode, n_trials=100_000):
    """Appendix A: vocabulary {A=0, B=1}, p_t = (0.7, 0.3), p_d = (0.5, 0.5),
    c_1 = 0.8, c_2 = 0.9 if x_1 = A else 0, SPS(1, 2, 3) = 1.0 / 0.5 / 0.45."""
    R = 10_000
    U = np.zeros((R, 2, 2), np.float32)
    T_rows = np.broadcast_to(np.log(np.array([0.7, 0.3], np.float32)), (R, 3, 2)).copy()
    sps = np.array([1.0, 0.5, 0.45])
    hits, accepted, tested = 0, 0, 0
    for cyc in range(n_trials // R):
        W1, W2t = _zero_bias(2)
        d = orc.draft_markov(U, np.zeros((R, 2, 1), np.float32), W1, W2t, np.zeros(2, np.float32),
                             np.zeros(R, np.int32), seed=21, cycle=cyc)
        ell = np.zeros(R, np.int64)
        for rq in range(R):
            c = np.array([[0.8, 0.9 if d["x"][rq, 0] == 0 else 0.0]], np.float32)
            ell[rq] = orc.schedule(c, sps, 1, mode=mode)["ell"][0]
        tags = wlmod.tags_from_ell(ell)
        T = np.stack([T_rows[rq, j] for rq, j in tags]).astype(np.float32)
        v = orc.verify(T, tags, np.zeros(R, np.int32), d["x"], d["logq"].astype(np.float32),
                       d["lse"].astype(np.float32), U, W1, W2t, seed=21, cycle=cyc)
        hits += int((v["out_tokens"][:, 0] == 0).sum())
        tested += int((ell >= 1).sum())
        accepted += int(((ell >= 1) & (v["n_accept"] >= 1)).sum())
    return hits / n_trials, accepted, tested


def test_appendix_a_two_token_bias(orc):
    n = 100_000
    tol = 5 * np.sqrt(0.25 / n)
    p_sync, _, tested = _two_token_trials(orc, orc.SCHED_SYNC, n)
    assert tested == 0  # Theta_1 = 0.9 < Theta_0 = 1.0: the break keeps l = 0
    assert abs(p_sync - 0.7) < tol
    p_lossy, accepted, tested = _two_token_trials(orc, orc.SCHED_NOBREAK, n)
    assert abs(p_lossy - 0.85) < tol  # x_1 = A admitted and always accepted
    assert accepted == tested  # min(1, 0.7 / 0.5) = 1 for the only admitted token A


def test_acceptance_rate_two_token(orc):
    # l forced to 1: acceptance probability sum min(p, q) = min(.7,.5) + min(.3,.5) = 0.8
    R, cycles = 10_000, 10
    U = np.zeros((R, 1, 2), np.float32)
    T_rows = np.broadcast_to(np.log(np.array([0.7, 0.3], np.float32)), (R, 2, 2)).copy()
    acc = 0
    for cyc in range(cycles):
        _, v = _draft_then_verify(orc, U, T_rows, np.ones(R, np.int64), seed=4, cycle=cyc)
        acc += int((v["n_accept"] == 1).sum())
    n = R * cycles
    assert abs(acc / n - 0.8) < 5 * np.sqrt(0.16 / n)


def test_identical_distributions_accept_everything(orc):
    R, gamma, V, r, d = 6, 4, 50, 4, 3
    rng = np.random.default_rng(1)
    U = (rng.standard_normal((R, gamma, V)) * 2).astype(np.float32)
    W1 = (rng.standard_normal((V, r)) * 0.3).astype(np.float32)
    W2t = (rng.standard_normal((V, r)) * 0.3).astype(np.float32)
    h = np.zeros((R, gamma, d), np.float32)
    w = np.zeros(d + r, np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    for cyc in range(20):
        dr = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=2, cycle=cyc, want_z=True)
        ell = np.full(R, gamma)
        tags = wlmod.tags_from_ell(ell)
        # target rows j < gamma: the draft's own logits; bonus row: anything
        T = np.stack([dr["z"][rq, j] if j < gamma else U[rq, 0] for rq, j in tags]).astype(np.float64)
        v = orc.verify(T.astype(np.float32), tags, anchor, dr["x"], dr["logq"].astype(np.float32),
                       dr["lse"].astype(np.float32), U, W1, W2t, seed=2, cycle=cyc)
        assert np.all(v["n_accept"] == gamma)
        assert np.array_equal(v["out_tokens"][:, :gamma], dr["x"])


def test_zero_target_probability_rejects_first(orc):
    R, V = 200, 12
    rng = np.random.default_rng(2)
    U = rng.standard_normal((R, 2, V)).astype(np.float32)
    W1, W2t = _zero_bias(V)
    h = np.zeros((R, 2, 1), np.float32)
    dr = orc.draft_markov(U, h, W1, W2t, np.zeros(2, np.float32), np.zeros(R, np.int32), seed=6)
    ell = np.full(R, 2)
    tags = wlmod.tags_from_ell(ell)
    T = rng.standard_normal((len(tags), V)).astype(np.float32)
    for i, (rq, j) in enumerate(tags):
        if j == 0:
            T[i, dr["x"][rq, 0]] = -1e30  # p(x_1) = 0
    v = orc.verify(T, tags, np.zeros(R, np.int32), dr["x"], dr["logq"].astype(np.float32),
                   dr["lse"].astype(np.float32), U, W1, W2t, seed=6)
    assert np.all(v["n_accept"] == 0)
    assert np.all(v["out_tokens"][:, 0] != dr["x"][:, 0])  # residual excludes x_1
    assert np.all(v["out_tokens"][:, 1:] == -1)
    assert np.array_equal(v["next_anchor"], v["out_tokens"][:, 0])


def test_bonus_token_follows_target(orc):
    # l = 0: no draft token is tested and the bonus token is a plain sample of p_0
    V, R, cycles = 5, 5000, 40
    rng = np.random.default_rng(8)
    p_logits = rng.standard_normal(V).astype(np.float32)
    U = np.zeros((R, 1, V), np.float32)
    T_rows = np.broadcast_to(p_logits, (R, 2, V)).copy()
    counts = np.zeros(V, np.int64)
    for cyc in range(cycles):
        _, v = _draft_then_verify(orc, U, T_rows, np.zeros(R, np.int64), seed=10, cycle=cyc)
        assert np.all(v["n_accept"] == 0)
        counts += np.bincount(v["out_tokens"][:, 0], minlength=V)
    p = special.softmax(p_logits.astype(np.float64))
    assert stats.chisquare(counts, p * counts.sum()).pvalue > 1e-4


def test_lse_p_and_logp(orc):
    R, gamma, V = 3, 3, 40
    rng = np.random.default_rng(3)
    U = rng.standard_normal((R, gamma, V)).astype(np.float32)
    ell = np.array([3, 0, 2])
    T_rows = rng.standard_normal((R, gamma + 1, V)).astype(np.float32)
    d, v = _draft_then_verify(orc, U, T_rows, ell, seed=1, cycle=0)
    tags = wlmod.tags_from_ell(ell)
    T = np.stack([T_rows[rq, j] for rq, j in tags]).astype(np.float64)
    np.testing.assert_allclose(v["lse_p"], special.logsumexp(T, axis=1), rtol=0, atol=1e-12)
    for i, (rq, j) in enumerate(tags):
        if j < ell[rq]:
            assert v["logp"][i] == pytest.approx(T[i, d["x"][rq, j]] - v["lse_p"][i], abs=1e-12)
        else:
            assert np.isnan(v["logp"][i])


def test_malformed_tags_rejected(orc):
    R, gamma, V = 2, 2, 8
    U = np.zeros((R, gamma, V), np.float32)
    W1, W2t = _zero_bias(V)
    x = np.zeros((R, gamma), np.int32)
    lq = np.zeros((R, gamma), np.float32)
    good = wlmod.tags_from_ell([1, 1])
    T = np.zeros((len(good), V), np.float32)
    orc.verify(T, good, np.zeros(R, np.int32), x, lq, lq, U, W1, W2t)
    for bad in ([[0, 0], [0, 2], [1, 0], [1, 1]],   # gap in positions
                [[0, 0], [0, 1], [0, 0], [1, 0]],   # request repeated
                [[0, 0], [0, 1], [1, 1], [1, 2]]):  # request 1 without position 0
        with pytest.raises(ValueError):
            orc.verify(T, np.array(bad, np.int32), np.zeros(R, np.int32), x, lq, lq, U, W1, W2t)


def test_final_sample_is_the_inverse_cdf_draw(orc):
    # l = 0: the final token is the inverse-CDF draw from p_0 with one stream-2
    # uniform (counter (0, position 0, request, cycle), word 0): the first v whose
    # cumulative probability exceeds u; gap holds the distances of u to the
    # lower and upper ends of that v's interval, runner the indices across them
    R, V = 40, 30
    rng = np.random.default_rng(12)
    U = rng.standard_normal((R, 1, V)).astype(np.float32)
    T_rows = rng.standard_normal((R, 2, V)).astype(np.float32)
    seed, cycle = 5, 9
    _, v = _draft_then_verify(orc, U, T_rows, np.zeros(R, np.int64), seed=seed, cycle=cycle)
    for rq in range(R):
        p = special.softmax(T_rows[rq, 0].astype(np.float64))
        cdf = np.cumsum(p)
        u = orc.uniform(orc.philox_word(seed, 0, 0, rq, cycle, 2, 0))
        y = int(np.searchsorted(cdf, u * cdf[-1], side="right"))
        assert v["out_tokens"][rq, 0] == y
        lo = u * cdf[-1] - (cdf[y - 1] if y > 0 else 0.0)
        hi = cdf[y] - u * cdf[-1]
        assert v["gap"][rq, 0] == pytest.approx(lo / cdf[-1], abs=1e-12)
        assert v["gap"][rq, 1] == pytest.approx(hi / cdf[-1], abs=1e-12)
        assert v["runner"][rq, 0] == (y - 1 if y > 0 else -1)
        assert v["runner"][rq, 1] == (y + 1 if y + 1 < V else -1)
