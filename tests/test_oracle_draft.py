"""Pins of the oracle's Markov-head draft (eqs. 4, 5 and 7 of the DSpark digest).

* eq. (5): the bias of step k equals row x_{k-1} of the explicit V x V matrix
  W_1 W_2 (numpy matmul on a tiny vocabulary), so a wrong gather index or a
  transposed operand fails.
* eq. (4): lse equals scipy's logsumexp of the logits; exp(log q) is the softmax
  probability of the sampled token.
* Gumbel-max sampling: 10^6 sampled tokens follow softmax(U + B) (chi-square).
* eq. (7): closed-form special cases (w = 0 gives 1/2; a weight vector that only
  sees the embedding part reads W_1[x_{k-1}], not W_1[x_k]; temperature divides
  the logit).
"""
import numpy as np
import pytest
from scipy import special, stats


def _inputs(R, gamma, V, r, d, seed=0, scale=3.0):
    rng = np.random.default_rng(seed)
    U = (rng.standard_normal((R, gamma, V)) * scale).astype(np.float32)
    W1 = (rng.standard_normal((V, r)) / np.sqrt(r)).astype(np.float32)
    W2t = (rng.standard_normal((V, r)) / np.sqrt(r)).astype(np.float32)
    h = rng.standard_normal((R, gamma, d)).astype(np.float32)
    w = (rng.standard_normal(d + r) / np.sqrt(d + r)).astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    return U, h, W1, W2t, w, anchor


def test_bias_equals_explicit_transition_matrix(orc):
    R, gamma, V, r, d = 3, 5, 64, 8, 16
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d, scale=1.0)
    out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=5, want_z=True)
    Bfull = W1.astype(np.float64) @ W2t.astype(np.float64).T  # V x V, eq. (5)
    for rq in range(R):
        prev = anchor[rq]
        for k in range(gamma):
            expect = U[rq, k].astype(np.float64) + Bfull[prev]
            np.testing.assert_allclose(out["z"][rq, k], expect, rtol=0, atol=1e-12)
            prev = out["x"][rq, k]


def test_lse_and_logq(orc):
    R, gamma, V, r, d = 2, 4, 300, 8, 8
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d)
    out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=1, cycle=3, want_z=True)
    z = out["z"]
    np.testing.assert_allclose(out["lse"], special.logsumexp(z, axis=-1), rtol=0, atol=1e-12)
    sm = special.softmax(z, axis=-1)
    q = np.take_along_axis(sm, out["x"][..., None].astype(np.int64), -1)[..., 0]
    np.testing.assert_allclose(np.exp(out["logq"]), q, rtol=1e-12)
    assert np.all(out["gap"] > 0)


def test_gumbel_max_frequencies_match_softmax(orc):
    # 1000 identical requests x 1000 cycles = 10^6 draws of x_1
    R, V, r, d, cycles = 1000, 8, 4, 4, 1000
    rng = np.random.default_rng(11)
    Urow = rng.standard_normal(V).astype(np.float32)
    U = np.broadcast_to(Urow, (R, 1, V)).copy()
    W1 = (rng.standard_normal((V, r)) * 0.5).astype(np.float32)
    W2t = (rng.standard_normal((V, r)) * 0.5).astype(np.float32)
    h = np.zeros((R, 1, d), np.float32)
    w = np.zeros(d + r, np.float32)
    anchor = np.full(R, 3, np.int32)
    counts = np.zeros(V, np.int64)
    z = None
    for cyc in range(cycles):
        out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=1234, cycle=cyc, want_z=(cyc == 0))
        if z is None:
            z = out["z"][0, 0]
        counts += np.bincount(out["x"][:, 0], minlength=V)
    p = special.softmax(z)
    res = stats.chisquare(counts, p * counts.sum())
    assert res.pvalue > 1e-4, (counts, p)


def test_confidence_closed_forms(orc):
    R, gamma, V, r, d = 2, 3, 50, 4, 6
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d)
    # w = 0 -> sigma(0) = 1/2 exactly
    out = orc.draft_markov(U, h, W1, W2t, np.zeros(d + r, np.float32), anchor)
    assert np.all(out["c"] == 0.5)
    # a weight vector that only reads the embedding block: c_k = sigma(sum W_1[x_{k-1}])
    we = np.concatenate([np.zeros(d), np.ones(r)]).astype(np.float32)
    out = orc.draft_markov(U, h, W1, W2t, we, anchor)
    for rq in range(R):
        prev = anchor[rq]
        for k in range(gamma):
            expect = special.expit(W1[prev].astype(np.float64).sum())
            np.testing.assert_allclose(out["c"][rq, k], expect, rtol=1e-14)
            prev = out["x"][rq, k]
    # only the hidden block: c_k = sigma(sum h_k), temperature divides the logit
    wh = np.concatenate([np.ones(d), np.zeros(r)]).astype(np.float32)
    T = np.array([1.0, 2.0, 0.5], np.float32)
    out = orc.draft_markov(U, h, W1, W2t, wh, anchor, sts_T=T)
    expect = special.expit(h.astype(np.float64).sum(-1) / T[None, :])
    np.testing.assert_allclose(out["c"], expect, rtol=1e-14)


def test_bf16_inputs_widen_exactly(orc):
    import torch
    R, gamma, V, r, d = 2, 2, 40, 8, 8
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d)
    to16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    tb = [to16(a) for a in (U, h, W1, W2t)]
    out16 = orc.draft_markov(*[bits(t) for t in tb], w, anchor, seed=2, want_z=True)
    out32 = orc.draft_markov(*[t.float().numpy() for t in tb], w, anchor, seed=2, want_z=True)
    for key in ("x", "logq", "lse", "c", "z"):
        np.testing.assert_array_equal(out16[key], out32[key])


def test_request_subset_matches_full(orc):
    R, gamma, V, r, d = 5, 3, 80, 4, 4
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d)
    full = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=9, cycle=2)
    sub = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=9, cycle=2, reqs=[4, 1])
    for key in ("x", "logq", "lse", "c"):
        np.testing.assert_array_equal(sub[key], full[key][[4, 1]])


def test_bad_anchor_rejected(orc):
    R, gamma, V, r, d = 2, 2, 10, 4, 4
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d)
    anchor[1] = V
    with pytest.raises(ValueError):
        orc.draft_markov(U, h, W1, W2t, w, anchor)


def test_sample_gap_and_runner_up_by_brute_force(orc):
    """The reported token is the argmax of z + g, the runner-up the second place and
    the gap their difference, with g = -log(-log u) of the stream-0 Philox words
    recomputed here word by word."""
    R, gamma, V, r, d = 2, 3, 40, 4, 2
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d, seed=4, scale=1.0)
    seed, cycle = 77, 5
    out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=seed, cycle=cycle, want_z=True)
    for rq in range(R):
        for k in range(gamma):
            g = np.array([-np.log(-np.log(orc.uniform(orc.philox_word(seed, v // 4, k + 1, rq, cycle, 0, v % 4))))
                          for v in range(V)])
            score = out["z"][rq, k] + g
            order = np.argsort(-score, kind="stable")
            assert out["x"][rq, k] == order[0]
            assert out["runner"][rq, k] == order[1]
            assert out["gap"][rq, k] == pytest.approx(score[order[0]] - score[order[1]], abs=1e-12)
