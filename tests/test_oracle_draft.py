"""Pins of the oracle's Markov-head draft (eqs. 4, 5 and 7 of the DSpark digest).

* eq. (5): the bias of step k equals row x_{k-1} of the explicit V x V matrix
  W_1 W_2 (numpy matmul on a tiny vocabulary), so a wrong gather index or a
  transposed operand fails.
* eq. (4): lse equals scipy's logsumexp of the logits; exp(log q) is the softmax
  probability of the sampled token.
* Sampling (a two-level draw: 16-entry vocabulary blocks by the Gumbel-max rule
  over their masses, then the entry inside the winning block by inverse CDF):
  10^6 sampled tokens follow softmax(U + B) (chi-square) on a vocabulary with
  a short last block; with equal logits the draw reduces to a closed form in
  the Philox words (the block with the largest race uniform, entry
  floor(16 u')); the near-tie records follow from the block scores and the
  cumulative sums, recomputed here from the words.
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


def _chi_square_draws(orc, V, Urow, cycles=1000, R=1000, seed=1234):
    """10^6 draws of x_1 (R identical requests x `cycles` cycles) against softmax."""
    r, d = 4, 4
    rng = np.random.default_rng(11)
    U = np.broadcast_to(Urow.astype(np.float32), (R, 1, V)).copy()
    W1 = (rng.standard_normal((V, r)) * 0.5).astype(np.float32)
    W2t = (rng.standard_normal((V, r)) * 0.5).astype(np.float32)
    h = np.zeros((R, 1, d), np.float32)
    w = np.zeros(d + r, np.float32)
    anchor = np.full(R, 3, np.int32)
    counts = np.zeros(V, np.int64)
    z = None
    for cyc in range(cycles):
        out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=seed, cycle=cyc, want_z=(cyc == 0))
        if z is None:
            z = out["z"][0, 0]
        counts += np.bincount(out["x"][:, 0], minlength=V)
    p = special.softmax(z)
    return stats.chisquare(counts, p * counts.sum()).pvalue, counts, p


def test_sampled_frequencies_match_softmax(orc):
    # V = 40: blocks of 16, 16 and 8 entries; the logits give the blocks very
    # different masses and spread each block's mass unevenly over its entries
    V = 40
    Urow = np.random.default_rng(5).standard_normal(V) * 1.5
    Urow[16:32] -= 2.0
    pval, counts, p = _chi_square_draws(orc, V, Urow)
    assert pval > 1e-4, (counts, p)


def test_equal_logits_reduce_to_the_words(orc):
    """With every logit equal each block of 16 has the same mass, so level 1 picks
    the block with the largest race uniform and level 2 the entry floor(16 u')."""
    R, gamma, V, r, d = 3, 4, 64, 4, 2
    U = np.zeros((R, gamma, V), np.float32)
    W1 = np.zeros((V, r), np.float32)
    W2t = np.zeros((V, r), np.float32)
    h = np.zeros((R, gamma, d), np.float32)
    w = np.zeros(d + r, np.float32)
    anchor = np.arange(R, dtype=np.int32)
    seed, cycle = 99, 7
    out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=seed, cycle=cycle)
    for rq in range(R):
        for k in range(gamma):
            u = [orc.uniform(orc.philox_word(seed, b // 2, k + 1, rq, cycle, 0, 2 * (b % 2))) for b in range(4)]
            b = int(np.argmax(u))
            ue = orc.uniform(orc.philox_word(seed, b // 2, k + 1, rq, cycle, 0, 2 * (b % 2) + 1))
            assert out["x"][rq, k] == 16 * b + int(np.floor(16 * ue)), (rq, k)
            assert out["logq"][rq, k] == pytest.approx(-np.log(V), abs=1e-12)


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


def test_sample_and_near_tie_records_by_brute_force(orc):
    """The reported token, the block-score gap and the runner-up block's token, and
    the entry draw's distances to both ends of the drawn entry's interval with the
    entries across them, recomputed from the
    stream-0 Philox words: block b (16 entries, the last one 8 here) takes words
    2 (b mod 2) and 2 (b mod 2) + 1 of counter (b / 2, k, request, cycle)."""
    R, gamma, V, r, d = 2, 3, 40, 4, 2
    U, h, W1, W2t, w, anchor = _inputs(R, gamma, V, r, d, seed=4, scale=1.0)
    seed, cycle = 77, 5
    out = orc.draft_markov(U, h, W1, W2t, w, anchor, seed=seed, cycle=cycle, want_z=True)
    blocks = [(0, 16), (16, 32), (32, 40)]

    def word(b, k, rq, lane):
        return orc.uniform(orc.philox_word(seed, b // 2, k + 1, rq, cycle, 0, 2 * (b % 2) + lane))

    def entry(e, lo, u):
        cum = np.cumsum(e[lo:])
        target = u * cum[-1]
        j = int(np.argmax(cum > target))
        below = cum[j - 1] if j > 0 else 0.0
        return lo + j, target - below, cum[j] - target, cum[-1]

    for rq in range(R):
        for k in range(gamma):
            z = out["z"][rq, k]
            e = np.exp(z - z.max())
            score = np.array([np.log(e[a:b].sum()) - np.log(-np.log(word(i, k, rq, 0)))
                              for i, (a, b) in enumerate(blocks)])
            order = np.argsort(-score, kind="stable")
            b0, b1 = order[0], order[1]
            x, lo, hi, S = entry(e[:blocks[b0][1]], blocks[b0][0], word(b0, k, rq, 1))
            assert out["x"][rq, k] == x
            assert out["gap"][rq, k] == pytest.approx(score[b0] - score[b1], abs=1e-12)
            assert out["runner"][rq, k] == entry(e[:blocks[b1][1]], blocks[b1][0], word(b1, k, rq, 1))[0]
            assert out["cdf_gap"][rq, k, 0] == pytest.approx(lo / S, abs=1e-12)
            assert out["cdf_gap"][rq, k, 1] == pytest.approx(hi / S, abs=1e-12)
            first, last = blocks[b0][0], blocks[b0][1] - 1
            assert out["cdf_runner"][rq, k, 0] == (x - 1 if x > first else -1)
            assert out["cdf_runner"][rq, k, 1] == (x + 1 if x < last else -1)
