"""Pins of the oracle's RNN-head draft (eq. 6 of the DSpark digest).

Special projections reduce eq. (6) to closed forms checked with numpy:
* W_o = [0 | I | 0] gives B_k = W_2^T tanh(W_1[x_{k-1}]) for any gate/candidate.
* W_o = [I | 0 | 0], W_c = [0 | I | 0] and a gate fixed at sigma(beta) through a
  constant hidden state give s_k = g s_{k-1} + (1 - g) tanh(W_1[x_{k-1}]),
  B_k = W_2^T tanh(s_{k-1}); this fixes the block order of z_k, which of g and
  1 - g multiplies the old state, and that B_k reads s_{k-1} (s_0 = 0).
"""
import numpy as np
from scipy import special


def _base(R, gamma, V, r, d, seed=0):
    rng = np.random.default_rng(seed)
    U = rng.standard_normal((R, gamma, V)).astype(np.float32)
    W1 = (rng.standard_normal((V, r))).astype(np.float32)
    W2t = (rng.standard_normal((V, r)) / np.sqrt(r)).astype(np.float32)
    w = (rng.standard_normal(d + r) / np.sqrt(d + r)).astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    return rng, U, W1, W2t, w, anchor


def test_output_projection_on_embedding(orc):
    R, gamma, V, r, d = 3, 4, 40, 6, 5
    rng, U, W1, W2t, w, anchor = _base(R, gamma, V, r, d)
    h = rng.standard_normal((R, gamma, d)).astype(np.float32)
    W = rng.standard_normal((3 * r, 2 * r + d)).astype(np.float32)
    W[2 * r:] = 0.0
    W[2 * r:, r:2 * r] = np.eye(r, dtype=np.float32)
    out = orc.draft_rnn(U, h, W1, W2t, W, w, anchor, seed=4, want_z=True)
    for rq in range(R):
        prev = anchor[rq]
        for k in range(gamma):
            A = np.tanh(W1[prev].astype(np.float64))
            np.testing.assert_allclose(out["A"][rq, k], A, rtol=0, atol=1e-14)
            expect = U[rq, k] + W2t.astype(np.float64) @ A
            np.testing.assert_allclose(out["z"][rq, k], expect, rtol=0, atol=1e-12)
            prev = out["x"][rq, k]


def test_state_recurrence(orc):
    R, gamma, V, r, d = 2, 5, 30, 4, 8
    rng, U, W1, W2t, w, anchor = _base(R, gamma, V, r, d, seed=3)
    h = np.ones((R, gamma, d), np.float32)
    beta = np.log(4.0)  # gate sigma(beta) = 0.8
    W = np.zeros((3 * r, 2 * r + d), np.float32)
    W[:r, 2 * r:] = beta / d                      # W_g: reads only h (constant 1)
    W[r:2 * r, r:2 * r] = np.eye(r)               # W_c: candidate = tanh(W_1[x_{k-1}])
    W[2 * r:, :r] = np.eye(r)                     # W_o: output = tanh(s_{k-1})
    out = orc.draft_rnn(U, h, W1, W2t, W, w, anchor, seed=8, cycle=1, want_z=True)
    g = special.expit(np.float64(np.float32(beta / d)) * d)
    for rq in range(R):
        s = np.zeros(r)
        prev = anchor[rq]
        for k in range(gamma):
            A = np.tanh(s)
            np.testing.assert_allclose(out["A"][rq, k], A, rtol=0, atol=1e-14)
            np.testing.assert_allclose(out["z"][rq, k], U[rq, k] + W2t.astype(np.float64) @ A,
                                       rtol=0, atol=1e-12)
            s = g * s + (1 - g) * np.tanh(W1[prev].astype(np.float64))
            prev = out["x"][rq, k]
    # B_1 = W_2^T tanh(s_0) = 0 exactly
    np.testing.assert_array_equal(out["z"][:, 0], U[:, 0].astype(np.float64))


def test_initial_state_and_confidence(orc):
    R, gamma, V, r, d = 2, 3, 20, 4, 3
    rng, U, W1, W2t, w, anchor = _base(R, gamma, V, r, d, seed=5)
    h = rng.standard_normal((R, gamma, d)).astype(np.float32)
    W = np.zeros((3 * r, 2 * r + d), np.float32)
    W[2 * r:, :r] = np.eye(r)                     # output reads s_{k-1}
    W[:r, 2 * r:] = 50.0                          # gate: saturated by |h| (sign of sum h)
    s0 = rng.standard_normal((R, r)).astype(np.float32)
    out = orc.draft_rnn(U, h, W1, W2t, W, w, anchor, s0=s0, want_z=True)
    np.testing.assert_allclose(out["A"][:, 0], np.tanh(s0.astype(np.float64)), atol=1e-14)
    # the confidence head is eq. (7), identical to the Markov head's
    ref = orc.draft_markov(U, h, W1, W2t, w, anchor)
    for rq in range(R):
        prev = anchor[rq]
        for k in range(gamma):
            feat = np.concatenate([h[rq, k].astype(np.float64), W1[prev].astype(np.float64)])
            np.testing.assert_allclose(out["c"][rq, k], special.expit(w.astype(np.float64) @ feat),
                                       rtol=1e-13)
            prev = out["x"][rq, k]
    assert ref["c"].shape == out["c"].shape
