"""Pin of the oracle's residual at later positions of the block.

"DSpark explained" section 06 gives the single-token rule: accept x with
probability min(1, p(x)/q(x)), otherwise draw from norm(max(0, p - q)).  The
DSpark digest (overview, step 3; the two-token chain of Appendix A) applies it
along the drafted prefix: position j+1 is tested against the target row j and
the draft distribution q_{j+1} = softmax(U_{j+1} + B(x_j, .)), and the first
rejection draws its replacement from max(0, p_j - q_{j+1}).  Whatever the draft,
the emitted tokens then follow the target exactly.

Here the target is a first-order Markov chain, p(. | prefix) = softmax(Tm[last
token]), so the first three emitted tokens of a stream started at x_0 have the
joint law p(y1 | x0) p(y2 | y1) p(y3 | y2).  The draft is a Markov head with a
strong bias (W_1, W_2 ~ N(0, 1), r = 4) and base logits that differ by
position, gamma = 3, every drafted token verified; a request that emits fewer
than three tokens in a cycle starts the next cycle from its last token.  10^6
streams are tallied over the V^3 = 125 joint outcomes and compared by
chi-square.  Rejections at positions 2 and 3 are frequent, so the U row, the
bias token (or RNN operand) and the draft normaliser the residual uses at j >= 1
all decide the outcome: the test compiles copies of the oracle with each of them
moved one position back (or the bias token one forward) and requires every copy
to fail the same test.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
from scipy import special, stats

import oracle as oracle_mod

V, R_DIM, GAMMA, K_TOKENS = 5, 4, 3, 3
X0 = 0


def _model(rnn):
    rng = np.random.default_rng(20261)
    Tm = rng.normal(0.0, 1.5, (V, V)).astype(np.float32)
    Ud = rng.normal(0.0, 2.0, (GAMMA, V)).astype(np.float32)
    W1 = rng.normal(0.0, 1.0, (V, R_DIM)).astype(np.float32)
    W2t = rng.normal(0.0, 1.0, (V, R_DIM)).astype(np.float32)
    W = rng.normal(0.0, 1.0, (3 * R_DIM, 2 * R_DIM + 1)).astype(np.float32) if rnn else None
    return Tm, Ud, W1, W2t, W


def _streams(orc, n, seed, rnn):
    """First K_TOKENS emitted tokens of n independent streams started at X0, and
    the number of residual draws at positions j >= 1."""
    Tm, Ud, W1, W2t, W = _model(rnn)
    toks = np.full((n, K_TOKENS), -1, np.int64)
    count = np.zeros(n, np.int64)
    anchors = np.full(n, X0, np.int32)
    late_rejections = 0
    cycle = 0
    while (count < K_TOKENS).any():
        act = np.nonzero(count < K_TOKENS)[0]
        m = len(act)
        U = np.ascontiguousarray(np.broadcast_to(Ud, (m, GAMMA, V)))
        h = np.zeros((m, GAMMA, 1), np.float32)
        w = np.zeros(1 + R_DIM, np.float32)
        anc = np.ascontiguousarray(anchors[act])
        if rnn:
            d = orc.draft_rnn(U, h, W1, W2t, W, w, anc, seed=seed, cycle=cycle)
        else:
            d = orc.draft_markov(U, h, W1, W2t, w, anc, seed=seed, cycle=cycle)
        # target row j of a request: the chain's logits after its prefix x_0..x_j
        prev = np.concatenate([anc[:, None], d["x"]], axis=1)
        T = np.ascontiguousarray(Tm[prev.reshape(-1)])
        tags = np.stack([np.repeat(np.arange(m), GAMMA + 1),
                         np.tile(np.arange(GAMMA + 1), m)], axis=1).astype(np.int32)
        v = orc.verify(T, tags, anc, d["x"], d["logq"].astype(np.float32),
                       d["lse"].astype(np.float32), U, W1, W2t,
                       A=d["A"].astype(np.float32) if rnn else None, seed=seed, cycle=cycle)
        n_acc = v["n_accept"]
        late_rejections += int(((n_acc >= 1) & (n_acc < GAMMA)).sum())
        out = v["out_tokens"]
        for j in range(GAMMA + 1):
            take = (j <= n_acc) & (count[act] < K_TOKENS)
            rows = act[take]
            toks[rows, count[rows]] = out[take, j]
            count[rows] += 1
        anchors[act] = v["next_anchor"]
        cycle += 1
    return toks, late_rejections


def _chain_pvalue(orc, n_streams, rnn, batches=4):
    Tm = _model(rnn)[0].astype(np.float64)
    P = special.softmax(Tm, axis=1)  # P[a, b] = p(b | a)
    joint = P[X0][:, None, None] * P[:, :, None] * P[None, :, :]  # [y1, y2, y3]
    counts = np.zeros(V ** K_TOKENS, np.int64)
    late = 0
    per = n_streams // batches
    for b in range(batches):  # a fresh key per batch keeps the streams independent
        toks, lr = _streams(orc, per, seed=9000 + b, rnn=rnn)
        late += lr
        counts += np.bincount((toks[:, 0] * V + toks[:, 1]) * V + toks[:, 2], minlength=V ** 3)
    expected = joint.reshape(-1) * counts.sum()
    # pool the rare outcomes (expected count below 5) into one cell
    rare = expected < 5
    obs = np.append(counts[~rare], counts[rare].sum())
    exp = np.append(expected[~rare], expected[rare].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return stats.chisquare(obs, exp).pvalue, late, counts.sum()


@pytest.mark.parametrize("rnn", [False, True], ids=["markov", "rnn"])
def test_emitted_tokens_follow_the_target_chain(orc, rnn):
    p, late, n = _chain_pvalue(orc, 1_000_000, rnn)
    assert n == 1_000_000
    assert late > 100_000, late  # the residual at j >= 1 decided many streams
    assert p > 1e-4, p


# (source text in the verification function, text of the planted mistake)
MUTANTS = {
    "U row n_r - 1": ("size_t urow = ((size_t)rq * gamma + (size_t)n_r) * (size_t)V;",
                      "size_t urow = ((size_t)rq * gamma + (size_t)(n_r > 0 ? n_r - 1 : 0)) * (size_t)V;"),
    "bias token x[n_r]": ("int32_t xn = n_r == 0 ? anchor[rq] : x[(size_t)rq * gamma + (n_r - 1)];",
                          "int32_t xn = x[(size_t)rq * gamma + n_r];"),
    "draft lse of position n_r": ("double lq = (double)lse[(size_t)rq * gamma + n_r];",
                                  "double lq = (double)lse[(size_t)rq * gamma + (n_r > 0 ? n_r - 1 : 0)];"),
    "RNN operand A row n_r - 1": (
        "b[i] = (double)A[((size_t)rq * gamma + n_r) * (size_t)r + i];",
        "b[i] = (double)A[((size_t)rq * gamma + (n_r > 0 ? n_r - 1 : 0)) * (size_t)r + i];"),
}


class _Mutant:
    """The oracle's Python wrapper bound to a mutated build of its C source."""

    def __init__(self, lib):
        self._lib = lib

    def __getattr__(self, name):
        return getattr(oracle_mod, name)

    def draft_markov(self, *a, **k):
        return self._call(oracle_mod.draft_markov, *a, **k)

    def draft_rnn(self, *a, **k):
        return self._call(oracle_mod.draft_rnn, *a, **k)

    def verify(self, *a, **k):
        return self._call(oracle_mod.verify, *a, **k)

    def _call(self, fn, *a, **k):
        saved = oracle_mod._lib
        oracle_mod._lib = self._lib
        try:
            return fn(*a, **k)
        finally:
            oracle_mod._lib = saved


def _mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "dspark_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site of '{name}' not found once in the oracle"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    inc = os.path.dirname(oracle_mod.__file__)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-I", inc, "-o", str(so), str(path), "-lm"])
    return _Mutant(oracle_mod.bind(ctypes.CDLL(str(so))))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_misplaced_residual_fails_the_chain_test(orc, tmp_path, name):
    mut = _mutant(tmp_path, name)
    p, late, _ = _chain_pvalue(mut, 200_000, rnn=name.startswith("RNN"))
    assert late > 20_000
    assert p < 1e-9, (name, p)
