"""Comparison rules between the CUDA path and the oracle.

Tolerances (absolute): log q, log p, confidences and confidence logits 1e-4;
log-sum-exp 1e-3.
Integer results (tokens, verify lengths, accepted counts) must match exactly,
except at a near tie of the oracle:
- a drafted token is drawn in two levels (a Gumbel-max race over 16-entry
  vocabulary blocks, then the entry of the winning block by inverse CDF); it may
  differ where the oracle's two best block scores are closer than 1e-3 -- and
  must then be the token the runner-up block gives -- or where the entry draw's
  target lies within 1e-4 of the block's mass from an end of the drawn entry's
  interval -- and must then be the entry across that end (either end: an entry
  narrower than the tolerance has both within it);
- an acceptance decision may differ where the oracle's margin
  (log p - log q) - log u is below 1e-4 in magnitude;
- a correction or bonus token may differ where its inverse-CDF target lies
  within 1e-4 of the total weight from an end of the drawn entry's interval
  (the positive-weight entry across that end).
Such "flips" end the comparison of that request,
whose later steps legitimately diverge, and are counted: per comparison they
must stay below 0.1 % of the compared tokens (at least one is allowed in a
small case), and LEDGER sums them over the whole test session, where the total
must stay below 0.1 % of all compared tokens (checked when the session ends).
"""
import numpy as np
import torch

TOL_LOGQ = 1e-4
TOL_C = 1e-4
TOL_LOGIT = 1e-4
TOL_LSE = 1e-3
TOL_LOGP = 1e-4
GAP_TOL = 1e-3
MARGIN_TOL = 1e-4
# the correction / bonus draw is an inverse CDF: its near ties are targets within
# this fraction of the total weight of a CDF boundary (fp32 sums over the
# vocabulary move a boundary by ~1e-6 of the total)
CDF_TOL = 1e-4


def host(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return np.asarray(t)


def allowed_flips(n):
    return max(1, int(0.001 * n))


# flips and compared tokens summed over every comparison of the session
LEDGER = {"flips": 0, "compared": 0, "comparisons": 0}


def record(flips, compared):
    LEDGER["flips"] += flips
    LEDGER["compared"] += compared
    LEDGER["comparisons"] += 1


def cdf_near_tie(token, gaps, runners):
    """An inverse-CDF draw landing across an end of the drawn entry's interval:
    `gaps` are the target's distances to the lower and upper ends (fractions of
    the total), `runners` the entries across them; both ends count (an entry
    narrower than the tolerance has both within it)."""
    return any(g < CDF_TOL and token == y for g, y in zip(gaps, runners))


def draft_near_tie(token, ref, t, k):
    """True when `token` is what the oracle's draw of (t, k) gives after a near tie:
    the runner-up block's token at a block-score gap below GAP_TOL, or an entry
    across an end of the drawn entry's interval within CDF_TOL of the target."""
    return ((ref["gap"][t, k] < GAP_TOL and token == ref["runner"][t, k]) or
            cdf_near_tie(token, ref["cdf_gap"][t, k], ref["cdf_runner"][t, k]))


def compare_draft(gpu, ref, reqs, gamma):
    """gpu: dict of [R, gamma] host arrays; ref: oracle output for `reqs`."""
    flips, compared = 0, 0
    for t, rq in enumerate(reqs):
        for k in range(gamma):
            # lse_k and c_k only depend on x_{k-1}, which matched so far
            assert abs(gpu["lse"][rq, k] - ref["lse"][t, k]) <= TOL_LSE, (rq, k)
            assert abs(gpu["c"][rq, k] - ref["c"][t, k]) <= TOL_C, (rq, k)
            if "conf_logit" in gpu:
                assert abs(gpu["conf_logit"][rq, k] - ref["conf_logit"][t, k]) <= TOL_LOGIT, (rq, k)
            compared += 1
            if gpu["x"][rq, k] != ref["x"][t, k]:
                assert draft_near_tie(gpu["x"][rq, k], ref, t, k), (
                    f"token mismatch at request {rq} step {k + 1}: gpu {gpu['x'][rq, k]} "
                    f"oracle {ref['x'][t, k]}; block score gap {ref['gap'][t, k]} "
                    f"(runner-up block's token {ref['runner'][t, k]}), entry CDF margin "
                    f"{ref['cdf_gap'][t, k]} (entry across it {ref['cdf_runner'][t, k]})")
                flips += 1
                break
            assert abs(gpu["logq"][rq, k] - ref["logq"][t, k]) <= TOL_LOGQ, (rq, k)
    assert flips <= allowed_flips(compared), (flips, compared)
    record(flips, compared)
    return flips, compared


def compare_verify(gpu, ref, reqs, tags, gamma):
    """Per-row lse_p / log p and per-request outcomes; near ties are counted."""
    flips, compared = 0, 0
    tags = np.asarray(tags)
    rows_of = {}
    for i, (rq, j) in enumerate(tags):
        rows_of.setdefault(int(rq), []).append(i)
    for rq in reqs:
        rows = rows_of[rq]
        for i in rows:
            assert abs(gpu["lse_p"][i] - ref["lse_p"][i]) <= TOL_LSE, (rq, i)
            if np.isnan(ref["logp"][i]):
                assert np.isnan(gpu["logp"][i]), (rq, i)
            else:
                assert abs(gpu["logp"][i] - ref["logp"][i]) <= TOL_LOGP, (rq, i)
        n = int(ref["n_accept"][rq])
        compared += n + 1
        decisive = [ref["margin"][rows[j]] for j in range(min(n + 1, len(rows) - 1))]
        near = any(abs(m) < MARGIN_TOL for m in decisive)
        if int(gpu["n_accept"][rq]) != n:
            assert near, f"acceptance mismatch at request {rq}: gpu {gpu['n_accept'][rq]} oracle {n}"
            flips += 1
            continue
        g_out, r_out = gpu["out_tokens"][rq], ref["out_tokens"][rq]
        assert np.array_equal(g_out[:n], r_out[:n])
        assert np.all(g_out[n + 1:] == -1)
        if g_out[n] != r_out[n]:
            assert cdf_near_tie(g_out[n], ref["gap"][rq], ref["runner"][rq]), (
                f"final token mismatch at request {rq}: gpu {g_out[n]} oracle {r_out[n]}; "
                f"target's distances to the ends of the oracle token's interval {ref['gap'][rq]}, "
                f"entries across them {ref['runner'][rq]}")
            flips += 1
        assert gpu["next_anchor"][rq] == g_out[n]
    assert flips <= allowed_flips(compared), (flips, compared)
    record(flips, compared)
    return flips, compared
