"""GPU parity of the sequential temperature-scaling fit (DSpark digest, Module D)
against the oracle, and its use on the draft's own confidence logits.

Comparison rule.  The kernel computes each product P_k in fp32 (MUFU exp and a
fast reciprocal), the oracle in fp64.  With EPS a bound on |P_gpu - P_oracle|,
the ECE of one grid point can differ in two ways:
- by at most EPS through the values themselves;
- by at most 2/M for every sample whose P lies within EPS of an interior bin
  edge (the only samples that can change bin).

The oracle counts those samples (``near_edge``).  The curves must therefore
agree within EPS + 2 near / M.  The oracle first runs on its own; the fitted
grid index may differ from the oracle's only where the two are that close on
the oracle's curve.  Such a near tie is counted, and only from then on does the
oracle hold the kernel's temperatures (T_prefix), so one near tie does not
derail the later positions.

EPS: per factor sigma(s/T), the exp argument carries (|x| + 2) 2^-23 relative
error and the reciprocal 2 ulp, which gives at most ~5e-7 absolute error per
factor (factors are <= 1).  A product of k factors is then within k * 5e-7.
The kernel also rounds P to units of 2^-16 / n_bins before binning and
summing, which adds at most 2^-17.  The test uses 2e-6 (gamma + 1) + 2^-17.
"""
import numpy as np
import pytest
import torch

from parity import host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _grid(lo, hi, n):
    return np.linspace(lo, hi, n).astype(np.float32)


def _gpu_fit(s, n, grid, n_bins, err=None):
    out = dsp.sts_fit(torch.as_tensor(s, device="cuda"), torch.as_tensor(n, device="cuda"),
                      torch.as_tensor(grid, device="cuda"), n_bins=n_bins, err=err)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items()}


def _check_parity(orc, s, n, grid, n_bins):
    M, gamma = s.shape
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu = _gpu_fit(s, n, grid, n_bins, err=err)
    assert int(err.item()) == 0
    eps = 2e-6 * (gamma + 1) + 2.0 ** -17
    ref = orc.sts_fit(s, n, grid, n_bins=n_bins, edge_eps=eps)  # free-standing
    agree = 0
    for k in range(gamma):
        tol = eps + 2.0 * ref["near_edge"][k] / M + 1e-9
        diff = np.abs(gpu["curve"][k] - ref["curve"][k])
        assert np.all(diff <= tol), (k, int(np.argmax(diff - tol)), diff.max())
        ig = int(np.nonzero(grid == gpu["T"][k])[0][0])
        assert gpu["curve"][k, ig] == gpu["curve"][k].min()   # its own minimum
        assert gpu["ece"][k] == gpu["curve"][k, ig]
        io = int(ref["index"][k])
        if ig == io:
            agree += 1
            continue
        # a counted near tie: both choices within the comparison margin on the oracle's curve
        assert ref["curve"][k, ig] <= ref["curve"][k, io] + tol[ig] + tol[io], k
        # from here on the oracle holds the kernel's temperatures
        ref = orc.sts_fit(s, n, grid, n_bins=n_bins, T_prefix=gpu["T"], edge_eps=eps)
    return gpu, ref, agree


CASES = [
    # (M, gamma, G, n_bins): ragged sample tiles, several grid blocks, 1 and 64 bins
    (1000, 4, 40, 15),
    (1, 3, 7, 10),
    (4096 + 17, 8, 300, 15),
    (2500, 2, 33, 1),
    (3000, 5, 64, 64),
    (777, 1, 256, 20),
]


@pytest.mark.parametrize("M,gamma,G,n_bins", CASES)
def test_parity_small(orc, M, gamma, G, n_bins):
    s, n = W.calibration_set(M, gamma, seed=M + gamma)
    grid = _grid(0.2, 4.0, G)
    _, _, agree = _check_parity(orc, s, n, grid, n_bins)
    assert agree >= gamma - 1


def test_parity_full_size(orc):
    """Held-out set of 65,536 draft blocks of gamma = 16 (e.g. 512 requests x 128
    cycles), 256 temperatures, 15 bins: the size the benchmark times."""
    T_true = np.linspace(1.2, 2.4, 16)
    s, n = W.calibration_set(65536, 16, seed=11, T_true=T_true)
    grid = _grid(0.05, 12.8, 256)
    gpu, ref, agree = _check_parity(orc, s, n, grid, 15)
    assert agree >= 14
    # the acceptance temperature is identified where enough blocks reach the
    # position: >= 5 % of them for positions 1..10 of this set
    assert (n >= 10).mean() > 0.05
    np.testing.assert_allclose(gpu["T"][:10], T_true[:10], rtol=0.1)


def test_deterministic():
    s, n = W.calibration_set(20000, 6, seed=2)
    grid = _grid(0.3, 3.0, 128)
    a = _gpu_fit(s, n, grid, 12)
    b = _gpu_fit(s, n, grid, 12)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_bad_inputs_reported():
    s, n = W.calibration_set(600, 3, seed=4)
    grid = _grid(0.5, 2.0, 16)
    # a non-positive grid point is skipped and reported
    bad = grid.copy()
    bad[0] = -1.0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu_fit(s, n, bad, 10, err=err)
    assert int(err.item()) == dsp.ERR_INVAL
    assert np.all(np.isnan(out["curve"][:, 0])) and np.all(out["T"] != -1.0)
    # NaN logit
    s2 = s.copy()
    s2[5, 1] = np.nan
    err.zero_()
    _gpu_fit(s2, n, grid, 10, err=err)
    assert int(err.item()) == dsp.ERR_NONFINITE
    # accepted length outside 0..gamma
    n2 = n.copy()
    n2[7] = 4
    err.zero_()
    _gpu_fit(s, n2, grid, 10, err=err)
    assert int(err.item()) == dsp.ERR_RANGE


def test_calibrates_the_drafts_own_confidences():
    """Draft with every position verified, collect (confidence logit, accepted
    length) over cycles, fit, and draft again with the fitted temperatures: the
    new confidences are sigma(logit / T_k) and the fitted ECE is no worse than
    the raw one (T = 1 is on the grid)."""
    wl = W.small("qwen4b", R=64, gamma=4, V=4096, r=64, d=64)
    inp = {k: v.cuda() for k, v in W.draft_inputs(wl, seed=6).items()}
    R, gamma = wl.R, wl.gamma
    logits, accepted = [], []
    for cycle in range(24):
        out = {"x": torch.empty((R, gamma), dtype=torch.int32, device="cuda"),
               **{k: torch.empty((R, gamma), device="cuda") for k in ("logq", "lse", "c", "conf_logit")}}
        d = dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                             seed=3, cycle=cycle, out=out)
        ell = np.full(R, gamma, np.int32)
        tags = torch.as_tensor(W.tags_from_ell(ell), device="cuda")
        T_rows = W.target_logits(wl, inp["U"], inp["U_bonus"], host(tags), seed=cycle,
                                 device="cuda")
        v = dsp.verify(T_rows, tags, inp["anchor"], d["x"], d["logq"], d["lse"], inp["U"],
                       inp["W1"], inp["W2t"], seed=3, cycle=cycle)
        logits.append(d["conf_logit"].clone())
        accepted.append(v["n_accept"].clone())
    s = torch.cat(logits)
    n = torch.cat(accepted)
    grid = torch.as_tensor(_grid(0.25, 4.0, 61), device="cuda")  # holds 1.0
    assert 1.0 in host(grid)
    fit = dsp.sts_fit(s, n, grid, n_bins=10)
    raw = dsp.sts_fit(s, n, torch.ones(1, device="cuda"), n_bins=10)
    torch.cuda.synchronize()
    assert np.all(host(fit["ece"])[:1] <= host(raw["ece"])[:1])
    T = fit["T"]
    d2 = dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                          seed=3, cycle=0, sts_T=T,
                          out={"x": torch.empty((R, gamma), dtype=torch.int32, device="cuda"),
                               **{k: torch.empty((R, gamma), device="cuda")
                                  for k in ("logq", "lse", "c", "conf_logit")}})
    torch.cuda.synchronize()
    expect = torch.sigmoid(d2["conf_logit"].double() / T.double()[None, :])
    assert torch.allclose(d2["c"].double(), expect, atol=1e-5)
