"""GPU parity of the acceptance diagnostics (DSpark digest, analysis 1) with the
oracle: integer counts, compared exactly.

* Random outcomes (n, ell) of many requests, several calls accumulating into
  the same counters, requests missing from a cycle (ell < 0), ell omitted.
* The outcomes of real decoding cycles (draft + verify of a small workload),
  counted on the GPU and, from the same outcomes copied to the host, by the
  oracle.
* A request with more accepted than verified tokens is reported in the error
  word and skipped.
"""
import numpy as np
import pytest
import torch

from parity import host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _cmp(gpu, ref):
    for k in ("reached", "accepted", "tau_hist", "ell_hist"):
        assert np.array_equal(host(gpu[k]).astype(np.uint64), ref[k]), k


@pytest.mark.parametrize("R,gamma", [(1, 1), (37, 5), (5000, 16), (300, 1024)])
def test_random_outcomes_accumulate(orc, R, gamma):
    rng = np.random.default_rng(R + gamma)
    gpu, ref = None, None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(3):
        ell = rng.integers(-1, gamma + 1, R).astype(np.int32)
        n = np.array([rng.integers(0, l + 1) if l >= 0 else rng.integers(0, gamma + 1) for l in ell], np.int32)
        ell_arg = None if call == 2 else ell
        if ell_arg is None:
            n = np.minimum(np.abs(n), gamma).astype(np.int32)
        gpu = dsp.accept_stats(torch.as_tensor(n, device="cuda"), gamma,
                               ell=None if ell_arg is None else torch.as_tensor(ell_arg, device="cuda"),
                               counters=gpu, err=err)
        ref = orc.accept_stats(n, ell_arg, gamma=gamma, into=ref)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _cmp(gpu, ref)


def test_counts_of_decoding_cycles(orc):
    wl = W.small("qwen4b", R=24, gamma=6, V=3000, r=64, d=32)
    inp = W.draft_inputs(wl, seed=4, device="cuda")
    tags = W.tags_from_ell(np.full(wl.R, wl.gamma))
    T = W.target_logits(wl, inp["U"], inp["U_bonus"], tags, seed=4)
    tags_d = torch.as_tensor(tags, device="cuda")
    gpu, ref = None, None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for cycle in range(4):
        d = dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                             seed=3, cycle=cycle, err=err)
        v = dsp.verify(T, tags_d, inp["anchor"], d["x"], d["logq"], d["lse"], inp["U"], inp["W1"], inp["W2t"],
                       seed=3, cycle=cycle, err=err)
        gpu = dsp.accept_stats(v["n_accept"], wl.gamma, counters=gpu, err=err)
        torch.cuda.synchronize()
        ref = orc.accept_stats(host(v["n_accept"]), None, gamma=wl.gamma, into=ref)
    assert int(err.item()) == 0
    _cmp(gpu, ref)
    assert int(host(gpu["tau_hist"]).sum()) == 4 * wl.R


def test_bad_request_reported_and_skipped(orc):
    n = torch.tensor([2, 3, 1], dtype=torch.int32, device="cuda")
    ell = torch.tensor([2, 2, 4], dtype=torch.int32, device="cuda")  # request 1: 3 accepted of 2
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu = dsp.accept_stats(n, 4, ell=ell, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dsp.ERR_RANGE
    ref = orc.accept_stats([2, 1], [2, 4], gamma=4)  # the two valid requests
    _cmp(gpu, ref)
