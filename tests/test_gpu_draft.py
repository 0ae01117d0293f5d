"""GPU parity of the draft calls (Markov and RNN heads) against the oracle.

Small cases run the oracle on every request; the standard full-size workloads
(the launch configuration the benchmark times) run it on every request of
qwen4b and on 64 requests spread over the batch elsewhere, split over the host
cores.
"""
import numpy as np
import pytest
import torch

import oracle_pool
from parity import compare_draft, host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(R, gamma):
    """The draft's outputs, with the optional confidence logit requested."""
    f32 = dict(dtype=torch.float32, device="cuda")
    return {"x": torch.empty((R, gamma), dtype=torch.int32, device="cuda"),
            "logq": torch.empty((R, gamma), **f32), "lse": torch.empty((R, gamma), **f32),
            "c": torch.empty((R, gamma), **f32), "conf_logit": torch.empty((R, gamma), **f32)}


def _gpu_draft(inp, seed, cycle, sts_T=None, rnn=False):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sts = None if sts_T is None else torch.as_tensor(sts_T, device="cuda")
    R, gamma, _ = inp["U"].shape
    if rnn:
        out = dsp.draft_rnn(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["W"], inp["w"],
                            inp["anchor"], seed=seed, cycle=cycle, sts_T=sts, err=err,
                            out=_outputs(R, gamma))
    else:
        out = dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                               seed=seed, cycle=cycle, sts_T=sts, err=err, out=_outputs(R, gamma))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, dsp.ERROR_NAMES[int(err.item())]
    return {k: host(v) for k, v in out.items()}


def _oracle_draft(orc, inp, seed, cycle, reqs=None, sts_T=None, rnn=False):
    """The oracle's draft of `reqs` (all when None), the requests split over host threads."""
    args = [host(inp[k]) for k in ("U", "h", "W1", "W2t")]
    reqs = list(range(inp["U"].shape[0])) if reqs is None else list(reqs)
    if rnn:
        return oracle_pool.draft(orc.draft_rnn, reqs, *args, host(inp["W"]), host(inp["w"]),
                                 host(inp["anchor"]), seed=seed, cycle=cycle, sts_T=sts_T)
    return oracle_pool.draft(orc.draft_markov, reqs, *args, host(inp["w"]), host(inp["anchor"]),
                             seed=seed, cycle=cycle, sts_T=sts_T)


def _to_cuda(inp):
    return {k: v.cuda() for k, v in inp.items()}


SMALL = [
    W.WORKLOADS["tiny"],
    W.small("qwen4b", R=10, gamma=3, V=1001, r=24, d=40),        # ragged V and r, bf16
    W.small("heavy", R=33, gamma=5, V=2048 + 63, r=64, d=96),    # several slices + tail
    W.small("prod", R=3, gamma=2, V=129, r=8, d=8, dtype="f32"),
    # tensor-core path: bf16, V % 8 == 0, r a multiple of 64 (partial tiles and M-tiles)
    W.small("qwen4b", R=40, gamma=3, V=5000, r=64, d=32),
    W.small("heavy", R=100, gamma=3, V=4104, r=128, d=16),
    W.small("prod", R=300, gamma=2, V=8192 + 72, r=256, d=16),
    W.small("heavy", R=65, gamma=5, V=2056, r=64, d=20),          # d % 8 != 0, 1 M-tile of 128
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("seed,cycle", [(0, 0), (12345678901, 7)])
def test_markov_small(orc, wl, seed, cycle):
    inp = _to_cuda(W.draft_inputs(wl, seed=seed % 1000))
    gpu = _gpu_draft(inp, seed, cycle)
    ref = _oracle_draft(orc, inp, seed, cycle)
    compare_draft(gpu, ref, list(range(wl.R)), wl.gamma)


def test_markov_temperature(orc):
    wl = W.small("qwen4b", R=6, gamma=4, V=700, r=16, d=32)
    inp = _to_cuda(W.draft_inputs(wl, seed=3))
    T = np.array([1.0, 1.7, 0.6, 2.5], np.float32)
    gpu = _gpu_draft(inp, 5, 1, sts_T=T)
    ref = _oracle_draft(orc, inp, 5, 1, sts_T=T)
    compare_draft(gpu, ref, list(range(wl.R)), wl.gamma)


def test_markov_deterministic():
    wl = W.small("heavy", R=17, gamma=4, V=3000, r=32, d=16)
    inp = _to_cuda(W.draft_inputs(wl, seed=4))
    a = _gpu_draft(inp, 9, 2)
    b = _gpu_draft(inp, 9, 2)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


STEP_CASES = [
    W.small("qwen4b", R=40, gamma=3, V=5000, r=64, d=32),
    W.small("heavy", R=130, gamma=4, V=4104, r=128, d=20),
    W.WORKLOADS["qwen4b"],
]


@pytest.mark.parametrize("wl", STEP_CASES, ids=lambda w: f"{w.name}-R{w.R}")
def test_step_calls_match_one_call(wl):
    """gamma single-step calls and the all-steps call give identical outputs."""
    inp = W.draft_inputs(wl, seed=6, device="cuda")
    whole = _gpu_draft(inp, 31, 2)
    out = {k: torch.empty((wl.R, wl.gamma), dtype=torch.int32 if k == "x" else torch.float32,
                          device="cuda") for k in ("x", "logq", "lse", "c")}
    nbytes = dsp.draft_markov_workspace_size(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"],
                                             inp["anchor"])
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in range(1, wl.gamma + 1):
        dsp.draft_markov_step(k, inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                              out=out, ws=ws, seed=31, cycle=2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for k in ("x", "logq", "lse", "c"):
        assert np.array_equal(host(out[k]), whole[k]), k


# full-size cases: every request at qwen4b, 64 requests spread over the batch
# elsewhere (the first and last included)
FULL_REQS = {"qwen4b": list(range(64)), "heavy": list(range(0, 256, 4)) + [255],
             "prod": list(range(0, 512, 8)) + [511], "rnn": list(range(0, 128, 2)) + [127]}


@pytest.mark.parametrize("name", ["qwen4b", "heavy", "prod"])
def test_markov_full_size_sampled(orc, name):
    reqs = FULL_REQS[name]
    wl = W.WORKLOADS[name]
    inp = W.draft_inputs(wl, seed=1, device="cuda")
    gpu = _gpu_draft(inp, 2024, 3)
    ref = _oracle_draft(orc, inp, 2024, 3, reqs=reqs)
    compare_draft(gpu, ref, reqs, wl.gamma)
    # every drafted token is a valid id and every confidence a probability
    assert gpu["x"].min() >= 0 and gpu["x"].max() < wl.V
    assert np.all((gpu["c"] > 0) & (gpu["c"] < 1))


RNN_SMALL = [
    W.small("rnn", R=5, gamma=4, V=900, r=16, d=24),
    W.small("rnn", R=3, gamma=3, V=257, r=8, d=8, dtype="f32"),
    W.small("rnn", R=70, gamma=3, V=2000, r=64, d=24),   # tensor cores, one M-tile of 128
    W.small("rnn", R=150, gamma=3, V=2000, r=64, d=24),  # tensor cores, 2 M-tiles (the second ragged)
    W.small("rnn", R=40, gamma=4, V=3000, r=128, d=20),  # tensor-core draft, CUDA-core h projection (d % 8)
    W.small("rnn", R=129, gamma=5, V=1024, r=256, d=72), # r = 256, two M-tiles, 2 K slabs of h
]


@pytest.mark.parametrize("wl", RNN_SMALL, ids=lambda w: f"{w.name}-{w.dtype}-r{w.r}")
def test_rnn_small(orc, wl):
    inp = _to_cuda(W.draft_inputs(wl, seed=2))
    gpu = _gpu_draft(inp, 77, 4, rnn=True)
    ref = _oracle_draft(orc, inp, 77, 4, rnn=True)
    compare_draft(gpu, ref, list(range(wl.R)), wl.gamma)
    # the bias operand A_k = tanh(W_o z_k) until the first flip
    for rq in range(wl.R):
        for k in range(wl.gamma):
            np.testing.assert_allclose(gpu["A"][rq, k], ref["A"][rq, k], atol=1e-4)
            if gpu["x"][rq, k] != ref["x"][rq, k]:
                break


def test_rnn_full_size_sampled(orc):
    wl = W.WORKLOADS["rnn"]
    inp = W.draft_inputs(wl, seed=1, device="cuda")
    gpu = _gpu_draft(inp, 11, 0, rnn=True)
    reqs = FULL_REQS["rnn"]
    ref = _oracle_draft(orc, inp, 11, 0, reqs=reqs, rnn=True)
    compare_draft(gpu, ref, reqs, wl.gamma)
    for t, rq in enumerate(reqs):  # the bias operand A_k until the first flip
        for k in range(wl.gamma):
            np.testing.assert_allclose(gpu["A"][rq, k], ref["A"][t, k], atol=1e-4)
            if gpu["x"][rq, k] != ref["x"][t, k]:
                break


def test_bad_anchor_reports_range():
    wl = W.small("qwen4b", R=4, gamma=2, V=300, r=8, d=8)
    inp = _to_cuda(W.draft_inputs(wl, seed=0))
    inp["anchor"][2] = wl.V + 5  # out of range: clamped on the device and reported
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"], err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dsp.ERR_RANGE
