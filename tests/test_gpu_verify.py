"""GPU parity of verification.  Draft tokens, log q and lse come from the oracle's
own draft (or from the seeded generator for requests the oracle does not
sample), so no input of the oracle comes from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle_pool
from parity import compare_verify, host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _case(orc, wl, seed, cycle, ell, reqs=None, device="cpu", rnn=False):
    """Inputs of one verify call: oracle draft for `reqs` (all when None),
    seeded synthetic tokens for the rest."""
    inp = W.draft_inputs(wl, seed=seed, device=device)
    hU, hh, hW1, hW2 = (host(inp[k]) for k in ("U", "h", "W1", "W2t"))
    all_reqs = list(range(wl.R)) if reqs is None else list(reqs)
    if rnn:
        ref = oracle_pool.draft(orc.draft_rnn, all_reqs, hU, hh, hW1, hW2, host(inp["W"]),
                                host(inp["w"]), host(inp["anchor"]), seed=seed, cycle=cycle)
    else:
        ref = oracle_pool.draft(orc.draft_markov, all_reqs, hU, hh, hW1, hW2, host(inp["w"]),
                                host(inp["anchor"]), seed=seed, cycle=cycle)
    R, gamma = wl.R, wl.gamma
    rng = np.random.default_rng(seed + 1)
    x = rng.integers(0, wl.V, (R, gamma)).astype(np.int32)
    logq = rng.uniform(-3.0, -0.01, (R, gamma)).astype(np.float32)
    lse = rng.uniform(5.0, 15.0, (R, gamma)).astype(np.float32)
    A = rng.uniform(-1, 1, (R, gamma, wl.r)).astype(np.float32) if rnn else None
    for t, rq in enumerate(reqs if reqs is not None else range(R)):
        x[rq], logq[rq], lse[rq] = ref["x"][t], ref["logq"][t], ref["lse"][t]
        if rnn:
            A[rq] = ref["A"][t]
    tags = W.tags_from_ell(ell)
    T = W.target_logits(wl, inp["U"], inp["U_bonus"], tags, seed=seed)
    return inp, x, logq, lse, A, tags, T


def _gpu_verify(inp, x, logq, lse, A, tags, T, seed, cycle, N_dev=None):
    dev = lambda a: torch.as_tensor(a, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dsp.verify(T.cuda(), dev(tags), inp["anchor"].cuda(), dev(x), dev(logq), dev(lse),
                     inp["U"].cuda(), inp["W1"].cuda(), inp["W2t"].cuda(),
                     A=None if A is None else dev(A), N_dev=N_dev, seed=seed, cycle=cycle, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, dsp.ERROR_NAMES[int(err.item())]
    return {k: host(v) for k, v in out.items()}


def _oracle_verify(orc, inp, x, logq, lse, A, tags, T, seed, cycle, reqs=None):
    reqs = list(range(x.shape[0])) if reqs is None else list(reqs)
    return oracle_pool.verify(orc.verify, reqs, host(T), tags, host(inp["anchor"]), x, logq, lse,
                              host(inp["U"]), host(inp["W1"]), host(inp["W2t"]), A=A, seed=seed,
                              cycle=cycle)


SMALL = [
    (W.WORKLOADS["tiny"], None),
    (W.small("qwen4b", R=12, gamma=4, V=1001, r=24, d=16), None),
    (W.small("heavy", R=20, gamma=6, V=4096 + 17, r=32, d=16), None),
    (W.small("prod", R=9, gamma=3, V=333, r=16, d=8, dtype="f32"), None),
    # tensor-core phase 2: bf16, V % 8 == 0, r a multiple of 64
    (W.small("qwen4b", R=12, gamma=4, V=1000, r=64, d=16), None),
    (W.small("heavy", R=100, gamma=5, V=4096 + 8, r=128, d=16), None),
]


@pytest.mark.parametrize("wl,_", SMALL, ids=lambda v: getattr(v, "name", ""))
@pytest.mark.parametrize("ell_kind", ["all", "random", "zero"])
def test_verify_small(orc, wl, _, ell_kind):
    rng = np.random.default_rng(3)
    ell = {"all": np.full(wl.R, wl.gamma), "zero": np.zeros(wl.R, np.int64),
           "random": rng.integers(0, wl.gamma + 1, wl.R)}[ell_kind]
    seed, cycle = 17, 5
    case = _case(orc, wl, seed, cycle, ell)
    gpu = _gpu_verify(*case, seed, cycle)
    ref = _oracle_verify(orc, *case, seed, cycle)
    compare_verify(gpu, ref, list(range(wl.R)), case[5], wl.gamma)


def test_verify_many_cycles_small(orc):
    wl = W.small("qwen4b", R=16, gamma=5, V=500, r=16, d=8)
    total_rej = 0
    for cycle in range(6):
        ell = np.random.default_rng(cycle).integers(0, wl.gamma + 1, wl.R)
        case = _case(orc, wl, 40 + cycle, cycle, ell)
        gpu = _gpu_verify(*case, 40 + cycle, cycle)
        ref = _oracle_verify(orc, *case, 40 + cycle, cycle)
        compare_verify(gpu, ref, list(range(wl.R)), case[5], wl.gamma)
        total_rej += int((ref["n_accept"] < ell).sum())
    assert total_rej > 0  # the residual path was exercised


@pytest.mark.parametrize("wl", [W.small("rnn", R=6, gamma=4, V=640, r=16, d=16),
                                W.small("rnn", R=70, gamma=3, V=1024, r=64, d=16)],
                         ids=["cuda-cores", "tensor-cores"])
def test_verify_rnn_small(orc, wl):
    ell = np.random.default_rng(2).integers(0, wl.gamma + 1, wl.R)
    case = _case(orc, wl, 8, 2, ell, rnn=True)
    gpu = _gpu_verify(*case, 8, 2)
    ref = _oracle_verify(orc, *case, 8, 2)
    compare_verify(gpu, ref, list(range(wl.R)), case[5], wl.gamma)


def test_verify_device_row_count(orc):
    # capacity rows beyond N_dev are ignored
    wl = W.small("qwen4b", R=5, gamma=3, V=400, r=8, d=8)
    ell = np.array([3, 1, 0, 2, 3])
    inp, x, logq, lse, A, tags, T = _case(orc, wl, 2, 0, ell)
    N = len(tags)
    cap = wl.R * (wl.gamma + 1)
    T_cap = torch.zeros((cap, wl.V), dtype=T.dtype)
    T_cap[:N] = T
    tags_cap = np.zeros((cap, 2), np.int32)
    tags_cap[:N] = tags
    N_dev = torch.tensor([N], dtype=torch.int32, device="cuda")
    gpu = _gpu_verify(inp, x, logq, lse, A, tags_cap, T_cap, 2, 0, N_dev=N_dev)
    ref = _oracle_verify(orc, inp, x, logq, lse, A, tags, T, 2, 0)
    compare_verify({k: (v[:N] if k in ("lse_p", "logp") else v) for k, v in gpu.items()}, ref,
                   list(range(wl.R)), tags, wl.gamma)


# every request at qwen4b, 64 spread over the batch elsewhere (first and last included)
FULL_REQS = {"qwen4b": list(range(64)), "heavy": list(range(0, 256, 4)) + [255],
             "prod": list(range(0, 512, 8)) + [511], "rnn": list(range(0, 128, 2)) + [127]}


@pytest.mark.parametrize("name,ell_kind", [("qwen4b", "all"), ("heavy", "random"), ("prod", "random"),
                                           ("rnn", "all")])
def test_verify_full_size_sampled(orc, name, ell_kind):
    wl = W.WORKLOADS[name]
    reqs = FULL_REQS[name]
    rnn = wl.head == "rnn"
    rng = np.random.default_rng(5)
    ell = np.full(wl.R, wl.gamma) if ell_kind == "all" else rng.integers(0, wl.gamma + 1, wl.R)
    case = _case(orc, wl, 6, 1, ell, reqs=reqs, device="cuda", rnn=rnn)
    gpu = _gpu_verify(*case, 6, 1)
    ref = _oracle_verify(orc, *case, 6, 1, reqs=reqs)
    compare_verify(gpu, ref, reqs, case[5], wl.gamma)
    assert int((ref["n_accept"][reqs] < ell[reqs]).sum()) > 0  # residuals exercised


def test_malformed_tags_report_inval():
    wl = W.small("qwen4b", R=3, gamma=2, V=64, r=8, d=8)
    inp = W.draft_inputs(wl, seed=0)
    tags = np.array([[0, 0], [0, 2], [1, 0], [2, 0]], np.int32)  # gap in request 0
    T = torch.zeros((4, wl.V), dtype=torch.bfloat16)
    z = np.zeros((wl.R, wl.gamma), np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.as_tensor(a, device="cuda")
    dsp.verify(T.cuda(), dev(tags), inp["anchor"].cuda(), dev(np.zeros((3, 2), np.int32)), dev(z),
               dev(z), inp["U"].cuda(), inp["W1"].cuda(), inp["W2t"].cuda(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dsp.ERR_INVAL


def test_verify_repeat_identical_with_dirty_workspace():
    """The tensor-core verification is deterministic: the tile order is dynamic
    (taken from a counter), but the draw's sums are indexed by vocabulary
    position and the tile level is integer arithmetic, so repeated calls give
    identical outputs bit for bit -- also when the caller's workspace holds
    stale data from another call (the tile sums are zeroed by every call)."""
    wl = W.small("heavy", R=300, gamma=4, V=20000, r=128, d=16)  # 3 M-tiles, ~157 tiles
    rng = np.random.default_rng(11)
    ell = rng.integers(0, wl.gamma + 1, wl.R)
    inp = W.draft_inputs(wl, seed=9, device="cuda")
    x = torch.as_tensor(rng.integers(0, wl.V, (wl.R, wl.gamma)).astype(np.int32), device="cuda")
    logq = torch.as_tensor(rng.uniform(-3.0, -0.01, (wl.R, wl.gamma)).astype(np.float32), device="cuda")
    lse = torch.as_tensor(rng.uniform(5.0, 15.0, (wl.R, wl.gamma)).astype(np.float32), device="cuda")
    tags = W.tags_from_ell(ell)
    T = W.target_logits(wl, inp["U"], inp["U_bonus"], tags, seed=9).cuda()
    tags_d = torch.as_tensor(tags, device="cuda")
    nbytes = dsp.verify_workspace_size(T, tags_d, inp["anchor"], x, logq, lse, inp["U"], inp["W1"],
                                       inp["W2t"])
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    outs = []
    for fill in (0, 0xFF, 0x5A):
        ws.fill_(fill)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = dsp.verify(T, tags_d, inp["anchor"], x, logq, lse, inp["U"], inp["W1"], inp["W2t"],
                         seed=3, cycle=7, ws=ws, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, dsp.ERROR_NAMES[int(err.item())]
        outs.append({k: host(v).copy() for k, v in out.items()})
    for o in outs[1:]:
        for k in outs[0]:
            assert np.array_equal(o[k].view(np.uint8), outs[0][k].view(np.uint8)), k
    assert (outs[0]["n_accept"] < ell).any()  # residual draws exercised
