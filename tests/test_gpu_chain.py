"""Chained decoding cycles on the GPU against the oracle's own chain.

The DSpark digest's production section runs the cycle without a pause: the
capacity K the asynchronous scheduler admits comes from the confidences of two
cycles earlier, the current order of the survival products decides which
positions fill it, there is no early-stop break, and the flattened verify
batch carries a (request, position) marker tensor.  Here 32 cycles of a
production-shaped case (R = 64, gamma = 16, V = 8192, r = 256, bf16 on the
tensor-core kernels, sawtooth SPS table, asynchronous scheduler) chain

    draft -> schedule (K from cycle t-2) -> marker tensor -> verify -> next anchor

on the GPU entirely through the library (device-side K history, row count and
tags), while the oracle runs its own chain from the same seeded inputs: its own
draft, its own scheduler with its own K history, its own verification and
anchors.  Every cycle compares the stages request by request:

- draft: tokens exact, log q / c within 1e-4, lse within 1e-3 (tests/parity.py);
- scheduler: the kernel reproduces the oracle's scheduler bit for bit on the
  confidences it was given; against the oracle's own chain, verify lengths and
  K exactly and Theta within 1e-5 relative (the confidences agree within 1e-4
  only, so the fixed-point sums differ in their last units);
- verification: accepted counts and emitted tokens exactly, per-row log p and
  log-sum-exp within tolerance.

A near tie (a draft token whose oracle block-score gap is below 1e-3 or whose
entry draw lies within 1e-4 of the block's mass from a CDF boundary, a correction or
bonus token whose inverse-CDF target lies within 1e-4 of the total weight from
a CDF boundary, an acceptance decision whose oracle margin is below 1e-4) is a
counted flip.  A
flipped request leaves that cycle's later comparisons; the scheduler sees the
confidences of every request, so a flip can move verify lengths anywhere.  A
difference in verify lengths or K from the oracle's chain counts as a flip (the
confidences agree within 1e-4, and the kernel matched the oracle's scheduler
bit for bit on its own confidences).  After a cycle with a flip the oracle's
chain continues from the GPU's anchors and K history (it follows the GPU only
after a counted near tie).  Flips must stay below 0.1 % of the compared tokens.
"""
import numpy as np
import pytest
import torch

import oracle_pool
from parity import TOL_C, compare_draft, compare_verify, host, record
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CYCLES = 32
SEED = 1234


def _cycle_inputs(wl, base, t):
    """Base logits and hidden states of cycle t (fresh each cycle); weights and
    the first anchors come from `base`, the inputs of cycle 0."""
    inp = W.draft_inputs(wl, seed=500 + t, device="cuda")
    out = {k: base[k] for k in ("W1", "W2t", "w")}
    out.update({k: inp[k] for k in ("U", "U_bonus", "h")})
    return out


def _rows_of(tags, gamma):
    t = np.asarray(tags, np.int64)
    return t[:, 0] * (gamma + 1) + t[:, 1]


@pytest.mark.parametrize("wl", [W.small("prod", R=64, gamma=16, V=8192, r=256, d=64)],
                         ids=lambda w: f"R{w.R}-g{w.gamma}-V{w.V}")
def test_async_chain_matches_oracle_chain(orc, wl):
    R, gm = wl.R, wl.gamma
    base = W.draft_inputs(wl, seed=499, device="cuda")
    B_min, _ = wl.B_range
    sps = W.sps_table(wl, seed=3)
    sps_dev = torch.as_tensor(sps, device="cuda")
    all_rows = W.tags_from_ell(np.full(R, gm))
    hw = {k: host(base[k]) for k in ("W1", "W2t", "w")}

    # GPU chain state (device) and oracle chain state (host)
    anchor_dev = base["anchor"].clone()
    anchor_orc = host(base["anchor"]).copy()
    K_dev = [torch.full((1,), -1, dtype=torch.int32, device="cuda") for _ in range(3)]
    K_orc = [-1, -1, -1]
    N_dev = torch.empty(1, dtype=torch.int32, device="cuda")
    tags_dev = torch.empty((R * (gm + 1), 2), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    flips = compared = admitted = rejections = async_cycles = 0
    for t in range(CYCLES):
        inp = _cycle_inputs(wl, base, t)
        hU, hh = host(inp["U"]), host(inp["h"])
        # the target's logits for every (request, position) of this cycle; each side
        # gathers the rows its own schedule admits
        T_all = W.target_logits(wl, inp["U"], inp["U_bonus"], all_rows, seed=t)

        # ---- GPU chain
        d = dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], anchor_dev,
                             seed=SEED, cycle=t, err=err)
        k_in = K_dev[(t + 1) % 3]  # written at cycle t - 2
        s_out = {"ell": torch.empty(R, dtype=torch.int32, device="cuda"), "K_out": K_dev[t % 3],
                 "theta_best": torch.empty(1, dtype=torch.float64, device="cuda")}
        dsp.schedule(d["c"], sps_dev, B_min, mode=dsp.SCHED_ASYNC, K_in=k_in, out=s_out, err=err)
        dsp.build_tags(s_out["ell"], gm, tags=tags_dev, N_out=N_dev, err=err)
        rows = tags_dev[:, 0].long() * (gm + 1) + tags_dev[:, 1].long()
        T_dev = torch.index_select(T_all, 0, rows.clamp(0, R * (gm + 1) - 1))
        v = dsp.verify(T_dev, tags_dev, anchor_dev, d["x"], d["logq"], d["lse"], inp["U"],
                       inp["W1"], inp["W2t"], N_dev=N_dev, seed=SEED, cycle=t, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, dsp.ERROR_NAMES[int(err.item())]
        gd = {k: host(val) for k, val in d.items()}
        gs = {k: host(val) for k, val in s_out.items()}
        n_rows = int(N_dev.item())
        gv = {k: host(val) for k, val in v.items()}
        gv["lse_p"], gv["logp"] = gv["lse_p"][:n_rows], gv["logp"][:n_rows]

        # ---- oracle chain
        od = oracle_pool.draft(orc.draft_markov, list(range(R)), hU, hh, hw["W1"], hw["W2t"], hw["w"],
                               anchor_orc, seed=SEED, cycle=t)
        K_in = K_orc[(t + 1) % 3]
        os_ = orc.schedule(od["c"].astype(np.float32), sps, B_min, mode=orc.SCHED_ASYNC, K_in=K_in)
        K_orc[t % 3] = os_["K_out"]
        tags_o = W.tags_from_ell(os_["ell"])
        T_o = host(T_all)[_rows_of(tags_o, gm)]
        ov = oracle_pool.verify(orc.verify, list(range(R)), T_o, tags_o, anchor_orc, od["x"],
                                od["logq"].astype(np.float32), od["lse"].astype(np.float32), hU,
                                hw["W1"], hw["W2t"], seed=SEED, cycle=t)
        async_cycles += K_in >= 0

        # ---- stage by stage
        f, n = compare_draft(gd, od, list(range(R)), gm)
        flips, compared = flips + f, compared + n
        flipped = {rq for rq in range(R) if not np.array_equal(gd["x"][rq], od["x"][rq])}
        cycle_flip = bool(flipped)
        # the scheduler kernel itself, bit for bit, on the confidences it was given
        chk = orc.schedule(gd["c"], sps, B_min, mode=orc.SCHED_ASYNC, K_in=int(host(k_in)[0]))
        assert np.array_equal(chk["ell"], gs["ell"]) and chk["K_out"] == int(gs["K_out"][0])
        assert chk["theta_best"] == float(gs["theta_best"][0])
        # against the oracle's own chain: the confidences agree within 1e-4, not bit for
        # bit, so Theta agrees to rounding and the integer decisions exactly, unless a
        # comparison of the scan sat at a near tie
        same_sched = np.array_equal(gs["ell"], os_["ell"]) and int(gs["K_out"][0]) == os_["K_out"]
        if not same_sched:
            assert np.abs(gd["c"] - od["c"]).max() <= TOL_C
            flips += 1
            record(1, 0)
            cycle_flip = True
        else:
            assert abs(float(gs["theta_best"][0]) - os_["theta_best"]) <= 1e-5 * os_["theta_best"]
            assert n_rows == len(tags_o)
            assert np.array_equal(host(tags_dev)[:n_rows], tags_o)
            keep = [rq for rq in range(R) if rq not in flipped]
            if keep:
                f, n = compare_verify(gv, ov, keep, tags_o, gm)
                flips, compared = flips + f, compared + n
                cycle_flip |= f > 0
            admitted += int(os_["ell"].sum())
            rejections += int((ov["n_accept"] < os_["ell"]).sum())

        # ---- next cycle's state
        if cycle_flip:  # follow the GPU after a counted near tie
            anchor_orc = gv["next_anchor"].copy()
            for i in range(3):
                K_orc[i] = int(host(K_dev[i])[0])
        else:
            assert np.array_equal(gv["next_anchor"], ov["next_anchor"])
            assert int(gs["K_out"][0]) == K_orc[t % 3]
            anchor_orc = ov["next_anchor"].copy()
        anchor_dev = v["next_anchor"].clone()

    assert async_cycles == CYCLES - 2  # K from cycle t - 2 from the third cycle on
    assert admitted > 0 and rejections > 0  # the schedule admitted tokens and residuals ran
    assert flips < max(1, 0.001 * compared), (flips, compared)
