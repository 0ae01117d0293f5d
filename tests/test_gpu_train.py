"""GPU parity of the drafter training losses (DSpark digest, Module F, eqs. 8-12)
with the oracle.

Tolerances, from the arithmetic: the kernel sums exp terms in fp32 with the
MUFU exponential (relative error about 2^-22 per term, arguments |z - lse| < 60
add about 60 * 2^-23), so a sum over V terms is within ~1e-5 relative; lse_d,
lse_t and ce (magnitude <= ~30) within 1e-4 absolute, tv and c* (<= 2) within
1e-4, bce within 1e-4, the fp64 loss totals within 1e-4 relative.  The gradient
element g = w/B [a_ce (p_d - onehot) + a_tv p_d (sgn - m)] is compared within
2e-5 relative to its row's scale w/B plus 1e-4 of |g|; an element may differ by
more only where p_d and p_t are so close that the sign sgn(p_d - p_t) is decided
by rounding (|p_d - p_t| < 1e-4 p_d, counted and required to be rare).
"""
import numpy as np
import pytest
import torch

from parity import host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _np(t):
    a = host(t)
    return a


def _probs(z):
    z = z.astype(np.float64)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _widen(t):
    return t.float().cpu().numpy()


def _check(orc, inp, gamma, rows=None, want_grad=True):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dsp.train_losses(inp["zd"], inp["zt"], inp["xs"], inp["s"], gamma, want_grad=want_grad, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    N, V = inp["zd"].shape
    sel = np.arange(N) if rows is None else np.asarray(rows)
    zd, zt = _np(inp["zd"]), _np(inp["zt"])
    xs, s = host(inp["xs"]), host(inp["s"])
    if rows is None:
        ref = orc.train_losses(zd, zt, xs, s, gamma, want_grad=want_grad)
        ref_rows = ref
    else:
        # whole blocks only: the oracle's position weights follow the row index
        ref_rows = orc.train_losses(zd[sel], zt[sel], xs[sel], s[sel], gamma, want_grad=want_grad)
        ref = None
    row = host(out["row"])[sel]
    for j, k in enumerate(("lse_d", "lse_t", "ce", "tv", "cstar", "bce")):
        assert np.abs(row[:, j] - ref_rows[k]).max() <= TOL, k
    if ref is not None:
        loss = host(out["loss"])
        for j, k in enumerate(("L_ce", "L_tv", "L_conf", "L")):
            assert abs(loss[j] - ref[k]) <= TOL * max(1.0, abs(ref[k])), k
    if want_grad:
        B_all = N // gamma
        B_sel = len(sel) // gamma
        # the oracle on a subset divides by its own block count: rescale to the full batch
        scale = B_sel / B_all
        gz = host(out["grad_z"])[sel]
        rz = ref_rows["grad_z"] * scale
        w = np.exp(-(sel % gamma) / gamma) / B_all
        tol = 2e-5 * w[:, None] + 1e-4 * np.abs(rz)
        bad = np.abs(gz - rz) > tol
        if bad.any():
            pd = _probs(_widen(inp["zd"])[sel]) if rows is not None else _probs(_widen(inp["zd"]))
            pt = _probs(_widen(inp["zt"])[sel]) if rows is not None else _probs(_widen(inp["zt"]))
            near = np.abs(pd - pt) < 1e-4 * pd
            assert np.all(near[bad]), "gradient differs away from a sign near-tie"
            assert bad.sum() <= max(3, 1e-5 * bad.size)
        gs = host(out["grad_s"])[sel]
        assert np.abs(gs - ref_rows["grad_s"] * scale).max() <= 1e-6
    return out


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_small_parity(orc, dtype):
    inp = W.train_loss_inputs(3, 4, 4104, dtype=dtype, seed=1, device="cuda")
    _check(orc, inp, 4)


def test_forward_only_and_single_row(orc):
    inp = W.train_loss_inputs(1, 1, 808, dtype=torch.bfloat16, seed=2, device="cuda")
    _check(orc, inp, 1, want_grad=False)


def test_full_size_sampled_blocks(orc):
    # the bench's workload: 64 blocks of 8 positions over V = 151936; two blocks checked
    B, gamma, V = 64, 8, 151936
    inp = W.train_loss_inputs(B, gamma, V, seed=3, device="cuda")
    rows = np.concatenate([np.arange(5 * gamma, 6 * gamma), np.arange(63 * gamma, 64 * gamma)])
    _check(orc, inp, gamma, rows=rows)


def test_many_rows_per_cluster(orc):
    # 160 rows over the resident kernel's clusters of 8 CTAs: every cluster
    # reloads its slices several times; every element checked
    inp = W.train_loss_inputs(40, 4, 4104, dtype=torch.bfloat16, seed=6, device="cuda")
    _check(orc, inp, 4)


def test_tiny_vocab_empty_slices(orc):
    # V = 16 over 8 CTAs: slices are rounded to 16 bytes, so six CTAs hold nothing
    inp = W.train_loss_inputs(2, 3, 16, dtype=torch.bfloat16, seed=7, device="cuda")
    _check(orc, inp, 3)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_streaming_kernel(orc, dtype):
    # V = 262144: a CTA's slice pair (128 KB for bf16, 256 KB for f32) leaves no
    # room for a second CTA on the SM, so the rows stream through L2 instead
    inp = W.train_loss_inputs(1, 2, 262144, dtype=dtype, seed=8, device="cuda")
    _check(orc, inp, 2)


def test_bad_token_reported():
    inp = W.train_loss_inputs(1, 2, 64, dtype=torch.float32, seed=5, device="cuda")
    inp["xs"][1] = 64
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsp.train_losses(inp["zd"], inp["zt"], inp["xs"], inp["s"], 2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dsp.ERR_RANGE
