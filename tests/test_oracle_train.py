"""Pins of the oracle's drafter training losses (DSpark digest, Module F,
eqs. 8-12).

Each position k of a block is weighted by w_k = exp(-(k - 1) / gamma). The
cross-entropy scores the target's token under the draft distribution, the total
variation term is the L1 distance between the draft and target distributions,
and the confidence head is trained by binary cross-entropy towards
c* = 1 - ||p_d - p_t||_1 / 2 (eq. 8). The total is 0.1 L_ce + 0.9 L_tv + L_conf
by default (eq. 12); the losses are averaged over the blocks.

* Closed forms: uniform logits (ce = ln V), equal distributions (tv = 0,
  c* = 1, also after a constant shift of one side), two tokens
  (tv = 2 |sigma(a) - sigma(b)|), c* = sum_v min(p_d, p_t) (the single-token
  acceptance probability, computed here with numpy).
* The position weights and the eq. (12) combination on hand-built rows.
* The gradients against central finite differences of the oracle's own loss,
  with respect to the draft logits (the label c* held fixed) and the
  confidence logits.
"""
import math

import numpy as np
import pytest


def _softmax(z):
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def test_uniform_and_equal_distributions(orc):
    V, gamma = 37, 3
    zd = np.zeros((gamma, V), np.float32)
    zt = np.zeros((gamma, V), np.float32) + 2.5  # a constant shift leaves p_t uniform
    out = orc.train_losses(zd, zt, [0, 5, 36], [0.0, 0.0, 0.0], gamma)
    assert np.allclose(out["ce"], math.log(V), rtol=0, atol=1e-12)
    assert np.allclose(out["tv"], 0.0, atol=1e-15)
    assert np.allclose(out["cstar"], 1.0, atol=1e-15)
    assert np.allclose(out["lse_d"], math.log(V), atol=1e-12)
    assert np.allclose(out["lse_t"], 2.5 + math.log(V), atol=1e-12)
    # sigma(0) = 1/2 against the label 1: bce = ln 2
    assert np.allclose(out["bce"], math.log(2.0), atol=1e-12)


def test_two_tokens_closed_form(orc):
    a, b = 1.3, -0.4
    zd = np.array([[0.0, a]], np.float32)
    zt = np.array([[0.0, b]], np.float32)
    out = orc.train_losses(zd, zt, [1], [0.7], 1)
    sa = 1 / (1 + math.exp(-float(np.float32(a))))
    sb = 1 / (1 + math.exp(-float(np.float32(b))))
    assert out["tv"][0] == pytest.approx(2 * abs(sa - sb), abs=1e-13)
    assert out["cstar"][0] == pytest.approx(1 - abs(sa - sb), abs=1e-13)
    assert out["ce"][0] == pytest.approx(-math.log(sa), abs=1e-13)
    c = 1 / (1 + math.exp(-float(np.float32(0.7))))
    cs = out["cstar"][0]
    assert out["bce"][0] == pytest.approx(-(cs * math.log(c) + (1 - cs) * math.log(1 - c)), abs=1e-12)


def test_cstar_is_the_acceptance_probability(orc):
    # eq. (8): 1 - TV/2 = sum_v min(p_d, p_t), the chance that one drafted token passes
    rng = np.random.default_rng(2)
    zd = rng.normal(0, 2, (6, 300)).astype(np.float32)
    zt = (zd + rng.normal(0, 1, zd.shape)).astype(np.float32)
    out = orc.train_losses(zd, zt, rng.integers(0, 300, 6), np.zeros(6, np.float32), 3)
    pd, pt = _softmax(zd.astype(np.float64)), _softmax(zt.astype(np.float64))
    assert np.allclose(out["cstar"], np.minimum(pd, pt).sum(axis=1), atol=1e-12)
    assert np.allclose(out["tv"], np.abs(pd - pt).sum(axis=1), atol=1e-12)


def test_position_weights_and_combination(orc):
    # two blocks of gamma = 4; only row (block 1, position 3) has a non-uniform draft
    gamma, V = 4, 8
    zd = np.zeros((2 * gamma, V), np.float32)
    zt = np.zeros((2 * gamma, V), np.float32)
    zd[gamma + 2, 3] = 2.0
    xs = np.zeros(2 * gamma, np.int32)
    s = np.full(2 * gamma, 1.5, np.float32)
    out = orc.train_losses(zd, zt, xs, s, gamma)
    w = np.exp(-np.arange(gamma) / gamma)
    ce_u = math.log(V)
    ce_x = math.log(7 + math.exp(2.0))  # -log p(0) with one logit raised to 2
    L_ce = (2 * w.sum() * ce_u - w[2] * ce_u + w[2] * ce_x) / 2
    assert out["L_ce"] == pytest.approx(L_ce, rel=1e-13)
    tv_x = out["tv"][gamma + 2]
    assert out["L_tv"] == pytest.approx(w[2] * tv_x / 2, rel=1e-13)
    assert out["L"] == pytest.approx(0.1 * out["L_ce"] + 0.9 * out["L_tv"] + 1.0 * out["L_conf"], rel=1e-14)
    custom = orc.train_losses(zd, zt, xs, s, gamma, a_ce=1.0, a_tv=0.0, a_conf=0.0)
    assert custom["L"] == pytest.approx(L_ce, rel=1e-13)


def test_gradients_match_finite_differences(orc):
    rng = np.random.default_rng(9)
    gamma, B, V = 3, 2, 11
    zd = rng.normal(0, 1.5, (B * gamma, V)).astype(np.float32)
    zt = rng.normal(0, 1.5, (B * gamma, V)).astype(np.float32)
    xs = rng.integers(0, V, B * gamma).astype(np.int32)
    s = rng.normal(0, 1, B * gamma).astype(np.float32)
    out = orc.train_losses(zd, zt, xs, s, gamma, want_grad=True)
    cstar = out["cstar"]

    def loss_at(zd2, s2):
        o = orc.train_losses(zd2, zt, xs, s2, gamma)
        # the confidence term with the label c* of the unperturbed logits
        w = np.exp(-(np.arange(B * gamma) % gamma) / gamma)
        sp = np.logaddexp(0.0, s2.astype(np.float64))
        conf = (w * (sp - cstar * s2.astype(np.float64))).sum() / B
        return 0.1 * o["L_ce"] + 0.9 * o["L_tv"] + conf

    h = 2.0 ** -9  # exact in fp32 next to these logits' magnitudes
    for (i, v) in [(0, 0), (1, 3), (4, int(xs[4])), (5, 10)]:
        zp, zm = zd.copy(), zd.copy()
        zp[i, v] += h
        zm[i, v] -= h
        fd = (loss_at(zp, s) - loss_at(zm, s)) / (float(zp[i, v]) - float(zm[i, v]))
        assert out["grad_z"][i, v] == pytest.approx(fd, rel=2e-4, abs=1e-7)
    for i in (0, 4):
        sp_, sm_ = s.copy(), s.copy()
        sp_[i] += h
        sm_[i] -= h
        fd = (loss_at(zd, sp_) - loss_at(zd, sm_)) / (float(sp_[i]) - float(sm_[i]))
        assert out["grad_s"][i] == pytest.approx(fd, rel=2e-4, abs=1e-9)
    # the cross-entropy gradient sums to zero over the vocabulary and so does the TV one
    assert np.allclose(out["grad_z"].sum(axis=1), 0.0, atol=1e-14)


def test_bf16_inputs_equal_their_widening(orc):
    rng = np.random.default_rng(4)
    z = rng.normal(0, 2, (4, 64)).astype(np.float32)
    bits_d = (z.view(np.uint32) >> 16).astype(np.uint16)
    bits_t = ((z + 0.5).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    wide_d = (bits_d.astype(np.uint32) << 16).view(np.float32)
    wide_t = (bits_t.astype(np.uint32) << 16).view(np.float32)
    xs, s = [1, 2, 3, 4], np.zeros(4, np.float32)
    a = orc.train_losses(bits_d, bits_t, xs, s, 2)
    b = orc.train_losses(wide_d, wide_t, xs, s, 2)
    for k in ("lse_d", "lse_t", "ce", "tv", "cstar", "bce"):
        assert np.array_equal(a[k], b[k]), k
    with pytest.raises(ValueError):
        orc.train_losses(wide_d, wide_t, [1, 2, 3, 64], s, 2)
