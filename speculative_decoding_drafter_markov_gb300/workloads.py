"""Seeded synthetic workloads for the DSpark per-cycle hot path.

This module only draws random inputs with the shapes and value distributions of
the five standard workloads; it holds none of the method's arithmetic (no bias
contraction, softmax, sampling, scheduling or acceptance test).  Both the CUDA
library's callers and the CPU checker take their inputs from here.

Workloads (shapes and distributions):
  tiny      R=4,   gamma=4,  V=1024,   r=32,  d=64,   fp32, planted +6 peak
  qwen4b    R=64,  gamma=8,  V=151936, r=256, d=2560, bf16, peak U(5,9) per position
  heavy     R=256, gamma=16, V=151936, r=256, d=2560, bf16, peak U(3,9) per request,
            smooth SPS(B) = 1000 / (20 + 0.01 B) on B = 256..4352, sync scheduler
  rnn       R=128, gamma=16, V=151936, r=256, d=4096, bf16, RNN head, as qwen4b
  prod      R=512, gamma=16, V=129280, r=256, d=4096, bf16, as heavy, sawtooth SPS on
            B = 512..8704 with a 5-15 % drop right after each multiple of 128,
            asynchronous scheduler, 32 cycles
Target logits for row (request, position j) are the base logits of position j+1
plus N(0, sigma^2) noise; row gamma (the bonus row) uses a fresh base-logit draw.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int
    gamma: int
    V: int
    r: int
    d: int
    dtype: str            # "f32" or "bf16"
    head: str = "markov"  # "markov" or "rnn"
    peak: str = "fixed"   # "fixed" (+6), "per_pos" (U(5,9)), "per_req" (U(3,9))
    sigma: float = 0.7    # target noise
    sps: str | None = None  # None, "linear", "smooth", "sawtooth"
    sched: str = "none"   # "none" (verify all), "sync", "async"
    cycles: int = 1

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def B_range(self):
        """(B_min, B_count) of the SPS table."""
        if self.sps is None:
            return None
        if self.sps == "linear":
            return 1, 20
        return self.R, self.R * self.gamma + 1


WORKLOADS = {
    "tiny": Workload("tiny", 4, 4, 1024, 32, 64, "f32", peak="fixed", sigma=0.5, sps="linear",
                     sched="sync"),
    "qwen4b": Workload("qwen4b", 64, 8, 151936, 256, 2560, "bf16", peak="per_pos"),
    "heavy": Workload("heavy", 256, 16, 151936, 256, 2560, "bf16", peak="per_req", sps="smooth",
                      sched="sync"),
    "rnn": Workload("rnn", 128, 16, 151936, 256, 4096, "bf16", head="rnn", peak="per_pos"),
    "prod": Workload("prod", 512, 16, 129280, 256, 4096, "bf16", peak="per_req", sps="sawtooth",
                     sched="async", cycles=32),
}


def small(name: str, **over) -> Workload:
    """A reduced-size copy of a standard workload (for CPU-checkable cases)."""
    return dataclasses.replace(WORKLOADS[name], name=f"{name}-small", **over)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _peaked_logits(wl: Workload, n_pos: int, g: torch.Generator, device) -> torch.Tensor:
    """[R, n_pos, V] fp32: N(0, 3^2) plus a planted peak on one token per position."""
    R, V = wl.R, wl.V
    base = torch.randn((R, n_pos, V), generator=g, device=device) * 3.0
    tok = torch.randint(0, V, (R, n_pos), generator=g, device=device)
    if wl.peak == "fixed":
        height = torch.full((R, n_pos), 6.0, device=device)
    elif wl.peak == "per_pos":
        height = 5.0 + 4.0 * torch.rand((R, n_pos), generator=g, device=device)
    elif wl.peak == "per_req":
        height = (3.0 + 6.0 * torch.rand((R, 1), generator=g, device=device)).expand(R, n_pos)
    else:
        raise ValueError(wl.peak)
    base.scatter_add_(2, tok.unsqueeze(-1), height.unsqueeze(-1).contiguous())
    return base


def draft_inputs(wl: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one draft call plus the extra base-logit row for the bonus
    target row.  Weights: W1, W2 ~ N(0, 1/r) (W2 stored transposed as [V, r]),
    h ~ N(0, 1), w ~ N(0, 1/(d + r)), RNN projection W [3r, 2r + d] ~ N(0, 1/(2r + d))."""
    g = _gen(seed, device)
    dt = wl.torch_dtype
    R, gm, V, r, d = wl.R, wl.gamma, wl.V, wl.r, wl.d
    U_all = _peaked_logits(wl, gm + 1, g, device)
    out = {
        "U": U_all[:, :gm].to(dt).contiguous(),
        "U_bonus": U_all[:, gm].to(dt).contiguous(),
    }
    del U_all
    out["W1"] = (torch.randn((V, r), generator=g, device=device) / math.sqrt(r)).to(dt)
    out["W2t"] = (torch.randn((V, r), generator=g, device=device) / math.sqrt(r)).to(dt)
    out["h"] = torch.randn((R, gm, d), generator=g, device=device).to(dt)
    out["w"] = torch.randn((d + r,), generator=g, device=device) / math.sqrt(d + r)
    out["anchor"] = torch.randint(0, V, (R,), generator=g, device=device, dtype=torch.int32)
    if wl.head == "rnn":
        out["W"] = (torch.randn((3 * r, 2 * r + d), generator=g, device=device)
                    / math.sqrt(2 * r + d)).to(dt)
    return out


def train_loss_inputs(B: int, gamma: int, V: int, dtype=torch.bfloat16, seed: int = 0, device="cpu",
                      sigma: float = 0.7) -> dict:
    """Inputs of the drafter's training losses for B blocks of gamma positions:
    draft logits zd = N(0, 3^2) plus a planted peak of U(5, 9) on one token per
    row (the draft workloads' base logits), target logits zt = zd + N(0, sigma^2),
    target tokens xs = the peak token in 80 % of the rows and a uniform token
    otherwise, confidence logits s ~ N(1, 1)."""
    g = _gen(seed, device)
    N = B * gamma
    zd = torch.randn((N, V), generator=g, device=device) * 3.0
    tok = torch.randint(0, V, (N,), generator=g, device=device)
    zd[torch.arange(N, device=device), tok] += 5.0 + 4.0 * torch.rand((N,), generator=g, device=device)
    zt = zd + torch.randn((N, V), generator=g, device=device) * sigma
    other = torch.randint(0, V, (N,), generator=g, device=device)
    keep = torch.rand((N,), generator=g, device=device) < 0.8
    xs = torch.where(keep, tok, other).to(torch.int32)
    s = torch.randn((N,), generator=g, device=device) + 1.0
    return {"zd": zd.to(dtype).contiguous(), "zt": zt.to(dtype).contiguous(), "xs": xs, "s": s}


def stand_in_target(d: int = 2560, layers: int = 2, max_B: int = 8704, device="cuda", seed: int = 0):
    """A stand-in for the target model's forward at verify batch B, whose timing
    gives a profiled SPS(B) table: per layer two bf16 GEMMs, [B, d] x [d, 3d] and
    [B, 3d] x [3d, d] (an MLP block); the values computed are not used."""
    g = _gen(seed, device)
    x = (torch.randn((max_B, d), generator=g, device=device) * 0.1).to(torch.bfloat16)
    ws = [((torch.randn((d, 3 * d), generator=g, device=device) * 0.02).to(torch.bfloat16),
           (torch.randn((3 * d, d), generator=g, device=device) * 0.02).to(torch.bfloat16)) for _ in range(layers)]

    def forward(B: int):
        y = x[:B]
        for w1, w2 in ws:
            y = torch.matmul(torch.matmul(y, w1), w2)
        return y
    return forward


def tags_from_ell(ell) -> np.ndarray:
    """Flattened batch layout: rows grouped by request, positions 0..ell_r."""
    ell = np.asarray(ell, dtype=np.int64)
    rows = [(rq, j) for rq in range(len(ell)) for j in range(int(ell[rq]) + 1)]
    return np.asarray(rows, dtype=np.int32).reshape(-1, 2)


def target_logits(wl: Workload, U: torch.Tensor, U_bonus: torch.Tensor, tags, seed: int = 0,
                  device=None) -> torch.Tensor:
    """[N, V] target logits for the flattened rows `tags` (N x 2 of request,
    position): row (r, j) = base logits of position j+1 of request r plus
    N(0, sigma^2) noise (position gamma takes the bonus base row)."""
    device = device or U.device
    tags_t = torch.as_tensor(np.asarray(tags), device=device, dtype=torch.long).reshape(-1, 2)
    g = _gen(seed + 7919, device)
    req, pos = tags_t[:, 0], tags_t[:, 1]
    gm = wl.gamma
    base = torch.empty((tags_t.shape[0], wl.V), device=device, dtype=torch.float32)
    inner = pos < gm
    if bool(inner.any()):
        base[inner] = U[req[inner], pos[inner]].float()
    if bool((~inner).any()):
        base[~inner] = U_bonus[req[~inner]].float()
    noise = torch.randn(base.shape, generator=g, device=device) * wl.sigma
    return (base + noise).to(wl.torch_dtype)


def sps_table(wl: Workload, seed: int = 0) -> np.ndarray:
    """Synthetic profiled cost table SPS(B) (steps per second) for B in
    [B_min, B_min + B_count)."""
    B_min, B_count = wl.B_range
    B = np.arange(B_min, B_min + B_count, dtype=np.float64)
    if wl.sps == "linear":
        return 1.0 - 0.7 * (B - 1.0) / 19.0
    smooth = 1000.0 / (20.0 + 0.01 * B)
    if wl.sps == "smooth":
        return smooth
    if wl.sps == "sawtooth":
        rng = np.random.default_rng(seed + 104729)
        blocks = int(math.ceil((B_min + B_count) / 128.0)) + 1
        delta = rng.uniform(0.05, 0.15, size=blocks)
        m = np.ceil(B / 128.0).astype(np.int64)
        rho = np.mod(B - 1.0, 128.0) / 128.0
        return smooth * (1.0 - delta[m] * (1.0 - rho))
    raise ValueError(wl.sps)


def confidences(R: int, gamma: int, seed: int = 0, low: float = 0.05, high: float = 0.999):
    """Random per-position confidences c [R, gamma] fp32 for scheduler cases."""
    rng = np.random.default_rng(seed)
    return rng.uniform(low, high, size=(R, gamma)).astype(np.float32)


def calibration_set(M: int, gamma: int, seed: int = 0, T_true=None, mean: float = 2.0,
                    spread: float = 1.5):
    """Held-out draft blocks for the sequential temperature-scaling fit: confidence
    logits s [M, gamma] fp32 ~ N(mean, spread^2) and accepted prefix lengths
    n [M] int32.  Acceptance model of the synthetic blocks: given that positions
    1..k-1 were accepted, position k is accepted with probability
    1 / (1 + exp(-s_k / T_true[k])) (T_true defaults to 1.5 everywhere, so a head
    reporting sigma(s_k) is over-confident, as the pages find raw confidences)."""
    rng = np.random.default_rng(seed + 7919)
    s = rng.normal(mean, spread, size=(M, gamma)).astype(np.float32)
    T = np.full(gamma, 1.5) if T_true is None else np.asarray(T_true, np.float64)
    pass_prob = 1.0 / (1.0 + np.exp(-s.astype(np.float64) / T[None, :]))
    u = rng.uniform(0.0, 1.0, size=(M, gamma))
    passed = u < pass_prob
    # accepted prefix length: index of the first rejection, gamma if none
    first_fail = np.where(~passed, np.arange(gamma)[None, :], gamma).min(axis=1)
    return s, first_fail.astype(np.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as uint16 bit patterns (fp32 stays fp32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
