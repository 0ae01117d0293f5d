"""CPU oracle for the DSpark per-cycle hot path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its Python
binding) never does and shares no code with it.

The arithmetic lives in ``dspark_oracle.c`` (plain single-threaded C, fp64); this
module only compiles it with gcc and marshals numpy arrays through ctypes.  Each
wrapper names the passage of the pages it follows:
  [D] "DSpark: confidence-scheduled speculative decoding" (ai-papers-daily digest)
  [E] "DSpark explained" (interactive explainer)

Every function here is pinned by tests/test_oracle_*.py; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

F32, BF16 = 0, 1
SCHED_SYNC, SCHED_ASYNC, SCHED_NOBREAK = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (no FMA contraction,
    so both the x86-64 and the aarch64 build round identically)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "dspark_oracle.h")))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def bind(L):
    """Declare the argument types of the oracle's C functions on a loaded library."""
    P = ctypes.c_void_p
    i32, u64, u32 = ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32
    L.oracle_philox4x32_10.argtypes = [P, P, P]
    L.oracle_philox4x32_10.restype = None
    L.oracle_uniform.argtypes = [u32]
    L.oracle_uniform.restype = ctypes.c_double
    L.oracle_philox_word.argtypes = [u64, u32, u32, u32, u64, u32, u32]
    L.oracle_philox_word.restype = u32
    L.oracle_draft_markov.argtypes = [i32] * 6 + [P] * 7 + [u64, u64, P, i32] + [P] * 10
    L.oracle_draft_markov.restype = i32
    L.oracle_draft_rnn.argtypes = [i32] * 6 + [P] * 9 + [u64, u64, P, i32] + [P] * 11
    L.oracle_draft_rnn.restype = i32
    L.oracle_schedule.argtypes = [i32, i32, P, P, i32, i32, i32, i32, P, P, P, P]
    L.oracle_schedule.restype = i32
    L.oracle_verify.argtypes = [i32] * 6 + [P] * 10 + [u64, u64, P, i32] + [P] * 8
    L.oracle_verify.restype = i32
    L.oracle_sts_fit.argtypes = [i32, i32, P, P, i32, P, i32, P, P, P, P, ctypes.c_double, P]
    L.oracle_sts_fit.restype = i32
    L.oracle_accept_stats.argtypes = [i32, i32, P, P, P, P, P, P]
    L.oracle_accept_stats.restype = i32
    d = ctypes.c_double
    L.oracle_train_losses.argtypes = [i32, i32, i32, i32, P, P, P, P, d, d, d, P, P, P, P]
    L.oracle_train_losses.restype = i32
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = bind(ctypes.CDLL(_LIB))
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _elem(a):
    """numpy array of float32 (F32) or uint16 bf16 bit patterns (BF16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"oracle tensors are float32 or uint16 (bf16 bits), got {a.dtype}")


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform(word: int) -> float:
    return lib().oracle_uniform(int(word) & 0xFFFFFFFF)


def philox_word(seed, w0, w1, req, cycle, stream, lane) -> int:
    return lib().oracle_philox_word(seed, w0, w1, req, cycle, stream, lane)


def draft_markov(U, h, W1, W2t, w, anchor, *, seed=0, cycle=0, sts_T=None, reqs=None,
                 want_z=False):
    """[D] eqs. (4), (5), (7).  U [R, gamma, V], h [R, gamma, d], W1 / W2t [V, r]."""
    U, dt = _elem(U)
    h, dt_h = _elem(h)
    W1, dt1 = _elem(W1)
    W2t, dt2 = _elem(W2t)
    assert dt == dt_h == dt1 == dt2
    R, gamma, V = U.shape
    r = W1.shape[1]
    d = h.shape[2]
    w = np.ascontiguousarray(w, dtype=np.float32)
    anchor = np.ascontiguousarray(anchor, dtype=np.int32)
    sts = None if sts_T is None else np.ascontiguousarray(sts_T, dtype=np.float32)
    rl = None if reqs is None else np.ascontiguousarray(reqs, dtype=np.int32)
    n = R if rl is None else len(rl)
    x = np.zeros((n, gamma), np.int32)
    logq = np.zeros((n, gamma)); lse = np.zeros((n, gamma)); c = np.zeros((n, gamma))
    gap = np.zeros((n, gamma)); logit = np.zeros((n, gamma)); cdf_gap = np.zeros((n, gamma, 2))
    runner = np.full((n, gamma), -1, np.int32); cdf_runner = np.full((n, gamma, 2), -1, np.int32)
    z = np.zeros((n, gamma, V)) if want_z else None
    rc = lib().oracle_draft_markov(R, gamma, V, r, d, dt, _p(U), _p(h), _p(W1), _p(W2t), _p(w),
                                   _p(sts), _p(anchor), seed, cycle, _p(rl), n, _p(x), _p(logq),
                                   _p(lse), _p(c), _p(gap), _p(runner), _p(cdf_gap),
                                   _p(cdf_runner), _p(z), _p(logit))
    if rc != 0:
        raise ValueError(f"oracle_draft_markov failed ({rc})")
    out = dict(x=x, logq=logq, lse=lse, c=c, gap=gap, runner=runner, cdf_gap=cdf_gap,
               cdf_runner=cdf_runner, conf_logit=logit)
    if want_z:
        out["z"] = z
    return out


def draft_rnn(U, h, W1, W2t, W, w, anchor, *, s0=None, seed=0, cycle=0, sts_T=None, reqs=None,
              want_z=False):
    """[D] eq. (6) with eqs. (4), (7).  W [3r, 2r + d] (gate, candidate, output rows)."""
    U, dt = _elem(U)
    h, _ = _elem(h)
    W1, _ = _elem(W1)
    W2t, _ = _elem(W2t)
    W, _ = _elem(W)
    R, gamma, V = U.shape
    r = W1.shape[1]
    d = h.shape[2]
    w = np.ascontiguousarray(w, dtype=np.float32)
    anchor = np.ascontiguousarray(anchor, dtype=np.int32)
    s0a = None if s0 is None else np.ascontiguousarray(s0, dtype=np.float32)
    sts = None if sts_T is None else np.ascontiguousarray(sts_T, dtype=np.float32)
    rl = None if reqs is None else np.ascontiguousarray(reqs, dtype=np.int32)
    n = R if rl is None else len(rl)
    x = np.zeros((n, gamma), np.int32)
    logq = np.zeros((n, gamma)); lse = np.zeros((n, gamma)); c = np.zeros((n, gamma))
    gap = np.zeros((n, gamma)); A = np.zeros((n, gamma, r)); logit = np.zeros((n, gamma))
    cdf_gap = np.zeros((n, gamma, 2))
    runner = np.full((n, gamma), -1, np.int32); cdf_runner = np.full((n, gamma, 2), -1, np.int32)
    z = np.zeros((n, gamma, V)) if want_z else None
    rc = lib().oracle_draft_rnn(R, gamma, V, r, d, dt, _p(U), _p(h), _p(W1), _p(W2t), _p(W),
                                _p(s0a), _p(w), _p(sts), _p(anchor), seed, cycle, _p(rl), n,
                                _p(x), _p(logq), _p(lse), _p(c), _p(gap), _p(runner),
                                _p(cdf_gap), _p(cdf_runner), _p(z), _p(A), _p(logit))
    if rc != 0:
        raise ValueError(f"oracle_draft_rnn failed ({rc})")
    out = dict(x=x, logq=logq, lse=lse, c=c, gap=gap, runner=runner, cdf_gap=cdf_gap,
               cdf_runner=cdf_runner, A=A, conf_logit=logit)
    if want_z:
        out["z"] = z
    return out


def schedule(c, sps, B_min, *, mode=SCHED_SYNC, K_in=-1):
    """[D] Module E, Algorithm 1 (mode SYNC) and the production asynchronous
    top-K variant (mode ASYNC); NOBREAK is the lossy backtracking search of
    Appendix A, kept for tests only."""
    c = np.ascontiguousarray(c, dtype=np.float32)
    R, gamma = c.shape
    sps = np.ascontiguousarray(sps, dtype=np.float64)
    ell = np.zeros(R, np.int32)
    K = np.zeros(1, np.int32)
    th = np.zeros(1, np.float64)
    a = np.zeros((R, gamma), np.float32)
    rc = lib().oracle_schedule(R, gamma, _p(c), _p(sps), int(B_min), len(sps), int(mode),
                               int(K_in), _p(ell), _p(K), _p(th), _p(a))
    if rc != 0:
        raise ValueError(f"oracle_schedule failed ({rc})")
    return dict(ell=ell, K_out=int(K[0]), theta_best=float(th[0]), a=a)


def verify(T, tags, anchor, x, logq, lse, U, W1, W2t, *, A=None, seed=0, cycle=0, reqs=None):
    """[E] section 06 rule along the scheduled prefix ([D] overview step 3)."""
    T, dt = _elem(T)
    U, _ = _elem(U)
    W1, _ = _elem(W1)
    W2t, _ = _elem(W2t)
    N, V = T.shape
    R, gamma = np.asarray(x).shape
    r = W1.shape[1]
    tags = np.ascontiguousarray(tags, dtype=np.int32).reshape(N, 2)
    anchor = np.ascontiguousarray(anchor, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.int32)
    logq = np.ascontiguousarray(logq, dtype=np.float32)
    lse = np.ascontiguousarray(lse, dtype=np.float32)
    Aa = None if A is None else np.ascontiguousarray(A, dtype=np.float32)
    rl = None if reqs is None else np.ascontiguousarray(reqs, dtype=np.int32)
    n = R if rl is None else len(rl)
    n_acc = np.full(R, -1, np.int32)
    out = np.full((R, gamma + 1), -1, np.int32)
    nxt = np.full(R, -1, np.int32)
    lse_p = np.full(N, np.nan); logp = np.full(N, np.nan); margin = np.full(N, np.nan)
    gap = np.full((R, 2), np.nan)
    runner = np.full((R, 2), -1, np.int32)
    rc = lib().oracle_verify(R, gamma, V, r, dt, N, _p(T), _p(tags), _p(anchor), _p(x), _p(logq),
                             _p(lse), _p(U), _p(W1), _p(W2t), _p(Aa), seed, cycle, _p(rl), n,
                             _p(n_acc), _p(out), _p(nxt), _p(lse_p), _p(logp), _p(margin), _p(gap),
                             _p(runner))
    if rc != 0:
        raise ValueError(f"oracle_verify failed ({rc})")
    return dict(n_accept=n_acc, out_tokens=out, next_anchor=nxt, lse_p=lse_p, logp=logp,
                margin=margin, gap=gap, runner=runner)


def sts_fit(logit, n_accept, grid, *, n_bins=15, T_prefix=None, edge_eps=0.0):
    """[D] Module D: sequential temperature scaling, one grid search per position,
    left to right, minimising the ECE of the cumulative products prod_{i<=k} c_i
    against the held-out outcome 1[n_accept >= k].  ``near_edge`` counts, per
    position and grid point, the samples within ``edge_eps`` of a bin edge."""
    logit = np.ascontiguousarray(logit, dtype=np.float32)
    M, gamma = logit.shape
    n_accept = np.ascontiguousarray(n_accept, dtype=np.int32)
    grid = np.ascontiguousarray(grid, dtype=np.float32)
    G = len(grid)
    Tp = None if T_prefix is None else np.ascontiguousarray(T_prefix, dtype=np.float32)
    T = np.zeros(gamma, np.float32)
    ece = np.zeros(gamma)
    curve = np.zeros((gamma, G))
    near = np.zeros((gamma, G), np.int32)
    rc = lib().oracle_sts_fit(M, gamma, _p(logit), _p(n_accept), G, _p(grid), int(n_bins), _p(Tp),
                              _p(T), _p(ece), _p(curve), float(edge_eps), _p(near))
    if rc != 0:
        raise ValueError(f"oracle_sts_fit failed ({rc})")
    return dict(T=T, ece=ece, curve=curve, index=np.argmin(curve, axis=1).astype(np.int32),
                near_edge=near)


def accept_stats(n_accept, ell=None, gamma=None, *, into=None):
    """[D] analysis 1: per-position conditional acceptance counts and the
    acceptance-length histogram of one cycle's verification outcomes, added to
    ``into`` (a dict from a previous call) or to fresh zero counters."""
    n_accept = np.ascontiguousarray(n_accept, dtype=np.int32)
    R = len(n_accept)
    ell_a = None if ell is None else np.ascontiguousarray(ell, dtype=np.int32)
    if gamma is None:
        raise ValueError("gamma is required")
    out = into if into is not None else dict(
        reached=np.zeros(gamma, np.uint64), accepted=np.zeros(gamma, np.uint64),
        tau_hist=np.zeros(gamma + 1, np.uint64), ell_hist=np.zeros(gamma + 1, np.uint64))
    rc = lib().oracle_accept_stats(R, gamma, _p(n_accept), _p(ell_a), _p(out["reached"]), _p(out["accepted"]),
                                   _p(out["tau_hist"]), _p(out["ell_hist"]))
    if rc != 0:
        raise ValueError("oracle_accept_stats: n_accept outside 0..min(ell, gamma)")
    return out


def train_losses(zd, zt, xs, s, gamma, *, a_ce=0.1, a_tv=0.9, a_conf=1.0, want_grad=False):
    """[D] Module F, eqs. (8)-(12): per-row (lse_d, lse_t, ce, tv, c*, bce), the
    losses (L_ce, L_tv, L_conf, L) averaged over the blocks, and optionally the
    gradients with respect to the draft logits and the confidence logits."""
    zd, dt = _elem(zd)
    zt, dt2 = _elem(zt)
    if dt != dt2:
        raise TypeError("draft and target logits must share a dtype")
    N, V = zd.shape
    if N % gamma:
        raise ValueError("rows must be blocks x gamma")
    xs = np.ascontiguousarray(xs, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    row = np.zeros((N, 6))
    loss = np.zeros(4)
    gz = np.zeros((N, V)) if want_grad else None
    gs = np.zeros(N) if want_grad else None
    rc = lib().oracle_train_losses(N // gamma, gamma, V, dt, _p(zd), _p(zt), _p(xs), _p(s), float(a_ce),
                                   float(a_tv), float(a_conf), _p(row), _p(loss), _p(gz), _p(gs))
    if rc != 0:
        raise ValueError("oracle_train_losses: token outside 0..V-1")
    out = dict(lse_d=row[:, 0], lse_t=row[:, 1], ce=row[:, 2], tv=row[:, 3], cstar=row[:, 4], bce=row[:, 5],
               L_ce=loss[0], L_tv=loss[1], L_conf=loss[2], L=loss[3])
    if want_grad:
        out.update(grad_z=gz, grad_s=gs)
    return out
