"""ctypes binding of libdspark.so (include/dspark.h).

Argument marshalling only: every step of the hot path runs in the library's CUDA
kernels.  PyTorch provides device memory (outputs and the scratch workspace are
torch tensors) and the current CUDA stream.  There is no fallback: if the
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

P = ctypes.c_void_p
i32 = ctypes.c_int32
u64 = ctypes.c_uint64

OK, ERR_INVAL, ERR_RANGE, ERR_NONFINITE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(7)
ERROR_NAMES = {0: "OK", 1: "INVAL", 2: "RANGE", 3: "NONFINITE", 4: "CUDA", 5: "TIMEOUT",
               6: "UNSUPPORTED"}
F32, BF16 = 0, 1
SCHED_SYNC, SCHED_ASYNC = 0, 1


class DraftArgs(ctypes.Structure):
    _fields_ = [("R", i32), ("gamma", i32), ("V", i32), ("r", i32), ("d", i32), ("dtype", i32),
                ("U", P), ("h", P), ("W1", P), ("W2t", P), ("w", P), ("sts_T", P), ("anchor", P),
                ("seed", u64), ("cycle", u64),
                ("x", P), ("logq", P), ("lse", P), ("c", P), ("err", P), ("conf_logit", P)]


class RnnArgs(ctypes.Structure):
    _fields_ = [("base", DraftArgs), ("W", P), ("s0", P), ("A", P), ("s_out", P)]


class SchedArgs(ctypes.Structure):
    _fields_ = [("R", i32), ("gamma", i32), ("c", P), ("sps", P), ("B_min", i32), ("B_count", i32),
                ("mode", i32), ("K_in", P), ("ell", P), ("K_out", P), ("theta_best", P), ("a", P),
                ("err", P)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("R", i32), ("gamma", i32), ("V", i32), ("r", i32), ("dtype", i32), ("N", i32),
                ("N_dev", P), ("T", P), ("tags", P), ("anchor", P), ("x", P), ("logq", P),
                ("lse", P), ("U", P), ("W1", P), ("W2t", P), ("A", P), ("seed", u64), ("cycle", u64),
                ("n_accept", P), ("out_tokens", P), ("next_anchor", P), ("lse_p", P), ("logp", P),
                ("err", P)]


class StsArgs(ctypes.Structure):
    _fields_ = [("M", i32), ("gamma", i32), ("G", i32), ("n_bins", i32), ("logit", P),
                ("n_accept", P), ("grid", P), ("T", P), ("ece", P), ("curve", P), ("err", P)]


class AcceptStatsArgs(ctypes.Structure):
    _fields_ = [("R", i32), ("gamma", i32), ("n_accept", P), ("ell", P), ("reached", P), ("accepted", P),
                ("tau_hist", P), ("ell_hist", P), ("err", P)]


class TrainLossArgs(ctypes.Structure):
    _fields_ = [("B", i32), ("gamma", i32), ("V", i32), ("dtype", i32), ("zd", P), ("zt", P), ("xs", P),
                ("s", P), ("a_ce", ctypes.c_float), ("a_tv", ctypes.c_float), ("a_conf", ctypes.c_float),
                ("row", P), ("loss", P), ("grad_z", P), ("grad_s", P), ("err", P)]


class DSparkError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"dspark error {ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None
_lock = threading.Lock()

SYMBOLS = {
    "dspark_draft_markov_workspace_size": ([ctypes.POINTER(DraftArgs)], ctypes.c_size_t),
    "dspark_draft_markov": ([ctypes.POINTER(DraftArgs), P, P], ctypes.c_int),
    "dspark_draft_markov_step": ([ctypes.POINTER(DraftArgs), i32, P, P], ctypes.c_int),
    "dspark_draft_markov_noalloc": ([ctypes.POINTER(DraftArgs), P], ctypes.c_int),
    "dspark_draft_rnn_workspace_size": ([ctypes.POINTER(RnnArgs)], ctypes.c_size_t),
    "dspark_draft_rnn": ([ctypes.POINTER(RnnArgs), P, P], ctypes.c_int),
    "dspark_schedule_workspace_size": ([ctypes.POINTER(SchedArgs)], ctypes.c_size_t),
    "dspark_schedule": ([ctypes.POINTER(SchedArgs), P, P], ctypes.c_int),
    "dspark_build_tags": ([i32, i32, P, P, P, P, P], ctypes.c_int),
    "dspark_verify_workspace_size": ([ctypes.POINTER(VerifyArgs)], ctypes.c_size_t),
    "dspark_verify": ([ctypes.POINTER(VerifyArgs), P, P], ctypes.c_int),
    "dspark_last_error": ([], ctypes.c_char_p),
    "dspark_version": ([], ctypes.c_int),
    "dspark_philox": ([P, u64, i32, P, P], ctypes.c_int),
    "dspark_wait_selfcheck": ([P, i32, i32, u64, P, P], ctypes.c_int),
    "dspark_sts_fit_workspace_size": ([ctypes.POINTER(StsArgs)], ctypes.c_size_t),
    "dspark_sts_fit": ([ctypes.POINTER(StsArgs), P, P], ctypes.c_int),
    "dspark_accept_stats": ([ctypes.POINTER(AcceptStatsArgs), P], ctypes.c_int),
    "dspark_train_losses": ([ctypes.POINTER(TrainLossArgs), P], ctypes.c_int),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libdspark.so (building it with nvcc first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libdspark.so not found at {path}")
            L = ctypes.CDLL(path)
            for name, (argt, rest) in SYMBOLS.items():
                fn = getattr(L, name)
                fn.argtypes = argt
                fn.restype = rest
            _lib = L
    return _lib


def _check(rc):
    if rc != OK:
        raise DSparkError(rc, load().dspark_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("dspark tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("dspark tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported element type {t.dtype}")


def _workspace(nbytes, device, ws):
    if nbytes == 0:
        nbytes = 256
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError(f"workspace of {ws.numel()} bytes, need {nbytes}")
        return ws
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# --------------------------------------------------------------------- draft
def _draft_struct(U, h, W1, W2t, w, anchor, seed, cycle, sts_T, out, err):
    R, gamma, V = U.shape
    a = DraftArgs()
    a.R, a.gamma, a.V, a.r, a.d = R, gamma, V, W1.shape[1], h.shape[2]
    a.dtype = _dtype_code(U)
    for t in (h, W1, W2t):
        if t.dtype != U.dtype:
            raise TypeError("U, h, W1 and W2t must share one element type")
    a.U, a.h, a.W1, a.W2t = _ptr(U), _ptr(h), _ptr(W1), _ptr(W2t)
    a.w, a.sts_T, a.anchor = _ptr(w), _ptr(sts_T), _ptr(anchor)
    a.seed, a.cycle = int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1)
    a.x, a.logq, a.lse, a.c = _ptr(out["x"]), _ptr(out["logq"]), _ptr(out["lse"]), _ptr(out["c"])
    a.conf_logit = _ptr(out.get("conf_logit"))
    a.err = _ptr(err)
    return a


def _draft_outputs(R, gamma, device, out):
    if out is not None:
        return out
    return {"x": torch.empty((R, gamma), dtype=torch.int32, device=device),
            "logq": torch.empty((R, gamma), dtype=torch.float32, device=device),
            "lse": torch.empty((R, gamma), dtype=torch.float32, device=device),
            "c": torch.empty((R, gamma), dtype=torch.float32, device=device)}


def draft_markov(U, h, W1, W2t, w, anchor, *, seed=0, cycle=0, sts_T=None, out=None, ws=None,
                 err=None, stream=None):
    """Markov-head draft of gamma tokens per request (see include/dspark.h)."""
    L = load()
    R, gamma, _ = U.shape
    out = _draft_outputs(R, gamma, U.device, out)
    a = _draft_struct(U, h, W1, W2t, w, anchor, seed, cycle, sts_T, out, err)
    ws = _workspace(L.dspark_draft_markov_workspace_size(ctypes.byref(a)), U.device, ws)
    _check(L.dspark_draft_markov(ctypes.byref(a), _ptr(ws), _stream(stream)))
    return out


def draft_markov_step(k, U, h, W1, W2t, w, anchor, *, out, ws, seed=0, cycle=0, sts_T=None,
                      err=None, stream=None):
    """Step k (1..gamma) of the Markov draft into preallocated `out` / `ws`."""
    L = load()
    a = _draft_struct(U, h, W1, W2t, w, anchor, seed, cycle, sts_T, out, err)
    _check(L.dspark_draft_markov_step(ctypes.byref(a), int(k), _ptr(ws), _stream(stream)))
    return out


def draft_markov_noalloc(U, h, W1, W2t, w, anchor, *, seed=0, cycle=0, sts_T=None, out=None,
                         err=None, stream=None):
    """Markov draft through the entry point that allocates nothing: its scratch
    is a fixed array inside the library (the draft workspace size -- 32 bytes per
    (request, vocabulary range) plus 256 -- must be <= 16 MiB)."""
    L = load()
    R, gamma, _ = U.shape
    out = _draft_outputs(R, gamma, U.device, out)
    a = _draft_struct(U, h, W1, W2t, w, anchor, seed, cycle, sts_T, out, err)
    _check(L.dspark_draft_markov_noalloc(ctypes.byref(a), _stream(stream)))
    return out


def draft_markov_workspace_size(U, h, W1, W2t, w, anchor):
    L = load()
    R, gamma, _ = U.shape
    out = _draft_outputs(R, gamma, U.device, None)
    a = _draft_struct(U, h, W1, W2t, w, anchor, 0, 0, None, out, None)
    return L.dspark_draft_markov_workspace_size(ctypes.byref(a))


def draft_rnn(U, h, W1, W2t, W, w, anchor, *, s0=None, seed=0, cycle=0, sts_T=None, out=None,
              ws=None, err=None, stream=None):
    """RNN-head draft (eq. 6); also returns A [R, gamma, r] and the final state."""
    L = load()
    R, gamma, _ = U.shape
    r = W1.shape[1]
    out = _draft_outputs(R, gamma, U.device, out)
    out.setdefault("A", torch.empty((R, gamma, r), dtype=torch.float32, device=U.device))
    out.setdefault("s_out", torch.empty((R, r), dtype=torch.float32, device=U.device))
    a = RnnArgs()
    a.base = _draft_struct(U, h, W1, W2t, w, anchor, seed, cycle, sts_T, out, err)
    if W.dtype != U.dtype:
        raise TypeError("W must share the element type of U")
    a.W, a.s0, a.A, a.s_out = _ptr(W), _ptr(s0), _ptr(out["A"]), _ptr(out["s_out"])
    ws = _workspace(L.dspark_draft_rnn_workspace_size(ctypes.byref(a)), U.device, ws)
    _check(L.dspark_draft_rnn(ctypes.byref(a), _ptr(ws), _stream(stream)))
    return out


def draft_rnn_workspace_size(U, h, W1, W2t, W, w, anchor):
    """Scratch bytes dspark_draft_rnn needs for this shape."""
    L = load()
    R, gamma, _ = U.shape
    r = W1.shape[1]
    out = _draft_outputs(R, gamma, U.device, None)
    a = RnnArgs()
    a.base = _draft_struct(U, h, W1, W2t, w, anchor, 0, 0, None, out, None)
    a.W, a.s0 = _ptr(W), None
    a.A = a.s_out = None
    return L.dspark_draft_rnn_workspace_size(ctypes.byref(a))


# --------------------------------------------------------------------- schedule
def schedule(c, sps, B_min, *, mode=SCHED_SYNC, K_in=None, out=None, err=None, want_a=True,
             stream=None):
    """Prefix scheduler (Algorithm 1 / async top-K).  c [R, gamma] f32, sps f64 (device)."""
    L = load()
    R, gamma = c.shape
    dev = c.device
    if out is None:
        out = {"ell": torch.empty(R, dtype=torch.int32, device=dev),
               "K_out": torch.empty(1, dtype=torch.int32, device=dev),
               "theta_best": torch.empty(1, dtype=torch.float64, device=dev)}
        if want_a:
            out["a"] = torch.empty((R, gamma), dtype=torch.float32, device=dev)
    a = SchedArgs()
    a.R, a.gamma = R, gamma
    a.c, a.sps = _ptr(c), _ptr(sps)
    a.B_min, a.B_count, a.mode = int(B_min), int(sps.numel()), int(mode)
    a.K_in = _ptr(K_in)
    a.ell, a.K_out, a.theta_best = _ptr(out["ell"]), _ptr(out["K_out"]), _ptr(out["theta_best"])
    a.a = _ptr(out.get("a"))
    a.err = _ptr(err)
    _check(L.dspark_schedule(ctypes.byref(a), None, _stream(stream)))
    return out


def build_tags(ell, gamma, *, tags=None, N_out=None, err=None, stream=None):
    """Flattened (request, position) rows from verify lengths ell (device)."""
    L = load()
    R = ell.numel()
    if tags is None:
        tags = torch.empty((R * (gamma + 1), 2), dtype=torch.int32, device=ell.device)
    if N_out is None:
        N_out = torch.empty(1, dtype=torch.int32, device=ell.device)
    _check(L.dspark_build_tags(R, gamma, _ptr(ell), _ptr(tags), _ptr(N_out), _ptr(err),
                               _stream(stream)))
    return tags, N_out


# --------------------------------------------------------------------- verify
def _verify_struct(T, tags, anchor, x, logq, lse, U, W1, W2t, A, N_dev, seed, cycle, out, err):
    R, gamma = x.shape
    a = VerifyArgs()
    a.R, a.gamma, a.V, a.r = R, gamma, T.shape[1], W1.shape[1]
    a.dtype = _dtype_code(T)
    a.N = T.shape[0]
    a.N_dev = _ptr(N_dev)
    a.T, a.tags, a.anchor, a.x = _ptr(T), _ptr(tags), _ptr(anchor), _ptr(x)
    a.logq, a.lse, a.U, a.W1, a.W2t, a.A = _ptr(logq), _ptr(lse), _ptr(U), _ptr(W1), _ptr(W2t), _ptr(A)
    a.seed, a.cycle = int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1)
    a.n_accept, a.out_tokens, a.next_anchor = (_ptr(out["n_accept"]), _ptr(out["out_tokens"]),
                                               _ptr(out["next_anchor"]))
    a.lse_p, a.logp = _ptr(out.get("lse_p")), _ptr(out.get("logp"))
    a.err = _ptr(err)
    return a


def verify(T, tags, anchor, x, logq, lse, U, W1, W2t, *, A=None, N_dev=None, seed=0, cycle=0,
           out=None, ws=None, err=None, want_rows=True, stream=None):
    """Lossless verification of the flattened batch (see include/dspark.h)."""
    L = load()
    R, gamma = x.shape
    N = T.shape[0]
    dev = T.device
    if out is None:
        out = {"n_accept": torch.empty(R, dtype=torch.int32, device=dev),
               "out_tokens": torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
               "next_anchor": torch.empty(R, dtype=torch.int32, device=dev)}
        if want_rows:
            out["lse_p"] = torch.empty(N, dtype=torch.float32, device=dev)
            out["logp"] = torch.empty(N, dtype=torch.float32, device=dev)
    a = _verify_struct(T, tags, anchor, x, logq, lse, U, W1, W2t, A, N_dev, seed, cycle, out, err)
    ws = _workspace(L.dspark_verify_workspace_size(ctypes.byref(a)), dev, ws)
    _check(L.dspark_verify(ctypes.byref(a), _ptr(ws), _stream(stream)))
    return out


def verify_workspace_size(T, tags, anchor, x, logq, lse, U, W1, W2t, *, A=None):
    """Scratch bytes dspark_verify needs for this batch shape."""
    L = load()
    R, gamma = x.shape
    dev = T.device
    dummy = {"n_accept": x, "out_tokens": x, "next_anchor": x}
    a = _verify_struct(T, tags, anchor, x, logq, lse, U, W1, W2t, A, None, 0, 0, dummy, None)
    return L.dspark_verify_workspace_size(ctypes.byref(a))


def philox(ctr, seed, stream=None):
    """Device Philox-4x32-10 of counters ctr [n, 4] (uint32 stored as int32)."""
    L = load()
    n = ctr.shape[0]
    out = torch.empty((n, 4), dtype=torch.int32, device=ctr.device)
    _check(L.dspark_philox(_ptr(ctr), int(seed), n, _ptr(out), _stream(stream)))
    return out


def wait_selfcheck(flag, target, mode, limit_ns, err, stream=None):
    """Run the kernels' bounded wait on `flag` (see include/dspark.h)."""
    L = load()
    _check(L.dspark_wait_selfcheck(_ptr(flag), int(target), int(mode), int(limit_ns), _ptr(err),
                                   _stream(stream)))


# --------------------------------------------------------------------- calibration
def sts_fit(logit, n_accept, grid, *, n_bins=15, want_curve=True, ws=None, err=None, stream=None):
    """Sequential temperature scaling of the confidences (include/dspark.h):
    logit [M, gamma] fp32 confidence logits of held-out draft blocks (the draft's
    ``conf_logit`` output), n_accept [M] int32 accepted prefix lengths, grid [G]
    fp32 candidate temperatures.  Returns {"T": [gamma] fp32 (the draft's sts_T),
    "ece": [gamma] fp64, "curve": [gamma, G] fp64 or None}."""
    L = load()
    M, gamma = logit.shape
    dev = logit.device
    if logit.dtype != torch.float32 or n_accept.dtype != torch.int32 or grid.dtype != torch.float32:
        raise TypeError("logit and grid are float32, n_accept int32")
    a = StsArgs()
    a.M, a.gamma, a.G, a.n_bins = M, gamma, grid.numel(), int(n_bins)
    out = {"T": torch.empty(gamma, dtype=torch.float32, device=dev),
           "ece": torch.empty(gamma, dtype=torch.float64, device=dev),
           "curve": torch.empty((gamma, grid.numel()), dtype=torch.float64, device=dev)
           if want_curve else None}
    a.logit, a.n_accept, a.grid = _ptr(logit), _ptr(n_accept), _ptr(grid)
    a.T, a.ece, a.curve, a.err = _ptr(out["T"]), _ptr(out["ece"]), _ptr(out["curve"]), _ptr(err)
    ws = _workspace(L.dspark_sts_fit_workspace_size(ctypes.byref(a)), dev, ws)
    _check(L.dspark_sts_fit(ctypes.byref(a), _ptr(ws), _stream(stream)))
    return out


# --------------------------------------------------------------------- diagnostics
def accept_stats_counters(gamma, device):
    """Zeroed device counters for accept_stats (uint64 stored as int64)."""
    z = lambda n: torch.zeros(n, dtype=torch.int64, device=device)
    return {"reached": z(gamma), "accepted": z(gamma), "tau_hist": z(gamma + 1), "ell_hist": z(gamma + 1)}


def accept_stats(n_accept, gamma, *, ell=None, counters=None, err=None, stream=None):
    """Per-position conditional acceptance counts and the acceptance-length
    histogram of one cycle (include/dspark.h), added into ``counters`` (a dict
    from accept_stats_counters; created when None).  n_accept [R] int32 from
    verify, ell [R] int32 verified lengths or None (gamma for all)."""
    L = load()
    dev = n_accept.device
    if n_accept.dtype != torch.int32 or (ell is not None and ell.dtype != torch.int32):
        raise TypeError("n_accept and ell are int32")
    c = counters if counters is not None else accept_stats_counters(gamma, dev)
    a = AcceptStatsArgs()
    a.R, a.gamma = n_accept.numel(), int(gamma)
    a.n_accept, a.ell = _ptr(n_accept), _ptr(ell)
    a.reached, a.accepted, a.tau_hist = _ptr(c["reached"]), _ptr(c["accepted"]), _ptr(c["tau_hist"])
    a.ell_hist, a.err = _ptr(c.get("ell_hist")), _ptr(err)
    _check(L.dspark_accept_stats(ctypes.byref(a), _stream(stream)))
    return c


# --------------------------------------------------------------------- training losses
def train_losses(zd, zt, xs, s, gamma, *, a_ce=0.1, a_tv=0.9, a_conf=1.0, want_row=True, want_grad=False,
                 err=None, stream=None):
    """The drafter's training losses (include/dspark.h; eqs. 8-12): zd, zt [N, V]
    draft and target logits (bf16 or fp32, N = B gamma), xs [N] int32 target
    tokens, s [N] fp32 confidence logits.  Returns {"loss": [4] fp64
    (L_ce, L_tv, L_conf, L), "row": [N, 6] fp32 or None, "grad_z": [N, V] fp32
    or None, "grad_s": [N] fp32 or None}."""
    L = load()
    N, V = zd.shape
    dev = zd.device
    if zt.shape != zd.shape or zt.dtype != zd.dtype:
        raise TypeError("zd and zt must match in shape and dtype")
    if xs.dtype != torch.int32 or s.dtype != torch.float32:
        raise TypeError("xs is int32 and s float32")
    if N % gamma:
        raise ValueError("rows must be blocks x gamma")
    a = TrainLossArgs()
    a.B, a.gamma, a.V, a.dtype = N // gamma, int(gamma), V, _dtype_code(zd)
    a.zd, a.zt, a.xs, a.s = _ptr(zd), _ptr(zt), _ptr(xs), _ptr(s)
    a.a_ce, a.a_tv, a.a_conf = float(a_ce), float(a_tv), float(a_conf)
    out = {"loss": torch.empty(4, dtype=torch.float64, device=dev),
           "row": torch.empty((N, 6), dtype=torch.float32, device=dev) if want_row else None,
           "grad_z": torch.empty((N, V), dtype=torch.float32, device=dev) if want_grad else None,
           "grad_s": torch.empty(N, dtype=torch.float32, device=dev) if want_grad else None}
    a.row, a.loss, a.grad_z, a.grad_s = _ptr(out["row"]), _ptr(out["loss"]), _ptr(out["grad_z"]), _ptr(out["grad_s"])
    a.err = _ptr(err)
    _check(L.dspark_train_losses(ctypes.byref(a), _stream(stream)))
    return out
