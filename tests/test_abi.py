"""The C-ABI library builds, loads without a GPU, exports every entry point that
include/dspark.h declares, matches the binding's struct layouts, and rejects bad
arguments on the host before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_drafter_markov_gb300 import _lib
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"DSPARK_API\s+[\w\s\*]+?\b(dspark_\w+)\s*\(", text)


def test_header_declares_the_four_calls():
    names = set(_declared())
    for n in ("dspark_draft_markov", "dspark_draft_rnn", "dspark_schedule", "dspark_verify"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_symbol():
    from speculative_decoding_drafter_markov_gb300 import _lib
    assert set(_declared()) == set(_lib.SYMBOLS)


def test_struct_layouts_match_header(tmp_path):
    from speculative_decoding_drafter_markov_gb300 import _lib
    src = tmp_path / "sizes.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "dspark.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\","
        "sizeof(dspark_draft_args),sizeof(dspark_rnn_args),sizeof(dspark_sched_args),"
        "sizeof(dspark_verify_args),offsetof(dspark_draft_args,seed),"
        "offsetof(dspark_sched_args,K_in),offsetof(dspark_verify_args,seed),"
        "offsetof(dspark_draft_args,conf_logit),sizeof(dspark_sts_args),"
        "offsetof(dspark_sts_args,curve));return 0;}\n")
    exe = tmp_path / "sizes"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    expect = [ctypes.sizeof(_lib.DraftArgs), ctypes.sizeof(_lib.RnnArgs),
              ctypes.sizeof(_lib.SchedArgs), ctypes.sizeof(_lib.VerifyArgs),
              _lib.DraftArgs.seed.offset, _lib.SchedArgs.K_in.offset, _lib.VerifyArgs.seed.offset,
              _lib.DraftArgs.conf_logit.offset, ctypes.sizeof(_lib.StsArgs), _lib.StsArgs.curve.offset]
    assert got == expect


def test_version_and_error_string(lib):
    assert lib.dspark_version() >= 100
    assert isinstance(lib.dspark_last_error(), bytes)


def test_host_side_validation(lib):
    from speculative_decoding_drafter_markov_gb300 import _lib
    byref = ctypes.byref
    # null argument structs
    assert lib.dspark_draft_markov(None, None, None) == _lib.ERR_INVAL
    assert lib.dspark_schedule(None, None, None) == _lib.ERR_INVAL
    assert lib.dspark_verify(None, None, None) == _lib.ERR_INVAL
    # bad draft shape
    a = _lib.DraftArgs()
    a.R, a.gamma, a.V, a.r, a.d, a.dtype = 0, 4, 100, 8, 8, 0
    assert lib.dspark_draft_markov(byref(a), None, None) == _lib.ERR_INVAL
    assert b"bad shape" in lib.dspark_last_error()
    a.R = 4
    a.dtype = 7
    assert lib.dspark_draft_markov(byref(a), None, None) == _lib.ERR_INVAL
    a.dtype = 1
    a.r = 4096
    assert lib.dspark_draft_markov(byref(a), None, None) == _lib.ERR_UNSUPPORTED
    a.r = 8
    assert lib.dspark_draft_markov(byref(a), None, None) == _lib.ERR_INVAL  # null tensors
    assert lib.dspark_draft_markov_workspace_size(byref(a)) == 0
    # scheduler: pool too large, table too short
    s = _lib.SchedArgs()
    s.R, s.gamma, s.mode = 1024, 16, 0
    assert lib.dspark_schedule(byref(s), None, None) == _lib.ERR_UNSUPPORTED
    dummy = ctypes.c_void_p(16)
    s.R, s.gamma = 4, 4
    s.c = s.sps = s.ell = s.K_out = s.theta_best = dummy
    s.B_min, s.B_count = 4, 10  # needs B up to 20
    assert lib.dspark_schedule(byref(s), None, None) == _lib.ERR_RANGE
    s.B_min = 5
    s.B_count = 30
    assert lib.dspark_schedule(byref(s), None, None) == _lib.ERR_RANGE
    s.mode = 9
    assert lib.dspark_schedule(byref(s), None, None) == _lib.ERR_INVAL
    # verify: fewer rows than requests
    v = _lib.VerifyArgs()
    v.R, v.gamma, v.V, v.r, v.dtype, v.N = 4, 4, 100, 8, 1, 3
    assert lib.dspark_verify(byref(v), None, None) == _lib.ERR_INVAL
    v.N = 21
    assert lib.dspark_verify(byref(v), None, None) == _lib.ERR_INVAL
    # calibration fit: shapes and limits are checked on the host
    t = _lib.StsArgs()
    assert lib.dspark_sts_fit(None, None, None) == _lib.ERR_INVAL
    t.M, t.gamma, t.G, t.n_bins = 0, 4, 8, 10
    assert lib.dspark_sts_fit(byref(t), None, None) == _lib.ERR_INVAL
    t.M = 16
    t.n_bins = 65
    assert lib.dspark_sts_fit(byref(t), None, None) == _lib.ERR_UNSUPPORTED
    t.n_bins, t.gamma = 10, 65
    assert lib.dspark_sts_fit(byref(t), None, None) == _lib.ERR_UNSUPPORTED
    t.gamma = 4
    assert lib.dspark_sts_fit(byref(t), None, None) == _lib.ERR_INVAL  # null tensors
    # bin sums (8 B each) + counters + two prefix buffers, each 256-byte aligned
    assert lib.dspark_sts_fit_workspace_size(byref(t)) == 4 * 8 * 10 * 8 + 256 + 2 * 256
    # acceptance diagnostics: shapes, limits and pointers are checked on the host
    d = _lib.AcceptStatsArgs()
    assert lib.dspark_accept_stats(None, None) == _lib.ERR_INVAL
    d.R, d.gamma = 4, 0
    assert lib.dspark_accept_stats(byref(d), None) == _lib.ERR_INVAL
    d.gamma = 1025
    assert lib.dspark_accept_stats(byref(d), None) == _lib.ERR_UNSUPPORTED
    d.gamma = 8
    assert lib.dspark_accept_stats(byref(d), None) == _lib.ERR_INVAL  # null counters
    d.reached = d.accepted = d.tau_hist = ctypes.c_void_p(16)
    d.R = 0
    assert lib.dspark_accept_stats(byref(d), None) == _lib.OK  # nothing to count: no launch
    # training losses
    tl = _lib.TrainLossArgs()
    assert lib.dspark_train_losses(None, None) == _lib.ERR_INVAL
    tl.B, tl.gamma, tl.V, tl.dtype = 2, 4, 100, _lib.BF16
    assert lib.dspark_train_losses(byref(tl), None) == _lib.ERR_UNSUPPORTED  # V % 8 for bf16
    tl.V = 96
    assert lib.dspark_train_losses(byref(tl), None) == _lib.ERR_INVAL  # null tensors
    tl.dtype = 7
    assert lib.dspark_train_losses(byref(tl), None) == _lib.ERR_INVAL
    tl.dtype = _lib.F32
    tl.zd = tl.zt = tl.xs = tl.s = tl.loss = ctypes.c_void_p(16)
    tl.grad_z = ctypes.c_void_p(24)
    assert lib.dspark_train_losses(byref(tl), None) == _lib.ERR_INVAL  # misaligned gradient rows
