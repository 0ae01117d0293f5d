"""The draft entry point that allocates nothing, checked against the regular one.

Some callers cannot allocate device memory (a plugin inside another runtime whose
allocator owns the device, a C host without an allocator, code that must not
risk the device synchronisation cudaMalloc can cause).  For them
dspark_draft_markov_noalloc takes no workspace: its scratch is a fixed array in
the library.  This test calls it through the C ABI twice in a row and compares
each result with dspark_draft_markov given a caller-owned workspace.  It sits in
a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity import TOL_C, TOL_LOGQ, TOL_LSE, host
from speculative_decoding_drafter_markov_gb300 import _lib as dsp
from speculative_decoding_drafter_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(R, gamma):
    return {"x": torch.full((R, gamma), -7, dtype=torch.int32, device="cuda"),
            "logq": torch.full((R, gamma), np.nan, device="cuda"),
            "lse": torch.full((R, gamma), np.nan, device="cuda"),
            "c": torch.full((R, gamma), np.nan, device="cuda")}


def _call_noalloc(inp, out, err, seed, cycle):
    L = dsp.load()
    a = dsp._draft_struct(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                          seed, cycle, None, out, err)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.dspark_draft_markov_noalloc(ctypes.byref(a), stream)


@pytest.mark.parametrize("wl", [W.small("qwen4b", R=40, gamma=4, V=5000, r=64, d=32),
                                W.WORKLOADS["qwen4b"],
                                # CUDA-core path: fp32, ragged V and r
                                W.small("qwen4b", R=10, gamma=3, V=1001, r=24, d=40, dtype="f32")],
                         ids=lambda w: f"{w.name}-{w.dtype}")
def test_noalloc_matches_workspace_version(wl):
    inp = W.draft_inputs(wl, seed=3, device="cuda")
    for call, (seed, cycle) in enumerate([(11, 0), (11, 1)]):  # two calls in a row
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = dsp.draft_markov(inp["U"], inp["h"], inp["W1"], inp["W2t"], inp["w"], inp["anchor"],
                               seed=seed, cycle=cycle, err=err)
        out = _outputs(wl.R, wl.gamma)
        assert _call_noalloc(inp, out, err, seed, cycle) == dsp.OK
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        r, o = {k: host(v) for k, v in ref.items()}, {k: host(v) for k, v in out.items()}
        assert np.array_equal(o["x"], r["x"]), f"call {call}"
        assert np.abs(o["logq"] - r["logq"]).max() <= TOL_LOGQ
        assert np.abs(o["lse"] - r["lse"]).max() <= TOL_LSE
        assert np.abs(o["c"] - r["c"]).max() <= TOL_C


def test_noalloc_rejects_sizes_beyond_the_array():
    # V not a multiple of 8 takes the CUDA-core path: 512 x ceil(V/64) x 32 B > 16 MiB
    R, gamma, V, r, d = 512, 1, 129281, 256, 8
    z = lambda *s, dt=torch.bfloat16: torch.zeros(s, dtype=dt, device="cuda")
    inp = {"U": z(R, gamma, V), "h": z(R, gamma, d), "W1": z(V, r), "W2t": z(V, r),
           "w": z(d + r, dt=torch.float32), "anchor": z(R, dt=torch.int32)}
    out = _outputs(R, gamma)
    rc = _call_noalloc(inp, out, None, 0, 0)
    assert rc == dsp.ERR_UNSUPPORTED
    assert b"fixed array" in dsp.load().dspark_last_error()
    torch.cuda.synchronize()
    assert int(host(out["x"]).max()) == -7  # nothing was launched
