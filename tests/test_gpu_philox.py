"""The device Philox-4x32-10 (the sampler's generator) against the published
known-answer vectors of Salmon et al., SC'11 (tests/golden/philox4x32_10_kat.txt),
and against the oracle's own Philox on many random counters and keys."""
import os

import numpy as np
import pytest
import torch

from speculative_decoding_drafter_markov_gb300 import _lib as dsp

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            v = [int(t, 16) for t in line.split()]
            rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


def _device_philox(ctr_u32, seed):
    ctr = torch.as_tensor(np.ascontiguousarray(ctr_u32, np.uint32).view(np.int32), device="cuda")
    out = dsp.philox(ctr, seed)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("ctr,key,expect", _kat())
def test_device_philox_known_answers(ctr, key, expect):
    seed = key[0] | (key[1] << 32)
    out = _device_philox(np.array([ctr], np.uint32), seed)
    assert [int(v) for v in out[0]] == expect


def test_device_philox_matches_oracle(orc):
    rng = np.random.default_rng(123)
    for seed in (0, 1234, int(rng.integers(0, 2**63))):
        ctr = rng.integers(0, 2**32, (4096, 4), dtype=np.uint64).astype(np.uint32)
        out = _device_philox(ctr, seed)
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i in range(0, 4096, 97):
            assert np.array_equal(out[i], orc.philox4x32_10(ctr[i], key)), (seed, i)
