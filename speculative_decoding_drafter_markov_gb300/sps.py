"""Profiled cost table SPS(B) for the prefix scheduler.

DSpark digest, Module E: the scheduler weighs the expected accepted tokens tau
against the engine's step rate SPS(B) at verify batch B, Theta = tau SPS(B); the
rate curve is profiled once offline, so at run time the scheduler only looks it
up.  The production section notes that real curves are not smooth: capacity
falls in steps (the tile quantisation of the target's kernels), which is why the
deployed scheduler searches the whole curve instead of stopping at the first
drop.

`profile_sps` times a caller's target forward at a grid of batch sizes with CUDA
events and returns the table dspark_schedule takes (steps per second for every
B in [B_min, B_max], float64).  It is host-side plumbing around the caller's
forward; nothing of the scheduler runs here.
"""
from __future__ import annotations

import statistics

import numpy as np
import torch


def _cuda_timer(forward, B, reps, warmup):
    """Median seconds of forward(B) over `reps` runs, CUDA events on the current stream."""
    for _ in range(warmup):
        forward(B)
    times = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        forward(B)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    return statistics.median(times)


def profile_sps(forward, B_min: int, B_max: int, *, step: int = 8, reps: int = 3, warmup: int = 1,
                timer=None) -> np.ndarray:
    """SPS(B) for B = B_min..B_max: forward(B) is timed at B_min, B_min + step,
    ..., B_max (the last size always included); between two timed sizes the
    rate is interpolated linearly.  `timer(forward, B, reps, warmup)` returns
    seconds per call (CUDA events by default)."""
    if B_min < 1 or B_max < B_min or step < 1:
        raise ValueError("need 1 <= B_min <= B_max and step >= 1")
    timer = timer or _cuda_timer
    sizes = list(range(B_min, B_max + 1, step))
    if sizes[-1] != B_max:
        sizes.append(B_max)
    secs = np.array([timer(forward, B, reps, warmup) for B in sizes], dtype=np.float64)
    if not np.all(np.isfinite(secs)) or np.any(secs <= 0):
        raise RuntimeError("profiling gave a non-positive step time")
    rate = 1.0 / secs
    return np.interp(np.arange(B_min, B_max + 1, dtype=np.float64), np.array(sizes, np.float64), rate)
