"""DSpark per-cycle hot path on one GB300 (sm_103a).

Semi-autoregressive Markov / RNN draft with confidences, the hardware-aware
prefix scheduler and lossless verification, as hand-written CUDA kernels behind
the C ABI in include/dspark.h.  This package is the thin Python binding.
"""
from ._lib import (  # noqa: F401
    BF16, F32, SCHED_ASYNC, SCHED_SYNC, DSparkError, build_tags, draft_markov,
    draft_markov_step, draft_markov_workspace_size, draft_rnn, load, philox, schedule, verify,
)

__all__ = ["draft_markov", "draft_rnn", "schedule", "build_tags", "verify", "philox", "load",
           "DSparkError"]
