"""Running the single-threaded oracle over many requests at once.

Requests are independent in the draft and in verification, so the tests split a
request list into chunks and run one oracle call per chunk on host threads: the
oracle is plain C behind ctypes, which releases the GIL during the call, and
its functions keep no global state.  Each call still computes its requests one
by one exactly as a single call would; only the wall-clock time shrinks.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunks(reqs, n):
    reqs = [int(r) for r in reqs]
    n = max(1, min(n, len(reqs)))
    return [list(c) for c in np.array_split(np.asarray(reqs, dtype=np.int64), n) if len(c)]


def draft(fn, reqs, *args, **kw):
    """fn is oracle.draft_markov or oracle.draft_rnn; outputs are indexed by
    position in `reqs`, as one call with reqs=reqs would give them."""
    chunks = _chunks(reqs, threads())
    with ThreadPoolExecutor(len(chunks)) as ex:
        outs = list(ex.map(lambda c: fn(*args, reqs=c, **kw), chunks))
    return {k: np.concatenate([o[k] for o in outs], axis=0) for k in outs[0]}


def verify(fn, reqs, T, tags, *args, **kw):
    """fn is oracle.verify: per-request outputs [R, ...] and per-row outputs [N]
    are written only for the listed requests; the chunks' results are merged."""
    chunks = _chunks(reqs, threads())
    with ThreadPoolExecutor(len(chunks)) as ex:
        outs = list(ex.map(lambda c: fn(T, tags, *args, reqs=c, **kw), chunks))
    tags = np.asarray(tags)
    merged = {k: v.copy() for k, v in outs[0].items()}
    for c, o in zip(chunks[1:], outs[1:]):
        rows = np.isin(tags[:, 0], c)
        for k, v in o.items():
            if v.shape[0] == tags.shape[0] and k in ("lse_p", "logp", "margin"):
                merged[k][rows] = v[rows]
            else:
                merged[k][c] = v[c]
    return merged
