"""The fp64 oracle's verify over every output column, run on all usable host
cores: contiguous column ranges, one oracle call per range (the C oracle is
called unchanged; it releases the GIL).  Columns are independent, so this is
the oracle over N in parallel, not a different computation.  Test helper."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def verify_all(fmt, parts, Xf, K, N, group):
    """(Y, A) of oracle.verify over all N columns."""
    nthr = max(1, len(os.sched_getaffinity(0)))
    ranges = [r for r in np.array_split(np.arange(N, dtype=np.int64), 2 * nthr) if r.size]
    with ThreadPoolExecutor(nthr) as ex:
        parts_out = list(ex.map(
            lambda c: oracle.verify(fmt, parts, Xf, K, N, group, cols=c), ranges))
    Y = np.concatenate([p[0] for p in parts_out], axis=1)
    A = np.concatenate([p[1] for p in parts_out], axis=1)
    return Y, A
