"""Full-size oracle runs spread over the host's cores.

The rows of a case are split into interleaved groups and each group is
computed by ``oracle.verify_case(case, rows=...)`` in a worker process.  The
workers are spawned (never forked: the parent may already hold a CUDA
context) and rebuild the seeded case from its recipe, the generator's name
and arguments, so no array crosses the process boundary; a fingerprint of
the rebuilt arrays is checked against the parent's case.  The arithmetic is
the oracle's own: this module only distributes rows.
"""
from __future__ import annotations

import hashlib
import multiprocessing as mp
import os

import numpy as np

_POOL = None


def workers() -> int:
    return max(1, min(os.cpu_count() or 1, 16))


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = mp.get_context("spawn").Pool(workers())
    return _POOL


def fingerprint(case) -> str:
    h = hashlib.sha256()
    for a in (case.q, case.k, case.v, case.ctx_len, case.cu_rows):
        a = np.ascontiguousarray(a)
        h.update(a.tobytes()[:1 << 20])
        h.update(str(a.shape).encode())
    return h.hexdigest()


def _rows_work(args):
    recipe, rows = args
    import oracle
    import synthetic as sy
    fn, kw = recipe
    case = getattr(sy, fn)(**kw)
    O, L = oracle.verify_case(case, rows=rows)
    return fingerprint(case), rows, O[rows], L[rows]


def oracle_full(recipe, case):
    """O [total_rows, H, D] and LSE [total_rows, H] (float64) of every
    (row, head) of ``case``, which ``recipe`` = (generator name, kwargs)
    rebuilds."""
    total = int(case.total_rows)
    n = min(total, 2 * workers())
    groups = [list(range(g, total, n)) for g in range(n)]
    O = np.full((total, case.num_heads, case.head_dim), np.nan)
    L = np.full((total, case.num_heads), np.nan)
    want = fingerprint(case)
    for fp, rows, o, l in _pool().imap_unordered(_rows_work, [(recipe, g) for g in groups]):
        assert fp == want, "worker rebuilt a different case"
        O[rows] = o
        L[rows] = l
    return O, L
