"""Row-parallel driver of the CPU oracle (test and baseline infrastructure, like the rest of
this package: only tests/, __graft_entry__.smoke() and bench.py's CPU legs use it).

The oracle itself is single-threaded C with per-call scratch in static storage, so it is run
unchanged in worker processes: each process loads its own copy of the oracle library, memory-
maps the blob from a temporary file (written once per Oracle object), and evaluates
oracle.gemv / oracle.abs_dot on a contiguous, row-block-aligned chunk of the requested rows. The
results are concatenated in row order, so every value is the one the single-process call gives,
bit for bit. Workers are started with the "spawn" method (safe after CUDA has been initialised
in the parent).
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

_pool = None
_pool_size = 0


def cores() -> int:
    """Host cores this process may run on."""
    return len(os.sched_getaffinity(0))


def _get_pool(workers: int):
    global _pool, _pool_size
    if _pool is None or _pool_size != workers:
        if _pool is not None:
            _pool.terminate()
        _pool = mp.get_context("spawn").Pool(workers)
        _pool_size = workers
    return _pool


def shutdown():
    global _pool, _pool_size
    if _pool is not None:
        _pool.terminate()
        _pool.join()
    _pool, _pool_size = None, 0


def _task(args):
    fn, path, x, rows = args
    import oracle
    blob = np.memmap(path, dtype=np.uint8, mode="r")
    return getattr(oracle, fn)(blob, x, rows)


def _chunks(rows: np.ndarray, parts: int):
    """Splits sorted-or-not row indices into about `parts` contiguous pieces, cutting only where
    the 8-row block changes so that no row block is decoded by two workers."""
    n = len(rows)
    if n == 0:
        return []
    cuts = [0]
    for p in range(1, parts):
        c = max(cuts[-1], p * n // parts)
        while 0 < c < n and rows[c] // 8 == rows[c - 1] // 8:
            c += 1
        if c >= n:
            break
        if c > cuts[-1]:
            cuts.append(c)
    cuts.append(n)
    return [rows[a:b] for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


class Oracle:
    """oracle.gemv / oracle.abs_dot of one blob over `workers` processes (all usable cores by
    default)."""

    def __init__(self, blob, workers: int | None = None):
        import oracle
        self.info = oracle.info(blob)
        self.workers = workers or cores()
        fd, self.path = tempfile.mkstemp(suffix=".nwcblob")
        with os.fdopen(fd, "wb") as f:
            f.write(bytes(blob))
        self.pool = _get_pool(self.workers)

    def _run(self, fn, x_bits, rows):
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        rows = np.arange(self.info["N"], dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
        parts = _chunks(rows, 2 * self.workers)
        outs = self.pool.map(_task, [(fn, self.path, x, r) for r in parts])
        return np.concatenate(outs) if outs else np.zeros(0, np.float64)

    def gemv(self, x_bits, rows=None) -> np.ndarray:
        return self._run("gemv", x_bits, rows)

    def abs_dot(self, x_bits, rows=None) -> np.ndarray:
        return self._run("abs_dot", x_bits, rows)

    def close(self):
        if self.path and os.path.exists(self.path):
            os.remove(self.path)
        self.path = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
