"""Run independent oracle calls on worker processes (test infrastructure).

Part of the oracle, which is test infrastructure: only the tests, the smoke
check and the CPU-baseline legs of the benchmark use it.  Nothing here does
any of the method's arithmetic: it hands whole calls of the token-by-token
definition (``recurrence``) to a pool of ``spawn``-started processes, one call
per independent (sequence, head) chain or batch slice, and returns their
results in order.  Chains of the method share nothing, so running them apart
changes no result.

``spawn`` (not ``fork``) keeps the pool safe to start from a process that has
already used the GPU.  Each worker's math libraries are limited to one thread,
so ``workers`` processes use ``workers`` cores.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _call(spec):
    name, args, kwargs = spec
    from . import recurrence, state_pass  # noqa: F401  (imported in the worker)
    mod = state_pass if name.startswith("chunk_state") else recurrence
    return getattr(mod, name)(*args, **kwargs)


def default_workers():
    return max(1, os.cpu_count() or 1)


class ChainPool:
    """A pool of ``workers`` spawn-started processes that stays up across
    several ``map`` calls (``with ChainPool(n) as pool: pool.map(specs)``)."""

    def __init__(self, workers=None):
        self.workers = default_workers() if workers is None else max(1, int(workers))
        self._ex = None
        self._saved = {}

    def __enter__(self):
        if self.workers > 1:
            self._saved = {v: os.environ.get(v) for v in _THREAD_VARS}
            for v in _THREAD_VARS:
                os.environ[v] = "1"
            self._ex = cf.ProcessPoolExecutor(max_workers=self.workers,
                                              mp_context=mp.get_context("spawn"))
        return self

    def map(self, specs):
        if self._ex is None:
            return [_call(s) for s in specs]
        return list(self._ex.map(_call, specs))

    def __exit__(self, *exc):
        if self._ex is not None:
            self._ex.shutdown()
            self._ex = None
        for v, old in self._saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        return False


def map_calls(specs, workers=None):
    """Results of ``[recurrence.<name>(*args, **kwargs) for name, args, kwargs in specs]``
    computed on up to ``workers`` processes (all host cores by default)."""
    specs = list(specs)
    workers = default_workers() if workers is None else max(1, int(workers))
    with ChainPool(min(workers, len(specs))) as pool:
        return pool.map(specs)
