"""Runs of the oracle for the full-size parity tests (test infrastructure).

The dense prefill oracle materialises a ``[q_len, kv_len]`` score matrix per
head in float64; the largest workload has 256 of them.  Here the heads of one
(batch, KV head) group go to one worker of a process pool started with the
``spawn`` method (so no worker inherits the parent's CUDA context), each worker
running the oracle unchanged, on its own input slice, with one BLAS thread.
The slice keeps the oracle's own GQA repeat: a worker receives the G query
heads of one KV head together with that KV head.

This module imports numpy and the oracle only.
"""

import contextlib
import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _prefill_group(task):
    import oracle
    b, kvh, q, k, v = task
    o, lse = oracle.prefill(q, k, v)
    return b, kvh, o, lse


@contextlib.contextmanager
def _single_threaded_children():
    saved = {k: os.environ.get(k) for k in _THREAD_VARS}
    for k in _THREAD_VARS:
        os.environ[k] = "1"
    try:
        yield
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def workers():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, 32))


def prefill_by_group(q, k, v):
    """Yield ``(b, kvh, o, lse)`` for every (batch, KV head) of a prefill:
    ``o [1, G, q_len, D]`` and ``lse [1, G, q_len]`` are ``oracle.prefill`` of
    query heads ``kvh*G .. kvh*G+G-1`` of batch ``b`` against KV head ``kvh``.
    ``q, k, v`` are float32 or float64 numpy arrays in the prefill layouts."""
    bsz, hq = q.shape[:2]
    hkv = k.shape[1]
    g = hq // hkv
    tasks = [(b, kvh, q[b:b + 1, kvh * g:(kvh + 1) * g], k[b:b + 1, kvh:kvh + 1], v[b:b + 1, kvh:kvh + 1])
             for b in range(bsz) for kvh in range(hkv)]
    ctx = multiprocessing.get_context("spawn")
    with _single_threaded_children():
        with ProcessPoolExecutor(max_workers=min(workers(), len(tasks)), mp_context=ctx) as ex:
            for res in ex.map(_prefill_group, tasks, chunksize=1):
                yield res


class WholeOutputCheck:
    """Accumulates the comparison of a whole output with the oracle, piece by
    piece: the maximum absolute error, the mean absolute error over every
    element of the output, and the LSE error and its -inf pattern."""

    def __init__(self):
        self.o_max = 0.0
        self.o_sum = 0.0
        self.o_count = 0
        self.lse_max = 0.0
        self.rows = 0

    def add(self, o_gpu, o_ref, lse_gpu, lse_ref):
        o_gpu = np.asarray(o_gpu, dtype=np.float64)
        assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
        assert np.all(np.isfinite(o_gpu)), "O: non-finite values"
        err = np.abs(o_gpu - o_ref)
        self.o_max = max(self.o_max, float(err.max()) if err.size else 0.0)
        self.o_sum += float(err.sum())
        self.o_count += err.size
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        assert lse_gpu.shape == lse_ref.shape
        dead = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), dead), "LSE: -inf pattern differs"
        live = ~dead
        if live.any():
            self.lse_max = max(self.lse_max, float(np.abs(lse_gpu[live] - lse_ref[live]).max()))
        self.rows += lse_ref.size

    @property
    def o_mean(self):
        return self.o_sum / max(1, self.o_count)
