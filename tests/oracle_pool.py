"""Float64 oracle checks of full-size workloads, spread over spawned worker processes.

Test infrastructure only. A task is one (sequence, KV-head group) of a batch: the worker
receives that group's inputs and the CUDA path's outputs as float32 numpy arrays (bf16 and
float32 values are exact in float32), runs the oracle of ``oracle.attention`` on chunks of
query rows and returns error statistics, or returns the oracle's whole-group gradient. The
pool is started with the "spawn" method (a process forked after CUDA has been initialised
can hang), its workers import numpy and the oracle only, and each worker's BLAS uses a
share of the host cores.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from contextlib import contextmanager
from typing import Dict, List

import numpy as np

from oracle import attention as A

_CHUNK = 256  # query rows per oracle call: keeps a worker's score matrices to about half a GB


def _new():
    return [0.0, 0.0, 0.0, 0, 0.0]


def _acc(stat: List[float], got: np.ndarray, ref: np.ndarray) -> None:
    """Accumulate [max |err|, sum |err|, sum |ref|, count, max |ref|] of one chunk (a row
    without visible keys has LSE = -inf on both sides and counts as no error)."""
    same_inf = np.isinf(ref) & (got == ref)
    e = np.where(same_inf, 0.0, np.abs(got.astype(np.float64) - ref))
    r = np.where(np.isinf(ref), 0.0, np.abs(ref))
    stat[0] = max(stat[0], float(e.max()))
    stat[1] += float(e.sum())
    stat[2] += float(r.sum())
    stat[3] += e.size
    stat[4] = max(stat[4], float(r.max()))


def rows_task(args) -> Dict[str, List[float]]:
    """O, LSE (and dQ when dO is given) of a range of query rows of one sequence and KV-head
    group.

    args: (q [G,n,D], k [m,D], v [m,D], do [G,n,D] or None, o [G,n,D], lse [G,n],
    dq [G,n,D] or None, row0, causal): rows row0 .. row0+n-1 of the sequence; k and v hold
    the keys the rows can see (causal: positions 0 .. row0+n-1; full mask: the whole
    sequence). Rows go to the oracle in chunks; under a causal mask a chunk ending at row r1
    reads only the keys before r1."""
    q, k, v, do, o, lse, dq, row0, causal = args
    n = q.shape[1]
    st = {"o": _new(), "lse": _new()}
    if do is not None:
        st["dq"] = _new()
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        rows = np.arange(row0 + c0, row0 + c1)
        kend = row0 + c1 if causal else k.shape[0]
        ro, rl = A.attention_rows(q[:, c0:c1], k[:kend], v[:kend], rows, causal)
        _acc(st["o"], o[:, c0:c1], ro)
        _acc(st["lse"], lse[:, c0:c1], rl)
        if do is not None:
            rdq = A.attention_dq_rows(q[:, c0:c1], do[:, c0:c1], k[:kend], v[:kend], rows, causal)
            _acc(st["dq"], dq[:, c0:c1], rdq)
    return st


def group_backward_task(args):
    """The oracle's whole gradient (dQ [G,L,D], dK [L,D], dV [L,D]) of one sequence and
    KV-head group. args: (q [G,L,D], k [L,D], v [L,D], do [G,L,D], causal)."""
    q, k, v, do, causal = args
    L = k.shape[0]
    dq, dk, dv = A.attention_backward(q, k[None], v[None], do, [L], causal)
    return dq, dk[0], dv[0]


def _available_gb() -> float:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 2 ** 20
    except OSError:
        pass
    return 32.0


@contextmanager
def pool(n_tasks: int, gb_per_task: float = 4.0):
    """A spawn-method pool of up to one worker per host core (at most 16, and no more than the
    available memory holds at gb_per_task each), each worker's BLAS with an equal share of
    the cores."""
    cores = os.cpu_count() or 1
    n = max(1, min(n_tasks, 16, cores, int(_available_gb() / gb_per_task)))
    threads = str(max(1, cores // n))
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {key: os.environ.get(key) for key in keys}
    for key in keys:
        os.environ[key] = threads  # read by the children when they import numpy
    try:
        with mp.get_context("spawn").Pool(n) as p:
            yield p
    finally:
        for key, val in saved.items():
            if val is None:
                os.environ.pop(key, None)
            else:
                os.environ[key] = val
