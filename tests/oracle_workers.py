"""Oracle evaluations run in worker processes (test infrastructure).

The full-length gate of the 100k-token workload evaluates 4096 query rows of
each sequence with the fp64 oracle; sequences are independent, so they run
in parallel processes.  The pool is started with the ``spawn`` method, which
is safe after the parent process has initialised CUDA.  Workers import only
numpy and the oracle.
"""
from __future__ import annotations

import multiprocessing as mp
import os


def _init_worker():
    # one BLAS thread per process: the processes already use every core
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"


def layer_rows(args):
    """One sequence through one layer, only the given query rows:
    args = (x [1, L, d], valid_len [1], layer params, n_heads, rows [1, R])."""
    import oracle
    x, vl, p, n_heads, rows = args
    return oracle.encoder_layer(x, vl, p, n_heads, rows=rows, check=False)


def make_pool(n: int | None = None):
    n = n or min(16, os.cpu_count() or 1)
    return mp.get_context("spawn").Pool(n, initializer=_init_worker)
