"""Run oracle calls on all host cores, for the parity tests at full workload
sizes (131072 and 65536 tokens), where one head's oracle backward takes
minutes on one core.

Workers are started with the ``spawn`` method, so the pool is safe to create
after the parent has initialised CUDA.  Each worker runs one BLAS thread.
Arrays go to the workers as float64 ``.npy`` files in a temporary directory,
memory-mapped read-only by each task, so a head is written once and shared
through the page cache; ``release`` deletes them.  The workers call the
oracle's own functions; this module adds no arithmetic.
"""
from __future__ import annotations

import atexit
import concurrent.futures as cf
import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

_pool = None
_dir = None


def workers() -> int:
    return max(1, min(32, len(os.sched_getaffinity(0))))


def pool() -> cf.ProcessPoolExecutor:
    global _pool
    if _pool is None:
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"      # inherited by the workers spawned below
        _pool = cf.ProcessPoolExecutor(workers(), mp_context=mp.get_context("spawn"))
        atexit.register(shutdown)
    return _pool


def shutdown():
    global _pool, _dir
    if _pool is not None:
        _pool.shutdown(cancel_futures=True)
        _pool = None
    if _dir is not None:
        shutil.rmtree(_dir, ignore_errors=True)
        _dir = None


def share(tag: str, **arrays) -> dict:
    """Write float64 copies of ``arrays`` for the workers; returns name -> path."""
    global _dir
    if _dir is None:
        _dir = tempfile.mkdtemp(prefix="ra_oracle_")
    out = {}
    for name, a in arrays.items():
        path = os.path.join(_dir, f"{tag}_{name}.npy")
        np.save(path, np.ascontiguousarray(a, dtype=np.float64))
        out[name] = path
    return out


def release(paths: dict):
    """Delete files written by ``share`` (tasks still running keep their maps)."""
    for path in paths.values():
        try:
            os.remove(path)
        except FileNotFoundError:
            pass


def _arr(path: str):
    return np.load(path, mmap_mode="r")


# ----------------------------------------------------------------- worker tasks
def _kv_rows_part(paths, keys, N, causal, layout, query_rows):
    import oracle as orc
    return orc.attention_bwd_kv_rows(_arr(paths["q"]), _arr(paths["k"]), _arr(paths["v"]), _arr(paths["do"]),
                                     keys, N, causal, layout, row_chunk=128, query_rows=query_rows)


def _dq_rows(paths, rows, N, causal, layout):
    import oracle as orc
    return orc.attention_bwd_dq_rows(_arr(paths["q"]), _arr(paths["k"]), _arr(paths["v"]), _arr(paths["do"]),
                                     rows, N, causal, layout)


def _fwd_rows(paths, rows, N, causal, layout):
    import oracle as orc
    return orc.attention_rows(_arr(paths["q"]), _arr(paths["k"]), _arr(paths["v"]), rows, N, causal, layout)


def _full_head(paths, out_prefix, N, causal, layout, with_bwd, row_chunk):
    import oracle as orc
    q, k, v = (np.asarray(_arr(paths[x])) for x in ("q", "k", "v"))
    o, lse = orc.naive_attention(q[None, None], k[None, None], v[None, None], N, causal, layout,
                                 row_chunk=row_chunk)
    res = {"o": o[0, 0], "lse": lse[0, 0]}
    if with_bwd:
        do = np.asarray(_arr(paths["do"]))
        res["dq"], res["dk"], res["dv"] = orc.attention_bwd_head_chunked(q, k, v, res["o"], res["lse"], do, N,
                                                                         causal, layout, row_chunk=row_chunk)
    out = {}
    for name, a in res.items():
        out[name] = out_prefix + name + ".npy"
        np.save(out[name], a)
    return out


# ------------------------------------------------------------------ parent API
def full_heads(head_paths: list, N, causal, layout, with_bwd: bool, row_chunk: int = 256):
    """The whole oracle of each head (``naive_attention`` over every row, and
    ``attention_bwd_head_chunked`` if ``with_bwd``), one head per task, on
    inputs shared with ``share``.  Yields (index, paths of the .npy results)
    as heads finish; the caller releases both."""
    global _dir
    if _dir is None:
        _dir = tempfile.mkdtemp(prefix="ra_oracle_")
    futs = {pool().submit(_full_head, p, os.path.join(_dir, f"full{n}_"), N, causal, layout, with_bwd,
                          row_chunk): n for n, p in enumerate(head_paths)}
    for f in cf.as_completed(futs):
        yield futs[f], f.result()



def kv_rows(paths, keys, N, causal, layout, S, part_rows=2048):
    """``oracle.attention_bwd_kv_rows`` for ``keys``, its sum over query rows
    split into parts of ``part_rows`` rows run in parallel and added up."""
    futs = [pool().submit(_kv_rows_part, paths, keys, N, causal, layout, np.arange(r0, min(S, r0 + part_rows)))
            for r0 in range(0, S, part_rows)]
    dk = dv = 0.0
    for f in futs:
        a, b = f.result()
        dk = dk + a
        dv = dv + b
    return dk, dv


def dq_rows(paths, rows, N, causal, layout, part=32):
    """``oracle.attention_bwd_dq_rows``, ``part`` rows per task."""
    rows = np.asarray(rows, dtype=np.int64)
    futs = [pool().submit(_dq_rows, paths, rows[c:c + part], N, causal, layout) for c in range(0, rows.size, part)]
    return np.concatenate([f.result() for f in futs])


def fwd_rows(paths, rows, N, causal, layout, part=32):
    """``oracle.attention_rows``, ``part`` rows per task."""
    rows = np.asarray(rows, dtype=np.int64)
    futs = [pool().submit(_fwd_rows, paths, rows[c:c + part], N, causal, layout) for c in range(0, rows.size, part)]
    res = [f.result() for f in futs]
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])
