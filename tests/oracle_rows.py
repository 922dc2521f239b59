"""The oracle on many selected query rows, spread over host processes.

Test harness only: it runs ``oracle.attention.attention_rows`` unchanged on
shares of the rows in spawned worker processes (spawn, never fork: the parent
has a CUDA context).  The parent writes the float64 K and V once to a
temporary directory; every worker memory-maps them read-only, so the large
KV buffers are neither pickled nor copied per worker.  Each row's result is
exactly what a single-process call gives for that row.
"""

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

_K = None
_V = None


def _init(k_path, k_shape, v_path, v_shape, v_cols):
    global _K, _V
    _K = np.memmap(k_path, dtype=np.float64, mode="r", shape=k_shape)
    if v_path is None:
        _V = _K[:, :, :v_cols]
    else:
        _V = np.memmap(v_path, dtype=np.float64, mode="r", shape=v_shape)


def _work(args):
    from oracle import attention as oatt

    idx, q, pos, kv0, scale, kv_lo, kv_hi = args
    O, L = oatt.attention_rows(q, _K, _V, pos, kv0, scale, kv_lo, kv_hi)
    return idx, O, L


def workers():
    return max(1, min(16, len(os.sched_getaffinity(0))))


def attention_rows_parallel(q_rows, k64, v64, positions, kv_row0, scale, kv_lo=0, kv_hi=None,
                            v_is_k_prefix=False, procs=None):
    """(O [R, Hq, dv], L [R, Hq]) of oracle.attention.attention_rows for the
    given rows, computed in ``procs`` spawned processes.  With v_is_k_prefix,
    V is the first dv = v64.shape[2] columns of K (v64 may then be a view)."""
    q_rows = np.asarray(q_rows, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    kv_row0 = np.asarray(kv_row0, dtype=np.int64)
    R, Hq = q_rows.shape[0], q_rows.shape[1]
    dv = v64.shape[2]
    procs = procs or workers()
    need = k64.size * 8 + (0 if v_is_k_prefix else v64.size * 8)
    base = None  # memory-backed /dev/shm when it has room, else the default temp dir
    try:
        if shutil.disk_usage("/dev/shm").free > 2 * need:
            base = "/dev/shm"
    except OSError:
        pass
    tmp = tempfile.mkdtemp(prefix="oracle_rows_", dir=base)
    try:
        k_path = os.path.join(tmp, "k.f64")
        np.ascontiguousarray(k64, dtype=np.float64).tofile(k_path)
        v_path = None
        if not v_is_k_prefix:
            v_path = os.path.join(tmp, "v.f64")
            np.ascontiguousarray(v64, dtype=np.float64).tofile(v_path)
        # heaviest rows first, dealt round-robin into ~4 chunks per process
        order = np.argsort(-positions, kind="stable")
        nchunks = max(1, min(R, 4 * procs))
        chunks = [order[c::nchunks] for c in range(nchunks)]
        tasks = [(c, q_rows[c], positions[c], kv_row0[c], scale, kv_lo, kv_hi)
                 for c in chunks if len(c)]
        O = np.zeros((R, Hq, dv))
        L = np.full((R, Hq), -np.inf)
        ctx = mp.get_context("spawn")
        with ctx.Pool(procs, initializer=_init,
                      initargs=(k_path, tuple(k64.shape), v_path, tuple(v64.shape), dv)) as pool:
            for idx, o, lse in pool.imap_unordered(_work, tasks):
                O[idx] = o
                L[idx] = lse
        return O, L
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
