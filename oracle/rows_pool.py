"""Run the fp64 oracle over many query rows on every host core.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by the
full-size parity tests and by the oracle timings of ``bench.py``.  It adds no
arithmetic of its own: each worker calls the oracle's functions on a subset
of query rows and returns what they return.

Inputs are written once to memory-mapped ``.npy`` files that every worker
maps read-only, so a production-width layer (1 GB per [b, sq, H, d] bf16
tensor) is held in host memory once, not once per process.  bf16 tensors are
stored as their 16-bit patterns and widened exactly to float64 one indexed
slice at a time (``Bf16Array``).  Workers are started with the ``spawn``
method, so a pool may be created after the parent has used the GPU.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile
from typing import Dict, Iterable, List

import numpy as np

__all__ = ["Bf16Array", "RowPool", "save_inputs"]


class Bf16Array:
    """Read-only view of a bf16 tensor stored as uint16 bit patterns: indexing
    returns float64 values (bf16 -> float64 is exact)."""

    def __init__(self, bits: np.ndarray):
        self.bits = bits
        self.shape = bits.shape
        self.ndim = bits.ndim

    def __getitem__(self, key):
        b = np.asarray(self.bits[key])
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def __len__(self):
        return self.shape[0]


def _to_numpy(t):
    """(array, is_bf16) of a torch tensor or numpy array (bf16 as its bits)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().to("cpu").contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), True
            return t.numpy(), False
    except ImportError:
        pass
    return np.ascontiguousarray(t), False


def _scratch_dir() -> str:
    shm = "/dev/shm"
    try:
        if os.path.isdir(shm) and shutil.disk_usage(shm).free > (16 << 30):
            return tempfile.mkdtemp(prefix="csa_oracle_", dir=shm)
    except OSError:
        pass
    return tempfile.mkdtemp(prefix="csa_oracle_")


def save_inputs(arrays: Dict[str, object], directory: str) -> Dict[str, tuple]:
    """Write each array to directory/<name>.npy; returns {name: (path, is_bf16)}."""
    out = {}
    for name, t in arrays.items():
        if t is None:
            out[name] = (None, False)
            continue
        a, is_bf16 = _to_numpy(t)
        path = os.path.join(directory, name + ".npy")
        np.save(path, a)
        out[name] = (path, is_bf16)
    return out


# ---------------------------------------------------------------------------
# worker side
# ---------------------------------------------------------------------------
_ARR: Dict[str, object] = {}
_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _worker_init(files: Dict[str, tuple]):
    for name, (path, is_bf16) in files.items():
        if path is None:
            _ARR[name] = None
            continue
        a = np.load(path, mmap_mode="r")
        _ARR[name] = Bf16Array(a) if is_bf16 else a


def _worker_call(task):
    fn, kwargs = task
    import importlib
    mod_name, fn_name = fn.rsplit(".", 1)
    f = getattr(importlib.import_module(mod_name), fn_name)
    return f(_ARR, **kwargs)


class RowPool:
    """A spawned pool of one process per host core over shared inputs.

    ``arrays``: name -> torch tensor or numpy array (saved once).
    ``map(fn, kwargs_list)`` calls ``fn(arrays, **kwargs)`` in the workers,
    where ``fn`` is a dotted path to a module-level function and ``arrays``
    maps each name to a read-only numpy array (float64 view for bf16).
    """

    def __init__(self, arrays: Dict[str, object], procs: int | None = None):
        self.procs = procs or (os.cpu_count() or 1)
        self.dir = _scratch_dir()
        self.files = save_inputs(arrays, self.dir)
        ctx = mp.get_context("spawn")
        # one BLAS thread per worker: the variables must be in the environment
        # the workers start with (their numpy is imported before any task runs)
        saved = {v: os.environ.get(v) for v in _BLAS_VARS}
        os.environ.update({v: "1" for v in _BLAS_VARS})
        try:
            self.pool = ctx.Pool(self.procs, initializer=_worker_init, initargs=(self.files,))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old

    def map(self, fn: str, kwargs_list: Iterable[dict]) -> List[object]:
        return self.pool.map(_worker_call, [(fn, kw) for kw in kwargs_list], chunksize=1)

    def close(self):
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def split_rows(rows: List[tuple], parts: int) -> List[List[tuple]]:
    """Interleaved split (row i to part i % parts), which balances the causal
    mix of short and long rows."""
    return [rows[i::parts] for i in range(parts) if rows[i::parts]]


# ---------------------------------------------------------------------------
# tasks (run in the workers; `A` is the mapping of shared arrays)
# ---------------------------------------------------------------------------

def attn_rows_vs(A, rows, scale, window, ratio):
    """Oracle forward and backward over `rows` [(b, t), ...] of the attention
    inputs A["q"], A["kv_full"], A["idx"], A["sink"], A["dO"], compared with
    a GPU run's outputs A["O"], A["L"], A["dq"] on the same rows.

    Returns (max |O - O_ref|, max |L - L_ref|, max |dq - dq_ref|,
    dkv contributions of these rows [b, n_kv, d], dsink contributions [H]).
    """
    from oracle import csa_oracle as orc
    kv = A["kv_full"]
    kv = kv[:] if isinstance(kv, Bf16Array) else np.asarray(kv, np.float64)
    sink = None if A["sink"] is None else np.asarray(A["sink"], np.float64)
    idx = A["idx"]
    O_ref, L_ref = orc.attn_fwd(A["q"], kv, idx, sink, scale, window, ratio, rows=rows)
    dq_ref, dkv, dsink = orc.attn_bwd(A["q"], kv, idx, sink, scale, window, ratio, A["dO"],
                                      rows=rows)
    e_o = e_l = e_dq = 0.0
    for n, (bi, t) in enumerate(rows):
        e_o = max(e_o, float(np.abs(A["O"][bi, t] - O_ref[n]).max()))
        e_l = max(e_l, float(np.abs(np.asarray(A["L"][bi, t], np.float64) - L_ref[n]).max()))
        e_dq = max(e_dq, float(np.abs(np.asarray(A["dq"][bi, t], np.float64) - dq_ref[n]).max()))
    return e_o, e_l, e_dq, dkv, dsink


def layer_rows(A, rows, scale, window, ratio, K, indexer):
    """The oracle's work for query rows [(b, t), ...] of one layer: the
    indexer scores and top-k of each row (when `indexer`), then attention
    forward and backward over the row's slots (the index list A["idx"] when it
    is given, else the row's own top-k) with the dKV scatter.  Returns the
    seconds spent."""
    import time
    from oracle import csa_oracle as orc
    kv = A["kv_full"]
    kv = kv[:] if isinstance(kv, Bf16Array) else np.asarray(kv, np.float64)
    sink = np.asarray(A["sink"], np.float64)
    b, sq = A["q"].shape[:2]
    n_c = kv.shape[1] - sq
    dkv = np.zeros(kv.shape[1:])
    t0 = time.perf_counter()
    for bi, t in rows:
        sel = None
        if indexer:
            scores = orc.indexer_scores_row(A["q_I"][bi, t], A["k_I"][bi],
                                            np.asarray(A["w"][bi, t], np.float64), t, ratio)
            sel = orc.topk_select_row(scores, K)
        if A.get("idx") is not None:
            sel = np.asarray(A["idx"][bi, t])
        slots = orc.query_slots(t, sel, sq, n_c, ratio, window)
        orc.attn_fwd_query(A["q"][bi, t], kv[bi], slots, sink, scale)
        _, dkv_s, _ = orc.attn_bwd_query(A["q"][bi, t], kv[bi], slots, sink, scale,
                                         A["dO"][bi, t])
        np.add.at(dkv, slots, dkv_s)
    return time.perf_counter() - t0
