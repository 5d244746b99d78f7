"""Shared helpers of the parity tests: oracle-side inputs and comparisons.

Every expected value here comes from the fp64 oracle (oracle/), never from
the CUDA path.  Inputs come from the seeded generator and are handed to both
sides unchanged.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

from compressed_sparse_attention_sum_gb300 import inputs as csa_inputs
from oracle import csa_oracle as orc

# Tolerances of the method: max abs error vs the oracle.
TOL = {"fp32": 2e-3, "bf16": 2e-2}
TOPK_GAP = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


@functools.lru_cache(maxsize=8)
def oracle_kv_full(cfg_name: str):
    """kv_full of a workload: raw rows + the oracle's pooled rows, rounded to
    the storage dtype (the one cast of the compressor)."""
    cfg = csa_inputs.CONFIGS[cfg_name]
    inp = csa_inputs.make_inputs(cfg, parts=("compress",))
    kv_raw = f64(inp["kv_raw"])
    kv_c = orc.compress(kv_raw, f64(inp["score"]), cfg.ratio, out_dtype=cfg.dtype)
    kv_full = np.concatenate([kv_raw, kv_c], axis=1)
    return torch.from_numpy(kv_full).to(cfg.torch_dtype)


@functools.lru_cache(maxsize=4)
def oracle_indexer(cfg_name: str):
    """Full oracle score matrix [b, sq, n_c] (-inf beyond vis) and top-k."""
    cfg = csa_inputs.CONFIGS[cfg_name]
    inp = csa_inputs.make_inputs(cfg, parts=("indexer",))
    I = orc.indexer_scores(f64(inp["q_I"]), f64(inp["k_I"]), f64(inp["w"]), cfg.ratio)
    idx = orc.topk_select(I, cfg.K)
    return I, idx


def attn_indices(cfg) -> torch.Tensor:
    """Index list fed to the attention of a workload (oracle top-k for the
    indexer workloads, the generator's list otherwise)."""
    if cfg.index_source == "indexer":
        return torch.from_numpy(oracle_indexer(cfg.name)[1])
    return csa_inputs.make_inputs(cfg, parts=("attn",))["idx"]


def compare_topk_row(gpu_idx: np.ndarray, scores_vis: np.ndarray, K: int, gap: float = TOPK_GAP):
    """Compare one row of GPU top-k with the oracle's scores of that row.

    Returns (ok, exact_required).  Bit-exact set equality is required where
    the K-th / (K+1)-th oracle score gap exceeds `gap` or where the boundary
    is an exact tie (ties go to the lower index); otherwise every selected
    block must be within `gap` of the K-th score and every block more than
    `gap` above it must be selected.  Always: ascending order, -1 tail,
    length min(K, vis).
    """
    v = scores_vis.shape[0]
    k = min(K, v)
    sel = gpu_idx[:k]
    if not (np.all(gpu_idx[k:] == -1) and np.all(sel >= 0) and np.all(sel < v)):
        return False, True
    if k > 1 and not np.all(np.diff(sel) > 0):
        return False, True
    ref = orc.topk_select_row(scores_vis, K)
    if k == v:
        return bool(np.array_equal(gpu_idx, ref)), True
    srt = np.sort(scores_vis)[::-1]
    kth, nxt = srt[k - 1], srt[k]
    if kth - nxt > gap or kth == nxt:
        return bool(np.array_equal(gpu_idx, ref)), True
    ok = np.all(scores_vis[sel] >= kth - gap) and set(np.nonzero(scores_vis > kth + gap)[0]) <= set(
        sel.tolist())
    return bool(ok), False


def maxabs(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0
