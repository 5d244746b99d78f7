"""One CSA layer split by query rows across ranks (one GPU each).

Every query's indexer row, top-k and attention read only inputs that all
ranks hold (kv_full, k_I, the sink), so each rank processes a subset of the
query rows with the row-range calls of the library (csa_indexer_topk_rows,
csa_attn_fwd_rows, csa_attn_bwd_rows) and no exchange; the backward's
scatter into the compact [b, n_kv, d] dKV buffer and the per-head dsink are
the only results that cross rows, and they sum, so one sum-reduction of
[dkv, dsink] completes the layer's gradients.  The pages keep the sink per
head and guard against splitting heads across ranks ("Add unfused SBHD
compressed sparse attention", attention-sink parameter and the review of its
tensor-parallel guard), which leaves the query rows as the axis to split.

Causal work grows with the query position (more visible compressed blocks,
up to the top-k), so equal row counts would leave the ranks unbalanced; the
rows are cut instead into N contiguous ranges of equal estimated work, with
the work of row t taken as its attention slots (window rows and selected
blocks) times the attention's flops per slot plus its visible blocks times
the indexer's flops per block.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np
import torch

ALIGN = 8   # range boundaries on multiples of 8 rows (the attention's query blocks)


def row_work(sq: int, ratio: int, window: int, K: int, H: int, d: int, H_I: int = 0,
             d_I: int = 0) -> np.ndarray:
    """Estimated work of each query row: 14 d H flops per attention slot
    (forward and backward) and 2 H_I d_I flops per visible block (indexer)."""
    t = np.arange(sq, dtype=np.float64)
    vis = np.floor((t + 1) / ratio)
    slots = np.minimum(t + 1, window) + np.minimum(vis, K)
    return 14.0 * d * H * slots + 2.0 * H_I * d_I * vis


def balanced_ranges(work: np.ndarray, world: int, rank: int,
                    align: int = ALIGN) -> List[Tuple[int, int]]:
    """The query rows [t_begin, t_end) of `rank` among `world` ranks: the
    rows are cut into `world` contiguous ranges of near-equal total work
    (boundaries on multiples of `align`).  The ranges of all ranks partition
    [0, sq); a rank may get none when sq is small."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    sq = work.shape[0]
    cum = np.cumsum(work)
    cuts = [0]
    for k in range(1, world):
        t = int(np.searchsorted(cum, cum[-1] * k / world))
        t = int(round(t / align)) * align
        cuts.append(min(sq, max(cuts[-1], t)))
    cuts.append(sq)
    lo, hi = cuts[rank], cuts[rank + 1]
    return [(lo, hi)] if hi > lo else []


def config_ranges(cfg, world: int, rank: int) -> List[Tuple[int, int]]:
    """balanced_ranges for a workload (inputs.CSAConfig)."""
    return balanced_ranges(row_work(cfg.sq, cfg.ratio, cfg.window, cfg.K, cfg.H, cfg.d, cfg.H_I,
                                    cfg.d_I), world, rank)


def allreduce_grads(dkv: torch.Tensor, dsink, group=None) -> None:
    """Sum the ranks' dKV and dsink contributions in place with one
    collective (dkv and dsink packed into one buffer)."""
    import torch.distributed as dist
    if dsink is None:
        dist.all_reduce(dkv, op=dist.ReduceOp.SUM, group=group)
        return
    flat = torch.cat([dkv.reshape(-1), dsink.reshape(-1)])
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    dkv.copy_(flat[:dkv.numel()].view_as(dkv))
    dsink.copy_(flat[dkv.numel():].view_as(dsink))


def layer_rows(csa, x, cfg, ranges, kv_full, ws, idx_out, O, L, dq, dkv, dsink, dscore,
               idx_given: bool, group=None, world: int = 1, mark=None):
    """One rank's share of a layer step on the current stream: compress
    (every rank pools all blocks: the attention of any row may select any of
    them), the indexer and the attention forward and backward over this
    rank's query rows, the reduction of [dkv, dsink] over the ranks, then the
    compressor backward (every rank, on the reduced dkv).  `x` holds the
    layer inputs; outputs are written in place.  `mark(i)` (optional) is
    called at the phase boundaries 0..6 (e.g. to record CUDA events)."""
    mark = mark or (lambda i: None)
    sq = cfg.sq
    kv_full[:, :sq].copy_(x["kv_raw"])
    mark(0)
    csa.csa_compress(kv_full[:, :sq], x["score"], cfg.ratio, out=kv_full[:, sq:])
    mark(1)
    idx = x["idx"] if idx_given else idx_out
    if cfg.H_I > 0:
        for r in ranges:
            csa.csa_indexer_topk(x["q_I"], x["k_I"], x["w"], cfg.topk, cfg.ratio, workspace=ws,
                                 out_idx=idx_out, rows=r)
    mark(2)
    for r in ranges:
        csa.csa_attn_fwd(x["q"], kv_full, idx, x["sink"], cfg.scale, cfg.ratio, cfg.window,
                         out=O, lse=L, rows=r)
    mark(3)
    if not ranges:                       # a rank without rows contributes zeros
        dkv.zero_()
        if dsink is not None:
            dsink.zero_()
    for i, r in enumerate(ranges):
        csa.csa_attn_bwd(x["q"], kv_full, idx, x["sink"], cfg.scale, cfg.ratio, cfg.window, O, L,
                         x["dO"], dq=dq, dkv=dkv, dsink=dsink, rows=r, accumulate=i > 0)
    mark(4)
    if world > 1:
        allreduce_grads(dkv, dsink, group)
    mark(5)
    csa.csa_compress_bwd(kv_full[:, :sq], x["score"], cfg.ratio, dkv[:, sq:], dkv[:, :sq],
                         dscore=dscore)
    mark(6)
