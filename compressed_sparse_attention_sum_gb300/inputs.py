"""Seeded synthetic workloads for the CSA hot path.

This module only draws random tensors and fixes shapes; it computes none of
the layer's arithmetic (no pooling, no indexer score, no top-k, no softmax).
Both the CUDA path (tests, benchmark) and the fp64 oracle take their inputs
from here, so the two sides always see bit-identical data.

The five workloads follow the shapes the Compressed Sparse Attention pages
discuss: the tiny fp32 case, the debug-scale bf16 case, the CSA-4 layer at
sq=4096 (Megatron-LM PR #6400, review of the gather backward: "sq=4096,
window=128, ratio=4 -> n_compressed=1024, n_kv=5120, v_head_dim=128"), an
HCA-style ratio-128 layer attending to every visible block, and a
production-width layer (DeepSeek-V4: 64 heads, head_dim 512, torchtitan PR
#4452).

Every tensor is drawn on the CPU from a ``torch.Generator`` seeded per
workload, in fp32, then cast to the storage dtype.  Indices fed to the
attention of the production-width workload are synthetic (Zipf-skewed,
10% padding); the other workloads take them from the indexer.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class CSAConfig:
    """Shape of one CSA layer problem.

    b: batch, sq: query tokens, H: query heads, d: shared K=V head dim,
    ratio: compress ratio, window: sliding-window length (raw tokens,
    including the query's own token), topk: indexer top-k, H_I / d_I:
    indexer heads and head dim (0 when the layer attends to every visible
    compressed block instead of running the indexer).
    """

    name: str
    b: int
    sq: int
    H: int
    d: int
    ratio: int
    window: int
    topk: int
    H_I: int
    d_I: int
    dtype: str  # "fp32" or "bf16"
    input_scale: str = "unit"  # "unit": N(0,1); "inv_sqrt_d": N(0,1)/sqrt(d)
    index_source: str = "indexer"  # "indexer" | "all_visible" | "zipf"
    zipf_exponent: float = 1.1
    pad_fraction: float = 0.0
    seed: int = 0

    @property
    def n_c(self) -> int:
        return self.sq // self.ratio

    @property
    def n_kv(self) -> int:
        return self.sq + self.n_c

    @property
    def K(self) -> int:
        """Top-k slots per query: min(topk, n_c)."""
        return min(self.topk, self.n_c)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def scale(self) -> float:
        """Softmax scale d**-0.5 (Megatron-LM PR #6400, CompressedSparseAttention init)."""
        return self.d ** -0.5

    def with_(self, **kw) -> "CSAConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: Dict[str, CSAConfig] = {
    "tiny_fp32": CSAConfig("tiny_fp32", b=1, sq=256, H=4, d=64, ratio=4, window=32,
                           topk=16, H_I=4, d_I=32, dtype="fp32"),
    "debug_bf16": CSAConfig("debug_bf16", b=1, sq=2048, H=16, d=128, ratio=4, window=128,
                            topk=256, H_I=8, d_I=64, dtype="bf16", input_scale="inv_sqrt_d"),
    "csa4_bf16": CSAConfig("csa4_bf16", b=1, sq=4096, H=32, d=128, ratio=4, window=128,
                           topk=512, H_I=64, d_I=128, dtype="bf16"),
    "hca_bf16": CSAConfig("hca_bf16", b=2, sq=8192, H=32, d=128, ratio=128, window=128,
                          topk=64, H_I=0, d_I=0, dtype="bf16", index_source="all_visible"),
    "prod_bf16": CSAConfig("prod_bf16", b=2, sq=8192, H=64, d=512, ratio=4, window=128,
                           topk=1024, H_I=64, d_I=128, dtype="bf16", index_source="zipf",
                           pad_fraction=0.10),
}

CONFIG_ORDER = ["tiny_fp32", "debug_bf16", "csa4_bf16", "hca_bf16", "prod_bf16"]


def _normal(g: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_inputs(cfg: CSAConfig, parts=("compress", "indexer", "attn"),
                index_override: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Draw the seeded inputs of one workload (CPU tensors, storage dtype).

    Returned keys (subset according to ``parts``):
      kv_raw  [b, sq, d]        raw shared K=V rows
      score   [b, sq, d]        pooling scores = kv_raw @ W_pool, W_pool ~ N(0, 0.02)
      q_I     [b, sq, H_I, d_I] indexer queries
      k_I     [b, n_c, d_I]     indexer keys (one head)
      w       [b, sq, H_I]      indexer head weights, fp32, N(0,1)/2
      q       [b, sq, H, d]     attention queries
      sink    [H]               per-head sink logits, fp32, N(0,1)
      dO      [b, sq, H, d]     upstream gradient of O
      idx     [b, sq, K] int32  (zipf / all_visible workloads only)
    The compressed rows of kv_full are not drawn here: they are the pooling
    of kv_raw, which the caller computes with the implementation under test
    or with the oracle.
    """
    g = torch.Generator().manual_seed(cfg.seed)
    dt = cfg.torch_dtype
    std = 1.0 if cfg.input_scale == "unit" else 1.0 / math.sqrt(cfg.d)
    out: Dict[str, torch.Tensor] = {}
    b, sq, d = cfg.b, cfg.sq, cfg.d
    # Draw order is fixed so that every key keeps its value when a part is skipped.
    kv_raw = _normal(g, (b, sq, d), std)
    w_pool = _normal(g, (d, d), 0.02)
    if "compress" in parts or "attn" in parts:
        out["kv_raw"] = kv_raw.to(dt)
    if "compress" in parts:
        # The pooling-score projection is the input of the compressor, not part of it.
        out["score"] = (kv_raw @ w_pool).to(dt)
    g_idx = torch.Generator().manual_seed(cfg.seed + 1)
    if cfg.H_I > 0 and "indexer" in parts:
        std_i = 1.0 if cfg.input_scale == "unit" else 1.0 / math.sqrt(cfg.d)
        out["q_I"] = _normal(g_idx, (b, sq, cfg.H_I, cfg.d_I), std_i).to(dt)
        out["k_I"] = _normal(g_idx, (b, cfg.n_c, cfg.d_I), std_i).to(dt)
        out["w"] = _normal(g_idx, (b, sq, cfg.H_I), 0.5)
    g_att = torch.Generator().manual_seed(cfg.seed + 2)
    if "attn" in parts:
        out["q"] = _normal(g_att, (b, sq, cfg.H, d), std).to(dt)
        out["sink"] = _normal(g_att, (cfg.H,), 1.0)
        out["dO"] = _normal(g_att, (b, sq, cfg.H, d), std).to(dt)
        if index_override is not None:
            out["idx"] = index_override
        elif cfg.index_source == "all_visible":
            out["idx"] = all_visible_indices(cfg.b, cfg.sq, cfg.ratio, cfg.K)
        elif cfg.index_source == "zipf":
            out["idx"] = zipf_indices(cfg, torch.Generator().manual_seed(cfg.seed + 3))
    return out


def visible_blocks(sq: int, ratio: int) -> torch.Tensor:
    """vis(t) = (t+1)//ratio for t in [0, sq): the number of complete blocks
    that end at or before token t (Megatron-LM PR #6400, causal compressed mask;
    torchtitan PR #4452: "j < (t+1)//ratio")."""
    return (torch.arange(1, sq + 1) // ratio).to(torch.int64)


def all_visible_indices(b: int, sq: int, ratio: int, K: int) -> torch.Tensor:
    """Index list of a layer that attends to every visible compressed block
    (HCA / dense mode): row t holds 0..vis(t)-1 followed by -1 padding."""
    vis = visible_blocks(sq, ratio)
    j = torch.arange(K).view(1, K)
    idx = torch.where(j < vis.view(sq, 1), j, torch.full_like(j, -1)).to(torch.int32)
    return idx.view(1, sq, K).expand(b, sq, K).contiguous()


def zipf_indices(cfg: CSAConfig, g: torch.Generator) -> torch.Tensor:
    """Synthetic top-k lists: per query, min(K, vis(t)) distinct visible blocks
    drawn with P(j) proportional to (j+1)^-s (Gumbel-top-k sampling), sorted
    ascending, then a seeded fraction of all slots set to -1 at random
    positions of the row."""
    b, sq, n_c, K = cfg.b, cfg.sq, cfg.n_c, cfg.K
    vis = visible_blocks(sq, cfg.ratio)
    logp = -cfg.zipf_exponent * torch.log(torch.arange(1, n_c + 1, dtype=torch.float32))
    out = torch.empty(b, sq, K, dtype=torch.int32)
    jj = torch.arange(n_c).view(1, n_c)
    chunk = 1024
    for bi in range(b):
        for t0 in range(0, sq, chunk):
            t1 = min(sq, t0 + chunk)
            u = torch.rand(t1 - t0, n_c, generator=g).clamp_(1e-12, 1.0 - 1e-7)
            key = logp.view(1, n_c) - torch.log(-torch.log(u))
            key = key.masked_fill(jj >= vis[t0:t1].view(-1, 1), float("-inf"))
            top = torch.topk(key, K, dim=1)
            sel = torch.where(torch.isinf(top.values), torch.full_like(top.indices, n_c + 1),
                              top.indices)
            sel, _ = torch.sort(sel, dim=1)
            sel = torch.where(sel > n_c, torch.full_like(sel, -1), sel)
            out[bi, t0:t1] = sel.to(torch.int32)
    if cfg.pad_fraction > 0:
        drop = torch.rand(b, sq, K, generator=g) < cfg.pad_fraction
        out = out.masked_fill(drop, -1)
    return out.contiguous()


def packed_doc_ids(b: int, sq: int, ratio: int, n_docs: int, seed: int = 0) -> torch.Tensor:
    """Per-token document ids [b, sq] int32 of n_docs packed documents per
    batch element.  Documents are consecutive runs whose boundaries fall on
    multiples of `ratio` (packing pads every document to a multiple of the
    compress ratio, torchtitan PR #4452), at seeded random positions; the
    ids are 0..n_docs-1 in order."""
    g = torch.Generator().manual_seed(1000 + seed)
    slots = sq // ratio
    assert 1 <= n_docs <= slots
    out = torch.empty(b, sq, dtype=torch.int32)
    for bi in range(b):
        cuts = torch.randperm(slots - 1, generator=g)[:n_docs - 1] + 1
        cuts, _ = torch.sort(cuts * ratio)
        ids = torch.zeros(sq, dtype=torch.int32)
        for c in cuts.tolist():
            ids[c:] += 1
        out[bi] = ids
    return out


def to_f64(t: torch.Tensor):
    """Exact widening of a stored tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()
