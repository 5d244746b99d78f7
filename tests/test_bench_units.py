"""The bench's algorithmic units (the numerators of its roofline fractions)
against brute force over the oracle's slot lists, on CPU."""
import numpy as np
import torch

import bench
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
from oracle import csa_oracle as orc


def test_algorithmic_work_counts_the_oracle_slots():
    cfg = CONFIGS["tiny_fp32"]
    g = torch.Generator().manual_seed(5)
    # an index list with repeats, padding, out-of-range and not-yet-visible entries
    idx = torch.randint(-1, cfg.n_c + 3, (cfg.b, cfg.sq, cfg.K), generator=g, dtype=torch.int32)
    w = bench.algorithmic_work(cfg, idx)
    slots = sum(len(orc.query_slots(t, idx[bi, t].numpy(), cfg.sq, cfg.n_c, cfg.ratio, cfg.window))
                for bi in range(cfg.b) for t in range(cfg.sq))
    assert w["slots"] == slots
    vis_sum = sum(min(orc.visible_blocks(t, cfg.ratio), cfg.n_c) for t in range(cfg.sq)) * cfg.b
    assert w["indexer_flops"] == 2.0 * cfg.H_I * cfg.d_I * vis_sum
    e = 4 if cfg.dtype == "fp32" else 2
    assert w["fwd_gathered_bytes"] == slots * cfg.d * e
    assert w["bwd_gathered_bytes"] == slots * (cfg.d * e + 4 * cfg.d)
    assert w["fwd_flops"] == 4.0 * cfg.d * cfg.H * slots


def test_algorithmic_work_ragged_sequence():
    """sq not a multiple of the ratio: the last tokens see no extra block."""
    cfg = CONFIGS["tiny_fp32"].with_(name="ragged", sq=250)
    n_c = 250 // cfg.ratio
    idx = torch.arange(cfg.K, dtype=torch.int32).repeat(cfg.b, 250, 1) % (n_c + 1)
    w = bench.algorithmic_work(cfg, idx)
    slots = sum(len(orc.query_slots(t, idx[0, t].numpy(), 250, n_c, cfg.ratio, cfg.window))
                for t in range(250)) * cfg.b
    assert w["slots"] == slots
