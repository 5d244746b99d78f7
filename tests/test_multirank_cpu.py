"""The multi-rank host logic on two gloo ranks (CPU).

A layer is split by query rows across ranks (compressed_sparse_attention_sum_gb300.shard):
the partition into contiguous ranges of equal estimated work covers every
row once and balances the causal work,
and one sum-reduction of the ranks' dKV / dsink contributions gives the
layer's gradients.  Here each rank's contributions come from the fp64 oracle
over its own rows, so the test checks the partition and the reduction, the
host side of the path; the GPU side (the row-range calls reproducing the
whole-layer calls) is tests/test_gpu_rows.py.  The job's step time is the
maximum over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from compressed_sparse_attention_sum_gb300.inputs import CONFIGS
from compressed_sparse_attention_sum_gb300.shard import (allreduce_grads, balanced_ranges,
                                                        config_ranges, row_work)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("name", ["tiny_fp32", "csa4_bf16", "hca_bf16", "prod_bf16"])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_partition_covers_every_row_once(name, world):
    cfg = CONFIGS[name]
    seen = np.zeros(cfg.sq, np.int64)
    for r in range(world):
        for lo, hi in config_ranges(cfg, world, r):
            assert 0 <= lo < hi <= cfg.sq and lo % 8 == 0
            seen[lo:hi] += 1
    assert np.all(seen == 1)


def test_partition_of_a_short_sequence_may_leave_ranks_empty():
    work = np.ones(16)
    got = [balanced_ranges(work, 4, r) for r in range(4)]
    assert sum(len(g) for g in got) >= 1
    assert sorted(x for g in got for x in g) == [(0, 8), (8, 16)]


@pytest.mark.parametrize("name", ["csa4_bf16", "hca_bf16", "prod_bf16"])
@pytest.mark.parametrize("world", [2, 4, 8])
def test_partition_balances_causal_work(name, world):
    """The ranks' estimated work agrees within 2% (top-k saturation and the
    window make per-row work piecewise linear, so equal row counts would not)."""
    cfg = CONFIGS[name]
    work = row_work(cfg.sq, cfg.ratio, cfg.window, cfg.K, cfg.H, cfg.d, cfg.H_I, cfg.d_I)
    tot = [sum(work[lo:hi].sum() for lo, hi in config_ranges(cfg, world, r))
           for r in range(world)]
    assert max(tot) / min(tot) < 1.02, tot


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
        from oracle import csa_oracle as orc
        cfg = CONFIGS["tiny_fp32"].with_(index_source="zipf", pad_fraction=0.1)
        inp = make_inputs(cfg, parts=("compress", "attn"))
        f = lambda t: t.double().numpy()
        kv_c = orc.compress(f(inp["kv_raw"]), f(inp["score"]), cfg.ratio)
        kv = np.concatenate([f(inp["kv_raw"]), kv_c], axis=1)
        idx = inp["idx"].numpy()
        args = (f(inp["q"]), kv, idx, f(inp["sink"]), cfg.scale, cfg.window, cfg.ratio,
                f(inp["dO"]))
        rows = [(bi, t) for (lo, hi) in config_ranges(cfg, world, rank)
                for bi in range(cfg.b) for t in range(lo, hi)]
        dq_part, dkv_part, ds_part = orc.attn_bwd(*args, rows=rows)
        dkv = torch.from_numpy(dkv_part)
        dsink = torch.from_numpy(ds_part)
        allreduce_grads(dkv, dsink)
        if rank == 0:
            dq_full, dkv_full, ds_full = orc.attn_bwd(*args)
            out["dkv_err"] = float(np.abs(dkv.numpy() - dkv_full).max())
            out["dsink_err"] = float(np.abs(dsink.numpy() - ds_full).max())
            out["dkv_max"] = float(np.abs(dkv_full).max())
        # a rank's dq rows are its share of the full dq
        dq_full = orc.attn_bwd(*args)[0]
        out[f"dq_err{rank}"] = float(max(np.abs(dq_part[n] - dq_full[bi, t]).max()
                                         for n, (bi, t) in enumerate(rows)))
        out[f"rows{rank}"] = len(rows)
        # a rank-dependent "step time": the job takes the slowest
        out[f"t{rank}"] = bench.max_over_ranks(1.0 + rank, world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_row_split_reduces_to_the_whole_layer():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res["rows0"] + res["rows1"] == 256
    assert res["dkv_err"] <= 1e-12 * max(1.0, res["dkv_max"]), res
    assert res["dsink_err"] <= 1e-12, res
    assert res["dq_err0"] == 0.0 and res["dq_err1"] == 0.0
    assert res["t0"] == res["t1"] == 2.0               # max over ranks
