"""The multi-rank host logic of bench.py on two gloo ranks (CPU): each rank
gets its own seeded layer, and the step time of the job is the maximum over
ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
        cfg = bench.rank_config(CONFIGS["tiny_fp32"], rank, world)
        x = make_inputs(cfg, parts=("attn",))["q"]
        sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, x.double().sum().view(1))
        # a rank-dependent "step time": the job takes the slowest
        t = bench.max_over_ranks(1.0 + rank, world)
        dist.barrier()
        out[rank] = (cfg.seed, t, sums[0].item() != sums[1].item())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_independent_layers_and_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] != res[1][0]                      # distinct seeds
    assert res[0][1] == res[1][1] == 2.0               # max over ranks
    assert res[0][2] and res[1][2]                     # distinct inputs
