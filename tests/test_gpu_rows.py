"""GPU parity of the row-range calls (csa_indexer_topk_rows,
csa_attn_fwd_rows, csa_attn_bwd_rows) that split one layer by query rows
across GPUs.

One GPU plays the ranks one after the other: every rank's rows go through the
row-range calls, and the ranks' dKV / dsink contributions are summed (here by
accumulating into one buffer, across GPUs by one all-reduce).  The result
must equal the whole-layer calls: the indexer rows and the forward and dq rows
bit for bit (the ranges start on multiples of 8 rows, so the tensor-core
kernels see the same query blocks), dKV and dsink up to the order of the fp32
sums.  The whole-layer calls are checked against the fp64 oracle in
test_gpu_parity.py; the sum is also checked against the oracle here.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
from compressed_sparse_attention_sum_gb300.shard import config_ranges
from oracle import csa_oracle as orc
from paritylib import TOL, f64, maxabs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    csa.load_library()
    yield
    assert csa.csa_get_device_status() == 0


CASES = {
    "csa4_bf16": CONFIGS["csa4_bf16"],                                   # tcgen05 kernels
    "prod_small": CONFIGS["prod_bf16"].with_(name="prod_small", sq=512, b=1, H=16),  # d=512
    "prod_tc": CONFIGS["prod_bf16"].with_(name="prod_tc", sq=264, b=2),   # tcgen05, d=512 H=64
    "hca_small": CONFIGS["hca_bf16"].with_(name="hca_small", sq=2048, b=2),      # dense lists
    "tiny_fp32": CONFIGS["tiny_fp32"],                                   # CUDA-core fp32
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("world", [2, 3])
def test_row_ranges_reproduce_the_whole_layer(name, world):
    cfg = CASES[name]
    x = {k: v.cuda() for k, v in make_inputs(cfg).items()}
    b, sq, d, n_c, H = cfg.b, cfg.sq, cfg.d, cfg.n_c, cfg.H
    kv_full = torch.empty(b, sq + n_c, d, dtype=cfg.torch_dtype, device="cuda")
    kv_full[:, :sq] = x["kv_raw"]
    csa.csa_compress(kv_full[:, :sq], x["score"], cfg.ratio, out=kv_full[:, sq:])
    ranges = [config_ranges(cfg, world, r) for r in range(world)]
    assert sum(len(r) for r in ranges) >= 2

    # the indexer over the ranks' rows equals the whole-layer indexer
    if cfg.H_I > 0:
        idx_full = csa.csa_indexer_topk(x["q_I"], x["k_I"], x["w"], cfg.topk, cfg.ratio)
        idx_rows = torch.full_like(idx_full, -7)
        for rr in ranges:
            for r in rr:
                csa.csa_indexer_topk(x["q_I"], x["k_I"], x["w"], cfg.topk, cfg.ratio,
                                     out_idx=idx_rows, rows=r)
        assert torch.equal(idx_rows, idx_full)
    idx = x["idx"] if "idx" in x else idx_full

    O, L = csa.csa_attn_fwd(x["q"], kv_full, idx, x["sink"], cfg.scale, cfg.ratio, cfg.window)
    dq, dkv, dsink = csa.csa_attn_bwd(x["q"], kv_full, idx, x["sink"], cfg.scale, cfg.ratio,
                                      cfg.window, O, L, x["dO"])
    O_r = torch.full_like(O, float("nan"))
    L_r = torch.full_like(L, float("nan"))
    dq_r = torch.full_like(dq, float("nan"))
    dkv_r = torch.full_like(dkv, float("nan"))
    ds_r = torch.full_like(dsink, float("nan"))
    for rr in ranges:
        for r in rr:
            csa.csa_attn_fwd(x["q"], kv_full, idx, x["sink"], cfg.scale, cfg.ratio, cfg.window,
                             out=O_r, lse=L_r, rows=r)
    first = True
    for rr in ranges:                      # every rank's contributions summed
        for r in rr:
            csa.csa_attn_bwd(x["q"], kv_full, idx, x["sink"], cfg.scale, cfg.ratio, cfg.window,
                             O_r, L_r, x["dO"], dq=dq_r, dkv=dkv_r, dsink=ds_r, rows=r,
                             accumulate=not first)
            first = False
    torch.cuda.synchronize()
    assert torch.equal(O_r, O) and torch.equal(L_r, L) and torch.equal(dq_r, dq)
    scale_kv = max(1.0, float(dkv.abs().max()))
    assert float((dkv_r - dkv).abs().max()) <= 1e-5 * scale_kv
    assert float((ds_r - dsink).abs().max()) <= 1e-5 * max(1.0, float(dsink.abs().max()))
    # and the summed gradients against the oracle
    _, dkv_ref, ds_ref = orc.attn_bwd(f64(x["q"]), f64(kv_full), idx.cpu().numpy(),
                                      f64(x["sink"]), cfg.scale, cfg.window, cfg.ratio,
                                      f64(x["dO"]))
    tol = TOL[cfg.dtype]
    assert maxabs(f64(dkv_r), dkv_ref) <= tol and maxabs(f64(ds_r), ds_ref) <= tol


def test_row_range_arguments_are_checked():
    cfg = CONFIGS["tiny_fp32"]
    x = {k: v.cuda() for k, v in make_inputs(cfg, parts=("attn",)).items()}
    kv = torch.zeros(cfg.b, cfg.sq + cfg.n_c, cfg.d, device="cuda")
    idx = torch.zeros(cfg.b, cfg.sq, cfg.K, dtype=torch.int32, device="cuda")
    for bad in ((0, 0), (-8, 8), (8, cfg.sq + 8), (16, 8)):
        with pytest.raises(csa.CSAError):
            csa.csa_attn_fwd(x["q"], kv, idx, x["sink"], cfg.scale, cfg.ratio, cfg.window,
                             rows=bad)
