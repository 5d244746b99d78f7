"""GPU parity of the overlapping compressor (csa_compress_overlap and its
backward, coff = 2: each compressed entry pools its own block and the one
before it) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, CONFIG_ORDER, make_inputs
from oracle import csa_oracle as orc
from paritylib import TOL, f64, maxabs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    yield
    assert csa.csa_get_device_status() == 0


def _dt(name):
    return torch.float32 if name == "fp32" else torch.bfloat16


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_overlap_layer_layout(name):
    """The workloads' KV and scores, written into and read from kv_full /
    dkv_full as the layer does; forward and backward against the oracle."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("compress",))
    b, sq, d, n_c = cfg.b, cfg.sq, cfg.d, cfg.n_c
    kv_full = torch.full((b, sq + n_c, d), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    kv_full[:, :sq] = inp["kv_raw"].cuda()
    score = inp["score"].cuda()
    csa.csa_compress_overlap(kv_full[:, :sq], score, cfg.ratio, 2, out=kv_full[:, sq:])
    g = torch.Generator().manual_seed(17)
    dout = torch.randn(b, n_c, d, generator=g)
    pre = torch.randn(b, sq, d, generator=g)
    dkv_full = torch.cat([pre, dout], dim=1).cuda()
    dscore = csa.csa_compress_overlap_bwd(kv_full[:, :sq], score, cfg.ratio, 2, dkv_full[:, sq:],
                                          dkv_full[:, :sq])
    torch.cuda.synchronize()
    tol = TOL[cfg.dtype]
    kv64, s64 = f64(inp["kv_raw"]), f64(inp["score"])
    got = f64(kv_full[:, sq:])
    assert np.all(np.isfinite(got))
    assert maxabs(got, orc.compress(kv64, s64, cfg.ratio, coff=2)) <= tol
    ref_dkv, ref_ds = orc.compress_bwd(kv64, s64, cfg.ratio, f64(dout), coff=2)
    e_kv = maxabs(f64(dkv_full[:, :sq]) - f64(pre), ref_dkv)
    e_s = maxabs(f64(dscore), ref_ds)
    assert e_kv <= tol and e_s <= tol, (e_kv, e_s)
    assert torch.equal(dkv_full[:, sq:].cpu(), dout)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("score_width", [1, "d"])
@pytest.mark.parametrize("ratio", [1, 4, 5])
def test_overlap_ragged_and_scalar_score(dtype, score_width, ratio):
    b, sq, d = 2, 43, 24                   # sq % ratio tokens past the last block
    g = torch.Generator().manual_seed(18)
    sw = d if score_width == "d" else 1
    kv = torch.randn(b, sq, d, generator=g).to(_dt(dtype))
    score = (torch.randn(b, sq, sw, generator=g) * 3).to(_dt(dtype))
    dout = torch.randn(b, sq // ratio, d, generator=g)
    out = csa.csa_compress_overlap(kv.cuda(), score.cuda(), ratio, 2)
    dkv = torch.zeros(b, sq, d, device="cuda")
    dscore = csa.csa_compress_overlap_bwd(kv.cuda(), score.cuda(), ratio, 2, dout.cuda(), dkv)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    assert maxabs(f64(out), orc.compress(f64(kv), f64(score), ratio, coff=2)) <= tol
    ref_dkv, ref_ds = orc.compress_bwd(f64(kv), f64(score), ratio, f64(dout), coff=2)
    assert maxabs(f64(dkv), ref_dkv) <= tol
    assert maxabs(f64(dscore), ref_ds) <= tol
    tail = (sq // ratio) * ratio
    assert torch.all(dkv[:, tail:] == 0) and torch.all(dscore[:, tail:] == 0)


def test_overlap_coff1_is_compress():
    """coff = 1 through the overlap entry points is bit-identical to
    csa_compress / csa_compress_bwd."""
    g = torch.Generator().manual_seed(19)
    b, sq, d, ratio = 1, 64, 32, 4
    kv = torch.randn(b, sq, d, generator=g).to(torch.bfloat16).cuda()
    score = torch.randn(b, sq, d, generator=g).to(torch.bfloat16).cuda()
    dout = torch.randn(b, sq // ratio, d, generator=g).cuda()
    assert torch.equal(csa.csa_compress_overlap(kv, score, ratio, 1),
                       csa.csa_compress(kv, score, ratio))
    dk1, dk2 = torch.zeros(b, sq, d, device="cuda"), torch.zeros(b, sq, d, device="cuda")
    ds1 = csa.csa_compress_overlap_bwd(kv, score, ratio, 1, dout, dk1)
    ds2 = csa.csa_compress_bwd(kv, score, ratio, dout, dk2)
    assert torch.equal(dk1, dk2) and torch.equal(ds1, ds2)


def test_overlap_rejects_unsupported_coff():
    kv = torch.zeros(1, 16, 8, device="cuda")
    with pytest.raises(csa.CSAError):
        csa.csa_compress_overlap(kv, kv, 4, 3)
    with pytest.raises(csa.CSAError):
        csa.csa_compress_overlap(kv, kv, 4, 0)
