"""GPU parity of csa_compress_norm_rope and its backward against the fp64
oracle (orc.compress, then orc.kv_norm_rope on the pooled rows rounded to the
storage dtype; orc.kv_norm_rope_bwd, then orc.compress_bwd).

The pooled row is cast to the storage dtype before the norm (the compressor
review's order), so a pooled value that lies next to a bf16 rounding boundary
may round differently on the two sides (fp32 on the GPU, fp64 in the oracle):
one bf16 step, 2^-8 of the value.  The norm weights are drawn in
[0.25, 0.5] so that the normalized rows stay below 2 in magnitude, where that
step and the output's own bf16 step together stay under the 2e-2 bound.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
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


CASES = [
    # workload, rope_dim, score_width, sq override
    ("tiny_fp32", 32, "d", None),
    ("tiny_fp32", 0, 1, 259),                   # no rotation, shared score, ragged tail
    ("debug_bf16", 64, "d", None),
    ("csa4_bf16", 64, "d", None),
    ("csa4_bf16", 128, 1, 4093),                 # every channel rotated, ragged tail
    ("hca_bf16", 64, "d", None),                 # ratio 128
    ("prod_bf16", 64, "d", 2048),                # d = 512
]


@pytest.mark.parametrize("name,rope_dim,sw,sq", CASES)
def test_compress_norm_rope_fwd_bwd(name, rope_dim, sw, sq):
    cfg = CONFIGS[name]
    if sq is not None:
        cfg = cfg.with_(sq=sq, b=1)
    inp = make_inputs(cfg, parts=("compress",))
    b, sq, d, ratio, n_c = cfg.b, cfg.sq, cfg.d, cfg.ratio, cfg.n_c
    g = torch.Generator().manual_seed(21)
    kv = inp["kv_raw"]
    score = inp["score"] if sw == "d" else inp["score"][..., :1].contiguous()
    w = 0.25 + 0.25 * torch.rand(d, generator=g)
    eps, base = 1e-6, 40000.0
    out = csa.csa_compress_norm_rope(kv.cuda(), score.cuda(), ratio, w.cuda(), eps, rope_dim,
                                     base)
    dout = torch.randn(b, n_c, d, generator=g)
    pre = torch.randn(b, sq, d, generator=g)
    dkv = pre.clone().cuda()
    dscore, dw = csa.csa_compress_norm_rope_bwd(kv.cuda(), score.cuda(), ratio, w.cuda(), eps,
                                                rope_dim, base, dout.cuda(), dkv)
    torch.cuda.synchronize()
    tol = TOL[cfg.dtype]
    kv_c = orc.compress(f64(kv), f64(score), ratio, out_dtype=cfg.dtype)
    ref = orc.kv_norm_rope(kv_c, f64(w), eps, rope_dim, base, ratio, out_dtype=cfg.dtype)
    e_out = maxabs(f64(out), ref)
    dx, dw_ref = orc.kv_norm_rope_bwd(kv_c, f64(w), eps, rope_dim, base, ratio, f64(dout))
    dkv_ref, ds_ref = orc.compress_bwd(f64(kv), f64(score), ratio, dx)
    e_dkv = maxabs(f64(dkv) - f64(pre), dkv_ref)
    e_ds = maxabs(f64(dscore), ds_ref)
    e_dw = maxabs(f64(dw), dw_ref)
    dw_scale = max(1.0, float(np.abs(dw_ref).max()))
    print(f"{name} rope {rope_dim} sw {sw}: out {e_out:.2e} dkv {e_dkv:.2e} dscore {e_ds:.2e} "
          f"dweight {e_dw:.2e} (|dweight| max {dw_scale:.1f})")
    assert e_out <= tol and e_dkv <= tol and e_ds <= tol, (e_out, e_dkv, e_ds)
    # dweight sums every row's contribution: the bound is relative to its size
    assert e_dw <= tol * dw_scale, (e_dw, dw_scale)


def test_norm_rope_arguments_are_checked():
    cfg = CONFIGS["tiny_fp32"]
    inp = make_inputs(cfg, parts=("compress",))
    kv, score = inp["kv_raw"].cuda(), inp["score"].cuda()
    w = torch.ones(cfg.d, device="cuda")
    for eps, rd, base in ((-1.0, 0, 1.0), (1e-6, 3, 40000.0), (1e-6, cfg.d + 2, 40000.0),
                          (1e-6, 8, 0.0)):
        with pytest.raises(csa.CSAError):
            csa.csa_compress_norm_rope(kv, score, cfg.ratio, w, eps, rd, base)
