"""Failure-detection paths on the GPU, exercised without faulting it.

Every device wait of the library is bounded (about one second of wall time):
a wait that gives up records CSA_ERR_TIMEOUT and a site code in the device
status word, its CTA frees its tensor memory and returns, and the context
stays usable.  Device checks record CSA_ERR_DEVICE_CHECK the same way.  The
test hook csa_debug_arm_fault makes the tensor-core forward (a) never request
its Q tile, so that the wait for it runs out with no copy or MMA in flight,
or (b) lower its union-size limit so that the check trips.  After each case
the hook is disarmed and the same call must match the oracle again.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
from oracle import csa_oracle as orc
from paritylib import TOL, f64, maxabs

pytestmark = pytest.mark.gpu

CSA_ERR_TIMEOUT, CSA_ERR_DEVICE_CHECK = 5, 6
SITE_FWD_Q, SITE_FWD_UNION = 0x21, 0x25


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    csa.load_library()
    csa.csa_get_device_status()
    yield
    csa.csa_debug_arm_fault(0)
    assert csa.csa_get_device_status() == 0


def _small_layer():
    """A small bf16 layer on the tensor-core forward (H=32, d=128: 4 queries
    per CTA, 64 CTAs, one wave)."""
    cfg = CONFIGS["tiny_fp32"].with_(name="tiny_tc", dtype="bf16", H=32, d=128)
    inp = make_inputs(cfg, parts=("compress", "attn"))
    kv_c = orc.compress(f64(inp["kv_raw"]), f64(inp["score"]), cfg.ratio, out_dtype="bf16")
    kv_full = torch.from_numpy(np.concatenate([f64(inp["kv_raw"]), kv_c], 1)).to(torch.bfloat16)
    g = torch.Generator().manual_seed(5)
    idx = torch.randint(-1, cfg.n_c, (cfg.b, cfg.sq, cfg.K), generator=g, dtype=torch.int32)
    return cfg, inp["q"], kv_full, idx, inp["sink"]


def _fwd(cfg, q, kv, idx, sink):
    O, L = csa.csa_attn_fwd(q.cuda(), kv.cuda(), idx.cuda(), sink.cuda(), cfg.scale, cfg.ratio,
                            cfg.window)
    return O, L


def _check_correct(cfg, q, kv, idx, sink):
    O, L = _fwd(cfg, q, kv, idx, sink)
    assert csa.csa_get_device_status(with_site=True) == (0, 0)
    O_ref, L_ref = orc.attn_fwd(f64(q), f64(kv), idx.numpy(), f64(sink), cfg.scale, cfg.window,
                                cfg.ratio)
    assert maxabs(f64(O), O_ref) <= TOL["bf16"]
    assert maxabs(f64(L), L_ref) <= TOL["bf16"]


@pytest.mark.parametrize("site,code", [(SITE_FWD_Q, CSA_ERR_TIMEOUT),
                                       (SITE_FWD_UNION, CSA_ERR_DEVICE_CHECK)])
def test_forward_failure_is_reported_and_the_context_survives(site, code):
    cfg, q, kv, idx, sink = _small_layer()
    _check_correct(cfg, q, kv, idx, sink)
    csa.csa_debug_arm_fault(site)
    try:
        _fwd(cfg, q, kv, idx, sink)
        got = csa.csa_get_device_status(with_site=True)
    finally:
        csa.csa_debug_arm_fault(0)
    assert got == (code, site), got
    # the status word was cleared by the read, and the next call is correct
    assert csa.csa_get_device_status(with_site=True) == (0, 0)
    _check_correct(cfg, q, kv, idx, sink)
