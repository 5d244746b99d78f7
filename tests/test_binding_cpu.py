"""The Python binding has no CPU path: every compute call rejects host
tensors before anything runs (on a machine without a GPU as on one with)."""
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa

bf = torch.bfloat16
f32 = torch.float32
i32 = torch.int32


def _t(*shape, dtype=bf):
    return torch.zeros(*shape, dtype=dtype)


CALLS = {
    "csa_compress": lambda: csa.csa_compress(_t(1, 8, 8), _t(1, 8, 8), 4),
    "csa_compress_bwd": lambda: csa.csa_compress_bwd(_t(1, 8, 8), _t(1, 8, 8), 4,
                                                     _t(1, 2, 8, dtype=f32), _t(1, 8, 8, dtype=f32)),
    "csa_compress_overlap": lambda: csa.csa_compress_overlap(_t(1, 8, 8), _t(1, 8, 8), 4, 2),
    "csa_compress_overlap_bwd": lambda: csa.csa_compress_overlap_bwd(
        _t(1, 8, 8), _t(1, 8, 8), 4, 2, _t(1, 2, 8, dtype=f32), _t(1, 8, 8, dtype=f32)),
    "csa_compress_norm_rope": lambda: csa.csa_compress_norm_rope(
        _t(1, 8, 8), _t(1, 8, 8), 4, _t(8, dtype=f32), 1e-6, 4),
    "csa_compress_norm_rope_bwd": lambda: csa.csa_compress_norm_rope_bwd(
        _t(1, 8, 8), _t(1, 8, 8), 4, _t(8, dtype=f32), 1e-6, 4, 40000.0,
        _t(1, 2, 8, dtype=f32), _t(1, 8, 8, dtype=f32)),
    "csa_indexer_topk": lambda: csa.csa_indexer_topk(_t(1, 8, 2, 16), _t(1, 2, 16),
                                                     _t(1, 8, 2, dtype=f32), 2, 4),
    "csa_quantize_e4m3": lambda: csa.csa_quantize_e4m3(_t(4, 16)),
    "csa_indexer_topk_fp8": lambda: csa.csa_indexer_topk_fp8(
        _t(1, 8, 2, 16, dtype=torch.uint8), _t(1, 8, 2, dtype=f32), _t(1, 2, 16, dtype=torch.uint8),
        _t(1, 2, dtype=f32), _t(1, 8, 2, dtype=f32), 2, 4),
    "csa_attn_fwd": lambda: csa.csa_attn_fwd(_t(1, 8, 2, 16), _t(1, 10, 16), _t(1, 8, 2, dtype=i32),
                                             None, 0.25, 4, 4),
    "csa_attn_bwd": lambda: csa.csa_attn_bwd(_t(1, 8, 2, 16), _t(1, 10, 16), _t(1, 8, 2, dtype=i32),
                                             None, 0.25, 4, 4, _t(1, 8, 2, 16),
                                             _t(1, 8, 2, dtype=f32), _t(1, 8, 2, 16)),
    "csa_indexer_topk_rows": lambda: csa.csa_indexer_topk(_t(1, 8, 2, 16), _t(1, 2, 16),
                                                          _t(1, 8, 2, dtype=f32), 2, 4,
                                                          rows=(0, 4)),
    "csa_attn_fwd_rows": lambda: csa.csa_attn_fwd(_t(1, 8, 2, 16), _t(1, 10, 16),
                                                  _t(1, 8, 2, dtype=i32), None, 0.25, 4, 4,
                                                  rows=(0, 4)),
    "csa_attn_bwd_rows": lambda: csa.csa_attn_bwd(_t(1, 8, 2, 16), _t(1, 10, 16),
                                                  _t(1, 8, 2, dtype=i32), None, 0.25, 4, 4,
                                                  _t(1, 8, 2, 16), _t(1, 8, 2, dtype=f32),
                                                  _t(1, 8, 2, 16), rows=(4, 8), accumulate=True),
    "csa_indexer_teacher": lambda: csa.csa_indexer_teacher(_t(1, 8, 2, 16), _t(1, 10, 16),
                                                           _t(1, 8, 2, dtype=i32),
                                                           _t(1, 8, 2, dtype=f32), 0.25, 4),
    "csa_indexer_loss": lambda: csa.csa_indexer_loss(_t(1, 8, 2, 16), _t(1, 2, 16),
                                                     _t(1, 8, 2, dtype=f32), _t(1, 8, 2, dtype=i32),
                                                     _t(1, 8, 2, dtype=f32), 4),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_rejected(name):
    with pytest.raises(ValueError, match="CUDA tensor"):
        CALLS[name]()


def test_every_compute_call_is_covered():
    compute = {n for n in csa.SIGNATURES if not n.endswith(("_size", "_workspace", "_string",
                                                             "_version", "_launches", "_status"))}
    compute.discard("csa_indexer_topk_noalloc")   # C-only entry point (no binding)
    compute.discard("csa_debug_arm_fault")        # test hook, takes no tensors
    assert compute <= set(CALLS), sorted(compute - set(CALLS))
