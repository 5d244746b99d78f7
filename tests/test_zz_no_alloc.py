"""GPU test of csa_indexer_topk_noalloc, the indexer entry point for callers
that cannot allocate device memory (a plugin inside a framework that owns the
device memory, a serving loop that must not call cudaMalloc, a C caller with
no spare buffer).  Instead of a caller workspace it keeps its score rows in a
fixed array of the library's own device memory.

The new entry point is called through the C ABI (ctypes) and its output is
compared with that of csa_indexer_topk, which takes a caller workspace, on the
same inputs, over two calls in a row: the array keeps the previous call's
contents, so the second call also shows that nothing stale leaks into a
result.  This file is collected last so that a run stopping at the first
failure has run every other test already; it also passes on its own in a
fresh process.
"""
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import build, csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

CSA_ERR_WORKSPACE = 4
SCRATCH_BYTES = 16 << 20   # CSA_NOALLOC_SCRATCH_BYTES in include/csa.h


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    return csa.load_library()


def _noalloc(lib, q_I, k_I, w, topk, ratio):
    b, sq, H_I, d_I = q_I.shape
    n_c = k_I.shape[1]
    K = min(topk, n_c)
    idx = torch.full((b, sq, K), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((b, sq, K), float("nan"), dtype=torch.float32, device="cuda")
    dt = 1 if q_I.dtype == torch.bfloat16 else 0
    st = lib.csa_indexer_topk_noalloc(q_I.data_ptr(), k_I.data_ptr(), w.data_ptr(), idx.data_ptr(),
                                      sc.data_ptr(), b, sq, n_c, H_I, d_I, ratio, topk, dt,
                                      torch.cuda.current_stream().cuda_stream)
    return st, idx, sc


def _same_as_workspace_call(lib, q_I, k_I, w, topk, ratio):
    ref_idx, ref_sc = csa.csa_indexer_topk(q_I, k_I, w, topk, ratio, return_scores=True)
    st, idx, sc = _noalloc(lib, q_I, k_I, w, topk, ratio)
    torch.cuda.synchronize()
    assert st == 0, lib.csa_status_string(st)
    assert torch.equal(idx, ref_idx)
    tol = 1e-3 * torch.clamp(ref_sc.abs(), min=1.0)
    assert bool(((sc - ref_sc).abs() <= tol).all())


def _case(name, **over):
    cfg = CONFIGS[name].with_(**over)
    inp = make_inputs(cfg, parts=("indexer",))
    return cfg, inp["q_I"].cuda(), inp["k_I"].cuda(), inp["w"].cuda()


@pytest.mark.parametrize("name,over", [
    ("csa4_bf16", {}),                                                 # one chunk, tensor cores
    ("csa4_bf16", dict(sq=16384, ratio=2, H_I=4, d_I=64, topk=64)),   # 32 chunks of 512 rows
    ("tiny_fp32", {}),                                                 # CUDA-core score kernel
])
def test_noalloc_matches_workspace_entry_point_twice(lib, name, over):
    cfg, q_I, k_I, w = _case(name, **over)
    # first call, then a second call in a row on other inputs
    _same_as_workspace_call(lib, q_I, k_I, w, cfg.topk, cfg.ratio)
    _same_as_workspace_call(lib, q_I.flip(1).contiguous(), k_I, -w, cfg.topk, cfg.ratio)
    assert csa.csa_get_device_status() == 0


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    b, n_c = 8, 16384               # smallest chunk: 8 * 128 rows * 16384 * 4 B = 64 MiB
    assert b * 128 * n_c * 4 > SCRATCH_BYTES
    sq, H_I, d_I = n_c, 1, 64
    q_I = torch.zeros(1, dtype=torch.bfloat16, device="cuda")   # never read
    idx = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    st = lib.csa_indexer_topk_noalloc(q_I.data_ptr(), q_I.data_ptr(), idx.data_ptr(),
                                      idx.data_ptr(), None, b, sq, n_c, H_I, d_I, 1, 16, 1,
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == CSA_ERR_WORKSPACE
    assert bool((idx == -7).all())
