"""GPU parity of the FP8 indexer against the fp64 oracle, through the C ABI:
per-row e4m3 quantization (csa_quantize_e4m3, bit-exact: every step is a
correctly rounded fp32 operation) and the indexer top-k on the codes
(csa_indexer_topk_fp8), tcgen05 kind::f8f6f4 and CUDA-core paths.

The oracle quantizes the same bf16 / fp32 inputs itself; nothing the GPU
computes is fed back to it.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs, packed_doc_ids
from oracle import csa_oracle as orc
from paritylib import compare_topk_row, f64

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


def _decode(codes: torch.Tensor) -> np.ndarray:
    """uint8 e4m3 bit patterns -> their values (torch's exact float8 decode)."""
    return codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _special_rows(d):
    """Rows that pin the rounding: amax 448 makes the multiplier exactly 1, so
    the codes are the e4m3 roundings of the inputs themselves (ties to even
    in the normal and the subnormal range, saturation never needed); an
    all-zero row; a row of one tiny value; a row with a huge value."""
    r = np.zeros((4, d), np.float32)
    ties = [448.0, 1.0625, 1.1875, -1.0625, 2.125, 2.0 ** -10, 3 * 2.0 ** -10, -5 * 2.0 ** -10,
            17.0, 19.0, -0.0]
    r[0, :len(ties)] = ties[:d]
    r[0, 0] = 448.0
    # r[1] stays zero
    r[2, d // 2] = 1e-30
    r[3, :] = np.linspace(-1, 1, d, dtype=np.float32)
    r[3, 1] = 3e4
    return r


@pytest.mark.parametrize("dtype,rows,d", [
    ("bf16", 1000, 128),
    ("fp32", 333, 64),
    ("bf16", 77, 8),
    ("fp32", 50, 136),      # not a multiple of 32 lanes x 8
])
def test_quantize_bit_exact(dtype, rows, d):
    g = torch.Generator().manual_seed(61)
    x = torch.randn(rows, d, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3)
    x[:4] = torch.from_numpy(_special_rows(d))
    x = x.to(_dt(dtype))
    codes, scale = csa.csa_quantize_e4m3(x.cuda())
    ref_codes, ref_scale = orc.quantize_rows_e4m3(x.float().numpy())
    assert codes.shape == x.shape and codes.dtype == torch.uint8
    assert np.array_equal(_decode(codes), ref_codes)
    assert np.array_equal(scale.cpu().numpy(), ref_scale)
    assert scale[1].item() == 0 and torch.all(codes[1] == 0)


def test_quantize_indexer_layout():
    """q_I [b, sq, H_I, d_I] quantizes per (b, t, h) row; scales [b, sq, H_I]."""
    cfg = CONFIGS["debug_bf16"]
    inp = make_inputs(cfg, parts=("indexer",))
    codes, scale = csa.csa_quantize_e4m3(inp["q_I"].cuda())
    ref_codes, ref_scale = orc.quantize_rows_e4m3(inp["q_I"].float().numpy())
    assert scale.shape == inp["q_I"].shape[:-1]
    assert np.array_equal(_decode(codes), ref_codes)
    assert np.array_equal(scale.cpu().numpy(), ref_scale)


def _quantize_both(q_I, k_I):
    q8, qs = csa.csa_quantize_e4m3(q_I.cuda())
    k8, ks = csa.csa_quantize_e4m3(k_I.cuda())
    rq, rqs = orc.quantize_rows_e4m3(q_I.float().numpy())
    rk, rks = orc.quantize_rows_e4m3(k_I.float().numpy())
    return (q8, qs, k8, ks), (rq, rqs, rk, rks)


def _check_rows(idx, sc, I, K, rows):
    exact = 0
    for bi, t in rows:
        ok, ex = compare_topk_row_finite(idx[bi, t], I[bi, t], K)
        assert ok, (bi, t, idx[bi, t][:8])
        exact += ex
        k = int(np.sum(idx[bi, t] >= 0))
        if k:
            ref = I[bi, t][idx[bi, t][:k]]
            assert np.max(np.abs(sc[bi, t, :k] - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
    return exact


def compare_topk_row_finite(gpu_row, I_row, K):
    """compare_topk_row over the finite (selectable) entries of a row, which
    need not be a prefix when documents are packed."""
    cand = np.flatnonzero(np.isfinite(I_row))
    k = min(K, cand.size)
    sel = gpu_row[:k]
    if np.any(gpu_row[k:] != -1):
        return False, True
    pos = np.searchsorted(cand, sel)
    if np.any(pos >= cand.size) or np.any(cand[np.minimum(pos, cand.size - 1)] != sel):
        return False, True
    full = np.concatenate([pos, gpu_row[k:]]).astype(np.int32)
    return compare_topk_row(full, I_row[cand], K)


@pytest.mark.parametrize("H_I,d_I,cores,docs", [
    (4, 128, False, False),     # tcgen05 kind::f8f6f4, one 128-byte K block
    (8, 256, False, True),      # two K blocks, packed documents
    (3, 128, True, False),      # CUDA-core kernel on request
    (5, 48, False, False),      # CUDA-core kernel: d_I outside the tensor-core set
])
def test_indexer_fp8_small(H_I, d_I, cores, docs, monkeypatch):
    if cores:
        monkeypatch.setenv("CSA_INDEXER_CUDA_CORES", "1")
    b, sq, ratio, topk = 2, 600, 4, 24
    g = torch.Generator().manual_seed(62)
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(torch.bfloat16)
    k_I = torch.randn(b, sq // ratio, d_I, generator=g).to(torch.bfloat16)
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    doc = packed_doc_ids(b, sq, ratio, 5) if docs else None
    (q8, qs, k8, ks), (rq, rqs, rk, rks) = _quantize_both(q_I, k_I)
    idx, sc = csa.csa_indexer_topk_fp8(q8, qs, k8, ks, w.cuda(), topk, ratio, return_scores=True,
                                       doc_ids=None if doc is None else doc.cuda())
    I = orc.indexer_scores_fp8(rq, rqs, rk, rks, w.numpy(), ratio,
                               doc_ids=None if doc is None else doc.numpy())
    rows = [(bi, t) for bi in range(b) for t in range(sq)]
    exact = _check_rows(idx.cpu().numpy(), sc.cpu().numpy(), I, topk, rows)
    assert exact > len(rows) // 2


def test_indexer_fp8_csa4():
    """The CSA-4 layer's indexer (H_I 64, d_I 128, n_c 1024, K 512) on e4m3
    codes: every row against the oracle's FP8 scores."""
    cfg = CONFIGS["csa4_bf16"]
    inp = make_inputs(cfg, parts=("indexer",))
    (q8, qs, k8, ks), (rq, rqs, rk, rks) = _quantize_both(inp["q_I"], inp["k_I"])
    idx, sc = csa.csa_indexer_topk_fp8(q8, qs, k8, ks, inp["w"].cuda(), cfg.topk, cfg.ratio,
                                       return_scores=True)
    I = orc.indexer_scores_fp8(rq, rqs, rk, rks, inp["w"].numpy(), cfg.ratio)
    rows = [(0, t) for t in range(cfg.sq)]
    _check_rows(idx.cpu().numpy(), sc.cpu().numpy(), I, cfg.K, rows)


def test_indexer_fp8_chunked_workspace():
    """A workspace of one 128-row chunk gives the same result as the default."""
    b, sq, ratio, topk, H_I, d_I = 1, 1000, 4, 40, 6, 128
    g = torch.Generator().manual_seed(63)
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(torch.bfloat16).cuda()
    k_I = torch.randn(b, sq // ratio, d_I, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(b, sq, H_I, generator=g) * 0.5).cuda()
    q8, qs = csa.csa_quantize_e4m3(q_I)
    k8, ks = csa.csa_quantize_e4m3(k_I)
    full = csa.csa_indexer_topk_fp8(q8, qs, k8, ks, w, topk, ratio)
    lib = csa.load_library()
    small = torch.empty(lib.csa_indexer_topk_min_workspace(b, sq // ratio), dtype=torch.uint8,
                        device="cuda")
    chunked = csa.csa_indexer_topk_fp8(q8, qs, k8, ks, w, topk, ratio, workspace=small)
    assert torch.equal(full, chunked)
