"""Seeded random configurations against the fp64 oracle, through the C ABI.

Each case draws its own shape from a fixed seed, so that the kernels meet
combinations no hand-written case lists: batch 1-3, a sequence length that
is rarely a multiple of the 128-row tile or of the ratio, every attention
kernel family (tcgen05 at d = 128 with 16, 32 or 64 heads and at d = 512
with 64 heads, warp-level MMA, CUDA-core fp32), ratios from 1 to 16,
windows from 1 past the sequence length, index lists from 1 to 300 entries
with repeated, -1, out-of-range and not-yet-visible entries, with or
without the sink, with or without packed documents.  The attention is
compared element by element (O, LSE, dq, every dkv row, dsink), the
indexer (bf16, fp32 and e4m3 codes) row by row with the tie-aware top-k
comparison, the indexer loss and its gradients element by element.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import packed_doc_ids
from oracle import csa_oracle as orc
from paritylib import TOL, compare_topk_row, f64, maxabs
from test_gpu_train import _check_loss, _messy_idx

pytestmark = pytest.mark.gpu

# (dtype, H, d): the kernel family each selects on a GB300
ATTN_KINDS = [("bf16", 16, 128), ("bf16", 32, 128), ("bf16", 64, 128), ("bf16", 64, 512),
              ("bf16", 6, 64), ("fp32", 4, 64), ("fp32", 3, 32)]
ATTN_SEEDS = list(range(1000, 1056))     # eight draws of each kernel family
IDX_SEEDS = list(range(2000, 2040))
FP8_SEEDS = list(range(3000, 3012))
LOSS_SEEDS = list(range(4000, 4012))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    yield
    assert csa.csa_get_device_status() == 0


def _dt(name):
    return torch.float32 if name == "fp32" else torch.bfloat16


def _attn_case(seed):
    rng = np.random.default_rng(seed)
    dtype, H, d = ATTN_KINDS[seed % len(ATTN_KINDS)]
    ratio = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    b = int(rng.integers(1, 4))
    big = d == 512 or H == 64
    sq = int(rng.integers(max(ratio, 20), 400 if big else 520))
    sq -= sq % ratio if rng.random() < 0.3 else 0          # sometimes a whole number of blocks
    window = int(rng.choice([1, 3, 17, 64, 128, 200, sq + 5]))
    K = int(rng.choice([1, 5, 33, 100, 300]))
    return dict(dtype=dtype, H=H, d=d, ratio=ratio, b=b, sq=sq, window=window, K=K,
                sink=bool(rng.random() < 0.75), docs=bool(rng.random() < 0.3),
                sorted_lists=bool(rng.random() < 0.5))


def _attn_inputs(seed, c):
    g = torch.Generator().manual_seed(seed)
    b, sq, H, d, ratio, K = c["b"], c["sq"], c["H"], c["d"], c["ratio"], c["K"]
    n_c = sq // ratio
    q = torch.randn(b, sq, H, d, generator=g).to(_dt(c["dtype"]))
    kv = torch.randn(b, sq + n_c, d, generator=g).to(_dt(c["dtype"]))
    if c["sorted_lists"]:
        # the indexer's shape of list: ascending visible blocks, then -1
        idx = torch.full((b, sq, K), -1, dtype=torch.int32)
        for bi in range(b):
            for t in range(sq):
                vis = min((t + 1) // ratio, n_c)
                k = min(K, vis)
                if k:
                    sel = torch.randperm(vis, generator=g)[:k].sort().values
                    idx[bi, t, :k] = sel.to(torch.int32)
    else:
        idx = torch.randint(-1, n_c + 2, (b, sq, K), generator=g, dtype=torch.int32)
        if K > 1:
            idx[:, :, 1] = idx[:, :, 0]                 # repeated entries
    snk = torch.randn(H, generator=g) if c["sink"] else None
    dO = torch.randn(b, sq, H, d, generator=g).to(_dt(c["dtype"]))
    doc = (torch.randint(0, 3, (b, sq), generator=g, dtype=torch.int32) if c["docs"] else None)
    return q, kv, idx, snk, dO, doc


@pytest.mark.parametrize("seed", ATTN_SEEDS)
def test_attention_random_configuration(seed):
    c = _attn_case(seed)
    q, kv, idx, snk, dO, doc = _attn_inputs(seed, c)
    b, sq, H, d = q.shape
    ratio, window = c["ratio"], c["window"]
    scale = d ** -0.5
    cu = lambda t: None if t is None else t.cuda()
    O, L = csa.csa_attn_fwd(cu(q), cu(kv), cu(idx), cu(snk), scale, ratio, window,
                            doc_ids=cu(doc))
    # both sides of the backward take the oracle's O (rounded to the storage
    # dtype) and LSE, so that the backward is checked on its own
    sn = None if snk is None else f64(snk)
    dn = None if doc is None else doc.numpy()
    O_ref, L_ref = orc.attn_fwd(f64(q), f64(kv), idx.numpy(), sn, scale, window, ratio,
                                doc_ids=dn)
    O_in = torch.from_numpy(orc.round_to_storage(O_ref, c["dtype"])).to(q.dtype).cuda()
    L_in = torch.from_numpy(L_ref).float().cuda()
    dq, dkv, dsink = csa.csa_attn_bwd(cu(q), cu(kv), cu(idx), cu(snk), scale, ratio, window,
                                      O_in, L_in, cu(dO), doc_ids=cu(doc))
    dq_ref, dkv_ref, ds_ref = orc.attn_bwd(f64(q), f64(kv), idx.numpy(), sn, scale, window,
                                           ratio, f64(dO), doc_ids=dn)
    errs = {"O": maxabs(f64(O), O_ref), "LSE": maxabs(f64(L), L_ref),
            "dq": maxabs(f64(dq), dq_ref), "dkv": maxabs(f64(dkv), dkv_ref)}
    if snk is not None:
        errs["dsink"] = maxabs(f64(dsink), ds_ref)
    assert max(errs.values()) <= TOL[c["dtype"]], (c, errs)
    assert csa.csa_get_device_status() == 0


def _idx_case(seed):
    rng = np.random.default_rng(seed)
    dtype = "fp32" if seed % 4 == 3 else "bf16"
    H_I = int(rng.choice([1, 3, 8, 32, 64]))
    d_I = int(rng.choice([32, 64, 128])) if dtype == "fp32" else int(rng.choice([64, 128]))
    ratio = int(rng.choice([1, 2, 4, 7]))
    b = int(rng.integers(1, 3))
    sq = int(rng.integers(max(ratio, 16), 900))
    topk = int(rng.choice([1, 16, 64, 300]))
    return dict(dtype=dtype, H_I=H_I, d_I=d_I, ratio=ratio, b=b, sq=sq, topk=topk,
                docs=bool(rng.random() < 0.3), scores=bool(rng.random() < 0.5))


@pytest.mark.parametrize("seed", IDX_SEEDS)
def test_indexer_random_configuration(seed):
    c = _idx_case(seed)
    g = torch.Generator().manual_seed(seed)
    b, sq, ratio, topk = c["b"], c["sq"], c["ratio"], c["topk"]
    n_c = sq // ratio
    q_I = torch.randn(b, sq, c["H_I"], c["d_I"], generator=g).to(_dt(c["dtype"]))
    k_I = torch.randn(b, n_c, c["d_I"], generator=g).to(_dt(c["dtype"]))
    w = torch.randn(b, sq, c["H_I"], generator=g) * 0.5
    doc = packed_doc_ids(b, sq, ratio, min(3, n_c), seed=seed) if c["docs"] else None
    out = csa.csa_indexer_topk(q_I.cuda(), k_I.cuda(), w.cuda(), topk, ratio,
                               return_scores=c["scores"],
                               doc_ids=None if doc is None else doc.cuda())
    idx = (out[0] if c["scores"] else out).cpu().numpy()
    assert csa.csa_get_device_status() == 0
    K = min(topk, n_c)
    I = orc.indexer_scores(f64(q_I), f64(k_I), f64(w), ratio,
                           doc_ids=None if doc is None else doc.numpy())
    for bi in range(b):
        for t in range(sq):
            row = I[bi, t]
            cand = np.flatnonzero(np.isfinite(row))
            k = min(K, cand.size)
            sel = idx[bi, t, :k]
            assert np.all(idx[bi, t, k:] == -1), (c, bi, t)
            pos = np.searchsorted(cand, sel)
            assert np.all(pos < cand.size) and np.array_equal(cand[np.minimum(pos, cand.size - 1)],
                                                              sel), (c, bi, t)
            full = np.concatenate([pos, idx[bi, t, k:]]).astype(np.int32)
            ok, _ = compare_topk_row(full, row[cand], K)
            assert ok, (c, bi, t, idx[bi, t, :8])
    if c["scores"]:
        sc = out[1].cpu().numpy()
        for bi in range(b):
            for t in range(sq):
                k = int((idx[bi, t] >= 0).sum())
                ref = I[bi, t, idx[bi, t, :k]]
                got = sc[bi, t, :k]
                tol = 1e-3 * np.maximum(np.abs(ref), 1.0) if c["dtype"] == "fp32" else \
                    2e-2 * np.maximum(np.abs(ref), 1.0)
                assert np.all(np.abs(got - ref) <= tol), (c, bi, t)
                assert np.all(sc[bi, t, k:] == 0.0), (c, bi, t)


def _finite_row_ok(gpu_row, I_row, K):
    """compare_topk_row over a row's selectable (finite) entries, which need
    not be a prefix when documents are packed."""
    cand = np.flatnonzero(np.isfinite(I_row))
    k = min(K, cand.size)
    sel = gpu_row[:k]
    if np.any(gpu_row[k:] != -1):
        return False
    pos = np.searchsorted(cand, sel)
    if np.any(pos >= cand.size) or np.any(cand[np.minimum(pos, cand.size - 1)] != sel):
        return False
    full = np.concatenate([pos, gpu_row[k:]]).astype(np.int32)
    return compare_topk_row(full, I_row[cand], K)[0]


@pytest.mark.parametrize("seed", FP8_SEEDS)
def test_indexer_fp8_random_configuration(seed):
    rng = np.random.default_rng(seed)
    H_I = int(rng.choice([1, 4, 16, 64]))
    d_I = int(rng.choice([128, 256, 48]))          # 48: the CUDA-core kernel
    ratio = int(rng.choice([1, 2, 4, 8]))
    b = int(rng.integers(1, 3))
    sq = int(rng.integers(max(ratio, 24), 800))
    topk = int(rng.choice([1, 24, 128, 300]))
    n_c = sq // ratio
    docs = bool(rng.random() < 0.3)
    g = torch.Generator().manual_seed(seed)
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(torch.bfloat16)
    k_I = torch.randn(b, n_c, d_I, generator=g).to(torch.bfloat16)
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    doc = packed_doc_ids(b, sq, ratio, min(3, n_c), seed=seed) if docs else None
    q8, qs = csa.csa_quantize_e4m3(q_I.cuda())
    k8, ks = csa.csa_quantize_e4m3(k_I.cuda())
    rq, rqs = orc.quantize_rows_e4m3(q_I.float().numpy())
    rk, rks = orc.quantize_rows_e4m3(k_I.float().numpy())
    idx, sc = csa.csa_indexer_topk_fp8(q8, qs, k8, ks, w.cuda(), topk, ratio, return_scores=True,
                                       doc_ids=None if doc is None else doc.cuda())
    assert csa.csa_get_device_status() == 0
    I = orc.indexer_scores_fp8(rq, rqs, rk, rks, w.numpy(), ratio,
                               doc_ids=None if doc is None else doc.numpy())
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    K = min(topk, n_c)
    cfg = (H_I, d_I, ratio, b, sq, topk, docs)
    for bi in range(b):
        for t in range(sq):
            assert _finite_row_ok(idx[bi, t], I[bi, t], K), (cfg, bi, t, idx[bi, t, :8])
            k = int((idx[bi, t] >= 0).sum())
            if k:
                ref = I[bi, t][idx[bi, t, :k]]
                assert np.max(np.abs(sc[bi, t, :k] - ref)) <= 1e-5 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("seed", LOSS_SEEDS)
def test_indexer_loss_random_configuration(seed):
    rng = np.random.default_rng(seed)
    # bf16 with d_I 128 and 32 or 64 heads: the tcgen05 kernel; the others
    # the warp-MMA and CUDA-core kernels
    dtype, H_I, d_I = [("bf16", 64, 128), ("bf16", 32, 128), ("bf16", 64, 128),
                       ("bf16", 12, 64), ("fp32", 5, 32)][seed % 5]
    ratio = int(rng.choice([1, 2, 4]))
    b = int(rng.integers(1, 3))
    sq = int(rng.integers(max(ratio, 12), 700))
    n_c = sq // ratio
    K = int(rng.choice([1, 16, 64, 200]))
    g = torch.Generator().manual_seed(seed)
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(_dt(dtype))
    k_I = torch.randn(b, n_c, d_I, generator=g).to(_dt(dtype))
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    idx = _messy_idx(g, b, sq, n_c, K)
    target = torch.rand(b, sq, K, generator=g)
    target[:, 7 % sq] = 0.0                  # a row without target mass
    target = target / target.sum(-1, keepdim=True).clamp_min(1e-30)
    loss, dq, dk, dw = _check_loss(q_I, k_I, w, idx, target, ratio, dtype)
    assert csa.csa_get_device_status() == 0
    r = 7 % sq
    assert torch.all(dq[:, r] == 0) and torch.all(dw[:, r] == 0) and torch.all(loss[:, r] == 0)
