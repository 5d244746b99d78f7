"""GPU parity of packed-document isolation (doc_ids) against the fp64 oracle,
through the C ABI.

"Refactor Deepseek v4 to use Attention Gym's Compressed Sparse Attention":
the window branch keeps key k for query t only when doc_ids[k] == doc_ids[t];
block j belongs to doc_ids[j*ratio] and the indexer may select it for t only
in t's document.  Covered: the CUDA-core and tensor-core indexer score
kernels with both select kernels (register rows and the shared-memory rows
beyond 2048 blocks), rows left with fewer than K candidates, arbitrary (not
contiguous) document ids, every attention kernel family (CUDA-core fp32,
warp MMA, tcgen05 forward/backward), and the isolation property itself:
changing one document leaves the other documents' outputs unchanged.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs, packed_doc_ids
from oracle import csa_oracle as orc
from paritylib import TOL, compare_topk_row, f64, maxabs, oracle_indexer, oracle_kv_full

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


def _random_doc_ids(seed, b, sq, n_docs):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, n_docs, (b, sq), generator=g, dtype=torch.int32)


def _topk_row_ok(gpu_row, I_row, K):
    """GPU top-k row vs the oracle scores of that row, where the candidates
    (finite entries) need not be a prefix: positions within the candidate
    list go through the same comparison as the prefix case."""
    cand = np.flatnonzero(np.isfinite(I_row))
    k = min(K, cand.size)
    sel = gpu_row[:k]
    if np.any(gpu_row[k:] != -1):
        return False
    pos = np.searchsorted(cand, sel)
    if np.any(pos >= cand.size) or np.any(cand[np.minimum(pos, cand.size - 1)] != sel):
        return False
    full = np.concatenate([pos, gpu_row[k:]]).astype(np.int32)
    ok, _ = compare_topk_row(full, I_row[cand], K)
    return ok


def _doc_mask(I, doc, ratio):
    """Oracle scores restricted to each query's selectable blocks."""
    I = I.copy()
    b, sq, n_c = I.shape
    for bi in range(b):
        for t in range(sq):
            I[bi, t, ~orc.indexer_selectable(t, n_c, ratio, doc[bi])] = -np.inf
    return I


# ---------------------------------------------------------------------------
# indexer + top-k
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H_I,d_I,docs", [
    ("fp32", 3, 32, "random"),     # CUDA-core scores, documents interleaved token by token
    ("bf16", 4, 64, "random"),     # tensor-core scores
    ("bf16", 8, 128, "packed"),    # packed documents on block boundaries
])
def test_indexer_docs_small(dtype, H_I, d_I, docs):
    b, sq, ratio, topk = 2, 600, 4, 24
    g = torch.Generator().manual_seed(31)
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(_dt(dtype))
    k_I = torch.randn(b, sq // ratio, d_I, generator=g).to(_dt(dtype))
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    doc = _random_doc_ids(32, b, sq, 3) if docs == "random" else packed_doc_ids(b, sq, ratio, 5)
    idx = csa.csa_indexer_topk(q_I.cuda(), k_I.cuda(), w.cuda(), topk, ratio,
                               doc_ids=doc.cuda()).cpu().numpy()
    # documents starting inside a block are reported (CSA_ERR_DEVICE_CHECK at
    # the document-boundary site 0x41); the selection still follows the rule
    # that a block belongs to the document of its first token
    status = csa.csa_get_device_status(with_site=True)
    assert status == ((6, 0x41) if docs == "random" else (0, 0)), status
    I = orc.indexer_scores(f64(q_I), f64(k_I), f64(w), ratio, doc_ids=doc.numpy())
    short = 0
    for bi in range(b):
        for t in range(sq):
            assert _topk_row_ok(idx[bi, t], I[bi, t], topk), (bi, t, idx[bi, t][:8])
            short += int(np.isfinite(I[bi, t]).sum() < topk)
    assert short > 0          # rows with fewer candidates than K were exercised


def test_indexer_docs_csa4():
    """The CSA-4 layer (tensor-core scores, register select) with 6 packed
    documents, every row checked against the oracle."""
    cfg = CONFIGS["csa4_bf16"]
    inp = make_inputs(cfg, parts=("indexer",))
    doc = packed_doc_ids(cfg.b, cfg.sq, cfg.ratio, 6, seed=1)
    idx = csa.csa_indexer_topk(inp["q_I"].cuda(), inp["k_I"].cuda(), inp["w"].cuda(), cfg.topk,
                               cfg.ratio, doc_ids=doc.cuda()).cpu().numpy()
    I = _doc_mask(oracle_indexer(cfg.name)[0], doc.numpy(), cfg.ratio)
    for t in range(cfg.sq):
        assert _topk_row_ok(idx[0, t], I[0, t], cfg.K), (t, idx[0, t][:8])


def test_indexer_docs_wide_rows_sampled():
    """More than 2048 blocks per row (shared-memory select kernel): sampled
    rows against the oracle's score rows."""
    b, sq, ratio, H_I, d_I, topk = 1, 9000, 4, 2, 64, 300
    g = torch.Generator().manual_seed(33)
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(torch.bfloat16)
    k_I = torch.randn(b, sq // ratio, d_I, generator=g).to(torch.bfloat16)
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    doc = packed_doc_ids(b, sq, ratio, 4, seed=2)
    idx = csa.csa_indexer_topk(q_I.cuda(), k_I.cuda(), w.cuda(), topk, ratio,
                               doc_ids=doc.cuda()).cpu().numpy()
    n_c = sq // ratio
    qn, kn, wn, dn = f64(q_I), f64(k_I), f64(w), doc.numpy()
    for t in list(range(0, sq, 97)) + [sq - 1]:
        row = np.full(n_c, -np.inf)
        v = orc.indexer_scores_row(qn[0, t], kn[0], wn[0, t], t, ratio)
        row[:v.shape[0]] = v
        row[~orc.indexer_selectable(t, n_c, ratio, dn[0])] = -np.inf
        assert _topk_row_ok(idx[0, t], row, topk), t


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _attn_both(q, kv, idx, snk, dO, ratio, window, dtype, doc, rows=None):
    b, sq, H, d = q.shape
    scale = d ** -0.5
    c = lambda t: None if t is None else t.cuda()
    O, L = csa.csa_attn_fwd(c(q), c(kv), c(idx), c(snk), scale, ratio, window, doc_ids=c(doc))
    dq, dkv, dsink = csa.csa_attn_bwd(c(q), c(kv), c(idx), c(snk), scale, ratio, window, O, L,
                                      c(dO), doc_ids=c(doc))
    sn = None if snk is None else f64(snk)
    idn, dn = idx.numpy(), doc.numpy()
    tol = TOL[dtype]
    if rows is None:
        O_ref, L_ref = orc.attn_fwd(f64(q), f64(kv), idn, sn, scale, window, ratio, doc_ids=dn)
        dq_ref, dkv_ref, ds_ref = orc.attn_bwd(f64(q), f64(kv), idn, sn, scale, window, ratio,
                                               f64(dO), doc_ids=dn)
        errs = {"O": maxabs(f64(O), O_ref), "LSE": maxabs(f64(L), L_ref),
                "dq": maxabs(f64(dq), dq_ref), "dkv": maxabs(f64(dkv), dkv_ref)}
        if snk is not None:
            errs["dsink"] = maxabs(f64(dsink), ds_ref)
    else:
        O_ref, L_ref = orc.attn_fwd(f64(q), f64(kv), idn, sn, scale, window, ratio, rows=rows,
                                    doc_ids=dn)
        dq_ref, _, _ = orc.attn_bwd(f64(q), f64(kv), idn, sn, scale, window, ratio, f64(dO),
                                    rows=rows, doc_ids=dn)
        bs, ts = [r[0] for r in rows], [r[1] for r in rows]
        errs = {"O": maxabs(f64(O)[bs, ts], O_ref), "LSE": maxabs(f64(L)[bs, ts], L_ref),
                "dq": maxabs(f64(dq)[bs, ts], dq_ref)}
    assert max(errs.values()) <= tol, errs
    return O, L, dq, dkv, dsink


@pytest.mark.parametrize("dtype,H,d", [
    ("fp32", 4, 64),      # CUDA-core kernels
    ("bf16", 6, 64),      # warp-level MMA kernels
    ("bf16", 16, 128),    # tcgen05 kernels, 8 queries per CTA
    ("bf16", 32, 128),    # tcgen05 kernels, 4 queries per CTA
])
def test_attn_docs_random_ids(dtype, H, d):
    b, sq, ratio, window, K = 2, 150, 4, 24, 10
    g = torch.Generator().manual_seed(34)
    n_c = sq // ratio
    q = torch.randn(b, sq, H, d, generator=g).to(_dt(dtype))
    kv = torch.randn(b, sq + n_c, d, generator=g).to(_dt(dtype))
    idx = torch.randint(-1, n_c + 2, (b, sq, K), generator=g, dtype=torch.int32)
    idx[:, :, 1] = idx[:, :, 0]
    snk = torch.randn(H, generator=g)
    dO = torch.randn(b, sq, H, d, generator=g).to(_dt(dtype))
    doc = _random_doc_ids(35, b, sq, 3)
    _attn_both(q, kv, idx, snk, dO, ratio, window, dtype, doc)


def test_attn_docs_debug_layer_full():
    """The debug layer (tcgen05, H=16) with 4 packed documents and the
    oracle's document-aware top-k, every output compared."""
    cfg = CONFIGS["debug_bf16"]
    inp = make_inputs(cfg)
    doc = packed_doc_ids(cfg.b, cfg.sq, cfg.ratio, 4, seed=3)
    I = _doc_mask(oracle_indexer(cfg.name)[0], doc.numpy(), cfg.ratio)
    idx = torch.from_numpy(orc.topk_select(I, cfg.K))
    kv = oracle_kv_full(cfg.name)
    _attn_both(inp["q"], kv, idx, inp["sink"], inp["dO"], cfg.ratio, cfg.window, "bf16", doc)


def test_attn_docs_csa4_sampled_rows():
    cfg = CONFIGS["csa4_bf16"]
    inp = make_inputs(cfg, parts=("attn",))
    doc = packed_doc_ids(cfg.b, cfg.sq, cfg.ratio, 6, seed=1)
    I = _doc_mask(oracle_indexer(cfg.name)[0], doc.numpy(), cfg.ratio)
    idx = torch.from_numpy(orc.topk_select(I, cfg.K))
    kv = oracle_kv_full(cfg.name)
    starts = [0] + [t for t in range(1, cfg.sq) if doc[0, t] != doc[0, t - 1]]
    rows = sorted({(0, min(cfg.sq - 1, max(0, s + o))) for s in starts for o in (-2, -1, 0, 1, 5)}
                  | {(0, t) for t in range(0, cfg.sq, 331)})
    _attn_both(inp["q"], kv, idx, inp["sink"], inp["dO"], cfg.ratio, cfg.window, "bf16", doc,
               rows=rows)


def test_documents_are_isolated_bit_exactly():
    """Changing every input of document 0 leaves the outputs of the other
    documents unchanged: the indexer selections of every later query, and O,
    LSE and dq bit for bit for the queries whose tensor-core block (128 / H
    consecutive queries) lies wholly after document 0.  A block that straddles
    the boundary walks the union of all its queries' slots, which changes with
    document 0's selections, so its later-document rows are equal only up to
    rounding order; dkv rows are compared the same way (fp32 atomics)."""
    cfg = CONFIGS["debug_bf16"]
    inp = make_inputs(cfg)
    doc = packed_doc_ids(cfg.b, cfg.sq, cfg.ratio, 3, seed=4)
    first_end = int((doc[0] == 0).sum())
    n0 = first_end // cfg.ratio
    kv = oracle_kv_full(cfg.name)

    def run(x, kv_full):
        dv = doc.cuda()
        idx = csa.csa_indexer_topk(x["q_I"].cuda(), x["k_I"].cuda(), x["w"].cuda(), cfg.topk,
                                   cfg.ratio, doc_ids=dv)
        O, L = csa.csa_attn_fwd(x["q"].cuda(), kv_full.cuda(), idx, x["sink"].cuda(), cfg.scale,
                                cfg.ratio, cfg.window, doc_ids=dv)
        dq, dkv, _ = csa.csa_attn_bwd(x["q"].cuda(), kv_full.cuda(), idx, x["sink"].cuda(),
                                      cfg.scale, cfg.ratio, cfg.window, O, L, x["dO"].cuda(),
                                      doc_ids=dv)
        return idx.cpu(), O.cpu(), L.cpu(), dq.cpu(), dkv.cpu()

    a = run(inp, kv)
    g = torch.Generator().manual_seed(36)
    x2 = dict(inp)
    for k in ("q_I", "q", "dO"):
        t = x2[k].clone()
        t[:, :first_end] = torch.randn(t[:, :first_end].shape, generator=g).to(t.dtype)
        x2[k] = t
    k_I = x2["k_I"].clone()
    k_I[:, :n0] = torch.randn(k_I[:, :n0].shape, generator=g).to(k_I.dtype)
    x2["k_I"] = k_I
    kv2 = kv.clone()
    kv2[:, :first_end] = torch.randn(kv2[:, :first_end].shape, generator=g).to(kv2.dtype)
    kv2[:, cfg.sq:cfg.sq + n0] = torch.randn(kv2[:, cfg.sq:cfg.sq + n0].shape,
                                             generator=g).to(kv2.dtype)
    b_ = run(x2, kv2)
    qb = 128 // cfg.H
    whole = slice(-(-first_end // qb) * qb, cfg.sq)
    rest = slice(first_end, cfg.sq)
    assert torch.equal(a[0][:, rest], b_[0][:, rest])
    for name, u, v in zip(("O", "LSE", "dq"), a[1:4], b_[1:4]):
        assert torch.equal(u[:, whole], v[:, whole]), name
        assert torch.allclose(u[:, rest].float(), v[:, rest].float(), atol=1e-2), name
    assert not torch.equal(a[1][:, :first_end], b_[1][:, :first_end])
    dkv_a, dkv_b = a[4], b_[4]
    assert torch.allclose(dkv_a[:, first_end:cfg.sq], dkv_b[:, first_end:cfg.sq], atol=1e-2)
    assert torch.allclose(dkv_a[:, cfg.sq + n0:], dkv_b[:, cfg.sq + n0:], atol=1e-2)
