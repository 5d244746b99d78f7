"""GPU parity of the four CSA entry points against the fp64 oracle, on the
five seeded workloads, through the C ABI (Python binding).

Full-size comparisons where the oracle finishes in seconds; on the
production-width workload (b=2, sq=8192, H=64, d=512) sampled rows that the
oracle computes one by one, plus identities that hold at any size.
Tolerances: max abs error 2e-3 (fp32 inputs) / 2e-2 (bf16 inputs) for O,
LSE and gradients; top-k sets bit-exact wherever the K-th/(K+1)-th score gap
exceeds 1e-3 or the boundary is an exact tie (lower index wins).
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, CONFIG_ORDER, make_inputs
from oracle import csa_oracle as orc
from paritylib import (TOL, attn_indices, compare_topk_row, f64, maxabs, oracle_indexer,
                       oracle_kv_full)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    csa.load_library()
    yield
    assert csa.csa_get_device_status() == 0


def _cuda(t):
    return t.cuda() if t is not None else None


# ---------------------------------------------------------------------------
# compressor
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_compress_parity(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("compress",))
    kv_raw, score = inp["kv_raw"].cuda(), inp["score"].cuda()
    b, sq, d, n_c = cfg.b, cfg.sq, cfg.d, cfg.n_c
    kv_full = torch.full((b, sq + n_c, d), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    kv_full[:, :sq] = kv_raw
    csa.csa_compress(kv_full[:, :sq], score, cfg.ratio, out=kv_full[:, sq:])
    torch.cuda.synchronize()
    ref = orc.compress(f64(inp["kv_raw"]), f64(inp["score"]), cfg.ratio)
    got = f64(kv_full[:, sq:])
    assert np.all(np.isfinite(got))
    err = maxabs(got, ref)
    assert err <= TOL[cfg.dtype], err
    assert torch.equal(kv_full[:, :sq], kv_raw)


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_compress_bwd_parity(name):
    """Gradient of the pooling in the layer layout: the compressed rows of
    dkv_full are the incoming gradient, the raw rows accumulate w*g."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("compress",))
    b, sq, d, n_c = cfg.b, cfg.sq, cfg.d, cfg.n_c
    g = torch.Generator().manual_seed(7)
    dout = torch.randn(b, n_c, d, generator=g)
    pre = torch.randn(b, sq, d, generator=g)
    kv_full = torch.zeros(b, sq + n_c, d, dtype=cfg.torch_dtype, device="cuda")
    kv_full[:, :sq] = inp["kv_raw"].cuda()
    dkv_full = torch.cat([pre, dout], dim=1).cuda()
    dscore = csa.csa_compress_bwd(kv_full[:, :sq], inp["score"].cuda(), cfg.ratio,
                                  dkv_full[:, sq:], dkv_full[:, :sq])
    torch.cuda.synchronize()
    ref_dkv, ref_ds = orc.compress_bwd(f64(inp["kv_raw"]), f64(inp["score"]), cfg.ratio, f64(dout))
    tol = TOL[cfg.dtype]
    e_kv = maxabs(f64(dkv_full[:, :sq]) - f64(pre), ref_dkv)
    e_s = maxabs(f64(dscore), ref_ds)
    assert e_kv <= tol and e_s <= tol, (e_kv, e_s)
    assert torch.equal(dkv_full[:, sq:].cpu(), dout)


# ---------------------------------------------------------------------------
# indexer + top-k
# ---------------------------------------------------------------------------

def _check_topk_rows(gpu_idx, gpu_sc, I_rows, t_list, K, ratio, n_c):
    bad, ties = [], 0
    for n, t in enumerate(t_list):
        v = min((t + 1) // ratio, n_c)
        ok, exact = compare_topk_row(gpu_idx[n], I_rows[n][:v], K)
        ties += (not exact)
        if not ok:
            bad.append(t)
        k = min(K, v)
        if gpu_sc is not None and k:
            sel = gpu_idx[n][:k]
            ref = I_rows[n][sel]
            assert np.all(np.abs(gpu_sc[n][:k] - ref) <= 1e-3 * np.maximum(1.0, np.abs(ref)))
            assert np.all(gpu_sc[n][k:] == 0)
    return bad, ties


@pytest.mark.parametrize("name", ["tiny_fp32", "debug_bf16", "csa4_bf16"])
def test_indexer_topk_parity_full(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("indexer",))
    idx, sc = csa.csa_indexer_topk(inp["q_I"].cuda(), inp["k_I"].cuda(), inp["w"].cuda(), cfg.topk,
                                   cfg.ratio, return_scores=True)
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    I, _ = oracle_indexer(name)
    total_ties = 0
    for bi in range(cfg.b):
        bad, ties = _check_topk_rows(idx[bi], sc[bi], I[bi], range(cfg.sq), cfg.K, cfg.ratio,
                                     cfg.n_c)
        assert not bad, f"batch {bi}: rows {bad[:10]} differ"
        total_ties += ties
    print(f"{name}: near-tie rows (gap <= 1e-3) {total_ties}")


def test_indexer_topk_parity_production_sampled():
    cfg = CONFIGS["prod_bf16"]
    inp = make_inputs(cfg, parts=("indexer",))
    idx, sc = csa.csa_indexer_topk(inp["q_I"].cuda(), inp["k_I"].cuda(), inp["w"].cuda(), cfg.topk,
                                   cfg.ratio, return_scores=True)
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    rng = np.random.default_rng(0)
    q_I, k_I, w = f64(inp["q_I"]), f64(inp["k_I"]), f64(inp["w"])
    for bi in range(cfg.b):
        ts = sorted(set(rng.integers(0, cfg.sq, 24).tolist()) | {cfg.sq - 1, cfg.sq - 2, 4095, 7})
        rows = [orc.indexer_scores_row(q_I[bi, t], k_I[bi], w[bi, t], t, cfg.ratio) for t in ts]
        rows = [np.concatenate([r, np.full(cfg.n_c - r.shape[0], -np.inf)]) for r in rows]
        bad, _ = _check_topk_rows(idx[bi, ts], sc[bi, ts], rows, ts, cfg.K, cfg.ratio, cfg.n_c)
        assert not bad, bad


# ---------------------------------------------------------------------------
# attention forward / backward
# ---------------------------------------------------------------------------

def _attn_inputs(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("attn",))
    kv_full = oracle_kv_full(name)
    idx = attn_indices(cfg)
    return cfg, inp["q"], kv_full, idx, inp["sink"], inp["dO"]


@pytest.mark.parametrize("name", ["tiny_fp32", "debug_bf16", "csa4_bf16", "hca_bf16"])
def test_attn_fwd_bwd_parity_full(name):
    cfg, q, kv_full, idx, sink, dO = _attn_inputs(name)
    O, L = csa.csa_attn_fwd(q.cuda(), kv_full.cuda(), idx.cuda(), sink.cuda(), cfg.scale, cfg.ratio,
                            cfg.window)
    O_ref, L_ref = orc.attn_fwd(f64(q), f64(kv_full), idx.numpy(), f64(sink), cfg.scale, cfg.window,
                                cfg.ratio)
    tol = TOL[cfg.dtype]
    e_o, e_l = maxabs(f64(O), O_ref), maxabs(f64(L), L_ref)
    assert e_o <= tol and e_l <= tol, (e_o, e_l)
    # backward: both sides get the oracle's O (stored dtype) and LSE (fp32)
    O_in = torch.from_numpy(orc.round_to_storage(O_ref, cfg.dtype)).to(cfg.torch_dtype).cuda()
    L_in = torch.from_numpy(L_ref).float().cuda()
    dq, dkv, dsink = csa.csa_attn_bwd(q.cuda(), kv_full.cuda(), idx.cuda(), sink.cuda(), cfg.scale,
                                      cfg.ratio, cfg.window, O_in, L_in, dO.cuda())
    dq_ref, dkv_ref, ds_ref = orc.attn_bwd(f64(q), f64(kv_full), idx.numpy(), f64(sink), cfg.scale,
                                           cfg.window, cfg.ratio, f64(dO))
    errs = (maxabs(f64(dq), dq_ref), maxabs(f64(dkv), dkv_ref), maxabs(f64(dsink), ds_ref))
    print(f"{name}: O {e_o:.2e} LSE {e_l:.2e} dq {errs[0]:.2e} dkv {errs[1]:.2e} "
          f"dsink {errs[2]:.2e} (|dkv|max {np.abs(dkv_ref).max():.1f})")
    assert max(errs) <= tol, errs


def test_attn_parity_production_sampled():
    """b=2, sq=8192, H=64, d=512, Zipf-skewed indices with 10% padding: sampled
    query rows (O, LSE, dq), complete dKV rows (raw rows from their window
    queries, cold compressed rows from their selecting queries), and two
    identities that hold at any size."""
    cfg, q, kv_full, idx, sink, dO = _attn_inputs("prod_bf16")
    qc, kvc, ic, sc, gc = q.cuda(), kv_full.cuda(), idx.cuda(), sink.cuda(), dO.cuda()
    O, L = csa.csa_attn_fwd(qc, kvc, ic, sc, cfg.scale, cfg.ratio, cfg.window)
    dq, dkv, dsink = csa.csa_attn_bwd(qc, kvc, ic, sc, cfg.scale, cfg.ratio, cfg.window, O, L, gc)
    torch.cuda.synchronize()
    qn, kvn, idn, sn, gn = f64(q), f64(kv_full), idx.numpy(), f64(sink), f64(dO)
    tol = TOL[cfg.dtype]
    rng = np.random.default_rng(1)
    rows = [(int(rng.integers(0, 2)), int(t)) for t in rng.integers(0, cfg.sq, 20)]
    rows += [(0, 0), (1, cfg.sq - 1), (0, 4095)]
    O_ref, L_ref = orc.attn_fwd(qn, kvn, idn, sn, cfg.scale, cfg.window, cfg.ratio, rows=rows)
    bi_l = [r[0] for r in rows]
    t_l = [r[1] for r in rows]
    assert maxabs(f64(O[bi_l, t_l]), O_ref) <= tol
    assert maxabs(f64(L[bi_l, t_l]), L_ref) <= tol
    dq_ref, _, _ = orc.attn_bwd(qn, kvn, idn, sn, cfg.scale, cfg.window, cfg.ratio, gn, rows=rows)
    assert maxabs(f64(dq[bi_l, t_l]), dq_ref) <= tol
    # complete dKV rows: raw row r gets contributions only from queries r..r+W-1
    for (bi, r) in [(0, 5000), (1, cfg.sq - 1)]:
        qs = [(bi, t) for t in range(r, min(cfg.sq, r + cfg.window))]
        _, dkv_part, _ = orc.attn_bwd(qn, kvn, idn, sn, cfg.scale, cfg.window, cfg.ratio, gn,
                                      rows=qs)
        assert maxabs(f64(dkv[bi, r]), dkv_part[bi, r]) <= tol
    # a cold compressed row: every query that selects it
    for bi in range(2):
        t_all = np.arange(cfg.sq)
        vis = (t_all + 1) // cfg.ratio
        sel = []
        for j in range(cfg.n_c - 1, 0, -1):
            sel = np.nonzero(((idn[bi] == j) & (j < vis[:, None])).any(axis=1))[0]
            if 0 < len(sel) <= 64:
                break
        assert 0 < len(sel) <= 64
        _, dkv_part, _ = orc.attn_bwd(qn, kvn, idn, sn, cfg.scale, cfg.window, cfg.ratio, gn,
                                      rows=[(bi, int(t)) for t in sel])
        assert maxabs(f64(dkv[bi, cfg.sq + j]), dkv_part[bi, cfg.sq + j]) <= tol
    # identity 1 (scaling kv): sum_rows kv.dkv = sum_{t,h} (dO.O + q.dq)
    lhs = (kv_full.cuda().double() * dkv.double()).sum().item()
    rhs = ((gc.double() * O.double()).sum() + (qc.double() * dq.double()).sum()).item()
    assert abs(lhs - rhs) <= 1e-2 * max(1.0, abs(rhs)), (lhs, rhs)
    # identity 2 (sink gradient): dsink_h = -sum_{b,t} exp(sink_h - LSE) (dO.O)
    Dh = (gc.double() * O.double()).sum(-1)
    ds_id = -(torch.exp(sc.double().view(1, 1, -1) - L.double()) * Dh).sum((0, 1))
    assert maxabs(f64(dsink), f64(ds_id)) <= tol * max(1.0, float(ds_id.abs().max()))
