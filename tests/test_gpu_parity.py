"""GPU parity of the four CSA entry points against the fp64 oracle, on the
five seeded workloads, through the C ABI (Python binding).

Full-size comparisons: the oracle finishes the small workloads in seconds,
and the production-width workload (b=2, sq=8192, H=64, d=512) in about a
minute on every host core (spawned processes over shared inputs); its
indexer is checked on sampled rows (its attention runs on synthetic lists).
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


def test_attn_parity_production_full():
    """b=2, sq=8192, H=64, d=512, Zipf-skewed indices with 10% padding, the
    whole layer against the oracle: O, LSE and dq of every query row, every
    row of dKV (raw and compressed, including the hottest Zipf rows, which
    sum thousands of repeated-index terms in fp32) and dsink.  The oracle runs
    over all 16384 query rows in spawned processes on every host core
    (oracle.rows_pool); each process returns the dKV / dsink contributions of
    its rows, which are summed here in float64."""
    from oracle.rows_pool import RowPool, split_rows
    cfg, q, kv_full, idx, sink, dO = _attn_inputs("prod_bf16")
    qc, kvc, ic, sc, gc = q.cuda(), kv_full.cuda(), idx.cuda(), sink.cuda(), dO.cuda()
    O, L = csa.csa_attn_fwd(qc, kvc, ic, sc, cfg.scale, cfg.ratio, cfg.window)
    dq, dkv, dsink = csa.csa_attn_bwd(qc, kvc, ic, sc, cfg.scale, cfg.ratio, cfg.window, O, L, gc)
    torch.cuda.synchronize()
    assert csa.csa_get_device_status() == 0
    idn = idx.numpy()
    arrays = {"q": q, "dO": dO, "kv_full": kv_full, "idx": idn, "sink": sink.numpy(),
              "O": O.cpu(), "L": L.cpu().numpy(), "dq": dq.cpu().numpy()}
    del qc, gc
    rows = [(bi, t) for bi in range(cfg.b) for t in range(cfg.sq)]
    with RowPool(arrays) as pool:
        parts = pool.map("oracle.rows_pool.attn_rows_vs",
                         [dict(rows=r, scale=cfg.scale, window=cfg.window, ratio=cfg.ratio)
                          for r in split_rows(rows, pool.procs)])
    tol = TOL[cfg.dtype]
    e_o = max(p[0] for p in parts)
    e_l = max(p[1] for p in parts)
    e_dq = max(p[2] for p in parts)
    dkv_ref = sum(p[3] for p in parts)
    ds_ref = sum(p[4] for p in parts)
    dkv_g = f64(dkv)
    err_rows = np.abs(dkv_g - dkv_ref).max(axis=2)              # [b, n_kv]
    e_dkv = float(err_rows.max())
    e_ds = maxabs(f64(dsink), ds_ref)
    # the hottest compressed rows: most (query, slot) selections
    vis = (np.arange(cfg.sq) + 1) // cfg.ratio
    valid = (idn >= 0) & (idn < vis[None, :, None])
    counts = np.zeros((cfg.b, cfg.n_c), np.int64)
    for bi in range(cfg.b):
        counts[bi] = np.bincount(idn[bi][valid[bi]], minlength=cfg.n_c)
    hot = np.argsort(counts.ravel())[::-1][:10]
    print(f"prod_bf16 full: O {e_o:.2e} LSE {e_l:.2e} dq {e_dq:.2e} dkv {e_dkv:.2e} "
          f"(|dkv|max {np.abs(dkv_ref).max():.1f}) dsink {e_ds:.2e} "
          f"(|dsink|max {np.abs(ds_ref).max():.1f})")
    for h in hot:
        bi, j = divmod(int(h), cfg.n_c)
        print(f"  hot compressed row b={bi} j={j}: selected {counts[bi, j]} times, "
              f"|dkv| max {np.abs(dkv_ref[bi, cfg.sq + j]).max():.2f}, "
              f"err {err_rows[bi, cfg.sq + j]:.2e}")
    assert max(e_o, e_l, e_dq, e_dkv, e_ds) <= tol, (e_o, e_l, e_dq, e_dkv, e_ds)
