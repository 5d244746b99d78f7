"""GPU edge cases against the fp64 oracle, through the C ABI.

Repeated indices with -1 / out-of-range / not-yet-visible entries at b=2
(the loop-oracle regression of the gather-backward review), no sink, dense
compressed mode, ragged tails (sq not a multiple of the ratio or of any
tile), n_c = 1, window 1 and window > sq, topk >= n_c, exact ties in the
indexer, chunked indexer workspaces, zeroing of dkv/dsink, odd head counts
and every supported head dim.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from oracle import csa_oracle as orc
from paritylib import TOL, compare_topk_row, f64, maxabs

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


def _rand_attn(seed, b, sq, H, d, ratio, window, K, dtype, sink=True, dup=True):
    g = torch.Generator().manual_seed(seed)
    n_c = sq // ratio
    q = torch.randn(b, sq, H, d, generator=g).to(_dt(dtype))
    kv = torch.randn(b, sq + n_c, d, generator=g).to(_dt(dtype))
    idx = torch.randint(-1, n_c + 2, (b, sq, K), generator=g, dtype=torch.int32)
    if dup and K > 1:
        idx[:, :, 1] = idx[:, :, 0]
    snk = torch.randn(H, generator=g) if sink else None
    dO = torch.randn(b, sq, H, d, generator=g).to(_dt(dtype))
    return q, kv, idx, snk, dO


def _run_both(q, kv, idx, snk, dO, ratio, window, dtype):
    b, sq, H, d = q.shape
    scale = d ** -0.5
    c = lambda t: None if t is None else t.cuda()
    O, L = csa.csa_attn_fwd(c(q), c(kv), c(idx), c(snk), scale, ratio, window)
    dq, dkv, dsink = csa.csa_attn_bwd(c(q), c(kv), c(idx), c(snk), scale, ratio, window, O, L, c(dO))
    idn = idx.numpy() if idx is not None else np.tile(
        np.arange(sq // ratio, dtype=np.int32), (b, sq, 1))
    sn = None if snk is None else f64(snk)
    O_ref, L_ref = orc.attn_fwd(f64(q), f64(kv), idn, sn, scale, window, ratio)
    dq_ref, dkv_ref, ds_ref = orc.attn_bwd(f64(q), f64(kv), idn, sn, scale, window, ratio, f64(dO))
    tol = TOL[dtype]
    errs = {"O": maxabs(f64(O), O_ref), "LSE": maxabs(f64(L), L_ref), "dq": maxabs(f64(dq), dq_ref),
            "dkv": maxabs(f64(dkv), dkv_ref)}
    if snk is not None:
        errs["dsink"] = maxabs(f64(dsink), ds_ref)
    assert max(errs.values()) <= tol, errs
    return O, L, dq, dkv, dsink


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("sink", [True, False])
def test_repeated_indices_padding_b2(dtype, sink):
    q, kv, idx, snk, dO = _rand_attn(1, b=2, sq=96, H=4, d=64, ratio=4, window=8, K=12,
                                     dtype=dtype, sink=sink)
    _run_both(q, kv, idx, snk, dO, 4, 8, dtype)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("shape", [
    dict(b=1, sq=4, H=2, d=64, ratio=4, window=1, K=1),        # n_c = 1, window 1
    dict(b=2, sq=131, H=20, d=128, ratio=4, window=200, K=40),  # ragged tails, window > sq, odd H
    dict(b=1, sq=77, H=3, d=256, ratio=3, window=5, K=30),      # topk > n_c, d 256
    dict(b=1, sq=64, H=16, d=512, ratio=8, window=16, K=4),     # d 512
    dict(b=1, sq=50, H=5, d=40, ratio=5, window=7, K=6),        # d not a power of two
])
def test_ragged_shapes(dtype, shape):
    q, kv, idx, snk, dO = _rand_attn(2, dtype=dtype, **shape)
    _run_both(q, kv, idx, snk, dO, shape["ratio"], shape["window"], dtype)


# ---------------------------------------------------------------------------
# the production-width tensor-core forward (bf16, d = 512, H = 64)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", [
    dict(b=2, sq=300, ratio=4, window=40, K=30, sink=True),     # repeats, -1, out of range
    dict(b=1, sq=261, ratio=3, window=1, K=200, sink=False),    # window 1, no sink, K > n_c
    dict(b=1, sq=700, ratio=4, window=128, K=175, sink=True),   # several slot tiles
    dict(b=1, sq=9, ratio=4, window=3, K=2, sink=True),         # n_c = 2, ragged tail
])
def test_tc512_forward_edges(case):
    """The transposed tcgen05 forward and backward at the production width
    against the oracle."""
    c = dict(case)
    sink = c.pop("sink")
    q, kv, idx, snk, dO = _rand_attn(12, H=64, d=512, dtype="bf16", sink=sink, **c)
    _run_both(q, kv, idx, snk, dO, c["ratio"], c["window"], "bf16")


def test_tc512_forward_large_logits_and_dense_mode():
    """The running maximum grows by far more than 2^8 between slot tiles, so
    O and the sums are rescaled: the window rows (the first tiles) are small
    and the compressed rows (later tiles, dense list) large in logit, while
    every row stays of unit size so that |O| <= 4 (the bf16 output's rounding
    stays inside the bound)."""
    b, sq, ratio, W = 1, 1100, 4, 256
    q, kv, _, snk, dO = _rand_attn(13, b, sq, 64, 512, ratio, W, 1, "bf16")
    kv[:, :sq] = (kv[:, :sq].float() * 0.05).to(torch.bfloat16)
    q = (q.float() * 4).to(torch.bfloat16)
    _run_both(q, kv, None, snk, dO, ratio, W, "bf16")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_dense_mode_matches_all_visible_list(dtype):
    b, sq, H, d, ratio, W = 2, 300, 8, 128, 16, 24
    q, kv, _, snk, dO = _rand_attn(3, b, sq, H, d, ratio, W, 1, dtype)
    n_c = sq // ratio
    vis = (torch.arange(1, sq + 1) // ratio).view(sq, 1)
    j = torch.arange(n_c).view(1, n_c)
    full = torch.where(j < vis, j, -1).to(torch.int32).expand(b, sq, n_c).contiguous()
    r_list = _run_both(q, kv, full, snk, dO, ratio, W, dtype)
    r_dense = _run_both(q, kv, None, snk, dO, ratio, W, dtype)
    assert torch.equal(r_list[0], r_dense[0]) and torch.equal(r_list[1], r_dense[1])
    assert torch.equal(r_list[2], r_dense[2])


def test_bwd_zeroes_outputs():
    q, kv, idx, snk, dO = _rand_attn(4, 1, 64, 4, 64, 4, 8, 8, "bf16")
    c = lambda t: t.cuda()
    O, L = csa.csa_attn_fwd(c(q), c(kv), c(idx), c(snk), 0.125, 4, 8)
    ref = csa.csa_attn_bwd(c(q), c(kv), c(idx), c(snk), 0.125, 4, 8, O, L, c(dO))
    dkv = torch.full_like(ref[1], 7.0)
    dsink = torch.full_like(ref[2], -3.0)
    got = csa.csa_attn_bwd(c(q), c(kv), c(idx), c(snk), 0.125, 4, 8, O, L, c(dO), dkv=dkv,
                           dsink=dsink)
    assert torch.allclose(got[1], ref[1], atol=1e-5) and torch.allclose(got[2], ref[2], atol=1e-5)


# ---------------------------------------------------------------------------
# indexer
# ---------------------------------------------------------------------------

def _indexer_case(seed, b, sq, H_I, d_I, ratio, dtype, ties=False):
    g = torch.Generator().manual_seed(seed)
    n_c = sq // ratio
    q_I = torch.randn(b, sq, H_I, d_I, generator=g)
    k_I = torch.randn(b, n_c, d_I, generator=g)
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    if ties:
        q_I = q_I.abs()
        w = w.abs()
        k_I[:, 1::5] = k_I[:, 0::5][:, :k_I[:, 1::5].shape[1]]      # duplicate key rows
        k_I[:, 3::7] = -k_I[:, 3::7].abs()                         # all dots < 0: score 0
    return q_I.to(_dt(dtype)), k_I.to(_dt(dtype)), w


def _check_indexer(q_I, k_I, w, topk, ratio, ws_bytes=None):
    b, sq, H_I, d_I = q_I.shape
    n_c = k_I.shape[1]
    K = min(topk, n_c)
    wsp = None
    if ws_bytes is not None:
        wsp = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    idx, sc = csa.csa_indexer_topk(q_I.cuda(), k_I.cuda(), w.cuda(), topk, ratio, workspace=wsp,
                                   return_scores=True)
    I = orc.indexer_scores(f64(q_I), f64(k_I), f64(w), ratio)
    idx = idx.cpu().numpy()
    for bi in range(b):
        for t in range(sq):
            v = min((t + 1) // ratio, n_c)
            ok, _ = compare_topk_row(idx[bi, t], I[bi, t, :v], K)
            assert ok, (bi, t, idx[bi, t][:8])
    return idx, sc


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_indexer_exact_ties(dtype):
    q_I, k_I, w = _indexer_case(5, 2, 200, 3, 64, 2, dtype, ties=True)
    _check_indexer(q_I, k_I, w, 17, 2)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("case", [
    dict(b=1, sq=4, H_I=1, d_I=32, ratio=4, topk=1),      # n_c = 1
    dict(b=2, sq=333, H_I=5, d_I=64, ratio=4, topk=500),  # topk > n_c, ragged
    dict(b=1, sq=515, H_I=8, d_I=128, ratio=4, topk=64),  # ragged tile tail
    dict(b=1, sq=260, H_I=2, d_I=256, ratio=1, topk=100), # d_I 256, ratio 1
])
def test_indexer_shapes(dtype, case):
    q_I, k_I, w = _indexer_case(6, case["b"], case["sq"], case["H_I"], case["d_I"], case["ratio"],
                                dtype)
    _check_indexer(q_I, k_I, w, case["topk"], case["ratio"])


@pytest.mark.parametrize("dtype,case", [
    # n_c 4100: more than 2048 blocks per row, the shared-memory select kernel
    ("bf16", dict(b=1, sq=8200, H_I=2, d_I=64, ratio=2, topk=300, ties=False)),
    # n_c 16384, the largest supported (the default workspace takes 8 chunks
    # of 2048 rows); duplicated key rows and ReLU zeros give exact ties
    ("bf16", dict(b=1, sq=16384, H_I=1, d_I=64, ratio=1, topk=64, ties=True)),
    # CUDA-core fp32 scores into the same select, b = 2, exact ties
    ("fp32", dict(b=2, sq=5000, H_I=3, d_I=32, ratio=2, topk=128, ties=True)),
])
def test_indexer_wide_rows_sampled(dtype, case):
    """Rows of more than 2048 visible blocks, up to the largest n_c: sampled
    rows (spread over the sequence, and its last two) against the oracle's
    score rows, bit-exact sets where the K-th gap exceeds 1e-3 or is a tie."""
    b, sq, ratio = case["b"], case["sq"], case["ratio"]
    q_I, k_I, w = _indexer_case(40, b, sq, case["H_I"], case["d_I"], ratio, dtype,
                                ties=case["ties"])
    n_c = sq // ratio
    K = min(case["topk"], n_c)
    idx = csa.csa_indexer_topk(q_I.cuda(), k_I.cuda(), w.cuda(), case["topk"],
                               ratio).cpu().numpy()
    qn, kn, wn = f64(q_I), f64(k_I), f64(w)
    rows = list(range(0, sq, max(1, sq // 48))) + [sq - 2, sq - 1]
    n_exact = 0
    for bi in range(b):
        for t in rows:
            v = orc.indexer_scores_row(qn[bi, t], kn[bi], wn[bi, t], t, ratio)
            ok, exact = compare_topk_row(idx[bi, t], v, K)
            assert ok, (bi, t, idx[bi, t][:8])
            n_exact += exact
    assert n_exact >= len(rows) // 2       # most rows are held to the exact set


@pytest.mark.parametrize("case", [
    dict(sq=480, ratio=1, topk=40),      # 256 < n_c <= 512: four keys per thread
    dict(sq=1600, ratio=1, topk=300),    # 1024 < n_c <= 2048: sixteen keys per thread
    dict(sq=1030, ratio=1, topk=1000),   # K close to n_c: few rows above K blocks
])
def test_indexer_select_cta_rows_with_ties(case):
    """Every row of layers whose rows above K visible blocks take a CTA each
    (duplicated key rows and ReLU zeros give exact ties at the K-th score),
    with the scores returned and without."""
    q_I, k_I, w = _indexer_case(12, 1, case["sq"], 2, 64, case["ratio"], "bf16", ties=True)
    idx, _ = _check_indexer(q_I, k_I, w, case["topk"], case["ratio"])
    plain = csa.csa_indexer_topk(q_I.cuda(), k_I.cuda(), w.cuda(), case["topk"], case["ratio"])
    assert np.array_equal(plain.cpu().numpy(), idx)


def test_indexer_chunked_workspace_identical():
    q_I, k_I, w = _indexer_case(7, 2, 1000, 4, 128, 4, "bf16")
    full, sc_full = _check_indexer(q_I, k_I, w, 96, 4)
    lib = csa.load_library()
    small = int(lib.csa_indexer_topk_min_workspace(2, 250))
    chunked, sc_chunk = _check_indexer(q_I, k_I, w, 96, 4, ws_bytes=small + 100)
    assert np.array_equal(full, chunked)
    assert torch.equal(sc_full, sc_chunk)


# ---------------------------------------------------------------------------
# tensor-core attention forward (d = 128, H in {16, 32, 64}: rows are
# (query, head) pairs of consecutive queries over the union of their slots)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H", [16, 32, 64])
@pytest.mark.parametrize("sink", [True, False])
@pytest.mark.parametrize("case", [
    dict(b=2, sq=203, ratio=4, window=16, K=24),    # ragged: sq not a multiple of the block
    dict(b=1, sq=300, ratio=2, window=130, K=64),   # window longer than one slot tile
])
def test_tc_forward_repeated_and_padded_indices(H, sink, case):
    q, kv, idx, snk, dO = _rand_attn(8, H=H, d=128, dtype="bf16", sink=sink, **case)
    # more repeats: a block listed three times in one row
    idx[:, :, 2] = idx[:, :, 0]
    _run_both(q, kv, idx, snk, dO, case["ratio"], case["window"], "bf16")


@pytest.mark.parametrize("H", [16, 32])
def test_tc_forward_dense_mode_and_large_logits(H):
    b, sq, ratio, W = 1, 260, 8, 40
    q, kv, _, snk, dO = _rand_attn(9, b, sq, H, 128, ratio, W, 1, "bf16")
    q = (q.float() * 4).bfloat16()           # logits spread over a wide range
    _run_both(q, kv, None, snk, dO, ratio, W, "bf16")


# ---------------------------------------------------------------------------
# compressor forward/backward: per-token score, ragged tail, fp32 and bf16
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("score_width", [1, "d"])
@pytest.mark.parametrize("b,sq,d,ratio", [
    (2, 43, 24, 5),        # one thread per block and 8 channels; 3 tokens past the last block
    (2, 200, 24, 37),      # token-split kernel: odd ratio, 3 channel groups, 15-token tail
    (1, 300, 512, 128),    # token-split kernel at the HCA ratio, d = 512, 44-token tail
    (1, 1091, 64, 17),     # token-split kernel, ratio just above its threshold
    (1, 70, 8, 16),        # token-split kernel, one channel group: most token lanes idle
    (1, 600, 64, 272),     # token-split kernel, 9 tokens a lane: past the register-held ones
])
def test_compress_fwd_bwd_ragged_and_scalar_score(dtype, score_width, b, sq, d, ratio):
    g = torch.Generator().manual_seed(11)
    sw = d if score_width == "d" else 1
    kv = torch.randn(b, sq, d, generator=g).to(_dt(dtype))
    score = (torch.randn(b, sq, sw, generator=g) * 3).to(_dt(dtype))
    dout = torch.randn(b, sq // ratio, d, generator=g)
    out = csa.csa_compress(kv.cuda(), score.cuda(), ratio)
    dkv = torch.zeros(b, sq, d, device="cuda")
    dscore = csa.csa_compress_bwd(kv.cuda(), score.cuda(), ratio, dout.cuda(), dkv)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    assert maxabs(f64(out), orc.compress(f64(kv), f64(score), ratio)) <= tol
    ref_dkv, ref_ds = orc.compress_bwd(f64(kv), f64(score), ratio, f64(dout))
    assert maxabs(f64(dkv), ref_dkv) <= tol
    assert maxabs(f64(dscore), ref_ds) <= tol
    n_tok = sq // ratio * ratio
    assert torch.all(dkv[:, n_tok:] == 0) and torch.all(dscore[:, n_tok:] == 0)
