"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against something independent of it:
a hand-derived worked example (tests/golden), a closed form, a special case
that reduces to a library routine (numpy matmul, torch's scaled-dot-product
attention and autograd in float64), brute-force enumeration, central finite
differences, or an invariant.  The cases are chosen so that a dropped term, a
wrong sign or index, or a transposed operand in the oracle fails one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import csa_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(x):
    """Evaluate a closed-form expression string of a golden fixture."""
    if isinstance(x, list):
        return [_ev(v) for v in x]
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"log": math.log, "exp": math.exp}))
    return float(x)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------

def test_round_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ours = orc.round_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_round_bf16_is_nearest_and_ties_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert orc.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert orc.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2 * 2.0 ** -7
    assert orc.round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == -(1.0 + 2.0 ** -7)


# ---------------------------------------------------------------------------
# compressor
# ---------------------------------------------------------------------------

def test_compress_golden():
    g = _load("compress_tiny.json")
    kv = np.array(_ev(g["kv"]))
    score = np.array(_ev(g["score"]))
    out = orc.compress(kv, score, g["ratio"])
    assert out.shape == (1, 1, 2)
    np.testing.assert_allclose(out, np.array(_ev(g["expected_kv_c"])), rtol=0, atol=1e-14)


def test_compress_ratio1_is_identity():
    rng = np.random.default_rng(1)
    kv = rng.standard_normal((2, 9, 5))
    score = rng.standard_normal((2, 9, 5)) * 10
    np.testing.assert_allclose(orc.compress(kv, score, 1), kv, rtol=0, atol=1e-15)


def test_compress_constant_score_is_block_mean():
    rng = np.random.default_rng(2)
    kv = rng.standard_normal((1, 12, 3))
    score = np.full((1, 12, 3), 0.7)
    ref = kv.reshape(1, 3, 4, 3).mean(axis=2)
    np.testing.assert_allclose(orc.compress(kv, score, 4), ref, rtol=0, atol=1e-14)


def test_compress_dominant_score_selects_token():
    rng = np.random.default_rng(3)
    kv = rng.standard_normal((1, 8, 4))
    score = np.zeros((1, 8, 4))
    score[0, 2, :] = 800.0   # block 0 -> token 2
    score[0, 4, :] = 800.0   # block 1 -> token 4
    out = orc.compress(kv, score, 4)
    np.testing.assert_allclose(out[0, 0], kv[0, 2], atol=1e-12)
    np.testing.assert_allclose(out[0, 1], kv[0, 4], atol=1e-12)


def test_compress_scalar_score_broadcasts():
    rng = np.random.default_rng(4)
    kv = rng.standard_normal((2, 8, 6))
    s1 = rng.standard_normal((2, 8, 1))
    np.testing.assert_allclose(orc.compress(kv, s1, 4), orc.compress(kv, np.repeat(s1, 6, 2), 4),
                               atol=1e-15)


def test_compress_rounds_once_to_storage():
    rng = np.random.default_rng(5)
    kv = orc.round_bf16(rng.standard_normal((1, 16, 8)))
    score = orc.round_bf16(rng.standard_normal((1, 16, 8)))
    exact = orc.compress(kv, score, 4)
    stored = orc.compress(kv, score, 4, out_dtype="bf16")
    np.testing.assert_array_equal(stored, orc.round_bf16(exact))
    assert np.abs(stored - exact).max() <= 2.0 ** -8 * np.abs(exact).max()


@pytest.mark.parametrize("d_s", [1, 3])
def test_compress_bwd_finite_differences(d_s):
    rng = np.random.default_rng(6)
    b, sq, d, r = 1, 7, 3, 3   # token 6 is past the last block: zero gradient
    kv = rng.standard_normal((b, sq, d))
    score = rng.standard_normal((b, sq, d_s))
    g = rng.standard_normal((b, sq // r, d))
    dkv, dscore = orc.compress_bwd(kv, score, r, g)
    h = 1e-6

    def loss(kv_, sc_):
        return float((orc.compress(kv_, sc_, r) * g).sum())
    for arr, grad in ((kv, dkv), (score, dscore)):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a0 = arr[i]
            arr[i] = a0 + h
            lp = loss(kv, score)
            arr[i] = a0 - h
            lm = loss(kv, score)
            arr[i] = a0
            fd[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-8)
    assert np.all(dkv[0, 6] == 0) and np.all(dscore[0, 6] == 0)


# overlapping compression (coff = 2): entry j pools blocks j-1 and j

def test_compress_overlap_is_shifted_double_ratio_pooling():
    """Odd entries pool the non-overlapping 2r-blocks of the sequence, even
    entries (j >= 2) those of the sequence shifted by r tokens, entry 0 the
    first r-block alone: three independent non-overlapping poolings."""
    rng = np.random.default_rng(7)
    r, sq, d = 4, 37, 5
    kv = rng.standard_normal((2, sq, d))
    score = rng.standard_normal((2, sq, d)) * 3
    out = orc.compress(kv, score, r, coff=2)
    n_c = sq // r
    assert out.shape == (2, n_c, d)
    odd = orc.compress(kv, score, 2 * r)                       # entries 1, 3, 5, ...
    even = orc.compress(kv[:, r:], score[:, r:], 2 * r)        # entries 2, 4, ...
    np.testing.assert_allclose(out[:, 1::2], odd[:, :len(range(1, n_c, 2))], atol=1e-14)
    np.testing.assert_allclose(out[:, 2::2], even[:, :len(range(2, n_c, 2))], atol=1e-14)
    np.testing.assert_allclose(out[:, 0], orc.compress(kv[:, :r], score[:, :r], r)[:, 0],
                               atol=1e-14)


def test_compress_overlap_constant_score_is_window_mean():
    rng = np.random.default_rng(8)
    kv = rng.standard_normal((1, 16, 3))
    out = orc.compress(kv, np.full((1, 16, 1), -2.5), 4, coff=2)
    np.testing.assert_allclose(out[0, 0], kv[0, 0:4].mean(axis=0), atol=1e-14)
    for j in range(1, 4):
        np.testing.assert_allclose(out[0, j], kv[0, 4 * j - 4:4 * j + 4].mean(axis=0), atol=1e-14)


@pytest.mark.parametrize("d_s", [1, 3])
def test_compress_overlap_bwd_finite_differences(d_s):
    rng = np.random.default_rng(9)
    b, sq, d, r = 1, 11, 3, 3   # tokens 9, 10 are past the last block: zero gradient
    kv = rng.standard_normal((b, sq, d))
    score = rng.standard_normal((b, sq, d_s))
    g = rng.standard_normal((b, sq // r, d))
    dkv, dscore = orc.compress_bwd(kv, score, r, g, coff=2)
    h = 1e-6

    def loss(kv_, sc_):
        return float((orc.compress(kv_, sc_, r, coff=2) * g).sum())
    for arr, grad in ((kv, dkv), (score, dscore)):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a0 = arr[i]
            arr[i] = a0 + h
            lp = loss(kv, score)
            arr[i] = a0 - h
            lm = loss(kv, score)
            arr[i] = a0
            fd[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-8)
    assert np.all(dkv[0, 9:] == 0) and np.all(dscore[0, 9:] == 0)


# ---------------------------------------------------------------------------
# indexer and top-k
# ---------------------------------------------------------------------------

def test_visible_blocks_values():
    # positions 1..8 // 4 -> 0,0,0,1,1,1,1,2
    assert [orc.visible_blocks(t, 4) for t in range(8)] == [0, 0, 0, 1, 1, 1, 1, 2]


def test_indexer_golden():
    g = _load("indexer_tiny.json")
    I = orc.indexer_scores(np.array(g["q_I"]), np.array(g["k_I"]), np.array(g["w"]), g["ratio"])
    exp = g["expected_rows"]
    for t, row in enumerate(exp):
        np.testing.assert_allclose(I[0, t, :len(row)], _ev(row), atol=1e-15)
        assert np.all(np.isneginf(I[0, t, len(row):]))


def test_indexer_single_head_unit_weight_is_relu_matmul():
    rng = np.random.default_rng(7)
    b, sq, d_I, r = 2, 24, 5, 3
    q_I = rng.standard_normal((b, sq, 1, d_I))
    k_I = rng.standard_normal((b, sq // r, d_I))
    w = np.ones((b, sq, 1))
    I = orc.indexer_scores(q_I, k_I, w, r)
    for bi in range(b):
        full = np.maximum(q_I[bi, :, 0] @ k_I[bi].T, 0)
        for t in range(sq):
            v = (t + 1) // r
            np.testing.assert_allclose(I[bi, t, :v], full[t, :v], atol=1e-13)
            assert np.all(np.isneginf(I[bi, t, v:]))


def test_indexer_linear_in_w_and_homogeneous_in_q():
    rng = np.random.default_rng(8)
    b, sq, H, d_I, r = 1, 16, 3, 4, 2
    q_I = rng.standard_normal((b, sq, H, d_I))
    k_I = rng.standard_normal((b, sq // r, d_I))
    w1 = rng.standard_normal((b, sq, H))
    w2 = rng.standard_normal((b, sq, H))
    fin = lambda x: np.where(np.isfinite(x), x, 0)
    I1 = fin(orc.indexer_scores(q_I, k_I, w1, r))
    I2 = fin(orc.indexer_scores(q_I, k_I, w2, r))
    I12 = fin(orc.indexer_scores(q_I, k_I, w1 + w2, r))
    np.testing.assert_allclose(I12, I1 + I2, atol=1e-12)
    np.testing.assert_allclose(fin(orc.indexer_scores(q_I, k_I, -w1, r)), -I1, atol=1e-12)
    np.testing.assert_allclose(fin(orc.indexer_scores(2.5 * q_I, k_I, w1, r)), 2.5 * I1, atol=1e-12)
    # ReLU: flipping q changes the score unless every dot is zero
    assert not np.allclose(fin(orc.indexer_scores(-q_I, k_I, w1, r)), -I1)


def test_topk_golden():
    g = _load("topk_tiny.json")
    s = np.array(g["scores"])
    for c in g["cases"]:
        assert orc.topk_select_row(s, c["K"]).tolist() == c["expected"]


def _brute_topk(scores, K):
    """Enumerate all subsets of size min(K, v); keep those in which every member
    beats every non-member under (score desc, index asc)."""
    v = len(scores)
    k = min(K, v)
    better = lambda i, j: scores[i] > scores[j] or (scores[i] == scores[j] and i < j)
    found = [S for S in itertools.combinations(range(v), k)
             if all(better(i, j) for i in S for j in range(v) if j not in S)]
    assert len(found) == 1
    return list(found[0]) + [-1] * (K - k)


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(9)
    for trial in range(300):
        v = int(rng.integers(0, 9))
        K = int(rng.integers(1, 7))
        s = rng.integers(-2, 3, size=v).astype(np.float64)   # many exact ties
        assert orc.topk_select_row(s, K).tolist() == _brute_topk(list(s), K)


def test_topk_ties_from_relu_zeros_and_duplicate_keys():
    rng = np.random.default_rng(10)
    b, sq, H, d_I, r, K = 1, 40, 2, 4, 2, 5
    q_I = np.abs(rng.standard_normal((b, sq, H, d_I)))
    k_I = rng.standard_normal((b, sq // r, d_I))
    k_I[0, 3] = k_I[0, 7]                  # duplicate key rows -> exact ties
    k_I[0, 10] = -np.abs(k_I[0, 10])       # all dots negative -> ReLU zeros
    k_I[0, 11] = -np.abs(k_I[0, 11])
    w = np.abs(rng.standard_normal((b, sq, H)))
    I = orc.indexer_scores(q_I, k_I, w, r)
    idx = orc.topk_select(I, K)
    for t in range(sq):
        v = (t + 1) // r
        assert idx[0, t].tolist() == _brute_topk(list(I[0, t, :v]), K)
    assert I[0, sq - 1, 3] == I[0, sq - 1, 7]
    assert I[0, sq - 1, 10] == 0.0 and I[0, sq - 1, 11] == 0.0


# ---------------------------------------------------------------------------
# attention: dense masked attention through torch's SDPA in float64
# ---------------------------------------------------------------------------

def _dense_sdpa(q, kv, idx, sink, scale, window, ratio, dO=None, doc_ids=None):
    """The same layer as dense attention over all n_kv rows plus one sink key,
    with an explicit additive mask: log(multiplicity) for allowed rows, -inf
    elsewhere (window rows of another document are not allowed).  Evaluated by
    torch.nn.functional.scaled_dot_product_attention in float64; gradients by
    torch autograd."""
    b, sq, H, d = q.shape
    n_kv = kv.shape[1]
    n_c = n_kv - sq
    count = np.zeros((b, sq, n_kv))
    for bi in range(b):
        for t in range(sq):
            count[bi, t, max(0, t - window + 1):t + 1] = 1.0
            if doc_ids is not None:
                count[bi, t, :sq] *= doc_ids[bi] == doc_ids[bi, t]
            for j in idx[bi, t]:
                if 0 <= j < n_c and j < (t + 1) // ratio:
                    count[bi, t, sq + j] += 1.0
    with np.errstate(divide="ignore"):
        bias = np.log(count)
    bias = np.concatenate([bias, np.zeros((b, sq, 1))], axis=2)          # sink column
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kvt = torch.tensor(kv, dtype=torch.float64, requires_grad=True)
    has_sink = sink is not None
    st = torch.tensor(sink if has_sink else np.zeros(H), dtype=torch.float64, requires_grad=True)
    qh = qt.permute(0, 2, 1, 3)                                          # [b,H,sq,d]
    q_ext = torch.cat([qh, torch.ones(b, H, sq, 1, dtype=torch.float64)], dim=3)
    k_rows = torch.cat([kvt, torch.zeros(b, n_kv, 1, dtype=torch.float64)], dim=2)
    k_rows = k_rows.unsqueeze(1).expand(b, H, n_kv, d + 1)
    k_sink = torch.cat([torch.zeros(H, d, dtype=torch.float64), (st / scale).view(H, 1)], dim=1)
    k_ext = torch.cat([k_rows, k_sink.view(1, H, 1, d + 1).expand(b, H, 1, d + 1)], dim=2)
    v_ext = torch.cat([kvt.unsqueeze(1).expand(b, H, n_kv, d),
                       torch.zeros(b, H, 1, d, dtype=torch.float64)], dim=2)
    mask = torch.tensor(bias).view(b, 1, sq, n_kv + 1)
    if not has_sink:
        mask = mask.clone()
        mask[..., -1] = -math.inf
    o = torch.nn.functional.scaled_dot_product_attention(q_ext, k_ext, v_ext, attn_mask=mask,
                                                         scale=scale)
    logits = scale * (q_ext @ k_ext.transpose(-1, -2)) + mask
    lse = torch.logsumexp(logits, dim=-1)                                # [b,H,sq]
    O = o.permute(0, 2, 1, 3)
    res = {"O": O.detach().numpy(), "LSE": lse.permute(0, 2, 1).detach().numpy()}
    if dO is not None:
        (O * torch.tensor(dO)).sum().backward()
        res["dq"] = qt.grad.numpy()
        res["dkv"] = kvt.grad.numpy()
        res["dsink"] = st.grad.numpy() if has_sink else np.zeros(H)
    return res


def _random_case(seed, b=2, sq=24, H=3, d=5, ratio=4, window=5, K=4, sink=True):
    rng = np.random.default_rng(seed)
    n_c = sq // ratio
    q = rng.standard_normal((b, sq, H, d))
    kv = rng.standard_normal((b, sq + n_c, d))
    # repeated indices, -1 padding, out-of-range and not-yet-visible entries
    idx = rng.integers(-1, n_c + 2, size=(b, sq, K)).astype(np.int32)
    idx[:, :, 1] = idx[:, :, 0]
    snk = rng.standard_normal(H) if sink else None
    dO = rng.standard_normal((b, sq, H, d))
    return q, kv, idx, snk, d ** -0.5, window, ratio, dO


@pytest.mark.parametrize("sink", [True, False])
def test_attn_matches_dense_sdpa(sink):
    q, kv, idx, snk, scale, W, r, dO = _random_case(11, sink=sink)
    O, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
    dq, dkv, dsink = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO)
    ref = _dense_sdpa(q, kv, idx, snk, scale, W, r, dO)
    np.testing.assert_allclose(O, ref["O"], atol=1e-12)
    np.testing.assert_allclose(L, ref["LSE"], atol=1e-12)
    np.testing.assert_allclose(dq, ref["dq"], atol=1e-12)
    np.testing.assert_allclose(dkv, ref["dkv"], atol=1e-12)
    np.testing.assert_allclose(dsink, ref["dsink"], atol=1e-12)


def test_attn_reduces_to_causal_dense_attention():
    """sink = -inf, every visible block selected, window = sq: plain masked
    attention over kv_full with M[t,i] = (i <= t) for raw rows and
    (i - sq < vis(t)) for compressed rows."""
    rng = np.random.default_rng(12)
    b, sq, H, d, r = 1, 16, 2, 4, 4
    n_c = sq // r
    q = rng.standard_normal((b, sq, H, d))
    kv = rng.standard_normal((b, sq + n_c, d))
    idx = np.tile(np.arange(n_c, dtype=np.int32), (b, sq, 1))
    O, L = orc.attn_fwd(q, kv, idx, None, 0.5, sq, r)
    for t in range(sq):
        allowed = [i for i in range(sq) if i <= t] + [sq + j for j in range(n_c) if j < (t + 1) // r]
        s = 0.5 * q[0, t] @ kv[0, allowed].T
        p = torch.softmax(torch.tensor(s), dim=1).numpy()
        np.testing.assert_allclose(O[0, t], p @ kv[0, allowed], atol=1e-13)
        np.testing.assert_allclose(L[0, t], torch.logsumexp(torch.tensor(s), 1).numpy(), atol=1e-13)


def test_attn_golden():
    g = _load("attn_tiny.json")
    q = np.array(_ev(g["q"]))
    kv = np.array(_ev(g["kv_full"]))
    idx = np.array(g["idx"], dtype=np.int32)
    sink = np.array(g["sink"])
    dO = np.array(g["dO"])
    O, L = orc.attn_fwd(q, kv, idx, sink, g["scale"], g["window"], g["ratio"])
    dq, dkv, dsink = orc.attn_bwd(q, kv, idx, sink, g["scale"], g["window"], g["ratio"], dO)
    e = g["expected"]
    np.testing.assert_allclose(O, np.array(_ev(e["O"])), atol=1e-14)
    np.testing.assert_allclose(L, np.array(_ev(e["LSE"])), atol=1e-14)
    np.testing.assert_allclose(dq, np.array(_ev(e["dq"])), atol=1e-14)
    np.testing.assert_allclose(dkv, np.array(_ev(e["dkv"])), atol=1e-14)
    np.testing.assert_allclose(dsink, np.array(_ev(e["dsink"])), atol=1e-14)


def test_attn_probabilities_plus_sink_sum_to_one():
    q, kv, idx, snk, scale, W, r, _ = _random_case(13)
    sq, n_c = q.shape[1], kv.shape[1] - q.shape[1]
    for bi in range(q.shape[0]):
        for t in range(sq):
            slots = orc.query_slots(t, idx[bi, t], sq, n_c, r, W)
            _, lse, p, _ = orc.attn_fwd_query(q[bi, t], kv[bi], slots, snk, scale)
            np.testing.assert_allclose(p.sum(axis=1) + np.exp(snk - lse), 1.0, atol=1e-14)


def test_attn_padding_and_batch_independence():
    q, kv, idx, snk, scale, W, r, dO = _random_case(14)
    O, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
    # appending -1 slots changes nothing
    idx_pad = np.concatenate([idx, -np.ones_like(idx)], axis=2)
    O2, L2 = orc.attn_fwd(q, kv, idx_pad, snk, scale, W, r)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(L, L2)
    # b=2 equals two b=1 runs
    for bi in range(2):
        Ob, Lb = orc.attn_fwd(q[bi:bi + 1], kv[bi:bi + 1], idx[bi:bi + 1], snk, scale, W, r)
        np.testing.assert_array_equal(Ob[0], O[bi])
        dqb, dkvb, _ = orc.attn_bwd(q[bi:bi + 1], kv[bi:bi + 1], idx[bi:bi + 1], snk, scale, W, r,
                                    dO[bi:bi + 1])
        dq, dkv, _ = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO)
        np.testing.assert_allclose(dqb[0], dq[bi], atol=1e-14)
        np.testing.assert_allclose(dkvb[0], dkv[bi], atol=1e-14)


def test_attn_large_logits_stable():
    """LSE near 1000 (two keys, two heads): finite results that match the
    dense float64 formulation."""
    rng = np.random.default_rng(15)
    b, sq, H, d, r = 1, 4, 2, 3, 2
    q = rng.standard_normal((b, sq, H, d)) * 300
    kv = rng.standard_normal((b, sq + sq // r, d)) * 3
    idx = np.zeros((b, sq, 1), np.int32)
    snk = np.array([1000.0, -5.0])
    dO = rng.standard_normal((b, sq, H, d))
    O, L = orc.attn_fwd(q, kv, idx, snk, 1.0, 2, r)
    dq, dkv, ds = orc.attn_bwd(q, kv, idx, snk, 1.0, 2, r, dO)
    ref = _dense_sdpa(q, kv, idx, snk, 1.0, 2, r, dO)
    assert np.all(np.isfinite(L)) and np.abs(L).max() > 500
    np.testing.assert_allclose(L, ref["LSE"], rtol=1e-13)
    np.testing.assert_allclose(O, ref["O"], atol=1e-9)
    np.testing.assert_allclose(dq, ref["dq"], atol=1e-7)
    np.testing.assert_allclose(dkv, ref["dkv"], atol=1e-7)
    np.testing.assert_allclose(ds, ref["dsink"], atol=1e-9)


def test_attn_bwd_finite_differences():
    q, kv, idx, snk, scale, W, r, dO = _random_case(16, b=1, sq=9, H=2, d=3, ratio=3, window=3, K=3)
    dq, dkv, dsink = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO)
    h = 1e-6

    def loss():
        O, _ = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
        return float((O * dO).sum())
    for arr, grad in ((q, dq), (kv, dkv), (snk, dsink)):
        for i in np.ndindex(arr.shape):
            a0 = arr[i]
            arr[i] = a0 + h
            lp = loss()
            arr[i] = a0 - h
            lm = loss()
            arr[i] = a0
            assert abs((lp - lm) / (2 * h) - grad[i]) < 1e-7, (i, grad[i])


def test_attn_rows_subset_matches_full():
    q, kv, idx, snk, scale, W, r, dO = _random_case(17)
    O, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
    dq, _, _ = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO)
    rows = [(1, 5), (0, 23), (0, 0)]
    Or, Lr = orc.attn_fwd(q, kv, idx, snk, scale, W, r, rows=rows)
    dqr, _, _ = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO, rows=rows)
    for n, (bi, t) in enumerate(rows):
        np.testing.assert_array_equal(Or[n], O[bi, t])
        np.testing.assert_array_equal(Lr[n], L[bi, t])
        np.testing.assert_allclose(dqr[n], dq[bi, t], atol=1e-15)


# ---------------------------------------------------------------------------
# packed documents (doc_ids)
# ---------------------------------------------------------------------------

def test_attn_doc_window_matches_dense_sdpa():
    """Arbitrary (not contiguous) document ids: the window keeps only rows of
    the query's own document; selected compressed entries are taken as given."""
    q, kv, idx, snk, scale, W, r, dO = _random_case(21, window=7)
    rng = np.random.default_rng(22)
    doc = rng.integers(0, 3, size=q.shape[:2]).astype(np.int32)
    O, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r, doc_ids=doc)
    dq, dkv, dsink = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO, doc_ids=doc)
    ref = _dense_sdpa(q, kv, idx, snk, scale, W, r, dO, doc_ids=doc)
    for name, got in [("O", O), ("LSE", L), ("dq", dq), ("dkv", dkv), ("dsink", dsink)]:
        np.testing.assert_allclose(got, ref[name], atol=1e-12, err_msg=name)
    # one document everywhere is the plain layer
    O1, _ = orc.attn_fwd(q, kv, idx, snk, scale, W, r, doc_ids=np.zeros_like(doc))
    O0, _ = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
    np.testing.assert_array_equal(O1, O0)


def test_indexer_topk_docs_brute_force():
    """Selectable set by explicit loops (j < vis(t) and doc[j*ratio] == doc[t])
    and the brute-force top-k over it, with many exact ties."""
    rng = np.random.default_rng(23)
    b, sq, H, d_I, r, K = 2, 48, 2, 3, 3, 4
    q_I = rng.integers(-1, 2, size=(b, sq, H, d_I)).astype(np.float64)
    k_I = rng.integers(-1, 2, size=(b, sq // r, d_I)).astype(np.float64)
    w = rng.integers(0, 3, size=(b, sq, H)).astype(np.float64)
    doc = rng.integers(0, 3, size=(b, sq)).astype(np.int32)
    I = orc.indexer_scores(q_I, k_I, w, r, doc_ids=doc)
    idx = orc.topk_select(I, K)
    for bi in range(b):
        for t in range(sq):
            cand = [j for j in range(sq // r) if j < (t + 1) // r and doc[bi, j * r] == doc[bi, t]]
            vals = [sum(w[bi, t, h] * max(0.0, float(q_I[bi, t, h] @ k_I[bi, j])) for h in range(H))
                    for j in cand]
            sel = [cand[i] for i in _brute_topk(vals, K) if i >= 0]
            assert idx[bi, t].tolist() == sorted(sel) + [-1] * (K - len(sel))


def test_packed_documents_equal_separate_runs():
    """Documents packed into one sequence (boundaries on multiples of ratio)
    give, for every document, exactly the results of running that document
    alone: indexer + top-k (block ids shifted by the document's first block),
    attention forward and backward (dkv rows and dsink summed over documents)."""
    from compressed_sparse_attention_sum_gb300.inputs import packed_doc_ids
    rng = np.random.default_rng(24)
    b, sq, H, d, r, W, K, H_I, d_I = 1, 40, 2, 4, 4, 6, 3, 2, 3
    n_c = sq // r
    doc = packed_doc_ids(b, sq, r, 3, seed=5).numpy()
    q_I = rng.standard_normal((b, sq, H_I, d_I))
    k_I = rng.standard_normal((b, n_c, d_I))
    w = rng.standard_normal((b, sq, H_I))
    q = rng.standard_normal((b, sq, H, d))
    kv_raw = rng.standard_normal((b, sq, d))
    kv_c = rng.standard_normal((b, n_c, d))
    kv = np.concatenate([kv_raw, kv_c], axis=1)
    snk = rng.standard_normal(H)
    dO = rng.standard_normal((b, sq, H, d))
    scale = d ** -0.5
    idx = orc.topk_select(orc.indexer_scores(q_I, k_I, w, r, doc_ids=doc), K)
    O, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r, doc_ids=doc)
    dq, dkv, dsink = orc.attn_bwd(q, kv, idx, snk, scale, W, r, dO, doc_ids=doc)
    starts = [0] + [t for t in range(1, sq) if doc[0, t] != doc[0, t - 1]]
    ends = starts[1:] + [sq]
    assert len(starts) == 3
    dsink_sum = np.zeros(H)
    for a, e in zip(starts, ends):
        ja, nc_s = a // r, (e - a) // r
        idx_s = orc.topk_select(orc.indexer_scores(q_I[:, a:e], k_I[:, ja:ja + nc_s], w[:, a:e], r), K)
        np.testing.assert_array_equal(np.where(idx_s >= 0, idx_s + ja, -1), idx[:, a:e])
        kv_s = np.concatenate([kv_raw[:, a:e], kv_c[:, ja:ja + nc_s]], axis=1)
        O_s, L_s = orc.attn_fwd(q[:, a:e], kv_s, idx_s, snk, scale, W, r)
        dq_s, dkv_s, ds_s = orc.attn_bwd(q[:, a:e], kv_s, idx_s, snk, scale, W, r, dO[:, a:e])
        np.testing.assert_allclose(O[:, a:e], O_s, atol=1e-12)
        np.testing.assert_allclose(L[:, a:e], L_s, atol=1e-12)
        np.testing.assert_allclose(dq[:, a:e], dq_s, atol=1e-12)
        np.testing.assert_allclose(dkv[:, a:e], dkv_s[:, :e - a], atol=1e-12)
        np.testing.assert_allclose(dkv[:, sq + ja:sq + ja + nc_s], dkv_s[:, e - a:], atol=1e-12)
        dsink_sum += ds_s
    np.testing.assert_allclose(dsink, dsink_sum, atol=1e-12)


# ---------------------------------------------------------------------------
# indexer training path (teacher, student rescoring, KL)
# ---------------------------------------------------------------------------

def _teacher_by_head_mass(q, kv, idx, sink, scale, window, ratio):
    """The teacher the other way round (review of the teacher normalization
    in "Add unfused SBHD compressed sparse attention"): per head, the
    compressed mass m_h = sigmoid(lse_compressed - lse_window_and_sink) times
    the softmax over the compressed entries, summed over heads and
    L1-normalized.  Log-space throughout; no attention LSE is used."""
    b, sq, H, d = q.shape
    n_c = kv.shape[1] - sq
    K = idx.shape[2]
    out = np.zeros((b, sq, K))
    for bi in range(b):
        for t in range(sq):
            pos, js = orc.selected_entries(idx[bi, t], t, n_c, ratio)
            if pos.size == 0:
                continue
            rows = list(range(max(0, t - window + 1), t + 1))
            lw = scale * q[bi, t] @ kv[bi, rows].T                       # [H, W]
            l_nc = np.logaddexp(np.log(np.exp(lw - lw.max(1, keepdims=True)).sum(1))
                                + lw.max(1), sink)
            lc = scale * q[bi, t] @ kv[bi, sq + js].T                    # [H, n]
            l_c = np.log(np.exp(lc - lc.max(1, keepdims=True)).sum(1)) + lc.max(1)
            soft = np.exp(lc - l_c[:, None])
            log_m = -np.logaddexp(0.0, -(l_c - l_nc))                    # log sigmoid
            T = (np.exp(log_m - log_m.max())[:, None] * soft).sum(0)
            out[bi, t, pos] = T / T.sum()
    return out


def test_teacher_matches_head_mass_formula():
    q, kv, idx, snk, scale, W, r, _ = _random_case(41, window=6, K=5)
    _, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
    T = orc.indexer_teacher(q, kv, idx, L, scale, r)
    np.testing.assert_allclose(T, _teacher_by_head_mass(q, kv, idx, snk, scale, W, r), atol=1e-12)
    s = T.sum(axis=2)
    assert np.all((np.abs(s - 1) < 1e-12) | (s == 0))


def test_teacher_survives_window_dominated_rows():
    """Window logits about 1000 above every compressed logit: exp(logit - lse)
    underflows even in float64, yet the shifted teacher is the proper
    distribution (the conditional softmax weighted by the log-space masses)."""
    q, kv, idx, snk, scale, W, r, _ = _random_case(42, b=1, sq=24, H=2, window=4, K=3)
    kv[:, :24] *= 0.0
    kv[:, :24, 0] = 1.0
    kv[:, 24:, 0] = 0.0
    q[..., 0] = 1000.0 / scale                     # window logits = 1000, compressed ones O(1)
    _, L = orc.attn_fwd(q, kv, idx, snk, scale, W, r)
    lc = scale * np.einsum("hd,nd->hn", q[0, 23], kv[0, 24:])
    assert np.all(np.exp(lc - L[0, 23][:, None]) == 0.0)       # the plain form underflows
    T = orc.indexer_teacher(q, kv, idx, L, scale, r)
    ref = _teacher_by_head_mass(q, kv, idx, snk, scale, W, r)
    np.testing.assert_allclose(T, ref, atol=1e-12)
    has = np.array([orc.selected_entries(idx[0, t], t, 24 // r, r)[0].size > 0 for t in range(24)])
    assert has.any() and np.allclose(T[0, has].sum(1), 1.0)
    assert np.all(T[0, ~has] == 0.0)


def test_indexer_loss_matches_autograd():
    """Student rescoring + KL against torch autograd in float64 (log_softmax
    over each row's valid slots), with repeated and invalid entries."""
    rng = np.random.default_rng(43)
    b, sq, H_I, d_I, r, K = 2, 20, 3, 4, 2, 6
    n_c = sq // r
    q_I = rng.standard_normal((b, sq, H_I, d_I))
    k_I = rng.standard_normal((b, n_c, d_I))
    w = rng.standard_normal((b, sq, H_I))
    idx = rng.integers(-1, n_c + 1, size=(b, sq, K)).astype(np.int32)
    idx[:, :, 1] = idx[:, :, 0]
    target = np.zeros((b, sq, K))
    for bi in range(b):
        for t in range(sq):
            pos, _ = orc.selected_entries(idx[bi, t], t, n_c, r)
            if pos.size:
                v = rng.random(pos.size)
                v[0] = 0.0                                   # a zero-target slot
                target[bi, t, pos] = v / v.sum() if v.sum() > 0 else 0.0
    loss, dq, dk, dw = orc.indexer_loss(q_I, k_I, w, idx, target, r)
    qt = torch.tensor(q_I, requires_grad=True)
    kt = torch.tensor(k_I, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    total = torch.zeros((), dtype=torch.float64)
    ref_loss = np.zeros((b, sq))
    for bi in range(b):
        for t in range(sq):
            pos, js = orc.selected_entries(idx[bi, t], t, n_c, r)
            if pos.size == 0:
                continue
            dots = qt[bi, t] @ kt[bi, torch.tensor(js)].T
            I = wt[bi, t] @ torch.relu(dots)
            logp = torch.log_softmax(I, dim=0)
            tg = torch.tensor(target[bi, t, pos])
            nz = tg > 0
            row = (tg[nz] * (torch.log(tg[nz]) - logp[nz])).sum()
            ref_loss[bi, t] = row.item()
            total = total + row
    total.backward()
    np.testing.assert_allclose(loss, ref_loss, atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), atol=1e-12)


def test_indexer_loss_zero_target_row_has_zero_gradient():
    rng = np.random.default_rng(44)
    q_I = rng.standard_normal((1, 8, 2, 3))
    k_I = rng.standard_normal((1, 4, 3))
    w = rng.standard_normal((1, 8, 2))
    idx = np.tile(np.arange(3, dtype=np.int32), (1, 8, 1))
    loss, dq, dk, dw = orc.indexer_loss(q_I, k_I, w, idx, np.zeros((1, 8, 3)), 2)
    assert np.all(loss == 0) and np.all(dq == 0) and np.all(dk == 0) and np.all(dw == 0)
    # a normalized target equal to the student's own distribution: zero gradient
    I = orc.indexer_student_row(q_I[0, 7], k_I[0], w[0, 7], idx[0, 7], 7, 2)
    p = np.exp(I - I.max()) / np.exp(I - I.max()).sum()
    l, dI = orc.indexer_kl_row(I, p)
    assert abs(l) < 1e-14 and np.abs(dI).max() < 1e-15


# ---------------------------------------------------------------------------
# FP8 (e4m3) indexer
# ---------------------------------------------------------------------------

def test_round_e4m3_matches_torch_float8():
    """torch's float8_e4m3fn conversion (round to nearest even) on values
    inside the finite range, including ties and subnormals."""
    rng = np.random.default_rng(61)
    vals = np.concatenate([
        rng.standard_normal(4000) * 50,
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 1000),                  # subnormal range
        np.array([0.0, 1.0625, 1.1875, 232.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -10]),
    ])
    vals = np.clip(vals, -448.0, 448.0).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(orc.round_e4m3(vals.astype(np.float64)), ref)


def test_quantize_rows_e4m3_properties():
    rng = np.random.default_rng(62)
    x = (rng.standard_normal((50, 128)) * rng.uniform(0.01, 100, (50, 1))).astype(np.float32)
    x[3] = 0.0
    q, sc = orc.quantize_rows_e4m3(x)
    amax_pos = np.abs(x).argmax(axis=1)
    for i in range(50):
        if i == 3:
            assert sc[i] == 0 and np.all(q[i] == 0)
            continue
        assert abs(q[i, amax_pos[i]]) == 448.0                 # the largest entry maps to 448
        # every code is an e4m3 value within half an e4m3 step of x * 448 / amax
        y = x[i].astype(np.float64) * 448.0 / np.abs(x[i]).max()
        assert np.all(np.abs(q[i] - y) <= np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) + 1e-4)
        np.testing.assert_array_equal(q[i], orc.round_e4m3(q[i]))


def test_indexer_scores_fp8_reduce_to_plain_scores():
    """With rows already on the e4m3 grid and unit scales, the fp8 scores are
    the plain indexer scores; scales factor out of the ReLU."""
    rng = np.random.default_rng(63)
    b, sq, H, d, r = 1, 24, 3, 16, 4
    q = orc.round_e4m3(rng.integers(-6, 7, (b, sq, H, d)).astype(np.float64))
    k = orc.round_e4m3(rng.integers(-6, 7, (b, sq // r, d)).astype(np.float64))
    w = rng.standard_normal((b, sq, H))
    ones_q, ones_k = np.ones((b, sq, H)), np.ones((b, sq // r))
    np.testing.assert_allclose(orc.indexer_scores_fp8(q, ones_q, k, ones_k, w, r),
                               orc.indexer_scores(q, k, w, r), atol=1e-12)
    sq_s, sk_s = rng.uniform(0.5, 2, (b, sq, H)), rng.uniform(0.5, 2, (b, sq // r))
    ref = orc.indexer_scores(q * sq_s[..., None], k * sk_s[..., None], w, r)
    np.testing.assert_allclose(orc.indexer_scores_fp8(q, sq_s, k, sk_s, w, r), ref, atol=1e-9)


# ---------------------------------------------------------------------------
# normalization and rotary embedding of the pooled rows
# ---------------------------------------------------------------------------

def test_kv_norm_unit_weight_has_the_closed_form_rms():
    """Weight 1, no rotation: each row is x / sqrt(mean(x^2) + eps), so its
    mean square is ms / (ms + eps) and x is recovered by the RMS factor."""
    rng = np.random.default_rng(40)
    x = rng.normal(size=(2, 5, 24)) * rng.uniform(0.1, 10, size=(2, 5, 1))
    eps = 1e-3
    y = orc.kv_norm_rope(x, np.ones(24), eps, 0, 40000.0, 4)
    ms = (x ** 2).sum(axis=2) / 24
    assert np.allclose((y ** 2).sum(axis=2) / 24, ms / (ms + eps), rtol=1e-12)
    assert np.allclose(y * np.sqrt(ms + eps)[..., None], x, rtol=1e-12)


def test_kv_norm_weight_scales_each_channel():
    rng = np.random.default_rng(41)
    x = rng.normal(size=(1, 3, 16))
    w = rng.normal(size=16)
    y1 = orc.kv_norm_rope(x, np.ones(16), 1e-6, 0, 40000.0, 4)
    yw = orc.kv_norm_rope(x, w, 1e-6, 0, 40000.0, 4)
    assert np.allclose(yw, y1 * w, rtol=1e-12, atol=0)


def test_rope_is_complex_multiplication_of_interleaved_pairs():
    """The rotary part equals (y[2i] + i y[2i+1]) * exp(i pos theta_i) with
    pos = (j+1)*ratio - 1 and theta_i = 40000^(-i/(rope_dim/2)), evaluated
    with numpy complex arithmetic; the other channels are untouched."""
    rng = np.random.default_rng(42)
    d, rd, ratio, n_c = 32, 12, 4, 7
    x = rng.normal(size=(2, n_c, d))
    w = rng.normal(size=d)
    plain = orc.kv_norm_rope(x, w, 1e-6, 0, 40000.0, ratio)
    got = orc.kv_norm_rope(x, w, 1e-6, rd, 40000.0, ratio)
    assert np.array_equal(got[..., :d - rd], plain[..., :d - rd])
    z = plain[..., d - rd::2] + 1j * plain[..., d - rd + 1::2]
    pos = np.array([(j + 1) * ratio - 1 for j in range(n_c)], np.float64)
    freq = 1.0 / 40000.0 ** (np.arange(rd // 2) / (rd // 2))
    zr = z * np.exp(1j * pos[:, None] * freq[None, :])
    assert np.allclose(got[..., d - rd::2], zr.real, atol=1e-12)
    assert np.allclose(got[..., d - rd + 1::2], zr.imag, atol=1e-12)


def test_rope_depends_only_on_relative_position():
    """Rows with identical content: the rotary parts' inner products depend
    only on the distance between the rows, and each pair keeps its norm."""
    rng = np.random.default_rng(43)
    d, rd, ratio, n_c = 16, 16, 4, 9
    u = rng.normal(size=d)
    x = np.broadcast_to(u, (1, n_c, d)).copy()
    y = orc.kv_norm_rope(x, np.ones(d), 0.0, rd, 40000.0, ratio)[0]
    dots = y @ y.T
    for k in range(1, 5):
        diag = np.diagonal(dots, offset=k)
        assert np.allclose(diag, diag[0], rtol=1e-10)
    pair = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    assert np.allclose(pair, pair[0], rtol=1e-12)


def test_rope_at_position_zero_is_identity():
    """ratio 1: entry 0 sits at position 0, where every angle is 0."""
    rng = np.random.default_rng(44)
    x = rng.normal(size=(1, 3, 16))
    w = rng.normal(size=16)
    a = orc.kv_norm_rope(x, w, 1e-6, 16, 40000.0, 1)
    b = orc.kv_norm_rope(x, w, 1e-6, 0, 40000.0, 1)
    assert np.array_equal(a[:, 0], b[:, 0]) and not np.allclose(a[:, 1], b[:, 1])


def test_kv_norm_rope_bwd_matches_torch_autograd():
    """Gradients against float64 autograd of torch's own RMS norm and a
    complex-number rotation (torch.view_as_complex / torch.polar)."""
    rng = np.random.default_rng(45)
    b, n_c, d, rd, ratio, eps = 2, 6, 32, 16, 4, 1e-5
    x = rng.normal(size=(b, n_c, d))
    w = rng.normal(size=d)
    g = rng.normal(size=(b, n_c, d))
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    y = torch.nn.functional.rms_norm(xt, (d,), weight=wt, eps=eps)
    pos = torch.tensor([(j + 1) * ratio - 1 for j in range(n_c)], dtype=torch.float64)
    freq = 40000.0 ** (-torch.arange(rd // 2, dtype=torch.float64) / (rd // 2))
    rot = torch.polar(torch.ones(n_c, rd // 2, dtype=torch.float64), pos[:, None] * freq[None])
    zc = torch.view_as_complex(y[..., d - rd:].reshape(b, n_c, rd // 2, 2).contiguous()) * rot
    out = torch.cat([y[..., :d - rd], torch.view_as_real(zc).reshape(b, n_c, rd)], dim=-1)
    out.backward(torch.tensor(g))
    assert np.allclose(orc.kv_norm_rope(x, w, eps, rd, 40000.0, ratio), out.detach().numpy(),
                       atol=1e-12)
    dx, dw = orc.kv_norm_rope_bwd(x, w, eps, rd, 40000.0, ratio, g)
    assert np.allclose(dx, xt.grad.numpy(), atol=1e-10)
    assert np.allclose(dw, wt.grad.numpy(), atol=1e-10)


def test_kv_norm_rope_bwd_finite_differences():
    rng = np.random.default_rng(46)
    b, n_c, d, rd, ratio, eps = 1, 3, 8, 4, 2, 1e-4
    x = rng.normal(size=(b, n_c, d))
    w = rng.normal(size=d)
    g = rng.normal(size=(b, n_c, d))
    dx, dw = orc.kv_norm_rope_bwd(x, w, eps, rd, 40000.0, ratio, g)
    f = lambda xx, ww: float((orc.kv_norm_rope(xx, ww, eps, rd, 40000.0, ratio) * g).sum())
    h = 1e-6
    for idx in [(0, 0, 0), (0, 1, 5), (0, 2, 7), (0, 2, 3)]:
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert abs((f(xp, w) - f(xm, w)) / (2 * h) - dx[idx]) < 1e-7
    for c in (0, 6):
        wp, wm = w.copy(), w.copy()
        wp[c] += h
        wm[c] -= h
        assert abs((f(x, wp) - f(x, wm)) / (2 * h) - dw[c]) < 1e-7
