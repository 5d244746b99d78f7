"""fp64 CPU oracle of the Compressed Sparse Attention (CSA) hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module: only
the tests, the smoke check of ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library (no
helpers, tables or constants); both sides only share the seeded input
generator, which computes none of the method's arithmetic.

Every function is the plain definition written out in float64 with numpy,
one query row at a time, in the order the pages describe the step.  Inputs
are read as stored (bf16 values widen exactly to float64).  Sources, by
page title and section:

* "Add unfused SBHD compressed sparse attention" (Megatron-LM PR #6400):
  compressor review (softmax-weighted pooling in fp32, cast once),
  causal compressed mask (block j visible to token t iff j < (t+1)//ratio),
  indexer/top-k block (k = min(index_topk, n_compressed), validity + offset,
  -1 padding), review of the gather backward (compact [b*n_kv, hn] KV buffer,
  index_add backward, repeated indices), attention-sink parameter (per-head
  fp32 logit), softmax_scale default v_head_dim**-0.5.
* "Refactor Deepseek v4 to use Attention Gym's Compressed Sparse Attention"
  (torchtitan PR #4452): one softmax over window + selected compressed
  entries + sink, returning the per-head LSE (the sink is in the
  denominator, contributes no value).
  Packed documents (same page, the selected_attention commit message): with
  per-token doc_ids, the window branch keeps key k for query t only when
  doc_ids[k] == doc_ids[t]; compressed block j covers tokens
  [j*ratio, (j+1)*ratio), belongs to doc_ids[j*ratio], and the indexer may
  select it for t only when doc_ids[t] == doc_ids[j*ratio] (and j < vis(t)).
  The attention takes the selected entries as given (the caller's indexer
  already filtered them).
* "Add the min-memory DSA attention kernels" (Megatron-LM PR #7152): exact
  ties after ReLU are common and routing must be tie-exact with one full
  top-k; the selected support is sorted by position; repeated keys
  accumulate their gradients in fp32.

Readings where the pages are silent (each one is listed with its reason in
the design notes of the repository):
  * window of query t = raw rows {t-W+1, ..., t} (its own token included);
  * KV row order = raw rows 0..sq-1 then compressed rows sq..sq+n_c-1;
  * tokens past the last complete block are never pooled;
  * top-k ties go to the lower block index; output ascending, -1 tail;
  * an index j is padding when j < 0, j >= n_c or j >= vis(t);
  * a repeated index is two separate softmax terms;
  * LSE = natural log including the sink; sink absent = -inf;
  * overlapping compression: coff counts the ratio-blocks an entry pools,
    ending with its own block (coff = 1 is the non-overlapping compressor the
    compressor review names);
  * FP8 indexer: per-row e4m3 codes with scale absmax / 448 (the pages list
    indexer quantization only as not yet included).
  * normalization of the pooled rows: RMS normalization over the d channels
    with a per-channel weight, on the pooled row after its one cast, result
    cast once more (the compressor review shows kv = self.norm(kv) after the
    cast; the norm's type is not shown);
  * rotary embedding of the pooled rows: interleaved channel pairs
    (2i, 2i+1) of the last rope_dim channels, angle pos * base^(-2i/rope_dim),
    entry j at the position of the last token it pools, (j+1)*ratio - 1
    (the pages give only the base, 40000, "for compressed KV positions").

All functions take and return numpy arrays; floating results are float64.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_storage", "round_bf16",
    "visible_blocks", "pooling_window", "compress", "compress_bwd",
    "indexer_selectable", "indexer_scores", "indexer_scores_row", "topk_select", "topk_select_row",
    "query_slots", "attn_fwd_query", "attn_fwd", "attn_bwd_query", "attn_bwd",
    "selected_entries", "indexer_teacher_row", "indexer_teacher",
    "indexer_student_row", "indexer_kl_row", "indexer_loss",
    "round_e4m3", "quantize_rows_e4m3", "indexer_scores_fp8",
    "compressed_position", "rope_angles", "kv_norm_rope", "kv_norm_rope_bwd",
]


# ---------------------------------------------------------------------------
# Storage rounding (the one cast of the pooled result and of O)
# ---------------------------------------------------------------------------

def round_bf16(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits; the value m * 2**e (0.5 <= |m| < 1) is
    rounded at 2**(e-8).  Values below the smallest normal (2**-126) round on
    the fixed subnormal grid 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    e = np.maximum(e, -125)
    step = np.ldexp(1.0, e - 8)
    return np.round(x / step) * step


def round_to_storage(x, dtype: str):
    """The single cast to the storage dtype ('fp32' or 'bf16'), as float64."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "fp32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "fp64":
        return x
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Step 1: compressor (softmax-weighted pooling of `ratio` consecutive tokens)
# ---------------------------------------------------------------------------

def visible_blocks(t: int, ratio: int) -> int:
    """vis(t): compressed blocks visible to token t (0-based) = (t+1)//ratio.

    PR #6400 builds the mask from positions = arange(1, sq+1) and marks block
    j invalid where j >= positions // ratio.
    """
    return (t + 1) // ratio


def pooling_window(j: int, ratio: int, coff: int = 1):
    """Tokens pooled into compressed entry j: the coff blocks of `ratio`
    tokens ending with block j, clipped at token 0.  coff = 1 is the
    non-overlapping compressor ("compress_ratio == 128 (non-overlapping,
    coff = 1)", compressor review of PR #6400); coff = 2 lets each entry also
    pool the previous block (the overlapping reading)."""
    return slice(max(0, (j + 1 - coff) * ratio), (j + 1) * ratio)


def compress(kv, score, ratio: int, out_dtype: str = "fp64", coff: int = 1):
    """Pool the tokens of each entry's window (`pooling_window`).

    kv    [b, sq, d]   raw KV rows
    score [b, sq, d_s] pooling scores, d_s in {1, d} (d_s = 1 broadcasts)
    returns kv_c [b, n_c, d], n_c = sq // ratio, rounded once to out_dtype.

    Per entry j and channel c: weights = softmax over the window's tokens of
    score[., c]; kv_c[j, c] = sum_t weights_t * kv[t, c].  The pages keep the
    weights, the products and the sum in fp32 and cast once (compressor
    review of PR #6400); the oracle does the same in fp64.
    """
    kv = np.asarray(kv, np.float64)
    score = np.asarray(score, np.float64)
    b, sq, d = kv.shape
    n_c = sq // ratio
    out = np.zeros((b, n_c, d))
    for bi in range(b):
        for j in range(n_c):
            rows = pooling_window(j, ratio, coff)
            s = score[bi, rows]                     # [window, d_s]
            s = s - s.max(axis=0, keepdims=True)
            e = np.exp(s)
            weights = e / e.sum(axis=0, keepdims=True)
            out[bi, j] = (weights * kv[bi, rows]).sum(axis=0)
    return round_to_storage(out, out_dtype)


def compress_bwd(kv, score, ratio: int, g, coff: int = 1):
    """Gradient of the pooling (unrounded) w.r.t. kv and score.

    g [b, n_c, d] = dL/dkv_c.  With weights w_t of an entry's window and a
    channel, each entry contributes
      dkv_t    += w_t * g
      dscore_t += w_t * (g*kv_t - sum_t' w_t' * g*kv_t')
    (a token in several windows, coff > 1, sums their contributions).
    Tokens past the last complete block get zero gradient.  A d_s = 1 score
    sums its per-channel gradient over channels.
    """
    kv = np.asarray(kv, np.float64)
    score = np.asarray(score, np.float64)
    g = np.asarray(g, np.float64)
    b, sq, d = kv.shape
    d_s = score.shape[2]
    n_c = sq // ratio
    dkv = np.zeros_like(kv)
    dscore = np.zeros_like(score)
    for bi in range(b):
        for j in range(n_c):
            rows = pooling_window(j, ratio, coff)
            n = rows.stop - rows.start
            s = score[bi, rows]
            s = s - s.max(axis=0, keepdims=True)
            e = np.exp(s)
            weights = np.broadcast_to(e / e.sum(axis=0, keepdims=True), (n, d))
            dkv[bi, rows] += weights * g[bi, j]
            gk = g[bi, j] * kv[bi, rows]                      # [window, d]
            ds = weights * (gk - (weights * gk).sum(axis=0, keepdims=True))
            dscore[bi, rows] += ds if d_s == d else ds.sum(axis=1, keepdims=True)
    return dkv, dscore


# ---------------------------------------------------------------------------
# Steps 2-3: lightning indexer and causal top-k
# ---------------------------------------------------------------------------

def indexer_scores_row(q_I_t, k_I_b, w_t, t: int, ratio: int):
    """I[t, j] = sum_h w[t,h] * max(0, q_I[t,h,:] . k_I[j,:]) for j < vis(t).

    q_I_t [H_I, d_I], k_I_b [n_c, d_I], w_t [H_I]; returns a length-vis
    float64 vector (the visible prefix of the row).
    """
    v = min(visible_blocks(t, ratio), k_I_b.shape[0])
    if v == 0:
        return np.zeros(0)
    dots = np.asarray(q_I_t, np.float64) @ np.asarray(k_I_b[:v], np.float64).T   # [H_I, v]
    return np.asarray(w_t, np.float64) @ np.maximum(dots, 0.0)


def indexer_selectable(t: int, n_c: int, ratio: int, doc_b=None):
    """Boolean mask [n_c] of the blocks query t may select: j < vis(t) and,
    with per-token document ids doc_b [sq], doc_b[j*ratio] == doc_b[t]."""
    j = np.arange(n_c)
    ok = j < visible_blocks(t, ratio)
    if doc_b is not None:
        doc_b = np.asarray(doc_b)
        ok &= doc_b[np.minimum(j * ratio, doc_b.shape[0] - 1)] == doc_b[t]
    return ok


def indexer_scores(q_I, k_I, w, ratio: int, doc_ids=None):
    """Full score matrix [b, sq, n_c]; entries query t may not select
    (j >= vis(t), or another document's block) are -inf."""
    b, sq = q_I.shape[:2]
    n_c = k_I.shape[1]
    out = np.full((b, sq, n_c), -np.inf)
    for bi in range(b):
        for t in range(sq):
            row = indexer_scores_row(q_I[bi, t], k_I[bi], w[bi, t], t, ratio)
            out[bi, t, :row.shape[0]] = row
            if doc_ids is not None:
                out[bi, t, ~indexer_selectable(t, n_c, ratio, doc_ids[bi])] = -np.inf
    return out


def topk_select_row(scores_vis, K: int):
    """Top-K of one row's visible scores.

    Sort the (score, j) pairs by score descending, then j ascending (ties go
    to the lower block index), keep the first min(K, vis), and return them in
    ascending j (support sorted by position) padded with -1 to length K.
    """
    v = scores_vis.shape[0]
    order = np.lexsort((np.arange(v), -np.asarray(scores_vis, np.float64)))
    sel = np.sort(order[:min(K, v)])
    out = np.full(K, -1, np.int32)
    out[:sel.shape[0]] = sel
    return out


def topk_select(scores, K: int):
    """Top-K of every row of a [b, sq, n_c] matrix whose non-selectable
    entries are -inf: the same rule as topk_select_row over the selectable
    entries (any subset of the row), ascending block ids, -1 tail."""
    b, sq, n_c = scores.shape
    out = np.full((b, sq, K), -1, np.int32)
    for bi in range(b):
        for t in range(sq):
            row = scores[bi, t]
            cand = np.flatnonzero(np.isfinite(row))
            sel = topk_select_row(row[cand], K)
            n = int((sel >= 0).sum())
            out[bi, t, :n] = cand[sel[:n]]
    return out


# ---------------------------------------------------------------------------
# Steps 4-5: sparse MQA over window + selected compressed rows + sink
# ---------------------------------------------------------------------------

def query_slots(t: int, idx_row, sq: int, n_c: int, ratio: int, window: int, doc_b=None):
    """KV rows that query t attends to, in the flat [n_kv] row space.

    Window: raw rows max(0, t-window+1) .. t (with document ids doc_b [sq],
    only those of t's document).  Compressed: row sq + j for every entry j of
    the index row with 0 <= j < n_c and j < vis(t); other entries are
    padding.  A repeated entry yields a repeated row (two terms).
    """
    raw = [k for k in range(max(0, t - window + 1), t + 1)
           if doc_b is None or doc_b[k] == doc_b[t]]
    vis = visible_blocks(t, ratio)
    comp = [sq + int(j) for j in idx_row if 0 <= int(j) < n_c and int(j) < vis]
    return np.asarray(raw + comp, dtype=np.int64)


def _sink_vec(sink, H):
    if sink is None:
        return np.full(H, -np.inf)
    return np.asarray(sink, np.float64)


def attn_fwd_query(q_t, kv_b, slots, sink_h, scale: float):
    """One query, all heads.

    s_i = scale * q_h . kv_i; LSE_h = log(exp(sink_h) + sum_i exp(s_i));
    O_h = sum_i exp(s_i - LSE_h) * kv_i.  The sink only enters the
    denominator.  Returns (O [H,d], LSE [H], P [H,S], gathered rows [S,d]).
    """
    kvg = np.asarray(kv_b, np.float64)[slots]
    s = scale * (np.asarray(q_t, np.float64) @ kvg.T)
    m = np.maximum(s.max(axis=1), sink_h)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1) + np.exp(sink_h - m)
    lse = m + np.log(z)
    p = e / z[:, None]
    return p @ kvg, lse, p, kvg


def attn_fwd(q, kv_full, idx, sink, scale: float, window: int, ratio: int,
             rows=None, out_dtype: str = "fp64", doc_ids=None):
    """O [b, sq, H, d] (rounded once to out_dtype) and LSE [b, sq, H].

    ``rows``: optional list of (b, t) pairs; only those rows are computed and
    the results come back as arrays of shape [len(rows), H, d] / [len(rows), H].
    ``doc_ids`` [b, sq]: optional document ids restricting the window.
    """
    b, sq, H, d = q.shape
    n_c = kv_full.shape[1] - sq
    sink_h = _sink_vec(sink, H)
    pairs = rows if rows is not None else [(bi, t) for bi in range(b) for t in range(sq)]
    O = np.zeros((len(pairs), H, d))
    L = np.zeros((len(pairs), H))
    for n, (bi, t) in enumerate(pairs):
        slots = query_slots(t, idx[bi, t], sq, n_c, ratio, window,
                            None if doc_ids is None else doc_ids[bi])
        o, lse, _, _ = attn_fwd_query(q[bi, t], kv_full[bi], slots, sink_h, scale)
        O[n], L[n] = o, lse
    O = round_to_storage(O, out_dtype)
    if rows is None:
        return O.reshape(b, sq, H, d), L.reshape(b, sq, H)
    return O, L


def attn_bwd_query(q_t, kv_b, slots, sink_h, scale: float, dO_t):
    """Exact gradients of L = sum_h dO_h . O_h for one query.

    D_h = dO_h . O_h;  p_i = exp(s_i - LSE);  ds_i = p_i (dO_h . kv_i - D_h);
    dq_h = scale * sum_i ds_i kv_i;  per slot: dkv_i = sum_h (p_i dO_h + scale ds_i q_h);
    dsink_h = -exp(sink_h - LSE_h) * D_h.
    Returns (dq [H,d], per-slot dkv contributions [S,d], dsink [H]).
    """
    o, lse, p, kvg = attn_fwd_query(q_t, kv_b, slots, sink_h, scale)
    dO_t = np.asarray(dO_t, np.float64)
    q_t = np.asarray(q_t, np.float64)
    D = (dO_t * o).sum(axis=1)
    dp = dO_t @ kvg.T
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ kvg)
    dkv_slots = p.T @ dO_t + scale * (ds.T @ q_t)
    dsink = -np.exp(sink_h - lse) * D
    return dq, dkv_slots, dsink


def attn_bwd(q, kv_full, idx, sink, scale: float, window: int, ratio: int, dO, rows=None,
             doc_ids=None):
    """dq [b, sq, H, d], dkv [b, n_kv, d] and dsink [H].

    The slot contributions scatter-add into the compact [b, n_kv, d] buffer
    (np.add.at sums repeated rows); dsink sums over b and t.  With ``rows``
    only those queries are processed: dq comes back as [len(rows), H, d] and
    dkv / dsink hold the contributions of those queries alone.
    """
    b, sq, H, d = q.shape
    n_kv = kv_full.shape[1]
    n_c = n_kv - sq
    sink_h = _sink_vec(sink, H)
    pairs = rows if rows is not None else [(bi, t) for bi in range(b) for t in range(sq)]
    dq = np.zeros((len(pairs), H, d))
    dkv = np.zeros((b, n_kv, d))
    dsink = np.zeros(H)
    for n, (bi, t) in enumerate(pairs):
        slots = query_slots(t, idx[bi, t], sq, n_c, ratio, window,
                            None if doc_ids is None else doc_ids[bi])
        dq_t, dkv_s, ds_t = attn_bwd_query(q[bi, t], kv_full[bi], slots, sink_h, scale, dO[bi, t])
        dq[n] = dq_t
        np.add.at(dkv[bi], slots, dkv_s)
        if sink is not None:
            dsink += ds_t
    if rows is None:
        dq = dq.reshape(b, sq, H, d)
    return dq, dkv, dsink


# ---------------------------------------------------------------------------
# Indexer training path: teacher target from the attention LSE, student
# rescoring of the selected entries, KL distillation loss and its gradients
# ---------------------------------------------------------------------------
#
# "Refactor Deepseek v4 to use Attention Gym's Compressed Sparse Attention"
# (selected_attention commit; indexer distillation): the teacher of query t
# over its selected entries is exp(logit - lse) summed over the heads and
# L1-normalized, with lse the attention's per-head LSE (window, selected
# entries and sink in the denominator); the student is a second pass of the
# indexer over the selected entries only.  "Add unfused SBHD compressed
# sparse attention" (review of the teacher normalization): one common
# per-row shift keeps the mass from underflowing and cancels in the L1
# normalization; a row without mass stays zero; the KL gradient with respect
# to the student scores is predict * sum(target) - target, so a zero row
# gets zero gradient.

def selected_entries(idx_row, t: int, n_c: int, ratio: int):
    """(slot positions, block ids) of the valid entries of one index row:
    0 <= j < n_c and j < vis(t); repeated entries are kept (one term each)."""
    vis = visible_blocks(t, ratio)
    pos = [s for s, j in enumerate(idx_row) if 0 <= int(j) < n_c and int(j) < vis]
    return np.asarray(pos, np.int64), np.asarray([int(idx_row[s]) for s in pos], np.int64)


def indexer_teacher_row(q_t, kv_b, idx_row, lse_t, t: int, sq: int, ratio: int, scale: float):
    """Teacher target [K] of query t.

    T_s = sum_h exp(scale * q_h . kv[sq + j_s] - lse_h) over the valid slots
    s (0 elsewhere), then target = T / sum(T).  Evaluated as
    exp(a - c) with a = logit - lse and c = max a over the row's valid
    (h, s): the shift cancels in the normalization and keeps the largest
    term at 1.  A row without valid slots is all zero.
    """
    K = len(idx_row)
    n_c = kv_b.shape[0] - sq
    out = np.zeros(K)
    pos, js = selected_entries(idx_row, t, n_c, ratio)
    if pos.size == 0:
        return out
    logits = scale * (np.asarray(q_t, np.float64) @ np.asarray(kv_b, np.float64)[sq + js].T)
    a = logits - np.asarray(lse_t, np.float64)[:, None]            # [H, n_valid]
    T = np.exp(a - a.max()).sum(axis=0)
    out[pos] = T / T.sum()
    return out


def indexer_teacher(q, kv_full, idx, lse, scale: float, ratio: int):
    """Teacher targets [b, sq, K] (fp64) from the attention inputs and LSE."""
    b, sq = q.shape[:2]
    K = idx.shape[2]
    out = np.zeros((b, sq, K))
    for bi in range(b):
        for t in range(sq):
            out[bi, t] = indexer_teacher_row(q[bi, t], kv_full[bi], idx[bi, t], lse[bi, t], t, sq,
                                             ratio, scale)
    return out


def indexer_student_row(q_I_t, k_I_b, w_t, idx_row, t: int, ratio: int):
    """Student scores [K] of query t: the indexer score of each valid slot's
    block, I_s = sum_h w_h max(0, q_I_h . k_I[j_s]); -inf at invalid slots."""
    n_c = k_I_b.shape[0]
    out = np.full(len(idx_row), -np.inf)
    pos, js = selected_entries(idx_row, t, n_c, ratio)
    if pos.size:
        dots = np.asarray(q_I_t, np.float64) @ np.asarray(k_I_b, np.float64)[js].T   # [H_I, n]
        out[pos] = np.asarray(w_t, np.float64) @ np.maximum(dots, 0.0)
    return out


def indexer_kl_row(I_row, target_row):
    """KL(target || softmax(I)) over the valid (finite) slots of one row and
    its gradient with respect to I: predict * sum(target) - target (zero at
    invalid slots).  Terms with target 0 contribute 0 to the loss."""
    I_row = np.asarray(I_row, np.float64)
    tg = np.asarray(target_row, np.float64)
    v = np.isfinite(I_row)
    dI = np.zeros_like(I_row)
    if not v.any():
        return 0.0, dI
    x = I_row[v]
    logp = x - x.max() - np.log(np.exp(x - x.max()).sum())
    tv = tg[v]
    nz = tv > 0
    loss = float((tv[nz] * (np.log(tv[nz]) - logp[nz])).sum())
    dI[v] = np.exp(logp) * tv.sum() - tv
    return loss, dI


def indexer_loss(q_I, k_I, w, idx, target, ratio: int):
    """Per-row KL loss [b, sq] and its gradients dq_I [b, sq, H_I, d_I],
    dk_I [b, n_c, d_I] (summed over every query and repeated slot that
    selected the block) and dw [b, sq, H_I], through the student rescoring.

    With G_hs = dI_s * w_h * [q_I_h . k_I[j_s] > 0]:
      dq_I[t, h]   = sum_s G_hs k_I[j_s]
      dk_I[j]     += sum_{t, s: j_s = j} sum_h G_hs q_I[t, h]
      dw[t, h]     = sum_s dI_s max(0, q_I_h . k_I[j_s])
    """
    q_I = np.asarray(q_I, np.float64)
    k_I = np.asarray(k_I, np.float64)
    w = np.asarray(w, np.float64)
    b, sq, H_I, d_I = q_I.shape
    n_c = k_I.shape[1]
    loss = np.zeros((b, sq))
    dq = np.zeros_like(q_I)
    dk = np.zeros_like(k_I)
    dw = np.zeros_like(w)
    for bi in range(b):
        for t in range(sq):
            I = indexer_student_row(q_I[bi, t], k_I[bi], w[bi, t], idx[bi, t], t, ratio)
            loss[bi, t], dI = indexer_kl_row(I, target[bi, t])
            pos, js = selected_entries(idx[bi, t], t, n_c, ratio)
            if pos.size == 0:
                continue
            dots = q_I[bi, t] @ k_I[bi][js].T                    # [H_I, n]
            g = dI[pos][None, :] * w[bi, t][:, None] * (dots > 0)
            dq[bi, t] = g @ k_I[bi][js]
            np.add.at(dk[bi], js, g.T @ q_I[bi, t])
            dw[bi, t] = np.maximum(dots, 0.0) @ dI[pos]
    return loss, dq, dk, dw


# ---------------------------------------------------------------------------
# FP8 indexer: q_I and k_I quantized per row to e4m3, scores from the codes
# ---------------------------------------------------------------------------
#
# The pages list "indexer quantization" as not included ("Refactor Deepseek
# v4 ...", model description); the quantization here is this repository's
# reading: every q_I head row and every k_I row is scaled by 448 / absmax(row)
# (448 = the largest finite e4m3 value), rounded to e4m3, and keeps the
# scale absmax / 448.  Both quantities are computed in fp32 (the reciprocal
# 448 / absmax, then x * reciprocal), so that both sides round the same fp32
# value.  The scores use the dequantized rows:
#   I[t, j] = sum_h w[t,h] * max(0, sq[t,h] sk[j] (q8[t,h] . k8[j]))
#           = sk[j] * sum_h (w[t,h] sq[t,h]) max(0, q8[t,h] . k8[j])   (scales > 0)

def round_e4m3(x):
    """Round to the nearest e4m3 value (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; no infinities), ties to even, saturating at +-448.
    Normal numbers have 4 significant bits; below 2^-6 the grid is 2^-9."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), 448.0)
    _, e = np.frexp(a)                     # a = m 2^e, 0.5 <= m < 1
    e = np.maximum(e, -5)                  # subnormal range shares the 2^-9 grid
    step = np.ldexp(1.0, e - 4)
    r = np.round(a / step) * step          # numpy rounds half to even
    return np.sign(x) * np.minimum(r, 448.0)


def quantize_rows_e4m3(x):
    """Per-row (last axis) e4m3 codes (as float64 values) and fp32 scales."""
    x32 = np.asarray(x, np.float32)
    amax = np.abs(x32).max(axis=-1)
    inv = np.where(amax > 0, np.float32(448.0) / np.where(amax > 0, amax, 1), 0).astype(np.float32)
    y = (x32 * inv[..., None]).astype(np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    return round_e4m3(y.astype(np.float64)), scale


def indexer_scores_fp8(q8, q_scale, k8, k_scale, w, ratio: int, doc_ids=None):
    """Indexer scores [b, sq, n_c] from e4m3 codes and scales; entries a query
    may not select are -inf (as indexer_scores)."""
    q8 = np.asarray(q8, np.float64)
    k8 = np.asarray(k8, np.float64)
    b, sq, H_I, _ = q8.shape
    n_c = k8.shape[1]
    out = np.full((b, sq, n_c), -np.inf)
    for bi in range(b):
        for t in range(sq):
            v = min(visible_blocks(t, ratio), n_c)
            if v == 0:
                continue
            dots = q8[bi, t] @ k8[bi, :v].T                                # [H_I, v]
            wq = np.asarray(w[bi, t], np.float64) * np.asarray(q_scale[bi, t], np.float64)
            out[bi, t, :v] = np.asarray(k_scale[bi, :v], np.float64) * (wq @ np.maximum(dots, 0.0))
            if doc_ids is not None:
                out[bi, t, ~indexer_selectable(t, n_c, ratio, doc_ids[bi])] = -np.inf
    return out


# ---------------------------------------------------------------------------
# Normalization and rotary embedding of the pooled rows
# ---------------------------------------------------------------------------
#
# "Add unfused SBHD compressed sparse attention" (compressor review): the
# pooled row is cast once to the storage dtype and then normalized,
# kv = self.norm(kv); its config fields give the rotary base of compressed KV
# positions, csa_compress_rotary_base = 40000.  "[DeepSeek-v4] Part 1": the
# KV norm is created over v_head_dim channels (one weight per channel), and
# the MLA rotary kernels keep the interleaved channel layout.  Neither the
# norm's type nor the rotary channels nor the compressed position are given;
# the readings are stated in the module header.

def compressed_position(j, ratio: int):
    """Position of compressed entry j: its last pooled token, (j+1)*ratio - 1
    (the token at which the entry becomes visible)."""
    return (np.asarray(j, np.int64) + 1) * ratio - 1


def rope_angles(pos, rope_dim: int, base: float):
    """Angles [len(pos), rope_dim/2]: pos * base^(-2i/rope_dim)."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / rope_dim)
    return np.asarray(pos, np.float64)[:, None] * theta[None, :]


def _rotate(y, ang, sign: float):
    """Rotate the interleaved pairs (2i, 2i+1) of y [..., 2m] by sign*ang [..., m]."""
    c, s = np.cos(ang), sign * np.sin(ang)
    a, b = y[..., 0::2], y[..., 1::2]
    out = np.empty_like(y)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def kv_norm_rope(kv_c, weight, eps: float, rope_dim: int, base: float, ratio: int,
                 out_dtype: str = "fp64"):
    """RMS-normalize each pooled row over its d channels and rotate its last
    rope_dim channels.

    kv_c [b, n_c, d] (the pooled rows as stored), weight [d]:
      y = kv_c / sqrt(mean_c(kv_c^2) + eps) * weight
      y[..., d-rope_dim:] rotated pairwise by pos_j * base^(-2i/rope_dim),
      pos_j = (j+1)*ratio - 1,
    rounded once to out_dtype.
    """
    x = np.asarray(kv_c, np.float64)
    b, n_c, d = x.shape
    rms = np.sqrt((x * x).mean(axis=2, keepdims=True) + eps)
    y = x / rms * np.asarray(weight, np.float64)
    if rope_dim:
        ang = rope_angles(compressed_position(np.arange(n_c), ratio), rope_dim, base)
        y[..., d - rope_dim:] = _rotate(y[..., d - rope_dim:], ang[None], 1.0)
    return round_to_storage(y, out_dtype)


def kv_norm_rope_bwd(kv_c, weight, eps: float, rope_dim: int, base: float, ratio: int, g):
    """Gradients of kv_norm_rope (unrounded) given g = dL/d(output) [b, n_c, d]:
    returns (dL/dkv_c [b, n_c, d], dL/dweight [d]).

    The rotation is orthogonal, so its gradient rotates g back (angle
    negated); with xh = x / rms and dy the unrotated gradient:
      dweight = sum over rows of dy * xh,
      dx = (dy*weight - xh * mean_c(dy*weight*xh)) / rms.
    """
    x = np.asarray(kv_c, np.float64)
    g = np.asarray(g, np.float64)
    w = np.asarray(weight, np.float64)
    b, n_c, d = x.shape
    dy = g.copy()
    if rope_dim:
        ang = rope_angles(compressed_position(np.arange(n_c), ratio), rope_dim, base)
        dy[..., d - rope_dim:] = _rotate(g[..., d - rope_dim:], ang[None], -1.0)
    rms = np.sqrt((x * x).mean(axis=2, keepdims=True) + eps)
    xh = x / rms
    dweight = (dy * xh).sum(axis=(0, 1))
    dxh = dy * w
    dx = (dxh - xh * (dxh * xh).mean(axis=2, keepdims=True)) / rms
    return dx, dweight
