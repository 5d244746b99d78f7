"""GPU parity of the indexer training path against the fp64 oracle, through
the C ABI: the distillation teacher (csa_indexer_teacher) and the student's
KL loss with its gradients (csa_indexer_loss).

Every kernel family is covered: the tcgen05 loss kernel for bf16 with
d_I = 128 and H_I in {32, 64}, warp-level MMA for the other bf16 shapes with
d (d_I) in the supported set, the CUDA-core kernel for fp32 and other shapes; index
rows carry repeated, padded, out-of-range and not-yet-visible entries, and
some rows have no valid entry at all or an all-zero target.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
from oracle import csa_oracle as orc
from paritylib import TOL, f64, maxabs, oracle_indexer, oracle_kv_full

pytestmark = pytest.mark.gpu

# The teacher and the loss are fp32 arithmetic on the stored inputs (products
# of bf16 values are exact in the fp32 accumulators); their outputs are
# probabilities and gradients of magnitude O(1), so they are held to
# 1e-4 / 2e-3, well inside the method's tolerance.
TEACHER_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    yield
    assert csa.csa_get_device_status() == 0


def _dt(name):
    return torch.float32 if name == "fp32" else torch.bfloat16


def _messy_idx(g, b, sq, n_c, K):
    idx = torch.randint(-1, n_c + 2, (b, sq, K), generator=g, dtype=torch.int32)
    if K > 1:
        idx[:, :, 1] = idx[:, :, 0]           # repeated entries
    idx[:, 5] = -1                            # a row without valid entries
    return idx


# ---------------------------------------------------------------------------
# teacher
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H,d", [
    ("fp32", 4, 64),      # CUDA-core kernel
    ("bf16", 6, 64),      # warp MMA, heads padded to 16
    ("bf16", 20, 40),     # CUDA-core kernel for a head dim outside the MMA set
    ("bf16", 16, 128),    # tcgen05 kernel, 8 queries per CTA
    ("bf16", 32, 128),    # tcgen05 kernel, 4 queries per CTA
    ("bf16", 64, 128),    # tcgen05 kernel, a query's heads over two column groups
    ("bf16", 64, 512),    # warp MMA, widest rows
])
def test_teacher_random_rows(dtype, H, d):
    b, sq, ratio, K = 2, 120, 4, 70
    g = torch.Generator().manual_seed(51)
    n_c = sq // ratio
    q = torch.randn(b, sq, H, d, generator=g).to(_dt(dtype))
    kv = torch.randn(b, sq + n_c, d, generator=g).to(_dt(dtype))
    idx = _messy_idx(g, b, sq, n_c, K)
    lse = torch.randn(b, sq, H, generator=g) + 6.0
    scale = d ** -0.5
    got = csa.csa_indexer_teacher(q.cuda(), kv.cuda(), idx.cuda(), lse.cuda(), scale, ratio)
    ref = orc.indexer_teacher(f64(q), f64(kv), idx.numpy(), f64(lse), scale, ratio)
    assert maxabs(f64(got), ref) <= TEACHER_TOL
    assert torch.all(got[:, 5] == 0)


@pytest.mark.parametrize("name", ["debug_bf16", "csa4_bf16"])
def test_teacher_layer_with_attention_lse(name):
    """The workload's layer: the GPU forward's LSE feeds the teacher on both
    sides; every row compared (invalid-slot zeros, row sums 1)."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("attn",))
    idx = torch.from_numpy(oracle_indexer(name)[1])
    kv = oracle_kv_full(name)
    q = inp["q"].cuda()
    _, lse = csa.csa_attn_fwd(q, kv.cuda(), idx.cuda(), inp["sink"].cuda(), cfg.scale, cfg.ratio,
                              cfg.window)
    got = csa.csa_indexer_teacher(q, kv.cuda(), idx.cuda(), lse, cfg.scale, cfg.ratio)
    ref = orc.indexer_teacher(f64(inp["q"]), f64(kv), idx.numpy(), f64(lse), cfg.scale, cfg.ratio)
    assert maxabs(f64(got), ref) <= TEACHER_TOL
    sums = got.sum(-1).cpu()
    has = torch.from_numpy((idx.numpy() >= 0).any(-1))          # rows with a selected block
    assert torch.all((sums[has] - 1).abs() < 1e-4) and torch.all(sums[~has] == 0)


# ---------------------------------------------------------------------------
# student loss and gradients
# ---------------------------------------------------------------------------

def _relu_mask_slack(q_I, k_I, w, idx, target, ratio):
    """Where a dot product q_I.k_I lies within the fp32 accumulation error of
    zero, the ReLU derivative [dot > 0] is decided by rounding, and the two
    sides may legitimately differ.  Per output element, the slack is the sum
    of |G| times the partner row over those ambiguous (head, slot) pairs
    (G = dI w), with the error bound d_I 2^-23 sum_k |q_k k_k| per dot."""
    qn, kn, wn, tn = f64(q_I), f64(k_I), f64(w), f64(target)
    b, sq, H_I, d_I = qn.shape
    n_c = kn.shape[1]
    s_dq = np.zeros_like(qn)
    s_dk = np.zeros_like(kn)
    n_amb = 0
    for bi in range(b):
        for t in range(sq):
            pos, js = orc.selected_entries(idx[bi, t], t, n_c, ratio)
            if pos.size == 0:
                continue
            kk = kn[bi][js]
            dots = qn[bi, t] @ kk.T
            bound = d_I * 2.0 ** -23 * (np.abs(qn[bi, t]) @ np.abs(kk).T)
            amb = np.abs(dots) <= bound
            if not amb.any():
                continue
            n_amb += int(amb.sum())
            I = orc.indexer_student_row(qn[bi, t], kn[bi], wn[bi, t], idx[bi, t], t, ratio)
            _, dI = orc.indexer_kl_row(I, tn[bi, t])
            gabs = np.abs(dI[pos][None, :] * wn[bi, t][:, None]) * amb
            s_dq[bi, t] = gabs @ np.abs(kk)
            np.add.at(s_dk[bi], js, gabs.T @ np.abs(qn[bi, t]))
    return s_dq, s_dk, n_amb


def _check_loss(q_I, k_I, w, idx, target, ratio, dtype):
    loss, dq, dk, dw = csa.csa_indexer_loss(q_I.cuda(), k_I.cuda(), w.cuda(), idx.cuda(),
                                            target.cuda(), ratio)
    r_loss, r_dq, r_dk, r_dw = orc.indexer_loss(f64(q_I), f64(k_I), f64(w), idx.numpy(),
                                                f64(target), ratio)
    s_dq, s_dk, _ = _relu_mask_slack(q_I, k_I, w, idx.numpy(), target, ratio)
    tol = TOL["fp32"]
    errs = {"loss": maxabs(f64(loss), r_loss), "dw": maxabs(f64(dw), r_dw),
            "dq_I": float(np.max(np.abs(f64(dq) - r_dq) - s_dq)),
            "dk_I": float(np.max(np.abs(f64(dk) - r_dk) - s_dk))}
    assert max(errs.values()) <= tol, errs
    return loss, dq, dk, dw


@pytest.mark.parametrize("dtype,H_I,d_I", [
    ("fp32", 3, 32),      # CUDA-core kernel
    ("bf16", 5, 64),      # warp MMA, heads padded to 16
    ("bf16", 24, 128),    # warp MMA, heads padded to 32
    ("bf16", 4, 40),      # CUDA-core kernel for a dim outside the MMA set
])
def test_loss_random_rows(dtype, H_I, d_I):
    b, sq, ratio, K = 2, 100, 2, 37
    g = torch.Generator().manual_seed(52)
    n_c = sq // ratio
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(_dt(dtype))
    k_I = torch.randn(b, n_c, d_I, generator=g).to(_dt(dtype))
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    idx = _messy_idx(g, b, sq, n_c, K)
    target = torch.rand(b, sq, K, generator=g)
    target[:, 7] = 0.0                        # a row without mass: no gradient
    target = target / target.sum(-1, keepdim=True).clamp_min(1e-30)
    loss, dq, dk, dw = _check_loss(q_I, k_I, w, idx, target, ratio, dtype)
    assert torch.all(dq[:, 7] == 0) and torch.all(dw[:, 7] == 0) and torch.all(loss[:, 7] == 0)


@pytest.mark.parametrize("H_I,sq,ratio,K,b", [
    (64, 101, 2, 37, 2),     # tensor-core kernel, 2 queries per CTA, a partial last block
    (32, 102, 2, 37, 2),     # 4 queries per CTA, a partial last block
    (64, 600, 2, 200, 2),    # unions of up to 300 blocks: three tiles of 128
    (32, 520, 2, 160, 2),    # 4 queries per CTA over three tiles
    (64, 2048, 1, 512, 1),   # n_c 2048, the largest its shared memory takes at H_I 64
])
def test_loss_tensor_core_shapes(H_I, sq, ratio, K, b):
    """bf16, d_I = 128 and H_I in {32, 64} take the tcgen05 kernel (queries
    sharing the union of their selections): messy index rows (repeats,
    padding, out-of-range and not-yet-visible entries), rows without valid
    entries or without target mass, and unions spanning several tiles."""
    d_I = 128
    g = torch.Generator().manual_seed(60 + H_I + sq)
    n_c = sq // ratio
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(torch.bfloat16)
    k_I = torch.randn(b, n_c, d_I, generator=g).to(torch.bfloat16)
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    idx = _messy_idx(g, b, sq, n_c, K)
    target = torch.rand(b, sq, K, generator=g)
    target[:, 7] = 0.0
    target = target / target.sum(-1, keepdim=True).clamp_min(1e-30)
    loss, dq, dk, dw = _check_loss(q_I, k_I, w, idx, target, ratio, "bf16")
    assert torch.all(dq[:, 7] == 0) and torch.all(dw[:, 7] == 0) and torch.all(loss[:, 7] == 0)
    assert torch.all(dq[:, 5] == 0) and torch.all(dw[:, 5] == 0) and torch.all(loss[:, 5] == 0)


@pytest.mark.parametrize("H_I", [32, 64])
def test_loss_tensor_core_zero_and_tiny_head_weights(H_I):
    """Head weights that are exactly zero or below 2^-60: the tcgen05 kernel
    forms dw from its dq_I products divided by w, so those rows take the
    weight-1 products and a zeroed Q row instead (dw from the same products,
    dq_I scaled by w, nothing added to dk_I)."""
    b, sq, ratio, K, d_I = 2, 150, 2, 40, 128
    g = torch.Generator().manual_seed(77 + H_I)
    n_c = sq // ratio
    q_I = torch.randn(b, sq, H_I, d_I, generator=g).to(torch.bfloat16)
    k_I = torch.randn(b, n_c, d_I, generator=g).to(torch.bfloat16)
    w = torch.randn(b, sq, H_I, generator=g) * 0.5
    w[:, :, 3] = 0.0                          # one head without weight everywhere
    w[:, 40:60, 5] = 1e-30                    # below 2^-60
    w[0, 90, :] = 0.0                         # a query whose heads all weigh nothing
    w[1, 100, 7] = -3e-19                     # just below 2^-60 in magnitude
    idx = _messy_idx(g, b, sq, n_c, K)
    target = torch.rand(b, sq, K, generator=g)
    target = target / target.sum(-1, keepdim=True).clamp_min(1e-30)
    _check_loss(q_I, k_I, w, idx, target, ratio, "bf16")


@pytest.mark.parametrize("name", ["debug_bf16", "csa4_bf16"])
def test_loss_layer_with_teacher(name):
    """The workload's indexer inputs and top-k, the oracle's teacher as the
    target: loss, dq_I, dk_I (summed over all queries) and dw."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    idx = torch.from_numpy(oracle_indexer(name)[1])
    kv = oracle_kv_full(name)
    _, lse = orc.attn_fwd(f64(inp["q"]), f64(kv), idx.numpy(), f64(inp["sink"]), cfg.scale,
                          cfg.window, cfg.ratio)
    target = torch.from_numpy(orc.indexer_teacher(f64(inp["q"]), f64(kv), idx.numpy(), lse,
                                                  cfg.scale, cfg.ratio)).float()
    _check_loss(inp["q_I"], inp["k_I"], inp["w"], idx, target, cfg.ratio, cfg.dtype)
