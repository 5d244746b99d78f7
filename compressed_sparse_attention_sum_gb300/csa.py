"""Python binding of the CSA C ABI (include/csa.h).

Argument marshalling only: each function checks the tensors it is given,
allocates missing outputs with PyTorch (device memory is PyTorch's job),
and calls the entry point of the same name in libcsa.so with raw device
pointers and the current CUDA stream.  All arithmetic runs in the library's
kernels; there is no fallback: if libcsa.so is missing or the call fails,
these functions raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

CSA_FP32, CSA_BF16 = 0, 1
STATUS = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARG", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_CUDA",
          4: "CSA_ERR_WORKSPACE", 5: "CSA_ERR_TIMEOUT", 6: "CSA_ERR_DEVICE_CHECK"}

_lib = None

_c_int, _c_ll, _c_p, _c_f, _c_sz = ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t

SIGNATURES = {
    "csa_status_string": (ctypes.c_char_p, [_c_int]),
    "csa_version": (_c_int, []),
    "csa_kernel_launches": (ctypes.c_ulonglong, []),
    "csa_compress": (_c_int, [_c_p, _c_ll, _c_p, _c_int, _c_p, _c_ll, _c_int, _c_int, _c_int, _c_int,
                              _c_int, _c_p]),
    "csa_compress_bwd": (_c_int, [_c_p, _c_ll, _c_p, _c_int, _c_p, _c_ll, _c_p, _c_ll, _c_p]
                         + [_c_int] * 5 + [_c_p]),
    "csa_compress_overlap": (_c_int, [_c_p, _c_ll, _c_p, _c_int, _c_p, _c_ll] + [_c_int] * 6
                             + [_c_p]),
    "csa_compress_overlap_bwd": (_c_int, [_c_p, _c_ll, _c_p, _c_int, _c_p, _c_ll, _c_p, _c_ll,
                                          _c_p] + [_c_int] * 6 + [_c_p]),
    "csa_compress_norm_rope": (_c_int, [_c_p, _c_ll, _c_p, _c_int, _c_p, _c_f, _c_int, _c_f,
                                        _c_p, _c_ll] + [_c_int] * 5 + [_c_p]),
    "csa_compress_norm_rope_bwd": (_c_int, [_c_p, _c_ll, _c_p, _c_int, _c_p, _c_f, _c_int, _c_f,
                                            _c_p, _c_ll, _c_p, _c_ll, _c_p, _c_p]
                                   + [_c_int] * 5 + [_c_p]),
    "csa_indexer_topk_workspace_size": (_c_sz, [_c_int] * 6 + [_c_int]),
    "csa_indexer_topk_min_workspace": (_c_sz, [_c_int, _c_int]),
    "csa_indexer_topk": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p] + [_c_int] * 7
                         + [_c_int, _c_p, _c_sz, _c_p]),
    "csa_indexer_topk_noalloc": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p] + [_c_int] * 7
                                 + [_c_int, _c_p]),
    "csa_quantize_e4m3": (_c_int, [_c_p, _c_ll, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "csa_indexer_topk_fp8": (_c_int, [_c_p] * 8 + [_c_int] * 7 + [_c_p, _c_sz, _c_p]),
    "csa_attn_fwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_p] + [_c_int] * 8
                     + [_c_int, _c_p]),
    "csa_attn_bwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_p, _c_p, _c_p, _c_p,
                              _c_p] + [_c_int] * 8 + [_c_int, _c_p]),
    "csa_indexer_teacher": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_f, _c_p] + [_c_int] * 7
                            + [_c_int, _c_p]),
    "csa_indexer_loss": (_c_int, [_c_p] * 9 + [_c_int] * 7 + [_c_int, _c_p]),
    "csa_indexer_topk_rows": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p] + [_c_int] * 7
                              + [_c_int, _c_p, _c_sz, _c_int, _c_int, _c_p]),
    "csa_attn_fwd_rows": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_p] + [_c_int] * 8
                          + [_c_int, _c_int, _c_int, _c_p]),
    "csa_attn_bwd_rows": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_p, _c_p, _c_p,
                                   _c_p, _c_p] + [_c_int] * 8 + [_c_int, _c_int, _c_int, _c_int,
                                                                 _c_p]),
    "csa_get_device_status": (_c_int, [_c_p, ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]),
    "csa_debug_arm_fault": (_c_int, [_c_int]),
}


def load_library(path: str = LIB_PATH):
    """Load libcsa.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CSA CUDA library not found at {path}; build it with "
                           "compressed_sparse_attention_sum_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class CSAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = load_library().csa_status_string(code).decode()
        super().__init__(f"{fn} failed: {msg}")
        self.code = code


def _check(fn: str, code: int):
    if code != 0:
        raise CSAError(fn, code)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CSA_BF16
    if t.dtype == torch.float32:
        return CSA_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, contiguous=True):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _compress_out(kv, score, ratio, out):
    _need(kv, "kv", contiguous=False)
    _need(score, "score", dtype=kv.dtype)
    b, sq, d = kv.shape
    n_c = sq // ratio
    if kv.stride(2) != 1 or kv.stride(1) != d:
        raise ValueError("kv rows must be contiguous")
    if out is None:
        out = torch.empty(b, n_c, d, dtype=kv.dtype, device=kv.device)
    _need(out, "out", dtype=kv.dtype, contiguous=False)
    if out.shape != (b, n_c, d) or out.stride(2) != 1 or out.stride(1) != d:
        raise ValueError("out must be [b, sq//ratio, d] with contiguous rows")
    return out


def csa_compress(kv: torch.Tensor, score: torch.Tensor, ratio: int,
                 out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Softmax-weighted pooling of `ratio` consecutive tokens.

    kv [b, sq, d] (rows contiguous; may be the raw-row view kv_full[:, :sq]),
    score [b, sq, d] or [b, sq, 1] packed, out [b, sq//ratio, d] (rows
    contiguous; may be the view kv_full[:, sq:]).
    """
    lib = load_library()
    out = _compress_out(kv, score, ratio, out)
    b, sq, d = kv.shape
    _check("csa_compress", lib.csa_compress(kv.data_ptr(), kv.stride(0), score.data_ptr(),
                                            score.shape[2], out.data_ptr(), out.stride(0), b, sq,
                                            d, ratio, _dt(kv), _stream(stream)))
    return out


def csa_compress_overlap(kv: torch.Tensor, score: torch.Tensor, ratio: int, coff: int,
                         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """csa_compress with windows of `coff` blocks ending at each entry's own
    block (coff = 1 is csa_compress)."""
    lib = load_library()
    out = _compress_out(kv, score, ratio, out)
    b, sq, d = kv.shape
    _check("csa_compress_overlap", lib.csa_compress_overlap(
        kv.data_ptr(), kv.stride(0), score.data_ptr(), score.shape[2], out.data_ptr(),
        out.stride(0), b, sq, d, ratio, coff, _dt(kv), _stream(stream)))
    return out


def _compress_bwd_args(kv, score, dout, dkv, dscore):
    _need(kv, "kv", contiguous=False)
    _need(score, "score", dtype=kv.dtype)
    _need(dout, "dout", dtype=torch.float32, contiguous=False)
    _need(dkv, "dkv", dtype=torch.float32, contiguous=False)
    b, sq, d = kv.shape
    for t, n in ((kv, "kv"), (dout, "dout"), (dkv, "dkv")):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{n} rows must be contiguous")
    if dscore is None:
        dscore = torch.empty(b, sq, score.shape[2], dtype=torch.float32, device=kv.device)
    _need(dscore, "dscore", dtype=torch.float32)
    return dscore


def csa_compress_bwd(kv: torch.Tensor, score: torch.Tensor, ratio: int, dout: torch.Tensor,
                     dkv: torch.Tensor, dscore: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """Gradient of the pooling: adds w*dout into dkv (in place) and returns
    dscore.  kv [b, sq, d] and dkv [b, sq, d] (fp32) may be row-contiguous
    views (kv_full[:, :sq], dkv_full[:, :sq]); dout [b, sq//ratio, d] fp32 may
    be dkv_full[:, sq:]."""
    lib = load_library()
    dscore = _compress_bwd_args(kv, score, dout, dkv, dscore)
    b, sq, d = kv.shape
    _check("csa_compress_bwd", lib.csa_compress_bwd(
        kv.data_ptr(), kv.stride(0), score.data_ptr(), score.shape[2], dout.data_ptr(),
        dout.stride(0), dkv.data_ptr(), dkv.stride(0), dscore.data_ptr(), b, sq, d, ratio,
        _dt(kv), _stream(stream)))
    return dscore


def csa_compress_overlap_bwd(kv: torch.Tensor, score: torch.Tensor, ratio: int, coff: int,
                             dout: torch.Tensor, dkv: torch.Tensor,
                             dscore: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Gradient of csa_compress_overlap (arguments as csa_compress_bwd)."""
    lib = load_library()
    dscore = _compress_bwd_args(kv, score, dout, dkv, dscore)
    b, sq, d = kv.shape
    _check("csa_compress_overlap_bwd", lib.csa_compress_overlap_bwd(
        kv.data_ptr(), kv.stride(0), score.data_ptr(), score.shape[2], dout.data_ptr(),
        dout.stride(0), dkv.data_ptr(), dkv.stride(0), dscore.data_ptr(), b, sq, d, ratio, coff,
        _dt(kv), _stream(stream)))
    return dscore


def csa_compress_norm_rope(kv: torch.Tensor, score: torch.Tensor, ratio: int,
                           norm_weight: torch.Tensor, eps: float, rope_dim: int,
                           rope_base: float = 40000.0, out: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """csa_compress, then the RMS normalization (norm_weight [d] fp32, eps) and
    the rotary embedding (last rope_dim channels, interleaved pairs, entry j
    at position (j+1)*ratio - 1) of each pooled row; arguments otherwise as
    csa_compress."""
    lib = load_library()
    out = _compress_out(kv, score, ratio, out)
    _need(norm_weight, "norm_weight", dtype=torch.float32)
    b, sq, d = kv.shape
    _check("csa_compress_norm_rope", lib.csa_compress_norm_rope(
        kv.data_ptr(), kv.stride(0), score.data_ptr(), score.shape[2], norm_weight.data_ptr(),
        float(eps), int(rope_dim), float(rope_base), out.data_ptr(), out.stride(0), b, sq, d,
        ratio, _dt(kv), _stream(stream)))
    return out


def csa_compress_norm_rope_bwd(kv: torch.Tensor, score: torch.Tensor, ratio: int,
                               norm_weight: torch.Tensor, eps: float, rope_dim: int,
                               rope_base: float, dout: torch.Tensor, dkv: torch.Tensor,
                               dscore: Optional[torch.Tensor] = None,
                               dnorm_weight: Optional[torch.Tensor] = None, stream=None):
    """Gradient of csa_compress_norm_rope: adds the pooling's share into dkv
    (in place) and returns (dscore, dnorm_weight)."""
    lib = load_library()
    dscore = _compress_bwd_args(kv, score, dout, dkv, dscore)
    _need(norm_weight, "norm_weight", dtype=torch.float32)
    b, sq, d = kv.shape
    if dnorm_weight is None:
        dnorm_weight = torch.empty(d, dtype=torch.float32, device=kv.device)
    _need(dnorm_weight, "dnorm_weight", dtype=torch.float32)
    _check("csa_compress_norm_rope_bwd", lib.csa_compress_norm_rope_bwd(
        kv.data_ptr(), kv.stride(0), score.data_ptr(), score.shape[2], norm_weight.data_ptr(),
        float(eps), int(rope_dim), float(rope_base), dout.data_ptr(), dout.stride(0),
        dkv.data_ptr(), dkv.stride(0), dscore.data_ptr(), dnorm_weight.data_ptr(), b, sq, d,
        ratio, _dt(kv), _stream(stream)))
    return dscore, dnorm_weight


def csa_indexer_topk_workspace_size(b: int, sq: int, n_c: int, H_I: int, d_I: int, topk: int,
                                    dtype=torch.bfloat16) -> int:
    lib = load_library()
    dt = CSA_BF16 if dtype == torch.bfloat16 else CSA_FP32
    return int(lib.csa_indexer_topk_workspace_size(b, sq, n_c, H_I, d_I, topk, dt))


def csa_indexer_topk(q_I: torch.Tensor, k_I: torch.Tensor, w: torch.Tensor, topk: int, ratio: int,
                     workspace: Optional[torch.Tensor] = None,
                     out_idx: Optional[torch.Tensor] = None,
                     out_score: Optional[torch.Tensor] = None, return_scores: bool = False,
                     stream=None, doc_ids: Optional[torch.Tensor] = None,
                     rows: Optional[Tuple[int, int]] = None):
    """Lightning-indexer scores + exact causal top-k.

    q_I [b, sq, H_I, d_I], k_I [b, n_c, d_I] (same dtype), w [b, sq, H_I] fp32,
    doc_ids [b, sq] int32 (optional: packed documents, a block is selectable
    only by queries of its own document).  Returns idx [b, sq, K] int32 (and
    the fp32 scores [b, sq, K] when return_scores or out_score is given).
    rows=(t_begin, t_end): only those query rows of every batch element
    (csa_indexer_topk_rows); the other rows of the outputs are not written.
    """
    lib = load_library()
    _need(q_I, "q_I")
    _need(k_I, "k_I", dtype=q_I.dtype)
    _need(w, "w", dtype=torch.float32)
    b, sq, H_I, d_I = q_I.shape
    n_c = k_I.shape[1]
    K = min(topk, n_c)
    dev = q_I.device
    if workspace is None:
        nbytes = csa_indexer_topk_workspace_size(b, sq, n_c, H_I, d_I, topk, q_I.dtype)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace")
    if out_idx is None:
        out_idx = torch.empty(b, sq, K, dtype=torch.int32, device=dev)
    _need(out_idx, "out_idx", dtype=torch.int32)
    if out_score is None and return_scores:
        out_score = torch.empty(b, sq, K, dtype=torch.float32, device=dev)
    if out_score is not None:
        _need(out_score, "out_score", dtype=torch.float32)
    if doc_ids is not None:
        _need(doc_ids, "doc_ids", dtype=torch.int32)
    args = (q_I.data_ptr(), k_I.data_ptr(), w.data_ptr(), _ptr(doc_ids), out_idx.data_ptr(),
            _ptr(out_score), b, sq, n_c, H_I, d_I, ratio, topk, _dt(q_I), workspace.data_ptr(),
            workspace.numel() * workspace.element_size())
    if rows is None:
        _check("csa_indexer_topk", lib.csa_indexer_topk(*args, _stream(stream)))
    else:
        _check("csa_indexer_topk_rows", lib.csa_indexer_topk_rows(*args, int(rows[0]),
                                                                  int(rows[1]), _stream(stream)))
    if out_score is not None:
        return out_idx, out_score
    return out_idx


def csa_quantize_e4m3(x: torch.Tensor, codes: Optional[torch.Tensor] = None,
                      scale: Optional[torch.Tensor] = None, stream=None
                      ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-row (last axis) e4m3 quantization of a bf16 / fp32 tensor.

    Returns codes (uint8 e4m3 bit patterns, x's shape) and scale (fp32,
    x.shape[:-1]) with x ~= e4m3(codes) * scale[..., None]."""
    lib = load_library()
    _need(x, "x")
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(codes, "codes", dtype=torch.uint8)
    _need(scale, "scale", dtype=torch.float32)
    _check("csa_quantize_e4m3", lib.csa_quantize_e4m3(
        x.data_ptr(), rows, d, _dt(x), codes.data_ptr(), scale.data_ptr(), _stream(stream)))
    return codes, scale


def csa_indexer_topk_fp8(q8: torch.Tensor, q_scale: torch.Tensor, k8: torch.Tensor,
                         k_scale: torch.Tensor, w: torch.Tensor, topk: int, ratio: int,
                         workspace: Optional[torch.Tensor] = None,
                         out_idx: Optional[torch.Tensor] = None,
                         out_score: Optional[torch.Tensor] = None, return_scores: bool = False,
                         stream=None, doc_ids: Optional[torch.Tensor] = None):
    """csa_indexer_topk on e4m3 codes: q8 [b, sq, H_I, d_I] and k8 [b, n_c, d_I]
    uint8 with fp32 per-row scales q_scale [b, sq, H_I], k_scale [b, n_c]
    (csa_quantize_e4m3); other arguments and the outputs as csa_indexer_topk."""
    lib = load_library()
    _need(q8, "q8", dtype=torch.uint8)
    _need(k8, "k8", dtype=torch.uint8)
    _need(q_scale, "q_scale", dtype=torch.float32)
    _need(k_scale, "k_scale", dtype=torch.float32)
    _need(w, "w", dtype=torch.float32)
    b, sq, H_I, d_I = q8.shape
    n_c = k8.shape[1]
    K = min(topk, n_c)
    dev = q8.device
    if workspace is None:
        nbytes = csa_indexer_topk_workspace_size(b, sq, n_c, H_I, d_I, topk)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace")
    if out_idx is None:
        out_idx = torch.empty(b, sq, K, dtype=torch.int32, device=dev)
    _need(out_idx, "out_idx", dtype=torch.int32)
    if out_score is None and return_scores:
        out_score = torch.empty(b, sq, K, dtype=torch.float32, device=dev)
    if out_score is not None:
        _need(out_score, "out_score", dtype=torch.float32)
    if doc_ids is not None:
        _need(doc_ids, "doc_ids", dtype=torch.int32)
    _check("csa_indexer_topk_fp8", lib.csa_indexer_topk_fp8(
        q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(), w.data_ptr(),
        _ptr(doc_ids), out_idx.data_ptr(), _ptr(out_score), b, sq, n_c, H_I, d_I, ratio, topk,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)))
    if out_score is not None:
        return out_idx, out_score
    return out_idx


def csa_attn_fwd(q: torch.Tensor, kv_full: torch.Tensor, idx: Optional[torch.Tensor],
                 sink: Optional[torch.Tensor], scale: float, ratio: int, window: int,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream=None, doc_ids: Optional[torch.Tensor] = None,
                 rows: Optional[Tuple[int, int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse MQA forward; idx None = every visible compressed block;
    doc_ids [b, sq] int32 (optional) keeps only window rows of the query's
    own document.  rows=(t_begin, t_end): only those query rows
    (csa_attn_fwd_rows)."""
    lib = load_library()
    _need(q, "q")
    _need(kv_full, "kv_full", dtype=q.dtype)
    b, sq, H, d = q.shape
    n_c = kv_full.shape[1] - sq
    K = 0
    if idx is not None:
        _need(idx, "idx", dtype=torch.int32)
        K = idx.shape[2]
    if sink is not None:
        _need(sink, "sink", dtype=torch.float32)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(b, sq, H, dtype=torch.float32, device=q.device)
    _need(out, "out", dtype=q.dtype)
    _need(lse, "lse", dtype=torch.float32)
    if doc_ids is not None:
        _need(doc_ids, "doc_ids", dtype=torch.int32)
    args = (q.data_ptr(), kv_full.data_ptr(), _ptr(idx), _ptr(sink), _ptr(doc_ids), float(scale),
            out.data_ptr(), lse.data_ptr(), b, sq, H, d, n_c, ratio, window, K, _dt(q))
    if rows is None:
        _check("csa_attn_fwd", lib.csa_attn_fwd(*args, _stream(stream)))
    else:
        _check("csa_attn_fwd_rows", lib.csa_attn_fwd_rows(*args, int(rows[0]), int(rows[1]),
                                                          _stream(stream)))
    return out, lse


def csa_attn_bwd(q: torch.Tensor, kv_full: torch.Tensor, idx: Optional[torch.Tensor],
                 sink: Optional[torch.Tensor], scale: float, ratio: int, window: int,
                 o: torch.Tensor, lse: torch.Tensor, dO: torch.Tensor,
                 dq: Optional[torch.Tensor] = None, dkv: Optional[torch.Tensor] = None,
                 dsink: Optional[torch.Tensor] = None, stream=None,
                 doc_ids: Optional[torch.Tensor] = None,
                 rows: Optional[Tuple[int, int]] = None, accumulate: bool = False):
    """Sparse MQA backward; returns (dq, dkv, dsink) in fp32.  doc_ids as in
    csa_attn_fwd.  rows=(t_begin, t_end): only those query rows
    (csa_attn_bwd_rows); with accumulate their dkv / dsink contributions are
    added to what dkv / dsink hold instead of overwriting them."""
    lib = load_library()
    _need(q, "q")
    _need(kv_full, "kv_full", dtype=q.dtype)
    _need(o, "o", dtype=q.dtype)
    _need(dO, "dO", dtype=q.dtype)
    _need(lse, "lse", dtype=torch.float32)
    b, sq, H, d = q.shape
    n_kv = kv_full.shape[1]
    n_c = n_kv - sq
    K = 0
    if idx is not None:
        _need(idx, "idx", dtype=torch.int32)
        K = idx.shape[2]
    if sink is not None:
        _need(sink, "sink", dtype=torch.float32)
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty(b, sq, H, d, **f32) if dq is None else dq
    dkv = torch.empty(b, n_kv, d, **f32) if dkv is None else dkv
    if dsink is None and sink is not None:
        dsink = torch.empty(H, **f32)
    _need(dq, "dq", dtype=torch.float32)
    _need(dkv, "dkv", dtype=torch.float32)
    if doc_ids is not None:
        _need(doc_ids, "doc_ids", dtype=torch.int32)
    args = (q.data_ptr(), kv_full.data_ptr(), _ptr(idx), _ptr(sink), _ptr(doc_ids), float(scale),
            o.data_ptr(), lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dkv.data_ptr(),
            _ptr(dsink), b, sq, H, d, n_c, ratio, window, K, _dt(q))
    if rows is None and not accumulate:
        _check("csa_attn_bwd", lib.csa_attn_bwd(*args, _stream(stream)))
    else:
        t0, t1 = (0, sq) if rows is None else rows
        _check("csa_attn_bwd_rows", lib.csa_attn_bwd_rows(*args, int(t0), int(t1),
                                                          int(bool(accumulate)),
                                                          _stream(stream)))
    return dq, dkv, dsink


def csa_get_device_status(stream=None, with_site: bool = False):
    """Synchronize the stream, then read and clear the device status word.

    Returns the status code (0 = OK), or (code, site) with `with_site`."""
    lib = load_library()
    v = ctypes.c_int(0)
    site = ctypes.c_int(0)
    _check("csa_get_device_status", lib.csa_get_device_status(_stream(stream), ctypes.byref(v),
                                                              ctypes.byref(site)))
    return (v.value, site.value) if with_site else v.value


def csa_debug_arm_fault(site: int):
    """Test hook: make later tensor-core attention forwards fake a failure at
    `site` (0x21: the Q-tile wait runs out; 0x25: the union check trips);
    0 disarms.  Synchronizes the device."""
    _check("csa_debug_arm_fault", load_library().csa_debug_arm_fault(int(site)))


def csa_indexer_teacher(q: torch.Tensor, kv_full: torch.Tensor, idx: torch.Tensor,
                        lse: torch.Tensor, scale: float, ratio: int,
                        out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Distillation target [b, sq, K] fp32 of the indexer: per valid slot,
    sum over heads of exp(scale q.kv - lse), L1-normalized per row."""
    lib = load_library()
    _need(q, "q")
    _need(kv_full, "kv_full", dtype=q.dtype)
    _need(idx, "idx", dtype=torch.int32)
    _need(lse, "lse", dtype=torch.float32)
    b, sq, H, d = q.shape
    n_c = kv_full.shape[1] - sq
    K = idx.shape[2]
    if out is None:
        out = torch.empty(b, sq, K, dtype=torch.float32, device=q.device)
    _need(out, "out", dtype=torch.float32)
    _check("csa_indexer_teacher", lib.csa_indexer_teacher(
        q.data_ptr(), kv_full.data_ptr(), idx.data_ptr(), lse.data_ptr(), float(scale),
        out.data_ptr(), b, sq, H, d, n_c, ratio, K, _dt(q), _stream(stream)))
    return out


def csa_indexer_loss(q_I: torch.Tensor, k_I: torch.Tensor, w: torch.Tensor, idx: torch.Tensor,
                     target: torch.Tensor, ratio: int, stream=None):
    """KL distillation loss of the indexer over its selected entries and its
    gradients: returns (loss [b, sq], dq_I, dk_I, dw), all fp32."""
    lib = load_library()
    _need(q_I, "q_I")
    _need(k_I, "k_I", dtype=q_I.dtype)
    _need(w, "w", dtype=torch.float32)
    _need(idx, "idx", dtype=torch.int32)
    _need(target, "target", dtype=torch.float32)
    b, sq, H_I, d_I = q_I.shape
    n_c = k_I.shape[1]
    K = idx.shape[2]
    f32 = dict(dtype=torch.float32, device=q_I.device)
    loss = torch.empty(b, sq, **f32)
    dq = torch.empty(b, sq, H_I, d_I, **f32)
    dk = torch.empty(b, n_c, d_I, **f32)
    dw = torch.empty(b, sq, H_I, **f32)
    _check("csa_indexer_loss", lib.csa_indexer_loss(
        q_I.data_ptr(), k_I.data_ptr(), w.data_ptr(), idx.data_ptr(), target.data_ptr(),
        loss.data_ptr(), dq.data_ptr(), dk.data_ptr(), dw.data_ptr(), b, sq, n_c, H_I, d_I, ratio,
        K, _dt(q_I), _stream(stream)))
    return loss, dq, dk, dw
