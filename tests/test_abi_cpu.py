"""The C ABI library on the host (no GPU needed): it loads, exports every
symbol include/csa.h declares, and rejects invalid arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

from compressed_sparse_attention_sum_gb300 import build, csa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return csa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_steps():
    names = declared_functions()
    for n in ("csa_compress", "csa_indexer_topk", "csa_attn_fwd", "csa_attn_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    # the binding declares a signature for each of them
    assert set(names) <= set(csa.SIGNATURES)


def test_status_strings(lib):
    for code in range(7):
        s = lib.csa_status_string(code).decode()
        assert s.startswith("CSA"), s
    assert lib.csa_version() >= 100


def test_workspace_sizes(lib):
    # full score matrix when small, capped at 128 MiB, never below one tile
    assert lib.csa_indexer_topk_workspace_size(1, 4096, 1024, 64, 128, 512, 1) == 4096 * 1024 * 4
    assert lib.csa_indexer_topk_workspace_size(2, 8192, 2048, 64, 128, 1024, 1) == 128 << 20
    assert lib.csa_indexer_topk_min_workspace(2, 2048) == 2 * 128 * 2048 * 4
    assert lib.csa_indexer_topk_workspace_size(0, 1, 1, 1, 8, 1, 1) == 0


P = ctypes.c_void_p


def test_invalid_arguments_rejected_on_host(lib):
    INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 4
    fake = 0x10000  # never dereferenced: validation fails first
    # null pointers
    assert lib.csa_attn_fwd(None, fake, None, None, None, 0.1, fake, fake, 1, 8, 1, 64, 2, 4, 4, 0, 1,
                            None) == INVALID
    # misaligned pointer
    assert lib.csa_attn_fwd(fake + 2, fake, None, None, None, 0.1, fake, fake, 1, 8, 1, 64, 2, 4, 4, 0, 1,
                            None) == INVALID
    # d not a multiple of 8
    assert lib.csa_attn_fwd(fake, fake, None, None, None, 0.1, fake, fake, 1, 8, 1, 60, 2, 4, 4, 0, 1,
                            None) == INVALID
    # n_c inconsistent with sq / ratio
    assert lib.csa_attn_fwd(fake, fake, None, None, None, 0.1, fake, fake, 1, 8, 1, 64, 3, 4, 4, 0, 1,
                            None) == INVALID
    # window < 1
    assert lib.csa_attn_bwd(fake, fake, None, None, None, 0.1, fake, fake, fake, fake, fake, None, 1, 8, 1,
                            64, 2, 4, 0, 0, 1, None) == INVALID
    # sink without dsink
    assert lib.csa_attn_bwd(fake, fake, None, fake, None, 0.1, fake, fake, fake, fake, fake, None, 1, 8, 1,
                            64, 2, 4, 4, 0, 1, None) == INVALID
    # d > 512
    assert lib.csa_attn_fwd(fake, fake, None, None, None, 0.1, fake, fake, 1, 8, 1, 520, 2, 4, 4, 0, 1,
                            None) == UNSUPPORTED
    # bad dtype
    assert lib.csa_attn_fwd(fake, fake, None, None, None, 0.1, fake, fake, 1, 8, 1, 64, 2, 4, 4, 0, 7,
                            None) == INVALID
    # compress: score width must be 1 or d
    assert lib.csa_compress(fake, 512, fake, 3, fake, 128, 1, 8, 64, 4, 1, None) == INVALID
    # compress: ratio larger than sq
    assert lib.csa_compress(fake, 512, fake, 64, fake, 128, 1, 8, 64, 16, 1, None) == INVALID
    # indexer: workspace too small
    assert lib.csa_indexer_topk(fake, fake, fake, None, fake, None, 1, 512, 128, 4, 64, 4, 16, 1, fake,
                                64, None) == WORKSPACE
    # indexer: topk < 1
    assert lib.csa_indexer_topk(fake, fake, fake, None, fake, None, 1, 512, 128, 4, 64, 4, 0, 1, fake,
                                1 << 20, None) == INVALID
    # misaligned document ids
    assert lib.csa_attn_fwd(fake, fake, None, None, fake + 4, 0.1, fake, fake, 1, 8, 1, 64, 2, 4, 4,
                            0, 1, None) == INVALID
    assert lib.csa_indexer_topk(fake, fake, fake, fake + 4, fake, None, 1, 512, 128, 4, 64, 4, 16,
                                1, fake, 1 << 30, None) == INVALID
    # teacher: null lse; head dim not a multiple of 8
    assert lib.csa_indexer_teacher(fake, fake, fake, None, 0.1, fake, 1, 8, 2, 64, 2, 4, 4, 1,
                                   None) == INVALID
    assert lib.csa_indexer_teacher(fake, fake, fake, fake, 0.1, fake, 1, 8, 2, 60, 2, 4, 4, 1,
                                   None) == INVALID
    # loss: null gradient output; d_I beyond the supported maximum
    assert lib.csa_indexer_loss(fake, fake, fake, fake, fake, fake, fake, None, fake, 1, 8, 2, 4,
                                64, 4, 4, 1, None) == INVALID
    assert lib.csa_indexer_loss(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 8, 2, 4,
                                512, 4, 4, 1, None) == UNSUPPORTED
    # e4m3 quantization: row width not a multiple of 8; misaligned codes; no rows is a no-op
    assert lib.csa_quantize_e4m3(fake, 4, 12, 1, fake, fake, None) == INVALID
    assert lib.csa_quantize_e4m3(fake, 4, 64, 1, fake + 8, fake, None) == INVALID
    assert lib.csa_quantize_e4m3(None, 0, 64, 1, None, None, None) == 0
    # FP8 indexer: null scale; d_I not a multiple of 16; workspace too small
    assert lib.csa_indexer_topk_fp8(fake, None, fake, fake, fake, None, fake, None, 1, 512, 128, 4,
                                    128, 4, 16, fake, 1 << 20, None) == INVALID
    assert lib.csa_indexer_topk_fp8(fake, fake, fake, fake, fake, None, fake, None, 1, 512, 128, 4,
                                    40, 4, 16, fake, 1 << 20, None) == INVALID
    assert lib.csa_indexer_topk_fp8(fake, fake, fake, fake, fake, None, fake, None, 1, 512, 128, 4,
                                    128, 4, 16, fake, 64, None) == WORKSPACE
    # overlapping compression: coff < 1 invalid, coff > 2 unsupported
    assert lib.csa_compress_overlap(fake, 512, fake, 64, fake, 128, 1, 8, 64, 4, 0, 1,
                                    None) == INVALID
    assert lib.csa_compress_overlap(fake, 512, fake, 64, fake, 128, 1, 8, 64, 4, 3, 1,
                                    None) == UNSUPPORTED
    assert lib.csa_compress_overlap_bwd(fake, 512, fake, 64, fake, 128, None, 512, fake, 1, 8,
                                        64, 4, 2, 1, None) == INVALID
    # device status needs an output pointer; the test hook takes no negative site
    assert lib.csa_get_device_status(None, None, None) == INVALID
    assert lib.csa_debug_arm_fault(-1) == INVALID


def test_binding_fails_loudly_without_library(tmp_path):
    saved = csa._lib
    try:
        csa._lib = None
        with pytest.raises(RuntimeError):
            csa.load_library(str(tmp_path / "missing.so"))
    finally:
        csa._lib = saved
