"""GB300-native (sm_103a) Compressed Sparse Attention hot path.

The library is the C ABI in include/csa.h, built as libcsa.so next to this
file.  ``csa`` is its Python binding (same function names); ``inputs`` holds
the seeded synthetic workloads.  Importing the package does not load the
library; the first call does, and raises if it is missing.
"""
from .csa import (csa_attn_bwd, csa_attn_fwd, csa_compress, csa_compress_bwd,  # noqa: F401
                  csa_compress_overlap, csa_compress_overlap_bwd,
                  csa_get_device_status, csa_indexer_loss, csa_indexer_teacher, csa_indexer_topk,
                  csa_indexer_topk_fp8, csa_indexer_topk_workspace_size, csa_quantize_e4m3, load_library, CSAError)
