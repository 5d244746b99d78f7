"""The library allocates no device memory: no CUDA allocation or free call
appears in its sources (every buffer, including the indexer workspace, is the
caller's; csa_indexer_topk_noalloc keeps a fixed file-scope array)."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "compressed_sparse_attention_sum_gb300", "csrc")

_ALLOC = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*|cuMemFree\w*|cudaMemPool\w*|"
                    r"malloc|free)\s*\(")


def _code(path):
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def test_sources_call_no_allocator():
    files = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                   + glob.glob(os.path.join(CSRC, "*.h")))
    assert files
    bad = [(os.path.basename(f), m.group(1)) for f in files for m in _ALLOC.finditer(_code(f))]
    assert not bad, bad
