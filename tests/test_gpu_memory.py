"""Peak device memory of one production-width layer step.

The gather-backward review of "Add unfused SBHD compressed sparse attention"
rejects any backward that materialises a [b, sq, n_kv, d] tensor (5.4 GB at
CSA-4; 343 GB in fp32 at the production width), and "Add the min-memory DSA
attention kernels" tests peak CUDA allocation against the planned tile.  The
library allocates no device memory at all: every buffer is the caller's.  So
with every output and the indexer workspace allocated up front, a whole layer
step (compress, indexer + top-k, forward, backward, compressor backward)
must leave the caller's allocator peak where it was and the device's free
memory unchanged.
"""
import pytest
import torch

from compressed_sparse_attention_sum_gb300 import csa
from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from compressed_sparse_attention_sum_gb300 import build
    build.build()
    csa.load_library()


def test_production_layer_allocates_nothing():
    cfg = CONFIGS["prod_bf16"]
    x = {k: v.cuda() for k, v in make_inputs(cfg).items()}
    b, sq, d, n_c, H = cfg.b, cfg.sq, cfg.d, cfg.n_c, cfg.H
    dev = x["q"].device
    kv_full = torch.empty(b, sq + n_c, d, dtype=cfg.torch_dtype, device=dev)
    ws = torch.empty(csa.csa_indexer_topk_workspace_size(b, sq, n_c, cfg.H_I, cfg.d_I, cfg.topk),
                     dtype=torch.uint8, device=dev)
    idx_i = torch.empty(b, sq, cfg.K, dtype=torch.int32, device=dev)
    O = torch.empty(b, sq, H, d, dtype=cfg.torch_dtype, device=dev)
    L = torch.empty(b, sq, H, dtype=torch.float32, device=dev)
    dq = torch.empty(b, sq, H, d, dtype=torch.float32, device=dev)
    dkv = torch.empty(b, sq + n_c, d, dtype=torch.float32, device=dev)
    dsink = torch.empty(H, dtype=torch.float32, device=dev)
    dscore = torch.empty(b, sq, d, dtype=torch.float32, device=dev)

    def step():
        kv_full[:, :sq].copy_(x["kv_raw"])
        csa.csa_compress(kv_full[:, :sq], x["score"], cfg.ratio, out=kv_full[:, sq:])
        csa.csa_indexer_topk(x["q_I"], x["k_I"], x["w"], cfg.topk, cfg.ratio, workspace=ws,
                             out_idx=idx_i)
        csa.csa_attn_fwd(x["q"], kv_full, x["idx"], x["sink"], cfg.scale, cfg.ratio, cfg.window,
                         out=O, lse=L)
        csa.csa_attn_bwd(x["q"], kv_full, x["idx"], x["sink"], cfg.scale, cfg.ratio, cfg.window,
                         O, L, x["dO"], dq=dq, dkv=dkv, dsink=dsink)
        csa.csa_compress_bwd(kv_full[:, :sq], x["score"], cfg.ratio, dkv[:, sq:], dkv[:, :sq],
                             dscore=dscore)

    step()                                  # first calls load the kernels
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    free0, total = torch.cuda.mem_get_info()
    step()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated()
    free1, _ = torch.cuda.mem_get_info()
    dense = b * sq * (sq + n_c) * d * 4
    print(f"prod_bf16 step: caller buffers {base / 2**30:.2f} GiB, peak above them "
          f"{(peak - base) / 2**20:.2f} MiB, device free memory change "
          f"{(free0 - free1) / 2**20:.2f} MiB; a dense fp32 [b, sq, n_kv, d] would be "
          f"{dense / 2**30:.0f} GiB")
    assert peak - base == 0, peak - base
    assert abs(free0 - free1) <= (2 << 20), free0 - free1
    assert csa.csa_get_device_status() == 0
