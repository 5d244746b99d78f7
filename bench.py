"""Benchmark of the CSA hot path on GB300: one step = one CSA layer,
forward + backward: csa_compress -> csa_indexer_topk -> csa_attn_fwd ->
csa_attn_bwd -> csa_compress_bwd (the compressed rows' gradient flowing back
through the pooling), by default on the CSA-4 workload (b=1, sq=4096, H=32,
d=128, ratio 4, n_c=1024, window 128, topk 512, indexer 64 heads x 128).

Prints one JSON line.  `value` is queries/s of the whole job (all ranks),
device-timed with CUDA events around each step on the launching stream; the
L2 is flushed before every timed step (a 256 MiB write, then a 256 MiB read
that leaves no dirty lines for the timed kernels to write back).  `e2e` is the same
metric through the C ABI from pinned host buffers, with every step's
host->device input copies and device->host result copies inside the timed
region.  `roofline` describes the kernel with the largest share of the
step.  `cpu_baseline` is the fp64 oracle on the host cores over a bounded
sample of query rows of the same workload.

--impl reference times the fp64 oracle on the host cores (the method's
published sources include no runnable implementation to time instead).
--workload picks one of the five workloads; --sweep times all of them.
Multi-GPU: one process per GPU (torchrun); the ranks split the layer's query
rows into contiguous ranges of equal estimated work (row-range calls of the
library) and sum their dkv / dsink contributions with one all-reduce, so the
layer is fixed as N grows (strong scaling); timing takes the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "csa4_bf16"
METRIC = "CSA fwd+bwd ms/layer & queries/s at sq=4096; % of HBM / tensor-core roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# oracle CPU baseline (spawned worker processes, one BLAS thread each)
# ---------------------------------------------------------------------------

# Query rows of the oracle sample per workload: the whole layer where the
# oracle finishes it in seconds, else a bounded sample (10-30 s of CPU work).
CPU_ROWS = {"tiny_fp32": 256, "debug_bf16": 2048, "csa4_bf16": 4096, "hca_bf16": 16384,
            "prod_bf16": 4096}


class OraclePool:
    """The oracle on every host core (oracle.rows_pool): one process per core
    over memory-mapped inputs of one workload."""

    def __init__(self, cfg_name, procs=None):
        import numpy as np
        from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs
        from oracle import csa_oracle as orc
        from oracle.rows_pool import RowPool
        self.cfg = cfg = CONFIGS[cfg_name]
        inp = make_inputs(cfg)
        f = lambda t: t.double().numpy()
        kv_raw = f(inp["kv_raw"])
        t0 = time.perf_counter()
        kv_c = orc.compress(kv_raw, f(inp["score"]), cfg.ratio, out_dtype=cfg.dtype)
        self.t_compress = time.perf_counter() - t0          # whole sequence, all batch rows
        arrays = {"kv_full": np.concatenate([kv_raw, kv_c], axis=1), "q": inp["q"],
                  "dO": inp["dO"], "sink": inp["sink"].numpy(), "idx": inp.get("idx"),
                  "q_I": inp.get("q_I"), "k_I": inp.get("k_I"), "w": inp.get("w")}
        self.pool = RowPool(arrays, procs)
        self.procs = self.pool.procs
        self.run(self.procs, seed=12345)                     # warm every worker

    def run(self, rows_total, seed):
        """Time `rows_total` query rows drawn uniformly over (b, t) (the causal
        mix of short and long rows); returns (seconds, rows)."""
        import numpy as np
        from oracle.rows_pool import split_rows
        cfg = self.cfg
        rng = np.random.default_rng(seed)
        flat = np.sort(rng.choice(cfg.b * cfg.sq, size=min(rows_total, cfg.b * cfg.sq),
                                  replace=False))
        rows = [(int(i // cfg.sq), int(i % cfg.sq)) for i in flat]
        kw = dict(scale=cfg.scale, window=cfg.window, ratio=cfg.ratio, K=cfg.K,
                  indexer=cfg.H_I > 0)
        t0 = time.perf_counter()
        self.pool.map("oracle.rows_pool.layer_rows",
                      [dict(rows=c, **kw) for c in split_rows(rows, self.procs)])
        wall = time.perf_counter() - t0
        # the pooling of the whole layer is charged pro rata
        return wall + self.t_compress * len(rows) / (cfg.b * cfg.sq), len(rows)

    def close(self):
        self.pool.close()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS)


def load_traffic():
    """Per-launch DRAM bytes of the kernels from the committed ncu summary,
    valid only while the kernel source is unchanged."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return {}
    out = {}
    for name, rec in d.items():
        src = os.path.join(ROOT, rec["source"])
        try:
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except OSError:
            continue
        if h == rec.get("source_sha256_16"):
            out[name] = rec
    return out


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def algorithmic_work(cfg, idx, ranges=None):
    """Algorithmic units of one step (valid slots only; MQA rows gathered once
    per query and shared by the heads); with `ranges`, of those query rows
    only (the attention and indexer units; the compressor runs whole)."""
    import torch
    sq, ratio, W, d, H = cfg.sq, cfg.ratio, cfg.window, cfg.d, cfg.H
    t = torch.arange(sq, device=idx.device)
    keep = torch.ones(sq, dtype=torch.bool, device=idx.device)
    if ranges is not None:
        keep = torch.zeros_like(keep)
        for lo, hi in ranges:
            keep[lo:hi] = True
    vis = ((t + 1) // ratio).view(1, sq, 1)
    valid_c = (((idx >= 0) & (idx < vis)) & keep.view(1, sq, 1)).sum().item()
    n_win = cfg.b * int((torch.clamp(t + 1, max=W) * keep).sum().item())
    slots = valid_c + n_win
    e = 2 if cfg.dtype == "bf16" else 4
    vis_sum = cfg.b * int((((t + 1) // ratio).clamp(max=cfg.n_c) * keep).sum().item())
    return {
        "slots": slots,
        "compress_bytes": cfg.b * (2 * cfg.sq * d + cfg.n_c * d) * e,
        # kv + score read, pooled-row gradient read, raw-row gradient read and
        # written, score gradient written
        "compress_bwd_bytes": cfg.b * (2 * cfg.sq * d * e + cfg.n_c * d * 4 + 3 * cfg.sq * d * 4),
        "indexer_flops": 2.0 * cfg.H_I * cfg.d_I * vis_sum,
        "fwd_gathered_bytes": slots * d * e,
        "bwd_gathered_bytes": slots * (d * e + 4 * d),
        "fwd_flops": 4.0 * d * H * slots,
        "bwd_flops": 10.0 * d * H * slots,
    }


def max_over_ranks(value_ms, world, device=None):
    """Max of a per-rank time over all ranks (the job finishes with the slowest)."""
    if world <= 1:
        return value_ms
    import torch
    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def workload_string(cfg):
    s = (f"{cfg.name}: b={cfg.b} sq={cfg.sq} H={cfg.H} d={cfg.d} ratio={cfg.ratio} "
         f"n_c={cfg.n_c} window={cfg.window}")
    if cfg.H_I > 0:
        s += f" topk={cfg.topk} H_I={cfg.H_I} d_I={cfg.d_I}"
    if cfg.index_source == "all_visible":
        s += " (no indexer: every visible block, K=n_c)"
    elif cfg.index_source == "zipf":
        s += (f" (attention on synthetic Zipf-{cfg.zipf_exponent} top-{cfg.K} lists with "
              f"{int(cfg.pad_fraction * 100)}% -1 padding; the indexer runs on its own inputs)")
    return s


def median(xs):
    return statistics.median(xs)


def run_gpu(args, rank, world, local_rank, workload=None, variants_on=True, e2e_on=True):
    import torch
    from compressed_sparse_attention_sum_gb300 import build as _build
    _build.build()
    from compressed_sparse_attention_sum_gb300 import csa
    from compressed_sparse_attention_sum_gb300.inputs import CONFIGS, make_inputs, packed_doc_ids
    lib = csa.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from compressed_sparse_attention_sum_gb300.shard import config_ranges, layer_rows
    cfg = CONFIGS[workload or args.workload]
    if getattr(args, "seq_len", 0) or getattr(args, "batch", 0):
        cfg = cfg.with_(name=cfg.name + "_resized", sq=args.seq_len or cfg.sq,
                        b=args.batch or cfg.b)
    # N > 1: the ranks split the layer's query rows (contiguous ranges of equal
    # estimated work) and sum their dkv / dsink contributions with one
    # all-reduce; N = 1 runs the whole layer
    ranges = config_ranges(cfg, world, rank) if world > 1 else None
    inp = make_inputs(cfg)
    host = {k: v.pin_memory() for k, v in inp.items()}
    d_in = {k: v.to(dev) for k, v in inp.items()}
    b, sq, d, n_c, H = cfg.b, cfg.sq, cfg.d, cfg.n_c, cfg.H
    has_indexer = cfg.H_I > 0
    # the attention's index list: the indexer's output, or the workload's own
    # list (every visible block; synthetic Zipf lists)
    idx_given = "idx" in d_in
    kv_full = torch.empty(b, sq + n_c, d, dtype=cfg.torch_dtype, device=dev)
    ws = (torch.empty(csa.csa_indexer_topk_workspace_size(b, sq, n_c, cfg.H_I, cfg.d_I, cfg.topk,
                                                           cfg.torch_dtype), dtype=torch.uint8,
                      device=dev) if has_indexer else None)
    idx_out = torch.empty(b, sq, cfg.K, dtype=torch.int32, device=dev)
    idx = d_in["idx"] if idx_given else idx_out
    O = torch.empty(b, sq, H, d, dtype=cfg.torch_dtype, device=dev)
    L = torch.empty(b, sq, H, dtype=torch.float32, device=dev)
    dq = torch.empty(b, sq, H, d, dtype=torch.float32, device=dev)
    dkv = torch.empty(b, sq + n_c, d, dtype=torch.float32, device=dev)
    dsink = torch.empty(H, dtype=torch.float32, device=dev)
    dscore = torch.empty(b, sq, d, dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        # write 256 MiB (evicts every cached input), then read another 256 MiB
        # so that the write's dirty lines are written back here, not inside
        # the next timed kernel
        flush.zero_()
        flush_rd.amax()
    stream = torch.cuda.current_stream(dev)

    side = torch.cuda.Stream(dev)

    def step_rows(x):
        # Events 0-6 at the phase boundaries of shard.layer_rows: compress,
        # indexer, forward, backward, all-reduce, compressor backward.
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        layer_rows(csa, x, cfg, ranges, kv_full, ws, idx_out, O, L, dq, dkv, dsink, dscore,
                   idx_given, world=world, mark=lambda i: ev[i].record(stream))
        return ev

    def step(x, doc=None):
        if ranges is not None:
            return step_rows(x)
        # Events: 0 step start; 1-2 the compressor on the side stream; 3 end of
        # the indexer; 4 both joined (fwd start); 5 fwd end; 6 bwd end; 7 step
        # end.  The compressor and the indexer are independent (the attention
        # needs both), so the compressor runs beside the indexer.
        kv_full[:, :sq].copy_(x["kv_raw"])          # raw rows of the KV buffer (layer input)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
        ev[0].record(stream)
        side.wait_event(ev[0])
        ev[1].record(side)
        csa.csa_compress(kv_full[:, :sq], x["score"], cfg.ratio, out=kv_full[:, sq:], stream=side)
        ev[2].record(side)
        if has_indexer:
            csa.csa_indexer_topk(x["q_I"], x["k_I"], x["w"], cfg.topk, cfg.ratio, workspace=ws,
                                 out_idx=idx_out, doc_ids=doc)
        ev[3].record(stream)
        stream.wait_event(ev[2])
        ev[4].record(stream)
        ix = x["idx"] if idx_given else idx_out
        csa.csa_attn_fwd(x["q"], kv_full, ix, x["sink"], cfg.scale, cfg.ratio, cfg.window, out=O,
                         lse=L, doc_ids=doc)
        ev[5].record(stream)
        csa.csa_attn_bwd(x["q"], kv_full, ix, x["sink"], cfg.scale, cfg.ratio, cfg.window, O, L,
                         x["dO"], dq=dq, dkv=dkv, dsink=dsink, doc_ids=doc)
        ev[6].record(stream)
        # the compressed rows' gradient flows back through the pooling into the
        # raw rows (accumulated in place) and the pooling scores
        csa.csa_compress_bwd(kv_full[:, :sq], x["score"], cfg.ratio, dkv[:, sq:], dkv[:, :sq],
                             dscore=dscore)
        ev[7].record(stream)
        return ev

    # (start, end) events of compress, indexer_topk, attn_fwd, attn_bwd,
    # compress_bwd (and the all-reduce of the row split), and of the whole step
    if ranges is None:
        seg_pairs = ((1, 2), (0, 3), (4, 5), (5, 6), (6, 7))
        last = 7
    else:
        seg_pairs = ((0, 1), (1, 2), (2, 3), (3, 4), (5, 6), (4, 5))
        last = 6

    def segments(e):
        return [e[a].elapsed_time(e[b]) for a, b in seg_pairs]

    def step_time(e):
        return e[0].elapsed_time(e[last])

    clk = ClockSampler(local_rank)
    clk.__enter__()          # samples from the warm-up through the end-to-end loop
    for _ in range(args.warmup):
        flush_l2()
        step(d_in)
    torch.cuda.synchronize()
    work = algorithmic_work(cfg, idx, ranges)

    # ---- device-timed region -------------------------------------------------
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = []
    launches0 = lib.csa_kernel_launches()
    for _ in range(args.steps):
        flush_l2()
        evs.append(step(d_in))
    torch.cuda.synchronize()
    launches = lib.csa_kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    seg = [list(c) for c in zip(*[segments(e) for e in evs])]
    step_ms = [step_time(e) for e in evs]
    ms = median(step_ms)
    ms_max = max_over_ranks(ms, world, dev)
    queries = b * sq
    # N = 1: one layer per GPU; N > 1: the ranks share one layer (strong scaling)
    value = queries / (ms_max / 1e3)

    # ---- variants (skipped with --no-variants) ----------------------------------
    variants = {}
    names = ("compress", "indexer_topk", "attn_fwd", "attn_bwd", "compress_bwd")
    if (variants_on and not args.no_variants and has_indexer and not idx_given
            and ranges is None):
        # the same layer holding 4 packed documents (window and indexer restricted
        # to each query's document; same timing rules)
        doc = packed_doc_ids(b, sq, cfg.ratio, 4, seed=rank).to(dev)
        for _ in range(args.warmup):
            flush_l2()
            step(d_in, doc)
        evs_doc = []
        for _ in range(args.steps):
            flush_l2()
            evs_doc.append(step(d_in, doc))
        torch.cuda.synchronize()
        doc_ms = max_over_ranks(median([step_time(e) for e in evs_doc]),
                                world, dev)
        variants["docs4"] = {
            "workload": f"{cfg.name} with 4 packed documents (boundaries on multiples of the ratio)",
            "ms_per_step": round(doc_ms, 4), "value": round(queries / (doc_ms / 1e3), 1),
            "unit": "queries/s",
            "kernels_ms": {n: round(median([segments(e)[i] for e in evs_doc]),
                                    4) for i, n in enumerate(names)},
        }
        # the indexer's training path on the same layer: teacher target from the
        # forward's LSE, then the student's KL loss and gradients over the
        # selected entries (L2 flushed before each pair)
        target = torch.empty(b, sq, cfg.K, dtype=torch.float32, device=dev)
        step(d_in)
        tr_ev = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            e3 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e3[0].record(stream)
            csa.csa_indexer_teacher(d_in["q"], kv_full, idx, L, cfg.scale, cfg.ratio, out=target)
            e3[1].record(stream)
            csa.csa_indexer_loss(d_in["q_I"], d_in["k_I"], d_in["w"], idx, target, cfg.ratio)
            e3[2].record(stream)
            if i >= args.warmup:
                tr_ev.append(e3)
        torch.cuda.synchronize()
        t_teach = median([e[0].elapsed_time(e[1]) for e in tr_ev])
        t_loss = median([e[1].elapsed_time(e[2]) for e in tr_ev])
        slots_sel = int((idx >= 0).sum().item())
        variants["indexer_training"] = {
            "workload": f"{cfg.name}: indexer distillation over the top-{cfg.K} entries",
            "teacher_ms": round(t_teach, 4), "loss_ms": round(t_loss, 4),
            "teacher_tflops": round(2.0 * H * d * slots_sel / (t_teach / 1e3) / 1e12, 2),
            "loss_tflops": round(3 * 2.0 * cfg.H_I * cfg.d_I * slots_sel / (t_loss / 1e3) / 1e12,
                                 2),
            "kernels": ("teacher and loss: tcgen05, 128 / H (128 / H_I) queries per job over the "
                        "union of their selections (teacher: persistent CTAs)"),
        }
        # the FP8 indexer: per-row e4m3 quantization of q_I and k_I, then the
        # indexer top-k on the codes (tcgen05 kind::f8f6f4); the overlap is the
        # mean fraction of the bf16 top-k that the FP8 top-k keeps
        q8, qs = csa.csa_quantize_e4m3(d_in["q_I"])
        k8, ks = csa.csa_quantize_e4m3(d_in["k_I"])
        idx8 = torch.empty_like(idx)
        f8_ev = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            e3 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e3[0].record(stream)
            csa.csa_quantize_e4m3(d_in["q_I"], codes=q8, scale=qs)
            csa.csa_quantize_e4m3(d_in["k_I"], codes=k8, scale=ks)
            e3[1].record(stream)
            csa.csa_indexer_topk_fp8(q8, qs, k8, ks, d_in["w"], cfg.topk, cfg.ratio, workspace=ws,
                                     out_idx=idx8)
            e3[2].record(stream)
            if i >= args.warmup:
                f8_ev.append(e3)
        torch.cuda.synchronize()
        t_q = median([e[0].elapsed_time(e[1]) for e in f8_ev])
        t_i8 = median([e[1].elapsed_time(e[2]) for e in f8_ev])
        hit = torch.zeros(b, sq, n_c + 1, dtype=torch.int32, device=dev)
        hit.scatter_(2, torch.where(idx >= 0, idx, n_c).long(), 1)
        hit[:, :, n_c] = 0
        kept = torch.gather(hit, 2, torch.where(idx8 >= 0, idx8, n_c).long()).sum().item()
        variants["indexer_fp8"] = {
            "workload": f"{cfg.name}: indexer top-{cfg.K} on per-row e4m3 codes of q_I and k_I",
            "quantize_ms": round(t_q, 4), "indexer_topk_ms": round(t_i8, 4),
            "indexer_topk_bf16_ms": round(median(seg[1]), 4),
            "topk_overlap_with_bf16": round(kept / max(1, int((idx >= 0).sum().item())), 5),
            "kernels": "quantize: a lane group per row; scores: tcgen05 kind::f8f6f4, same select",
        }
        # overlapping compression (coff = 2: each entry pools its own block and
        # the previous one), forward and backward in the layer layout
        kvc = torch.empty(b, n_c, d, dtype=cfg.torch_dtype, device=dev)
        dkv_raw = torch.zeros(b, sq, d, dtype=torch.float32, device=dev)
        ov_ev = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            e3 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e3[0].record(stream)
            csa.csa_compress_overlap(kv_full[:, :sq], d_in["score"], cfg.ratio, 2, out=kvc)
            e3[1].record(stream)
            csa.csa_compress_overlap_bwd(kv_full[:, :sq], d_in["score"], cfg.ratio, 2,
                                         dkv[:, sq:], dkv_raw, dscore=dscore)
            e3[2].record(stream)
            if i >= args.warmup:
                ov_ev.append(e3)
        torch.cuda.synchronize()
        variants["compress_overlap"] = {
            "workload": f"{cfg.name}: compressor with coff = 2 (windows of 2 x ratio tokens)",
            "compress_ms": round(median([e[0].elapsed_time(e[1]) for e in ov_ev]), 4),
            "compress_bwd_ms": round(median([e[1].elapsed_time(e[2]) for e in ov_ev]), 4),
            "coff1_compress_ms": round(median(seg[0]), 4),
            "coff1_compress_bwd_ms": round(median(seg[4]), 4),
        }

    # ---- end-to-end through host buffers -------------------------------------
    # Every step copies all of its inputs host -> device (pinned) and all of its
    # results device -> host.  Three streams pipeline consecutive steps: step
    # i+1's inputs arrive while step i computes and step i-1's results leave;
    # inputs and results are double-buffered.  Each step moves more bytes in
    # than L2 holds (137.6 MB at CSA-4), so no flush is added here.
    e2e_res = None
    if e2e_on:
        def make_out():
            o = {"O": torch.empty_like(O), "L": torch.empty_like(L), "dq": torch.empty_like(dq),
                 "dkv": torch.empty_like(dkv), "dsink": torch.empty_like(dsink),
                 "dscore": torch.empty_like(dscore)}
            if has_indexer:
                o["idx"] = torch.empty_like(idx_out)
            return o
        d_out = [make_out(), make_out()]
        d_e2e = [{k: torch.empty_like(v) for k, v in d_in.items()} for _ in range(2)]
        out_host = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                     for n, t in o.items()} for o in d_out]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(v.numel() * v.element_size() for v in d_out[0].values())
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            sl = i & 1
            x, y = d_e2e[sl], d_out[sl]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[sl])          # inputs of slot free again
                for k in host:
                    x[k].copy_(host[k], non_blocking=True)
                ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            if i >= 2:
                stream.wait_event(ev_out[sl])             # results of slot read back
            if ranges is not None:
                layer_rows(csa, x, cfg, ranges, kv_full, ws, y.get("idx", idx_out), y["O"],
                           y["L"], y["dq"], y["dkv"], y["dsink"], y["dscore"], idx_given,
                           world=world)
            else:
                kv_full[:, :sq].copy_(x["kv_raw"])
                csa.csa_compress(kv_full[:, :sq], x["score"], cfg.ratio, out=kv_full[:, sq:])
                if has_indexer:
                    csa.csa_indexer_topk(x["q_I"], x["k_I"], x["w"], cfg.topk, cfg.ratio,
                                         workspace=ws, out_idx=y["idx"])
                ix = x["idx"] if idx_given else y["idx"]
                csa.csa_attn_fwd(x["q"], kv_full, ix, x["sink"], cfg.scale, cfg.ratio,
                                 cfg.window, out=y["O"], lse=y["L"])
                csa.csa_attn_bwd(x["q"], kv_full, ix, x["sink"], cfg.scale, cfg.ratio,
                                 cfg.window, y["O"], y["L"], x["dO"], dq=y["dq"], dkv=y["dkv"],
                                 dsink=y["dsink"])
                csa.csa_compress_bwd(kv_full[:, :sq], x["score"], cfg.ratio, y["dkv"][:, sq:],
                                     y["dkv"][:, :sq], dscore=y["dscore"])
            ev_comp[sl].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[sl])
                for n in y:
                    out_host[sl][n].copy_(y[n], non_blocking=True)
                ev_out[sl].record(s_out)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(s_in)
        for i in range(args.warmup, args.warmup + args.steps):
            e2e_step(i)
        t_end.record(s_out)
        torch.cuda.synchronize()
        e2e = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, world, dev)
        e2e_res = {"value": round(queries / (e2e / 1e3), 1), "unit": "queries/s",
                   "ms_per_step": round(e2e, 4), "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h,
                   "method": "pinned host buffers; every step copies all inputs in and all "
                             "results out; copy-in / compute / copy-out streams pipelined "
                             "across steps"}
    clk.__exit__(None, None, None)

    # ---- roofline ---------------------------------------------------------------
    peaks = load_peaks()
    traffic = load_traffic()
    names = ("compress", "indexer_topk", "attn_fwd", "attn_bwd", "compress_bwd")
    k_ms = {n: median(s) for n, s in zip(names, seg)}
    allreduce_ms = median(seg[5]) if ranges is not None else None
    if not has_indexer:
        del k_ms["indexer_topk"]
    per = {
        "compress": ("hbm", work["compress_bytes"] / (k_ms["compress"] / 1e3) / 1e9,
                     peaks["hbm_gbs"], "GB/s"),
        "attn_fwd": ("hbm", work["fwd_gathered_bytes"] / (k_ms["attn_fwd"] / 1e3) / 1e9,
                     peaks["hbm_gbs"], "GB/s"),
        "attn_bwd": ("hbm", work["bwd_gathered_bytes"] / (k_ms["attn_bwd"] / 1e3) / 1e9,
                     peaks["hbm_gbs"], "GB/s"),
        "compress_bwd": ("hbm", work["compress_bwd_bytes"] / (k_ms["compress_bwd"] / 1e3) / 1e9,
                         peaks["hbm_gbs"], "GB/s"),
    }
    if has_indexer:
        per["indexer_topk"] = ("tensor",
                               work["indexer_flops"] / (k_ms["indexer_topk"] / 1e3) / 1e12,
                               peaks["bf16_tflops"], "TFLOP/s")
    kernels = {}
    for n in names:
        if n not in per:
            continue
        bound, ach, peak, unit = per[n]
        kernels[n] = {"ms": round(k_ms[n], 4), "share": round(k_ms[n] / ms, 4), "bound": bound,
                      "achieved": round(ach, 2), "peak": peak, "unit": unit,
                      "frac": round(ach / peak, 4)}
    # the attention's contraction, against the sustained bf16 peak (a kernel
    # timed inside a long step)
    for n, key in (("attn_fwd", "fwd_flops"), ("attn_bwd", "bwd_flops")):
        tf = work[key] / (k_ms[n] / 1e3) / 1e12
        kernels[n]["tflops"] = round(tf, 2)
        kernels[n]["tensor_frac_sustained"] = round(tf / peaks["bf16_tflops_sustained"], 4)
    dom = max(k_ms, key=k_ms.get)
    bound, ach, peak, unit = per[dom]
    tr = traffic.get(f"{dom}@{cfg.name}") or (traffic.get(dom) if cfg.name == WORKLOAD else None)
    roofline = {"kernel": dom, "bound": bound, "achieved": round(ach, 2), "peak": peak,
                "unit": unit, "frac": round(ach / peak, 4),
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "peak_source": peaks["source"]}
    attn_ms = k_ms["attn_fwd"] + k_ms["attn_bwd"]
    attn_gb = (work["fwd_gathered_bytes"] + work["bwd_gathered_bytes"]) / (attn_ms / 1e3) / 1e9
    targets = {"attn_fwd_bwd_hbm_frac": round(attn_gb / peaks["hbm_gbs"], 4)}
    if has_indexer:
        targets["indexer_tensor_frac"] = kernels["indexer_topk"]["frac"]
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": workload_string(cfg),
                   "global_batch": b, "seq_len": sq,
                   "parallelism": "replicas" if world == 1 else
                   f"{world} ranks split the query rows; one all-reduce of dkv and dsink",
                   "l2": "flushed before every timed step (256 MiB written, then 256 MiB read)"},
        "ms_per_layer": round(ms_max, 4),
        "rows": ranges,
        "allreduce_ms": None if allreduce_ms is None else round(allreduce_ms, 4),
        "step_stat": f"median of {args.steps} timed steps",
        "e2e": e2e_res,
        "roofline": roofline,
        "kernels": kernels,
        "targets": targets,
        "variants": variants,
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    return res


def run_cpu_baseline(cfg_name, rows, seed=0):
    from compressed_sparse_attention_sum_gb300.inputs import CONFIGS
    cfg = CONFIGS[cfg_name]
    pool = OraclePool(cfg_name)
    try:
        sec, n = pool.run(rows, seed)
    finally:
        pool.close()
    what = ("indexer scores + top-k + " if cfg.H_I > 0 else "") + "attention fwd + bwd"
    if cfg.index_source == "zipf":
        what += " (attention on the workload's Zipf lists)"
    return {"value": round(n / sec, 2), "unit": "queries/s", "cores": pool.procs,
            "kind": "oracle",
            "sample": f"{n} of {cfg.b * cfg.sq} query rows of {cfg_name} (uniform over b, t), "
                      f"each row: {what} in fp64; pooling of the whole layer charged pro rata; "
                      "one process per host core"}


# Query rows per step of the reference arm, per workload.
REF_ROWS = {"tiny_fp32": 256, "debug_bf16": 1024, "csa4_bf16": 1024, "hca_bf16": 2048,
            "prod_bf16": 256}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on the host cores.  Each step is a
    bounded sample of the workload's query rows (drawn uniformly over b and t);
    `value` is those rows over the measured time, `ms_per_step` the measured
    time of one sampled step."""
    from compressed_sparse_attention_sum_gb300.inputs import CONFIGS
    cfg = CONFIGS[args.workload]
    rows = args.ref_rows or REF_ROWS.get(args.workload, 256)
    pool = OraclePool(args.workload)
    try:
        for i in range(args.warmup):
            pool.run(rows, seed=100 + i)
        times = []
        for i in range(args.steps):
            sec, n = pool.run(rows, seed=i)
            times.append(sec)
    finally:
        pool.close()
    ms = 1e3 * median(times)
    value = n / (ms / 1e3)
    sample = (f"{n} of {cfg.b * cfg.sq} query rows per step (uniform over b, t), fp64 oracle, "
              "one process per host core; ms_per_step is the measured time of one such step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_string(cfg), "global_batch": cfg.b, "seq_len": cfg.sq,
                   "parallelism": "replicas",
                   "l2": "flushed before every timed step (256 MiB written, then 256 MiB read)"},
        "ms_per_layer_extrapolated": round(ms * cfg.b * cfg.sq / n, 2),
        "step_stat": f"median of {args.steps} timed steps",
        "cpu_baseline": {"value": round(value, 2), "unit": "queries/s", "cores": pool.procs,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="query rows of the oracle CPU baseline sample (0: per-workload default)")
    ap.add_argument("--ref-rows", type=int, default=0,
                    help="query rows per step of the reference arm (0: per-workload default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the packed-documents, indexer-training, FP8 and overlap timings")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end timing")
    ap.add_argument("--sweep", action="store_true",
                    help="time every workload (one JSON line each, no variants, no e2e)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="profiling aid: run the workload at this sq (not a bench line)")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling aid: run the workload at this b (not a bench line)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if args.sweep:
        from compressed_sparse_attention_sum_gb300.inputs import CONFIG_ORDER
        for name in CONFIG_ORDER:
            cpu = None
            if not args.no_cpu_baseline:
                cpu = run_cpu_baseline(name, args.cpu_rows or CPU_ROWS.get(name, 1024))
            res = run_gpu(args, 0, 1, local_rank, workload=name, variants_on=False, e2e_on=False)
            res["cpu_baseline"] = cpu
            print(json.dumps(res), flush=True)
        return
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle pool is spawned before the first GPU call
        cpu = run_cpu_baseline(args.workload, args.cpu_rows or CPU_ROWS.get(args.workload, 1024))
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank, e2e_on=not args.no_e2e)
    res["cpu_baseline"] = cpu
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
