"""Benchmark of block-sparse retrieval decode on GB300.

One step = one decode step of one layer through srkv_retrieval_decode: score + top-k of
the offload blocks, then split-K sparse paged attention and its combine; steps of the rotated
layers are captured in CUDA graphs, as a model's decode step would be.  The representation
vectors are built once per page at prefill (as on the method's page: the store is written at
prefill and read at decode) and reported separately under "prefill_reps".

Workloads (--workload): the default, and the metric's, is one Llama-3-8B-shaped layer
(batch 1, 32 q / 8 kv heads, d 128, bf16, 65536 cached tokens, init 1024, window 7192,
top-k 20 %, 5 % planted blocks, shuffled 128-token pages); the others are a ragged batch of
16 requests, batch 4 x 131072 at top-k 1.0 / 0.1 / 0.2 / 0.4, and 64 requests sharing a
16384-token prefix.  The default run measures those too, under "workloads" (each over about
--load-seconds of graph replays with its own clock record); --no-workloads skips them.

Timing: exactly --steps steps (whole replays of a graph holding one step of every rotated
layer, then a graph of the remaining steps) between barriers and device synchronizations,
timed with CUDA events on the launching stream.  Around them, --load-seconds of replays
before and after keep the GPU under the same load while nvidia-smi samples its clocks; their
rate is reported as "sustained".

L2: the step rotates over --layers layer caches (default: about 2 GB of K/V, 8 x 268 MB for
the default workload; one block table and one set of lengths shared by all layers, as in a
model); between two uses of one layer the others stream far more than the 129 MB L2, so
every step reads its pages from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload W]

--impl reference times the oracle (plain fp64 C on the host cores) on the default workload.
Under torchrun each rank runs an independent replica (the method shards by request with
no exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
METRIC = "decode steps/s and achieved HBM GB/s (% of GB300 peak) for sparse paged attention"
# name -> (case factory, description, longest sequence).  The first is the metric's workload;
# the others are the remaining configurations, measured with --workload.
WORKLOADS = {
    "llama8b-65536": (
        lambda seed, dev: __import__("block_sparse_retrieval_gb300.synth", fromlist=["x"]).llama8b_layer(seed=seed, device=dev),
        "llama8b-layer-65536-bf16 (batch 1, 32/8 heads, d 128, init 1024, window 7192, top-k 0.2, 5% planted, shuffled pages)",
        65536),
    "ragged-16": (
        lambda seed, dev: __import__("block_sparse_retrieval_gb300.synth", fromlist=["x"]).ragged_batch(seed=seed, device=dev),
        "ragged-16x[32768,131072]-bf16 (16 requests, lengths U[32768, 131072], 32/8 heads, d 128, top-k 0.2, shuffled pages)",
        131072),
    "prefix-shared-64": (
        lambda seed, dev: __import__("block_sparse_retrieval_gb300.synth", fromlist=["x"]).prefix_shared(seed=seed, device=dev),
        "prefix-shared-64 (64 requests, 64/8 heads, d 128, 16384-token shared prefix + U[2048, 8192], top-k 0.2, DENSE_BOUNDARY 0; srkv_retrieval_decode_prefix: the shared pages attended once per kv head for all requests)",
        24576),
}
# The same shared-prefix batch through the plain call (every request attends its own view of
# the shared pages).
WORKLOADS["prefix-shared-64-plain"] = (
    WORKLOADS["prefix-shared-64"][0],
    "prefix-shared-64-plain (as prefix-shared-64, through srkv_retrieval_decode: no cascade)",
    24576)
# A shared prefix four times longer (65536 tokens, 512 pages: 256 MB of K/V per layer, more
# than the L2), through both calls.
WORKLOADS["prefix-shared-64-long"] = (
    lambda seed, dev: __import__("block_sparse_retrieval_gb300.synth", fromlist=["x"]).prefix_shared(prefix=65536, seed=seed, device=dev),
    "prefix-shared-64-long (64 requests, 64/8 heads, d 128, 65536-token shared prefix + U[2048, 8192], top-k 0.2, DENSE_BOUNDARY 0; srkv_retrieval_decode_prefix)",
    73728)
WORKLOADS["prefix-shared-64-long-plain"] = (
    WORKLOADS["prefix-shared-64-long"][0],
    "prefix-shared-64-long-plain (as prefix-shared-64-long, through srkv_retrieval_decode: no cascade)",
    73728)
PREFIX_WORKLOADS = ("prefix-shared-64", "prefix-shared-64-long")
for _p in (1.0, 0.1, 0.2, 0.4):
    WORKLOADS[f"dense-vs-sparse-p{_p}"] = (
        (lambda p: lambda seed, dev: __import__("block_sparse_retrieval_gb300.synth", fromlist=["x"]).dense_vs_sparse(p, seed=seed, device=dev))(_p),
        f"dense-vs-sparse-4x131072-bf16 (batch 4, 32/8 heads, d 128, top-k {_p}, 3% planted, shuffled pages)",
        131072)
# Mid-size batches of the same cache shape: 2 and 3 requests (16 and 24 (request, kv head)
# units); at top-k 0.2 one kernel on clusters of 6 and 5.
for _b in (2, 3):
    for _p in (0.2, 0.4):
        WORKLOADS[f"dense-vs-sparse-b{_b}-p{_p}"] = (
            (lambda b, p: lambda seed, dev: __import__("block_sparse_retrieval_gb300.synth", fromlist=["x"]).dense_vs_sparse(p, batch=b, seed=seed, device=dev))(_b, _p),
            f"dense-vs-sparse-{_b}x131072-bf16 (batch {_b}, 32/8 heads, d 128, top-k {_p}, 3% planted, shuffled pages)",
            131072)
# The offload tier: the same layer with every page that holds only offload-range tokens
# ([INIT, L - LOCAL)) in a pinned host pool, read in place over NVLink-C2C.
WORKLOADS["offload-65536"] = (
    WORKLOADS["llama8b-65536"][0],
    "offload-llama8b-layer-65536-bf16 (batch 1, 32/8 heads, d 128, top-k 0.2; the offload-range "
    "pages in a pinned host pool, initial and window pages in HBM)",
    65536)
OFFLOAD_WORKLOADS = ("offload-65536",)
# Compressed pages: the same caches as E4M3 codes with one fp32 scale per row (vectors and
# selection from the bf16 keys, at prefill).
WORKLOADS["fp8-65536"] = (
    WORKLOADS["llama8b-65536"][0],
    "fp8-llama8b-layer-65536 (batch 1, 32/8 heads, d 128, top-k 0.2, 5% planted, shuffled "
    "pages; K/V as E4M3 codes with fp32 row scales, bf16 q/out)",
    65536)
WORKLOADS["fp8-dense-vs-sparse-p0.2"] = (
    WORKLOADS["dense-vs-sparse-p0.2"][0],
    "fp8-dense-vs-sparse-4x131072 (batch 4, 32/8 heads, d 128, top-k 0.2, 3% planted, shuffled "
    "pages; K/V as E4M3 codes with fp32 row scales, bf16 q/out)",
    131072)
FP8_WORKLOADS = ("fp8-65536", "fp8-dense-vs-sparse-p0.2")
DATA = "synthetic (seeded N(0,1) q/K/V, 5% planted blocks, shuffled pages)"
DEFAULT_WORKLOAD = "llama8b-65536"
WORKLOAD = WORKLOADS[DEFAULT_WORKLOAD][1]
FALLBACK_HBM = 6800.0
DECODE_SOURCES = ("score_topk.cu", "decode_split_mma.cu", "decode_combine.cu",
                  "decode_fused.cu", "decode_mma.cuh", "select.cuh", "decode_plan.cuh",
                  "srkv_internal.cuh", "srkv_api.cu")


# ---- distributed plumbing -----------------------------------------------------------------

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(local)
            dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- measurement helpers ------------------------------------------------------------------

def peaks() -> tuple[float, str]:
    try:
        with open(PEAKS) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM, "fallback"


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_retrieval_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per step (the kernels of one srkv_retrieval_decode call) from the committed
    ncu summary, if it was taken on the current sources; else None."""
    try:
        with open(TRAFFIC) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_hash") != decode_source_hash():
        return None
    return t.get("bytes_per_launch")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        time.sleep(0.1)
        self.lines = []
        if self.proc:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        busy = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": mx or None, "reasons": sorted(reasons), "samples": len(sm)}


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(summary: dict) -> str | None:
    """Why a timed region's clock record disqualifies its number (None: the number stands).
    A hardware or thermal slowdown does, and so do SM clocks well below their maximum with no
    reason given (a clock lock left behind by another process).  A power cap does not: it is
    reported with the number."""
    bad = [r for r in summary.get("reasons") or [] if r in REJECT_REASONS]
    if bad:
        return ", ".join(bad)
    sm, mx = summary.get("sm_mhz"), summary.get("sm_max_mhz")
    if sm and mx and sm < 0.85 * mx and not summary.get("reasons"):
        return f"SM clock {sm:.0f} MHz of {mx:.0f} MHz with no reason"
    return None


def attended_tokens(L: int, sel, INIT: int, LOCAL: int, S: int = 128) -> tuple[int, int]:
    """|initial u selected-offload u window| and the number of pages it touches."""
    W = L - LOCAL
    ie, ws = min(INIT, L), max(W, 0)
    base = ie + (L - ws if ws < L else 0) - max(0, ie - ws)
    blocks = set(range((ie + S - 1) // S)) | set(range(ws // S, (L + S - 1) // S) if ws < L else [])
    extra = 0
    for b in sel:
        b = int(b)
        lo, hi = max(b * S, INIT), min(b * S + S, W)
        if lo < hi:
            extra += hi - lo
            blocks.add(int(b))
    return base + extra, len(blocks)


def unique_kv_bytes(case, sel, nsel, S: int = 128, row_bytes: int | None = None) -> int:
    """K/V bytes of the distinct (physical page, kv head, row) triples the step attends: a
    page shared by several requests counts once.  row_bytes: bytes of one K (or V) row."""
    cfg = case.cfg
    d, Hkv = cfg["head_dim"], cfg["num_kv_heads"]
    INIT, LOCAL = cfg["init_tokens"], cfg["local_tokens"]
    bt = case.block_table.cpu().numpy()
    L = case.seq_lens.cpu().numpy()
    masks = {}
    for r in range(case.batch):
        Lr = int(L[r])
        W = Lr - LOCAL
        ranges = [(0, min(INIT, Lr))]
        if W < Lr:
            ranges.append((max(W, 0), Lr))
        for h in range(Hkv):
            rr = list(ranges) + [(max(int(b) * S, INIT), min(int(b) * S + S, W))
                                 for b in sel[r, h, :nsel[r, h]]]
            for lo, hi in rr:
                t = lo
                while t < hi:
                    b = t // S
                    e = min(hi, (b + 1) * S)
                    key = (int(bt[r, b]), h)
                    masks[key] = masks.get(key, 0) | (((1 << (e - b * S)) - 1) ^ ((1 << (t - b * S)) - 1))
                    t = e
    rows = sum(bin(m).count("1") for m in masks.values())
    return rows * 2 * (row_bytes if row_bytes is not None else d * case.k_cache.element_size())


# ---- our arm --------------------------------------------------------------------------------

def shared_prefix_blocks(case, S: int = 128) -> int:
    """Leading logical blocks that every request maps to the same physical page and holds
    whole."""
    bt = case.block_table.cpu().numpy()
    L = case.seq_lens.cpu().numpy()
    n = 0
    while n < bt.shape[1] and all(n < int(x) // S for x in L) and np.all(bt[:, n] == bt[0, n]):
        n += 1
    return n


class Layer:
    """One attention layer's cache.  As in a model's paged cache, every layer has its own
    queries, K/V pages and representation vectors, while the block table and the sequence
    lengths (per request) are shared by all layers."""

    def __init__(self, seed: int, device, shared=None, workload: str = DEFAULT_WORKLOAD):
        from block_sparse_retrieval_gb300 import srkv
        self.case = WORKLOADS[workload][0](seed, device)
        if shared is not None:
            for name in ("block_table", "seq_lens", "prompt_lens"):
                assert torch.equal(getattr(self.case, name), getattr(shared, name))
                setattr(self.case, name, getattr(shared, name))
        c = self.case
        # leading blocks every request maps to the same pages (the shared-prefix call)
        self.prefix_blocks = shared_prefix_blocks(c) if workload in PREFIX_WORKLOADS else None
        self.buf = srkv.DecodeBuffers(c.cfg, c.batch, c.max_blocks, c.num_pages, device=device,
                                      prefix=self.prefix_blocks is not None)
        self.srkv = srkv
        self.k_host = self.v_host = None  # the host pool of the offload workload
        self.k_scale = self.v_scale = None  # row scales of compressed pages

    def to_fp8(self):
        """Compresses every page (srkv_quantize_kv_fp8) and drops the bf16 caches."""
        c, b = self.case, self.buf
        dev = c.k_cache.device
        ids = torch.arange(c.num_pages, dtype=torch.int32, device=dev)
        k8 = torch.empty(c.k_cache.shape, dtype=torch.uint8, device=dev)
        v8 = torch.empty_like(k8)
        self.k_scale = torch.empty(c.k_cache.shape[:3], dtype=torch.float32, device=dev)
        self.v_scale = torch.empty_like(self.k_scale)
        self.srkv.quantize_kv_fp8(c.cfg, c.k_cache, c.v_cache, ids, k8, v8, self.k_scale,
                                  self.v_scale, b.error_flags)
        c.k_cache, c.v_cache = k8, v8

    def to_host(self, dev_ids, host_ids, new_id):
        """Moves pages host_ids into a pinned host pool: the device pool keeps dev_ids (in that
        order), the vectors are renumbered; the caller renumbers the shared block table."""
        c, b = self.case, self.buf
        d_idx = torch.as_tensor(dev_ids, device=c.k_cache.device)
        h_idx = torch.as_tensor(host_ids, device=c.k_cache.device)
        self.k_host = c.k_cache[h_idx].cpu().contiguous().pin_memory()
        self.v_host = c.v_cache[h_idx].cpu().contiguous().pin_memory()
        c.k_cache = c.k_cache[d_idx].contiguous()
        c.v_cache = c.v_cache[d_idx].contiguous()
        reps = torch.empty_like(b.reps)
        reps[torch.as_tensor(new_id, device=reps.device)] = b.reps
        b.reps.copy_(reps)

    def prefill(self):
        c, b = self.case, self.buf
        self.srkv.build_block_reps(c.cfg, c.k_cache, c.page_ids, c.page_valid, b.reps,
                                   b.error_flags)

    def step(self):
        """One decode step: srkv_retrieval_decode (score + top-k, then split + combine), or
        srkv_retrieval_decode_tiered when pages live in a host pool."""
        c, b = self.case, self.buf
        if self.k_scale is not None:
            self.srkv.retrieval_decode_fp8(c.cfg, c.q, c.k_cache, c.v_cache, self.k_scale,
                                           self.v_scale, b.reps, c.block_table, c.seq_lens,
                                           c.prompt_lens, b.sel, b.nsel, b.out, b.workspace,
                                           b.error_flags)
            return
        if self.prefix_blocks is not None:
            self.srkv.retrieval_decode_prefix(c.cfg, c.q, c.k_cache, c.v_cache, b.reps,
                                              c.block_table, c.seq_lens, c.prompt_lens,
                                              self.prefix_blocks, b.sel, b.nsel, b.out,
                                              b.workspace, b.error_flags)
            return
        if self.k_host is not None:
            self.srkv.retrieval_decode_tiered(c.cfg, c.q, c.k_cache, c.v_cache, self.k_host,
                                              self.v_host, b.reps, c.block_table, c.seq_lens,
                                              c.prompt_lens, b.sel, b.nsel, b.out, b.workspace,
                                              b.error_flags)
            return
        self.srkv.retrieval_decode(c.cfg, c.q, c.k_cache, c.v_cache, b.reps, c.block_table,
                                   c.seq_lens, c.prompt_lens, b.sel, b.nsel, b.out,
                                   b.workspace, b.error_flags)

    def plain(self) -> bool:
        """True when the step is srkv_retrieval_decode over device pages (not compressed,
        not tiered, no shared-prefix call): the step srkv_retrieval_decode_host runs."""
        return self.k_scale is None and self.prefix_blocks is None and self.k_host is None

    def step_bytes(self) -> dict:
        """Algorithmic bytes of one step: what the method must read and write."""
        c, b = self.case, self.buf
        cfg = c.cfg
        d, Hkv, Hq = cfg["head_dim"], cfg["num_kv_heads"], cfg["num_q_heads"]
        sel, nsel = b.sel.cpu().numpy(), b.nsel.cpu().numpy()
        L = c.seq_lens.cpu().numpy()
        from block_sparse_retrieval_gb300 import srkv
        # bytes of one attended K (or V) row: bf16 values, or E4M3 codes and a fp32 scale
        row = d * 2 if self.k_scale is None else d + 4
        kv = pages = n_cand = 0
        for r in range(c.batch):
            n_cand += srkv.num_candidates(cfg, int(L[r])) * Hkv
            for h in range(Hkv):
                toks, pg = attended_tokens(int(L[r]), sel[r, h, :nsel[r, h]],
                                           cfg["init_tokens"], cfg["local_tokens"])
                kv += toks * 2 * row
                pages += pg
        qo = c.batch * Hq * d * 2
        score = n_cand * (d * 4 + 4) + qo + int(nsel.sum()) * 4 + nsel.size * 4
        decode = kv + pages * 4 + qo * 2 + int(nsel.sum()) * 4 + nsel.size * 4
        host_kv = 0  # K/V of kept blocks read from the host pool (whole 128-token pages)
        if self.k_host is not None:
            bt = c.block_table.cpu().numpy()
            P_dev = c.k_cache.shape[0]
            for r in range(c.batch):
                for h in range(Hkv):
                    blocks = sel[r, h, :nsel[r, h]]
                    host_kv += int((bt[r, blocks] >= P_dev).sum()) * 128 * d * 2 * 2
        return {"score": score, "decode": decode, "kv": kv, "total": score + decode,
                "kv_unique": unique_kv_bytes(c, sel, nsel, row_bytes=row), "host_kv": host_kv}


def launches_per_step(layer) -> int:
    """Kernels one decode call of the layer launches (the shared-prefix call adds one)."""
    c = layer.case
    if layer.prefix_blocks:
        return 4
    return layer.srkv.retrieval_decode_launches(c.cfg, c.batch, c.max_blocks)


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def build_layers(wl: str, n_layers, rank: int, dev):
    """The rotated layer caches of a workload (prefill included): (layers, prefill record).
    Same seed for every layer: one page structure and one block table shared by all."""
    first = Layer(1000 + 1000003 * rank, dev, workload=wl)
    if n_layers is None:
        layer_bytes = 2 * first.case.k_cache.numel() * first.case.k_cache.element_size()
        n_layers = max(2, min(8, -(-2_000_000_000 // layer_bytes)))
    layers = [first] + [Layer(1000 + 1000003 * rank, dev, shared=first.case, workload=wl)
                        for _ in range(n_layers - 1)]
    # prefill: representation vectors of every page of every layer, one launch per layer,
    # queued behind a short device sleep so that the events time the kernels, not the host
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for ly in layers:                        # warm the kernel once
        ly.prefill()
    torch.cuda.synchronize()
    rep_bytes = 0  # counted first: a read of a device tensor would wait for the queue
    for ly in layers:
        c = ly.case
        rep_bytes += int(c.page_valid.sum()) * c.cfg["num_kv_heads"] * c.cfg["head_dim"] * 2 \
            + c.page_ids.numel() * c.cfg["num_kv_heads"] * c.cfg["head_dim"] * 4
    torch.cuda._sleep(int(2e7))
    ev[0].record()
    for ly in layers:
        ly.prefill()
    ev[1].record()
    torch.cuda.synchronize()
    rep_ms = ev[0].elapsed_time(ev[1])
    if wl in OFFLOAD_WORKLOADS:
        offload_layers(layers)
    if wl in FP8_WORKLOADS:
        for ly in layers:
            ly.to_fp8()
        torch.cuda.synchronize()
    for ly in layers:                        # the step must run clean before it is timed
        ly.step()
    torch.cuda.synchronize()
    flags = [int(ly.buf.error_flags.item()) for ly in layers]
    if any(flags):
        raise RuntimeError(f"device error flags {flags}")
    prefill = {"kernel": "srkv_build_block_reps", "launches": len(layers),
               "pages": sum(ly.case.page_ids.numel() for ly in layers),
               "bytes": rep_bytes, "us": round(rep_ms * 1e3, 1),
               "GB_s": round(rep_bytes / (rep_ms / 1e3) / 1e9, 1)}
    return layers, prefill


def step_graphs(layers, K: int, stream):
    """CUDA graphs that together run exactly K steps: `full` holds one step of every rotated
    layer (replayed K // R times), `tail` the first K % R of them (None if K % R == 0)."""
    R = len(layers)
    with torch.cuda.stream(stream):
        full = capture(lambda: [ly.step() for ly in layers], stream)
        tail = capture(lambda: [ly.step() for ly in layers[:K % R]], stream) if K % R else None
    torch.cuda.synchronize()
    return full, tail


def roofline_of(layers, step_bytes, call_ms: float, peak: float, peak_kind: str, wl: str,
                dev) -> dict:
    avg_step_bytes = statistics.mean(sb["total"] for sb in step_bytes)
    avg_unique = statistics.mean(sb["total"] - sb["kv"] + sb["kv_unique"] for sb in step_bytes)
    achieved = avg_step_bytes / (call_ms / 1e3) / 1e9
    roofline = {"kernel": None, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "bytes_per_launch": int(avg_step_bytes), "unique_bytes_per_launch": int(avg_unique),
                "unique_frac": round(avg_unique / (call_ms / 1e3) / 1e9 / peak, 4),
                "us_per_launch": round(call_ms * 1e3, 3), "traffic": None}
    if wl in OFFLOAD_WORKLOADS:
        # bound by the host pool's reads over the chip-to-chip link
        host = statistics.mean(sb["host_kv"] for sb in step_bytes)
        c2c = c2c_copy_peak(dev)
        roofline.update({"bound": "c2c", "achieved": round(host / (call_ms / 1e3) / 1e9, 1),
                         "peak": c2c, "frac": round(host / (call_ms / 1e3) / 1e9 / c2c, 4),
                         "peak_kind": "measured in this run: pinned host to device copy",
                         "bytes_per_launch": int(host),
                         "unique_bytes_per_launch": int(host), "unique_frac": None,
                         "device_bytes_per_launch": int(avg_step_bytes - host),
                         "device_GB_s": round((avg_step_bytes - host) / (call_ms / 1e3) / 1e9, 1)})
    launches = launches_per_step(layers[0])
    roofline["kernel"] = "srkv_retrieval_decode_prefix call: score_topk, shared-prefix cascade, " \
        "split-K decode and combine kernels, overlapped by programmatic launch" if launches == 4 else (
        "srkv_retrieval_decode call: one kernel (a thread-block cluster per (request, kv head) "
        "scores, selects and attends)" if launches == 1 else
        "srkv_retrieval_decode call: score_topk, split-K decode and combine kernels, "
        "overlapped by programmatic launch")
    return roofline


def replay_for(full, stream, seconds: float, est_ms: float) -> tuple[int, float]:
    """Replays `full` for about `seconds` of device time; returns (replays, ms)."""
    n = max(1, int(seconds * 1e3 / max(est_ms, 1e-3)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            full.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return n, e0.elapsed_time(e1)


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_kind = peaks()
    wl = args.workload
    layers, prefill = build_layers(wl, args.layers, rank, dev)
    R = len(layers)
    step_bytes = [ly.step_bytes() for ly in layers]
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    K = args.steps
    full, tail = step_graphs(layers, K, stream)
    with torch.cuda.stream(stream):           # W warm-up steps (whole replays, at least W)
        for _ in range(max(1, -(-args.warmup // R))):
            full.replay()
    torch.cuda.synchronize()
    _, probe_ms = replay_for(full, stream, 0.0, 1.0)
    est_step_ms = probe_ms / R

    def timed_region():
        """Exactly K steps between barriers and synchronizations, inside a window of load
        (about 0.15 s of replays before and after) over which nvidia-smi samples the clocks;
        the window's replays give the sustained rate."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with ClockSampler(local) as clocks:
            n0, ms0 = replay_for(full, stream, args.load_seconds, est_step_ms * R)
            barrier(world)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                torch.cuda._sleep(int(2e7))  # the host queues the K steps before they start
                ev[0].record(stream)
                for _ in range(K // R):
                    full.replay()
                if tail is not None:
                    tail.replay()
                ev[1].record(stream)
            torch.cuda.synchronize()
            barrier(world)
            n1, ms1 = replay_for(full, stream, args.load_seconds, est_step_ms * R)
        sustained = {"steps": (n0 + n1) * R, "ms": round(ms0 + ms1, 3),
                     "us_per_step": round((ms0 + ms1) * 1e3 / ((n0 + n1) * R), 3)}
        return ev[0].elapsed_time(ev[1]), clocks.summary(), sustained

    region_ms, clk, sustained = timed_region()
    # A region whose clocks disqualify it is measured once more; every rank takes the same
    # path (the decision is the maximum over ranks), and the line keeps the first record.
    why = clocks_rejected(clk)
    remeasured = None
    if max_over_ranks(1.0 if why else 0.0, world, dev) > 0:
        remeasured = {"first_clocks": clk, "reason": why or "clocks of another rank"}
        region_ms, clk, sustained = timed_region()
    total_ms = max_over_ranks(region_ms, world, dev)
    ms_per_step = total_ms / K
    value = world * K / (total_ms / 1e3)
    sustained["value"] = round(world * 1e3 / sustained["us_per_step"] * 1e3, 2)
    roofline = roofline_of(layers, step_bytes, ms_per_step, peak, peak_kind, wl, dev)
    roofline["traffic"] = committed_traffic() if wl == DEFAULT_WORKLOAD else None
    roofline["us_per_launch_sustained"] = sustained["us_per_step"]
    launches = launches_per_step(layers[0])

    e2e = run_e2e(layers, args.e2e_steps, world, dev) if args.e2e_steps > 0 else None
    append = time_append(dev, layers[0].case.cfg)
    prefill["frac"] = round(prefill["GB_s"] / peak, 4)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 K/V with fp32 row scales, bf16 q/out" if wl in FP8_WORKLOADS else "bf16",
        "data": DATA,
        "config": {"workload": WORKLOADS[wl][1], "global_batch": world * layers[0].case.batch,
                   "seq_len": WORKLOADS[wl][2], "parallelism": f"replicas x{world}",
                   "layers_rotated": R,
                   "l2": f"inputs larger than L2: {R} layer caches rotated per step"},
        "roofline": roofline,
        "sustained": sustained,
        "prefill_reps": prefill,
        "clocks": clk,
        "e2e": e2e["per_call"] if e2e else None,
        "e2e_graph": e2e["graph"] if e2e else None,
        "append_kv": append,
        "gpu_launches": K * launches,  # kernels per srkv_retrieval_decode call x steps
    }
    if remeasured:
        line["remeasured"] = remeasured
    base_case = base_arr = None
    if rank == 0 and not args.no_cpu_baseline and wl == DEFAULT_WORKLOAD:
        from block_sparse_retrieval_gb300 import synth
        base_case = layers[0].case
        base_arr = synth.to_oracle_arrays(base_case)
    del layers, full, tail
    torch.cuda.empty_cache()
    if wl == DEFAULT_WORKLOAD and not args.no_workloads:
        line["workloads"] = {name: measure_workload(name, args, world, rank, dev, peak, peak_kind)
                             for name in EXTRA_WORKLOADS}
    if rank == 0 and not args.no_cpu_baseline and wl == DEFAULT_WORKLOAD:
        line["cpu_baseline"] = cpu_baseline(base_case, base_arr, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


# The other configurations of the method's evaluation, measured in the default run beside the
# metric's workload: the batch-4 x 131072 cache at four ratios, the ragged batch, the shared
# prefix.
EXTRA_WORKLOADS = ("dense-vs-sparse-p0.2", "dense-vs-sparse-p0.1", "dense-vs-sparse-p0.4",
                   "dense-vs-sparse-p1.0", "dense-vs-sparse-b2-p0.2", "dense-vs-sparse-b3-p0.2",
                   "ragged-16", "prefix-shared-64", "prefix-shared-64-plain")


def measure_workload(wl: str, args, world: int, rank: int, dev, peak: float,
                     peak_kind: str) -> dict:
    """One workload's decode step: about args.load_seconds of CUDA-graph replays over two
    rotated layer caches (each larger than L2), timed with CUDA events, clocks sampled over
    them.  Its prefill is one srkv_build_block_reps launch per layer over every page."""
    layers, prefill = build_layers(wl, 2, rank, dev)
    R = len(layers)
    step_bytes = [ly.step_bytes() for ly in layers]
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    full, _ = step_graphs(layers, R, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            full.replay()
    torch.cuda.synchronize()
    _, probe_ms = replay_for(full, stream, 0.0, 1.0)
    barrier(world)
    with ClockSampler(dev.index or 0) as clocks:  # the rank's local GPU
        n, ms = replay_for(full, stream, max(args.load_seconds, 0.1), probe_ms)
    ms = max_over_ranks(ms, world, dev)
    call_ms = ms / (n * R)
    roofline = roofline_of(layers, step_bytes, call_ms, peak, peak_kind, wl, dev)
    prefill["frac"] = round(prefill["GB_s"] / peak, 4)
    out = {"workload": WORKLOADS[wl][1], "steps": n * R, "us_per_launch": roofline["us_per_launch"],
           "steps_per_s": round(world * 1e3 / call_ms, 2), "roofline": roofline,
           "prefill_reps": prefill, "clocks": clocks.summary(),
           "gpu_launches_per_step": launches_per_step(layers[0])}
    del layers, full
    torch.cuda.empty_cache()
    return out


def offload_layers(layers):
    """Moves every page holding only offload-range tokens of some request (blocks b with
    INIT <= b*S and (b+1)*S <= L - LOCAL) of every layer into a pinned host pool; the layers
    share one block table, renumbered once."""
    c = layers[0].case
    cfg = c.cfg
    bt = c.block_table.cpu().numpy()
    to_host = np.zeros(c.num_pages, bool)
    for r, L in enumerate(c.seq_lens.cpu().numpy()):
        W = int(L) - cfg["local_tokens"]
        for b in range(-(-cfg["init_tokens"] // 128), max(W, 0) // 128):
            if bt[r, b] >= 0:
                to_host[bt[r, b]] = True
    dev_ids, host_ids = np.nonzero(~to_host)[0], np.nonzero(to_host)[0]
    new_id = np.empty(c.num_pages, np.int64)
    new_id[dev_ids] = np.arange(len(dev_ids))
    new_id[host_ids] = len(dev_ids) + np.arange(len(host_ids))
    for ly in layers:
        ly.to_host(dev_ids, host_ids, new_id)
    ok = bt >= 0
    bt[ok] = new_id[bt[ok]]
    c.block_table.copy_(torch.from_numpy(bt))


def c2c_copy_peak(dev, nbytes: int = 1 << 30, reps: int = 5) -> float:
    """GB/s of a pinned host to device copy (the copy engines over NVLink-C2C)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return round(reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9, 1)


def time_append(dev, cfg, n: int = 200) -> dict:
    """Decode-time maintenance of the same layer shape: srkv_append_kv of one new token
    (every kv head) and the refresh of its page's representation vector, per call."""
    from block_sparse_retrieval_gb300 import srkv, synth
    case = synth.llama8b_layer(seq_len=65536 - 128 + n, device=dev, seed=7)
    lens = case.seq_lens - n
    buf = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=dev)
    Hkv, d = case.cfg["num_kv_heads"], case.cfg["head_dim"]
    kn = torch.randn(n, case.batch, Hkv, d, device=dev).to(case.k_cache.dtype)
    lens_all = torch.stack([lens + i for i in range(n)])  # position of every call
    srkv.append_kv(case.cfg, kn[0], kn[0], case.k_cache, case.v_cache, case.block_table,
                   lens_all[0], buf.reps, buf.error_flags)
    torch.cuda.synchronize()
    # The n calls go into one CUDA graph, as a decode step would hold them: the figure is
    # device time per call, not the host cost of n Python calls.
    stream = torch.cuda.Stream(dev)
    graph = capture(lambda: [srkv.append_kv(case.cfg, kn[i], kn[i], case.k_cache, case.v_cache,
                                            case.block_table, lens_all[i], buf.reps,
                                            buf.error_flags) for i in range(n)], stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return {"kernel": "srkv_append_kv", "us_per_call": round(e0.elapsed_time(e1) * 1e3 / n, 2),
            "calls": n, "note": "one token per call (all kv heads), n calls replayed from one CUDA graph, same layer shape"}


def run_e2e(layers, K, world, dev) -> dict:
    """The same steps through the public entry points with host buffers, as a serving loop runs
    them.  `per_call`: one srkv_retrieval_decode_host call per step through the binding (its
    argument checks included): the step's query and lengths copied from pinned host memory,
    the decode, the output copied back into pinned host memory, and the wait for it.  Steps
    that srkv_retrieval_decode_host does not run (compressed or host-pool pages, the
    shared-prefix call) are, per step from Python, one copy of the query and lengths from a
    pinned host buffer, the layer's own entry point through the binding, the copy of the
    output into pinned host memory and the wait.  `graph`: the same copies and decode call
    replayed from one CUDA graph per layer (what a serving loop that captures its step would
    see), then the wait."""
    plain = all(ly.plain() for ly in layers)
    steps = []
    for ly in layers:
        c, b = ly.case, ly.buf
        qb = c.q.numel() * c.q.element_size()
        nb = c.seq_lens.numel() * 4
        host = torch.empty(qb + 2 * nb, dtype=torch.uint8).pin_memory()
        host[:qb].copy_(c.q.cpu().contiguous().view(-1).view(torch.uint8))
        host[qb:qb + nb].copy_(c.seq_lens.cpu().view(torch.uint8))
        host[qb + nb:].copy_(c.prompt_lens.cpu().view(torch.uint8))
        hq = hlens = hprompt = staging = None
        if plain:
            # the host call's own buffers: page-locked inputs laid out like its staging (one
            # copy), a page-locked output, the device staging
            hin = ly.srkv.host_inputs(c.cfg, c.batch)
            hq, hlens, hprompt = hin["q"], hin["seq_lens"], hin["prompt_lens"]
            hq.copy_(c.q.cpu())
            hlens.copy_(c.seq_lens.cpu())
            hprompt.copy_(c.prompt_lens.cpu())
            staging = torch.empty(ly.srkv.host_staging_size(c.cfg, c.batch), dtype=torch.uint8,
                                  device=dev)
        packed = torch.empty_like(host, device=dev)
        # the layer reads its query and lengths from the packed device buffer
        c.q = packed[:qb].view(c.q.dtype).view(c.q.shape)
        c.seq_lens = packed[qb:qb + nb].view(torch.int32)
        c.prompt_lens = packed[qb + nb:].view(torch.int32)
        out = torch.empty_like(b.out, device="cpu").pin_memory()
        steps.append(dict(ly=ly, host=host, packed=packed, out=out, hq=hq, hlens=hlens,
                          hprompt=hprompt, staging=staging))
    stream = torch.cuda.Stream(dev)
    for st in steps:  # the host call over each layer's fixed buffers, marshalled once
        if not plain:
            break
        ly = st["ly"]
        c, b = ly.case, ly.buf
        st["host_step"] = ly.srkv.HostDecodeStep(
            c.cfg, st["hq"], st["hlens"], st["hprompt"], st["out"], st["staging"], c.k_cache,
            c.v_cache, b.reps, c.block_table, b.sel, b.nsel, b.out, b.workspace, b.error_flags,
            stream)
    h2d = steps[0]["host"].nbytes
    d2h = steps[0]["out"].nbytes
    stream.wait_stream(torch.cuda.current_stream())

    def one(st):
        st["packed"].copy_(st["host"], non_blocking=True)
        st["ly"].step()
        st["out"].copy_(st["ly"].buf.out, non_blocking=True)

    graphs = []
    with torch.cuda.stream(stream):
        for st in steps:
            one(st)
        stream.synchronize()
        for st in steps:
            graphs.append(capture(lambda st=st: one(st), stream))
    torch.cuda.synchronize()

    def timed(step) -> float:
        with torch.cuda.stream(stream):
            for i in range(3):
                step(i)
            barrier(world)
            t0 = time.perf_counter()
            for i in range(K):
                step(i)
            return max_over_ranks(time.perf_counter() - t0, world, dev)

    def per_call(i):
        st = steps[i % len(steps)]
        if plain:
            st["host_step"]()
        else:
            one(st)
            stream.synchronize()

    def replay(i):
        graphs[i % len(graphs)].replay()
        stream.synchronize()

    dt_call, dt_graph = timed(per_call), timed(replay)
    base = {"unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "copies_declared": True}
    return {
        "per_call": dict(base, value=round(world * K / dt_call, 2),
                         how="per step from Python: one srkv_retrieval_decode_host call "
                             "through the binding (srkv.HostDecodeStep: arguments checked and "
                             "marshalled once per buffer set; one copy of q and lengths from a "
                             "pinned host buffer laid out like the staging, the decode, copy of "
                             "the output to pinned host memory, stream synchronize)" if plain
                         else "per step from Python: copy of q and lengths from pinned host "
                              "memory, the layer's decode entry point through the binding, "
                              "copy of the output to pinned host memory, stream synchronize"),
        "graph": dict(base, value=round(world * K / dt_graph, 2),
                      how="the same three per step replayed from one CUDA graph per layer, "
                          "host synchronize"),
    }


# ---- the oracle on the host --------------------------------------------------------------------

def oracle_step_fn(case, threads, arr=None):
    import oracle
    from block_sparse_retrieval_gb300 import synth
    arr = arr or synth.to_oracle_arrays(case)
    args = [arr[k] for k in ("q", "k_cache", "v_cache", "block_table", "seq_lens",
                             "prompt_lens")]
    return lambda: oracle.decode(case.cfg, *args, threads=threads)


def time_oracle(fn, seconds: float) -> tuple[int, float]:
    fn()
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        fn()
        n += 1
    return n, time.perf_counter() - t0


def cpu_baseline(case, arr, seconds: float) -> dict:
    """The oracle as it stands on the host cores: all of them (one thread per kv-head unit,
    at most the core count) and a single thread, full decode steps of the metric's layer."""
    units = case.batch * case.cfg["num_kv_heads"]
    threads = max(1, min(os.cpu_count() or 1, units))
    n, dt = time_oracle(oracle_step_fn(case, threads, arr), seconds)
    n1, dt1 = time_oracle(oracle_step_fn(case, 1, arr), seconds * 0.75)
    return {"value": round(n / dt, 3), "unit": "steps/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full decode steps of one 65536-token layer (all {units} kv-head "
                      "units; the oracle recomputes block means from K as it scores)",
            "host_cores": os.cpu_count(),
            "single_thread": {"value": round(n1 / dt1, 3), "unit": "steps/s", "cores": 1,
                              "sample": f"{n1} full decode steps, one thread"}}


def run_reference(args, world, rank):
    """The oracle on the host cores, on the workload --workload names (its first seed's
    case): per step one full decode of every (request, kv head) unit.  Over compressed pages a
    step is the attention over the E4M3 codes with the selection of the bf16 cache, taken
    once before timing; the offload and shared-prefix calls compute the plain decode's
    result, so their step is the plain decode."""
    if rank != 0:
        return
    import oracle
    from block_sparse_retrieval_gb300 import synth
    wl = args.workload
    case = WORKLOADS[wl][0](1000, "cpu")
    units = case.batch * case.cfg["num_kv_heads"]
    threads = max(1, min(os.cpu_count() or 1, units))
    arr = synth.to_oracle_arrays(case)
    fn = oracle_step_fn(case, threads, arr)
    what = "full decode steps"
    if wl in FP8_WORKLOADS:
        ids = np.arange(case.num_pages, dtype=np.int32)
        k8, ks = oracle.quantize_e4m3(case.cfg, arr["k_cache"], ids)
        v8, vs = oracle.quantize_e4m3(case.cfg, arr["v_cache"], ids)
        cfg8 = dict(case.cfg, dtype=2)
        rest = [arr[k] for k in ("block_table", "seq_lens", "prompt_lens")]
        sel = oracle.decode(case.cfg, arr["q"], arr["k_cache"], arr["v_cache"], *rest,
                            threads=threads)

        def fn():
            return oracle.decode(cfg8, arr["q"], k8, v8, *rest, sel=sel["sel"],
                                 nsel=sel["nsel"], threads=threads, k_scale=ks, v_scale=vs)
        what = ("decode steps over the E4M3 codes (the selection, from the bf16 cache, taken "
                "once before timing: the oracle's step is the cheaper for it)")
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA,
        "config": {"workload": WORKLOADS[wl][1], "global_batch": case.batch,
                   "seq_len": WORKLOADS[wl][2], "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 3), "unit": "steps/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{args.steps} {what} of the workload ({units} units)"},
        "e2e": {"value": round(value, 3), "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=None,
                    help="rotated layer caches (default: 2 to 8, about 2 GB of K/V, far more than L2)")
    ap.add_argument("--workload", choices=list(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=1000,
                    help="steps of each end-to-end loop (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only --workload (the default run adds the other configurations)")
    ap.add_argument("--load-seconds", type=float, default=0.15,
                    help="seconds of replays before and after the timed steps (clock sampling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
