#!/usr/bin/env python3
"""Quantized-KV decode attention benchmark (one JSON line on stdout).

Metric: achieved HBM GB/s of one decode step = algorithmic bytes (packed cache
blocks the step must read, fp32 staging tail, bf16 Q and output) / device time
of the step (one launch of the split kernel, whose last CTA per (sequence, kv
head) merges the splits), with the cache resident in HBM; L2 is flushed before
every timed step where the step's bytes do not already exceed three times the
L2 size.  ms_per_step gives the time per decode step.  The default workload is
tiered_32k (B64, Hkv8, Hq64, D128, context 32768, FP8 pages for the 10% of
pages with the largest synthetic attention mass, 2-bit codebook + e4m3 outliers
elsewhere), the largest of the five workloads; the same line carries the other
measured workloads (cb2_4k, fp4_32k, longctx_128k) under "configs", each with
its own roofline, and "append": kvq_quantize_append timed on 1-token appends and
a 4096-token prefill chunk of the longctx_128k shape (--no-append skips it);
--project adds the fused projection + append comparison.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

--impl reference times the CPU oracle (plain fp64 C) on the host cores on a
bounded sample of the same workload and prints the same line with
"impl": "reference".  Under torchrun (N > 1) every rank runs an independent
replica (weak scaling: the path shards by (sequence, kv head) with no exchange);
value sums the ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import re
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sub_byte_quantized_kvq_gb300 import kvq, synth, workloads  # noqa: E402

METRIC = "quantized-KV decode attention: achieved HBM GB/s vs peak; us per decode step"
FMT_NAME = {0: "INT4_G32", 1: "FP4_E2M1_S16", 2: "CB2_OUTLIER", 3: "TIERED", 4: "CB2_STATIC", 5: "ASYM3_OUTLIER",
            6: "CB2_GROUP4"}
DECODE_MATH = {"auto": kvq.KVQ_DECODE_AUTO, "tensor_cores": kvq.KVQ_DECODE_TENSOR_CORES,
               "cuda_cores": kvq.KVQ_DECODE_CUDA_CORES}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_split_traffic.json")
KERNEL_SOURCES = ["kvq_common.cuh", "kvq_decode.cuh", "kvq_internal.cuh"]


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    p.add_argument("--workload", default="tiered_32k", choices=sorted(synth.WORKLOADS))
    p.add_argument("--batch", type=int, default=0, help="override the workload's sequence count (profiling)")
    p.add_argument("--q-heads", type=int, default=0, help="override the workload's query heads (GQA group size)")
    p.add_argument("--decode-math", default="auto", choices=sorted(DECODE_MATH),
                   help="tensor or CUDA cores for the dense products of the codebook pages")
    p.add_argument("--no-configs", action="store_true",
                   help="time only --workload (skip the other workloads carried under \"configs\")")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--splits", type=int, default=-1, help="-1: the workload's own (0 = library choice)")
    p.add_argument("--flush-mb", type=int, default=512)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-append", action="store_true",
                   help="skip timing kvq_quantize_append (1-token appends and a 4096-token prefill chunk)")
    p.add_argument("--append-workload", default="longctx_128k", choices=sorted(synth.WORKLOADS),
                   help="shape of the kvq_quantize_append timing")
    p.add_argument("--project", action="store_true",
                   help="also time kvq_project_append against a cuBLAS projection + kvq_quantize_append")
    p.add_argument("--project-only", action="store_true",
                   help="time only the projection + append comparison (no decode cache, no decode timing)")
    p.add_argument("--project-b", type=int, default=0, help="sequences for the projection timing (0: the workload's)")
    return p.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- byte accounting
def block_meta(fmt: int, D: int, blocks):
    """The bytes of each main-pool block that the algorithmic count needs, as
    numpy (blocks: [n_blocks, stride] uint8, a torch tensor on any device or a
    numpy array): the side-list's channel-record count (CB2, TIERED, ASYM3,
    CB2_GROUP4) or the outlier count of each block (INT4); None otherwise."""
    if fmt in (synth.FMT_CB2, synth.FMT_TIERED, synth.FMT_CB2G):
        col = blocks[:, 12 * D]
    elif fmt == synth.FMT_A3:
        col = blocks[:, 10 * D]
    elif fmt == synth.FMT_INT4:
        col = blocks[:, 10 * D:10 * D + 16]
        col = col.to(torch.int64).sum(1) if isinstance(col, torch.Tensor) else col.astype(np.int64).sum(1)
    else:
        return None
    return (col.cpu().numpy() if isinstance(col, torch.Tensor) else np.asarray(col)).astype(np.int64)


def step_bytes(fmt: int, D: int, Hkv: int, Hq: int, B: int, N: int, page_table: np.ndarray, meta,
               static_channels: int = 0) -> dict:
    """Bytes one decode step must move when every one of the B sequences holds
    N tokens: the packed contents of every block it reads (codes, scales or
    codebooks, and the outlier side-list or per-token outliers actually
    present), the fp32 staging tail of the page formats, Q (bf16) and the
    output (bf16).

    page_table: int32 [B, pages] (bit 31 = FP8 tier page); meta: block_meta()
    of the main pool, indexed by block (phys * Hkv + head) * 2 + role."""
    pt = np.asarray(page_table).astype(np.int64) & 0xFFFFFFFF
    paged = fmt in (synth.FMT_CB2, synth.FMT_TIERED, synth.FMT_CB2S, synth.FMT_A3, synth.FMT_CB2G)
    unit = 64 if fmt == synth.FMT_CB2G else 16                 # tokens quantized together
    full = (N // unit) * (unit // 16) if paged else (N + 15) // 16   # pages stored as blocks
    ent = pt[:, :full].reshape(-1)
    tier = (ent >> 31) != 0
    phys = ent[~tier] & 0x7FFFFFFF
    blk = ((phys[:, None] * Hkv + np.arange(Hkv)[None, :])[:, :, None] * 2 + np.arange(2)[None, None, :]).reshape(-1)
    n_main = blk.size
    n_tier = int(tier.sum()) * Hkv * 2
    if fmt in (synth.FMT_CB2, synth.FMT_TIERED):
        cache = n_main * 12 * D + int((4 + 20 * meta[blk]).sum()) + n_tier * (16 * D + 4)
    elif fmt == synth.FMT_CB2G:
        groups = full // 4 * B                                  # one 8D codebook per (group, head, role)
        cache = n_main * 4 * D + int((4 + 20 * meta[blk]).sum()) + groups * Hkv * 2 * 8 * D
    elif fmt == synth.FMT_A3:
        cache = n_main * 10 * D + int((4 + 20 * meta[blk]).sum())
    elif fmt == synth.FMT_CB2S:
        cache = n_main * (12 * D + 16 + 32 * static_channels)
    elif fmt == synth.FMT_INT4:
        cache = n_main * (10 * D + 16) + 3 * int(meta[blk].sum())   # 1-byte channel + fp16 value per outlier
    else:
        cache = n_main * 9 * D
    tail = (N - (N // unit) * unit) * D * 4 * 2 * B * Hkv if paged else 0
    q_bytes = B * Hq * D * 2
    out_bytes = B * Hq * D * 2
    return {"cache": int(cache), "tail": int(tail), "q": q_bytes, "out": out_bytes,
            "split_kernel": int(cache + tail + q_bytes), "step": int(cache + tail + q_bytes + out_bytes)}


def algorithmic_bytes(built: workloads.Built) -> dict:
    """step_bytes() of a workload built on the device."""
    w, cache = built.w, built.cache
    meta = block_meta(w.fmt, w.D, cache.pool.view(-1, cache.block_bytes(0)))
    return step_bytes(w.fmt, w.D, w.Hkv, w.Hq, w.B, w.N, built.page_table, meta, w.static_channels)


_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|//[^\n]*|/\*.*?\*/', re.S)


def code_only(text: str) -> str:
    """C++ source with comments removed and white space collapsed (string
    literals, such as inline PTX, kept)."""
    code = _CODE_TOKENS.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(code.split())


def kernel_source_sha() -> str:
    """Hash of the decode kernel's code: a comment or layout edit leaves the
    stored traffic record valid, any code change invalidates it."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(open(os.path.join(ROOT, "sub_byte_quantized_kvq_gb300", "csrc", f)).read()).encode())
    return h.hexdigest()[:16]


def measured_peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        self.path = os.path.join(tempfile.gettempdir(), f"kvq_bench_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[4]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r[2] >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_busy": len(busy)}


# ----------------------------------------------------------------------------- GPU timing
L2_BYTES = 129 * 1024 * 1024


class L2Flush:
    """Write one buffer and read another, each larger than L2, so a step starts
    with none of its inputs cached (and no dirty lines to write back)."""

    def __init__(self, mb: int, device):
        n = max(mb, 2 * 160) * 1024 * 1024 // 2
        self.a = torch.empty(n, dtype=torch.uint8, device=device)
        self.b = torch.ones(n // 4, dtype=torch.int32, device=device)
        self.sink = torch.empty((), dtype=torch.int32, device=device)
        self.k = 0

    def __call__(self):
        self.k += 1
        self.a.fill_(self.k & 0xFF)
        torch.sum(self.b, dim=0, out=self.sink)


def time_gpu(built: workloads.Built, args, world: int, dev) -> dict:
    w, cache = built.w, built.cache
    S = w.splits if args.splits < 0 else args.splits
    S_eff = S if S > 0 else kvq.kvq_decode_num_splits(cache, w.Hq, w.N)
    q = synth.queries_bf16(args.seed, w.B, w.Hq, w.D, device=dev)
    scale = w.D ** -0.5
    ws = kvq.alloc_workspace(cache, w.Hq, w.N, S)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    nbytes = algorithmic_bytes(built)
    flush = L2Flush(args.flush_mb, dev) if nbytes["step"] < 3 * L2_BYTES else None

    def step(q_in, evs):
        # one launch: the split kernel with the split merge fused into its last CTAs
        evs[0].record()
        kvq.kvq_decode_attention(cache, q_in, scale, w.N, S, out=out, workspace=ws)
        evs[1].record()

    mk = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]  # noqa: E731
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for _ in range(args.warmup):
        if flush:
            flush()
        step(q, mk(2))
    torch.cuda.synchronize()
    barrier(world)
    evs = [mk(2) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush:
            flush()
        step(q, evs[i])
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    assert cache.status_word() == 0, f"device status {cache.status_word():#x}"

    # end to end through the C ABI with host buffers: pinned Q in, output back, every step
    q_host = q.cpu().pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_dev = torch.empty_like(q)
    e2e_evs = [mk(2) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        if flush:
            flush()
        e = e2e_evs[i - args.warmup] if i >= args.warmup else mk(2)
        e[0].record()
        q_dev.copy_(q_host, non_blocking=True)
        kvq.kvq_decode_attention(cache, q_dev, scale, w.N, S, out=out, workspace=ws)
        out_host.copy_(out, non_blocking=True)
        e[1].record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = [e[0].elapsed_time(e[1]) for e in e2e_evs]
    return {"step_ms": float(np.mean(step_ms)),
            "step_ms_median": float(np.median(step_ms)), "e2e_ms": float(np.mean(e2e_ms)), "bytes": nbytes,
            "splits": S_eff, "clocks": clocks, "flushed": flush is not None,
            "h2d": q.numel() * q.element_size(), "d2h": out.numel() * out.element_size()}


# ----------------------------------------------------------------------------- CPU oracle
ORACLE_SAMPLE_TOKENS = 8192


def oracle_sample(w: synth.Workload, seed: int):
    """Oracle cache for a bounded sample: sequence 0, all kv heads, the first
    min(N, 8192) tokens (same distributions; drawn with the CPU generator)."""
    import oracle
    N = min(w.N, ORACLE_SAMPLE_TOKENS)
    pages = (N + 15) // 16
    tiers = synth.tier_pages(seed, 1, N, w.tier_frac, w.zipf_s) if w.tier_frac > 0 else None
    pt, nm, nt = synth.page_table(seed, 1, pages, False, tiers)
    st = None
    if w.fmt == synth.FMT_CB2S:   # the oracle's own static channels, from the same calibration values
        kc, vc = workloads.calibration_kv(w, seed, "cpu")
        st = np.stack([oracle.select_static(kc.numpy(), w.static_channels),
                       oracle.select_static(vc.numpy(), w.static_channels)], 1)
    ref = oracle.OracleCache(w.fmt, 1, w.Hkv, w.D, pages, max(nm, 1), nt, page_table=pt, static_channels=st)
    for t0, T in workloads.chunks(N):
        k, v = workloads.seq_kv(w, seed, 0, t0, T, "cpu")
        ref.append(k[None].numpy(), v[None].numpy())
    q = synth.queries_bf16(seed, 1, w.Hq, w.D).view(torch.int16).numpy().view(np.uint16)
    # bytes the same step reads for this sample (same accounting as the GPU line; one sequence)
    meta = block_meta(w.fmt, w.D, ref.pool.reshape(-1, ref.stride))
    nbytes = step_bytes(w.fmt, w.D, w.Hkv, w.Hq, 1, N, pt, meta, w.static_channels)["step"]
    return ref, q, nbytes, N


def time_oracle(w: synth.Workload, seed: int, target_s: float, reps: int | None = None):
    ref, q, nbytes, N = oracle_sample(w, seed)
    cores = os.cpu_count() or 1
    scale = w.D ** -0.5
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        ref.decode(q, scale, nthreads=cores)
        times.append(time.perf_counter() - t0)
        if reps is not None and len(times) >= reps:
            break
        if reps is None and time.perf_counter() - t_start >= target_s:
            break
    mean = float(np.mean(times))
    return {"value": nbytes / mean / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"sequence 0 of {w.name}, all {w.Hkv} kv heads x {w.G} query heads, first {N} tokens, "
                      f"fp64 dequantize + attention, {len(times)} runs of {mean * 1e3:.1f} ms",
            "ms_per_step": mean * 1e3, "bytes_per_step": nbytes}


# ----------------------------------------------------------------------------- append timing (optional)
def time_append(w: synth.Workload, dev, flush_mb: int) -> dict:
    """kvq_quantize_append for every sequence of the workload: one token into
    staging, one token that completes a page (its 15 earlier tokens appended
    beforehand; page quantizer), and a 4096-token prefill chunk (bf16 inputs,
    N(0,1)).  L2 flushed before every timed call;
    CUDA events on the current stream; mean of 5 calls after 3 warm-up calls."""
    flush = L2Flush(flush_mb, dev)
    res = {"l2": "flushed before every timed call"}
    for label, T, start in (("1_token_staging", 1, 0), ("1_token_completes_page", 1, 15), ("prefill_4096", 4096, 0)):
        pages = -(-((start + T + 15) // 16) // 4) * 4   # whole groups for the CB2 group format
        c = kvq.QuantizedKVCache(w.fmt, w.B, w.Hkv, w.D, pages, w.B * pages, 0, device=dev,
                                 static_channels=w.static_channels)
        kk = torch.randn((w.B, T, w.Hkv, w.D), device=dev).to(torch.bfloat16)
        vv = torch.randn_like(kk)
        if w.fmt == synth.FMT_CB2S:
            kvq.kvq_select_static_channels(c, kk[0].contiguous(), vv[0].contiguous())
        if start:   # the page's earlier tokens, appended beforehand (untimed): the serving case
            k0 = torch.randn((w.B, start, w.Hkv, w.D), device=dev).to(torch.bfloat16)
            kvq.kvq_quantize_append(c, k0, torch.randn_like(k0))
        ts = []
        for r in range(8):
            c.seq_lens.fill_(start)
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            kvq.kvq_quantize_append(c, kk, vv)
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        t = float(np.mean(ts))
        res[label] = {"us": t * 1e6, "tokens": w.B * T, "input_gbs": 2 * kk.numel() * kk.element_size() / t / 1e9}
        del c, kk, vv
    return res


# ----------------------------------------------------------------------------- fused projection timing (optional)
def time_project(w: synth.Workload, dev, flush_mb: int, reps: int = 10, warmup: int = 3, B: int = 0) -> dict:
    """K/V projection + quantize-on-append for every sequence of the workload,
    hidden = Hq * D: the fused kvq_project_append against the unfused pair
    (two cuBLAS bf16 GEMMs writing K and V in bf16, then kvq_quantize_append),
    for a 4096-token prefill chunk and a 1-token append.  L2 flushed before
    every timed call; CUDA events on the current stream."""
    hidden = w.Hq * w.D
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak = float(json.load(f)["bf16_tflops"])   # burst: the call is timed alone
    except Exception:
        bf16_peak = 1900.0   # fallback
    if B:
        w = dataclasses.replace(w, B=B)
    flush = L2Flush(flush_mb, dev)
    res = {"hidden": hidden, "B": w.B, "l2": "flushed before every timed call"}

    def timed(fn, c):
        ts = []
        for r in range(warmup + reps):
            c.seq_lens.zero_()
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if r >= warmup:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        return float(np.mean(ts))

    for label, T in (("prefill_4096", 4096), ("1_token", 1)):
        pages = -(-((T + 15) // 16) // 4) * 4
        c = kvq.QuantizedKVCache(w.fmt, w.B, w.Hkv, w.D, pages, w.B * pages, 0, device=dev,
                                 static_channels=w.static_channels)
        x, wk, wv = synth.projection_inputs(0, w.B, T, hidden, w.Hkv, w.D, device=dev)
        if w.fmt == synth.FMT_CB2S:
            n = min(T, synth.CALIBRATION_TOKENS)
            kc = torch.matmul(x[0, :n].float(), wk.float().t()).view(n, w.Hkv, w.D).contiguous()
            vc = torch.matmul(x[0, :n].float(), wv.float().t()).view(n, w.Hkv, w.D).contiguous()
            kvq.kvq_select_static_channels(c, kc, vc)

        def unfused():
            k = torch.matmul(x, wk.t()).view(w.B, T, w.Hkv, w.D)
            v = torch.matmul(x, wv.t()).view(w.B, T, w.Hkv, w.D)
            kvq.kvq_quantize_append(c, k, v)

        def gemm_only():
            torch.matmul(x, wk.t())
            torch.matmul(x, wv.t())

        k_pre = torch.matmul(x, wk.t()).view(w.B, T, w.Hkv, w.D)
        v_pre = torch.matmul(x, wv.t()).view(w.B, T, w.Hkv, w.D)
        t_f = timed(lambda: kvq.kvq_project_append(c, x, wk, wv), c)
        t_u = timed(unfused, c)
        t_g = timed(gemm_only, c)
        t_a = timed(lambda: kvq.kvq_quantize_append(c, k_pre, v_pre), c)
        flops = 2.0 * w.B * T * hidden * 2 * w.Hkv * w.D
        res[label] = {"fused_us": t_f * 1e6, "unfused_us": t_u * 1e6, "cublas_gemms_us": t_g * 1e6,
                      "append_bf16_us": t_a * 1e6, "fused_tflops": flops / t_f / 1e12,
                      "fused_frac_of_bf16_peak": flops / t_f / 1e12 / bf16_peak,
                      "speedup_vs_unfused": t_u / t_f}
        del c, x, wk, wv, k_pre, v_pre
    return res


# ----------------------------------------------------------------------------- main
CONFIG_WORKLOADS = ("cb2_4k", "fp4_32k", "longctx_128k")   # carried beside the headline workload


def traffic_record(workload: str, other_launch):
    """DRAM bytes per launch of decode_split_kernel for `workload` from the
    committed ncu record, or None when the record is for other kernel sources
    (the kernel changed since the counters were taken) or the timed launch is
    not the recorded one (`other_launch`: another shape or decode math)."""
    try:
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
    except Exception:
        return None
    if tr.get("kernel_src_sha") != kernel_source_sha():
        return None
    rec = tr.get("workloads", {}).get(workload)
    if rec is None or other_launch:
        return None
    return rec.get("dram_bytes_per_launch")


def measure_workload(w: synth.Workload, args, world: int, rank: int, dev, peak: float, peak_kind: str) -> dict:
    """Build the workload's cache on the device, time its decode step, and
    return the timing with its roofline (the split kernel is the whole step)."""
    built = workloads.build(w, seed=args.seed + rank, device=dev)
    built.cache.cfg.decode_math = DECODE_MATH[args.decode_math]
    torch.cuda.synchronize()
    t = time_gpu(built, args, world, dev)
    del built
    torch.cuda.empty_cache()
    t["step_ms"] = all_max(t["step_ms"], world)
    t["e2e_ms"] = all_max(t["e2e_ms"], world)
    t["step_ms_median"] = all_max(t["step_ms_median"], world)
    nb = t["bytes"]
    achieved = nb["step"] / (t["step_ms"] * 1e-3) / 1e9
    t["roofline"] = {"bound": "hbm", "kernel": "decode_split_kernel", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic_record(w.name, args.batch or args.q_heads or args.decode_math != "auto"),
                     "algorithmic_bytes_per_launch": nb["step"], "us_per_launch": t["step_ms"] * 1e3,
                     "frac_of_nominal_8000_gbs": achieved / 8000.0}
    t["l2"] = ("flushed before every step (write 256 MB + read 256 MB)" if t["flushed"]
               else f"inputs exceed L2 ({nb['step'] / L2_BYTES:.1f} x its 129 MB; no flush)")
    return t


def main():
    args = parse_args()
    rank, world = dist_setup(args)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    if args.q_heads:
        w = dataclasses.replace(w, Hq=args.q_heads)
    config = {"workload": w.name, "format": FMT_NAME[w.fmt], "B": w.B, "Hkv": w.Hkv, "Hq": w.Hq, "D": w.D,
              "context": w.N, "page_tokens": 16}
    if args.decode_math != "auto":
        config["decode_math"] = args.decode_math

    if args.impl == "reference":
        if rank != 0:
            return
        r = time_oracle(w, args.seed, 0.0, reps=args.warmup + args.steps)
        line = {"metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": dict(config, sample=r["sample"]),
                "cpu_baseline": {"value": r["value"], "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    dev = torch.device("cuda", torch.cuda.current_device())
    if args.project_only:
        if rank == 0:
            print(json.dumps({"workload": w.name, "format": FMT_NAME[w.fmt],
                              "project": time_project(w, dev, args.flush_mb, B=args.project_b)}), flush=True)
        return
    peak, peak_kind = measured_peak_gbs()
    t = measure_workload(w, args, world, rank, dev, peak, peak_kind)
    nb = t["bytes"]
    step_ms, e2e_ms = t["step_ms"], t["e2e_ms"]
    line = {
        "metric": METRIC,
        "value": world * nb["step"] / (step_ms * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_ms, "us_per_step": step_ms * 1e3,
        "us_per_step_median": t["step_ms_median"] * 1e3,   # event timestamps tick in ~2 us steps
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 mma / f32 accumulate over 2-4 bit codes", "data": "synthetic",
        "config": dict(config, splits=t["splits"], l2=t["l2"], bytes_per_step=nb["step"],
                       partial_bytes_per_step=2 * w.B * w.Hq * t["splits"] * (w.D + 2) * 4),
        "roofline": t["roofline"],
        "e2e": {"value": world * nb["step"] / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": t["h2d"], "d2h_bytes_per_step": t["d2h"], "us_per_step": e2e_ms * 1e3,
                "us_host_and_copies_beyond_device_step": (e2e_ms - step_ms) * 1e3},
        "gpu_launches": args.steps,
        "clocks": t["clocks"],
    }
    if not args.no_configs and not args.batch and not args.q_heads:
        configs = {}
        for name in CONFIG_WORKLOADS:
            if name == w.name:
                continue
            wc = synth.WORKLOADS[name]
            tc = measure_workload(wc, args, world, rank, dev, peak, peak_kind)
            configs[name] = {"format": FMT_NAME[wc.fmt], "B": wc.B, "Hkv": wc.Hkv, "Hq": wc.Hq, "D": wc.D,
                             "context": wc.N, "splits": tc["splits"], "l2": tc["l2"],
                             "bytes_per_step": tc["bytes"]["step"], "us_per_step": tc["step_ms"] * 1e3,
                             "us_per_step_median": tc["step_ms_median"] * 1e3,
                             "value": world * tc["bytes"]["step"] / (tc["step_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                             "roofline": tc["roofline"], "clocks": tc["clocks"]}
        line["configs"] = configs
    if not args.no_append:
        line["append"] = dict(time_append(synth.WORKLOADS[args.append_workload], dev, args.flush_mb),
                              workload=args.append_workload)
    if args.project:
        line["project"] = time_project(w, dev, args.flush_mb, B=args.project_b)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = time_oracle(w, args.seed, args.cpu_seconds)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
