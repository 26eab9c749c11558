#!/usr/bin/env python3
"""Benchmark of the quantized KV-cache hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {kvq,reference}]

One JSON line on stdout (rank 0).

Workload (the decode configuration the headline metric is quoted on): a
Llama-3-8B-shaped decode layer -- batch 16, 32 query / 8 KV heads, head_dim
128, context 4096, K and V INT4 token-wise with Hadamard block 128, page 16 --
replicated over 32 distinct layer caches (2.3 GB of packed KV, far above the
126 MB L2), so every step streams its cache from HBM.

A step is one serving decode step through all 32 layers: per layer, one
kvq_decode_step call quantizes the new token of each of the 16 sequences into
the paged cache (rotation, scale/zero, codes, paged store) and runs split-K
attention over the 4096 cached tokens (query rotation, page streaming,
dequantization in registers, online softmax, merge) in a single launch.  The
bit-widths come from kvq_alloc_bits at set-up (this workload's widths are
uniform: 4 and 4).  The step is captured once in a CUDA graph and replayed.

value = algorithmic bytes of a step / step time, summed over ranks.  Bytes per
layer: packed codes + fp16 scale/zero of the cached tokens (136 B per (token,
KV head) for K4V4), the new tokens' bf16 K/V read and their codes written, q
read, o written, the page-table rows read.  The "roofline" object is the
decode-step kernel alone, timed by CUDA-event nodes around each launch inside
the replayed step.  "append" adds the quantize-on-append sweep (8 sequences x
8192 new tokens, every Hadamard block and bit width) in tokens/s.
"cpu_baseline" times the CPU oracle on a bounded sample.

Further sections of the same line, each with its own roofline object:
"mixed_bits" (32 layers x 8 KV heads, batch 64, context 2048, per-head bits
from kvq_alloc_bits fed by kvq_distortion + kvq_fit_distortion, at 3.0 and
3.5 average bits), "long_context" (1 sequence x 131072 tokens, K4V2, a
128-token bf16 window), "logquant" (the same shape at K2V2 with LogQuant's
log-spaced bf16 tokens, W = 128) and "quant_error" (error of the cache's
attention against float64 attention over the original bf16 K/V, with and
without the rotation, computed with torch on the device), "key_per_channel"
(the Llama-3-8B-shaped layer with keys quantized per channel, decode attention
alone).  --only {append,mixed,long,logquant,key_channel} runs one of them (or the
append sweep) alone over --layers layer caches.

--impl reference times the CPU oracle itself as the reference arm (this
library has no third-party reference implementation to install).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (APPEND_BITS, APPEND_BLOCKS, APPEND_SWEEP, LLAMA3_8B_LAYER,  # noqa: E402
                       LONG_CONTEXT, MIXED_32L, TINY, kv_tokens, page_table, queries,
                       sensitivities)

METRIC = "quantized-KV decode attention GB/s (% of HBM peak); append tokens/s"
N_LAYERS = 32
W = LLAMA3_8B_LAYER


def unit_bytes(d: int, bk: int, bv: int) -> int:
    """Algorithmic bytes per (token, KV head): packed K and V codes + fp16 (s, z) x 2."""
    return d * (bk + bv) // 8 + 8


def decode_bytes_per_layer() -> int:
    """Algorithmic bytes one decode step of one layer moves (see the module docstring)."""
    d, hkv, hq, bsz, ctx = W.head_dim, W.hkv, W.hq, W.batch, W.ctx
    cache = bsz * ctx * hkv * unit_bytes(d, 4, 4)      # codes + (s, z) read
    new_tok = bsz * hkv * 2 * (2 * d + d * 4 // 8 + 4)  # bf16 K, V read; codes, (s, z) written
    q_o = bsz * hq * d * (2 + 4)                        # bf16 q read, fp32 o written
    ptab = bsz * (ctx // 16) * 4
    return cache + new_tok + q_o + ptab


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "source": "fallback"}


def ncu_traffic() -> "int | None":
    """DRAM bytes (read + write) of one decode-step launch from the committed ncu
    capture (profiles/traffic.json), or None once the kernel sources changed."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get("decode_kernel<128> llama3-8b-decode-layer step")
    if not rec:
        return None
    h = hashlib.sha256()
    for name in rec["sources"]:
        with open(os.path.join(ROOT, "quantized_decode_attention_diag_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return int(rec["per_launch_bytes"]) if h.hexdigest()[:16] == rec["source_sha256_16"] else None


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.window = None   # (start, end) of the timed region, local wall clock
        # raw samples: $KVQ_CLOCKS_CSV (a path template with {rank}) or a temporary file
        tmpl = os.environ.get("KVQ_CLOCKS_CSV")
        if tmpl:
            self.path = tmpl.format(rank=gpu_index)
        else:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix=f"kvq_clocks_rank{gpu_index}_", suffix=".csv")
            os.close(fd)

    def __enter__(self):
        try:
            if os.path.dirname(self.path):
                os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(1.5)          # nvidia-smi needs a moment before its first sample
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def mark(self, start, end) -> None:
        self.window = (start, end)

    def summary(self) -> dict:
        import datetime as _dt
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(f[2]), float(f[3])
            except ValueError:
                continue
            if self.window and not (self.window[0] - 0.25 <= ts <= self.window[1] + 0.25):
                continue
            sm.append(clk)
            smax.append(cmax)
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------- oracle legs

class OracleSample:
    """The CPU oracle on a bounded sample of the workload.

    The sample is n_seqs of the 16 sequences of one layer: the oracle fills its
    own cache for them at construction (untimed); step() is one decode step for
    them -- append of the new token and attention over 4096 tokens for all 8
    KV heads / 32 query heads."""

    def __init__(self, n_seqs: int):
        from oracle import cache as ocache
        try:
            from threadpoolctl import threadpool_info
            self.threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
        except Exception:  # noqa: BLE001
            self.threads = 1
        d, hkv, ctx = W.head_dim, W.hkv, W.ctx
        self.n = n_seqs
        self.k = kv_tokens(W.seed, 0, n_seqs, ctx, hkv, d, W.k_outliers, W.outlier_lo,
                           W.outlier_hi)
        self.v = kv_tokens(W.seed, 1, n_seqs, ctx, hkv, d, W.v_outliers, W.outlier_lo,
                           W.outlier_hi)
        mp = ctx // 16
        self.pt = page_table(W.seed, n_seqs, mp)
        self.st = ocache.new_state(1, n_seqs * mp, d, W.had_block, np.full((1, hkv, 2), 4))
        ocache.append(self.st, 0, self.k[:, :ctx - 1], self.v[:, :ctx - 1], self.pt,
                      np.zeros(n_seqs, np.int32))
        self.q = queries(W.seed, 0, n_seqs, W.hq, d, False).astype(np.float64)
        self.before = np.full(n_seqs, ctx - 1, np.int32)
        self.nbytes = decode_bytes_per_layer() * n_seqs // W.batch   # same byte count, pro rata

    def step(self) -> float:
        from oracle import attention, cache as ocache
        ctx = W.ctx
        t0 = time.perf_counter()
        ocache.append(self.st, 0, self.k[:, ctx - 1:], self.v[:, ctx - 1:], self.pt, self.before)
        attention.decode(self.st, 0, self.q, self.pt, self.before + 1)
        return time.perf_counter() - t0

    def describe(self, repeats: int) -> str:
        return (f"{self.n} of {W.batch} sequences x {W.hkv} KV heads x {W.ctx} tokens of one "
                f"layer (one decode step: append 1 token + attention), median of {repeats}")


def oracle_baseline(n_seqs: int = 4, repeats: int = 5) -> dict:
    o = OracleSample(n_seqs)
    o.step()
    sec = statistics.median([o.step() for _ in range(repeats)])
    return {"value": round(o.nbytes / sec / 1e9, 4), "unit": "GB/s", "cores": o.threads,
            "host_cpus": os.cpu_count(), "kind": "oracle", "sample": o.describe(repeats)}


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    o = OracleSample(2)
    for _ in range(args.warmup):
        o.step()
    times = [o.step() for _ in range(max(1, min(args.steps, 50)))]
    sec = sum(times) / len(times)
    gbs = o.nbytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": o.threads,
                         "host_cpus": os.cpu_count(), "kind": "oracle",
                         "sample": o.describe(len(times))},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict() -> dict:
    return {"workload": "llama3-8b-decode-layer x 32 layer caches",
            "batch": W.batch, "q_heads": W.hq, "kv_heads": W.hkv, "head_dim": W.head_dim,
            "context": W.ctx, "bits": "K4V4", "had_block": W.had_block, "page": 16,
            "layers": N_LAYERS,
            "step": "per layer: kvq_decode_step (append 1 token/seq fused with split-K decode)",
            "l2": (f"inputs larger than L2: {N_LAYERS} distinct layer caches, "
                   f"{N_LAYERS * decode_bytes_per_layer() / 1e9:.2f} GB of packed KV per step"),
            "parallelism": "replicas (weak scaling), no collective on the data path"}


# ------------------------------------------------------------------------- GPU leg

def init_distributed(world: int, local: int):
    """One process per GPU (NCCL) for N > 1; gloo on a machine without CUDA."""
    import torch
    import torch.distributed as dist
    if world <= 1:
        return
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist.init_process_group("gloo")


def max_over_ranks(value: float, world: int, dev) -> float:
    """The largest of the ranks' values (a step time): one all-reduce of a
    scalar, nothing on the data path."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_kvq(args) -> None:
    import torch
    import torch.distributed as dist

    import quantized_decode_attention_diag_b300 as kvq
    from quantized_decode_attention_diag_b300 import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    init_distributed(world, local)
    dev = torch.device("cuda", local if world > 1 else 0)
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()

    # CPU baseline first (rank 0 only), before the first kernel runs
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_baseline(4, 5)

    d, hkv, hq, bsz, ctx = W.head_dim, W.hkv, W.hq, W.batch, W.ctx
    # bit-widths from the allocator (uniform sensitivities, only width 4 allowed)
    bits, _ = kvq.kvq_alloc_bits([1.0] * (N_LAYERS * hkv * 2), [4.0] * (N_LAYERS * hkv * 2),
                                 4 * N_LAYERS * hkv * 2, [kvq.mask_of([4])] * (N_LAYERS * hkv * 2))
    bits = np.array(bits).reshape(N_LAYERS, hkv, 2)
    mp = ctx // 16
    # programmatic dependent launch: a layer's decode step starts its page copies
    # while the previous layer's kernel finishes (no kernel of the step writes
    # another layer's pool, the page table or the lengths)
    cache = kvq.Cache(N_LAYERS, hkv, d, W.had_block, bits, bsz * mp, device=dev, overlap=True)
    pt = torch.from_numpy(page_table(W.seed, bsz, mp)).to(dev)

    # prefill every layer cache with the first ctx-1 tokens (one layer's data, 32 caches)
    k = kv_tokens(W.seed, 0, bsz, ctx, hkv, d, W.k_outliers, W.outlier_lo, W.outlier_hi)
    v = kv_tokens(W.seed, 1, bsz, ctx, hkv, d, W.v_outliers, W.outlier_lo, W.outlier_hi)
    kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
    vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    zero = torch.zeros(bsz, dtype=torch.int32, device=dev)
    for l in range(N_LAYERS):
        cache.append(l, kd[:, :ctx - 1].contiguous(), vd[:, :ctx - 1].contiguous(), pt, zero)
    knew = kd[:, ctx - 1].contiguous().unsqueeze(0).repeat(N_LAYERS, 1, 1, 1).contiguous()
    vnew = vd[:, ctx - 1].contiguous().unsqueeze(0).repeat(N_LAYERS, 1, 1, 1).contiguous()
    del kd, vd
    q_host = np.stack([queries(W.seed, l, bsz, hq, d, False) for l in range(N_LAYERS)])
    q_all = torch.from_numpy(q_host).to(dev).to(torch.bfloat16)
    o_all = torch.empty((N_LAYERS, bsz, hq, d), dtype=torch.float32, device=dev)
    before = torch.full((bsz,), ctx - 1, dtype=torch.int32, device=dev)
    after = before + 1
    ws = cache.workspace(bsz, hq, mp)
    torch.cuda.synchronize(dev)
    assert cache.get_status() == 0

    stream = torch.cuda.Stream(device=dev)
    ev = [(torch.cuda.Event(enable_timing=True, external=True),
           torch.cuda.Event(enable_timing=True, external=True)) for _ in range(N_LAYERS)]

    def step():
        for l in range(N_LAYERS):
            cache.decode_step(l, knew[l], vnew[l], q_all[l], pt, after, o=o_all[l], workspace=ws)

    def step_events():   # each launch between events: no overlap, per-launch times
        for l in range(N_LAYERS):
            ev[l][0].record()
            cache.decode_step(l, knew[l], vnew[l], q_all[l], pt, after, o=o_all[l], workspace=ws)
            ev[l][1].record()

    with torch.cuda.stream(stream):
        step()                                   # eager warm-up outside capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        step_events()
    torch.cuda.synchronize(dev)

    def timed(fn, k_steps):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record()
            for _ in range(k_steps):
                fn()
            t1.record()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        return max_over_ranks(t0.elapsed_time(t1) / k_steps, world, dev)

    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        t_start = time.time()
        ms = nvtx(torch, "decode step graph (timed)", timed, graph.replay, args.steps)
        clocks.mark(t_start, time.time())
    # isolated launches (events between them), after the timed region
    for _ in range(3):
        with torch.cuda.stream(stream):
            graph_ev.replay()
    torch.cuda.synchronize(dev)
    dec_ms = [ev[l][0].elapsed_time(ev[l][1]) for l in range(N_LAYERS)]   # last replay
    assert cache.get_status() == 0, f"device status {cache.get_status():#x}"

    # end to end: pinned host inputs -> device, step, o -> pinned host
    knew_h = knew.cpu().pin_memory()
    vnew_h = vnew.cpu().pin_memory()
    q_h = q_all.cpu().pin_memory()
    o_h = torch.empty(o_all.shape, dtype=torch.float32).pin_memory()

    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    inputs_in = [torch.cuda.Event() for _ in range(N_LAYERS)]
    layer_done = [torch.cuda.Event() for _ in range(N_LAYERS)]

    # upload groups of growing size (layers [0, 1), [1, 4), [4, 12), [12, L)):
    # the decode steps wait on a group only at its first layer, so the
    # launches inside a group keep their programmatic overlap; the first group
    # is small, so little of the upload is exposed
    bounds = sorted({0, N_LAYERS} | {b for b in (1, 4, 12) if b < N_LAYERS})
    groups = list(zip(bounds[:-1], bounds[1:]))
    # read-back groups of shrinking size ([0, L - 20), ..., [L - 1, L)): few
    # cross-stream waits, and only the last layer's o is left after the step
    rb = sorted({0, N_LAYERS} | {N_LAYERS - x for x in (1, 4, 12, 20) if x < N_LAYERS})
    rb_first = {b - 1: a for a, b in zip(rb[:-1], rb[1:])}   # last layer -> first

    def e2e_body():
        # the inputs go over on one copy stream in a few large copies, ahead of
        # the decode steps; the o of finished layers comes back on another
        # stream while the next layers run; the step ends when the last copy has
        # landed.  (A wait before every layer's step cut the overlap of
        # consecutive launches; uploading everything first exposed the whole
        # upload.)
        cur = torch.cuda.current_stream()
        h2d_stream.wait_stream(cur)
        d2h_stream.wait_stream(cur)
        with torch.cuda.stream(h2d_stream):
            for gi, (a, b) in enumerate(groups):
                q_all[a:b].copy_(q_h[a:b], non_blocking=True)
                knew[a:b].copy_(knew_h[a:b], non_blocking=True)
                vnew[a:b].copy_(vnew_h[a:b], non_blocking=True)
                inputs_in[gi].record(h2d_stream)
        first = {a: gi for gi, (a, _) in enumerate(groups)}
        for l in range(N_LAYERS):
            if l in first:
                cur.wait_event(inputs_in[first[l]])
            cache.decode_step(l, knew[l], vnew[l], q_all[l], pt, after, o=o_all[l], workspace=ws)
            if l in rb_first:
                a = rb_first[l]
                layer_done[l].record(cur)
                d2h_stream.wait_event(layer_done[l])
                with torch.cuda.stream(d2h_stream):
                    o_h[a:l + 1].copy_(o_all[a:l + 1], non_blocking=True)
        cur.wait_stream(h2d_stream)
        cur.wait_stream(d2h_stream)

    with torch.cuda.stream(stream):
        e2e_body()                               # eager warm-up outside capture
    torch.cuda.synchronize(dev)
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_body()
    torch.cuda.synchronize(dev)

    for _ in range(max(1, args.warmup)):
        with torch.cuda.stream(stream):
            e2e_graph.replay()
    ms_e2e = nvtx(torch, "e2e step graph (timed)", timed, e2e_graph.replay, args.steps)
    o_check = torch.from_numpy(o_h.numpy().copy())
    assert torch.equal(o_check, o_all.cpu()), "e2e: host copy of o differs from the device o"
    h2d = q_h.numel() * 2 + knew_h.numel() * 2 + vnew_h.numel() * 2
    d2h = o_h.numel() * 4

    del cache, ws, knew, vnew, q_all, o_all
    torch.cuda.synchronize(dev)
    # append sweep: 8 sequences x 8192 new tokens into empty caches
    append = nvtx(torch, "append sweep", append_sweep, kvq, torch, dev) \
        if not args.skip_append else None
    calib = nvtx(torch, "calibration", calibration_bench, kvq, torch, dev) \
        if not args.skip_append else None
    mixed = long_ctx = qerr = lq = kpc = None
    if not args.skip_configs:
        # the mixed-bits allocation takes (alpha, beta) from the calibration
        if calib is not None:
            alpha, beta = calib["_alpha"], calib["_beta"]
        else:
            alpha = np.ones(N_LAYERS * hkv * 2)
            beta = np.full(N_LAYERS * hkv * 2, 4.0)
        if N_LAYERS == MIXED_32L.num_layers:
            mixed = nvtx(torch, "mixed bits", mixed_bits_bench, kvq, torch, dev, alpha, beta,
                         min(args.steps, 10), args.warmup)
        long_ctx = nvtx(torch, "long context", long_context_bench, kvq, torch, dev, N_LAYERS,
                        args.steps, args.warmup)
        lq = nvtx(torch, "LogQuant", logquant_bench, kvq, torch, dev, N_LAYERS, args.steps,
                  args.warmup)
        kpc = nvtx(torch, "key-per-channel", key_channel_bench, kvq, torch, dev, N_LAYERS,
                   args.steps, args.warmup)
        qerr = nvtx(torch, "quantization error", quant_error_report, kvq, torch, dev)
    if calib is not None:
        calib.pop("_alpha")
        calib.pop("_beta")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    pk = peaks()
    step_bytes = N_LAYERS * decode_bytes_per_layer()
    gbs = world * step_bytes / (ms * 1e-3) / 1e9
    # the timed region holds only the N_LAYERS decode-step launches of each step
    launch_ms = ms / N_LAYERS
    achieved = decode_bytes_per_layer() / (launch_ms * 1e-3) / 1e9
    dec_avg = statistics.mean(dec_ms)
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u4 codes, fp16 MMA, fp32 accumulate", "data": "synthetic",
        "config": config_dict(),
        "frac_of_hbm": round(gbs / world / pk["hbm_gbs"], 4),
        "roofline": {"bound": "hbm",
                     "kernel": "decode_kernel<128> (decode step: append + split-K decode + merge)",
                     "achieved": round(achieved, 2), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4),
                     "peak_source": pk["source"], "traffic": ncu_traffic(),
                     "algorithmic_bytes_per_launch": decode_bytes_per_layer(),
                     "avg_launch_us": round(launch_ms * 1e3, 3),
                     "isolated_launch_us": round(dec_avg * 1e3, 3)},
        "e2e": {"value": round(world * step_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(ms_e2e, 4)},
        "gpu_launches": N_LAYERS * args.steps,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "append": append,
        "calibration": calib,
        "mixed_bits": mixed,
        "long_context": long_ctx,
        "logquant": lq,
        "key_per_channel": kpc,
        "quant_error": qerr,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def append_sweep(kvq, torch, dev) -> dict:
    w = APPEND_SWEEP
    bsz, t, hkv, d = w.batch, w.new_tokens, w.hkv, w.head_dim
    k = kv_tokens(w.seed, 0, bsz, t, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, t, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi)
    kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
    vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    del k, v
    mp = t // 16
    pt = torch.from_numpy(page_table(w.seed, bsz, mp)).to(dev)
    zero = torch.zeros(bsz, dtype=torch.int32, device=dev)
    pk = peaks()
    points = []
    tokens = bsz * t
    for block in APPEND_BLOCKS:
        for bits in APPEND_BITS:
            c = kvq.Cache(1, hkv, d, block, np.full((1, hkv, 2), bits), bsz * mp, device=dev)
            for _ in range(3):
                c.append(0, kd, vd, pt, zero)
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            reps = 10
            e0.record()
            for _ in range(reps):
                c.append(0, kd, vd, pt, zero)
            e1.record()
            torch.cuda.synchronize(dev)
            assert c.get_status() == 0
            sec = e0.elapsed_time(e1) / reps * 1e-3
            nbytes = tokens * hkv * 2 * (d * 2 + d * bits // 8 + 4)
            points.append({"block": block, "bits": bits, "us": round(sec * 1e6, 2),
                           "tokens_per_s": round(tokens / sec, 1),
                           "GB_s": round(nbytes / sec / 1e9, 1),
                           "frac": round(nbytes / sec / 1e9 / pk["hbm_gbs"], 4)})
            del c
    return {"workload": "append-sweep 8 seqs x 8192 new tokens, 8 KV heads, head_dim 128",
            "bytes": "bf16 K/V read + packed codes + fp16 (s, z) written",
            "unit": "tokens/s", "points": points}


def calibration_bench(kvq, torch, dev) -> dict:
    """Distortion calibration of a 32-layer cache: per layer, K and V of 16
    calibration sequences x 512 tokens (8 KV heads, head_dim 128), MSE at widths
    2 .. 6 (kvq_distortion), then the host fit of (alpha, beta) per component."""
    w = LLAMA3_8B_LAYER
    seqs, t, hkv, d, widths = 16, 512, w.hkv, w.head_dim, [2, 3, 4, 5, 6]
    T = seqs * t
    xs = [torch.from_numpy(kv_tokens(w.seed + 7, kv, seqs, t, hkv, d,
                                     w.k_outliers if kv == 0 else w.v_outliers,
                                     w.outlier_lo, w.outlier_hi).reshape(T, hkv, d))
          .to(dev).to(torch.bfloat16) for kv in range(2)]
    outs = [torch.empty((hkv, len(widths)), dtype=torch.float64, device=dev)
            for _ in range(2 * N_LAYERS)]

    def run():   # 2 * N_LAYERS calls: the two sample tensors stand in for every layer's
        for i in range(2 * N_LAYERS):
            kvq.kvq_distortion(d, w.had_block, xs[i % 2], widths, mse=outs[i])

    for _ in range(3):
        run()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    reps = 5
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / reps * 1e-3 / (2 * N_LAYERS)
    t0 = time.perf_counter()
    # call i = 2 layer + kv holds [head][width]: into the allocator's component
    # order (layer * Hkv + head) * 2 + kv
    mse = (torch.stack(outs).cpu().numpy().reshape(N_LAYERS, 2, hkv, len(widths))
           .transpose(0, 2, 1, 3).reshape(-1, len(widths)))
    alpha, beta = kvq.kvq_fit_distortion(mse, widths)
    fit_s = time.perf_counter() - t0
    nbytes = T * hkv * d * 2
    pk = peaks()
    return {"workload": f"calibration: {N_LAYERS} layers x (K, V) x {seqs} seqs x {t} tokens, "
                        f"{hkv} KV heads, head_dim {d}, widths 2..6",
            "us_per_call": round(sec * 1e6, 2), "vectors_per_s": round(T * hkv / sec, 1),
            "GB_s": round(nbytes / sec / 1e9, 1),
            "frac_of_hbm": round(nbytes / sec / 1e9 / pk["hbm_gbs"], 4),
            "bytes": "bf16 vectors read once per call",
            "fit_ms": round(fit_s * 1e3, 3),
            "beta_range": [round(float(beta.min()), 3), round(float(beta.max()), 3)],
            "_alpha": alpha, "_beta": beta}


def nvtx(torch, name, fn, *a, **kw):
    """fn(*a, **kw) inside an NVTX range named `name` (visible to a timeline
    profiler; no effect otherwise)."""
    torch.cuda.nvtx.range_push(name)
    try:
        return fn(*a, **kw)
    finally:
        torch.cuda.nvtx.range_pop()


def graph_step_bench(torch, dev, cache, n_layers, knew, vnew, q_all, pt, after, o_all, ws,
                     steps, warmup, decode_only=False) -> tuple:
    """Times one step of n_layers fused decode steps (one per layer cache;
    with decode_only, decode attention alone), captured once as a CUDA graph
    with layer-to-layer launch overlap, and the same launches with events
    between them.  Returns (ms per step, average isolated launch in ms)."""
    stream = torch.cuda.Stream(device=dev)
    ev = [(torch.cuda.Event(enable_timing=True, external=True),
           torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n_layers)]

    def layer(l):
        if decode_only:
            cache.decode(l, q_all[l], pt, after, o=o_all[l], workspace=ws)
        else:
            cache.decode_step(l, knew[l], vnew[l], q_all[l], pt, after, o=o_all[l], workspace=ws)

    def step():
        for l in range(n_layers):
            layer(l)

    def step_events():
        for l in range(n_layers):
            ev[l][0].record()
            layer(l)
            ev[l][1].record()

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        step_events()
    for _ in range(warmup):
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record()
        for _ in range(steps):
            graph.replay()
        t1.record()
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    for _ in range(3):
        with torch.cuda.stream(stream):
            graph_ev.replay()
    torch.cuda.synchronize(dev)
    iso = statistics.mean(ev[l][0].elapsed_time(ev[l][1]) for l in range(n_layers))
    assert cache.get_status() == 0, f"device status {cache.get_status():#x}"
    return ms, iso


def step_bytes_layer(bits_layer, bsz, ctx, hq, d, window=0, partial_floats=0) -> int:
    """Algorithmic bytes of one layer's decode step: the quantized tokens'
    codes and (s, z), the bf16 window, the new token (bf16 K/V read, one
    vector per head quantized and written), q read, o written, page-table rows,
    and split partials (written and read once) where the merge keeps them in
    memory."""
    lq = ctx - window
    cache_b = bsz * lq * sum(unit_bytes(d, int(bk), int(bv)) for bk, bv in bits_layer)
    win_b = bsz * window * len(bits_layer) * 2 * 2 * d
    new_tok = bsz * sum(2 * 2 * d + d * (int(bk) + int(bv)) // 8 + 8 for bk, bv in bits_layer)
    q_o = bsz * hq * d * (2 + 4)
    ptab = bsz * ((ctx + 15) // 16) * 4
    return cache_b + win_b + new_tok + q_o + ptab + 2 * 4 * partial_floats


def _roofline(step_bytes, ms, n_layers, iso_ms, bytes_per_launch) -> dict:
    pk = peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
            "peak_source": pk["source"], "traffic": None,
            "algorithmic_bytes_per_launch": int(bytes_per_launch),
            "avg_launch_us": round(ms / n_layers * 1e3, 3),
            "isolated_launch_us": round(iso_ms * 1e3, 3)}


def mixed_bits_bench(kvq, torch, dev, alpha, beta, steps, warmup, n_layers=None) -> dict:
    """The mixed per-head bits workload: 32 layers x 8 KV heads, batch 64,
    context 2048, 32 query heads, bits from the RateQuant greedy (sensitivities
    lognormal x U-shape over depth, times alpha; beta per component from the
    calibration section) at the stated 3-bit average (which leaves K4V2 on
    every head) and at 3.5 bits.  One step = one fused decode step per layer,
    each over its own cache (3.5-4.3 GB per step: far above L2).  Layer 0's
    K/V streams fill every layer's cache (the values do not change the work)."""
    w = MIXED_32L
    L, hkv, hq, d, bsz, ctx = w.num_layers, w.hkv, w.hq, w.head_dim, w.batch, w.ctx
    if n_layers is not None:
        L = n_layers                  # a smaller case for profiling
    mp = ctx // 16
    sens = sensitivities(w.seed, L, hkv).reshape(-1)
    allowed = [kvq.mask_of([4, 8]), kvq.mask_of([2, 4])] * (L * hkv)
    k = kv_tokens(w.seed, 0, bsz, ctx, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, ctx, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi)
    kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
    vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    del k, v
    kpre, vpre = kd[:, :ctx - 1].contiguous(), vd[:, :ctx - 1].contiguous()
    knew = kd[:, ctx - 1].contiguous().unsqueeze(0).repeat(L, 1, 1, 1).contiguous()
    vnew = vd[:, ctx - 1].contiguous().unsqueeze(0).repeat(L, 1, 1, 1).contiguous()
    del kd, vd
    pt = torch.from_numpy(page_table(w.seed, bsz, mp)).to(dev)
    q_all = torch.from_numpy(np.stack([queries(w.seed, l, bsz, hq, d, False) for l in range(L)])
                             ).to(dev).to(torch.bfloat16)
    o_all = torch.empty((L, bsz, hq, d), dtype=torch.float32, device=dev)
    zero = torch.zeros(bsz, dtype=torch.int32, device=dev)
    after = torch.full((bsz,), ctx, dtype=torch.int32, device=dev)
    out = {"workload": f"mixed per-head bits: {L} layers x {hkv} KV heads, {hq} q heads, "
                       f"head_dim {d}, batch {bsz}, context {ctx}, Hadamard {w.had_block}",
           "step": "per layer: kvq_decode_step over its own cache", "variants": []}
    a = np.asarray(alpha, np.float64)
    b = np.asarray(beta, np.float64)
    for avg in (3.0, 3.5):
        budget = int(round(avg * L * hkv * 2))
        bits, left = kvq.kvq_alloc_bits(sens * a, b, budget, allowed)
        bits = np.array(bits).reshape(L, hkv, 2)
        cache = kvq.Cache(L, hkv, d, w.had_block, bits, bsz * mp, device=dev, overlap=True)
        for l in range(L):
            cache.append(l, kpre, vpre, pt, zero)
        ws = cache.workspace(bsz, hq, mp)
        torch.cuda.synchronize(dev)
        ms, iso = graph_step_bench(torch, dev, cache, L, knew, vnew, q_all, pt, after, o_all, ws,
                                   steps, warmup)
        per_layer = [step_bytes_layer(bits[l], bsz, ctx, hq, d) for l in range(L)]
        sb = sum(per_layer)
        mix = {}
        for bk, bv in bits.reshape(-1, 2):
            key = f"K{bk}V{bv}"
            mix[key] = mix.get(key, 0) + 1
        out["variants"].append({
            "avg_bits": avg, "budget_bits": budget, "leftover_bits": left, "heads_by_bits": mix,
            "ms_per_step": round(ms, 4), "GB_per_step": round(sb / 1e9, 4),
            "roofline": _roofline(sb, ms, L, iso, sb / L)})
        del cache, ws
        torch.cuda.synchronize(dev)
    return out


def long_context_bench(kvq, torch, dev, n_layers, steps, warmup) -> dict:
    """Long context: one sequence of 131072 tokens, 32 query / 8 KV heads,
    head_dim 128, K INT4 / V INT2 with Hadamard 128, the last 128 tokens kept
    in a bf16 window.  One step = one fused decode step per layer over
    n_layers distinct layer caches (109.5 MB each: together far above L2)."""
    w = LONG_CONTEXT
    hkv, hq, d, ctx, r = w.hkv, w.hq, w.head_dim, w.ctx, w.window
    mp = ctx // 16
    k = kv_tokens(w.seed, 0, 1, ctx, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, 1, ctx, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi)
    kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
    vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    del k, v
    bits = np.tile(np.array([w.k_bits, w.v_bits]), (n_layers, hkv, 1))
    cache = kvq.Cache(n_layers, hkv, d, w.had_block, bits, mp, window=r, max_batch=1,
                      device=dev, overlap=True)
    pt = torch.from_numpy(page_table(w.seed, 1, mp)).to(dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    kpre, vpre = kd[:, :ctx - 1].contiguous(), vd[:, :ctx - 1].contiguous()
    for l in range(n_layers):
        cache.append(l, kpre, vpre, pt, zero)
    knew = kd[:, ctx - 1].contiguous().unsqueeze(0).repeat(n_layers, 1, 1, 1).contiguous()
    vnew = vd[:, ctx - 1].contiguous().unsqueeze(0).repeat(n_layers, 1, 1, 1).contiguous()
    del kd, vd, kpre, vpre
    q_all = torch.from_numpy(np.stack([queries(w.seed, l, 1, hq, d, False)
                                       for l in range(n_layers)])).to(dev).to(torch.bfloat16)
    o_all = torch.empty((n_layers, 1, hq, d), dtype=torch.float32, device=dev)
    after = torch.full((1,), ctx, dtype=torch.int32, device=dev)
    ws = cache.workspace(1, hq, mp)
    torch.cuda.synchronize(dev)
    ms, iso = graph_step_bench(torch, dev, cache, n_layers, knew, vnew, q_all, pt, after, o_all,
                               ws, steps, warmup)
    # the split-K partials of the ticket merge: (workspace - tickets) floats
    partial_floats = (ws.numel() - (hkv * 4 + 255) // 256 * 256) // 4
    per = step_bytes_layer(bits[0], 1, ctx, hq, d, window=r, partial_floats=partial_floats)
    sb = per * n_layers
    del cache
    return {"workload": f"long context: 1 sequence x {ctx} tokens, {hq} q / {hkv} KV heads, "
                        f"head_dim {d}, K{w.k_bits}V{w.v_bits}, Hadamard {w.had_block}, "
                        f"{r}-token bf16 window, {n_layers} layer caches",
            "step": "per layer: kvq_decode_step (ticket merge over the splits)",
            "ms_per_step": round(ms, 4), "GB_per_step": round(sb / 1e9, 4),
            "roofline": _roofline(sb, ms, n_layers, iso, per)}


def logquant_bench(kvq, torch, dev, n_layers, steps, warmup, w=128) -> dict:
    """LogQuant mode on the long-context shape: one sequence of 131072 tokens,
    32 query / 8 KV heads, head_dim 128, K and V INT2 (the method's 2-bit
    setting) with Hadamard 128, base window W = 128: every token quantized,
    the log-spaced set B (< 3W positions) kept in bf16 in the reserve.  One
    step = one fused decode step per layer over n_layers layer caches."""
    L = LONG_CONTEXT
    hkv, hq, d, ctx = L.hkv, L.hq, L.head_dim, L.ctx
    mp = ctx // 16
    k = kv_tokens(L.seed, 0, 1, ctx, hkv, d, L.k_outliers, L.outlier_lo, L.outlier_hi)
    v = kv_tokens(L.seed, 1, 1, ctx, hkv, d, L.v_outliers, L.outlier_lo, L.outlier_hi)
    kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
    vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
    del k, v
    bits = np.full((n_layers, hkv, 2), 2)
    cache = kvq.Cache(n_layers, hkv, d, L.had_block, bits, mp, max_batch=1, device=dev,
                      overlap=True, logquant_w=w)
    pt = torch.from_numpy(page_table(L.seed, 1, mp)).to(dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    kpre, vpre = kd[:, :ctx - 1].contiguous(), vd[:, :ctx - 1].contiguous()
    for l in range(n_layers):
        cache.append(l, kpre, vpre, pt, zero)
    knew = kd[:, ctx - 1].contiguous().unsqueeze(0).repeat(n_layers, 1, 1, 1).contiguous()
    vnew = vd[:, ctx - 1].contiguous().unsqueeze(0).repeat(n_layers, 1, 1, 1).contiguous()
    del kd, vd, kpre, vpre
    q_all = torch.from_numpy(np.stack([queries(L.seed, l, 1, hq, d, False)
                                       for l in range(n_layers)])).to(dev).to(torch.bfloat16)
    o_all = torch.empty((n_layers, 1, hq, d), dtype=torch.float32, device=dev)
    after = torch.full((1,), ctx, dtype=torch.int32, device=dev)
    ws = cache.workspace(1, hq, mp)
    torch.cuda.synchronize(dev)
    ms, iso = graph_step_bench(torch, dev, cache, n_layers, knew, vnew, q_all, pt, after, o_all,
                               ws, steps, warmup)
    members = len(kvq.kvq_logquant_members(ctx, w))
    partial_floats = (ws.numel() - (hkv * 4 + 255) // 256 * 256) // 4
    per = (step_bytes_layer(bits[0], 1, ctx, hq, d, partial_floats=partial_floats)
           + hkv * members * 2 * 2 * d)            # the members' bf16 K and V rows
    sb = per * n_layers
    del cache
    return {"workload": f"LogQuant: 1 sequence x {ctx} tokens, {hq} q / {hkv} KV heads, "
                        f"head_dim {d}, K2V2, Hadamard {L.had_block}, base window W = {w} "
                        f"({members} full-precision positions), {n_layers} layer caches",
            "step": "per layer: kvq_decode_step (members masked in the quantized splits, "
                    "reserve CTAs attend over their bf16 rows)",
            "ms_per_step": round(ms, 4), "GB_per_step": round(sb / 1e9, 4),
            "roofline": _roofline(sb, ms, n_layers, iso, per)}


def key_channel_bench(kvq, torch, dev, n_layers, steps, warmup) -> dict:
    """Key-per-channel mode on the Llama-3-8B-shaped decode layer: batch 16,
    32 query / 8 KV heads, head_dim 128, context 4096, Hadamard 128, keys
    quantized per channel (one fp16 scale per page, head and channel), values
    token-wise, no window; K4V4 (as the token-wise headline) and K2V2 (the
    2-bit setting of KIVI and LogQuant).  One step = decode attention over
    n_layers distinct layer caches (the append of a step's token is a separate
    launch in this mode; the decode is the kernel measured)."""
    w = LLAMA3_8B_LAYER
    hkv, hq, d, bsz, ctx = w.hkv, w.hq, w.head_dim, w.batch, w.ctx
    mp = ctx // 16
    variants = []
    for kb, vb in ((4, 4), (2, 2)):
        bits = np.tile(np.array([kb, vb]), (n_layers, hkv, 1))
        cache = kvq.Cache(n_layers, hkv, d, w.had_block, bits, bsz * mp, max_batch=bsz,
                          device=dev, overlap=True, key_per_channel=True)
        pt = torch.from_numpy(page_table(w.seed, bsz, mp)).to(dev)
        zero = torch.zeros(bsz, dtype=torch.int32, device=dev)
        for half in range(2):       # the inputs for 8 sequences at a time, shared by the layers
            rows = slice(8 * half, 8 * half + 8)
            k = kv_tokens(w.seed, 0, 8, ctx, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi,
                          seq0=8 * half)
            v = kv_tokens(w.seed, 1, 8, ctx, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi,
                          seq0=8 * half)
            kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
            vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
            del k, v
            for l in range(n_layers):
                cache.append(l, kd, vd, pt[rows].contiguous(), zero[rows].contiguous(),
                             window_row=8 * half)
            del kd, vd
        q_all = torch.from_numpy(np.stack([queries(w.seed, l, bsz, hq, d, False)
                                           for l in range(n_layers)])).to(dev).to(torch.bfloat16)
        o_all = torch.empty((n_layers, bsz, hq, d), dtype=torch.float32, device=dev)
        lens = torch.full((bsz,), ctx, dtype=torch.int32, device=dev)
        ws = cache.workspace(bsz, hq, mp)
        torch.cuda.synchronize(dev)
        ms, iso = graph_step_bench(torch, dev, cache, n_layers, None, None, q_all, pt, lens, o_all,
                                   ws, steps, warmup, decode_only=True)
        seg = cache.page_bytes[0] // hkv                 # one (page, head) segment
        per = bsz * mp * hkv * seg + bsz * hq * d * (2 + 4) + bsz * mp * 4
        sb = per * n_layers
        variants.append({"bits": f"K{kb} per channel / V{vb}", "bytes_per_token_head": seg // 16,
                         "ms_per_step": round(ms, 4), "GB_per_step": round(sb / 1e9, 4),
                         "roofline": _roofline(sb, ms, n_layers, iso, per)})
        del cache, ws, q_all, o_all
        torch.cuda.synchronize(dev)
    return {"workload": f"key-per-channel: batch {bsz} x {ctx} tokens, {hq} q / {hkv} KV heads, "
                        f"head_dim {d}, Hadamard {w.had_block}, {n_layers} layer caches",
            "step": "per layer: kvq_decode_attn (cluster merge; the last split attends to "
                    "the open page's bf16 rows)",
            "variants": variants}


def _exact_attention_torch(torch, q, k, v, scale):
    """softmax(q k^T scale) v in float64 on the device for one KV head:
    q [G, d], k/v [T, d] (bf16 values)."""
    s = (q.double() @ k.double().T) * scale
    return torch.softmax(s, dim=-1) @ v.double()


def quant_error_report(kvq, torch, dev) -> dict:
    """Error of the decode output over the quantized cache against attention
    over the original bf16 K/V (float64, computed with torch on the device),
    with the configuration's Hadamard block and with no rotation (block 1):
    max / mean absolute difference, relative L2 and the L1 output perturbation
    per query row (CriticalKV technical summary, Methodology)."""
    out = {}
    cases = [(TINY, 1, TINY.ctx, None), (LLAMA3_8B_LAYER, 2, LLAMA3_8B_LAYER.ctx, None),
             (LONG_CONTEXT, 1, LONG_CONTEXT.ctx, [0, 3, 6])]
    for w, bsz, n, heads in cases:
        k = kv_tokens(w.seed, 0, bsz, n, w.hkv, w.head_dim, w.k_outliers, w.outlier_lo,
                      w.outlier_hi)
        v = kv_tokens(w.seed, 1, bsz, n, w.hkv, w.head_dim, w.v_outliers, w.outlier_lo,
                      w.outlier_hi)
        qn = queries(w.seed, 0, bsz, w.hq, w.head_dim, w.q_fp32)
        kd = torch.from_numpy(k).to(dev).to(torch.bfloat16)
        vd = torch.from_numpy(v).to(dev).to(torch.bfloat16)
        del k, v
        q = torch.from_numpy(qn).to(dev)
        if not w.q_fp32:
            q = q.to(torch.bfloat16)
        mp = n // 16
        pt = torch.from_numpy(page_table(w.seed, bsz, mp)).to(dev)
        lens = torch.full((bsz,), n, dtype=torch.int32, device=dev)
        g = w.hq // w.hkv
        scale = 1.0 / np.sqrt(w.head_dim)
        hs = heads if heads is not None else list(range(w.hkv))
        ref = torch.stack([torch.stack([_exact_attention_torch(
            torch, q[b, h * g:(h + 1) * g], kd[b, :, h], vd[b, :, h], scale) for h in hs])
            for b in range(bsz)])
        bits = np.tile(np.array([w.k_bits, w.v_bits]), (1, w.hkv, 1))
        res = {}
        for block in (w.had_block, 1):
            c = kvq.Cache(1, w.hkv, w.head_dim, block, bits, bsz * mp, window=w.window,
                          max_batch=bsz, device=dev)
            c.append(0, kd, vd, pt, torch.zeros(bsz, dtype=torch.int32, device=dev))
            o = c.decode(0, q, pt, lens)
            torch.cuda.synchronize(dev)
            assert c.get_status() == 0
            got = torch.stack([torch.stack([o[b, h * g:(h + 1) * g].double() for h in hs])
                               for b in range(bsz)])
            diff = (got - ref)
            rows = diff.shape[0] * diff.shape[1] * diff.shape[2]
            res[f"block_{block}"] = {
                "max_abs": round(float(diff.abs().max()), 6),
                "mean_abs": round(float(diff.abs().mean()), 6),
                "rel_l2": round(float(diff.norm() / ref.norm()), 6),
                "l1_per_row": round(float(diff.abs().sum()) / rows, 4)}
            del c
        out[w.name] = {"bits": f"K{w.k_bits}V{w.v_bits}", "rows": f"{bsz} seqs x heads {hs}",
                       **res}
        del kd, vd
    return {"reference": "float64 attention over the original bf16 K/V (torch, on the device)",
            "configs": out}


def run_section(args) -> None:
    """One configuration section alone on one GPU, over --layers layer caches."""
    import torch
    import quantized_decode_attention_diag_b300 as kvq
    from quantized_decode_attention_diag_b300 import build
    build.build()
    dev = torch.device("cuda", 0)
    if args.only == "mixed":
        n = N_LAYERS * MIXED_32L.hkv * 2
        out = mixed_bits_bench(kvq, torch, dev, np.ones(n), np.full(n, 4.0), args.steps,
                               args.warmup, n_layers=N_LAYERS)
    elif args.only == "long":
        out = long_context_bench(kvq, torch, dev, N_LAYERS, args.steps, args.warmup)
    elif args.only == "append":
        out = append_sweep(kvq, torch, dev)
    elif args.only == "logquant":
        out = logquant_bench(kvq, torch, dev, N_LAYERS, args.steps, args.warmup)
    else:
        out = key_channel_bench(kvq, torch, dev, N_LAYERS, args.steps, args.warmup)
    print(json.dumps({"section": args.only, **out}), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-append", action="store_true")
    ap.add_argument("--skip-configs", action="store_true",
                    help="leave out the mixed-bits, long-context and quantization-error sections")
    ap.add_argument("--only", default="all",
                    choices=["all", "append", "mixed", "long", "logquant", "key_channel"],
                    help="run one section alone and print it (profiling a small case)")
    ap.add_argument("--layers", type=int, default=32,
                    help="distinct layer caches per step (profiling uses a small case)")
    args = ap.parse_args()
    global N_LAYERS
    N_LAYERS = args.layers
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only != "all":
        run_section(args)
    else:
        run_kvq(args)


if __name__ == "__main__":
    main()
