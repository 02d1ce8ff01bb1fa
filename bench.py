"""Benchmark of the NVFP4 paged-KV decode step on GB300.

A step is one pass of the hot path over one batch: the newest token of every
sequence is quantised into the NVFP4 cache and one query token per sequence
attends over the whole cache (nvfp4kv_append_paged_decode: the fused
append + split-KV attention kernel, then the merge kernel).  value =
KV-tokens attended per second per layer (sum of sequence lengths / step
time), summed over ranks.  The headline workload defaults to the largest that
runs on one GPU (160K context, batch 15); the same step over the FP8-E4M3
comparison cache is timed beside it, every other decode workload gets a row
of its own, and the step's achieved HBM bandwidth is reported against the
measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own copy of the workload (its own
sequences; no collective on the data path) and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "NVFP4 paged decode KV-tokens/s per layer and achieved HBM GB/s vs GB300 peak"
UNIT = "KV-tokens/s"
WORKLOADS = {
    "llama70b_b12": ("llama70b", 12),
    "llama70b_b21": ("llama70b", 21),
    "ctx32k_b44": ("ctx32k", 44),
    "ctx32k_b70": ("ctx32k", 70),
    "ctx160k_b10": ("ctx160k", 10),
    "ctx160k_b15": ("ctx160k", 15),
    "ctx1m_b1": ("ctx1m", 1),
    "ctx1m_b2": ("ctx1m", 2),
}
NVFP4_BYTES_PER_TOKEN_HEAD = 2 * (64 + 8)        # K and V: packed data + scales
FP8_BYTES_PER_TOKEN_HEAD = 2 * 128


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="ctx160k_b15", choices=sorted(WORKLOADS),
                    help="the headline workload (default: the largest single-GPU one)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--num-workers", type=int, default=0)
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="untimed load before the timed region so clock samples see load clocks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the quantize / prefix-dequant rows")
    ap.add_argument("--no-decode-rows", action="store_true",
                    help="skip the decode rows of the other workloads")
    ap.add_argument("--row-only", default=None,
                    choices=["ext160k", "ext8k_c2k", "ext160k_e4m3", "ext8k_c2k_e4m3", "quantize8k", "prefix160k",
                             "prefill8k"],
                    help="time only this row (extend attention on a workload, quantize_append of 8,192 "
                         "bf16 tokens, dequant_prefix_fp8 of a 163,840-token prefix, or FP8 initial prefill "
                         "of 8,192 tokens) and print it")
    a = ap.parse_args()
    a.warmup = max(3, a.warmup)
    a.steps = max(1, a.steps)
    return a


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return None


# the sources each profiled kernel is compiled from (a summary's counters are
# used only while the hash of these files matches the one it records)
KERNEL_SOURCES = {
    "decode_nvfp4": ["abi.cpp", "decode_common.cuh", "decode_nvfp4.cu", "device_common.cuh", "merge.cu",
                     "nvfp4kv_internal.h", "record_write.cuh"],
    "extend_attention": ["abi.cpp", "device_common.cuh", "extend_attention.cu", "nvfp4kv_internal.h",
                         "record_write.cuh", "tcgen05.cuh"],
    "quantize_append": ["abi.cpp", "device_common.cuh", "nvfp4kv_internal.h", "quantize_append.cu",
                        "record_write.cuh"],
    "dequant_prefix": ["abi.cpp", "dequant_prefix.cu", "device_common.cuh", "nvfp4kv_internal.h"],
}


def kernel_sources_hash(kernel_tag: str) -> str:
    import hashlib
    csrc = os.path.join(ROOT, "nvfp4_quantized_paged_nvfp4kv_gb300", "csrc")
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel_tag]:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current sources of that kernel (the summary records their hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            v = v.strip()
            if v.startswith("`") and "`" in v[1:]:
                v = v[1:v.index("`", 1)]             # the quoted value, without a trailing note
            fields[k.strip()] = v
    if fields.get("kernel_sources_sha256") != kernel_sources_hash(kernel_tag):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is loaded."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm

def fill_caches(w, bt, num_pages, dev, fmts):
    """Caches of workload w in each format of fmts ("nvfp4", "fp8"), filled by the
    library's own quantize_append from the seeded bf16 K/V rows (each chunk of
    rows generated once and written into every format)."""
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    caches = {}
    for f in fmts:
        if f == "nvfp4":
            caches[f] = nv.NVFP4Cache.allocate(num_pages, w.num_kv_heads, device=dev, zero=False)
        else:
            caches[f] = nv.FP8Cache.allocate(num_pages, w.num_kv_heads, device=dev, zero=False)
    app = {"nvfp4": nv.nvfp4kv_quantize_append, "fp8": nv.fp8kv_quantize_append}
    for b, L in enumerate(w.seq_lens):
        for t0 in range(0, L, workloads.CHUNK):
            t1 = min(L, t0 + workloads.CHUNK)
            sm = torch.from_numpy(workloads.slot_mapping(w, bt, b, t0, t1)).to(dev)
            k = workloads.kv_rows(w, "k", b, t0, t1, device=dev).to(torch.bfloat16)
            v = workloads.kv_rows(w, "v", b, t0, t1, device=dev).to(torch.bfloat16)
            for f in fmts:
                app[f](caches[f], k, v, sm)
    return caches


def replicas_for(w, bytes_per_token_head, l2):
    """Cache copies rotated between steps so that no step finds its pages in
    L2: enough to cover 3x L2 when one cache is smaller than 4x L2."""
    one = w.total_tokens * w.num_kv_heads * bytes_per_token_head
    return max(2, math.ceil(3 * l2 / max(1, one)) + 1) if one < 4 * l2 else 1


class DecodeSetup:
    """Cache replicas (rotated to defeat L2), tables, queries and the new token."""

    def __init__(self, w, fmt: str, dev, replicas: int, num_workers: int, first=None, tables=None):
        import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
        self.nv, self.w, self.fmt, self.dev = nv, w, fmt, dev
        bt, num_pages = workloads.block_table(w) if tables is None else tables
        self.num_pages = num_pages
        self.bt = torch.from_numpy(bt).to(dev)
        self.sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
        if first is None:
            first = fill_caches(w, bt, num_pages, dev, [fmt])[fmt]
        self.caches = [first] + [self._clone(first) for _ in range(replicas - 1)]
        self.q = workloads.query(w, device=dev)
        self.out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
        self.num_workers = num_workers
        self.ws = nv.new_workspace(num_workers, device=dev)
        # newest token of every sequence: its slot and fresh K/V rows
        last = np.array([workloads.slot_mapping(w, bt, b, L - 1, L)[0] for b, L in enumerate(w.seq_lens)],
                        np.int32)
        self.new_slots = torch.from_numpy(last).to(dev)
        self.k_new, self.v_new = workloads.new_tokens(w, w.batch, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def _clone(self, c):
        return type(c)(c.pool.clone())

    def cache_bytes(self):
        return self.caches[0].nbytes()

    def append(self, i, k=None, v=None, slots=None):
        nv = self.nv
        c = self.caches[i % len(self.caches)]
        fn = nv.nvfp4kv_quantize_append if self.fmt == "nvfp4" else nv.fp8kv_quantize_append
        fn(c, self.k_new if k is None else k, self.v_new if v is None else v,
           self.new_slots if slots is None else slots, self.status)

    def decode(self, i, q=None, sl=None):
        nv = self.nv
        c = self.caches[i % len(self.caches)]
        fn = nv.nvfp4kv_paged_decode if self.fmt == "nvfp4" else nv.fp8kv_paged_decode
        fn(c, self.q if q is None else q, self.bt, self.sl if sl is None else sl, self.out, self.ws,
           num_workers=self.num_workers, dev_status=self.status)

    def step(self, i, q=None, k=None, v=None, sl=None):
        """quantize the newest token of every sequence and decode, one fused call"""
        nv = self.nv
        c = self.caches[i % len(self.caches)]
        fn = nv.nvfp4kv_append_paged_decode if self.fmt == "nvfp4" else nv.fp8kv_append_paged_decode
        fn(c, self.k_new if k is None else k, self.v_new if v is None else v, self.q if q is None else q,
           self.bt, self.sl if sl is None else sl, self.out, self.ws, num_workers=self.num_workers,
           dev_status=self.status)


def time_steps(setup: DecodeSetup, steps: int, warmup: int, world: int):
    """Device time of `steps` back-to-back steps (barrier + synchronize on both
    sides), on the launching stream, and the mean device time of one decode
    call (the timed region over the number of calls).  No event sits between
    the steps: an event between two kernels would stop the next one from
    starting its prologue while the previous drains, as it does in a serving
    loop."""
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        setup.step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        setup.step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    return total_ms, total_ms / steps


def time_e2e(setup: DecodeSetup, steps: int, world: int):
    """Same step through the public API with the step's inputs in pinned host
    memory: every step copies its queries, new K/V rows and lengths host to
    device (one copy of one packed buffer) and its output back; all copies are
    inside the timed region.  A serving loop would not pay a host launch per
    call: each step is one CUDA graph (captured once per input slot) that
    decodes from one device slot while, on a second stream, it copies the next
    step's inputs into the other slot and reads the previous step's output
    back."""
    parts = [setup.q, setup.k_new, setup.v_new, setup.sl]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in sizes:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    host_in = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, sizes):
        host_in[o:o + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
    dev_in = [torch.empty(offs[-1], dtype=torch.uint8, device=setup.dev) for _ in range(2)]
    dev_views = [[b[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, sizes)]
                 for b in dev_in]
    outs = [torch.empty_like(setup.out) for _ in range(2)]
    host_out = [torch.empty(setup.out.shape, dtype=setup.out.dtype).pin_memory() for _ in range(2)]
    h2d, d2h = sum(sizes), host_out[0].numel() * host_out[0].element_size()
    out_saved = setup.out
    side = torch.cuda.Stream(device=setup.dev)

    def body(s, i):
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            dev_in[1 - s].copy_(host_in, non_blocking=True)      # the next step's inputs
            host_out[1 - s].copy_(outs[1 - s], non_blocking=True)  # the previous step's output
        setup.out = outs[s]
        q, k, v, sl = dev_views[s]
        setup.step(i, q, k, v, sl)
        main.wait_stream(side)

    # warm up both slots eagerly, then capture one graph per slot
    dev_in[0].copy_(host_in)
    for i in range(4):
        body(i % 2, i)
    torch.cuda.synchronize()
    graphs = []
    for s in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body(s, s)
        graphs.append(g)
    dev_in[0].copy_(host_in)
    for i in range(4):
        graphs[i % 2].replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    dev_in[0].copy_(host_in, non_blocking=True)                  # step 0's inputs
    for i in range(steps):
        graphs[i % 2].replay()
    last = (steps - 1) % 2
    host_out[last].copy_(outs[last], non_blocking=True)         # the last step's output
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    setup.out = out_saved
    return t0.elapsed_time(t1), h2d, d2h


def decode_alg_bytes(w, bytes_per_token_head: int) -> int:
    """Algorithmic bytes of one step: the K/V bytes of every cached token read
    once, the queries and outputs (bf16), the block table and lengths, and the
    new token's fp32 K/V rows."""
    return (w.total_tokens * w.num_kv_heads * bytes_per_token_head
            + 2 * w.batch * w.num_q_heads * w.head_dim * 2
            + w.batch * w.max_pages * 4 + w.batch * 4
            + w.batch * w.num_kv_heads * w.head_dim * 2 * 4)


def hbm_peak():
    hbm = (measured_peaks() or {}).get("hbm_gbs")
    return (hbm, "measured") if hbm is not None else (6800.0, "fallback")


def decode_row(name: str, dev, steps: int, warmup: int, num_workers: int, world: int = 1):
    """One decode workload: the fused append + decode step over the NVFP4 cache
    and over the FP8 cache at the same batch, timed as the headline is."""
    wname, batch = WORKLOADS[name]
    w = workloads.make(wname, batch=batch)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    bt, num_pages = workloads.block_table(w)
    caches = fill_caches(w, bt, num_pages, dev, ["nvfp4", "fp8"])
    hbm, _ = hbm_peak()
    row = {"batch": w.batch, "kv_tokens_per_step": w.total_tokens}
    for fmt, bpt in (("nvfp4", NVFP4_BYTES_PER_TOKEN_HEAD), ("fp8", FP8_BYTES_PER_TOKEN_HEAD)):
        setup = DecodeSetup(w, fmt, dev, replicas_for(w, bpt, l2), num_workers, first=caches.pop(fmt),
                            tables=(bt, num_pages))
        total_ms, ms = time_steps(setup, steps, warmup, world)
        alg = decode_alg_bytes(w, bpt)
        gbs = alg / (ms / 1e3) / 1e9
        row[fmt] = {"us": ms * 1e3, "kv_tokens_per_s": w.total_tokens / (ms / 1e3), "alg_bytes": alg,
                    "alg_gbs": gbs, "frac_of_measured": gbs / hbm, "frac_of_8tbs": gbs / 8000.0,
                    "device_status": int(setup.status.item())}
        del setup
        torch.cuda.empty_cache()
    row["nvfp4_over_fp8"] = row["nvfp4"]["kv_tokens_per_s"] / row["fp8"]["kv_tokens_per_s"]
    return row


def run_ours(args, world, rank, local):
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    nv.load()
    dev = torch.device("cuda", local)
    name, batch = WORKLOADS[args.workload]
    w = workloads.make(name, batch=batch)
    tokens = w.total_tokens
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    replicas = replicas_for(w, NVFP4_BYTES_PER_TOKEN_HEAD, l2)
    bt, num_pages = workloads.block_table(w)
    fmts = ["nvfp4"] if args.no_fp8 else ["nvfp4", "fp8"]
    caches = fill_caches(w, bt, num_pages, dev, fmts)
    setup = DecodeSetup(w, "nvfp4", dev, replicas, args.num_workers, first=caches.pop("nvfp4"),
                        tables=(bt, num_pages))
    sampler = ClockSampler(local)
    sampler.start()
    # soak: keep the GPU loaded for ~1 s so the clock samples see load clocks
    t_end = time.time() + args.soak_seconds
    i = 0
    while time.time() < t_end:
        setup.step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    total_ms, dec_ms = time_steps(setup, args.steps, args.warmup, world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = tokens * world / (ms_per_step / 1e3)
    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(setup, args.steps, world)
        e2e_ms = max_over_ranks(e2e_ms, world)
        e2e = {"value": tokens * world / (e2e_ms / args.steps / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    st = int(setup.status.item())
    hbm, peak_src = hbm_peak()
    alg_bytes = decode_alg_bytes(w, NVFP4_BYTES_PER_TOKEN_HEAD)
    achieved = alg_bytes / (dec_ms / 1e3) / 1e9
    traffic = profiled_traffic("decode_nvfp4", args.workload)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "dtype_detail": "NVFP4 cache (E2M1 codes, E4M3 block scales) dequantised to f16 MMA operands, "
                        "f32 accumulation and softmax",
        "data": "synthetic (seeded generators; shapes and distributions of the workload, no real weights)",
        "config": {"workload": args.workload, "batch": w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                   "seq_len": (w.seq_lens[0] if len(set(w.seq_lens)) == 1 else "ragged"),
                   "kv_tokens_per_step": tokens,
                   "l2": (f"{replicas} rotating cache replicas of {setup.cache_bytes() / 1e6:.1f} MB "
                          f"(L2 {l2 / 1e6:.0f} MB)") if replicas > 1 else
                         f"cache {setup.cache_bytes() / 1e6:.1f} MB > 4x L2",
                   "parallelism": f"replicas x{world} (each rank its own sequences)",
                   "step": "append_paged_decode: newest token per sequence quantised into the cache, "
                           "then split-KV decode + merge (2 kernels)"},
        "roofline": {"bound": "hbm", "kernel": "nvfp4 append + paged decode (split-KV attention + merge)",
                     "achieved": achieved, "peak": hbm, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / hbm, "frac_of_8tbs_nominal": achieved / 8000.0,
                     "alg_bytes_per_launch": alg_bytes, "decode_ms": dec_ms, "traffic": traffic,
                     "traffic_over_alg": (traffic / alg_bytes) if traffic else None},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "device_status": st,
    }
    del setup
    torch.cuda.empty_cache()
    if not args.no_fp8:
        fs = DecodeSetup(w, "fp8", dev, replicas_for(w, FP8_BYTES_PER_TOKEN_HEAD, l2), args.num_workers,
                         first=caches.pop("fp8"), tables=(bt, num_pages))
        f_total, f_dec = time_steps(fs, args.steps, args.warmup, world)
        f_total = max_over_ranks(f_total, world)
        f_value = tokens * world / (f_total / args.steps / 1e3)
        f_bytes = decode_alg_bytes(w, FP8_BYTES_PER_TOKEN_HEAD)
        result["fp8_comparison"] = {
            "value": f_value, "unit": UNIT, "ms_per_step": f_total / args.steps, "decode_ms": f_dec,
            "achieved_gbs": f_bytes / (f_dec / 1e3) / 1e9,
            "nvfp4_over_fp8_step": value / f_value, "nvfp4_over_fp8_decode": f_dec / dec_ms}
        del fs
        torch.cuda.empty_cache()
    rows = {}
    if not args.no_decode_rows and world == 1:
        head = {"batch": w.batch, "kv_tokens_per_step": tokens,
                "nvfp4": {"us": dec_ms * 1e3, "kv_tokens_per_s": tokens / (dec_ms / 1e3), "alg_bytes": alg_bytes,
                          "alg_gbs": achieved, "frac_of_measured": achieved / hbm,
                          "frac_of_8tbs": achieved / 8000.0, "device_status": st}}
        if "fp8_comparison" in result:
            fc = result["fp8_comparison"]
            head["fp8"] = {"us": fc["decode_ms"] * 1e3, "kv_tokens_per_s": tokens / (fc["decode_ms"] / 1e3),
                           "alg_gbs": fc["achieved_gbs"], "frac_of_measured": fc["achieved_gbs"] / hbm,
                           "frac_of_8tbs": fc["achieved_gbs"] / 8000.0}
            head["nvfp4_over_fp8"] = fc["nvfp4_over_fp8_decode"]
        for other in WORKLOADS:
            rows[other] = head if other == args.workload else decode_row(other, dev, args.steps, args.warmup,
                                                                         args.num_workers)
        rows["timing"] = ("each workload's fused append + decode step, back to back, CUDA events over the "
                          "timed steps; caches smaller than 4x L2 rotated among replicas")
    if not args.no_rows:
        result["other_rows"] = other_rows(dev)
    if rows:
        result.setdefault("other_rows", {})["decode"] = rows
    cpu = (cpu_baseline(args.workload, budget_s=24.0)
           if rank == 0 and world == 1 and not args.no_cpu_baseline else None)
    if cpu is not None:
        result["cpu_baseline"] = cpu
    return result


# Per-call rows time one short launch between two events.  A GPU-side spin of
# this many cycles before the start event keeps the GPU busy while the host
# enqueues the call, so the interval holds the kernel, not the host's launch.
HOST_COVER_CYCLES = 400_000


class L2Flush:
    """Evicts the timed call's inputs from L2 before each timed call: a
    256 MB buffer is written (twice the L2), then a second one is read, so
    that the dirty lines of the write are written back before the timed call
    rather than inside it."""

    def __init__(self, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(32 << 20, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def other_rows(dev):
    """The write side and the extend path on the long-context workload: quantize_append
    of one 8192-token bf16 prefill chunk (Hkv=8) and dequant_prefix_fp8 of a
    163840-token prefix, each timed with CUDA events (mean of 20 after 3 warm-ups)."""
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    w = workloads.make("ctx160k", batch=1)
    bt, num_pages = workloads.block_table(w)
    cache = nv.NVFP4Cache.allocate(num_pages, w.num_kv_heads, device=dev, zero=False)
    bt_d = torch.from_numpy(bt).to(dev)
    for t0 in range(0, w.seq_lens[0], workloads.CHUNK):
        t1 = min(w.seq_lens[0], t0 + workloads.CHUNK)
        sm = torch.from_numpy(workloads.slot_mapping(w, bt, 0, t0, t1)).to(dev)
        nv.nvfp4kv_quantize_append(cache, workloads.kv_rows(w, "k", 0, t0, t1, device=dev).to(torch.bfloat16),
                                   workloads.kv_rows(w, "v", 0, t0, t1, device=dev).to(torch.bfloat16), sm)
    T = 8192
    k = workloads.kv_rows(w, "k", 0, 0, T, device=dev).to(torch.bfloat16)
    v = workloads.kv_rows(w, "v", 0, 0, T, device=dev).to(torch.bfloat16)
    sm = torch.from_numpy(workloads.slot_mapping(w, bt, 0, 0, T)).to(dev)
    L = w.seq_lens[0]
    kf = torch.empty((L, w.num_kv_heads, 128), dtype=torch.uint8, device=dev)
    vf = torch.empty_like(kf)
    pl = torch.tensor([L], dtype=torch.int32, device=dev)
    ip = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(20):
            flush()                                          # evict the inputs from L2
            torch.cuda._sleep(HOST_COVER_CYCLES)             # the GPU waits here, not on the host launch
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.mean(ms)

    # Back to back, as in a prefill loop over layers: the mean of n calls
    # between two events (a single short call's event interval is quantised
    # to ~2 us on this GPU).  Each quantize call reads its own copy of the
    # 8K-token rows and writes its own cache (as each layer has its own),
    # rotated among enough copies that none is still in L2 when it comes round.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(2, math.ceil(3 * l2 / (2 * k.numel() * k.element_size())) + 1)
    kv_copies = [(k.clone(), v.clone()) for _ in range(copies)]
    pools = [nv.NVFP4Cache.allocate(num_pages, w.num_kv_heads, device=dev, zero=False) for _ in range(copies)]

    def back_to_back(call, n=2 * copies, passes=5):
        """median over `passes` passes of the mean of n calls between two events"""
        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        means = []
        for _ in range(passes):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(n):
                call(i)
            b.record()
            torch.cuda.synchronize()
            means.append(a.elapsed_time(b) / n)
        return statistics.median(means)

    def quantize_into(g=1.0, factors=None):
        cs = [nv.NVFP4Cache(c.pool, global_scale=g, head_scales=factors) for c in pools]
        return lambda i: nv.nvfp4kv_quantize_append(cs[i % copies], kv_copies[i % copies][0],
                                                    kv_copies[i % copies][1], sm)

    q_ms = back_to_back(quantize_into())
    q_bytes = T * w.num_kv_heads * (2 * 128 * 2 + NVFP4_BYTES_PER_TOKEN_HEAD) + T * 4
    p_ms = back_to_back(lambda i: nv.nvfp4kv_dequant_prefix_fp8(cache, bt_d, pl, ip, kf, vf), n=10)
    p_bytes = L * w.num_kv_heads * (NVFP4_BYTES_PER_TOKEN_HEAD + 2 * 128)
    # the same cache read as one with a calibrated tensor scale G = 0.37: the
    # decode of the 160K sequence and the quantise path cost what G = 1 costs
    cache_g = nv.NVFP4Cache(cache.pool, global_scale=0.37)
    q = workloads.query(w, device=dev)
    sl = torch.tensor([L], dtype=torch.int32, device=dev)
    out = torch.empty((1, w.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
    ws = nv.new_workspace(device=dev)
    d1_ms = back_to_back(lambda i: nv.nvfp4kv_paged_decode(cache, q, bt_d, sl, out, ws), n=20)
    dg_ms = back_to_back(lambda i: nv.nvfp4kv_paged_decode(cache_g, q, bt_d, sl, out, ws), n=20)
    qg_ms = back_to_back(quantize_into(0.37))
    # and with per-head factors on top (K and V of each kv head their own scale)
    factors = [[0.5 + 0.25 * h for h in range(w.num_kv_heads)], [2.0 - 0.2 * h for h in range(w.num_kv_heads)]]
    cache_h = nv.NVFP4Cache(cache.pool, global_scale=0.37, head_scales=factors)
    dh_ms = back_to_back(lambda i: nv.nvfp4kv_paged_decode(cache_h, q, bt_d, sl, out, ws), n=20)
    qh_ms = back_to_back(quantize_into(0.37, factors))
    del kv_copies, pools
    d_bytes = L * w.num_kv_heads * NVFP4_BYTES_PER_TOKEN_HEAD
    multi = multi_query_rows(dev, timed)
    extend = extend_rows(dev)
    extend8 = extend_rows(dev, chunk="e4m3")
    prefill = prefill_rows(dev)
    return {
        "quantize_append_8k_bf16": {"us": q_ms * 1e3, "tokens_per_s": T / (q_ms / 1e3),
                                    "alg_gbs": q_bytes / (q_ms / 1e3) / 1e9, "alg_bytes": q_bytes,
                                    "traffic": profiled_traffic("quantize_append", "nvfp4_8k_bf16")},
        "dequant_prefix_fp8_160k": {"us": p_ms * 1e3, "tokens_per_s": L / (p_ms / 1e3),
                                    "alg_gbs": p_bytes / (p_ms / 1e3) / 1e9, "alg_bytes": p_bytes,
                                    "traffic": profiled_traffic("dequant_prefix", "fp8_160k")},
        "tensor_scale_0.37": {"decode_160k_b1_us": dg_ms * 1e3, "decode_160k_b1_unit_scale_us": d1_ms * 1e3,
                              "decode_alg_gbs": d_bytes / (dg_ms / 1e3) / 1e9,
                              "quantize_append_8k_bf16_us": qg_ms * 1e3,
                              "per_head_factors": {"decode_160k_b1_us": dh_ms * 1e3,
                                                   "quantize_append_8k_bf16_us": qh_ms * 1e3}},
        "multi_query": multi,
        "extend_160k_chunk8k": extend,
        "extend_160k_chunk8k_e4m3": extend8,
        "prefill_fp8_8k": prefill,
        "timing": "quantize, prefix and 160K decode rows: calls back to back between two CUDA events (the "
                  "median of five such passes), each "
                  "quantize call with its own copy of the inputs and its own cache, rotated among copies "
                  "totalling over 3x L2 (the other inputs exceed L2); "
                  "multi-query rows: one call per event pair after a 256 MB write and a 256 MB read (L2 "
                  "evicted) and a GPU spin covering the host launch",
    }


def write_side_row(dev, name: str, steps: int, warmup: int):
    """One write-side row alone: quantize_append of 8,192 bf16 tokens (Hkv 8)
    into a 163,840-token cache, or dequant_prefix_fp8 of that 163,840-token
    prefix; CUDA events per call, L2 evicted before each call (L2Flush)."""
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    w = workloads.make("ctx160k", batch=1)
    bt, num_pages = workloads.block_table(w)
    cache = nv.NVFP4Cache.allocate(num_pages, w.num_kv_heads, device=dev, zero=False)
    L = w.seq_lens[0]
    flush = L2Flush(dev)
    if name == "quantize8k":
        T = 8192
        k = workloads.kv_rows(w, "k", 0, 0, T, device=dev).to(torch.bfloat16)
        v = workloads.kv_rows(w, "v", 0, 0, T, device=dev).to(torch.bfloat16)
        sm = torch.from_numpy(workloads.slot_mapping(w, bt, 0, 0, T)).to(dev)
        fn = lambda: nv.nvfp4kv_quantize_append(cache, k, v, sm)  # noqa: E731
        alg, units = T * w.num_kv_heads * (2 * 128 * 2 + NVFP4_BYTES_PER_TOKEN_HEAD) + T * 4, T
    else:
        for t0 in range(0, L, workloads.CHUNK):
            t1 = min(L, t0 + workloads.CHUNK)
            sm = torch.from_numpy(workloads.slot_mapping(w, bt, 0, t0, t1)).to(dev)
            nv.nvfp4kv_quantize_append(cache, workloads.kv_rows(w, "k", 0, t0, t1, device=dev),
                                       workloads.kv_rows(w, "v", 0, t0, t1, device=dev), sm)
        bt_d = torch.from_numpy(bt).to(dev)
        kf = torch.empty((L, w.num_kv_heads, 128), dtype=torch.uint8, device=dev)
        vf = torch.empty_like(kf)
        pl = torch.tensor([L], dtype=torch.int32, device=dev)
        ip = torch.zeros(1, dtype=torch.int32, device=dev)
        fn = lambda: nv.nvfp4kv_dequant_prefix_fp8(cache, bt_d, pl, ip, kf, vf)  # noqa: E731
        alg, units = L * w.num_kv_heads * (NVFP4_BYTES_PER_TOKEN_HEAD + 2 * 128), L
    for _ in range(warmup):
        fn()
    ms = []
    for _ in range(steps):
        flush()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    t = statistics.mean(ms)
    hbm = (measured_peaks() or {}).get("hbm_gbs", 6800.0)
    return {"row": name, "us": t * 1e3, "tokens_per_s": units / (t / 1e3), "alg_bytes": alg,
            "alg_gbs": alg / (t / 1e3) / 1e9, "frac": alg / (t / 1e3) / 1e9 / hbm, "peak_gbs": hbm}


def extend_flops(e) -> float:
    """Algorithmic FLOPs of extend attention: 2 d for q.k and 2 d for p.v per
    (chunk token, query head, visible key); token t sees P + t + 1 keys."""
    tot = 0
    for P, C in zip(e.prefix_lens, e.chunk_lens):
        tot += C * P + C * (C + 1) // 2
    return 4.0 * e.head_dim * e.num_q_heads * tot


def extend_rows(dev, name: str = "ext160k", steps: int = 5, warmup: int = 3, compare_fused: bool = True,
                chunk: str = "bf16"):
    """Extend attention of the last 8,192-token chunk of a 163,840-token
    prefill (Hq 48, Hkv 8) over the 155,648-row FP8 prefix workspace (319 MB,
    larger than L2) and the chunk (bf16, or E4M3 as the pages' FP8 prefill
    has it), bf16 out; mean of `steps` launches after `warmup`, CUDA events on
    the launching stream.  Then the same step fused with the NVFP4 write of
    the chunk against attention + quantize_append."""
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    e = workloads.extend_make(name)
    x = workloads.extend_inputs(e, device=dev, chunk=chunk)
    out = torch.empty((e.q_rows, e.num_q_heads, e.head_dim), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mql = max(e.chunk_lens)

    def call():
        nv.nvfp4kv_extend_attention_fp8(x["q"], x["q_indptr"], x["k_prefix"], x["v_prefix"], x["kv_indptr"],
                                        x["prefix_lens"], x["k_chunk"], x["v_chunk"], out, max_q_len=mql,
                                        dev_status=status)
    for _ in range(warmup):
        call()
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    t = statistics.mean(ms)
    flops = extend_flops(e)
    peaks = measured_peaks() or {}
    peak = peaks.get("bf16_tflops")
    src = "measured"
    if peak is None:
        peak, src = 1900.0, "fallback"
    tf = flops / (t / 1e3) / 1e12
    f8 = ("tcgen05.mma M128: Q K^T kind::f8f6f4 (E4M3 key tiles by TMA, Q as two E4M3 terms), P V kind::f16; "
          "fp32 accumulators in tensor memory")
    if chunk == "e4m3":
        mma = f8
    elif e.prefix_rows >= 8 * e.q_rows:        # the library's dispatch: a bf16 chunk behind a long prefix
        mma = f8 + "; the bf16 chunk tiles split into two E4M3 terms by the converter warps"
    else:
        mma = "tcgen05.mma kind::f16 M128 (f16 operands, fp32 accumulators in tensor memory)"
    row = {"workload": name, "chunk": chunk, "us": t * 1e3, "chunk_tokens_per_s": e.q_rows / (t / 1e3),
           "alg_tflops": tf, "alg_flops": flops, "bound": "tensor", "peak_tflops": peak, "peak_source": src,
           "frac": tf / peak, "mma": mma + "; peak: measured bf16 dense burst",
           "traffic": profiled_traffic("extend_attention", name if chunk == "bf16" else name + "_e4m3")}
    if not compare_fused:
        row["device_status"] = int(status.item())
        return row

    # the same step fused with the NVFP4 write of the chunk, against the
    # attention followed by a separate quantize_append
    P = e.prefix_lens[0]
    cache = nv.NVFP4Cache.allocate((P + e.q_rows) // 16 + 1, e.num_kv_heads, device=dev, zero=False)
    slots = torch.arange(P, P + e.q_rows, dtype=torch.int32, device=dev)
    args = (x["q"], x["q_indptr"], x["k_prefix"], x["v_prefix"], x["kv_indptr"], x["prefix_lens"],
            x["k_chunk"], x["v_chunk"], out)

    def fused():
        nv.nvfp4kv_extend_attention_fp8_append(cache, slots, *args, max_q_len=mql, dev_status=status)

    # the separate write quantises the same values (E4M3 codes held exactly in bf16)
    kq, vq = ((x["k_chunk"].view(torch.float8_e4m3fn).to(torch.bfloat16),
               x["v_chunk"].view(torch.float8_e4m3fn).to(torch.bfloat16)) if chunk == "e4m3" else
              (x["k_chunk"], x["v_chunk"]))

    def separate():
        nv.nvfp4kv_extend_attention_fp8(*args, max_q_len=mql, dev_status=status)
        nv.nvfp4kv_quantize_append(cache, kq, vq, slots, status)

    def mean_ms(fn):
        for _ in range(2):
            fn()
        res = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            res.append(a.elapsed_time(b))
        return statistics.mean(res)
    f_ms, s_ms = mean_ms(fused), mean_ms(separate)
    row.update({"fused_append_us": f_ms * 1e3, "attention_then_quantize_append_us": s_ms * 1e3,
                "device_status": int(status.item())})
    return row


def prefill_rows(dev, steps: int = 10, warmup: int = 3):
    """Initial prefill of one 8,192-token prompt (Hq 48, Hkv 8, no prefix) on
    the prompt's FP8 keys and values, attention alone and fused with the NVFP4
    write of the same values, and the same fused step with the K/V in bf16;
    mean of `steps` launches after `warmup`, CUDA events on the launching
    stream."""
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    e = workloads.extend_make("prefill8k")
    C = e.chunk_lens[0]
    out = torch.empty((C, e.num_q_heads, e.head_dim), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cache = nv.NVFP4Cache.allocate(C // 16 + 1, e.num_kv_heads, device=dev, zero=False)
    slots = torch.arange(C, dtype=torch.int32, device=dev)
    flops = extend_flops(e)
    peak = (measured_peaks() or {}).get("bf16_tflops", 1900.0)
    row = {"workload": "prefill8k", "alg_flops": flops, "peak_tflops": peak}
    for chunk in ("e4m3", "bf16"):
        x = workloads.extend_inputs(e, device=dev, chunk=chunk)
        args = (x["q"], x["q_indptr"], x["k_prefix"], x["v_prefix"], x["kv_indptr"], x["prefix_lens"],
                x["k_chunk"], x["v_chunk"], out)
        calls = {"fused_append": lambda: nv.nvfp4kv_extend_attention_fp8_append(cache, slots, *args, max_q_len=C,
                                                                                  dev_status=status)}
        if chunk == "e4m3":
            calls["attention"] = lambda: nv.nvfp4kv_extend_attention_fp8(*args, max_q_len=C, dev_status=status)
        for what, fn in calls.items():
            for _ in range(warmup):
                fn()
            ms = []
            for _ in range(steps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                ms.append(a.elapsed_time(b))
            t = statistics.mean(ms)
            tf = flops / (t / 1e3) / 1e12
            row[f"{chunk}_{what}"] = {"us": t * 1e3, "tokens_per_s": C / (t / 1e3), "alg_tflops": tf,
                                      "frac": tf / peak}
    row["device_status"] = int(status.item())
    return row


def multi_query_rows(dev, timed):
    """Multi-query decode (q_len new tokens per sequence, causal) against q_len
    single-token decodes of the same cache: Llama-3.3-70B layer (group 8, two
    row groups per kv head at q_len 2) and the 32K workload shape with group 4
    (Hq 32, Hkv 8: both tokens' rows share one row group)."""
    import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
    res = {}
    for name, w in (("llama70b_b12_q2", workloads.make("llama70b", batch=12)),
                    ("g4_b12_8k_q2", workloads.custom(12, 32, 8, (8192,) * 12, seed=41))):
        q_len = 2
        bt, num_pages = workloads.block_table(w)
        cache = nv.NVFP4Cache.allocate(num_pages, w.num_kv_heads, device=dev, zero=False)
        for b in range(w.batch):
            for t0 in range(0, w.seq_lens[b], workloads.CHUNK):
                t1 = min(w.seq_lens[b], t0 + workloads.CHUNK)
                sm = torch.from_numpy(workloads.slot_mapping(w, bt, b, t0, t1)).to(dev)
                nv.nvfp4kv_quantize_append(cache, workloads.kv_rows(w, "k", b, t0, t1, device=dev),
                                           workloads.kv_rows(w, "v", b, t0, t1, device=dev), sm)
        bt_d = torch.from_numpy(bt).to(dev)
        sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
        sl_prev = sl - 1
        q2 = torch.randn((w.batch, q_len, w.num_q_heads, 128), device=dev).to(torch.bfloat16)
        q1 = q2[:, 0].contiguous()
        out2 = torch.empty((w.batch, q_len, w.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
        out1 = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
        ws = nv.new_workspace(device=dev)
        m_ms = timed(lambda: nv.nvfp4kv_paged_decode_multi(cache, q2, bt_d, sl, out2, ws))

        def two_singles():
            nv.nvfp4kv_paged_decode(cache, q1, bt_d, sl_prev, out1, ws)
            nv.nvfp4kv_paged_decode(cache, q1, bt_d, sl, out1, ws)
        s_ms = timed(two_singles)
        kv = sum(w.seq_lens) * w.num_kv_heads * NVFP4_BYTES_PER_TOKEN_HEAD
        res[name] = {"us": m_ms * 1e3, "two_single_decodes_us": s_ms * 1e3,
                     "query_tokens_per_s": w.batch * q_len / (m_ms / 1e3),
                     "kv_alg_gbs": kv / (m_ms / 1e3) / 1e9}
        del cache
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# CPU oracle: the baseline line and the reference arm

CPU_SAMPLE_TOKENS = 2048       # tokens of sequence 0 per CPU-baseline pass
REF_SAMPLE_TOKENS = 8192       # tokens of sequence 0 per reference-arm step


def _cpu_sample(w, n_tokens: int):
    """CPU cache of the first n_tokens tokens of sequence 0, every kv head,
    quantised by the oracle, and the sequence's queries (all query heads)."""
    import oracle
    L = min(w.seq_lens[0], n_tokens)
    npg = (L + 15) // 16
    bt = np.arange(npg, dtype=np.int32)[None, :]
    sm = np.arange(L, dtype=np.int32)
    pools = [np.zeros((npg, w.num_kv_heads, 16, s), np.uint8) for s in (64, 8, 64, 8)]
    for t0 in range(0, L, workloads.CHUNK):
        t1 = min(L, t0 + workloads.CHUNK)
        k = workloads.kv_rows(w, "k", 0, t0, t1).contiguous().numpy()
        v = workloads.kv_rows(w, "v", 0, t0, t1).contiguous().numpy()
        oracle.quantize_append(k, sm[t0:t1], pools[0], pools[1])
        oracle.quantize_append(v, sm[t0:t1], pools[2], pools[3])
    q = workloads.query(w)[:1].float().numpy()
    return pools, bt, q, L


def _time_oracle_decode(pools, bt, q, L, budget_s: float):
    import oracle
    reps, total = 0, 0.0
    while total < budget_s or reps == 0:
        t = time.perf_counter()
        oracle.paged_decode(*pools, q, bt, np.int32([L]))
        total += time.perf_counter() - t
        reps += 1
    return reps, total


def cpu_baseline(headline: str, budget_s: float = 24.0):
    """The oracle decode timed on this host's cores, for every decode workload,
    on all cores and on one: each pass decodes every query head of sequence 0
    over its first CPU_SAMPLE_TOKENS tokens (the oracle's cost per KV token
    does not depend on the context length); passes repeat until about
    budget_s / 16 seconds are timed per (workload, thread count)."""
    import oracle
    cores = oracle.num_threads()
    per = budget_s / (2 * len(WORKLOADS))
    rows = {}
    try:
        for name, (wname, batch) in WORKLOADS.items():
            w = workloads.make(wname, batch=batch)
            pools, bt, q, L = _cpu_sample(w, CPU_SAMPLE_TOKENS)
            row = {"sample_tokens": L, "query_heads": w.num_q_heads}
            for key, threads in (("all_cores", cores), ("one_core", 1)):
                oracle.set_num_threads(threads)
                reps, total = _time_oracle_decode(pools, bt, q, L, per)
                row[key] = {"value": L * reps / total, "threads": threads, "passes": reps, "seconds": total}
            rows[name] = row
    finally:
        oracle.set_num_threads(cores)
    h = rows[headline]
    return {"value": h["all_cores"]["value"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_thread_value": h["one_core"]["value"],
            "sample": (f"{headline}: sequence 0, its first {h['sample_tokens']} tokens, all {h['query_heads']} "
                       f"query heads (fp64 oracle decode over the oracle's own NVFP4 cache), repeated for "
                       f"{h['all_cores']['seconds']:.1f} s on {cores} threads; every workload below on "
                       f"{cores} threads and on 1"),
            "per_workload": rows}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step decodes a bounded sample of
    the workload (every query head of sequence 0 over its first
    REF_SAMPLE_TOKENS tokens) on the host cores."""
    import oracle
    name, batch = WORKLOADS[args.workload]
    w = workloads.make(name, batch=batch)
    pools, bt, q, L = _cpu_sample(w, REF_SAMPLE_TOKENS)
    for _ in range(args.warmup):
        oracle.paged_decode(*pools, q, bt, np.int32([L]))
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_decode(*pools, q, bt, np.int32([L]))
    el = time.perf_counter() - t
    value = L * args.steps / el
    sample = (f"per step: sequence 0, its first {L} tokens, all {w.num_q_heads} query heads, "
              f"fp64 oracle decode")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": w.batch, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                       "seq_len": (w.seq_lens[0] if len(set(w.seq_lens)) == 1 else "ragged"),
                       "kv_tokens_per_step": w.total_tokens,
                       "step": "a bounded sample of the workload per step (see cpu_baseline.sample), "
                               "the rate in KV-tokens/s of that sample"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world, rank)))
        return 0
    if args.row_only:
        import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
        nv.load()
        dev = torch.device("cuda", 0)
        warm = max(args.warmup, 3)
        if args.row_only == "prefill8k":
            row = prefill_rows(dev, steps=args.steps, warmup=warm)
        elif args.row_only.startswith("ext"):
            row = extend_rows(dev, args.row_only.replace("_e4m3", ""), steps=args.steps, warmup=warm,
                              compare_fused=False, chunk="e4m3" if args.row_only.endswith("_e4m3") else "bf16")
        else:
            row = write_side_row(dev, args.row_only, args.steps, warm)
        print(json.dumps(row))
        return 0
    world, rank, local = dist_init(args)
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
