"""Benchmark of the fused GQA flash-attention prefill on one GB300.

Headline workload (one "step"): a gpt-oss-20b-like prefill of 16,384 tokens
processed as 32 chunks of 512 over a growing cached prefix, through 24 layers
alternating full-causal and window-128 attention -- 768 calls, chunk-major
(the order a chunked prefill runs them).  Hq=64 / Hkv=8, d=64, bf16 Q/K/V
~ N(0,1) (synthetic: no model weights), per-head sinks ~ N(0,1).  All
inputs are resident in HBM before timing starts; they are far larger than
L2 (3.8 GB read per step), and a 256 MiB buffer is also written between
steps, outside the timed events.

Metric: useful attention TFLOP/s = 4 * d * Hq * (unmasked query-key pairs) /
time, counting only pairs the mask keeps; also prefill tokens/s (attention
only) and the fraction of the measured dense bf16 tensor peak.

The line also carries the gpt-oss layer pair (4096 tokens, one full-causal
and one window-128 layer) as a sub-object, the per-kernel rooflines, an
end-to-end figure through the C ABI from pinned host buffers, and the CPU
oracle timed on a bounded sample.  `--impl reference` times the CPU oracle
instead (a bounded sample of rows of the same workload); `--workload`
selects the supplementary configurations.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "useful attention TFLOP/s & prefill tok/s at 1 GB300; % of bf16 tensor peak"
UNIT = "TFLOP/s"
WORKLOAD = ("gpt-oss-20b-like 16k prefill: 24 layers alternating full-causal and window-128 "
            "(12 each), Hq=64, Hkv=8, d=64, bf16, 16384 tokens as 32 chunks of 512 over a "
            "growing prefix, per-head sinks (768 calls per step)")
PAIR_WORKLOAD = ("gpt-oss layer pair, pure prefill: B=1, seq 4096, Hq=64, Hkv=8, d=64, bf16, "
                 "full-causal + window-128, per-head sinks")
SEQ, CHUNK, LAYERS = 16384, 512, 24


def useful_pairs(prefix_lens, extend_lens, window):
    """Unmasked (query, key) pairs per head: sum over rows of the keys the
    causal / window mask keeps."""
    total = 0
    for p, e in zip(prefix_lens, extend_lens):
        for i in range(e):
            n = p + i + 1
            total += min(n, window) if window > 0 else n
    return total


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_tflops": pk["bf16_tflops"], "bf16_tflops_sustained": pk["bf16_tflops_sustained"],
                "hbm_gbs": pk["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


# The sources that define the roofline kernel (the d=64 single-tile prefill
# kernel) and its launch: the split-KV merge, the paged and split
# instantiations and the other head dims do not change it.
ROOFLINE_KERNEL_SOURCES = ("host.cu", "inst_d64.cu", "inst_balanced.cu", "launch.h", "prefill_kernel.cuh", "ptx.cuh",
                           "tile_math.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gqa_flash_attention_prefill_gb300", "csrc")
    for name in ROOFLINE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """DRAM bytes per launch recorded under `key` in the committed ncu summary
    (profiles/traffic.json), or None when the kernel sources changed since
    the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get(key)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (arrival time, line)
        self.window = None  # (start, end) of the timed region, perf_counter seconds

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, start, end):
        """Keep only samples that arrived inside the timed region."""
        self.window = (start, end)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for when, line in self.lines:
            if self.window is not None and not (self.window[0] <= when <= self.window[1] + 0.06):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[2:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    """One process per GPU under torchrun: each rank runs its own replica of
    the workload (the layer pair shards with no exchange step); returns
    (rank, world)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("GQA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return rank, world


def dist_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_layer_pair(args, rank, world):
    """The gpt-oss layer pair as the workload (`--workload layer_pair`)."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg
    from gqa_flash_attention_prefill_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    pkg.load()
    layers_cpu = W.layer_pair(seq=args.seq, seed=1)
    layers = [b.to("cuda") for b in layers_cpu]
    outs = [torch.empty_like(b.q) for b in layers]
    lses = [torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda") for b in layers]
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def step():
        for b, o, l in zip(layers, outs, lses):
            pkg.prefill(b, out=o, lse=l, stream=stream)

    pairs = [useful_pairs(b.prefix_lens.tolist(), b.extend_lens, b.window) for b in layers]
    flops = [4.0 * b.d * b.hq * n for b, n in zip(layers, pairs)]
    tokens = sum(b.total_q for b in layers)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised during warm-up")

    # Timed region: per step, flush L2 (untimed), then time each layer's
    # launch with events on the launching stream.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            pkg.prefill(layers[0], out=outs[0], lse=lses[0], stream=stream)
            ev[i][1].record(stream)
            pkg.prefill(layers[1], out=outs[1], lse=lses[1], stream=stream)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.perf_counter()
        clk.mark(t_wall0, t_wall1)
    dist_barrier(world)
    t_full = [e[0].elapsed_time(e[1]) for e in ev]
    t_win = [e[1].elapsed_time(e[2]) for e in ev]
    ms_step = statistics.median(a + b for a, b in zip(t_full, t_win))
    ms_step = dist_max(ms_step, world)
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised during the timed region")

    peaks = load_peaks()
    value = world * sum(flops) / (ms_step * 1e-3) / 1e12
    full_ms = statistics.median(t_full)
    achieved = flops[0] / (full_ms * 1e-3) / 1e12

    # The same launches without the L2 flush (the layer pair's 75 MB of
    # operands can then stay in the 129 MB L2 between steps): reported beside
    # the flushed figure, which remains `value`.
    n_warm = max(3, min(args.steps, 200))
    ev_w = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_warm)]
    for i in range(n_warm):
        ev_w[i][0].record(stream)
        pkg.prefill(layers[0], out=outs[0], lse=lses[0], stream=stream)
        pkg.prefill(layers[1], out=outs[1], lse=lses[1], stream=stream)
        ev_w[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = dist_max(statistics.median(e[0].elapsed_time(e[1]) for e in ev_w), world)

    # End to end through the C ABI from pinned host buffers: per step, copy
    # this step's inputs host->device, run both layers, read the outputs back.
    host = []
    for b in layers_cpu:
        hb = {n: getattr(b, n).pin_memory() for n in ("q", "k", "v", "cu_seqlens_q",
                                                       "prefix_lens", "kv_indptr", "sinks")}
        host.append(hb)
    host_out = [torch.empty(b.q.shape, dtype=b.q.dtype).pin_memory() for b in layers_cpu]
    host_lse = [torch.empty(b.q.shape[:2], dtype=torch.float32).pin_memory() for b in layers_cpu]
    h2d = sum(t.numel() * t.element_size() for hb in host for t in hb.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out + host_lse)

    # Three streams, as a caller would pipeline it: host->device copies of the
    # next layer's inputs and device->host copies of the previous layer's
    # outputs overlap the current layer's kernel.  Events keep every buffer
    # reuse ordered across layers and steps.
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    n_l = len(layers)
    in_ready = [torch.cuda.Event() for _ in range(n_l)]
    in_free = [torch.cuda.Event() for _ in range(n_l)]   # kernel done reading inputs
    out_free = [torch.cuda.Event() for _ in range(n_l)]  # copy-out done reading outputs
    for e in in_free + out_free:
        e.record(stream)

    def e2e_step():
        for L, (hb, b) in enumerate(zip(host, layers)):
            h2d_s.wait_event(in_free[L])
            with torch.cuda.stream(h2d_s):
                for n, t in hb.items():
                    getattr(b, n).copy_(t, non_blocking=True)
            in_ready[L].record(h2d_s)
        for L, (b, o, l, ho, hl) in enumerate(zip(layers, outs, lses, host_out, host_lse)):
            stream.wait_event(in_ready[L])
            stream.wait_event(out_free[L])
            pkg.prefill(b, out=o, lse=l, stream=stream)
            in_free[L].record(stream)
            d2h_s.wait_event(in_free[L])
            with torch.cuda.stream(d2h_s):
                ho.copy_(o, non_blocking=True)
                hl.copy_(l, non_blocking=True)
            out_free[L].record(d2h_s)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    dist_barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    d2h_s.wait_event(e0)
    for _ in range(e2e_steps):
        e2e_step()
    for e in out_free:
        stream.wait_event(e)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist_max(e0.elapsed_time(e1) / e2e_steps, world)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/K/V and sinks; no model weights)",
        "config": {"workload": PAIR_WORKLOAD, "global_batch": world, "seq_len": args.seq,
                   "layers": ["full-causal", "window-128"], "l2": "flushed between steps (256 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": round(world * tokens / 2 / (ms_step * 1e-3), 1),
        "pct_of_bf16_peak": round(100.0 * value / (world * peaks["bf16_tflops"]), 2),
        "per_layer_ms": {"full_causal": round(full_ms, 5),
                         "window_128": round(statistics.median(t_win), 5)},
        "per_layer_tflops": {"full_causal": round(achieved, 2),
                             "window_128": round(flops[1] / (statistics.median(t_win) * 1e-3) / 1e12, 2)},
        "roofline": {"bound": "tensor", "kernel": "prefill_kernel<64,128,...,full-causal>",
                     "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": recorded_traffic("full_layer_dram_bytes_per_launch"), "peak_source": peaks["source"] + " burst bf16"},
        "e2e": {"value": round(world * sum(flops) / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipeline": "copies in / kernel / copies out on three streams, overlapped across layers"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "timed_wall_s": round(t_wall1 - t_wall0, 3),
        "warm_l2": {"ms_per_step": round(warm_ms, 5), "steps": n_warm,
                    "value": round(world * sum(flops) / (warm_ms * 1e-3) / 1e12, 2),
                    "unit": UNIT, "note": "no L2 flush between steps; not the headline"},
    }
    return line


# ----------------------------------------------------------------- headline: 16k prefill

def chunk_pairs(prefix, extend, window):
    """Unmasked (query, key) pairs per head of one call with a single
    sequence: rows i < extend see min(prefix + i + 1, window) keys (all
    prefix + i + 1 without a window)."""
    n = sum(prefix + i + 1 for i in range(extend)) if window <= 0 else \
        sum(min(prefix + i + 1, window) for i in range(extend))
    return n


def window_call_bytes(prefix, extend, hq, hkv, d, window, elt=2):
    """Minimum HBM bytes of one windowed call: Q read and O written once, lse
    written, and of K and V only the rows some query's window reaches
    (min(prefix, window - 1) prefix rows plus the chunk's own)."""
    keys = min(prefix, window - 1) + extend
    return extend * hq * d * elt * 2 + extend * hq * 4 + keys * hkv * d * elt * 2


class Cudart:
    """cudaMemcpy2DAsync from the CUDA runtime already loaded by torch: one
    strided copy moves a chunk's rows of every layer (a layer-stacked device
    tensor and a chunk-major host buffer)."""

    H2D, D2H = 1, 2

    def __init__(self):
        import ctypes
        lib = None
        for name in ("libcudart.so.13", "libcudart.so.12", "/usr/local/cuda/lib64/libcudart.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("CUDA runtime library not found")
        c = ctypes
        lib.cudaMemcpy2DAsync.argtypes = [c.c_void_p, c.c_size_t, c.c_void_p, c.c_size_t,
                                          c.c_size_t, c.c_size_t, c.c_int, c.c_void_p]
        lib.cudaMemcpy2DAsync.restype = c.c_int
        self.lib = lib

    def copy2d(self, dst, dpitch, src, spitch, width, height, kind, stream):
        rc = self.lib.cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind,
                                        stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"cudaMemcpy2DAsync failed: {rc}")


def oss20b_setup(device="cuda", num_layers=LAYERS, seq=SEQ, chunk=CHUNK):
    """The 16k prefill's tensors (layer-stacked), its 768 calls in chunk-major
    order, and per call its kind, useful flops and minimum bytes."""
    from gqa_flash_attention_prefill_gb300 import workloads as W
    st = W.oss20b_stack(num_layers=num_layers, seq=seq, chunk_len=chunk, seed=3, device=device)
    metas = [st.chunk_meta(c, device) for c in range(st.num_chunks)]
    calls = []
    for c in range(st.num_chunks):
        for layer in range(st.num_layers):
            b = st.call(c, layer, metas[c])
            p = c * chunk
            fl = 4.0 * b.d * b.hq * chunk_pairs(p, chunk, b.window)
            nb = window_call_bytes(p, chunk, b.hq, b.hkv, b.d, b.window) if b.window > 0 else 0
            calls.append({"chunk": c, "layer": layer, "batch": b, "flops": fl, "bytes": nb,
                          "kind": "window_128" if b.window > 0 else "full_causal"})
    return st, metas, calls


def split_request(pkg, splits):
    """num_splits for --splits: None (the plain entry point), an int >= 0, or
    SPLITS_BALANCED."""
    if splits in (None, "none"):
        return None
    if splits == "balanced":
        return pkg.SPLITS_BALANCED
    k = int(splits)
    if k < 0:
        raise ValueError("--splits takes none, balanced or an integer >= 0")
    return k


def step_workspace(pkg, mode):
    """The one workspace the 16k step's balanced-split calls share (they run
    in stream order), or None when `mode` is "none"."""
    import torch
    if mode == "none":
        return None
    nbytes = max(pkg.splitkv_workspace(1, CHUNK, CHUNK, 64, 8, 64, "bf16", w,
                                       pkg.SPLITS_BALANCED)[1] for w in (0, 128))
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda")


# --balanced long: the default prefix from which a full-causal chunk call
# takes the balanced split (--long-prefix changes it).
LONG_PREFIX = 6144


def step_uses_balanced(kind, mode, prefix, long_prefix=None):
    lp = LONG_PREFIX if long_prefix is None else long_prefix
    return (mode == "all" or (mode == "full" and kind == "full_causal")
            or (mode == "long" and kind == "full_causal" and prefix >= lp))


def step_prepare(pkg, batch, kind, mode, ws, out, lse, stream, prefix=0, long_prefix=None):
    """A prepared call of the 16k step: the plain entry point, or the
    balanced split for the full-causal calls (`mode` "full"), for the
    full-causal calls over at least `long_prefix` (default LONG_PREFIX)
    cached tokens ("long"), or for all calls ("all")."""
    bal = step_uses_balanced(kind, mode, prefix, long_prefix)
    return pkg.prepare(batch, out=out, lse=lse, stream=stream,
                       num_splits=pkg.SPLITS_BALANCED if bal else None,
                       workspace=ws if bal else None)


def run_oss20b(args, rank, world):
    """Headline: the 16k chunked prefill, 768 calls per step."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    pkg.load()
    st, metas, calls = oss20b_setup()
    # The chunks' metadata is uploaded once, before any call (and, in the e2e
    # object, by copies the compute stream waits for): no kernel writes it, so
    # the kernels may read it before waiting on the previous kernel.
    pkg.set_call_flags(0 if args.no_metadata_ready else pkg.FLAG_METADATA_READY)
    out = torch.empty_like(st.q)
    lse = torch.empty(st.q.shape[:3], dtype=torch.float32, device="cuda")
    # Everything runs on one side stream: a CUDA graph is captured from it.
    stream = torch.cuda.Stream()
    L = CHUNK
    ws = step_workspace(pkg, args.balanced)
    for cl in calls:
        c, layer = cl["chunk"], cl["layer"]
        cl["run"] = step_prepare(pkg, cl["batch"], cl["kind"], args.balanced, ws,
                                 out[layer, c * L:(c + 1) * L], lse[layer, c * L:(c + 1) * L],
                                 stream, prefix=c * L, long_prefix=args.long_prefix)
    flops = sum(cl["flops"] for cl in calls)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def step():
        for cl in calls:
            cl["run"]()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            step()
    torch.cuda.synchronize()
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised during warm-up")
    # The step's 768 calls as one CUDA graph (their programmatic dependent
    # launches become programmatic edges), unless --eager: replaying it saves
    # the per-launch submission cost (1% of the step on GB300).
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        torch.cuda.synchronize()
    run_step = graph.replay if graph is not None else step

    # Timed region: K steps, each bracketed by events on the launching stream;
    # the L2 flush sits between steps, outside the events.
    steps = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush.fill_(float(i))
                ev[i][0].record(stream)
                run_step()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.perf_counter()
        clk.mark(t_wall0, t_wall1)
    dist_barrier(world)
    t_steps = [e[0].elapsed_time(e[1]) for e in ev]
    ms_step = dist_max(statistics.median(t_steps), world)
    ms_mean = dist_max(statistics.mean(t_steps), world)
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised during the timed region")

    # Per-kernel durations: the same steps again with an event between every
    # two launches (on the launching stream), so each call's duration is known.
    # The events keep each kernel from overlapping its neighbour, so these are
    # the kernels' isolated times; the headline above has no such events.
    n_b = max(1, min(steps, 10))
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
           for _ in range(n_b)]
    with torch.cuda.stream(stream):
        for i in range(n_b):
            flush.fill_(float(i))
            evb[i][0].record(stream)
            for j, cl in enumerate(calls):
                cl["run"]()
                evb[i][j + 1].record(stream)
    torch.cuda.synchronize()
    kind_ms = {"full_causal": 0.0, "window_128": 0.0}
    for i in range(n_b):
        for j, cl in enumerate(calls):
            kind_ms[cl["kind"]] += evb[i][j].elapsed_time(evb[i][j + 1]) / n_b
    kind_ms = {k: dist_max(v, world) for k, v in kind_ms.items()}
    # isolated time per chunk and kind, averaged over the layers and steps
    chunk_ms = {"full_causal": [0.0] * st.num_chunks, "window_128": [0.0] * st.num_chunks}
    for i in range(n_b):
        for j, cl in enumerate(calls):
            chunk_ms[cl["kind"]][cl["chunk"]] += (evb[i][j].elapsed_time(evb[i][j + 1])
                                                  / n_b / (st.num_layers // 2))
    kind_flops = {k: sum(cl["flops"] for cl in calls if cl["kind"] == k) for k in kind_ms}
    win_bytes = sum(cl["bytes"] for cl in calls if cl["kind"] == "window_128")
    n_kind = {k: sum(1 for cl in calls if cl["kind"] == k) for k in kind_ms}
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised during the per-kernel pass")

    peaks = load_peaks()
    value = world * flops / (ms_step * 1e-3) / 1e12
    full_tf = kind_flops["full_causal"] / (kind_ms["full_causal"] * 1e-3) / 1e12
    win_gbs = win_bytes / (kind_ms["window_128"] * 1e-3) / 1e9
    e2e = oss20b_e2e(args, st, metas, calls, out, lse, stream, world, flops, ws)
    n_bal = sum(1 for cl in calls if cl["kind"] == "full_causal"
                and step_uses_balanced(cl["kind"], args.balanced, cl["chunk"] * CHUNK,
                                       args.long_prefix))
    full_kernel_desc = (f"prefill_kernel<64,128,...> full-causal calls ({n_kind['full_causal']} "
                        f"per step: {n_kind['full_causal'] - n_bal} unsplit, {n_bal} through the "
                        f"balanced split)")
    del flush
    pair = layer_pair_summary(args, world, peaks)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/K/V and sinks; no model weights)",
        "config": bench_config(world, args.balanced, args.eager, args.long_prefix,
                               not args.no_metadata_ready),
        "ms_per_step_mean": round(ms_mean, 4),
        "tokens_per_s": round(world * SEQ / (ms_step * 1e-3), 1),
        "pct_of_bf16_peak": round(100.0 * value / (world * peaks["bf16_tflops"]), 2),
        "pct_of_bf16_peak_sustained": round(100.0 * value / (world * peaks["bf16_tflops_sustained"]), 2),
        "roofline": {"bound": "tensor",
                     "kernel": full_kernel_desc,
                     "achieved": round(full_tf, 2), "peak": peaks["bf16_tflops_sustained"],
                     "unit": "TFLOP/s", "frac": round(full_tf / peaks["bf16_tflops_sustained"], 4),
                     "frac_of_burst": round(full_tf / peaks["bf16_tflops"], 4),
                     "traffic": recorded_traffic("oss20b_full_dram_bytes_per_launch"),
                     "peak_source": peaks["source"] + " sustained bf16 (kernel timed inside a "
                                                      "seconds-long loop)",
                     "work": "useful flops (4 d Hq per unmasked pair) of the full-causal calls / "
                             "their summed isolated durations"},
        "roofline_window": {"bound": "hbm",
                            "kernel": "prefill_kernel<64,64,...> window-128 calls (384 per step)",
                            "achieved": round(win_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(win_gbs / peaks["hbm_gbs"], 4),
                            "traffic": recorded_traffic("oss20b_window_dram_bytes_per_launch"),
                            "algorithmic_bytes_per_launch": round(win_bytes / n_kind["window_128"]),
                            "work": "Q read, O and lse written, K and V rows inside some "
                                    "query's window read once"},
        "per_kind": {k: {"calls": n_kind[k], "ms_per_step": round(kind_ms[k], 4),
                         "useful_tflops": round(kind_flops[k] / (kind_ms[k] * 1e-3) / 1e12, 2)}
                     for k in kind_ms},
        "per_chunk_us": {k: [round(1e3 * x, 1) for x in v] for k, v in chunk_ms.items()},
        "layer_pair": pair,
        "e2e": e2e,
        "gpu_launches": len(calls) * steps,
        "clocks": clk.summary(),
        "timed_wall_s": round(t_wall1 - t_wall0, 3),
    }
    return line


def run_profile(args):
    """`--profile step`: the warm-up steps and one more step of the 16k
    prefill (768 calls), untimed, for an ncu launch list or a counter capture
    of every launch of a step.  `--profile chunk31`: chunk 31's full-causal and
    window-128 calls once each (the largest calls of the step), for a full
    ncu capture.  `--profile pair`: the layer pair's two calls once each.
    Prints nothing but a completion line; no bench values."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg
    from gqa_flash_attention_prefill_gb300 import workloads as W
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    pkg.load()
    pkg.set_call_flags(0 if args.no_metadata_ready else pkg.FLAG_METADATA_READY)
    stream = torch.cuda.current_stream()
    if args.profile == "pair":
        for b in W.layer_pair(seq=4096, seed=1):
            pkg.prefill(b.to("cuda"), stream=stream)
        n = 2
    elif args.profile == "chunk31":
        st = W.oss20b_stack(num_layers=2, seq=SEQ, chunk_len=CHUNK, seed=3, device="cuda")
        ws = step_workspace(pkg, args.balanced)
        for layer in (0, 1):
            b = st.call(SEQ // CHUNK - 1, layer)
            kind = "window_128" if b.window > 0 else "full_causal"
            step_prepare(pkg, b, kind, args.balanced, ws, torch.empty_like(b.q),
                         torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda"), stream,
                         prefix=SEQ - CHUNK, long_prefix=args.long_prefix)()
        n = 2
    else:
        st, metas, calls = oss20b_setup()
        out = torch.empty_like(st.q)
        lse = torch.empty(st.q.shape[:3], dtype=torch.float32, device="cuda")
        L = CHUNK
        ws = step_workspace(pkg, args.balanced)
        runs = [step_prepare(pkg, cl["batch"], cl["kind"], args.balanced, ws,
                             out[cl["layer"], cl["chunk"] * L:(cl["chunk"] + 1) * L],
                             lse[cl["layer"], cl["chunk"] * L:(cl["chunk"] + 1) * L], stream,
                             prefix=cl["chunk"] * L, long_prefix=args.long_prefix)
                for cl in calls]
        for _ in range(args.warmup + 1):
            for r in runs:
                r()
        n = len(runs) * (args.warmup + 1)
    torch.cuda.synchronize()
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised")
    print(f"profile run done: {n} prefill launches", flush=True)


def bench_config(world, balanced="long", eager=False, long_prefix=None, metadata_ready=True):
    lp = LONG_PREFIX if long_prefix is None else long_prefix
    entry = {"none": "gqa_flash_prefill",
             "full": "gqa_flash_prefill_splitkv (balanced split) for the full-causal calls, "
                     "gqa_flash_prefill for the window-128 calls",
             "long": f"gqa_flash_prefill_splitkv (balanced split) for the full-causal calls "
                     f"over >= {lp} cached tokens, gqa_flash_prefill for the others",
             "all": "gqa_flash_prefill_splitkv (balanced split)"}[balanced]
    return {"workload": WORKLOAD, "global_batch": world, "seq_len": SEQ, "chunk_len": CHUNK,
            "layers": LAYERS, "calls_per_step": LAYERS * (SEQ // CHUNK),
            "l2": "inputs larger than L2 (3.8 GB read per step); 256 MiB written between steps",
            "parallelism": "replicas (one per GPU)" if world > 1 else "single GPU",
            "entry": entry,
            "launch": ("each call launched by the host" if eager else
                       "the step's calls replayed as one CUDA graph, captured once after "
                       "the warm-up (the e2e object launches them one by one)"),
            "call_flags": ("GQA_FLAG_METADATA_READY (metadata uploaded once per chunk, "
                           "read before the kernel waits on its predecessor)"
                           if metadata_ready else "none")}


def oss20b_e2e(args, st, metas, calls, out, lse, stream, world, flops, ws=None):
    """The 16k prefill end to end through the C ABI from pinned host memory:
    every step uploads each chunk's Q rows, its new K and V rows and its
    metadata for all 24 layers, runs the chunk's 24 calls, and downloads the
    chunk's output and lse rows.  Copies run on their own streams, one
    strided copy per tensor and chunk, so uploads and downloads overlap the
    kernels.  Consecutive steps alternate between two sets of device buffers
    (as a server alternates between requests), so a step's uploads need not
    wait for the previous step's last kernel, which still reads the K/V rows
    they would overwrite."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg
    from gqa_flash_attention_prefill_gb300 import workloads as W
    cr = Cudart()
    n_l, n_c, L = st.num_layers, st.num_chunks, st.chunk_len
    hq, hkv, d = st.q.shape[2], st.k.shape[2], st.q.shape[3]
    # Chunk-major pinned host buffers: [chunk][layer][row][head][dim].
    hq_ = torch.empty((n_c, n_l, L, hq, d), dtype=st.q.dtype, pin_memory=True)
    hk_ = torch.empty((n_c, n_l, L, hkv, d), dtype=st.k.dtype, pin_memory=True)
    hv_ = torch.empty((n_c, n_l, L, hkv, d), dtype=st.v.dtype, pin_memory=True)
    hm_ = torch.stack([m.cpu() for m in metas]).pin_memory()
    ho_ = torch.empty((n_c, n_l, L, hq, d), dtype=out.dtype, pin_memory=True)
    hl_ = torch.empty((n_c, n_l, L, hq), dtype=torch.float32, pin_memory=True)
    for c in range(n_c):
        hq_[c].copy_(st.q[:, c * L:(c + 1) * L])
        hk_[c].copy_(st.k[:, c * L:(c + 1) * L])
        hv_[c].copy_(st.v[:, c * L:(c + 1) * L])
    # Two device sets: the resident tensors and a second set of the same shapes.
    st2 = W.PrefillStack(torch.empty_like(st.q), torch.empty_like(st.k), torch.empty_like(st.v),
                         st.sinks, st.windows, st.chunk_len, st.scale)
    metas2 = [torch.empty_like(m) for m in metas]
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    sets = []
    for s_, m_, o_, l_ in ((st, metas, out, lse), (st2, metas2, out2, lse2)):
        runs = [[step_prepare(pkg, s_.call(c, layer, m_[c]),
                              "window_128" if s_.windows[layer] > 0 else "full_causal",
                              args.balanced, ws, o_[layer, c * L:(c + 1) * L],
                              l_[layer, c * L:(c + 1) * L], stream, prefix=c * L,
                              long_prefix=args.long_prefix)
                 for layer in range(n_l)] for c in range(n_c)]
        sets.append({"st": s_, "metas": m_, "out": o_, "lse": l_, "runs": runs,
                     "in_ready": [torch.cuda.Event() for _ in range(n_c)],
                     "done": [torch.cuda.Event() for _ in range(n_c)],
                     "out_free": [torch.cuda.Event() for _ in range(n_c)],
                     "step_done": torch.cuda.Event()})
    for S in sets:
        for e in S["out_free"] + [S["step_done"]]:
            e.record(stream)
    elt = st.q.element_size()
    q_row, kv_row, o_row, l_row = hq * d * elt, hkv * d * elt, hq * d * out.element_size(), hq * 4
    seq = st.q.shape[1]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def up(dev_t, host_t, c, row_bytes):
        # rows [c L, (c+1) L) of every layer: n_l blocks of L rows, one layer apart
        cr.copy2d(dev_t.data_ptr() + c * L * row_bytes, seq * row_bytes, host_t[c].data_ptr(),
                  L * row_bytes, L * row_bytes, n_l, Cudart.H2D, h2d_s)

    def down(host_t, dev_t, c, row_bytes):
        cr.copy2d(host_t[c].data_ptr(), L * row_bytes, dev_t.data_ptr() + c * L * row_bytes,
                  seq * row_bytes, L * row_bytes, n_l, Cudart.D2H, d2h_s)

    def e2e_step(S):
        # This set's K/V rows were last read by its previous step's last kernel.
        h2d_s.wait_event(S["step_done"])
        s_ = S["st"]
        for c in range(n_c):
            up(s_.q, hq_, c, q_row)
            up(s_.k, hk_, c, kv_row)
            up(s_.v, hv_, c, kv_row)
            with torch.cuda.stream(h2d_s):
                S["metas"][c].copy_(hm_[c], non_blocking=True)
            S["in_ready"][c].record(h2d_s)
        for c in range(n_c):
            stream.wait_event(S["in_ready"][c])
            stream.wait_event(S["out_free"][c])
            for r in S["runs"][c]:
                r()
            S["done"][c].record(stream)
            d2h_s.wait_event(S["done"][c])
            down(ho_, S["out"], c, o_row)
            down(hl_, S["lse"], c, l_row)
            S["out_free"][c].record(d2h_s)
        S["step_done"].record(stream)

    n_e = max(4, min(args.steps, 10))
    for i in range(2):
        e2e_step(sets[i % 2])
    torch.cuda.synchronize()
    dist_barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    d2h_s.wait_event(e0)
    for i in range(n_e):
        e2e_step(sets[i % 2])
    for S in sets:
        for e in S["out_free"]:
            stream.wait_event(e)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist_max(e0.elapsed_time(e1) / n_e, world)
    # the outputs of the last step match the device-resident run's
    last = sets[(n_e - 1) % 2]
    ok = bool(torch.equal(last["out"], out)) if last["out"] is not out else True
    h2d = n_c * (n_l * L * (q_row + 2 * kv_row) + hm_[0].numel() * 4)
    d2h = n_c * n_l * L * (o_row + l_row)
    del st2, out2, lse2, sets
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": n_e, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "outputs_match_resident_run": ok,
            "pipeline": "per chunk: strided uploads of Q, new K/V rows and metadata (all 24 "
                        "layers), 24 calls, strided downloads of out and lse; copy-in, compute "
                        "and copy-out streams; steps alternate between two device buffer sets"}


def layer_pair_summary(args, world, peaks):
    """The gpt-oss layer pair (4096 tokens), each layer timed alone with
    events, L2 flushed before every step: per-layer time and the two
    rooflines (full-causal: tensor, burst peak; window-128: HBM)."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg
    from gqa_flash_attention_prefill_gb300 import workloads as W
    layers = [b.to("cuda") for b in W.layer_pair(seq=4096, seed=1)]
    stream = torch.cuda.current_stream()
    outs = [torch.empty_like(b.q) for b in layers]
    lses = [torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda") for b in layers]
    runs = [pkg.prepare(b, out=o, lse=l, stream=stream) for b, o, l in zip(layers, outs, lses)]
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    n = max(20, min(10 * args.steps, 200))
    for _ in range(5):
        flush.fill_(1.0)
        for r in runs:
            r()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        runs[0]()
        ev[i][1].record(stream)
        runs[1]()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised in the layer pair")
    t_full = dist_max(statistics.median(e[0].elapsed_time(e[1]) for e in ev), world)
    t_win = dist_max(statistics.median(e[1].elapsed_time(e[2]) for e in ev), world)
    fl = [4.0 * b.d * b.hq * chunk_pairs(0, b.total_q, b.window) for b in layers]
    wb = window_call_bytes(0, layers[1].total_q, 64, 8, 64, 128)
    full_tf = fl[0] / (t_full * 1e-3) / 1e12
    return {"workload": PAIR_WORKLOAD, "steps": n,
            "ms_per_step": round(t_full + t_win, 5),
            "value": round(world * sum(fl) / ((t_full + t_win) * 1e-3) / 1e12, 2),
            "per_layer_ms": {"full_causal": round(t_full, 5), "window_128": round(t_win, 5)},
            "full_causal": {"bound": "tensor", "achieved": round(full_tf, 2),
                            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": round(full_tf / peaks["bf16_tflops"], 4),
                            "traffic": recorded_traffic("full_layer_dram_bytes_per_launch"),
                            "peak_source": peaks["source"] + " burst bf16 (one launch timed alone)"},
            "window_128": {"bound": "hbm", "achieved": round(wb / (t_win * 1e-3) / 1e9, 1),
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(wb / (t_win * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                           "algorithmic_bytes": wb,
                           "useful_tflops": round(fl[1] / (t_win * 1e-3) / 1e12, 2)},
            "l2": "flushed before every step (256 MiB write)"}


def run_ragged_grid(args, rank, world):
    """Throughput per cell of a grid over head counts, head dims and windows,
    on one ragged batch shape (16 sequences, prefixes U[0,16384], extends
    U[1,8192], seed 4): one call per cell, L2 flushed before each timed call.
    The inputs are generated on the GPU from a seeded CUDA generator."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg
    from gqa_flash_attention_prefill_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    pkg.load()
    gen = torch.Generator().manual_seed(4 * 7919 + 17)  # the lengths of workloads.ragged(seed=4)
    pre = torch.randint(0, 16384 + 1, (16,), generator=gen).tolist()
    ext = torch.randint(1, 8192 + 1, (16,), generator=gen).tolist()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    peaks = load_peaks()
    steps = max(3, min(args.steps, args.grid_steps))
    cells, tot_flops, tot_ms, launches = [], 0.0, 0.0, 0
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for hq, hkv in ((64, 8), (32, 4)):
            for d in (64, 128, 256):
                for window in (0, 128):
                    b = W.make_batch(pre, ext, hq, hkv, d, "bf16", window=window,
                                     sink_mode="head", seed=4, device="cuda",
                                     name=f"grid-{hq}/{hkv}-d{d}-w{window}")
                    out = torch.empty_like(b.q)
                    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device="cuda")
                    for _ in range(args.warmup):
                        flush.fill_(1.0)
                        pkg.prefill(b, out=out, lse=lse, stream=stream)
                    ts = []
                    for i in range(steps):
                        flush.fill_(float(i))
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        pkg.prefill(b, out=out, lse=lse, stream=stream)
                        e1.record(stream)
                        e1.synchronize()
                        ts.append(e0.elapsed_time(e1))
                    launches += steps
                    if pkg.get_device_status() != 0:
                        raise RuntimeError("device status word raised in " + b.name)
                    ms = dist_max(statistics.median(ts), world)
                    fl = 4.0 * d * hq * useful_pairs(pre, ext, window)
                    tf = world * fl / (ms * 1e-3) / 1e12
                    cells.append({"hq": hq, "hkv": hkv, "d": d, "window": window, "ms": round(ms, 4),
                                  "tflops": round(tf, 1),
                                  "pct_of_bf16_peak": round(100.0 * tf / (world * peaks["bf16_tflops"]), 1)})
                    tot_flops += fl
                    tot_ms += ms
                    del b, out, lse
        clk.mark(t0, time.perf_counter())
    value = world * tot_flops / (tot_ms * 1e-3) / 1e12
    return {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(tot_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V and sinks, generated on the GPU)",
            "config": {"workload": "ragged grid: 16 sequences, prefixes U[0,16384], extends "
                                   "U[1,8192]; {64/8, 32/4} x d {64, 128, 256} x window "
                                   "{none, 128}; bf16, per-head sinks; one call per cell, "
                                   "median of the steps; value = all cells' flops / summed times",
                       "l2": "flushed before every timed call (256 MiB write)"},
            "cells": cells, "gpu_launches": launches, "clocks": clk.summary()}


def run_workload(args, rank, world):
    """Supplementary workloads: one step = every call of the workload, timed as
    a whole with CUDA events (L2 flushed before each step, outside the
    events)."""
    import torch
    import gqa_flash_attention_prefill_gb300 as pkg
    from gqa_flash_attention_prefill_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    pkg.load()
    dev = "cuda"
    masks = None
    if args.workload == "chunked_prefix":
        full = W.chunked_prefix(8, 8192, 8192, 128, seed=2)
        b = W.window_bounded(full, 128) if args.layout == "window-bounded" else full
        calls = [b.to(dev)]
        desc = (f"chunked prefill over cached prefix: B=8, prefix 8192 + extend 8192, 64/8, d 64, "
                f"bf16, window 128, sinks, {args.layout} KV layout")
        tokens = 8 * 8192
    elif args.workload == "ragged":
        b = W.ragged(hq=64, hkv=8, d=64, dtype="bf16", window=128, sink_mode="head", seed=4)
        calls = [b.to(dev)]
        desc = ("ragged varlen: 16 sequences, prefixes U[0,16384], extends U[1,8192], 64/8, d 64, "
                "bf16, window 128, sinks")
        tokens = b.total_q
    elif args.workload == "ragged_full":
        b = W.ragged(hq=64, hkv=8, d=64, dtype="bf16", window=0, sink_mode="head", seed=4)
        calls = [b.to(dev)]
        desc = ("ragged varlen, full causal: 16 sequences, prefixes U[0,16384], extends "
                "U[1,8192], 64/8, d 64, bf16, sinks")
        tokens = b.total_q
    elif args.workload == "decode":
        b = W.decode(num_seqs=128, min_prefix=1024, max_prefix=16384, window=128,
                     sink_mode="head", seed=6,
                     window_bounded_layout=(args.layout == "window-bounded"))
        calls = [b.to(dev)]
        desc = (f"windowed decode: 128 sequences x 1 new token over prefixes U[1024,16384], "
                f"64/8, d 64, bf16, window 128, sinks, {args.layout} KV layout")
        tokens = 128
    elif args.workload == "decode_full":
        b = W.decode(num_seqs=256, min_prefix=1024, max_prefix=16384, window=0,
                     sink_mode="head", seed=6)
        calls = [b.to(dev)]
        desc = ("full-attention decode: 256 sequences x 1 new token over prefixes "
                "U[1024,16384], 64/8, d 64, bf16, sinks (every prefix key read once)")
        tokens = 256
    elif args.workload == "short_chunk":
        calls = [W.make_batch([16384, 16384], [64, 64], 64, 8, 64, "bf16", window=w,
                              sink_mode="head", seed=5 + i, name=f"short-chunk-w{w}").to(dev)
                 for i, w in enumerate((0, 128))]
        desc = ("short chunks over long prefixes: 2 sequences x (prefix 16384 + extend 64), "
                "64/8, d 64, bf16, sinks; one full-causal and one window-128 call per step")
        tokens = 2 * 128
    elif args.workload == "tree_verify":
        # custom mask with and without a sliding window: 8 sequences, 8192
        # cached tokens each, 64 draft tokens in a random tree per sequence
        trees = [W.random_tree_mask(64, seed=50 + s_) for s_ in range(8)]
        full = W.make_batch([8192] * 8, [64] * 8, 64, 8, 64, "bf16", window=0,
                            sink_mode="head", seed=7, name="tree-verify-full")
        win = W.window_bounded(W.make_batch([8192] * 8, [64] * 8, 64, 8, 64, "bf16", window=128,
                                            sink_mode="head", seed=8), 128)
        calls = [full.to(dev), win.to(dev)]
        words, indptr = W.pack_custom_mask(trees)
        masks = [(words.to(dev), indptr.to(dev))] * 2
        desc = ("custom-mask verify: 8 sequences x (8192 cached + 64 draft tokens in a random "
                "tree), 64/8, d 64, bf16, sinks; one full-attention and one window-128 "
                "(window-bounded KV) call per step")
        tokens = 2 * 8 * 64
    else:
        raise ValueError(args.workload)
    flops = 0.0
    for i, b in enumerate(calls):
        if masks is not None:  # kept pairs under causal, window and custom mask
            pre = [int(x) for x in b.prefix_lens.tolist()]
            for s_, (p_, e) in enumerate(zip(pre, b.extend_lens)):
                for row in range(e):
                    pos = p_ + row
                    lo = 0 if b.window <= 0 else max(0, pos - b.window + 1)
                    n = (min(p_, pos + 1) - min(lo, p_)) + int(
                        sum(trees[s_][row, j - p_] for j in range(max(lo, p_), pos + 1)))
                    flops += 4.0 * b.d * b.hq * n
        else:
            flops += 4.0 * b.d * b.hq * useful_pairs([int(x) for x in b.prefix_lens.tolist()],
                                                     b.extend_lens, b.window)
    outs = [torch.empty_like(b.q) for b in calls]
    lses = [torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev) for b in calls]
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    # --splits k (k >= 0) or balanced: the split-KV entry point (0 = the
    # library's choice; balanced = GQA_SPLITS_BALANCED), with a workspace per
    # call allocated here, outside the timed region.
    split_req = split_request(pkg, args.splits)
    splits_used, workspaces = [], []
    if split_req is not None:
        for b in calls:
            used, nbytes = pkg.splitkv_workspace(b.num_seqs, b.total_q, b.max_seqlen_q, b.hq,
                                                 b.hkv, b.d, b.dtype_name, b.window, split_req)
            splits_used.append(used)
            workspaces.append(torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev))

    # --paged P: the same K/V laid out as a shuffled pool of P-token pages.
    paged_calls = ([W.paged(b.to("cpu"), args.paged, seed=i).to(dev) for i, b in enumerate(calls)]
                   if args.paged > 0 else [])

    def step():
        for i, (b, o, l) in enumerate(zip(calls, outs, lses)):
            if masks is not None:
                pkg.prefill_masked(b, masks[i][0], masks[i][1], out=o, lse=l, stream=stream)
            elif args.paged > 0:
                pkg.prefill_paged(paged_calls[i], out=o, lse=l, stream=stream)
            elif split_req is not None:
                pkg.prefill_splitkv(b, num_splits=split_req, workspace=workspaces[i], out=o,
                                    lse=l, stream=stream)
            else:
                pkg.prefill(b, out=o, lse=l, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if pkg.get_device_status() != 0:
        raise RuntimeError("device status word raised during warm-up")
    # Timed steps: as asked, but at most about 30 s of timed work (the 16k
    # prefill's 768 calls take ~35 ms a step); every rank takes the same count.
    e0_, e1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0_.record(stream)
    step()
    e1_.record(stream)
    torch.cuda.synchronize()
    probe_ms = dist_max(e0_.elapsed_time(e1_), world)
    steps = max(3, min(args.steps, int(30000.0 / max(probe_ms, 1e-3))))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        clk.mark(t0, time.perf_counter())
    dist_barrier(world)
    ms_step = dist_max(statistics.median(e[0].elapsed_time(e[1]) for e in ev), world)
    peaks = load_peaks()
    value = world * flops / (ms_step * 1e-3) / 1e12
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V and sinks; no model weights)",
            "config": {"workload": desc, "l2": "flushed between steps (256 MiB write)",
                       "calls_per_step": len(calls),
                       "entry": (f"gqa_flash_prefill_paged, page_size {args.paged}"
                                 if args.paged > 0 else
                                 ("gqa_flash_prefill_splitkv, splits " + str(splits_used))
                                 if split_req is not None else "gqa_flash_prefill")},
            "tokens_per_s": round(world * tokens / (ms_step * 1e-3), 1),
            "pct_of_bf16_peak": round(100.0 * value / (world * peaks["bf16_tflops"]), 2),
            "gpu_launches": len(calls) * steps + sum(1 for s_ in splits_used if s_ > 1) * steps,
            "clocks": clk.summary()}
    if masks is not None:
        line["config"]["entry"] = "gqa_flash_prefill_masked"
    if args.workload in ("chunked_prefix", "decode", "decode_full", "tree_verify"):
        # HBM-bound: Q read and O (+ lse) written once; of K and V only the rows some
        # window reaches (the window-bounded layout's rows) must be read, in either layout.
        nbytes = 0
        for b in calls:
            keys = sum((min(p_, b.window) if b.window > 0 else p_) + e for p_, e in
                       zip([int(x) for x in b.prefix_lens.tolist()], b.extend_lens))
            nbytes += b.q.numel() * 2 * 2 + keys * b.hkv * b.d * 2 * 2 + b.q.shape[0] * b.hq * 4
        gbs = nbytes / (ms_step * 1e-3) / 1e9
        line["roofline"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                            "traffic": None, "algorithmic_bytes": nbytes}
    if args.workload == "ragged_full":
        # Tensor-bound: useful flops over the measured dense bf16 peak (burst; one call).
        line["roofline"] = {"bound": "tensor", "achieved": round(value / world, 1),
                            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": round(value / world / peaks["bf16_tflops"], 4),
                            "traffic": None}
    return line


def oracle_inputs(layers_cpu):
    """Widen each layer's inputs to float64 once, outside any timing."""
    import numpy as np
    out = []
    for b in layers_cpu:
        x = {n: np.ascontiguousarray(getattr(b, n).double().numpy()) for n in ("q", "k", "v")}
        x["out"] = np.empty(x["q"].shape)            # result buffers, reused by every call
        x["lse"] = np.empty(x["q"].shape[:2])
        out.append((b, x))
    return out


def oracle_sample_run(layers64, rows_per_layer, offset=0):
    """Runs the CPU oracle on `rows_per_layer` evenly spaced query rows of
    each layer (inputs from oracle_inputs); returns (seconds, useful flops,
    rows)."""
    import numpy as np
    import oracle
    total_s, total_flops, total_rows = 0.0, 0.0, 0
    for b, x in layers64:
        e = b.total_q
        step = max(1, e // rows_per_layer)
        rows = (np.arange(rows_per_layer) * step + offset) % e
        t0 = time.perf_counter()
        oracle.prefill(x["q"], x["k"], x["v"], b.cu_seqlens_q, b.prefix_lens, b.kv_indptr,
                       b.scale, b.window, sinks=b.sinks, smooth_softmax=b.smooth, rows=rows,
                       out=x["out"], lse=x["lse"])
        total_s += time.perf_counter() - t0
        pre = int(b.prefix_lens[0])
        for r in rows:
            n = pre + int(r) + 1
            total_flops += 4.0 * b.d * b.hq * (min(n, b.window) if b.window > 0 else n)
        total_rows += len(rows)
    return total_s, total_flops, total_rows


def size_oracle_sample(layers64, target_s):
    """Rows per layer so that one oracle sample takes about target_s."""
    probe = 32
    t, _, _ = oracle_sample_run(layers64, probe)
    per_row = max(t / probe, 1e-6)
    return int(max(8, min(layers64[0][0].total_q, target_s / per_row)))


def oracle_sample_calls():
    """The calls the CPU oracle times, on the host: chunks 0, 10, 21 and 31 of
    the 16k prefill's first full-causal and first window-128 layer (the same
    seeded tensors as layers 0 and 1 of the GPU run)."""
    from gqa_flash_attention_prefill_gb300 import workloads as W
    st = W.oss20b_stack(num_layers=2, seq=SEQ, chunk_len=CHUNK, seed=3, device="cpu")
    return [st.call(c, layer) for c in (0, 10, 21, 31) for layer in (0, 1)]


SAMPLE_DESC = ("evenly spaced query rows of each of 8 calls of the 16k prefill (chunks 0, 10, "
               "21, 31 of a full-causal and a window-128 layer), all 64 heads, fp64 CPU oracle")


def cpu_baseline(args):
    import oracle
    oracle.build()
    layers64 = oracle_inputs(oracle_sample_calls())
    rows = size_oracle_sample(layers64, args.cpu_seconds)
    t, fl, n = oracle_sample_run(layers64, rows)
    return {"value": fl / t / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{rows} {SAMPLE_DESC}; {n} rows in {t:.1f} s, {fl / t / 1e9:.2f} useful "
                      f"GFLOP/s; rate of the sample, not extrapolated"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on this workload's metric: each
    step a bounded sample of rows of the headline workload's calls."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    layers64 = oracle_inputs(oracle_sample_calls())
    # About --ref-seconds (150 s by default) of oracle work in total, however
    # many steps are asked for.
    per_step_s = max(0.005, min(5.0, args.ref_seconds / max(1, args.steps + args.warmup)))
    rows = size_oracle_sample(layers64, per_step_s)
    for i in range(args.warmup):
        oracle_sample_run(layers64, rows, offset=i)
    secs, fl_total = 0.0, 0.0
    for i in range(args.steps):
        t, fl, n = oracle_sample_run(layers64, rows, offset=args.warmup + i)
        secs += t
        fl_total += fl
    value = fl_total / secs / 1e12
    cores = oracle.num_threads()
    sample = f"each step: {rows} {SAMPLE_DESC}"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) Q/K/V and sinks; no model weights)",
            "config": bench_config(world, args.balanced, args.eager, args.long_prefix,
                               not args.no_metadata_ready),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seq", type=int, default=4096, help="layer_pair workload: tokens")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU work of the oracle baseline sample (rank 0, N=1)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="--impl reference: total CPU seconds of oracle work over all steps")
    ap.add_argument("--workload", default="oss20b_16k",
                    choices=["oss20b_16k", "layer_pair", "chunked_prefix", "ragged", "ragged_full",
                             "ragged_grid", "short_chunk", "decode", "decode_full",
                             "tree_verify"],
                    help="oss20b_16k is the headline configuration; the others are "
                         "supplementary measurements")
    ap.add_argument("--layout", default="window-bounded", choices=["window-bounded", "full-prefix"],
                    help="KV layout of the chunked_prefix and decode workloads")
    ap.add_argument("--paged", type=int, default=0,
                    help="supplementary workloads: K/V as a page pool with this page size "
                         "(0: contiguous)")
    ap.add_argument("--grid-steps", type=int, default=10,
                    help="ragged_grid: timed calls per cell (capped by --steps)")
    ap.add_argument("--splits", default="none",
                    help="supplementary workloads: none, the plain entry point; 0, split-KV "
                         "with the library's split count; k >= 1, split-KV with k splits; "
                         "balanced, the balanced split")
    ap.add_argument("--balanced", choices=["none", "long", "full", "all"], default="long",
                    help="16k prefill: the balanced split (gqa_flash_prefill_splitkv with "
                         "GQA_SPLITS_BALANCED) for no call, the full-causal calls over long "
                         "prefixes, all full-causal calls, or all calls")
    ap.add_argument("--long-prefix", type=int, default=LONG_PREFIX,
                    help="--balanced long: cached tokens from which a full-causal call takes "
                         "the balanced split")
    ap.add_argument("--no-metadata-ready", action="store_true",
                    help="16k prefill: do not set GQA_FLAG_METADATA_READY (the kernels then "
                         "read the metadata only after waiting on the previous kernel)")
    ap.add_argument("--eager", action="store_true",
                    help="16k prefill: launch the step's calls one by one instead of replaying "
                         "them as one CUDA graph")
    ap.add_argument("--profile", choices=["step", "chunk31", "pair"], default=None,
                    help="untimed run for an ncu capture: the warm-up steps plus one step of "
                         "the 16k prefill, chunk 31's two calls, or the layer pair's two "
                         "calls; prints no bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile is not None:
        run_profile(args)
        return
    rank, world = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.workload == "ragged_grid":
        line = run_ragged_grid(args, rank, world)
    elif args.workload == "layer_pair":
        line = run_layer_pair(args, rank, world)
    elif args.workload != "oss20b_16k":
        line = run_workload(args, rank, world)
    else:
        line = run_oss20b(args, rank, world)
        if rank == 0:
            if world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(args)
            else:
                line["cpu_baseline"] = None
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
