"""Benchmark of the fused causal GQA attention forward on GB300 (one JSON line on stdout).

Default workload (one "step"): the chunked-prefill call of GQA 32/8, head dim 128, a 2048-row
query chunk at the end of 16384 keys (bottom-right causal), f16 -- the shape the throughput gate
of "perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)" is stated at.
``value`` is TFLOP/s under the FLOP convention 4 * D * Hq * B * (visible query-key pairs).

The same run also times, each in its own loop, the other hot-path workloads and reports them as
secondary legs: the q4_0 decode (``decode``: KV GB/s against the HBM roofline), the q4_0 chunked
prefill, the 2K/8K and bf16 prefill shapes and the q4_0 cache build.

Timing: CUDA events on the launching stream around each launch; the L2 cache is flushed (a
256 MiB write) before every timed prefill launch; decode reads 302 MB per call, more than L2.
The legs of 2048 keys or fewer also report ``graph_us``: the device time per call of 20 calls
replayed from one CUDA graph (no launch cost between calls, no L2 flush), beside their
per-launch event time, which for calls this short includes microseconds of launch overhead.
Multi-GPU: one process per GPU (torchrun); every rank runs a replica of the workload (independent
problems, weak scaling); barrier + synchronize around the timed region, time = max over ranks.

``--impl reference`` times the CPU oracle instead (bounded samples of the same workload).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import fa_inputs  # noqa: E402

METRIC = "causal GQA attn TFLOP/s (% of GB300 tensor peak); q4_0 decode KV GB/s"
DEFAULT_WORKLOAD = "prefill_gqa32x8_d128_sq2048_sk16384_f16"
DECODE_WORKLOAD = "decode_q4_0_b4_gqa32x8_d128_sk65536_f16"
# the pages' figure for the same metric and workload: 429.2 ms/call = 1.20 TFLOP/s at 16K keys,
# f16, on a Radeon 8060S (gfx1151) -- another machine's number, context only
PAGES_TFLOPS_16K_F16 = 1.20
L2_BYTES = 129 * 1000 * 1000  # GB300 L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------------------------------
# helpers (host logic, testable without a GPU)
# ------------------------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha16(files) -> str:
    import hashlib

    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "quantized_kv_cache_sm_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def measured_traffic(kernel_key: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel's sources
    changed since that capture (or no capture exists for this workload)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for ln in open(path):
        parts = ln.split()
        if len(parts) >= 5 and not ln.startswith("#") and parts[0] == kernel_key \
                and parts[4] == workload:
            if source_sha16(parts[1].split("+")) == parts[2]:
                return int(parts[3])
    return None


def kv_bytes_q4_0(w: fa_inputs.Workload) -> int:
    """Algorithmic K+V bytes one decode call reads: every visible key of every (b, kv head),
    nibbles (D/2 bytes) + fp16 scales (D/32 * 2 bytes), for K and for V."""
    keys = (w.q_pos_offset + 1) if w.causal else w.Sk
    per_row = w.D // 2 + (w.D // 32) * 2
    return 2 * w.B * w.Hkv * keys * per_row


def kv_bytes(w: fa_inputs.Workload) -> int:
    """Algorithmic K+V bytes one call of a decode workload reads (q4_0 or 16-bit cache)."""
    if w.kv_format == "q4_0":
        return kv_bytes_q4_0(w)
    keys = (w.q_pos_offset + 1) if w.causal else w.Sk
    return 2 * w.B * w.Hkv * keys * w.D * 2


def is_decode(w: fa_inputs.Workload) -> bool:
    return w.Sq == 1


def rate(w: fa_inputs.Workload, ms: float, share: float = 1.0):
    """The workload's metric for `share` of one call taking `ms`: KV GB/s for a decode workload
    (bound by HBM), TFLOP/s otherwise (bound by the tensor cores)."""
    if is_decode(w):
        return kv_bytes(w) * share / (ms * 1e-3) / 1e9, "GB/s"
    return w.flops() * share / (ms * 1e-3) / 1e12, "TFLOP/s"


def aggregate(local_ms: float, world: int) -> float:
    """Max over ranks of a per-rank time (ms); identity without a process group."""
    import torch.distributed as dist

    if world > 1 and dist.is_available() and dist.is_initialized():
        t = torch.tensor([local_ms], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return local_ms


def barrier(world: int):
    import torch.distributed as dist

    if world > 1 and dist.is_available() and dist.is_initialized():
        dist.barrier()


def parse_clocks(lines: list[str]) -> dict:
    """nvidia-smi csv rows (index, sm MHz, max sm MHz, power, active mask, hw_slowdown,
    hw_thermal, sw_thermal, sw_power_cap) -> median SM clock under load and the active reasons."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for n, val in zip(names, parts[5:9]):
            if val.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.file = None
        self.dev = device_index

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", sel], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.seek(0)
        return parse_clocks(self.file.read().splitlines())


# ------------------------------------------------------------------------------------------
# our implementation
# ------------------------------------------------------------------------------------------

def time_calls(fn, steps: int, warmup: int, flush=None, stream=None):
    """Average device time (ms) of fn() over `steps` launches, CUDA events on the launching
    stream, optional L2 flush before each timed launch (outside the events)."""
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def run_ours(args, rank, world, local_rank):
    import quantized_kv_cache_sm_gb300 as fa
    from quantized_kv_cache_sm_gb300 import build as fa_build

    fa_build.build()
    fa.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peaks_src = load_peaks()
    w = fa_inputs.WORKLOADS[args.workload]
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    if w.kv_format == "q4_0":
        k, v = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    o = torch.empty_like(q)
    rc = None
    # scratch: the decode partials, or the prefill's cut schedule (D = 128) where the
    # library plans one for this device; without it the prefill runs one work unit per CTA
    n_ws = fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset, w.causal)
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev) if n_ws > 0 else None
    if is_decode(w):
        kernel = "decode_split_kernel"
    else:
        kernel = "prefill_seg_kernel" if n_ws > 0 and w.D == 128 else "prefill_kernel"
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # inputs larger than L2 (a decode call's K/V cache) are not flushed between launches: the
    # flush's dirty lines would be written back inside the next timed launch
    in_bytes = sum((t.buf if hasattr(t, "buf") else t).numel() *
                   (t.buf if hasattr(t, "buf") else t).element_size() for t in (q, k, v))
    flush_each = in_bytes <= L2_BYTES

    def step():
        fa.fa_fwd_ex(q, k, v, o, causal=w.causal, q_pos_offset=w.q_pos_offset, scale=w.scale,
                     workspace=ws, rescale_count=rc, stream=stream)

    # warm-up
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert fa.fa_get_status() == fa.FA_OK

    # timed region: K steps, events per launch, clocks sampled throughout
    sampler = ClockSampler(local_rank)
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for a, b in evs:
        if flush_each:
            flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    kernel_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    ms = aggregate(kernel_ms, world)
    status = fa.fa_get_status()
    assert status == fa.FA_OK, fa.status_name(status)

    flops = w.flops()
    value, unit = rate(w, ms, world)
    achieved, _ = rate(w, kernel_ms)
    if is_decode(w):
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "peak_source": f"{peaks_src} HBM copy",
                "algorithmic_bytes_per_launch": kv_bytes(w)}
    else:
        peak = peaks["bf16_tflops"]  # f16 and bf16 share the dense tensor rate
        roof = {"bound": "tensor",
                "peak_source": f"{peaks_src} bf16 dense burst (f16 runs at the same rate)",
                "algorithmic_flops_per_launch": flops}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (round(value / PAGES_TFLOPS_16K_F16, 1)
                        if args.workload == DEFAULT_WORKLOAD else None),
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {
            "workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
            "D": w.D, "causal": w.causal, "q_pos_offset": w.q_pos_offset,
            "kv_format": w.kv_format,
            "l2": ("flushed before every timed launch (256 MiB write)" if flush_each else
                   f"not flushed: the inputs ({in_bytes / 1e6:.0f} MB) exceed L2"),
            "parallelism": f"replicas x{world} (independent problems per rank)",
        },
        "roofline": {
            "kernel": kernel,
            "bound": roof["bound"],
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": unit,
            "frac": round(achieved / peak, 4),
            "peak_source": roof["peak_source"],
            "traffic": measured_traffic(f"{kernel}_{w.dtype}_{w.kv_format}", w.name),
            "traffic_unit": "bytes per launch (ncu dram read + write)",
            **{k: v for k, v in roof.items() if k.startswith("algorithmic")},
        },
        "gpu_launches": args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }

    # end to end through the public API with host buffers: pinned H2D of Q, K, V, the call,
    # D2H of O, every step
    line["e2e"] = e2e_leg(fa, w, dev, stream, min(args.steps, 100), max(3, min(args.warmup, 10)),
                          world)

    if rank == 0 and not args.no_legs:
        line["decode"] = decode_leg(fa, dev, stream, peaks, peaks_src)
        line["legs"] = other_legs(fa, dev, stream, flush, peaks)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    return line


def e2e_leg(fa, w, dev, stream, steps, warmup, world):
    """End to end through the public API with host buffers: every step copies its Q, K, V from
    pinned host memory to the device, (q4_0 workloads: quantizes K and V,) runs the call and reads
    O back into pinned host memory.  Two timings on the device clock:
    - `sequential`: one step at a time, nothing overlapped (latency of a single request);
    - the reported value: consecutive steps alternate between two streams with their own device
      buffers, so step i+1's host-to-device copies run while step i computes and step i's
      read-back overlaps step i+1 -- the steady state of a serving loop; every step still moves
      all of its own bytes over the one host link, whose two directions share its bandwidth."""
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    bufs = []
    for _ in range(2):
        bf = {"q": torch.empty_like(q), "k": torch.empty_like(k), "v": torch.empty_like(v),
              "o": torch.empty_like(q), "ho": torch.empty(q.shape, dtype=q.dtype).pin_memory(),
              "ws": None}
        n = fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset, w.causal)
        if n > 0:  # decode partials, or the prefill's cut schedule
            bf["ws"] = torch.empty(n, dtype=torch.uint8, device=dev)
        bufs.append(bf)

    def step(i):
        bf, st = bufs[i % 2], streams[i % 2]
        with torch.cuda.stream(st):
            bf["q"].copy_(hq, non_blocking=True)
            bf["k"].copy_(hk, non_blocking=True)
            bf["v"].copy_(hv, non_blocking=True)
            if w.kv_format == "q4_0":
                kk, vv = fa.fa_quantize_q4_0(bf["k"]), fa.fa_quantize_q4_0(bf["v"])
            else:
                kk, vv = bf["k"], bf["v"]
            fa.fa_fwd_ex(bf["q"], kk, vv, bf["o"], causal=w.causal, q_pos_offset=w.q_pos_offset,
                         scale=w.scale, workspace=bf["ws"], stream=st)
            bf["ho"].copy_(bf["o"], non_blocking=True)

    def span(n):
        """device time (ms) of n consecutive steps, both streams joined to `stream`"""
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for st in streams:
            st.wait_stream(stream)
        for i in range(n):
            step(i)
        for st in streams:
            stream.wait_stream(st)
        e.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(e)

    span(max(2, warmup))
    seq_ms = aggregate(sum(span(1) for _ in range(steps)) / steps, world)
    ms = aggregate(span(steps) / steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = q.numel() * q.element_size()
    unit = rate(w, 1.0)[1]
    tflops = lambda t: round(rate(w, t, world)[0], 2)
    return {"value": tflops(ms), "unit": unit, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "steps alternate between two streams: step i+1's host-to-device copies "
                       "overlap step i's kernel and read-back",
            "sequential": {"value": tflops(seq_ms), "unit": unit,
                           "ms_per_step": round(seq_ms, 4)}}


def decode_leg(fa, dev, stream, peaks, peaks_src):
    w = fa_inputs.WORKLOADS[DECODE_WORKLOAD]
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    kq, vq = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    del k, v
    o = torch.empty_like(q)
    ws = torch.empty(fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset,
                                           w.causal), dtype=torch.uint8, device=dev)

    def call():
        fa.fa_fwd_ex(q, kq, vq, o, causal=True, q_pos_offset=w.q_pos_offset, scale=w.scale,
                     workspace=ws, stream=stream)

    ms = time_calls(call, 200, 10, stream=stream)
    nbytes = kv_bytes_q4_0(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "workload": w.name, "metric": "q4_0 decode KV GB/s", "value": round(gbs, 1),
        "unit": "GB/s", "ms_per_call": round(ms, 5), "kv_bytes_per_call": nbytes,
        "launches_per_call": 1,
        "roofline": {"kernel": "decode_split_kernel (one call: splits and their merge)",
                     "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peaks_src} HBM copy",
                     "traffic": measured_traffic("decode_split_kernel_f16_q4_0", w.name)},
    }


def graph_time_us(make_call, calls: int = 20, replays: int = 30) -> float:
    """Device time per call (us) of `calls` back-to-back calls replayed from one CUDA graph, as
    a serving loop runs short calls: no host launch cost between them and no L2 flush (a short
    call's inputs stay in L2).  make_call(stream) returns the call bound to that stream."""
    gs = torch.cuda.Stream()
    call = make_call(gs)
    torch.cuda.synchronize()
    with torch.cuda.stream(gs):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for _ in range(calls):
            call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gs):
        g.replay()
        e0.record(gs)
        for _ in range(replays):
            g.replay()
        e1.record(gs)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (calls * replays)


def other_legs(fa, dev, stream, flush, peaks):
    out = {}
    peak = peaks["bf16_tflops"]
    for name in ("prefill_gqa32x8_d128_sq2048_sk2048_f16", "prefill_gqa32x8_d128_sq2048_sk8192_f16",
                 "prefill_gqa32x8_d128_sq2048_sk16384_bf16",
                 "prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16",
                 "selfattn_b2_s512_h8_d64_f16"):
        w = fa_inputs.WORKLOADS[name]
        q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
        if w.kv_format == "q4_0":
            k, v = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
        o = torch.empty_like(q)
        # the call's scratch is allocated once, outside the timed loop, as for the headline leg
        n = fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset, w.causal)
        ws = torch.empty(n, dtype=torch.uint8, device=dev) if n > 0 else None

        def bound(st):
            return lambda: fa.fa_fwd_ex(q, k, v, o, causal=True, q_pos_offset=w.q_pos_offset,
                                        scale=w.scale, workspace=ws, stream=st)

        ms = time_calls(bound(stream), 50, 5, flush=flush, stream=stream)
        tf = w.flops() / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 2), "frac": round(tf / peak, 4)}
        if w.Sk <= 2048:
            # a call this short is paced by its launch as much as by the kernel: also its time
            # per call replayed from a CUDA graph (warm L2, no launch cost between calls)
            out[name]["graph_us"] = round(graph_time_us(bound), 2)
    # f16 K with a q4_0 V (independent cache formats): 16K chunked prefill and 64K decode
    w = fa_inputs.WORKLOADS["prefill_gqa32x8_d128_sq2048_sk16384_f16"]
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    vq = fa.fa_quantize_q4_0(v)
    del v
    o = torch.empty_like(q)
    # the call's scratch (the cut schedule's partial rows) is allocated once, as for the
    # headline prefill: querying and allocating it inside the timed loop adds host time that
    # can leave the GPU idle between the events
    ws = torch.empty(max(16, fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D,
                                                   w.q_pos_offset, w.causal)),
                     dtype=torch.uint8, device=dev)
    ms = time_calls(lambda: fa.fa_fwd_kv(q, k, vq, o, causal=True, workspace=ws), 50, 5,
                    flush=flush, stream=stream)
    tf = w.flops() / (ms * 1e-3) / 1e12
    out["prefill_f16k_q4_0v_gqa32x8_d128_sq2048_sk16384"] = {
        "ms": round(ms, 4), "TFLOP/s": round(tf, 2), "frac": round(tf / peak, 4)}
    del q, k, vq, o, ws
    w = fa_inputs.WORKLOADS[DECODE_WORKLOAD]
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    vq = fa.fa_quantize_q4_0(v)
    del v
    o = torch.empty_like(q)
    ws = torch.empty(fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset,
                                           w.causal), dtype=torch.uint8, device=dev)
    ms = time_calls(lambda: fa.fa_fwd_kv(q, k, vq, o, causal=True, workspace=ws), 100, 5,
                    stream=stream)
    keys = w.q_pos_offset + 1
    nbytes = w.B * w.Hkv * keys * (2 * w.D + w.D // 2 + w.D // 16)
    out["decode_f16k_q4_0v_b4_gqa32x8_d128_sk65536"] = {
        "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "kv_bytes_per_call": nbytes}
    del q, k, vq, o
    # the chunk appended to q4_0 caches inside the prefill launch, against the two-launch flow
    # (append, then the prefill over the cache): the q4_0 16K workload's last 2048 tokens are
    # the chunk, the caches hold the 14336 tokens before it
    w = fa_inputs.WORKLOADS["prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16"]
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    pos0 = w.q_pos_offset
    kc, vc = fa.q4_0_cache(w.B, w.Hkv, w.Sk, w.D), fa.q4_0_cache(w.B, w.Hkv, w.Sk, w.D)
    fa.fa_append_q4_0(k[:, :, :pos0].contiguous(), kc, 0, v[:, :, :pos0].contiguous(), vc)
    kn, vn = k[:, :, pos0:].contiguous(), v[:, :, pos0:].contiguous()
    del k, v
    o = torch.empty_like(q)
    ws = torch.empty(max(16, fa.fa_prefill_append_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk,
                                                                  w.D, pos0)),
                     dtype=torch.uint8, device=dev)
    ms_fused = time_calls(lambda: fa.fa_prefill_append_q4_0(q, kn, vn, kc, vc, pos0, o,
                                                            workspace=ws, stream=stream),
                          50, 5, flush=flush, stream=stream)

    def two_launches():
        fa.fa_append_q4_0(kn, kc, pos0, vn, vc, stream=stream)
        fa.fa_fwd_kv(q, kc, vc, o, Sk=w.Sk, causal=True, q_pos_offset=pos0, workspace=ws,
                     stream=stream)

    ms_two = time_calls(two_launches, 50, 5, flush=flush, stream=stream)
    out["prefill_append_q4_0_gqa32x8_d128_chunk2048_at14336"] = {
        "ms_fused": round(ms_fused, 4), "ms_append_then_prefill": round(ms_two, 4),
        "TFLOP/s_fused": round(w.flops() / (ms_fused * 1e-3) / 1e12, 2),
        "frac_fused": round(w.flops() / (ms_fused * 1e-3) / 1e12 / peak, 4)}
    del q, kn, vn, kc, vc, o, ws
    # the explicit (non-flash) path on the q4_0 16K chunk: dequant, S in f32, softmax, O = P V
    w = fa_inputs.WORKLOADS["prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16"]
    q, k, v = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    kq, vq = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    del k, v
    o = torch.empty_like(q)
    ws = torch.empty(fa.load().fa_explicit_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, 1, 1),
                     dtype=torch.uint8, device=dev)
    ms = time_calls(lambda: fa.fa_fwd_explicit(q, kq, vq, o, causal=True, workspace=ws), 10, 2,
                    flush=flush, stream=stream)
    tf = w.flops() / (ms * 1e-3) / 1e12
    out["explicit_q4_0_gqa32x8_d128_sq2048_sk16384_f16"] = {
        "ms": round(ms, 4), "TFLOP/s": round(tf, 2), "frac": round(tf / peak, 4),
        "note": "non-flash path: dequant, S in f32 (tcgen05 GEMM), softmax, O = P V (tcgen05 "
                "GEMM)"}
    del q, kq, vq, o, ws
    # paged q4_0 decode: the 4 x 65536-key workload through 256-token pages in shuffled order,
    # and a batch of four different lengths
    w = fa_inputs.WORKLOADS[DECODE_WORKLOAD]
    page = 256
    for name, lens in (("decode_paged_q4_0_b4_gqa32x8_d128_page256_65536x4", [65536] * 4),
                       ("decode_paged_q4_0_varlen_gqa32x8_d128_page256_65536_32768_16384_8192",
                        [65536, 32768, 16384, 8192])):
        B = len(lens)
        npages = [n // page for n in lens]
        NP = sum(npages)
        g = torch.Generator(device=dev).manual_seed(1006)
        perm = torch.randperm(NP, generator=g, device=dev).to(torch.int32)
        table = torch.zeros(B, max(npages), dtype=torch.int32, device=dev)
        at = 0
        for b, n in enumerate(npages):
            table[b, :n] = perm[at:at + n]
            at += n
        pool = torch.randn(NP, w.Hkv, page, w.D, generator=g, device=dev).to(torch.float16)
        kp = fa.fa_quantize_q4_0(pool)
        pool.normal_(generator=g)
        vp = fa.fa_quantize_q4_0(pool)
        del pool
        q = torch.randn(B, w.Hq, 1, w.D, generator=g, device=dev).to(torch.float16)
        o = torch.empty_like(q)
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)
        ws = torch.empty(fa.load().fa_decode_paged_workspace_bytes(B, w.Hq, w.Hkv, w.D, page,
                                                                  table.shape[1]),
                         dtype=torch.uint8, device=dev)
        ms = time_calls(lambda: fa.fa_decode_paged(q, kp, vp, table, sl, o, workspace=ws), 100, 5,
                        stream=stream)
        nbytes = 2 * w.Hkv * sum(lens) * (w.D // 2 + w.D // 16)
        out[name] = {"us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "kv_bytes_per_call": nbytes}
        del kp, vp, q, o, table, sl, ws
    # append a 16K-token chunk of K and V (B 4, 8 kv heads) into q4_0 caches of 64K tokens
    w = fa_inputs.WORKLOADS[DECODE_WORKLOAD]
    kn = torch.randn(w.B, w.Hkv, 16384, w.D, device=dev).to(torch.float16)
    vn = torch.randn_like(kn)
    kc, vc = fa.q4_0_cache(w.B, w.Hkv, w.Sk, w.D), fa.q4_0_cache(w.B, w.Hkv, w.Sk, w.D)
    ms = time_calls(lambda: fa.fa_append_q4_0(kn, kc, 32768, vn, vc), 20, 3, stream=stream)
    rows = 2 * w.B * w.Hkv * 16384
    nbytes = rows * (w.D * 2 + w.D // 2 + w.D // 16)
    out["append_q4_0_kv_b4_h8_d128_chunk16384"] = {
        "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    del kn, vn, kc, vc
    # q4_0 cache build: reads f16 K (D*2 B per row), writes D/2 + D/16 B per row
    w = fa_inputs.WORKLOADS[DECODE_WORKLOAD]
    _, k, _ = fa_inputs.make_qkv(w, device=dev, generate_on_device=True)
    ms = time_calls(lambda: fa.fa_quantize_q4_0(k), 20, 3, stream=stream)
    rows = w.B * w.Hkv * w.Sk
    nbytes = rows * (w.D * 2 + w.D // 2 + w.D // 16)
    out["quantize_q4_0_" + w.name.split("_", 2)[2]] = {
        "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    return out


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline key)
# ------------------------------------------------------------------------------------------

def _oracle_inputs(w):
    import numpy as np

    q, k, v = fa_inputs.make_qkv(w)
    qn = q.double().numpy()
    if w.kv_format == "q4_0":
        import oracle

        kp = oracle.quantize_q4_0(k.float().numpy())
        vp = oracle.quantize_q4_0(v.float().numpy())
        return qn, (kp, vp), np
    return qn, (k.double().numpy(), v.double().numpy()), np


def _oracle_call(w, qn, kv, rows, threads):
    import oracle

    if w.kv_format == "q4_0":
        return oracle.attention_q4_0(qn, kv[0], kv[1], causal=w.causal,
                                     q_pos_offset=w.q_pos_offset, scale=w.scale, rows=rows,
                                     threads=threads)
    return oracle.attention(qn, kv[0], kv[1], causal=w.causal, q_pos_offset=w.q_pos_offset,
                            scale=w.scale, rows=rows, threads=threads)


def _rows_flops(w, rows):
    i = rows % w.Sq
    vis = (w.q_pos_offset + i + 1) if w.causal else (i * 0 + w.Sk)
    vis = vis.clip(max=w.Sk)
    return 4 * w.D * int(vis.sum())


def cpu_baseline(w, budget_s=15.0):
    import oracle

    oracle.build()
    threads = oracle.default_threads()
    qn, kv, np = _oracle_inputs(w)
    rng = np.random.default_rng(0)
    n = w.B * w.Hq * w.Sq
    # calibrate on a small sample, then size the timed sample to the budget
    rows = np.sort(rng.choice(n, size=min(n, 2 * threads), replace=False))
    t0 = time.perf_counter()
    _oracle_call(w, qn, kv, rows, threads)
    t_cal = max(time.perf_counter() - t0, 1e-3)
    nrows = int(min(n, max(len(rows), len(rows) * budget_s / t_cal)))
    rows = np.sort(rng.choice(n, size=nrows, replace=False))
    t0 = time.perf_counter()
    _oracle_call(w, qn, kv, rows, threads)
    dt = time.perf_counter() - t0
    fl = _rows_flops(w, rows)
    value, unit = (rate(w, dt * 1e3, nrows / n) if is_decode(w) else (fl / dt / 1e12, "TFLOP/s"))
    return {"value": round(value, 6), "unit": unit, "cores": threads,
            "kind": "oracle",
            "sample": f"{nrows} random query rows of {w.name} (of {n}), all their visible keys, "
                      f"f64, {dt:.1f} s wall",
            "seconds": round(dt, 2)}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, bounded samples of the same workload."""
    import oracle

    if rank != 0:
        return None
    oracle.build()
    w = fa_inputs.WORKLOADS[args.workload]
    threads = oracle.default_threads()
    qn, kv, np = _oracle_inputs(w)
    n = w.B * w.Hq * w.Sq
    rng = np.random.default_rng(1)
    # size each step so the whole run stays within a few minutes
    cal = np.sort(rng.choice(n, size=min(n, 2 * threads), replace=False))
    t0 = time.perf_counter()
    _oracle_call(w, qn, kv, cal, threads)
    t_row = max(time.perf_counter() - t0, 1e-4) / len(cal)
    per_step_s = min(1.0, 150.0 / max(1, args.steps + args.warmup))
    rows_per_step = int(max(1, min(n, per_step_s / t_row)))
    for _ in range(args.warmup):
        _oracle_call(w, qn, kv, np.sort(rng.choice(n, size=rows_per_step, replace=False)),
                     threads)
    tot_fl, tot_t = 0, 0.0
    for _ in range(args.steps):
        rows = np.sort(rng.choice(n, size=rows_per_step, replace=False))
        t0 = time.perf_counter()
        _oracle_call(w, qn, kv, rows, threads)
        tot_t += time.perf_counter() - t0
        tot_fl += _rows_flops(w, rows)
    # a decode workload: the share of the call's KV bytes behind the sampled query rows
    value, unit = (rate(w, tot_t * 1e3 / args.steps, rows_per_step / n) if is_decode(w)
                   else (tot_fl / tot_t / 1e12, "TFLOP/s"))
    sample = (f"{rows_per_step} random query rows of {w.name} per step (of {n}), all their "
              f"visible keys, f64")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq,
                   "Sk": w.Sk, "D": w.D, "kv_format": w.kv_format,
                   "sample_rows_per_step": rows_per_step},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of the run; must equal WORLD_SIZE when launched by torchrun")
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--no-legs", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {world}: launch one process per GPU "
                 "(torchrun --nproc-per-node N) for N > 1")
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if args.impl == "reference":
            if rank != 0:
                return 0
            world_for_line = world
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
            world_for_line = world
    else:
        world_for_line = 1

    if args.impl == "reference":
        line = run_reference(args, 0, world_for_line)
    else:
        line = run_ours(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
