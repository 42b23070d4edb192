#!/usr/bin/env python
"""Benchmark of the RoPE hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic inputs:
  1. in-place partial interleave RoPE, x bf16 [4,4096,32,128], slice [64,128),
     cos/sin fp32 [1,4096,1,64];
  2. cache RoPE, NeoX, bf16, 16384 tokens, 32 query + 8 key heads of 128;
  3. cache RoPE, GPT-J, fp16, 8192 tokens (8 x 1024), 16 + 16 heads of 256, R = 64;
  4. cache mrope [16,24,24], NeoX, bf16, 32768 tokens, 28 + 4 heads of 128.
Metric: achieved HBM GB/s of algorithmic bytes (read + write of rotated
elements, cos/sin or one gathered cache row per token, positions), plus
tokens/s, against the measured peak bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores on bounded samples of the same workloads.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RoPE achieved HBM GB/s and tokens/s on 1 GB300 vs peak-bandwidth roofline"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
E2E_WINDOW = 40  # steps per sub-window of the end-to-end region
WORKLOAD_NAME = ("rope hot path: inplace bf16x/f32cs [4,4096,32,128] slice[64,128) + cache NeoX bf16 16384tok "
                 "32q8k h128 + cache GPT-J f16 8192tok 16q16k h256 r64 + mrope[16,24,24] NeoX bf16 32768tok "
                 "28q4k h128")


# ----------------------------------------------------------------------------
# workloads and byte model
# ----------------------------------------------------------------------------

def build_workloads():
    import workloads as W
    return [W.inplace_bf16_mixed(), W.cache_neox_bf16(), W.cache_gptj_f16_partial(), W.mrope_neox_bf16()]


def algorithmic_bytes(case) -> int:
    """Read + write of rotated elements, cos/sin (or one gathered cache row per
    token), positions.  Pass-through columns are never touched and not counted.
    Fused QKV operator: read of qkv, write of q_out and of the cached K/V rows,
    one gathered cache row per token, gammas and the int64 metadata."""
    if hasattr(case, "qkv"):
        e = case.qkv.element_size()
        T, D = case.tokens, case.head_size
        cached = int((case.slot_mapping >= 0).sum())
        meta = (case.seq_lens.numel() + case.query_start_loc.numel() + case.slot_mapping.numel()) * 8
        return (T * (case.nq + case.nk + case.nv) * D * e + T * case.nq * D * e + cached * (case.nk + case.nv) * D * e
                + T * D * e + 2 * D * e + meta)
    if hasattr(case, "x"):
        B, S, N, D = case.x.shape
        L = D if (case.start, case.end) == (0, 0) else case.end - case.start
        xb = B * S * N * L * case.x.element_size() * 2
        return xb + 2 * case.cos.numel() * case.cos.element_size()
    T = case.tokens
    heads = (case.query.shape[1] + case.key.shape[1]) // case.head_size
    e = case.query.element_size()
    return (T * heads * case.rotary_dim * e * 2 + T * case.rotary_dim * e
            + case.positions.numel() * case.positions.element_size())


def kernel_label(case) -> str:
    return case.name


# ----------------------------------------------------------------------------
# distributed helpers
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []  # (monotonic time, sm, sm_max, power, hw, hw_thermal, sw_thermal, sw_power)
        self.proc = None
        self.thread = None
        ident = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            u = getattr(props, "uuid", None)
            if u is not None:
                s = str(u)
                ident = s if s.startswith("GPU-") else "GPU-" + s
        except Exception:  # noqa: BLE001
            ident = None
        self.ident = ident

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50"]
        if self.ident:
            cmd += ["-i", self.ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            flags = [p.lower() == "active" for p in parts[4:8]]
            self.samples.append((time.monotonic(), sm, smax, parts[2], *flags))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed_region"
        if not inside:
            inside = self.samples
            window = "whole_run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in inside:
            for n, f in zip(names, s[4:8]):
                if f:
                    reasons.add(n)
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------
# roofline helpers
# ----------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_tokens(text: str) -> str:
    """C/CUDA source with comments removed and whitespace runs collapsed (the
    sources hold no string literal containing a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


# The C ABI's argument checks: host code that runs before any launch and
# changes neither a kernel nor its launch configuration.
ARGUMENT_CHECKS = "rope_api.cu"


def kernel_source_hash() -> str:
    """sha256[:16] of the kernel sources' code (comments and layout excluded):
    the kernels, their launchers and launch bookkeeping, not the argument
    checks; so that a profile stays tied to the code it measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_rope_positional_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name != ARGUMENT_CHECKS:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + source_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(label: str):
    """DRAM bytes per launch from the committed ncu summary of ``label``, or
    None when there is none or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"^kernel_source_sha256_16:\s*(\S+)", text, re.M)
    if not src or src.group(1) != kernel_source_hash():
        return None
    m = re.search(r"^%s:\s*([0-9]+)" % re.escape(label), text, re.M)
    return int(m.group(1)) if m else None


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def step_config(total_bytes: int, step_tokens: int) -> dict:
    """The ``config`` of the bench line, the same for both arms: the step's
    workload, its algorithmic bytes and tokens, the L2 rule and the parallelism."""
    return {"workload": WORKLOAD_NAME, "bytes_per_step": total_bytes, "tokens_per_step": step_tokens,
            "l2": "inputs larger than L2: %.2f GB per step vs %d MB L2; each kernel's buffers are "
                  "evicted by the others between its launches" % (total_bytes / 1e9, L2_BYTES >> 20),
            "parallelism": "replicas of the per-GPU workload (weak scaling), no collective"}


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)  # before the process group, so its collectives use this GPU
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from transformer_rope_positional_gb300 import build as B
    B.build()
    import transformer_rope_positional_gb300 as R

    cases = build_workloads()
    step_bytes = [algorithmic_bytes(c) for c in cases]
    step_tokens = sum(c.tokens for c in cases)
    total_bytes = sum(step_bytes)

    # device-resident inputs and prepared launches
    dev_tensors = []
    calls = []
    for c in cases:
        if hasattr(c, "x"):
            x, cs, sn = c.x.to(dev), c.cos.to(dev), c.sin.to(dev)
            dev_tensors.append((x, cs, sn))
            calls.append(R.prepare_inplace_partial(x, cs, sn, c.rotary_mode, [c.start, c.end]))
        else:
            p, q, k, cc = c.positions.to(dev), c.query.to(dev), c.key.to(dev), c.cache.to(dev)
            dev_tensors.append((p, q, k, cc))
            calls.append(R.prepare_with_sin_cos_cache(p, q, k, cc, c.head_size, c.rotary_dim, c.is_neox,
                                                      c.mrope_section))
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        for call in calls:
            call()
    torch.cuda.synchronize()
    if R.get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    K = args.steps
    nk = len(calls)
    # ---- timed region: K steps, events only at its two ends
    launches0 = R.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t_host0 = time.monotonic()
    # keep the GPU busy while the host queues the timed steps (outside the timed region)
    torch.cuda._sleep(int(4e6))
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(K):
        for call in calls:
            call()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    t_host1 = time.monotonic()
    launches = R.launch_count() - launches0
    total_ms = start.elapsed_time(end)

    # ---- per-kernel region: the same steps with an event between launches
    # (each event costs about a microsecond, so these durations are upper bounds)
    Kk = min(K, args.kernel_steps)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(Kk)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(4e6))
    for s_ in range(Kk):
        ev = events[s_]
        for i, call in enumerate(calls):
            ev[i].record()
            call()
        ev[nk].record()
    torch.cuda.synchronize()
    per_kernel_ms = [[events[s_][i].elapsed_time(events[s_][i + 1]) for s_ in range(Kk)] for i in range(nk)]

    # ---- rows beyond the hot path (backward, half mode), each timed cold: a
    # large cache-op launch runs between two of them and flushes their data from L2
    specs = operator_specs(cases, dev_tensors)
    next_rows = time_next_rows(specs, calls, Kk)
    streams = time_streams(specs)
    copy_us = {b: copy_stream_us(b) for b in set(step_bytes) | {nb for _, nb, _, _ in specs}}
    del specs
    for entry in next_rows:
        entry.update(streams.get(entry["workload"], {}))
        if "stream_us" in entry:
            entry["copy_stream_us"] = round(copy_us[entry["bytes_per_launch"]], 3)
            entry["vs_copy"] = round(copy_us[entry["bytes_per_launch"]] / entry["stream_us"], 4)
    small = time_small_rows(dev)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    ms_step_local = total_ms / K
    ms_step = max_over_ranks(ms_step_local, world, dev)
    value = world * total_bytes / (ms_step * 1e-3) / 1e9
    tokens_per_s = world * step_tokens / (ms_step * 1e-3)

    peak, peak_kind = measured_peak()
    kernels = []
    for c, b, ms in zip(cases, step_bytes, per_kernel_ms):
        avg = sum(ms) / len(ms)
        kernels.append({"workload": kernel_label(c), "bytes_per_launch": b, "launches": len(ms),
                        "avg_us": round(avg * 1e3, 3),
                        "median_us": round(statistics.median(ms) * 1e3, 3),
                        "gbs": round(b / (avg * 1e-3) / 1e9, 1), "frac_of_peak": round(b / (avg * 1e-3) / 1e9 / peak, 4),
                        "tokens": c.tokens, **streams.get(kernel_label(c), {}),
                        "copy_stream_us": round(copy_us[b], 3),
                        "vs_copy": round(copy_us[b] / streams[kernel_label(c)]["stream_us"], 4)})
    dom = max(range(nk), key=lambda i: sum(per_kernel_ms[i]))
    dom_label = kernel_label(cases[dom])
    dom_avg_s = sum(per_kernel_ms[dom]) / Kk * 1e-3
    achieved_evented = step_bytes[dom] / dom_avg_s / 1e9
    # average launch duration of the dominant kernel in a stream of its own
    # launches (the kernel's own time, as ncu's gpu__time_duration measures it);
    # the evented figure also carries the launch latency after each event
    dom_stream_us = streams[dom_label]["stream_us"]
    achieved = step_bytes[dom] / (dom_stream_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dom_label, "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                if peak_kind == "measured" else "fallback", "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(dom_label),
                "algorithmic_bytes": step_bytes[dom],
                "method": "average launch duration over 200 back-to-back launches on rotating buffer copies "
                          "(>3x L2 of other data between reuses), CUDA events at both ends",
                "launch_us": dom_stream_us,
                "achieved_evented": round(achieved_evented, 1), "frac_evented": round(achieved_evented / peak, 4)}

    e2e = run_e2e(args, cases, dev_tensors, calls, world, dev, total_bytes)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cases, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtypes": "bf16,f16 (x: bf16; cos/sin f32)",
                "data": "synthetic (seeded SplitMix64 + Box-Muller N(0,1); cos/sin tables from base 1e4 / 1e6)",
                "tokens_per_s": round(tokens_per_s, 1),
                "config": step_config(total_bytes, step_tokens),
                "per_kernel": kernels, "next_rows": next_rows, "small_rows": small, "roofline": roofline, "e2e": e2e,
                "gpu_launches": launches,
                "clocks": clocks, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


DECODE_TOKENS = (1, 8, 64, 256)
GRAPH_LAUNCHES = 100


def small_workloads():
    """Latency-bound calls: the small in-place workload (slice [16,48), the
    whole-D [0,0] variant and the [8,8] no-op), decode-sized batches of the
    cache operator on the head layouts of the three cache workloads, and the
    fused QKV op on decode batches (one new token per sequence)."""
    import workloads as W
    out = [W.inplace_f32_small(v) for v in ("slice", "full", "noop")]
    for T in DECODE_TOKENS:
        out.append(W.cache_case("decode_rope_neox_bf16_%dtok_32q8k_h128" % T, 20, T, 32, 8, 128, 128, 32768,
                                torch.bfloat16, True))
        out.append(W.cache_case("decode_rope_gptj_f16_%dtok_16q16k_h256_r64" % T, 21, T, 16, 16, 256, 64, 65536,
                                torch.float16, False))
        out.append(W.cache_case("decode_mrope_neox_bf16_%dtok_28q4k_h128_s16_24_24" % T, 22, T, 28, 4, 128, 128,
                                40960, torch.bfloat16, True, base=1e6, mrope_section=[16, 24, 24]))
    for T in DECODE_TOKENS:  # the fused op on T decode requests, one new token each
        ctx = W.uniform_int(W.stream_seed(23, 3), T, 16, 1024).tolist()
        out.append(W.qkv_case("decode_qkv_rmsnorm_rope_bf16_%dseq_32q8k8v_h128" % T, 23, [1] * T, ctx, 32, 8, 8, 128,
                              16, torch.bfloat16))
    return out


def latency_us(enqueue, reps: int = 200):
    """(median evented us, us per launch replayed from a CUDA graph) of a call
    that ``enqueue()`` puts on the current stream.  Evented: each call between
    two events, all queued behind a sleep kernel so that the host's own time
    per call never shows.  Graph: GRAPH_LAUNCHES calls captured once, the graph
    replayed 20 times between two events (the device's time per call, launch
    overhead included, with no host in the loop)."""
    for _ in range(5):
        enqueue()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda._sleep(int(7e4 * reps))  # about 35 us of queueing time per call
    for e0, e1 in ev:
        e0.record()
        enqueue()
        e1.record()
    torch.cuda.synchronize()
    evented = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(GRAPH_LAUNCHES):
                enqueue()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(20):
        graph.replay()
    g1.record()
    torch.cuda.synchronize()
    return evented, g0.elapsed_time(g1) / (20 * GRAPH_LAUNCHES) * 1e3


def host_us(call, n: int = 1000) -> float:
    """Host microseconds per call of ``call`` (binding and C ABI: argument checks,
    marshalling and the launch itself), n calls in a row, the GPU synchronised
    after them."""
    for _ in range(10):
        call()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(n):
        call()
    us = (time.perf_counter() - h0) / n * 1e6
    torch.cuda.synchronize()
    return round(us, 2)


def time_small_rows(dev):
    """Per-call latency of the small workloads, next to the floor of an empty
    kernel launch timed the same two ways."""
    import transformer_rope_positional_gb300 as R
    floor_ev, floor_graph = latency_us(lambda: torch.cuda._sleep(0))
    rows = []
    for c in small_workloads():
        if hasattr(c, "qkv"):
            t = [v.to(dev) for v in (c.qkv, c.q_gamma, c.k_gamma, c.cache, c.seq_lens, c.query_start_loc,
                                     c.slot_mapping, c.q_out, c.k_cache, c.v_cache)]
            enqueue = (lambda t=t, c=c: R.qkv_rmsnorm_rope_cache(t[0], c.nq, c.nk, c.nv, t[1], t[2], c.eps, *t[3:]))
            prepared = R.prepare_qkv_rmsnorm_rope_cache(t[0], c.nq, c.nk, c.nv, t[1], t[2], c.eps, *t[3:])
        elif hasattr(c, "x"):
            t = (c.x.to(dev), c.cos.to(dev), c.sin.to(dev))
            enqueue = (lambda t=t, c=c: R.rope_inplace_partial(t[0], t[1], t[2], c.rotary_mode, [c.start, c.end]))
            prepared = R.prepare_inplace_partial(t[0], t[1], t[2], c.rotary_mode, [c.start, c.end])
        else:
            t = (c.positions.to(dev), c.query.to(dev), c.key.to(dev), c.cache.to(dev))
            enqueue = (lambda t=t, c=c: R.rope_with_sin_cos_cache(t[0], t[1], t[2], t[3], c.head_size, c.rotary_dim,
                                                                 c.is_neox, c.mrope_section))
            prepared = R.prepare_with_sin_cos_cache(t[0], t[1], t[2], t[3], c.head_size, c.rotary_dim, c.is_neox,
                                                    c.mrope_section)
        torch.cuda.synchronize()
        l0 = R.launch_count()
        enqueue()
        torch.cuda.synchronize()
        launches = R.launch_count() - l0
        row = {"workload": c.name, "tokens": c.tokens, "launches_per_call": launches,
               "host_us_per_call": host_us(enqueue), "host_us_per_prepared_call": host_us(prepared)}
        if launches == 0:  # the no-op: the call returns before any CUDA call
            row["bytes_per_call"] = 0
            rows.append(row)
            continue
        nbytes = algorithmic_bytes(c)
        ev, gr = latency_us(enqueue)
        row.update({"bytes_per_call": nbytes, "evented_us": round(ev, 3), "graph_us": round(gr, 3),
                    "tokens_per_s": round(c.tokens / (gr * 1e-6), 1), "gbs": round(nbytes / (gr * 1e-6) / 1e9, 2),
                    "floor_over_evented": round(floor_ev / ev, 3), "floor_over_graph": round(floor_graph / gr, 3)})
        rows.append(row)
        del t
    return {"empty_kernel_floor": {"evented_us": round(floor_ev, 3), "graph_us": round(floor_graph, 3),
                                   "kernel": "torch.cuda._sleep(0), a kernel that returns at once"},
            "method": "evented: median of 200 calls each between two events, queued behind a sleep kernel; "
                      "graph: %d calls replayed from one CUDA graph, per call" % GRAPH_LAUNCHES,
            "rows": rows}


def copies(*ts, n):
    """The given tensors, then n - 1 clones of them (the originals come first)."""
    return [ts] + [tuple(t.clone() for t in ts) for _ in range(n - 1)]


def operator_specs(cases, dev_tensors):
    """Every operator timed by the bench, as (label, algorithmic bytes per
    launch, factory, flush index): factory(n) prepares n launches on n copies of
    the operator's buffers (the first on the step's own tensors); read-only
    tables (positions, cos/sin, gammas) are shared, as in serving.  The first
    four are the hot-path kernels of the step, the rest the rows beyond it: the
    in-place operator's backward and half mode, the V2 cache operator with the
    interleaved mrope splice, with separate outputs and on strided views of a
    fused QKV buffer, and the fused QKV split + RMSNorm + RoPE + paged cache
    write.  The flush index names the step kernel (NeoX 1 or mrope 3) whose
    launch on other buffers evicts a row's data between its evented launches."""
    import transformer_rope_positional_gb300 as R
    import workloads as W
    inplace, neox, gptj, mrope = cases
    x, cs, sn = dev_tensors[0]
    p3, q3, k3, c3 = dev_tensors[1]
    p4, q4, k4, c4 = dev_tensors[2]
    p5, q5, k5, c5 = dev_tensors[3]
    ib = algorithmic_bytes(inplace)
    sl = [inplace.start, inplace.end]
    specs = [(kernel_label(inplace), ib, lambda n: [R.prepare_inplace_partial(t[0], cs, sn, 1, sl)
                                                     for t in copies(x, n=n)], None)]
    for c, (p, q, k, cc) in ((neox, dev_tensors[1]), (gptj, dev_tensors[2]), (mrope, dev_tensors[3])):
        specs.append((kernel_label(c), algorithmic_bytes(c),
                      lambda n, c=c, p=p, q=q, k=k, cc=cc: [
                          R.prepare_with_sin_cos_cache(p, t[0], t[1], cc, c.head_size, c.rotary_dim, c.is_neox,
                                                       c.mrope_section) for t in copies(q, k, n=n)], None))
    tag = inplace.name.split("_", 1)[1]
    specs.append(("inplace_backward_interleave_" + tag, ib, lambda n: [
        R.prepare_inplace_partial(t[0], cs, sn, 1, sl, backward=True) for t in copies(x, n=n)], 1))
    specs.append(("inplace_half_forward_" + tag, ib, lambda n: [
        R.prepare_inplace_partial(t[0], cs, sn, 0, sl) for t in copies(x, n=n)], 3))
    specs.append(("mrope_interleaved_splice_" + mrope.name.split("_", 1)[1], algorithmic_bytes(mrope), lambda n: [
        R.prepare_with_sin_cos_cache(p5, t[0], t[1], c5, mrope.head_size, mrope.rotary_dim, True,
                                     mrope.mrope_section, cache_mode=1) for t in copies(q5, k5, n=n)], 1))
    # NeoX workload, R == head size: no pass-through columns to copy
    qo, ko = torch.empty_like(q3), torch.empty_like(k3)
    specs.append(("rope_neox_out_of_place_" + neox.name.split("_", 2)[2], algorithmic_bytes(neox), lambda n: [
        R.prepare_with_sin_cos_cache(p3, t[0], t[1], c3, neox.head_size, neox.rotary_dim, True,
                                     query_out=t[2], key_out=t[3]) for t in copies(q3, k3, qo, ko, n=n)], 3))
    # GPT-J workload on q/k views of a fused [T, (16+16+16)*256] QKV buffer
    wq, wk = q4.shape[1], k4.shape[1]
    qkv4 = torch.empty(gptj.tokens, wq + 2 * wk, dtype=q4.dtype, device=q4.device)
    qkv4[:, :wq].copy_(q4)
    qkv4[:, wq:wq + wk].copy_(k4)
    specs.append(("rope_gptj_fused_qkv_views_" + gptj.name.split("_", 2)[2], algorithmic_bytes(gptj), lambda n: [
        R.prepare_with_sin_cos_cache(p4, t[0][:, :wq], t[0][:, wq:wq + wk], c4, gptj.head_size, gptj.rotary_dim,
                                     False) for t in copies(qkv4, n=n)], 1))
    # mixed prefill/decode batch
    qc = W.qkv_rmsnorm_rope_bf16()
    qt = [t.to(q3.device) for t in (qc.qkv, qc.q_gamma, qc.k_gamma, qc.cache, qc.seq_lens, qc.query_start_loc,
                                    qc.slot_mapping, qc.q_out, qc.k_cache, qc.v_cache)]
    specs.append((qc.name, algorithmic_bytes(qc), lambda n: [
        R.prepare_qkv_rmsnorm_rope_cache(t[0], qc.nq, qc.nk, qc.nv, qt[1], qt[2], qc.eps, qt[3], qt[4], qt[5],
                                         qt[6], t[1], t[2], t[3])
        for t in copies(qt[0], qt[7], qt[8], qt[9], n=n)], 3))
    return specs


def time_streams(specs, launches=200):
    """Steady-state time per launch of each operator in a stream of its own
    launches: back to back (launches overlap through programmatic stream
    serialization, as in the step), with events only at the two ends, cycling
    over enough copies of the operator's buffers that at least 3x the L2
    capacity of other data passes between two uses of one copy."""
    peak, _ = measured_peak()
    out = {}
    for label, nbytes, factory, _ in specs:
        us, n = stream_us(factory, nbytes, launches)
        out[label] = {"stream_us": round(us, 3), "stream_frac_of_peak": round(nbytes / (us * 1e-6) / 1e9 / peak, 4),
                      "stream_buffer_sets": n}
    return out


def copy_stream_us(nbytes: int, launches: int = 200) -> float:
    """Microseconds per launch of the device copy that defines the peak
    (``copy_`` of bf16 buffers, nbytes / 2 read and nbytes / 2 written), timed
    as stream_us times an operator: back to back over rotating buffer copies."""
    n = max(1, nbytes // 4)  # bf16 elements per buffer
    return stream_us(lambda k: [lambda s=torch.empty(n, dtype=torch.bfloat16, device="cuda"),
                                       d=torch.empty(n, dtype=torch.bfloat16, device="cuda"): d.copy_(s)
                                for _ in range(k)], 4 * n, launches)[0]


def stream_us(factory, nbytes, launches=200):
    """(microseconds per launch, buffer copies) of back-to-back launches cycling
    over enough copies that 3x L2 of other data passes between two uses."""
    import math
    n = max(2, math.ceil(3 * L2_BYTES / nbytes) + 1)
    calls = factory(n)
    for call in calls:
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e6))
    e0.record()
    for j in range(launches):
        calls[j % n]()
    e1.record()
    torch.cuda.synchronize()
    del calls
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / launches * 1e3, n


def time_next_rows(specs, calls, steps):
    """Per-launch time of the rows beyond the hot path on the hot path's own
    workloads, each launch between two events and followed by a launch of a
    large step kernel on other buffers, so every timed launch starts cold."""
    rows = [(name, b, factory(1)[0], calls[flush]) for name, b, factory, flush in specs if flush is not None]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(rows))] for _ in range(steps)]
    for _ in range(3):
        for _, _, call, flush in rows:
            call()
            flush()
    torch.cuda.synchronize()
    torch.cuda._sleep(int(4e6))
    for s_ in range(steps):
        for i, (_, _, call, flush) in enumerate(rows):
            ev[s_][2 * i].record()
            call()
            ev[s_][2 * i + 1].record()
            flush()
    torch.cuda.synchronize()
    peak, _ = measured_peak()
    out = []
    for i, (name, b, _, _) in enumerate(rows):
        ms = [ev[s_][2 * i].elapsed_time(ev[s_][2 * i + 1]) for s_ in range(steps)]
        avg = sum(ms) / len(ms)
        out.append({"workload": name, "bytes_per_launch": b, "launches": steps, "avg_us": round(avg * 1e3, 3),
                    "gbs": round(b / (avg * 1e-3) / 1e9, 1), "frac_of_peak": round(b / (avg * 1e-3) / 1e9 / peak, 4)})
    return out


def run_e2e(args, cases, dev_tensors, calls, world, dev, total_bytes):
    """Host buffers in, host buffers out: per step every input of every
    workload is copied from pinned host memory, the operators run through the
    public API, and the results are copied back to pinned host memory.  Copies
    in, kernels and copies out run on three streams with two sets of buffers,
    so the copies of one workload overlap the kernels and copies of the others
    (and of the next step), as a serving loop would pipeline them."""
    import transformer_rope_positional_gb300 as R
    compute = torch.cuda.current_stream()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def device_set(src):
        return [tuple(t.clone() for t in group) for group in src]

    def prepared(c, dt):
        if hasattr(c, "x"):
            return R.prepare_inplace_partial(dt[0], dt[1], dt[2], c.rotary_mode, [c.start, c.end], stream=compute)
        return R.prepare_with_sin_cos_cache(dt[0], dt[1], dt[2], dt[3], c.head_size, c.rotary_dim, c.is_neox,
                                            c.mrope_section, stream=compute)

    sets = [dev_tensors, device_set(dev_tensors)]
    set_calls = [calls, [prepared(c, dt) for c, dt in zip(cases, sets[1])]]
    host_in, host_out = [], [[], []]
    h2d = d2h = 0
    for c in cases:
        ins = ([c.x, c.cos, c.sin] if hasattr(c, "x") else [c.positions, c.query, c.key, c.cache])
        host_in.append([t.pin_memory() for t in ins])
        outs = [0] if hasattr(c, "x") else [1, 2]  # indices of the device tensors read back
        for b in range(2):
            host_out[b].append([(torch.empty_like(ins[j]).pin_memory(), j) for j in outs])
        h2d += sum(t.numel() * t.element_size() for t in ins)
        d2h += sum(ins[j].numel() * ins[j].element_size() for j in outs)
    n = len(cases)
    ev = {key: [[torch.cuda.Event() for _ in range(n)] for _ in range(2)] for key in ("in", "run", "out")}

    def step(s_):
        b = s_ % 2
        for i in range(n):
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(ev["out"][b][i])  # the previous readback of this buffer set is done
                for h, d in zip(host_in[i], sets[b][i]):
                    d.copy_(h, non_blocking=True)
                ev["in"][b][i].record(h2d_stream)
            compute.wait_event(ev["in"][b][i])
            set_calls[b][i]()
            ev["run"][b][i].record(compute)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev["run"][b][i])
                for h, j in host_out[b][i]:
                    h.copy_(sets[b][i][j], non_blocking=True)
                ev["out"][b][i].record(d2h_stream)

    # its own step count (about a second of copies), whatever --steps is: the
    # host copy path stalls now and then, and a short region would be a lottery
    K = max(3, args.e2e_steps)
    window = min(E2E_WINDOW, K)
    for s_ in range(max(2, min(args.warmup, 4))):
        step(s_)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # the GPU waits (outside the timed region) while the host queues the timed
    # steps, so a pause of the host thread cannot leave the copy engines idle
    torch.cuda._sleep(int(4e7))
    e0.record(compute)
    h2d_stream.wait_stream(compute)
    d2h_stream.wait_stream(compute)
    # sub-window marks: the readbacks of every window-th step done
    marks = []
    for s_ in range(K):
        step(s_)
        if (s_ + 1) % window == 0:
            marks.append(torch.cuda.Event(enable_timing=True))
            marks[-1].record(d2h_stream)
    compute.wait_stream(d2h_stream)
    e1.record(compute)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    ends = [0.0] + [e0.elapsed_time(m) for m in marks]
    windows = [round(world * total_bytes * window / ((b - a) * 1e-3) / 1e9, 1) for a, b in zip(ends, ends[1:])]
    ms = max_over_ranks(ms, world, dev)
    return {"value": round(world * total_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "steps": K,
            "path": "pinned host -> device copies, C-ABI calls, device -> pinned host copies on three streams "
                    "with double-buffered device and host buffers",
            "windows_gbs": windows, "median_window_gbs": statistics.median(windows) if windows else None,
            "window_steps": window,
            "note": "value: every timed step, the host copy path's occasional 30-60 ms stalls included; "
                    "windows_gbs: rank 0's rate per window of window_steps steps"}


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(case, tokens: int):
    """The first ``tokens`` tokens of a workload as a standalone case."""
    import workloads as W
    if hasattr(case, "x"):
        B, S, N, D = case.x.shape
        if tokens >= S:  # whole batches (b, s order)
            nb = min(B, tokens // S)
            x = case.x[:nb].contiguous()
            cos = case.cos[:nb].contiguous() if case.cos.shape[0] != 1 else case.cos
            sin = case.sin[:nb].contiguous() if case.sin.shape[0] != 1 else case.sin
            return W.InplaceCase(case.name, x, cos, sin, case.start, case.end)
        s = max(1, tokens)
        x = case.x[:1, :s].contiguous()
        cos = case.cos[:1, :s].contiguous() if case.cos.shape[1] != 1 else case.cos[:1]
        sin = case.sin[:1, :s].contiguous() if case.sin.shape[1] != 1 else case.sin[:1]
        return W.InplaceCase(case.name, x, cos, sin, case.start, case.end)
    t = max(1, min(case.tokens, tokens))
    return W.CacheCase(case.name, case.positions[..., :t].contiguous(), case.query[:t].contiguous(),
                       case.key[:t].contiguous(), case.cache, case.head_size, case.rotary_dim, case.is_neox,
                       case.mrope_section)


def run_oracle(case):
    """The oracle on one workload; returns its outputs (x, or (query, key))."""
    import oracle
    if hasattr(case, "x"):
        return oracle.inplace_partial_rotary_mul(case.x, case.cos, case.sin, case.start, case.end)
    return oracle.rope_with_sin_cos_cache(case.positions, case.query, case.key, case.cache, case.head_size,
                                          case.is_neox, case.mrope_section)[:2]


def _bounds(n: int, parts: int):
    parts = max(1, min(parts, n))
    return [(n * i // parts, n * (i + 1) // parts) for i in range(parts)]


def oracle_shards(case, parts: int):
    """A workload cut into ``parts`` contiguous token ranges (in-place op:
    ranges of S, with cos/sin cut alongside unless broadcast over S; cache op:
    ranges of tokens), each a standalone workload.  Tokens are independent
    under both operators, so the shards' outputs put together are the whole
    workload's."""
    import workloads as W
    if hasattr(case, "x"):
        S = case.x.shape[1]
        out = []
        for s0, s1 in _bounds(S, parts):
            cut = (lambda t: t[:, s0:s1].contiguous()) if case.cos.shape[1] != 1 else (lambda t: t)
            out.append(W.InplaceCase(case.name, case.x[:, s0:s1].contiguous(), cut(case.cos), cut(case.sin),
                                     case.start, case.end))
        return out
    return [W.CacheCase(case.name, case.positions[..., t0:t1].contiguous(), case.query[t0:t1].contiguous(),
                        case.key[t0:t1].contiguous(), case.cache, case.head_size, case.rotary_dim, case.is_neox,
                        case.mrope_section) for t0, t1 in _bounds(case.tokens, parts)]


def run_oracle_threaded(case, threads: int, pool=None):
    """The oracle on ``threads`` token shards of ``case`` at once, outputs put
    back together.  A thin driver: the oracle's arithmetic is unchanged, each
    shard is one plain call, and the C code runs without the GIL."""
    import concurrent.futures as cf
    shards = oracle_shards(case, threads)
    own = pool is None
    pool = pool or cf.ThreadPoolExecutor(max_workers=threads)
    try:
        outs = list(pool.map(run_oracle, shards))
    finally:
        if own:
            pool.shutdown()
    if hasattr(case, "x"):
        return torch.cat(outs, 1)
    return torch.cat([o[0] for o in outs], 0), torch.cat([o[1] for o in outs], 0)


def usable_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu() -> dict:
    """nproc, the cores this process may use, and the CPU model (lscpu, else
    /proc/cpuinfo)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "usable_cores": usable_cores(), "cpu_model": model or "unknown",
            "machine": platform.machine()}


def time_oracle(samples, threads: int = 1):
    """Seconds of oracle work over the samples: one thread in order, or every
    sample's token shards spread over ``threads`` threads (shards cut before
    the clock starts)."""
    if threads <= 1:
        t0 = time.perf_counter()
        for s in samples:
            run_oracle(s)
        return time.perf_counter() - t0
    import concurrent.futures as cf
    shards = [sh for s in samples for sh in oracle_shards(s, 4 * threads)]
    with cf.ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        list(pool.map(run_oracle, shards))
        return time.perf_counter() - t0


def sized_samples(cases, budget_s: float, threads: int = 1):
    """Per-workload token samples whose oracle time on ``threads`` threads adds
    up to about budget_s, keeping each workload's share of the step's bytes."""
    probe = [oracle_sample(c, 64) for c in cases]
    t = time_oracle(probe)
    probe_bytes = sum(algorithmic_bytes(p) for p in probe)
    rate = probe_bytes / max(t, 1e-6) * threads
    total = sum(algorithmic_bytes(c) for c in cases)
    frac = min(1.0, budget_s * rate / total)
    return [oracle_sample(c, max(1, int(c.tokens * frac))) for c in cases], frac


def _sample_text(samples, cases, threads):
    b = sum(algorithmic_bytes(s) for s in samples)
    tok = sum(s.tokens for s in samples)
    total_tok = sum(c.tokens for c in cases)
    how = "one thread" if threads == 1 else "%d threads over token shards" % threads
    return ("leading tokens of each of the four workloads, %d of the step's %d tokens (%.1f%%), %d bytes; "
            "binary64 scalar C oracle, %s" % (tok, total_tok, 100 * tok / total_tok, b, how))


def cpu_baseline(cases, budget_s: float):
    """The oracle on the host cores: on every usable core (token shards, one
    thread per core; the headline figure) and on one core."""
    import oracle
    oracle.build()
    host = host_cpu()
    threads = host["usable_cores"]
    single, _ = sized_samples(cases, budget_s)
    secs1 = time_oracle(single)
    b1 = sum(algorithmic_bytes(s) for s in single)
    many, _ = sized_samples(cases, budget_s, threads)
    secs, reps = 0.0, 0
    while reps < 1 or (secs < 2.0 and reps < 20):  # repeat a short sample for a stable figure
        secs += time_oracle(many, threads)
        reps += 1
    b = sum(algorithmic_bytes(s) for s in many) * reps
    tok = sum(s.tokens for s in many) * reps
    return {"value": round(b / secs / 1e9, 5), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "tokens_per_s": round(tok / secs, 1), "seconds": round(secs, 2), "repeats": reps,
            "nproc": host["nproc"], "cpu_model": host["cpu_model"], "machine": host["machine"],
            "sample": _sample_text(many, cases, threads) + (", run %d times" % reps if reps > 1 else ""),
            "single_core": {"value": round(b1 / secs1 / 1e9, 5), "unit": "GB/s", "cores": 1,
                            "tokens_per_s": round(sum(s.tokens for s in single) / secs1, 1),
                            "seconds": round(secs1, 2), "sample": _sample_text(single, cases, 1)}}


def run_reference(args):
    """The reference arm: the oracle, as it stands, on every usable host core
    (token shards, one thread per core), bounded samples of the workload."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    host = host_cpu()
    threads = host["usable_cores"]
    cases = build_workloads()
    steps = args.steps + args.warmup
    per_step = max(0.02, min(0.5, args.reference_seconds / max(1, steps)))
    samples, frac = sized_samples(cases, per_step, threads)
    for _ in range(args.warmup):
        time_oracle(samples, threads)
    times = [time_oracle(samples, threads) for _ in range(args.steps)]
    secs = sum(times) / len(times)
    b = sum(algorithmic_bytes(s) for s in samples)
    tok = sum(s.tokens for s in samples)
    value = b / secs / 1e9
    sample = _sample_text(samples, cases, threads) + ", per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "tokens_per_s": round(tok / secs, 1),
            "config": step_config(sum(algorithmic_bytes(c) for c in cases), sum(c.tokens for c in cases)),
            "sample": sample,
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "nproc": host["nproc"], "cpu_model": host["cpu_model"], "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_stream_only(args):
    """One operator of the bench alone: its launches back to back over the
    rotating buffer copies of the stream region (at least 3x L2 of other data
    between two uses of a copy), ``--warmup`` then ``--steps`` launches, for a
    profiler capture of consecutive launches in steady state (each launch's
    DRAM write-back of the previous one's dirty lines included)."""
    import math
    from transformer_rope_positional_gb300 import build as B
    B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cases = build_workloads()
    dev_tensors = []
    for c in cases:
        if hasattr(c, "x"):
            dev_tensors.append((c.x.to(dev), c.cos.to(dev), c.sin.to(dev)))
        else:
            dev_tensors.append((c.positions.to(dev), c.query.to(dev), c.key.to(dev), c.cache.to(dev)))
    specs = {label: (nbytes, factory) for label, nbytes, factory, _ in operator_specs(cases, dev_tensors)}
    if args.stream_only not in specs:
        raise SystemExit("unknown operator %r; one of %s" % (args.stream_only, ", ".join(sorted(specs))))
    nbytes, factory = specs[args.stream_only]
    n = max(2, math.ceil(3 * L2_BYTES / nbytes) + 1)
    calls = factory(n)
    for j in range(args.warmup):
        calls[j % n]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host = []
    e0.record()
    for j in range(args.steps):
        h0 = time.perf_counter()
        calls[(args.warmup + j) % n]()
        host.append((time.perf_counter() - h0) * 1e6)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / args.steps * 1e3
    print(json.dumps({"mode": "stream_only", "workload": args.stream_only, "buffer_sets": n, "warmup": args.warmup,
                      "launches": args.steps, "us_per_launch": round(us, 3), "bytes_per_launch": nbytes,
                      "host_us_per_call": [round(h, 1) for h in host]}), flush=True)


def run_fetch_granularity(args):
    """The in-place workload's aligned slice [64,128) and the slice [4,68)
    (which crosses a 128-byte line of every 256-byte row) under L2 fetch
    granularity limits of 32, 64 and 128 bytes, set on this process's CUDA
    context (cuCtxSetLimit; the setting ends with the process, and the
    context's own value is restored at the end).  Default: stream time per
    launch of each.  ``--steps 1``: one launch of each, for a profiler capture
    of the DRAM bytes."""
    import ctypes
    import workloads as W
    from transformer_rope_positional_gb300 import build as B
    B.build()
    import transformer_rope_positional_gb300 as R
    limit_id = 0x05  # CU_LIMIT_MAX_L2_FETCH_GRANULARITY
    cu = ctypes.CDLL("libcuda.so.1")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    torch.zeros(1, device=dev)  # the primary context is current on this thread

    def limit():
        v = ctypes.c_size_t(0)
        if cu.cuCtxGetLimit(ctypes.byref(v), limit_id) != 0:
            raise RuntimeError("cuCtxGetLimit failed")
        return int(v.value)

    def set_limit(n):
        if cu.cuCtxSetLimit(limit_id, ctypes.c_size_t(n)) != 0:
            raise RuntimeError("cuCtxSetLimit failed")

    default = limit()
    full = W.inplace_bf16_mixed()
    cases = [full, W.inplace_case("inplace_bf16x_f32cs_4x4096x32x128_slice4_68", 1, tuple(full.x.shape), 4, 68,
                                  torch.bfloat16, torch.float32)]
    peak, _ = measured_peak()
    rows = []
    try:
        for lim in (32, 64, 128):
            set_limit(lim)
            for c in cases:
                x, cs, sn = c.x.to(dev), c.cos.to(dev), c.sin.to(dev)
                row = {"workload": c.name, "fetch_limit_bytes": limit()}
                if args.steps == 1:
                    R.rope_inplace_partial(x, cs, sn, 1, [c.start, c.end])
                    torch.cuda.synchronize()
                else:
                    nbytes = algorithmic_bytes(c)
                    us = min(stream_us(lambda n: [R.prepare_inplace_partial(t[0], cs, sn, 1, [c.start, c.end])
                                                  for t in copies(x, n=n)], nbytes)[0] for _ in range(3))
                    row.update({"stream_us": round(us, 3), "frac_of_peak": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)})
                rows.append(row)
                del x
                torch.cuda.empty_cache()
    finally:
        set_limit(default)
    print(json.dumps({"mode": "fetch_granularity", "context_default_limit_bytes": default, "rows": rows}),
          flush=True)


def run_size_sweep(args):
    """Each operator stream-timed (as in the step's stream region) on its
    workload at 0.5x, 1x, 1.5x and 2x the tokens, and a least-squares line
    time = fixed + bytes / rate through the four points: `rate` is the
    streaming rate of the kernel, `fixed_us` the per-launch cost (ramp-up,
    drain) that the launch cannot amortise."""
    import workloads as W
    from transformer_rope_positional_gb300 import build as B
    B.build()
    import transformer_rope_positional_gb300 as R
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, _ = measured_peak()

    def mrope(f):
        pos = W.mrope_positions(int(8192 * f), (int(6 * f), 64, 64))
        return W.cache_case("mrope_%dtok" % pos.shape[1], 4, pos.shape[1], 28, 4, 128, 128, 40960, torch.bfloat16,
                            True, base=1e6, positions=pos, mrope_section=[16, 24, 24])

    def qkv(f):  # the prefill chunks and the number of decode requests both scale
        nd = int(256 * f)
        ctx = W.uniform_int(W.stream_seed(5, 3), nd, 16, 1024).tolist()
        return W.qkv_case("qkv_%dtok" % (4 * int(1984 * f) + nd), 5, [int(1984 * f)] * 4 + [1] * nd,
                          [4096] * 4 + ctx, 32, 8, 8, 128, 16, torch.bfloat16)

    def factory(c, mode=1, backward=False, cache_mode=0, out_of_place=False, views=False):
        if hasattr(c, "qkv"):
            ro = [t.to(dev) for t in (c.q_gamma, c.k_gamma, c.cache, c.seq_lens, c.query_start_loc, c.slot_mapping)]
            ts = [t.to(dev) for t in (c.qkv, c.q_out, c.k_cache, c.v_cache)]
            return lambda n: [R.prepare_qkv_rmsnorm_rope_cache(t[0], c.nq, c.nk, c.nv, ro[0], ro[1], c.eps, ro[2],
                                                               ro[3], ro[4], ro[5], t[1], t[2], t[3])
                              for t in copies(*ts, n=n)]
        if hasattr(c, "x"):
            cs, sn = c.cos.to(dev), c.sin.to(dev)
            x = c.x.to(dev)
            return lambda n: [R.prepare_inplace_partial(t[0], cs, sn, mode, [c.start, c.end], backward=backward)
                              for t in copies(x, n=n)]
        p, cc = c.positions.to(dev), c.cache.to(dev)
        q, k = c.query.to(dev), c.key.to(dev)
        if out_of_place:
            return lambda n: [R.prepare_with_sin_cos_cache(p, t[0], t[1], cc, c.head_size, c.rotary_dim, c.is_neox,
                                                           c.mrope_section, query_out=t[2], key_out=t[3])
                              for t in copies(q, k, torch.empty_like(q), torch.empty_like(k), n=n)]
        if views:  # q and k as row views of a fused [T, q | k | k-sized v] buffer
            wq, wk = q.shape[1], k.shape[1]
            buf = torch.empty(q.shape[0], wq + 2 * wk, dtype=q.dtype, device=dev)
            buf[:, :wq].copy_(q)
            buf[:, wq:wq + wk].copy_(k)
            return lambda n: [R.prepare_with_sin_cos_cache(p, t[0][:, :wq], t[0][:, wq:wq + wk], cc, c.head_size,
                                                           c.rotary_dim, c.is_neox, c.mrope_section)
                              for t in copies(buf, n=n)]
        return lambda n: [R.prepare_with_sin_cos_cache(p, t[0], t[1], cc, c.head_size, c.rotary_dim, c.is_neox,
                                                       c.mrope_section, cache_mode=cache_mode)
                          for t in copies(q, k, n=n)]

    inplace = lambda f: W.inplace_bf16_mixed(int(4 * f))  # noqa: E731
    neox = lambda f: W.cache_neox_bf16(int(16384 * f))  # noqa: E731
    gptj = lambda f: W.cache_gptj_f16_partial(int(8 * f))  # noqa: E731
    families = [("inplace_bf16x_f32cs_Bx4096x32x128_slice64_128", inplace, {}),
                ("rope_neox_bf16_32q8k_h128", neox, {}),
                ("rope_gptj_f16_16q16k_h256_r64", gptj, {}),
                ("mrope_neox_bf16_28q4k_h128_s16_24_24", mrope, {}),
                ("qkv_rmsnorm_rope_bf16_32q8k8v_h128", qkv, {}),
                ("inplace_backward_interleave_bf16x_f32cs", inplace, {"backward": True}),
                ("inplace_half_forward_bf16x_f32cs", inplace, {"mode": 0}),
                ("mrope_interleaved_splice_neox_bf16", mrope, {"cache_mode": 1}),
                ("rope_neox_out_of_place_bf16", neox, {"out_of_place": True}),
                ("rope_gptj_fused_qkv_views_f16", gptj, {"views": True})]
    out = []
    for name, make, opts in families:
        pts = []
        for f in (0.5, 1.0, 1.5, 2.0):
            c = make(f)
            nbytes = algorithmic_bytes(c)
            us, _ = stream_us(factory(c, **opts), nbytes)
            pts.append({"tokens": c.tokens, "bytes": nbytes, "us": round(us, 3)})
            del c
            torch.cuda.empty_cache()
        xs = [p["bytes"] for p in pts]
        ys = [p["us"] for p in pts]
        mx, my = sum(xs) / len(xs), sum(ys) / len(ys)
        slope = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sum((x - mx) ** 2 for x in xs)  # us per byte
        rate = 1e-3 / slope  # GB/s
        out.append({"family": name, "points": pts, "stream_rate_gbs": round(rate, 1),
                    "stream_rate_frac_of_peak": round(rate / peak, 4), "fixed_us": round(my - slope * mx, 3)})
        print(json.dumps(out[-1]), flush=True)
    print(json.dumps({"metric": "stream rate and per-launch fixed cost from a size sweep", "peak_gbs": peak,
                      "families": out}), flush=True)


def run_marginal(args):
    """Each hot-path kernel alone, at its token count and at twice that, with a
    read-only sweep of 384 MB before every launch (clean, cold L2).  Reports the
    clean single-launch GB/s, the marginal GB/s (extra bytes / extra time) and
    the fixed cost (launch, ramp-up, drain) that separates the two."""
    import workloads as W
    from transformer_rope_positional_gb300 import build as B
    B.build()
    import transformer_rope_positional_gb300 as R
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sweep = torch.empty(384 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1, dtype=torch.float32, device=dev)

    def prep(c):
        if hasattr(c, "x"):
            return R.prepare_inplace_partial(c.x.to(dev), c.cos.to(dev), c.sin.to(dev), 1, [c.start, c.end])
        return R.prepare_with_sin_cos_cache(c.positions.to(dev), c.query.to(dev), c.key.to(dev), c.cache.to(dev),
                                            c.head_size, c.rotary_dim, c.is_neox, c.mrope_section)

    def median_us(call, reps=30):
        ts = []
        for _ in range(3):
            call()
        for _ in range(reps):
            sink.copy_(sweep.sum().reshape(1))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return sorted(ts)[len(ts) // 2] * 1e3

    mrope = W.mrope_neox_bf16()
    pairs = [(W.inplace_bf16_mixed(4), W.inplace_bf16_mixed(8)),
             (W.cache_neox_bf16(16384), W.cache_neox_bf16(32768)),
             (W.cache_gptj_f16_partial(8, 1024), W.cache_gptj_f16_partial(16, 1024)),
             (mrope, W.cache_case(mrope.name + "_x2", 4, 2 * mrope.tokens, 28, 4, 128, 128, 40960, torch.bfloat16,
                                  True, base=1e6, positions=torch.cat([mrope.positions] * 2, 1).contiguous(),
                                  mrope_section=[16, 24, 24]))]
    peak, _ = measured_peak()
    out = []
    for c1, c2 in pairs:
        t1, t2 = median_us(prep(c1)), median_us(prep(c2))
        b1, b2 = algorithmic_bytes(c1), algorithmic_bytes(c2)
        marg = (b2 - b1) / ((t2 - t1) * 1e-6) / 1e9
        out.append({"workload": c1.name, "us_1x": round(t1, 2), "us_2x": round(t2, 2),
                    "gbs_1x": round(b1 / (t1 * 1e-6) / 1e9, 1), "frac_1x": round(b1 / (t1 * 1e-6) / 1e9 / peak, 4),
                    "marginal_gbs": round(marg, 1), "fixed_us": round(t1 - b1 / (marg * 1e9) * 1e6, 2)})
    print(json.dumps({"mode": "marginal", "peak_gbs": peak, "kernels": out}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--kernel-steps", type=int, default=500, help="steps of the per-kernel timing region")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle work for cpu_baseline")
    ap.add_argument("--reference-seconds", type=float, default=120.0, help="oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--marginal", action="store_true",
                    help="instead of the step: each kernel alone at 1x and 2x tokens on a clean L2")
    ap.add_argument("--size-sweep", action="store_true",
                    help="instead of the step: each operator stream-timed at 0.5x..2x tokens; rate and fixed cost")
    ap.add_argument("--fetch-granularity", action="store_true",
                    help="instead of the step: aligned and unaligned in-place slices under L2 fetch limits")
    ap.add_argument("--stream-only", metavar="WORKLOAD",
                    help="instead of the step: one operator's launches back to back (--warmup, then --steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.stream_only:
        run_stream_only(args)
    elif args.fetch_granularity:
        run_fetch_granularity(args)
    elif args.marginal:
        run_marginal(args)
    elif args.size_sweep:
        run_size_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
