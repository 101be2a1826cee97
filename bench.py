#!/usr/bin/env python3
"""Benchmark of the fused KDA decode step on GB300.

One step = one decode token through a stack of 69 independent KDA layers
(H=48 heads of 128, a 96-slot state pool per layer, N=64 rows of which the
last 4 are slot-0 padding), all 69 launches captured in one CUDA graph and
replayed.  The metric is (sequence, head) state updates per second; the
roofline object reports the algorithmic HBM bytes of one launch over its
measured duration against the measured copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (under torchrun) every rank runs its own stack on its own GPU
with no data exchange (weak scaling); rank 0 prints the line.
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
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused KDA decode: seq·head updates/s and achieved HBM GB/s vs GB300 peak"
UNIT = "updates/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_NOTE = os.path.join(ROOT, "profiles", "kda_decode_stack69_traffic.md")
KERNEL_SRC = os.path.join(ROOT, "linear_attention_decode_04_gb300", "csrc", "kda_decode_kernel.cuh")
PREFILL_TRAFFIC_NOTE = os.path.join(ROOT, "profiles", "kda_prefill_traffic.md")
PREFILL_SRC = os.path.join(ROOT, "linear_attention_decode_04_gb300", "csrc", "kda_prefill.cu")


# ----------------------------------------------------------------- host logic

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate(ms_local: float, units_local: int, world: int, device=None) -> tuple[float, int]:
    """Max step time and total units over ranks (identity at world 1)."""
    if world == 1:
        return ms_local, units_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    u = torch.tensor([float(units_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), int(u.item())


def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(path: str | None = None) -> str:
    with open(path or KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(note: str | None = None, src: str | None = None) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None).  Defaults: the decode note and
    the decode kernel source."""
    note, src = note or TRAFFIC_NOTE, src or KERNEL_SRC
    try:
        text = open(note).read()
    except OSError:
        return None
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not h or not b or h.group(1) != kernel_source_hash(src):
        return None
    return float(b.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self) -> dict:
        try:
            rows = [r.split(",") for r in open(self.file.name).read().strip().splitlines() if r.strip()]
        finally:
            os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- oracle leg

def oracle_rate(host_layers, budget_s: float) -> dict:
    """Time the fp64 oracle (as it stands) on the given layers' inputs,
    repeating passes until ``budget_s`` of wall time; returns units/s."""
    import oracle
    threads = os.cpu_count() or 1
    units = done = 0
    t0 = time.perf_counter()
    passes = 0
    while True:
        for x in host_layers:
            r = oracle.decode(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state,
                              state=x.state, g=x.g, beta=x.beta, slot_idx=x.slot_idx, H=x.H,
                              gate=x.gate, norm_weight=x.norm_weight, eps=x.spec.eps,
                              out_norm=x.spec.out_norm, update_conv_state=x.spec.update_conv_state,
                              threads=threads, want_f64=False, in_place=True)
            assert r.n_out_of_range == 0
            units += len(x.active_rows()) * x.H
        passes += 1
        done = time.perf_counter() - t0
        if done >= budget_s:
            break
    return {"units": units, "seconds": done, "value": units / done, "threads": threads, "passes": passes}


# ----------------------------------------------------------------- main

def build_stack(device, n_layers: int, keep_host: int):
    from linear_attention_decode_04_gb300 import workloads as W
    return build_stack_specs(device, [W.stack_layer_spec(ell) for ell in range(n_layers)], keep_host)


def build_stack_specs(device, specs, keep_host: int = 0):
    import torch

    from linear_attention_decode_04_gb300 import workloads as W
    layers, host = [], []
    for ell, sp in enumerate(specs):
        x = W.make_inputs(sp)
        L = dict(
            qkv=torch.from_numpy(x.qkv.view(np.int16)).view(torch.bfloat16).to(device),
            conv_weight=torch.from_numpy(x.conv_weight).to(device),
            conv_state=torch.from_numpy(x.conv_state.view(np.int16)).view(torch.bfloat16).to(device),
            state=torch.from_numpy(x.state).to(device),
            g=torch.from_numpy(x.g).to(device),
            beta=torch.from_numpy(x.beta.view(np.int16)).view(torch.bfloat16).to(device),
            gate=torch.from_numpy(x.gate.view(np.int16)).view(torch.bfloat16).to(device),
            norm_weight=torch.from_numpy(x.norm_weight).to(device),
            slot_idx=torch.from_numpy(x.slot_idx).to(device),
            out=torch.empty(x.N, x.H * W.HEAD_DIM, dtype=torch.bfloat16, device=device),
            err_flag=torch.zeros(1, dtype=torch.int32, device=device),
        )
        layers.append(L)
        if ell < keep_host:
            host.append(x)
        n_active = len(x.active_rows())
    return layers, host, x.spec, n_active


def replay_stats(step, stream, n: int) -> dict:
    """Run ``step`` ``n`` times on ``stream`` with a CUDA event before each
    run and one after the last; per-run device times in ms (median, p10,
    p90, mean)."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        for i in range(n):
            evs[i].record(stream)
            step()
        evs[n].record(stream)
    torch.cuda.synchronize(stream.device)
    t = np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(n)])
    return {"n": n, "median_ms": float(np.median(t)), "p10_ms": float(np.percentile(t, 10)),
            "p90_ms": float(np.percentile(t, 90)), "mean_ms": float(t.mean())}


def single_launch(device, spec, warmup: int, n: int, graph: bool = True) -> dict:
    """One decode launch of ``spec`` on its own (replayed from a CUDA graph,
    or launched eagerly), timed per launch over ``n`` runs."""
    import torch

    from linear_attention_decode_04_gb300 import workloads as W
    from linear_attention_decode_04_gb300.stack import DecodeStack
    layers, _, spec, n_active = build_stack_specs(device, [spec])
    stack = DecodeStack(layers, eps=spec.eps, out_norm=spec.out_norm,
                        update_conv_state=spec.update_conv_state)
    stream = torch.cuda.Stream(device)
    if graph:
        stack.capture(stream)
    step = stack.replay if graph else (lambda: stack.run_eager(stream))
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize(device)
    st = replay_stats(step, stream, n)
    if int(layers[0]["err_flag"].item()):
        raise SystemExit("device error flag raised")
    nbytes = W.algorithmic_bytes(spec.N, spec.H, n_active, spec.out_norm)
    peak, kind = measured_peak()
    ms = st["mean_ms"]
    gbs = nbytes / (ms / 1e3) / 1e9
    res = {"workload": spec.name, "graph": graph, "ms_per_launch": ms, "stats": st,
           "updates_per_s": n_active * spec.H / (ms / 1e3), "achieved_gbs": gbs, "peak_gbs": peak,
           "frac": gbs / peak, "frac_median": nbytes / (st["median_ms"] / 1e3) / 1e9 / peak,
           "peak_source": f"{kind} hbm_gbs", "algorithmic_bytes_per_launch": nbytes,
           "work_queue": stack.queue is not None}
    del stack, layers
    torch.cuda.empty_cache()
    return res


def spec_launch(device, spec, warmup: int, n: int, reset_timeline_before_last: bool = False) -> dict:
    """One multi-token (speculative) decode launch of ``spec`` (work queue)
    replayed from a CUDA graph, timed per launch over ``n`` replays."""
    import torch

    from linear_attention_decode_04_gb300 import KdaDecodeCall
    from linear_attention_decode_04_gb300 import workloads as W
    from linear_attention_decode_04_gb300.stack import warm_up
    x = W.make_multi_inputs(spec)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    t = dict(qkv=bf(x.qkv), conv_weight=f(x.conv_weight), conv_state=bf(x.conv_state), state=f(x.state),
             g=f(x.g), beta=bf(x.beta), gate=bf(x.gate), norm_weight=f(x.norm_weight), src=f(x.src_slot),
             dst=f(x.dst_slots), out=torch.empty(x.N * x.T, x.H * 128, dtype=torch.bfloat16, device=device),
             err=torch.zeros(1, dtype=torch.int32, device=device),
             queue=torch.zeros(2, dtype=torch.int32, device=device))
    call = KdaDecodeCall(t["qkv"], t["conv_weight"], t["conv_state"], t["state"], t["g"], t["beta"], t["dst"],
                         t["out"], gate=t["gate"], norm_weight=t["norm_weight"], eps=spec.eps,
                         out_norm=spec.out_norm, update_conv_state=spec.update_conv_state, err_flag=t["err"],
                         work_queue=t["queue"], tokens_per_seq=x.T, src_slot=t["src"])
    warm_up(device)
    stream = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize(device)
    st = replay_stats(graph.replay, stream, n)
    timeline = None
    if reset_timeline_before_last:  # one more replay, recorded (timeline build)
        from linear_attention_decode_04_gb300 import binding
        binding.timeline_reset()
        torch.cuda.synchronize(device)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize(device)
        timeline = binding.timeline_read()
    if int(t["err"].item()):
        raise SystemExit("device error flag raised")
    valid = lambda sl: 0 < sl < spec.num_slots  # noqa: E731
    units = sum(1 for nn in range(x.N) if valid(x.src_slot[nn])) * x.H
    tokens = sum(1 for nn in range(x.N) for tt in range(x.T)
                 if valid(x.src_slot[nn]) and valid(x.dst_slots[nn, tt])) * x.H
    nbytes = W.multi_algorithmic_bytes(spec, x.src_slot, x.dst_slots)
    peak, kind = measured_peak()
    ms = st["mean_ms"]
    gbs = nbytes / (ms / 1e3) / 1e9
    res = {"workload": spec.name, "tokens_per_seq": x.T, "graph": True, "ms_per_launch": ms, "stats": st,
           "token_updates_per_s": tokens / (ms / 1e3), "sequence_head_units_per_s": units / (ms / 1e3),
           "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak, "peak_source": f"{kind} hbm_gbs",
           "algorithmic_bytes_per_launch": nbytes,
           "bytes_note": "per (sequence, head): 64 KiB state read once + 64 KiB written per present token, "
                         "plus windows and per-token inputs / outputs"}
    if timeline is not None:
        res["_timeline"] = timeline
    del call, graph, t
    torch.cuda.empty_cache()
    return res


def run_ours(args) -> dict | None:
    import torch

    from linear_attention_decode_04_gb300 import workloads as W
    from linear_attention_decode_04_gb300.stack import STEP_INPUTS, DecodeStack

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    n_layers = W.STACK_LAYERS
    keep_host = 2 if (rank == 0 and not args.no_cpu_baseline) else 0
    layers, host, spec, n_active = build_stack(device, n_layers, keep_host)
    stack = DecodeStack(layers, eps=spec.eps, out_norm=spec.out_norm,
                        update_conv_state=spec.update_conv_state)
    stream = torch.cuda.Stream(device)
    stack.capture(stream)

    units_step = n_layers * n_active * spec.H
    launch_bytes = W.algorithmic_bytes(spec.N, spec.H, n_active, spec.out_norm)
    state_bytes = n_layers * spec.num_slots * spec.H * 128 * 128 * 4

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-resident timing (graph replay)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            stack.replay()
    torch.cuda.synchronize(device)
    barrier()
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                stack.replay()
            ev1.record(stream)
        torch.cuda.synchronize(device)
    barrier()
    torch.cuda.synchronize(device)
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms_step, units_total = aggregate(ms_local, units_step, world, device)
    clocks = clk.summary()

    # ---- spread: per-replay device times over at least 100 graph replays
    n_stats = max(args.steps, 100)
    stats = replay_stats(stack.replay, stream, n_stats)
    # ---- the same step launched eagerly (69 C-ABI calls per step, no graph)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            stack.run_eager(stream)
    torch.cuda.synchronize(device)
    eager = replay_stats(lambda: stack.run_eager(stream), stream, max(args.steps, 50))

    # ---- end to end: pinned host inputs -> device, graph, output -> host
    # ---- end to end: every layer's per-token inputs and its output live in
    # pinned host memory; the kernels read and write them directly over the
    # CPU-GPU link (no copy engine), state and weights stay in HBM.
    host_layers = []
    for L in layers:
        HL = dict(L)
        for k in STEP_INPUTS + ("out",):
            HL[k] = torch.empty(L[k].shape, dtype=L[k].dtype).pin_memory()
            HL[k].copy_(L[k])
        host_layers.append(HL)
    h2d = sum(HL[k].numel() * HL[k].element_size() for HL in host_layers for k in STEP_INPUTS)
    d2h = sum(HL["out"].numel() * HL["out"].element_size() for HL in host_layers)
    e2e_stack = DecodeStack(host_layers, eps=spec.eps, out_norm=spec.out_norm,
                            update_conv_state=spec.update_conv_state, host_token_io=True)
    e2e_stack.capture(stream)
    e2e_steps = max(args.steps, 20)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_stack.replay()
    torch.cuda.synchronize(device)
    barrier()
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_stack.replay()
        ev1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    e2e_ms, _ = aggregate(ev0.elapsed_time(ev1) / e2e_steps, units_step, world, device)

    errs = sum(int(L["err_flag"].item()) for L in layers)
    if errs:
        raise SystemExit(f"device error flag raised ({errs})")
    del e2e_stack, host_layers

    # ---- the N=256, H=96, 1024-slot step as one launch under graph replay,
    # the configuration the >= 75% roofline target is judged on
    cfg3 = None
    if not args.no_cfg3:
        cfg3 = single_launch(device, W.ROOFLINE, args.warmup, max(args.steps, 50))
    spec_decode = None
    if not args.no_cfg3:
        spec_decode = spec_launch(device, W.MULTI_BENCH, args.warmup, max(args.steps, 50))
    prefill = None
    if not args.no_cfg3:
        prefill, _ = prefill_timing(device, W.PREFILL_BENCH, args.warmup, max(args.steps, 50))
        prefill.pop("mode", None)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r = oracle_rate(host, args.cpu_budget)
        cpu = {"value": r["value"], "unit": UNIT, "cores": r["threads"], "kind": "oracle",
               "sample": (f"fp64 C oracle, OpenMP {r['threads']} threads, {len(host)} of the 69 layers "
                          f"({r['units']} (row, head) updates over {r['passes']} passes, "
                          f"{r['seconds']:.1f} s)")}

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    peak, peak_kind = measured_peak()
    per_launch_s = ms_step / 1e3 / stack.launches_per_step
    achieved = launch_bytes / per_launch_s / 1e9
    traffic = recorded_traffic()
    return {
        "metric": METRIC, "value": units_total / (ms_step / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; distributions of the decode-step workload)",
        "config": {"workload": W.STACK_LAYER.name, "layers": n_layers, "N": spec.N, "H": spec.H,
                   "head_dim": 128, "pool_slots": spec.num_slots, "pad_rows": spec.pad_tail,
                   "active_units_per_step": units_step, "graph": "one CUDA graph per step",
                   "l2": f"inputs larger than L2: {state_bytes / 1e9:.1f} GB state pools",
                   "parallelism": f"replicas x{world} (no exchange)"},
        "achieved_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": launch_bytes},
        "e2e": {"value": units_total / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "one CUDA graph per step; every layer's per-token inputs and output in "
                       "pinned host memory, read and written by the kernels directly over "
                       "NVLink-C2C (no copy engine); state and weights resident in HBM"},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": stack.launches_per_step * args.steps,
        "stats": dict(stats, what=f"per-replay device time of the 69-layer graph step over "
                                  f"{stats['n']} replays after the timed region",
                      updates_per_s_median=units_step / (stats["median_ms"] / 1e3)),
        "eager": {"ms_per_step": eager["mean_ms"], "median_ms": eager["median_ms"],
                  "p10_ms": eager["p10_ms"], "p90_ms": eager["p90_ms"], "steps": eager["n"],
                  "updates_per_s": units_step / (eager["mean_ms"] / 1e3),
                  "graph_ms_per_step": ms_step,
                  "how": "the same 69 launches issued one C-ABI call at a time from Python, no graph"},
        "cfg3": cfg3,
        "spec_decode": spec_decode,
        "prefill": prefill,
        "impl": "ours",
    }


def run_case(args) -> dict | None:
    """Timing of one launch configuration on its own (also the small case
    for ncu captures): ``layer`` = one layer of the stack, launched eagerly;
    ``roofline`` = N=256, H=96, pool 1024 as one launch replayed from a CUDA
    graph.  Prints a line with ``mode`` set; not the headline line."""
    import torch

    from linear_attention_decode_04_gb300 import workloads as W
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    spec = W.stack_layer_spec(0) if args.case == "layer" else W.ROOFLINE
    with ClockSampler(0) as clk:
        res = single_launch(device, spec, args.warmup, args.steps, graph=args.case != "layer")
    res.update(mode=args.case, clocks=clk.summary(), steps=args.steps, warmup=args.warmup)
    return res


def measured_tf32_peak() -> tuple[float, str]:
    """Dense tf32 tensor peak: the measured bf16 burst figure scaled by the
    nominal tf32 / bf16 ratio (1.1 / 2.25 PFLOP/s)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        return bf16 * 1.1 / 2.25, "measured bf16_tflops x 1.1/2.25"
    except Exception:
        return 1900.0 * 1.1 / 2.25, "fallback 1.9 PFLOP/s bf16 x 1.1/2.25"


def run_prefill(args) -> dict:
    """Chunked prefill of one varlen batch (16 sequences, 16,384 tokens,
    H = 48): each step is one kda_prefill launch over the whole batch, inputs
    resident in HBM (1.5 GB, larger than L2).  The state pools carry over from
    step to step.  ``value`` = (token, head) updates per second."""
    import torch

    from linear_attention_decode_04_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    spec = W.PREFILL_PROFILE if args.prefill_workload == "profile" else W.PREFILL_BENCH
    res, x = prefill_timing(dev, spec, args.warmup, args.steps)
    act_tokens = sum(n for b, n in enumerate(spec.lens) if b not in spec.pad_seqs)
    if not args.no_cpu_baseline:
        import oracle
        threads = os.cpu_count() or 1
        updates = passes = 0
        t0 = time.perf_counter()
        while True:  # whole batch, repeated until the time budget is spent
            oracle.prefill(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state,
                           g=x.g, beta=x.beta, gate=x.gate, norm_weight=x.norm_weight, slot_idx=x.slot_idx,
                           cu_seqlens=x.cu_seqlens, H=spec.H, eps=spec.eps, threads=threads, want_f64=False)
            updates += act_tokens * spec.H
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= args.cpu_budget:
                break
        res["cpu_baseline"] = {"value": updates / dt, "unit": "updates/s", "cores": threads, "kind": "oracle",
                               "sample": f"fp64 C prefill oracle, OpenMP {threads} threads, the whole batch "
                                         f"x{passes} ({updates} (token, head) updates, {dt:.1f} s)"}
    return res


def prefill_timing(dev, spec, warmup: int, steps: int):
    """``steps`` kda_prefill launches over one varlen batch timed between
    CUDA events (after ``warmup`` untimed ones); the result line's fields and
    the host inputs."""
    import torch

    from linear_attention_decode_04_gb300 import KdaPrefillCall
    from linear_attention_decode_04_gb300 import workloads as W
    x = W.make_prefill_inputs(spec)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    t = dict(qkv=bf(x.qkv), conv_weight=torch.from_numpy(x.conv_weight).to(dev), conv_state=bf(x.conv_state),
             state=torch.from_numpy(x.state).to(dev), g=torch.from_numpy(x.g).to(dev), beta=bf(x.beta),
             cu_seqlens=torch.from_numpy(x.cu_seqlens).to(dev), slot_idx=torch.from_numpy(x.slot_idx).to(dev),
             out=torch.empty(spec.T, spec.H * 128, dtype=torch.bfloat16, device=dev), gate=bf(x.gate),
             norm_weight=torch.from_numpy(x.norm_weight).to(dev),
             err_flag=torch.zeros(1, dtype=torch.int32, device=dev))
    call = KdaPrefillCall(t["qkv"], t["conv_weight"], t["conv_state"], t["state"], t["g"], t["beta"],
                          t["cu_seqlens"], t["slot_idx"], t["out"],
                          cu_seqlens_cpu=torch.from_numpy(x.cu_seqlens), gate=t["gate"],
                          norm_weight=t["norm_weight"], eps=spec.eps, out_norm=spec.out_norm,
                          err_flag=t["err_flag"])
    stream = torch.cuda.Stream(dev)
    for _ in range(warmup):
        call(stream)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        ev0.record(stream)
        for _ in range(steps):
            call(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    if int(t["err_flag"].item()):
        raise SystemExit("device error flag raised")
    ms = ev0.elapsed_time(ev1) / steps
    act_tokens = sum(n for b, n in enumerate(spec.lens) if b not in spec.pad_seqs)
    nbytes = W.prefill_algorithmic_bytes(spec)
    flops = W.prefill_algorithmic_flops(spec)
    peak, kind = measured_peak()
    tpeak, tkind = measured_tf32_peak()
    gbs = nbytes / (ms / 1e3) / 1e9
    tflops = flops / (ms / 1e3) / 1e12
    res = {"mode": "prefill", "metric": "chunked KDA prefill: (token, head) updates/s",
           "value": act_tokens * spec.H / (ms / 1e3), "unit": "updates/s", "ms_per_launch": ms,
           "workload": spec.name, "tokens": spec.T, "sequences": spec.B, "H": spec.H,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                        "traffic": (recorded_traffic(PREFILL_TRAFFIC_NOTE, PREFILL_SRC)
                                    if spec is W.PREFILL_BENCH else None),
                        "traffic_note": "both kernels; includes the workspace written and read back",
                        "peak_source": f"{kind} hbm_gbs", "algorithmic_bytes_per_launch": nbytes},
           "tensor": {"achieved_tflops": tflops, "peak_tflops": tpeak, "frac": tflops / tpeak,
                      "peak_source": tkind, "algorithmic_flops_per_launch": flops,
                      "note": "chunk-form contractions counted once; the kernel issues three tf32 "
                              "products per contraction (split operands)"},
           "clocks": clk.summary(), "steps": steps, "warmup": warmup,
           "gpu_launches": 3 * steps,
           "kernels": "per step: chunk metadata, chunk-parallel kernel, scan kernel",
           "scan_order": "longest sequence first" if call.seq_order is not None else "index"}
    del call, t
    torch.cuda.empty_cache()
    return res, x


def run_chunk_metadata(args) -> dict:
    """Timing of the device-side chunk metadata build for a prefill batch
    (256 sequences, lengths 1..8192 tokens, chunk size 64): 20 builds
    captured back to back in one CUDA graph, so that the per-call figure is
    the kernel's and not the graph launch's."""
    import torch

    from linear_attention_decode_04_gb300 import kda_chunk_metadata
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 8193, 256)
    cu_cpu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    cu = cu_cpu.to(dev)
    kda_chunk_metadata(cu, cu_cpu, 64)
    s = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    per_graph = 20
    with torch.cuda.graph(g, stream=s):
        for _ in range(per_graph):
            idx, off = kda_chunk_metadata(cu, cu_cpu, 64)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(args.steps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / args.steps / per_graph * 1e3
    total = int(off[-1].item())
    return {"mode": "chunk_metadata", "sequences": 256, "tokens": int(lens.sum()), "chunk_size": 64,
            "chunks": total, "us_per_call": us, "bound": "latency (one CTA, a scan then an expansion)",
            "bytes": 257 * 4 + 257 * 8 + total * 8, "steps": args.steps, "warmup": args.warmup}


def timeline_summary(rec: np.ndarray, ctas: int) -> dict:
    """Per-launch figures from the decode kernel's per-CTA records of one
    step (records sorted by start: each launch's CTAs all start before any
    CTA of the next launch), medians over the launches after the first; us."""
    rec = rec[np.argsort(rec[:, 2])].astype(np.float64)
    per = []
    for ell in range(len(rec) // ctas):
        r = rec[ell * ctas:(ell + 1) * ctas]
        start, first, end, units, comp, wait = (r[:, i] for i in range(2, 8))
        d = {"duration": end.max() - start.min(), "first_unit_ready_after_cta_start": np.median(first - start),
             "end_spread": end.max() - end.min(), "tail_after_median_end": end.max() - np.median(end),
             "consumer_compute_per_unit": comp.sum() / units.sum(),
             "consumer_wait_per_unit": wait.sum() / units.sum(),
             "units_per_cta_min": units.min(), "units_per_cta_max": units.max()}
        if ell > 0:
            prev_end = rec[(ell - 1) * ctas:ell * ctas, 4].max()
            d["first_unit_ready_after_previous_launch_end"] = np.median(first) - prev_end
        per.append(d)
    out = {}
    for k in per[-1]:
        vals = [p[k] for p in per[1:] if k in p]
        scale = 1.0 if k.startswith("units") else 1e-3
        out[k] = round(float(np.median(vals)) * scale, 3)
    out["launches"] = len(per)
    return out


def run_timeline(args) -> dict:
    """One 69-layer graph step with the timeline build of the library: the
    per-CTA records summarised per launch, for the dynamic (work queue) and
    the static schedule.  The recording itself slows the kernel slightly;
    the step times here are not bench figures."""
    import torch

    from linear_attention_decode_04_gb300 import binding
    from linear_attention_decode_04_gb300 import workloads as W
    from linear_attention_decode_04_gb300.stack import DecodeStack
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    layers, _, spec, _ = build_stack(dev, W.STACK_LAYERS, 0)
    res = {"mode": "timeline", "workload": W.STACK_LAYER.name, "layers": W.STACK_LAYERS,
           "note": "timeline build (per-CTA %globaltimer records); us; medians over launches 2..69"}
    for name, q in (("work_queue", True), ("static", False)):
        stack = DecodeStack(layers, eps=spec.eps, work_queue=q)
        stream = torch.cuda.Stream(dev)
        stack.capture(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                stack.replay()
        torch.cuda.synchronize(dev)
        binding.timeline_reset()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            stack.replay()
        torch.cuda.synchronize(dev)
        rec = binding.timeline_read()
        if len(rec) != W.STACK_LAYERS * min(sms, spec.N * spec.H):
            raise SystemExit(f"timeline: {len(rec)} records")
        res[name] = timeline_summary(rec, min(sms, spec.N * spec.H))
        del stack
    return res


def run_spec_timeline(args) -> dict:
    """The multi-token batch with the timeline build: per CTA the time
    waiting for a unit's data, in the state-independent phase, in the token
    loop (including waits for an output buffer), medians over the CTAs of
    one launch, per unit and per token; us."""
    import torch

    from linear_attention_decode_04_gb300 import binding
    from linear_attention_decode_04_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    spec_res = spec_launch(dev, W.MULTI_BENCH, args.warmup, 3, reset_timeline_before_last=True)
    rec = spec_res.pop("_timeline").astype(np.float64)
    units = rec[:, 5]
    tokens = units * W.MULTI_BENCH.T
    per_unit = lambda col: float(np.median(rec[:, col] / np.maximum(units, 1))) / 1e3  # noqa: E731
    res = {"mode": "spec_timeline", "workload": W.MULTI_BENCH.name, "ctas": int(len(rec)),
           "units_per_cta_median": float(np.median(units)),
           "launch_us": float((rec[:, 4].max() - rec[:, 2].min()) / 1e3),
           "per_unit_us": {"waiting_for_data": per_unit(7), "state_independent_phase": per_unit(3),
                           "token_loop": per_unit(6), "of_which_waiting_for_an_output_buffer": per_unit(1)},
           "token_loop_per_token_us": float(np.median(rec[:, 6] / np.maximum(tokens, 1))) / 1e3,
           "note": "timeline build; padding sequences count as units with no tokens"}
    return res


def run_reference(args) -> dict | None:
    """The oracle as it stands, timed on the host cores on a bounded sample
    of the same workload (rank 0 only)."""
    from linear_attention_decode_04_gb300 import workloads as W
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    host = [W.make_inputs(W.stack_layer_spec(ell)) for ell in range(args.ref_layers)]
    n_active = len(host[0].active_rows())
    units = n_active * host[0].H * len(host)
    import oracle
    threads = os.cpu_count() or 1

    def step():
        for x in host:
            oracle.decode(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state,
                          g=x.g, beta=x.beta, slot_idx=x.slot_idx, H=x.H, gate=x.gate,
                          norm_weight=x.norm_weight, eps=x.spec.eps, threads=threads,
                          want_f64=False, in_place=True)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = units / dt
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": W.STACK_LAYER.name, "layers_sampled": len(host), "N": 64, "H": 48},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{len(host)} of 69 layers per step ({units} updates)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing")
    ap.add_argument("--ref-layers", type=int, default=2, help="layers per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-workload", choices=("bench", "profile"), default="bench",
                    help="--case prefill: the measured 16,384-token batch, or a 4,096-token batch for "
                         "profiler captures")
    ap.add_argument("--no-cfg3", action="store_true",
                    help="skip the N=256/H=96 single-launch, multi-token and prefill measurements in the "
                         "headline line")
    ap.add_argument("--case", choices=("stack69", "layer", "roofline", "chunk_metadata", "prefill", "spec",
                                       "configs", "timeline", "spec_timeline"),
                    default="stack69",
                    help="stack69: the headline 69-layer graph step; layer / roofline: one "
                         "launch configuration timed on its own (profiling aid); prefill: the "
                         "chunked varlen prefill")
    args = ap.parse_args(argv)
    if args.case in ("timeline", "spec_timeline"):  # the library with the per-CTA timeline compiled in
        os.environ["KDA_DECODE_TIMELINE"] = "1"
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        res = run_reference(args)
    elif args.case == "chunk_metadata":
        res = run_chunk_metadata(args)
    elif args.case == "prefill":
        res = run_prefill(args)
    elif args.case == "timeline":
        res = run_timeline(args)
    elif args.case == "spec_timeline":
        res = run_spec_timeline(args)
    elif args.case == "configs":
        import torch

        from linear_attention_decode_04_gb300 import workloads as W
        torch.cuda.set_device(0)
        rows = []
        with ClockSampler(0) as clk:
            for spec in W.SPECS.values():
                rows.append(single_launch(torch.device("cuda", 0), spec, args.warmup, max(args.steps, 50)))
        res = {"mode": "configs", "configs": rows, "clocks": clk.summary(), "steps": args.steps,
               "warmup": args.warmup,
               "note": "each decode workload as one launch replayed from a CUDA graph; the state evolves "
                       "across replays; configurations whose pools fit in L2 read part of them from L2"}
    elif args.case == "spec":
        import torch

        from linear_attention_decode_04_gb300 import workloads as W
        torch.cuda.set_device(0)
        with ClockSampler(0) as clk:
            res = spec_launch(torch.device("cuda", 0), W.MULTI_BENCH, args.warmup, args.steps)
        res.update(mode="spec", clocks=clk.summary(), steps=args.steps, warmup=args.warmup)
    elif args.case != "stack69":
        res = run_case(args)
    else:
        res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
