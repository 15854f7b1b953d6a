#!/usr/bin/env python
"""Benchmark of the W8A8 projection path on one GB300 (replicas for N > 1).

A step is one pass of the whole workload's hot path over one batch: every
activation quantizer call and every projection GEMM (with its fused epilogue;
LoRA adds where the workload has them).  Headline workload (the largest one
that fits one GPU): all INT8 projections of one 27B-shaped decoder layer at
24,032 tokens (16 records of 1,502) -- q|k|v packed 5120 -> 6144 + 1024 +
1024, o 6144 -> 5120, gate/up 5120 -> 2 x 17408 with SwiGLU, down 17408 ->
5120 -- each with a rank-256 runtime LoRA pair.

Printed (rank 0, one JSON line): whole-step W8A8 GEMM throughput in TOPS
(2*M*N*K per projection, counted once), the end-to-end figure through the
C ABI with host buffers, the roofline of the dominant kernel from CUDA events
recorded on its stream (in a separate pass of up to 100 steps with an event
pair around every launch; the timed steps carry only the step's own pair),
the quantizer's GB/s, clocks sampled during the timed region, the CPU oracle
timed on a bounded sample on the host cores, and under "configs" the other
four workloads timed in the same process (step throughput, every GEMM's
fraction of its tensor peak, kernel times; the FP8 layer among them).
``--impl reference`` times that oracle as the reference arm instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import clef_synth as S  # noqa: E402

METRIC = "W8A8 linear TOPS & % of GB300 dense INT8/FP8 peak; quantizer GB/s vs HBM"
L2_FLUSH_BYTES = 256 << 20
CPU_SAMPLE_S = 10.0   # target length of the timed oracle sample
INSTRUMENTED_STEPS = 100   # steps of the per-kernel timing pass
HOST_AHEAD_CYCLES = 2_000_000   # about 1 ms of device sleep before each timed or instrumented step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="clef", choices=["clef", "reference"])
    ap.add_argument("--config", default="int8-layer-27b-m24032-lora256",
                    help="workload name (or its position 0-4 in the workload table) of the headline line")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads in the same process")
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the headline workload at this many tokens instead (a smaller case of the "
                         "same kernels, for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch in plain stream order (no programmatic dependent launch)")
    return ap.parse_args()


def measured_traffic(cfg, proj):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when that kernel's source changed since the capture.
    The record names the gemm.cu it was captured on, and may list later
    gemm.cu sources whose changes lie outside the captured kernel's
    instantiation (each with its reason in the summary)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        src = os.path.join(ROOT, "w8a8_quantized_projections_gb300", "csrc", "gemm.cu")
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        same = [rec["gemm_cu_sha256_prefix"]] + rec.get("same_kernel_sources", [])
        if h not in same or not rec["workload"].startswith(cfg.name + " " + proj):
            return None
        return rec["dram_read_bytes"] + rec["dram_write_bytes"]
    except Exception:
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mp = json.load(f)
        return mp["hbm_gbs"], mp["bf16_tflops"], mp.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
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
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle sample

def _par(fn, n, threads):
    from concurrent.futures import ThreadPoolExecutor
    chunk = max(1, -(-n // threads))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda a: fn(a, min(n, a + chunk)), range(0, n, chunk)))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(len(parts[0]))) \
        if isinstance(parts[0], tuple) else np.concatenate(parts)


def oracle_weights(cfg, weights, threads):
    """The oracle's own quantisation of every weight (set-up, not timed)."""
    import oracle as O
    qfn = (lambda x: O.quant_fp8(x)) if cfg.scheme == "fp8" else O.quant_int8_h128
    return {name: _par(lambda a, b: qfn(W[a:b]), W.shape[0], threads) for name, (W, _) in weights.items()}


def oracle_sample(cfg, acts, weights, qw, lora, rows, threads):
    """Run the oracle over `rows` (row indices) of the workload; returns
    (seconds, algorithmic GEMM ops covered)."""
    import oracle as O

    def par(fn, n):
        return _par(fn, n, threads)

    fp8 = cfg.scheme == "fp8"
    qfn = (lambda x: O.quant_fp8(x)) if fp8 else O.quant_int8_h128
    R = len(rows)
    xs = {name: np.ascontiguousarray(x[rows]) for name, x in acts.items()}
    t0 = time.perf_counter()

    def run_rows(a, b):
        q = {name: qfn(x[a:b]) for name, x in xs.items()}
        h = None
        out = None
        for p in cfg.projections:
            wq, ws = qw[p.name]
            bias = weights[p.name][1]
            qx, sx = qfn(h) if p.chained else q[p.act]
            if p.kind == "gateup":
                if lora:
                    y = (O.fp8_linear if fp8 else O.int8_linear)(qx, sx, wq, ws, bias)
                    N = p.N
                    x = xs[p.act][a:b]
                    y[:, :N] = O.lora_add(x, *lora[p.name + "/gate"], y[:, :N])
                    y[:, N:] = O.lora_add(x, *lora[p.name + "/up"], y[:, N:])
                    h = O.swiglu_bf16(y)
                elif fp8:
                    h = O.fp8_gateup_swiglu(qx, sx, wq, ws, bias)
                else:
                    h = O.int8_gateup_swiglu(qx, sx, wq, ws, bias)
                out = h
            else:
                out = (O.fp8_linear if fp8 else O.int8_linear)(qx, sx, wq, ws, bias)
                if lora and p.name in lora:
                    A, B = lora[p.name]
                    out = O.lora_add(xs[p.act][a:b] if not p.chained else h, A, B, out)
        return (out,)

    par(run_rows, R)
    dt = time.perf_counter() - t0
    ops = sum(p.ops(R) for p in cfg.projections)
    return dt, ops


def cpu_threads():
    return max(1, os.cpu_count() or 1)


def sample_rows(cfg, n):
    rng = np.random.default_rng(1234)
    return np.sort(rng.choice(cfg.M, size=min(n, cfg.M), replace=False))


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = S.workload(args.config)
    acts, weights, lora = S.layer_inputs(cfg, seed=0)
    threads = cpu_threads()
    per_step_rows = threads  # one row per host thread per step
    rows = sample_rows(cfg, per_step_rows)
    qw = oracle_weights(cfg, weights, threads)
    for _ in range(args.warmup):
        oracle_sample(cfg, acts, weights, qw, lora, rows, threads)
    times, ops = [], 0
    for _ in range(args.steps):
        dt, ops = oracle_sample(cfg, acts, weights, qw, lora, rows, threads)
        times.append(dt)
    tot = sum(times)
    value = ops * args.steps / tot / 1e12
    sample = f"{len(rows)} of {cfg.M} token rows per step through every projection of {cfg.name}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8" if cfg.scheme == "fp8" else "int8", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PDL = True   # the library's programmatic-dependent-launch switch for this run


def workload_config(cfg):
    d = {"workload": cfg.name, "tokens": cfg.M, "scheme": cfg.scheme,
         "projections": {p.name: [p.K, p.weight_rows] for p in cfg.projections},
         "l2": "flushed between steps (256 MiB write, outside the per-step events)",
         "launch": "programmatic dependent launch" if PDL else "plain stream order"}
    if cfg.lora_rank:
        d["lora_rank"] = cfg.lora_rank
    return d


# ---------------------------------------------------------------- replicas (N > 1)

def replica_activations(cfg, acts_np, rank):
    """Each rank's own batch: rank 0 keeps the workload's seed-0 activations,
    rank r > 0 draws its own seeded tensors of the same shapes (weights are
    shared by seed, so every rank runs the same layer)."""
    if rank == 0:
        return acts_np
    return {n: S.activation(rank, f"{cfg.name}/act/{n}", cfg.M, x.shape[1]) for n, x in acts_np.items()}


def max_over_ranks(value, world, dist, device):
    """The largest of the ranks' values (timed seconds): the whole job takes as
    long as its slowest replica."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tops(ops_per_step, steps, world, seconds):
    """Throughput of all replicas together: every rank ran `steps` steps."""
    return ops_per_step * steps * world / seconds / 1e12


# ---------------------------------------------------------------- GPU arm

def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    import w8a8_quantized_projections_gb300 as clef
    global PDL
    PDL = not args.no_pdl
    clef.set_pdl(PDL)
    dev = torch.device("cuda", local)
    cfg = S.workload(args.config)
    if args.tokens:
        import dataclasses
        cfg = dataclasses.replace(cfg, M=args.tokens)
    env = Env(args, rank, world, dev, dist, torch)

    line = measure(env, cfg, args.steps, headline=True)
    line["peaks"] = env.peaks_line()
    # ---- CPU oracle on a bounded sample of the headline workload (rank 0,
    # N = 1): a probe of two rows per host thread sizes a sample of about
    # CPU_SAMPLE_S seconds
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        acts_np, weights_np, lora_np = env.inputs
        threads = cpu_threads()
        qw = oracle_weights(cfg, weights_np, threads)
        probe = sample_rows(cfg, 2 * threads)
        dt0, _ = oracle_sample(cfg, acts_np, weights_np, qw, lora_np, probe, threads)
        n = int(min(cfg.M, max(len(probe), len(probe) * CPU_SAMPLE_S / max(dt0, 1e-3))))
        rows = sample_rows(cfg, n)
        dt, ops = oracle_sample(cfg, acts_np, weights_np, qw, lora_np, rows, threads)
        line["cpu_baseline"] = {"value": ops / dt / 1e12, "unit": "TOPS", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{len(rows)} of {cfg.M} token rows through every projection "
                                          f"of {cfg.name} ({dt:.1f} s on {threads} threads)"}
        del qw
    env.inputs = None
    # the other workloads, timed in the same process (rank 0 at N = 1): each
    # with its own step throughput, dominant kernel fraction and kernel times
    if rank == 0 and world == 1 and not args.no_configs:
        line["configs"] = {}
        for c in S.CONFIGS.values():
            if c.name == cfg.name:
                continue
            line["configs"][c.name] = measure(env, c, max(args.steps, MIN_STEPS_OTHER), headline=False)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


MIN_STEPS_OTHER = 100   # timed steps of each further workload (their steps take 0.03-1.5 ms)
# CTAs of the end-to-end copies (clef_copy_sm): 4 move 1.62 GB from pinned host
# memory in 7.98 ms (203 GB/s, the link's rate within 4%; 2 CTAs: 102 GB/s), and
# the compute keeps 148 of 152 SMs (the headline step 11.88 -> 12.03 ms)
E2E_COPY_CTAS = 4
MMA_PEAK_ITERS = {"bf16": 100_000, "e4m3": 100_000, "s8_mma_sync": 10_000}


class Env:
    """What every measurement shares: arguments, ranks, device, library, peaks."""

    def __init__(self, args, rank, world, dev, dist, torch):
        import w8a8_quantized_projections_gb300 as clef
        self.args, self.rank, self.world, self.dev, self.dist, self.torch = args, rank, world, dev, dist, torch
        self.clef = clef
        self.hbm_gbs, self.bf16_peak, self.bf16_sust, self.peak_src = peaks()
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # dense tensor rates of the three instruction routes, from the
        # library's own microbenchmark on this device (TFLOP/s)
        self.mma = {k: clef.mma_peak(k, n) for k, n in MMA_PEAK_ITERS.items()}

    def peaks_line(self):
        return {"bf16_matmul_measured": self.bf16_peak, "bf16_source": f"{self.peak_src} (cuBLAS bf16, burst)",
                "microbenchmark_tflops": self.mma,
                "note": "clef_mma_peak: tcgen05 kind::f16 (bf16) and kind::f8f6f4 (e4m3) MMAs issued back "
                        "to back from shared memory by one CTA pair per two SMs; mma.sync m16n8k32 s8 "
                        "(the legacy integer route) on register operands"}

    def fp8_ratio(self):
        """e4m3 over bf16 dense rate of the tensor pipe, measured by the
        microbenchmark (both routes at the same clock in one process)."""
        return self.mma["e4m3"] / self.mma["bf16"]

    def tensor_peak(self, scheme):
        """(peak TFLOP/s, source) of the tensor pipe a scheme's GEMMs run on.

        The bf16 figure is the measured cuBLAS bf16 matmul rate; the e4m3 one
        is that figure times the e4m3/bf16 ratio the microbenchmark measures
        on this GPU, so both denominators are full GEMMs under the same power
        and clock behaviour.  The microbenchmark's own figures (MMAs issued
        from shared memory with no copies, a short burst at full clock) are
        higher and are reported beside them."""
        if scheme == "fp8":
            r = self.fp8_ratio()
            return (self.bf16_peak * r,
                    f"{self.peak_src} bf16 dense burst x {r:.3f}, the e4m3/bf16 ratio measured by the "
                    f"tcgen05 microbenchmark (kind::f8f6f4 {self.mma['e4m3']:.0f}, kind::f16 "
                    f"{self.mma['bf16']:.0f} TFLOP/s)")
        return (self.bf16_peak, f"{self.peak_src} bf16 dense burst (INT8 runs exactly on the fp16 "
                                f"tensor pipe: sm_103a has no tcgen05 integer MMA; the legacy mma.sync "
                                f"s8 route measures {self.mma['s8_mma_sync']:.0f})")


def measure(env, cfg, steps, headline):
    """One workload: its step timed `steps` times (L2 flushed between steps),
    per-kernel times from a separate instrumented pass, the dominant GEMM's
    roofline, the LoRA and quantizer figures, and the step replayed from a
    CUDA graph.  The headline workload also gets the clocks, the quantizer
    streaming figure and the end-to-end figure with host buffers, its dict is
    the bench line itself, and its host inputs are kept in env.inputs for the
    CPU oracle baseline."""
    torch, clef, args = env.torch, env.clef, env.args
    from w8a8_quantized_projections_gb300.layer import QuantizedLayer
    dev, stream, flush, world, rank = env.dev, env.stream, env.flush, env.world, env.rank

    # replicas: each rank works on its own batch (seeded by rank), weights shared by seed
    acts_np, weights_np, lora_np = S.layer_inputs(cfg, seed=0)
    acts_np = replica_activations(cfg, acts_np, rank)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    weights = {k: (bf(W), bf(b)) for k, (W, b) in weights_np.items()}
    lora = {k: (bf(A), bf(B)) for k, (A, B) in lora_np.items()}
    acts = {k: bf(x) for k, x in acts_np.items()}
    layer = QuantizedLayer(cfg, weights, lora or None, device=dev)
    del weights
    ops_step = cfg.gemm_ops()

    for _ in range(args.warmup):
        layer.step(acts)
    torch.cuda.synchronize(dev)
    assert layer.poll_status() == 0
    # a step shorter than about 2 ms can be host-bound (its launches issued
    # from Python while the device waits): such steps are each queued behind a
    # short device sleep, outside their events, so that the host is ahead and
    # the events hold device time only (the 298-token step read 560-600 us in
    # two runs without it, 31 us otherwise).  Longer steps run back to back.
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    layer.step(acts)
    w1.record(stream)
    torch.cuda.synchronize(dev)
    host_ahead = w0.elapsed_time(w1) < 2.0

    # ---- device-timed steps (inputs resident in HBM)
    events = {}
    step_ev = []
    clocks = ClockSampler(dev.index) if headline else None
    if clocks:
        clocks.start()
    if world > 1 and headline:
        env.dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for _ in range(steps):
        flush.zero_()
        if host_ahead:
            torch.cuda._sleep(HOST_AHEAD_CYCLES)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        layer.step(acts)
        s1.record(stream)
        step_ev.append((s0, s1))
    torch.cuda.synchronize(dev)
    if world > 1 and headline:
        env.dist.barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop() if clocks else None
    status = layer.poll_status()
    if status:
        raise RuntimeError(f"device status word reported {status}")
    # per-kernel times from a separate pass with an event pair around every
    # launch (the events themselves cost about 2 us each, so the timed steps
    # above carry only the step's own pair); each instrumented step is queued
    # behind a short device sleep so that the host has issued all of its
    # launches before the first one starts, and no host gap sits between an
    # event pair
    n_inst = min(steps, INSTRUMENTED_STEPS)
    for _ in range(n_inst):
        flush.zero_()
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        layer.step(acts, events=events)
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    t_sum = sum(step_ms) / 1e3
    if headline:
        t_sum = max_over_ranks(t_sum, world, env.dist, dev)
    value = whole_job_tops(ops_step, steps, world if headline else 1, t_sum)

    kt = {key: [a.elapsed_time(b) / 1e3 for a, b in lst] for key, lst in events.items()}
    gemm_keys = [k for k in kt if k[0] == "gemm"]
    units = {u[0]: u for u in layer.units()}   # name -> (name, weight rows, K, ops, fused LoRA flops)
    dom = max(gemm_keys, key=lambda k: sum(kt[k]))
    dom_name, dom_rows, dom_K, dom_base, dom_lora = units[dom[1]]
    dom_ops = dom_base + dom_lora   # a fused LoRA expand's tensor work is part of the launch
    dom_t = statistics.mean(kt[dom])
    achieved = dom_ops / dom_t / 1e12
    peak, peak_source = env.tensor_peak(cfg.scheme)
    q_bytes, q_time = 0, 0.0
    for key, lst in kt.items():
        if key[0] != "quant":
            continue
        K = acts_np[key[1]].shape[1] if key[1] in acts_np else proj_input_K(cfg, key[1])
        q_bytes += (3 * cfg.M * K + 4 * cfg.M) * len(lst)
        q_time += sum(lst)
    q_gbs = q_bytes / q_time / 1e9 if q_time else None
    gemm_time = sum(sum(kt[k]) for k in gemm_keys)
    gemm_tops = ops_step * n_inst / gemm_time / 1e12
    gemms = {}
    for k in gemm_keys:
        _, rows, K, base, lora_fl = units[k[1]]
        ops = base + lora_fl
        t = statistics.mean(kt[k])
        gemms[k[1]] = {"shape": f"{cfg.M}x{rows}x{K}", "ms": 1e3 * t, "tops": ops / t / 1e12,
                       "fused_lora_flops": lora_fl,
                       "frac": ops / t / 1e12 / peak,
                       "frac_of_microbenchmark": ops / t / 1e12 / env.mma["e4m3" if cfg.scheme == "fp8" else "bf16"]}

    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_sum / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8" if cfg.scheme == "fp8" else "int8", "data": "synthetic",
        "config": dict(workload_config(cfg), step_timing="each step queued behind a 1 ms device sleep outside its events (steps under 2 ms)" if host_ahead else "steps back to back"),
        "roofline": {
            "kernel": f"{'fp8' if cfg.scheme == 'fp8' else 'w8a8'} {dom_name} GEMM "
                      f"({cfg.M}x{dom_rows}x{dom_K})",
            "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "traffic": measured_traffic(cfg, dom_name) if headline else None,
            "traffic_unit": "bytes per launch",
            "ops_per_launch": dom_ops, "fused_lora_flops_per_launch": dom_lora, "launch_ms": 1e3 * dom_t,
            "peak_source": peak_source,
        },
        "gemm_only_tops": gemm_tops,
        "gemms": gemms,
        "quantizer": {"achieved": q_gbs, "unit": "GB/s", "peak": env.hbm_gbs,
                      "frac": (q_gbs / env.hbm_gbs) if q_gbs else None,
                      "bytes_per_element": 3, "bytes_per_row": 4},
        "kernel_ms": {f"{k[0]}:{k[1]}": 1e3 * statistics.mean(v) for k, v in kt.items()},
        "gpu_launches": layer.launches_per_step() * steps,
    }
    if headline:
        line["clocks"] = clk
        line["wall_s_timed_region"] = wall

    # ---- LoRA launches (runtime adapters): bf16 tensor-core work, near the ridge
    lora_keys = [k for k in kt if k[0] == "lora"]
    if lora_keys:
        l_fl, l_by = layer.lora_work()
        l_t = sum(statistics.mean(kt[k]) for k in lora_keys)
        line["lora"] = {"ms_per_step": 1e3 * l_t, "launches_per_step": len(lora_keys),
                        "tflops": l_fl / l_t / 1e12, "tflops_frac": l_fl / l_t / 1e12 / env.bf16_peak,
                        "gbs": l_by / l_t / 1e9, "gbs_frac": l_by / l_t / 1e9 / env.hbm_gbs,
                        "flops_per_step": l_fl, "min_bytes_per_step": l_by,
                        "note": ("LoRA expands fused into the INT8 GEMMs: these launches are the x A^T "
                                 "shrinks (2 M r K flops per adapter; x read, t written); the expand's "
                                 "2 M N r flops count in the GEMMs' figures" if layer.fused else
                                 "2 M r (K + N) flops per adapter; bytes: x once per shrink launch, "
                                 "t written and read, y read and written (gate/up: base halves "
                                 "read, h written)") + "; against the bf16 burst peak and the copy bandwidth"}

    # ---- the quantizer streaming: alone on 16 records of the widest activation
    if headline:
        line["quantizer"]["stream"] = quantizer_stream(cfg, acts_np, dev, stream, flush, env.hbm_gbs,
                                                       clef, torch)

    # ---- the same step replayed from a CUDA graph (launch overhead removed)
    layer.capture(acts)
    g_ev = []
    for _ in range(args.warmup):
        layer.replay()
    torch.cuda.synchronize(dev)
    for _ in range(steps):
        flush.zero_()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        layer.replay()
        g1.record(stream)
        g_ev.append((g0, g1))
    torch.cuda.synchronize(dev)
    g_t = sum(a.elapsed_time(b) for a, b in g_ev) / 1e3
    line["graph"] = {"value": ops_step * steps / g_t / 1e12, "unit": "TOPS",
                     "ms_per_step": 1e3 * g_t / steps,
                     "note": "the step captured once in a CUDA graph and replayed (one launch per step)"}

    # ---- end to end through the C ABI with host buffers
    if headline and not args.no_e2e:
        line["e2e"] = e2e(args, layer, acts, acts_np, cfg, dev, stream, world, torch)

    if headline:
        env.inputs = (acts_np, weights_np, lora_np)
    del layer, acts, lora
    torch.cuda.empty_cache()
    return line


def proj_input_K(cfg, act):
    for p in cfg.projections:
        if p.act == act:
            return p.K
    raise KeyError(act)


def quantizer_stream(cfg, acts_np, dev, stream, flush, hbm_gbs, clef, torch, records=16, reps=20):
    """The workload's quantizer on `records` x M rows of its widest activation
    (the batched size of the pages' throughput note), L2 flushed before each
    call: its streaming bandwidth, apart from the start-up cost that dominates
    the step's small calls."""
    K = max(p.K for p in cfg.projections)    # the widest projection input (h for the MLP)
    # 16 records, but at least 512 MB of bf16 input (4x the 126 MB L2) and at most 1 GB
    rows = max(cfg.M * records, -(-(512 << 20) // (2 * K)))
    rows = min(rows, (1 << 30) // (2 * K))
    mode = "fp8" if cfg.scheme == "fp8" else "int8_h128"
    x = torch.empty((rows, K), dtype=torch.bfloat16, device=dev).normal_()
    q = torch.empty((rows, K), dtype=torch.uint8 if mode == "fp8" else torch.int8, device=dev)
    s = torch.empty((rows,), dtype=torch.float32, device=dev)
    clef.quant_act(x, mode, q=q, scale=s)
    ts = []
    for _ in range(reps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        clef.quant_act(x, mode, q=q, scale=s)
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize(dev)
    t = statistics.median(a.elapsed_time(b) for a, b in ts) / 1e3
    gbs = (3 * rows * K + 4 * rows) / t / 1e9
    del x, q, s
    return {"rows": rows, "K": K, "achieved": gbs, "unit": "GB/s", "peak": hbm_gbs, "frac": gbs / hbm_gbs,
            "note": f"the same kernel alone on {rows} rows of the widest activation, median of "
                    f"{reps} calls with L2 flushed; the step's own calls are start-up bound"}


def weight_bytes(layer):
    """Bytes of quantized weights one step reads (codes and scales)."""
    return sum(qw.numel() * qw.element_size() + sw.numel() * sw.element_size()
               for qw, sw, _ in layer.unit_w)


def e2e(args, layer, acts, acts_np, cfg, dev, stream, world, torch):
    """Same metric with host buffers: every step copies its activations in
    from pinned host memory and its final output back, inside the timing.
    The copies run on a second stream, pipelined with the compute: step i+1's
    inputs are copied into the other of two device input sets while step i
    computes, and step i's output is read back while step i+1's first kernels
    run (its last projection waits for that read before overwriting the
    output buffer).  The copies are the library's clef_copy_sm on
    E2E_COPY_CTAS CTAs, and the compute runs under an SM budget that leaves
    them those SMs: copy-engine transfers from pinned host memory stalled
    for 20-180 ms about every half second on some boxes (200 steps at
    14.8-17.5 ms against 11.8 ms without the stalls) and rarely on others
    (1,000 steps at 12.01 ms against 12.35 ms with the SM copies); SM loads
    over the same link did not stall on any box tried."""
    host_in = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).pin_memory()
               for k, v in acts_np.items()}
    last = cfg.projections[-1].name
    out_dev = layer.out[last]
    host_out = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    dev_in = [{k: torch.empty_like(v) for k, v in acts.items()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    copy = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    import w8a8_quantized_projections_gb300 as clef
    ctas = E2E_COPY_CTAS
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def move(dst, src):
        clef.copy_sm(dst, src, ctas, stream=copy)

    def run(n):
        in_ready = [ev(), ev()]
        used = [None, None]          # step that last read input set b has finished
        read_back = None             # the previous step's output has been read
        with torch.cuda.stream(copy):
            for k in dev_in[0]:
                move(dev_in[0][k], host_in[k])
            in_ready[0].record(copy)
        for i in range(n):
            b = i % 2
            if i + 1 < n:            # next step's inputs, into the other set
                with torch.cuda.stream(copy):
                    if used[1 - b] is not None:
                        copy.wait_event(used[1 - b])
                    for k in dev_in[1 - b]:
                        move(dev_in[1 - b][k], host_in[k])
                    in_ready[1 - b].record(copy)
            stream.wait_event(in_ready[b])
            layer.step(dev_in[b], final_wait=read_back)
            done = ev()
            done.record(stream)
            used[b] = done
            with torch.cuda.stream(copy):
                copy.wait_event(done)
                move(host_out, out_dev)
                read_back = ev()
                read_back.record(copy)
        stream.wait_event(read_back)

    clef.set_sm_budget(sms - ctas)
    try:
        run(2)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(args.steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    finally:
        clef.set_sm_budget(0)
    t = e0.elapsed_time(e1) / 1e3
    return {"value": cfg.gemm_ops() * args.steps * world / t / 1e12, "unit": "TOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": f"clef_copy_sm on {ctas} CTAs beside the compute, which runs under an SM "
                      f"budget of {sms - ctas} of {sms}",
            "note": "input copies of step i+1 and the read-back of step i overlap the compute "
                    "on a second stream; every step's copies are inside the timed region; no "
                    "L2 flush between steps (each step streams all weights, "
                    f"{weight_bytes(layer) / 1e6:.0f} MB, against a 126 MB L2)"}


if __name__ == "__main__":
    main()
