"""Benchmark of the frame-locked batched decode step (one JSON line).

Default workload: the 7B-class temporal-transformer frame step (32 layers,
d=4096, 32 heads x 128, SwiGLU 11008, bf16 weights, FP8 e4m3 K/V history
with per-(session, head, token) scales), S = 80 sessions, positions uniform
in [0, 3000).  Metric: session-frames/s = S / step time, with p50/p99 step
latency and the HBM roofline fraction of the step kernel.

  python bench.py [--gpus N --steps K --warmup W] [--S 80] [--impl reference]
  python bench.py --sweep 1,8,16,32,48,56,64,80,96,128 --steps 20
  python bench.py --beat 2
  python bench.py --depth [--phases]
  python bench.py --hybrid [--phases] [--layers 6k]
  python bench.py --phases [--layers L]      (per-phase times of one step)

Inputs are seeded and synthetic and are drawn on the device (weights and the
raw history by the generator's device twin, the history quantised by the
library's own quantiser); every input is far larger than L2, so no flush is
needed between steps.  With --gpus N > 1 (launched by torchrun) every rank
runs an independent replica of S sessions on its own GPU: sessions shard
with no collective on the data path.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "session-frames/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "step_kernel_7b_traffic.txt")
FALLBACK_HBM_GBS = 6800.0
# Every source the step kernel compiles from, in a fixed order: the committed
# traffic figure holds only while their joint hash is the one it was taken on.
STEP_SRCS = [os.path.join(ROOT, "frame_step_decode_gb300", "csrc", f)
             for f in ("step.cu", "internal.h", "ptx.cuh", "fp8.cuh")]


def step_sources_sha():
    h = hashlib.sha256()
    for path in STEP_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(w, pos) -> int:
    """Weights once + FP8 K/V codes and scales of slots 0..pos read + the
    appended slot written, per step."""
    L, H, D = w.n_layers, w.n_heads, w.head_dim
    weights = 2 * synth.weight_elems(w)
    kv_read = sum(L * 2 * H * (int(p) + 1) * (D + 4) for p in pos)
    kv_write = L * 2 * len(pos) * H * (D + 4)
    return weights + kv_read + kv_write


# The read-bound model of ttlab "voice-agent principles", §2 "Conversational
# LLM": a step reads every weight once, so it cannot be shorter than its bytes
# over the memory bandwidth; batching adds 2 flops per parameter per request
# but no reads.  The page works examples of each relation;
# tests/golden/roofline_examples.txt holds them.
def read_bound_per_s(bandwidth_gbs, gb_per_unit):
    """Units (tokens, steps) per second at most when each reads gb_per_unit GB."""
    return bandwidth_gbs / gb_per_unit


def fixed_cost_ms(rate_per_s, gb_per_unit, bandwidth_gbs):
    """Time per unit beyond reading its bytes: 1 / rate - bytes / bandwidth (ms)."""
    return 1e3 / rate_per_s - 1e3 * gb_per_unit / bandwidth_gbs


def compute_bound_concurrency(tflops, bandwidth_gbs, bytes_per_param):
    """Requests sharing one weight read past which their 2 flops per parameter
    outrun the read: F * bytes_per_param / (2 * BW)."""
    return tflops * 1e12 * bytes_per_param / (2.0 * bandwidth_gbs * 1e9)


def matmul_tflops(params, rate_per_s):
    """2 flops per parameter per token at rate_per_s tokens/s, in TFLOP/s."""
    return 2.0 * params * rate_per_s / 1e12


def algorithmic_flops(w, pos) -> int:
    L, H, D, d, F = w.n_layers, w.n_heads, w.head_dim, w.d_model, w.ffn
    HD = H * D
    gemm = 2 * len(pos) * L * (3 * HD * d + d * HD + 2 * F * d + d * F)
    attn = sum(4 * D * L * H * (int(p) + 1) for p in pos)
    return gemm + attn


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def traffic_per_launch():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    vals = {}
    with open(PROFILE_TRAFFIC) as f:
        lines = f.readlines()
    for line in lines:
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("step_sources_sha256_16") != step_sources_sha():
        return None
    try:
        return int(float(vals["dram_bytes_per_full_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- oracle arm
def oracle_session_time(w, sessions, pos):
    """Time the CPU oracle for the listed sessions of workload w (its inputs
    prepared outside the timed region).  Returns (seconds, threads)."""
    import oracle
    W = synth.weights_host(w)
    x = synth.x_bf16(w)[sessions]
    p = np.asarray(pos)[sessions].astype(np.int32)
    kv, sc = oracle.prefill_history(w, sessions, p, poison=False)
    t0 = time.perf_counter()
    oracle.step(w, W, kv, sc, p, x)
    dt = time.perf_counter() - t0
    return dt, os.cpu_count()


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    pos = synth.positions(w, args.S)
    W = synth.weights_host(w)
    sess = [0]
    x = synth.x_bf16(w)[sess]
    p = pos[sess]
    kv, sc = oracle.prefill_history(w, sess, p, poison=False)
    kv0, sc0 = kv.copy(), sc.copy()
    for _ in range(min(args.warmup, 1)):
        oracle.step(w, W, kv, sc, p, x)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        kv[...] = kv0
        sc[...] = sc0
        t0 = time.perf_counter()
        oracle.step(w, W, kv, sc, p, x)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    ms = 1000 * total / args.steps
    value = len(sess) / (total / args.steps)
    sample = f"1 of {args.S} sessions (session 0, pos {int(p[0])}) of {w.name}, per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": METRIC, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": min(args.warmup, 1), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "S": args.S, "T_max": w.T_max,
                   "positions": f"uniform [{w.pos_lo}, {w.pos_hi})"},
        "cpu_baseline": {"value": value, "unit": METRIC, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": METRIC, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_all,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------ multi-GPU replicas
def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    replica sets the job's time); identity without a process group."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world: int, S: int, ms_per_step: float) -> float:
    """Whole-job session-frames/s: every rank advances its own S sessions
    (replicas, no collective on the data path) in the max-over-ranks time."""
    return world * S / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ GPU arm
def build_inputs(w, S, device):
    import torch
    import frame_step_decode_gb300 as fsd
    stream = torch.cuda.current_stream().cuda_stream
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    rm = torch.empty(synth.weight_elems(w), dtype=torch.bfloat16, device=device)
    synth.weights_device(w, rm, stream)
    weights = fsd.pack_weights(fsd.WaveConfig.of(w), rm)   # the packed blob the step reads
    del rm
    kv = torch.empty((L, 2, S, H, T, D), dtype=torch.uint8, device=device)
    sc = torch.empty((L, 2, S, H, T), dtype=torch.float32, device=device)
    raw = torch.empty((S, H, T, D), dtype=torch.float32, device=device)
    for l in range(L):
        for which in range(2):
            synth.kv_raw_device(w, l, which, 0, S, T, raw.data_ptr(), T, stream)
            fsd.kv_quantize(raw, kv[l, which], sc[l, which])
    del raw
    pos_h = synth.positions(w, S)
    pos = torch.from_numpy(pos_h).to(device)
    x = torch.empty((S, w.d_model), dtype=torch.bfloat16, device=device)
    synth.x_device(w, S, x.data_ptr(), stream)
    y = torch.empty_like(x)
    torch.cuda.synchronize()
    return weights, kv, sc, pos, pos_h, x, y


def run_gpu(args, w):
    import torch
    import frame_step_decode_gb300 as fsd
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    S = args.S
    weights, kv, sc, pos, pos_h, x, y = build_inputs(w, S, device)
    wave = fsd.Wave(fsd.WaveConfig.of(w), S, w.T_max)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        wave.step(S, weights, kv, sc, pos, x, y, stream=stream)
    rc = wave.status()
    if rc != fsd.WAVE_OK:
        raise RuntimeError(f"warm-up step failed: {fsd.strerror(rc)}")

    # ---- device-resident timed region
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev0[i].record(stream)
        wave.step(S, weights, kv, sc, pos, x, y, stream=stream)
        ev1[i].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    rc = wave.status()
    if rc != fsd.WAVE_OK:
        raise RuntimeError(f"timed step failed: {fsd.strerror(rc)}")
    per = [ev0[i].elapsed_time(ev1[i]) for i in range(args.steps)]
    total_ms = t_start.elapsed_time(t_end)

    # ---- end to end through the C ABI with host buffers
    x_host = x.cpu().pin_memory()
    pos_host = pos.cpu().pin_memory()
    y_host = torch.empty_like(y, device="cpu").pin_memory()
    for _ in range(2):
        x.copy_(x_host, non_blocking=True)
        pos.copy_(pos_host, non_blocking=True)
        wave.step(S, weights, kv, sc, pos, x, y, stream=stream)
        y_host.copy_(y, non_blocking=True)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        x.copy_(x_host, non_blocking=True)
        pos.copy_(pos_host, non_blocking=True)
        wave.step(S, weights, kv, sc, pos, x, y, stream=stream)
        y_host.copy_(y, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    h2d = x.numel() * 2 + pos.numel() * 4
    d2h = y.numel() * 2

    ms_per_step, e2e_ms = max_over_ranks([total_ms / args.steps, e2e_ms], dist, device)
    if rank == 0:
        bytes_step = algorithmic_bytes(w, pos_h)
        flops_step = algorithmic_flops(w, pos_h)
        kern_ms = statistics.mean(per)
        peak, peak_kind = measured_peaks()
        achieved = bytes_step / (kern_ms * 1e-3) / 1e9
        traffic = traffic_per_launch()
        line = {
            "metric": METRIC,
            "value": job_throughput(world, S, ms_per_step),
            "unit": METRIC,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "p50_ms": statistics.median(per),
            "p99_ms": float(np.percentile(per, 99)),
            "late_frames_over_80ms": int(sum(1 for t in per if t > 80.0)),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded; weights N(0,0.02) bf16, x N(0,1), FP8 e4m3 history of N(0,1))",
            "config": {"workload": w.name, "S": S, "T_max": w.T_max,
                       "positions": f"uniform [{w.pos_lo}, {w.pos_hi})", "kv": "e4m3 + fp32 scales",
                       "parallelism": f"replicas x{world} (sessions shard, no collective)",
                       "l2": "inputs larger than L2 (no flush needed)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                         "frac_of_8000": achieved / 8000.0,
                         "algorithmic_bytes_per_launch": bytes_step,
                         "ceiling_value": S * world * read_bound_per_s(peak, bytes_step / 1e9),
                         "tflops": flops_step / (kern_ms * 1e-3) / 1e12},
            "e2e": {"value": job_throughput(world, S, e2e_ms), "unit": METRIC, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps,
            "clocks": clk,
        }
        if world == 1 and not args.no_cpu_baseline:
            try:
                dt, cores = oracle_session_time(w, [0], pos_h)
                line["cpu_baseline"] = {"value": 1.0 / dt, "unit": METRIC, "cores": cores,
                                        "kind": "oracle",
                                        "sample": f"1 of {S} sessions (session 0, pos {int(pos_h[0])}) of "
                                                  f"{w.name}, one frame"}
            except Exception as e:  # the GPU number stands without it
                line["cpu_baseline"] = {"value": None, "unit": METRIC, "cores": os.cpu_count(),
                                        "kind": "oracle", "sample": f"failed: {e}"}
        print(json.dumps(line), flush=True)
    wave.close()
    if dist is not None:
        dist.destroy_process_group()


def run_phases(args, w):
    """Per-phase times of one step from the kernel's phase-end marks
    (profiling hook): for every phase, when the last CTA finished it minus
    when the last CTA finished the phase before (the critical path; no grid
    barrier separates the phases), averaged over the layers, with the spread
    of the CTAs' finishing times; three steps averaged."""
    import torch
    import frame_step_decode_gb300 as fsd
    device = torch.device("cuda", 0)
    S = args.S
    weights, kv, sc, pos, pos_h, x, y = build_inputs(w, S, device)
    wave = fsd.Wave(fsd.WaveConfig.of(w), S, w.T_max)
    for _ in range(max(3, args.warmup)):
        wave.step(S, weights, kv, sc, pos, x, y)
    n, grid = wave.phases_per_step, wave.grid
    ts = torch.zeros((n, grid), dtype=torch.int64, device=device)
    wave.debug_arrival_times(ts)
    ends, spreads = [], []
    for _ in range(3):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        wave.step(S, weights, kv, sc, pos, x, y)
        ev1.record()
        if wave.status() != fsd.WAVE_OK:
            raise RuntimeError("step failed")
        t = ts.cpu().numpy().astype(np.float64) / 1000.0
        last = t.max(axis=1)
        ends.append(np.diff(np.concatenate([[t.min()], last])))
        spreads.append(last - t.min(axis=1))
    wave.debug_arrival_times(None)
    dur, spr = np.mean(ends, axis=0), np.mean(spreads, axis=0)
    names = ["prologue"]
    for l in range(w.n_layers):
        names += (["norm1"] if l > 0 else []) + ["qkv", "attn", "o", "norm2", "gu", "down"]
    d, HD, F = w.d_model, w.HD, w.ffn
    kvb = sum(2 * w.n_heads * (int(q) + 1) * (w.head_dim + 4) for q in pos_h)
    nbytes = {"qkv": 3 * HD * d * 2, "o": d * HD * 2, "gu": 2 * F * d * 2, "down": d * F * 2, "attn": kvb}
    print(f"{w.name} S={S}: {dur.sum():.1f} us from the first mark (phase = the last CTA's finish minus "
          "the last CTA's finish of the phase before; spread = last minus first CTA)")
    agg = {}
    for nm, v, sp in zip(names, dur, spr):
        agg.setdefault(nm, []).append((v, sp))
    for nm, vs in agg.items():
        m = float(np.mean([v for v, _ in vs]))
        sp = float(np.mean([q for _, q in vs]))
        extra = f"  {nbytes[nm] / m / 1e3:6.0f} GB/s" if nm in nbytes else ""
        print(f"  {nm:8s} x{len(vs):3d}  mean {m:7.1f} us  spread {sp:6.1f} us  total {m * len(vs):9.1f} us "
              f"({100 * m * len(vs) / dur.sum():5.1f}%){extra}")
    wave.close()


# -------------------------------------------------- the other workloads
def timed_runs(launch, steps, runs, stream, gpu_index):
    """`runs` runs of `steps` launches each, every launch timed by its own
    CUDA event pair on `stream`, with nvidia-smi clocks sampled across all
    of them.  Returns ([per-launch ms of each run], clocks)."""
    import torch
    clocks = ClockSampler(gpu_index)
    clocks.start()
    time.sleep(0.3)
    per_run = []
    for _ in range(runs):
        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            ev0[i].record(stream)
            launch()
            ev1[i].record(stream)
        torch.cuda.synchronize()
        per_run.append([a.elapsed_time(b) for a, b in zip(ev0, ev1)])
    return per_run, clocks.stop()


def run_stats(per_run, deadline_ms=None):
    """Mean, p50 and p99 over every timed launch, the same per run, and the
    launches over the deadline."""
    allv = [t for r in per_run for t in r]
    out = {"ms_mean": statistics.mean(allv), "p50_ms": statistics.median(allv),
           "p99_ms": float(np.percentile(allv, 99)),
           "runs": [{"ms_mean": statistics.mean(r), "p50_ms": statistics.median(r),
                     "p99_ms": float(np.percentile(r, 99))} for r in per_run]}
    if deadline_ms is not None:
        out["over_deadline"] = int(sum(1 for t in allv if t > deadline_ms))
        out["deadline_ms"] = deadline_ms
    return out


def roofline_of(bytes_per_launch, ms):
    """The HBM roofline object of a launch moving bytes_per_launch in ms."""
    peak, peak_kind = measured_peaks()
    achieved = bytes_per_launch / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_kind": peak_kind, "frac_of_8000": achieved / 8000.0,
            "algorithmic_bytes_per_launch": bytes_per_launch, "traffic": None}


def cpu_baseline_of(seconds, units, sample):
    """The oracle's rate on one sampled unit of the same workload."""
    return {"value": units / seconds, "unit": METRIC, "cores": os.cpu_count(), "kind": "oracle",
            "sample": sample}


def _oracle_frames_seconds(w, s, pos, frames):
    """Seconds of the oracle for `frames` successive frames of session s of
    the decoder workload w (inputs prepared outside the timing)."""
    import oracle
    W = synth.weights_host(w)
    x = synth.x_bf16(w)[[s]]
    p = np.asarray([pos[s]], dtype=np.int32)
    kv, sc = oracle.prefill_history(w, [s], p, poison=False)
    t0 = time.perf_counter()
    for f in range(frames):
        oracle.step(w, W, kv, sc, p + f, x)
    return time.perf_counter() - t0


def run_sweep(args, w):
    """Session sweep on one GPU: one history of S_max = max(S) sessions, and
    for each S the first S of them (positions are the first S of one draw,
    so the sweeps nest).  One JSON line per S: session-frames/s, p50/p99
    step ms over --runs runs of --steps steps, the HBM roofline fraction of
    the step, clocks, and the oracle on one session as the CPU baseline."""
    import torch
    import frame_step_decode_gb300 as fsd
    device = torch.device("cuda", 0)
    sizes = [int(v) for v in args.sweep.split(",")]
    S_max = max(sizes)
    weights, kv, sc, pos, pos_h, x, y = build_inputs(w, S_max, device)
    wave = fsd.Wave(fsd.WaveConfig.of(w), S_max, w.T_max)
    stream = torch.cuda.current_stream()
    cpu = None
    if not args.no_cpu_baseline:
        sec = _oracle_frames_seconds(w, 0, pos_h, 1)
        cpu = cpu_baseline_of(sec, 1, f"session 0 (pos {int(pos_h[0])}) of {w.name}, one frame; "
                                       "sessions are independent, so the rate holds at any S")
    for S in sizes:
        launch = lambda: wave.step(S, weights, kv, sc, pos, x, y, stream=stream)
        for _ in range(max(3, args.warmup)):
            launch()
        if wave.status() != fsd.WAVE_OK:
            raise RuntimeError(f"warm-up failed at S={S}")
        per_run, clk = timed_runs(launch, args.steps, args.runs, stream, 0)
        if wave.status() != fsd.WAVE_OK:
            raise RuntimeError(f"timed step failed at S={S}")
        st = run_stats(per_run, 80.0)
        b = algorithmic_bytes(w, pos_h[:S])
        print(json.dumps({"mode": "sweep", "metric": METRIC, "value": S / (st["ms_mean"] * 1e-3), "unit": METRIC,
                          "higher_is_better": True, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": st["ms_mean"], "stats": st, "dtype": "bf16",
                          "data": "synthetic (seeded)",
                          "config": {"workload": w.name, "S": S, "T_max": w.T_max,
                                     "positions": f"first {S} of one uniform [{w.pos_lo}, {w.pos_hi}) draw",
                                     "l2": "inputs larger than L2 (no flush needed)"},
                          "roofline": roofline_of(b, st["ms_mean"]), "clocks": clk, "cpu_baseline": cpu}),
              flush=True)
    wave.close()


def run_beat(args, w):
    """Beats of `--beat` frames per launch (the pages' beat is two 80 ms
    frames with a 160 ms deadline): per-beat CUDA-event times over --runs
    runs, p50/p99, beats over the deadline, roofline, clocks and the oracle
    on one session's beat.  Positions are held fixed between beats (advance
    off) so that every timed beat moves the same bytes."""
    import torch
    import frame_step_decode_gb300 as fsd
    device = torch.device("cuda", 0)
    S, F = args.S, args.beat
    weights, kv, sc, pos, pos_h, x, y = build_inputs(w, S, device)
    pos_h = np.minimum(pos_h, w.T_max - F)
    pos = torch.from_numpy(pos_h).to(device)
    xs = x.unsqueeze(0).repeat(F, 1, 1).contiguous()
    ys = torch.empty_like(xs)
    wave = fsd.Wave(fsd.WaveConfig.of(w), S, w.T_max)
    stream = torch.cuda.current_stream()
    launch = lambda: wave.beat(S, F, weights, kv, sc, pos, xs, ys, advance=False, stream=stream)
    for _ in range(max(3, args.warmup)):
        launch()
    if wave.status() != fsd.WAVE_OK:
        raise RuntimeError("warm-up beat failed")
    per_run, clk = timed_runs(launch, args.steps, args.runs, stream, 0)
    if wave.status() != fsd.WAVE_OK:
        raise RuntimeError("timed beat failed")
    st = run_stats(per_run, 80.0 * F)
    b = sum(algorithmic_bytes(w, pos_h + f) for f in range(F))
    line = {"mode": "beat", "metric": METRIC, "value": F * S / (st["ms_mean"] * 1e-3), "unit": METRIC,
            "higher_is_better": True, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "frames_per_launch": F, "ms_per_beat": st["ms_mean"], "stats": st, "dtype": "bf16",
            "data": "synthetic (seeded)",
            "config": {"workload": w.name, "S": S, "T_max": w.T_max, "frames": F,
                       "positions": f"uniform [{w.pos_lo}, {w.pos_hi}), at most T_max - {F}",
                       "l2": "inputs larger than L2 (no flush needed)"},
            "roofline": roofline_of(b, st["ms_mean"]), "clocks": clk, "cpu_baseline": None}
    if not args.no_cpu_baseline:
        sec = _oracle_frames_seconds(w, 0, pos_h, F)
        line["cpu_baseline"] = cpu_baseline_of(sec, F, f"session 0 (pos {int(pos_h[0])}) of {w.name}, "
                                                       f"one beat of {F} frames")
    print(json.dumps(line), flush=True)
    wave.close()


def run_depth(args):
    """The inner depth loop: 8 dependent steps per frame of the 6-layer
    d=1024 model, S = 80, one launch per frame (wave_depth).  Per-frame CUDA
    events over --runs runs; reports session-frames/s (a session's frame is
    its 8 dependent steps), session-steps/s, p50/p99 frame ms, the
    algorithmic bytes per frame (weights once per step + W_p once per chained
    step + the depth cache read and written) against the HBM peak, clocks,
    and the oracle's depth loop for one session."""
    import torch
    import frame_step_decode_gb300 as fsd
    w = synth.DEPTH
    steps = w.extra["depth_steps"]
    S, d = args.S if args.S != 80 else w.S, w.d_model
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    rm = torch.empty(synth.weight_elems(w), dtype=torch.bfloat16, device=device)
    synth.weights_device(w, rm, stream.cuda_stream)
    weights = fsd.pack_weights(fsd.WaveConfig.of(w), rm)
    del rm
    wp = torch.empty((d, d), dtype=torch.bfloat16, device=device)
    synth.proj_device(w, wp.data_ptr(), stream.cuda_stream)
    x0 = torch.empty((S, d), dtype=torch.bfloat16, device=device)
    synth.x_device(w, S, x0.data_ptr(), stream.cuda_stream)
    kv = torch.zeros((L, 2, S, H, T, D), dtype=torch.uint8, device=device)
    sc = torch.zeros((L, 2, S, H, T), dtype=torch.float32, device=device)
    xs = torch.empty((steps, S, d), dtype=torch.bfloat16, device=device)
    y = torch.empty((steps, S, d), dtype=torch.bfloat16, device=device)
    wave = fsd.Wave(fsd.WaveConfig.of(w), S, T)
    launch = lambda: wave.depth(S, steps, weights, wp, kv, sc, x0, xs, y, stream=stream)
    for _ in range(max(3, args.warmup)):
        launch()
    if wave.status() != fsd.WAVE_OK:
        raise RuntimeError("warm-up depth loop failed")
    per_run, clk = timed_runs(launch, args.steps, args.runs, stream, 0)
    if wave.status() != fsd.WAVE_OK:
        raise RuntimeError("timed depth loop failed")
    st = run_stats(per_run, 80.0)
    ms = st["ms_mean"]
    b = sum(algorithmic_bytes(w, np.full(S, k)) for k in range(steps)) + (steps - 1) * 2 * d * d
    line = {"mode": "depth", "metric": METRIC, "value": S / (ms * 1e-3), "unit": METRIC,
            "higher_is_better": True, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "session_steps_per_s": S * steps / (ms * 1e-3), "ms_per_frame": ms, "us_per_step": 1000.0 * ms / steps,
            "stats": st, "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "S": S, "steps_per_frame": steps, "T_max": T,
                       "l2": "weights re-read every dependent step (154 MB, larger than L2)"},
            "roofline": roofline_of(b, ms), "clocks": clk, "cpu_baseline": None,
            "grid_barriers_per_frame": steps * wave.barriers_per_step + 2 * (steps - 1)}
    if not args.no_cpu_baseline:
        import oracle
        Wh, wp_h, x_h = synth.weights_host(w), synth.proj_host(w), synth.x_bf16(w, 1)
        t0 = time.perf_counter()
        oracle.depth_loop(w, Wh, wp_h, x_h, steps)
        line["cpu_baseline"] = cpu_baseline_of(time.perf_counter() - t0, 1,
                                               f"session 0 of {w.name}: one frame of {steps} dependent steps")
    print(json.dumps(line), flush=True)
    wave.close()


def hybrid_bytes(w, pos) -> int:
    """Algorithmic bytes of one hybrid step: the weights once, the attention
    blocks' history read and the appended slot written, and every selective-
    state block's fp32 state read and written."""
    La, H, D = w.n_attn, w.n_heads, w.head_dim
    weights = 2 * synth.hybrid_weight_elems(w)
    live = [int(p) for p in pos if p >= 0]
    kv = sum(La * 2 * H * (p + 1) * (D + 4) for p in live) + La * 2 * len(live) * H * (D + 4)
    state = 2 * w.n_mamba * len(live) * w.ssm_heads * w.ssm_head_dim * w.ssm_state * 4
    return weights + kv + state


def run_hybrid(args):
    """The hybrid recurrent step (48 layers: selective-state blocks with an
    attention block every sixth layer), S = 56: per-step CUDA events over
    --runs runs, p50/p99, session-frames/s, the HBM fraction of its
    algorithmic bytes, clocks, and the oracle on one session."""
    import torch
    import frame_step_decode_gb300 as fsd
    w = synth.HYBRID
    if args.layers:  # a shorter copy (whole groups of attn_every layers) for profiling a small case
        if args.layers % w.attn_every:
            raise SystemExit(f"--layers with --hybrid must be a multiple of {w.attn_every}")
        from dataclasses import replace
        w = replace(w, n_layers=args.layers, name=f"{w.name}-L{args.layers}")
    S = w.S
    aw = w.attention_view()
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    La, H, T, D = w.n_attn, w.n_heads, w.T_max, w.head_dim
    rm = torch.empty(synth.hybrid_weight_elems(w), dtype=torch.bfloat16, device=device)
    synth.hybrid_weights_device(w, rm, stream.cuda_stream)
    weights = fsd.hybrid_pack_weights(fsd.WaveHybridConfig.of(w), rm)
    del rm
    kv = torch.empty((La, 2, S, H, T, D), dtype=torch.uint8, device=device)
    sc = torch.empty((La, 2, S, H, T), dtype=torch.float32, device=device)
    raw = torch.empty((S, H, T, D), dtype=torch.float32, device=device)
    for l in range(La):
        for which in range(2):
            synth.kv_raw_device(aw, l, which, 0, S, T, raw.data_ptr(), T, stream.cuda_stream)
            fsd.kv_quantize(raw, kv[l, which], sc[l, which])
    del raw
    state = torch.empty((w.n_mamba, S, w.ssm_heads, w.ssm_head_dim, w.ssm_state), dtype=torch.float32,
                        device=device)
    for lm in range(w.n_mamba):
        synth.hybrid_state_device(w, lm, 0, S, state[lm].data_ptr(), stream.cuda_stream)
    pos_h = synth.positions(aw, S)
    pos = torch.from_numpy(pos_h).to(device)
    x = torch.empty((S, w.d_model), dtype=torch.bfloat16, device=device)
    synth.x_device(aw, S, x.data_ptr(), stream.cuda_stream)
    y = torch.empty_like(x)
    wave = fsd.HybridWave(fsd.WaveHybridConfig.of(w), S, T)
    for _ in range(max(3, args.warmup)):
        wave.hybrid_step(S, weights, kv, sc, state, pos, x, y, stream=stream)
    if wave.status() != fsd.WAVE_OK:
        raise RuntimeError("warm-up hybrid step failed")
    if args.phases:
        # phase-end marks: each phase's time is the last CTA's finish minus
        # the last CTA's finish of the phase before (the hand-overs overlap)
        n, grid = wave.phases_per_step, wave.grid
        ts = torch.zeros((n, grid), dtype=torch.int64, device=device)
        wave.debug_arrival_times(ts)
        ends = []
        for _ in range(3):
            wave.hybrid_step(S, weights, kv, sc, state, pos, x, y, stream=stream)
            if wave.status() != fsd.WAVE_OK:
                raise RuntimeError("step failed")
            tm = ts.cpu().numpy().astype(np.float64) / 1000.0
            ends.append(np.diff(np.concatenate([[tm.min()], tm.max(axis=1)])))
        wave.debug_arrival_times(None)
        t = np.mean(ends, axis=0)
        names = ["prologue"]
        for l in range(w.n_layers):
            if l > 0:
                names.append("norm")
            names += ["qkv", "attn", "o"] if w.is_attn(l) else ["in", "ssm", "out"]
        print(f"{w.name} S={S}: {t.sum():.1f} us from the first mark (phase = the last CTA's finish minus "
              "the last CTA's finish of the phase before)")
        agg = {}
        for n_, v in zip(names, t):
            agg.setdefault(n_, []).append(v)
        blk = w.ssm_heads * w.ssm_head_dim * w.ssm_state * 4 * 2 * S
        for n_, v in agg.items():
            m = float(np.mean(v))
            extra = f"  {blk / m / 1e3:6.0f} GB/s of state" if n_ == "ssm" else ""
            print(f"  {n_:8s} x{len(v):3d}  mean {m:8.1f} us  total {np.sum(v):9.1f} us "
                  f"({100 * np.sum(v) / t.sum():5.1f}%){extra}")
        wave.close()
        return
    launch = lambda: wave.hybrid_step(S, weights, kv, sc, state, pos, x, y, stream=stream)
    per_run, clk = timed_runs(launch, args.steps, args.runs, stream, 0)
    if wave.status() != fsd.WAVE_OK:
        raise RuntimeError("timed hybrid step failed")
    st = run_stats(per_run, 80.0)
    b = hybrid_bytes(w, pos_h)
    line = {"mode": "hybrid", "metric": METRIC, "value": S / (st["ms_mean"] * 1e-3), "unit": METRIC,
            "higher_is_better": True, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": st["ms_mean"], "stats": st, "dtype": "bf16 (fp32 state)", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "S": S, "T_max": T,
                       "positions": f"uniform [{aw.pos_lo}, {aw.pos_hi})",
                       "l2": "inputs larger than L2 (no flush needed)"},
            "roofline": roofline_of(b, st["ms_mean"]), "clocks": clk, "cpu_baseline": None}
    wave.close()
    if not args.no_cpu_baseline:
        import oracle
        W = synth.hybrid_weights_host(w)
        p1 = pos_h[:1]
        kv1, sc1, st1 = oracle.hybrid_prefill(w, [0], p1, poison=False)
        x1 = synth.x_bf16(aw, 1)
        t0 = time.perf_counter()
        oracle.hybrid_step(w, W, kv1, sc1, st1, p1, x1)
        line["cpu_baseline"] = cpu_baseline_of(time.perf_counter() - t0, 1,
                                               f"session 0 (pos {int(p1[0])}) of {w.name}, one frame")
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--S", type=int, default=80)
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (profiling a small case)")
    ap.add_argument("--tmax", type=int, default=None, help="shorter history (profiling a small case)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--hybrid", action="store_true",
                    help="time the hybrid recurrent step (48 layers, S = 56)")
    ap.add_argument("--depth", action="store_true",
                    help="time the inner depth loop (8 chained steps of the 6-layer d=1024 model)")
    ap.add_argument("--beat", type=int, default=0,
                    help="time beats of this many frames per launch (one JSON line, one GPU)")
    ap.add_argument("--sweep", default=None,
                    help="comma-separated session counts: one JSON line per S (one GPU)")
    ap.add_argument("--phases", action="store_true",
                    help="print the per-phase time table of one step instead of the JSON line")
    ap.add_argument("--runs", type=int, default=3,
                    help="runs of --steps launches per point in the --sweep/--beat/--depth/--hybrid modes")
    args = ap.parse_args()
    # --gpus N: one process per GPU.  Launched by torchrun, WORLD_SIZE must
    # say the same; launched plainly with N > 1, start the N ranks here.
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        import socket
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
        sys.exit(subprocess.call(cmd))
    if world is not None and int(world) != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU")
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    w = synth.SEVEN_B
    if args.layers or args.tmax:
        from dataclasses import replace
        T = args.tmax or w.T_max
        w = replace(w, n_layers=args.layers or w.n_layers, T_max=T, pos_hi=min(w.pos_hi, T),
                    name=f"{w.name}-L{args.layers or w.n_layers}-T{T}")
    if args.hybrid:
        run_hybrid(args)
    elif args.depth:
        if args.phases:  # one dependent step of the loop's model, phase by phase
            run_phases(args, synth.DEPTH)
        else:
            run_depth(args)
    elif args.beat:
        run_beat(args, w)
    elif args.sweep:
        run_sweep(args, w)
    elif args.phases:
        run_phases(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
