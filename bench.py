#!/usr/bin/env python3
"""Benchmark: fused exact attention, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole path over one batch of synthetic input:
attn_fwd (fused forward), then the two backward kernels as attn_bwd runs
them (dQ, which also forms the row terms D_i = dO_i . O_i, then dK/dV).  The default workload is B=1, H=16, N=8192, d=128, causal, bf16
(the N=8192 causal forward is the case the forward target is stated on).
Prints ONE JSON line (rank 0).

Timing: inputs resident in HBM; L2 is flushed (a 256 MiB write) before every
step, outside the timed events; each kernel is bracketed by CUDA events on
the launching stream; the step time is the sum of its kernels' event times.
After the K timed steps a repeat phase of at least 200 ms of device time
gives per-kernel and per-step medians (the "median" object); nvidia-smi
clocks are sampled across both.
TFLOPS use the algorithmic FLOP model 4*B*H*N^2*d (halved when causal) for
the forward and 2.5x that for the backward.

Under torchrun (N > 1) every rank runs its own copy of the workload (heads
are independent: weak scaling, no data-path collective); the reported value
is the FLOPs of all ranks over the slowest rank's time.  --gpus N > 1 outside
torchrun relaunches this script under torchrun with N ranks; a --gpus that
differs from WORLD_SIZE is refused.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOPS (fwd, fwd+bwd) on 1 GB300 and % of dense BF16 tensor peak"
UNIT = "TFLOPS"
FALLBACK_PEAK_TFLOPS = 1900.0   # profiling recipe fallback (bf16 burst) if no measured file
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, help="workload number 1-5 (default 4)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks of the default
    process group (the slowest rank's times); the identity without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return flops_per_rank * world / ms / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p.get("hbm_gbs", 0.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": FALLBACK_PEAK_TFLOPS, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def code_tokens(text: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of white
    space made one blank: what the compiler sees, so that editing a comment
    does not mark a profiled kernel as changed.  String and character
    literals are kept as written."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif c == "/" and text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_sha(name: str) -> str:
    src = {"attn_fwd_kernel": "fwd.cu", "bwd_dkdv_kernel": "bwd.cu", "bwd_dq_kernel": "dq.cu"}[name]
    h = hashlib.sha256()
    for f in (src, "ptx.cuh", "kernels.cuh"):
        with open(os.path.join(ROOT, "exact_attention_67_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def dram_traffic(name: str, workload: str):
    """Per-launch DRAM bytes of `name` from the committed ncu summary, if it was
    taken on the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[workload][name]
        if e.get("source_sha") != kernel_source_sha(name):
            return None
        return float(e["bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples with host timestamps."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.proc = None
        self.path = None
        self.idx = device_index
        if not enabled:
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float, label: str = "timed region"):
        if self.proc is None or not self.path:
            return None
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                        ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                        rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
                    except (ValueError, IndexError):
                        continue
        finally:
            os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = label
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:3]
            window = "nearest samples to a short timed region"
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


# ------------------------------------------------------------ CPU oracle legs
def oracle_head_flops(w, n_rows: int) -> float:
    """Algorithmic fwd+bwd FLOPs of an n_rows x n_rows leading block of one head."""
    f = 4.0 * n_rows * n_rows * w.d
    if w.causal:
        f /= 2
    return 3.5 * f


def run_oracle_sample(w, q, k, v, do, head: int, n_rows: int):
    """The oracle's full fwd + bwd on the leading n_rows x n_rows block of one
    head (under the causal mask these rows see only these keys).  Returns
    (seconds, threads)."""
    import oracle
    orc = oracle._load()
    b, h = divmod(head, w.H)

    def f64(t):
        return t[b, h, :n_rows].float().double().numpy()

    qf, kf, vf, dof = f64(q), f64(k), f64(v), f64(do)
    nt = orc.default_threads()
    t0 = time.perf_counter()
    orc.head_fwd(qf, kf, vf, w.causal, w.scale, nthreads=nt)
    orc.head_bwd(qf, kf, vf, dof, w.causal, w.scale, nthreads=nt)
    return time.perf_counter() - t0, nt


def cpu_baseline(w, q, k, v, do):
    """The oracle timed on this host's cores: full fwd + bwd of whole heads
    (exact outputs for those heads), ~10-30 s of CPU work."""
    secs, flops, heads, nt = 0.0, 0.0, 0, 1
    for head in range(w.B * w.H):
        s, nt = run_oracle_sample(w, q, k, v, do, head, w.N)
        secs += s
        flops += oracle_head_flops(w, w.N)
        heads += 1
        if secs > 10.0:
            break
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": nt, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of {heads} whole head(s) (N={w.N}, d={w.d}) of {w.name}, "
                      f"{secs:.1f} s on {nt} threads ({cpu_model()})",
            "seconds": secs}


def reference_arm(args, w, rank: int, world: int):
    """--impl reference: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return 0
    from exact_attention_67_gb300.synth import make_inputs
    q, k, v, do = make_inputs(w, with_grad=True)
    # size each step's sample so that warmup + steps end within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_rows = min(512, w.N)
    s, _ = run_oracle_sample(w, q, k, v, do, 0, n_rows)
    while n_rows * 2 <= w.N and s * 4.2 < budget:
        n_rows *= 2
        s, _ = run_oracle_sample(w, q, k, v, do, 0, n_rows)
    for i in range(max(0, args.warmup - 1)):
        run_oracle_sample(w, q, k, v, do, i % (w.B * w.H), n_rows)
    total, nt = 0.0, 1
    for i in range(args.steps):
        s, nt = run_oracle_sample(w, q, k, v, do, i % (w.B * w.H), n_rows)
        total += s
    flops = oracle_head_flops(w, n_rows) * args.steps
    value = flops / total / 1e12
    sample = (f"per step: fp64 oracle fwd+bwd of the leading {n_rows}x{n_rows} block of one head of "
              f"{w.name} (heads in turn); {nt} threads ({cpu_model()})")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, world: int):
    # Every step times the forward and the backward, also for a workload whose
    # published figure is forward-only (its fwd_tflops is that figure).
    return {"workload": f"{w.name} fwd+bwd",
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "scale": "1/sqrt(d)", "inputs": "bf16 N(0,1) (Q,K sigma %g), seeded" % w.sigma_qk,
            "l2": "flushed before every step (256 MiB write, outside the timed events)",
            "parallelism": "replicas" if world == 1 else f"replicas x{world} (independent heads per rank)"}


# ------------------------------------------------------------------ launch
def relaunch_under_torchrun(args) -> int:
    """--gpus N > 1 outside torchrun: run this script as N ranks on this node
    (one per GPU) and return their exit status.  Every rank must come up: a
    replicas run never quietly measures fewer GPUs than asked."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def check_world(args):
    """Exit status for a --gpus / WORLD_SIZE mismatch (None when consistent)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if "WORLD_SIZE" in os.environ and world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU "
              f"(torchrun --nproc-per-node {args.gpus}) or pass --gpus {world}", file=sys.stderr)
        return 2
    return None


def kernel_stats(ms_lists):
    """Per kernel: mean and median of its per-step event times (ms)."""
    return [(statistics.fmean(v), statistics.median(v)) for v in ms_lists]


# ------------------------------------------------------------------ our arm
def main():
    args = parse_args()
    if args.gpus < 1:
        print("bench.py: --gpus must be >= 1", file=sys.stderr)
        return 2
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return relaunch_under_torchrun(args)
    bad = check_world(args)
    if bad is not None:
        return bad
    from exact_attention_67_gb300.synth import WORKLOADS
    w = WORKLOADS[args.config]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, w, rank, world)

    import torch
    import torch.distributed as dist

    import exact_attention_67_gb300 as ex
    from exact_attention_67_gb300 import build as exbuild
    from exact_attention_67_gb300.synth import make_inputs

    if not torch.cuda.is_available() or torch.cuda.device_count() <= local:
        print(f"bench.py: rank {rank} needs CUDA device {local}; {torch.cuda.device_count()} visible",
              file=sys.stderr)
        return 1
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        exbuild.build()
    if world > 1:
        dist.barrier()
    ex.load()
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    q_h, k_h, v_h, do_h = make_inputs(w, seed_base=1000 * w.cfg + 100 * rank, with_grad=True)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    Dws = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    causal, scale = w.causal, w.scale
    stream = torch.cuda.current_stream()
    F = w.flops_fwd()
    # The backward as attn_bwd runs it: the dQ kernel also forms the row terms
    # D_i = dO_i . O_i (stored for dK/dV), then dK/dV.
    kernels = ["attn_fwd_kernel", "bwd_dq_kernel", "bwd_dkdv_kernel"]
    nk = len(kernels)
    # algorithmic FLOPs per launch: fwd = 2 GEMMs (QK^T, PV); dK/dV = 4 (S, dP, dV, dK);
    # dQ = 1 (dQ; its S/dP recomputation and the row dots are not counted).
    alg = {"attn_fwd_kernel": F, "bwd_dkdv_kernel": 2.0 * F, "bwd_dq_kernel": 0.5 * F}

    def step(evs):
        evs[0].record(stream)
        ex.attn_fwd(q, k, v, o, lse, causal, scale)
        evs[1].record(stream)
        ex.attn_bwd_d_and_dq(q, k, v, o, do, lse, Dws, dq, causal, scale)
        evs[2].record(stream)
        ex.attn_bwd_dkdv(q, k, v, do, lse, Dws, dk, dv, causal, scale)
        evs[3].record(stream)

    def new_events(n):
        return [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(n)]

    def run_steps(n):
        """n steps, L2 flushed before each (outside its events); per-kernel ms lists."""
        evs = new_events(n)
        for i in range(n):
            flush.zero_()
            step(evs[i])
        return evs

    def per_kernel_ms(evs):
        return [[e[j].elapsed_time(e[j + 1]) for e in evs] for j in range(nk)]

    evw = run_steps(max(3, args.warmup))
    torch.cuda.synchronize()
    if ex.device_error() != 0:
        raise RuntimeError("kernel watchdog fired during warm-up")
    step_est = sum(statistics.median(x) for x in per_kernel_ms(evw))

    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.3 if not args.no_clocks else 0.0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev = run_steps(args.steps)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    # Repeat phase for order statistics and a clock record over >= 200 ms of
    # device time, whatever --steps is: the per-kernel medians reported
    # beside the K-step means.
    n_rep = max(50, int(math.ceil(200.0 / max(step_est, 1e-3))))
    ev_rep = run_steps(n_rep)
    torch.cuda.synchronize()
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall2, "timed steps and the repeat phase after them")
    if ex.device_error() != 0:
        raise RuntimeError("kernel watchdog fired during the timed region")

    timed = per_kernel_ms(ev)
    per_kernel = [sum(x) for x in timed]
    reduced = max_over_ranks([sum(per_kernel)] + per_kernel, dev)
    total_ms, per_kernel = reduced[0], reduced[1:]
    rep = per_kernel_ms(ev_rep)
    rep_steps = [sum(rep[j][i] for j in range(nk)) for i in range(n_rep)]
    med = max_over_ranks([statistics.median(rep_steps)] + [statistics.median(x) for x in rep], dev)
    med_step, med_kernel = med[0], med[1:]

    steps = args.steps
    t_fwd = per_kernel[0] / steps
    t_bwd = sum(per_kernel[1:]) / steps
    value = job_tflops(3.5 * F, world, total_ms / steps)   # TFLOPS over all ranks
    fwd_tflops = F / t_fwd / 1e9
    bwd_tflops = 2.5 * F / t_bwd / 1e9
    peak = peaks["bf16_tflops"]
    rows = []
    for j, (name, ms) in enumerate(zip(kernels, per_kernel)):
        per = ms / steps
        r = {"kernel": name, "ms": per, "median_ms": med_kernel[j], "share": ms / total_ms}
        r["tflops"] = alg[name] / per / 1e9
        r["frac_of_peak"] = r["tflops"] / peak
        rows.append(r)
    dom = max(range(nk), key=lambda j: per_kernel[j])
    dname = kernels[dom]
    traffic = dram_traffic(dname, w.name)
    roofline = {"bound": "tensor", "kernel": dname, "achieved": rows[dom].get("tflops"), "peak": peak,
                "unit": "TFLOP/s", "frac": rows[dom].get("frac_of_peak"), "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                "algorithmic_flops_per_launch": alg.get(dname)}
    median = {"ms_per_step": med_step, "value": job_tflops(3.5 * F, world, med_step),
              "fwd_tflops": F / med_kernel[0] / 1e9, "bwd_tflops": 2.5 * F / sum(med_kernel[1:]) / 1e9,
              "steps": n_rep, "device_ms": sum(rep_steps),
              "note": "medians over a repeat phase run right after the timed steps (same L2 flush per step)"}

    # ---------------------------------------------------------------- e2e
    e2e = None
    if not args.no_e2e:
        pin = [t.pin_memory() for t in (q_h, k_h, v_h, do_h)]
        outs_h = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (o, lse, dq, dk, dv))
        n_e2e = max(3, min(steps, 20))
        e2e_groups = min(4, w.B * w.H)
        ws_host = torch.empty(ex.attn_fwd_bwd_host_workspace_size(w.B, w.H, w.N, w.d, causal), dtype=torch.uint8,
                              device=dev)
        s_in, s_out, s_two = (torch.cuda.Stream(device=dev) for _ in range(3))

        def e2e_step():
            # Host in, host out through the C ABI: attn_fwd_bwd_host copies each
            # group's inputs in on s_in and its results out on s_out while the
            # kernels of other groups (on `stream` and s_two) or later stages run.
            ex.attn_fwd_bwd_host(*pin, *outs_h, causal, scale, ws_host, groups=e2e_groups, stream=stream,
                                 copy_in_stream=s_in, copy_out_stream=s_out, stream2=s_two)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks([e0.elapsed_time(e1) / n_e2e], dev)[0]
        h2d = sum(t.numel() * t.element_size() for t in pin)
        d2h = sum(t.numel() * t.element_size() for t in outs_h)
        e2e = {"value": job_tflops(3.5 * F, world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n_e2e,
               "path": "C ABI attn_fwd_bwd_host with host buffers, called every step: pinned host inputs -> "
                       "device, forward and backward kernels, device -> pinned host outputs, copies overlapped "
                       f"with the kernels ({e2e_groups} groups of heads on 2 compute streams)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q_h, k_h, v_h, do_h)

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, world),
            "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
            "fwd_pct_peak": 100.0 * fwd_tflops / peak, "fwd_bwd_pct_peak": 100.0 * value / world / peak,
            "median": median, "kernels": rows, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": nk * steps, "clocks": clocks,
            "gpu": torch.cuda.get_device_name(dev)}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
