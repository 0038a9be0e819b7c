"""Benchmark of the fused SwiGLU projection Y = SiLU(A W1) * (A W2) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--secondary NAMES] [--impl ours|reference] [--no-cpu-baseline]

One step = one swiglu_forward call over one batch of synthetic input (the
packed weight is prepared once, before timing, as at model load). Prints one
JSON line (rank 0). Metric: TFLOP/s counted as 4*M*K*N per step, and its
fraction of the dense BF16 tensor peak. Default workload: the Qwen-2.5-72B
MLP gate/up projection on 8192 tokens (M=8192, K=8192, N=29568), the largest
prefill shape; the 7B decode batch (M=16) follows as a secondary record.

* value: whole-job TFLOP/s with inputs resident in HBM; K steps timed with
  CUDA events between barriers + synchronisations, max over ranks. The K steps
  replay from one CUDA graph of exactly K kernel nodes captured from
  swiglu_forward calls (longer runs: whole-rotation graphs plus a remainder
  graph; --eager: one host call per step).
* roofline: the fused kernel's achieved bytes/s (HBM-bound workloads) or
  FLOP/s (tensor-bound workloads) per launch (timed region over launches: one
  launch per step), against the measured peaks in MEASURED_PEAKS.json.
* e2e: the same metric through swiglu_forward_from_host, with each step's
  activations copied from pinned host memory and its output copied back;
  alternate steps go to two streams with their own staging buffers.
* secondary: other workloads through the same device-timed path (value,
  roofline, clocks), one record each.
* cpu_baseline: the CPU oracle (float64) on a bounded sample of the workload.
* --impl reference: the CPU oracle timed as the reference arm (the method has
  no runnable reference implementation).
N > 1 runs independent replicas (the op has no exchange step), one per rank.
"""
from __future__ import annotations

import os
import re

# BLAS threads of the CPU oracle: the cores this process may run on.
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

import argparse  # noqa: E402
import dataclasses  # noqa: E402
import glob  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from swiglu_gated_mlp_gb300.workloads import (WORKLOADS, Workload, bf16_bits,  # noqa: E402
                                              make_inputs, make_inputs_fp8, make_inputs_mxfp8,
                                              make_workload_inputs, sample_rows, sweep_32b)

METRIC = "fused SwiGLU-GEMM TFLOP/s (4·M·K·N) and % of GB300 dense BF16 peak"
METRIC_DOWN = "MLP down-projection TFLOP/s (2·M·N·H), Out = Y·W3 + R"
# the metric is a fraction of the dense BF16 tensor peak: its headline is the
# largest prefill shape (Qwen-2.5-72B, 8192 tokens); the 7B decode batch, the
# HBM-bound case, is reported beside it as a secondary record
DEFAULT_WORKLOAD = "qwen2.5-72b-prefill-m8192"
DEFAULT_SECONDARY = "qwen2.5-7b-decode-m16"
# swiglu_forward_variant's kernel choice (auto = what swiglu_forward does)
VARIANTS = {"auto": 0, "large": 1, "small": 2, "pair": 3, "sequential": 4, "split": 5,
            "resident": 6}
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["swiglu_gated_mlp_gb300/csrc/" + f for f in
                  ("fused_small_m.cu", "fused_large_m.cu", "fused_large_m_pair.cu", "fused_sequential.cu",
                   "fused_split_k.cu", "fused_resident_pair.cu", "ptx.cuh", "kernels.h",
                   "swiglu_api.cu")]


def workload_by_name(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("qwen2.5-32b-m"):
        return sweep_32b(int(name.rsplit("m", 1)[1]))
    raise SystemExit(f"unknown workload {name}; known: {sorted(WORKLOADS)}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured (MEASURED_PEAKS.json)"
    return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


def _code_only(text: str) -> str:
    """C++/CUDA source without comments and blank lines (comment edits keep the stamp)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def host_copy_rates(a_host, a_dev, y_dev, y_host, stream, reps: int = 3) -> dict:
    """This box's pinned host <-> device copy rates at the step's own sizes
    (best of `reps` single copies, CUDA events on `stream`): the end-to-end
    figure is bound by them when a step's copies outlast its kernel."""
    def best(dst, src):
        t = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                dst.copy_(src, non_blocking=True)
                e1.record(stream)
            e1.synchronize()
            t.append(e0.elapsed_time(e1) * 1e-3)
        return round(src.numel() * src.element_size() / min(t) / 1e9, 1)
    return {"h2d_gbs": best(a_dev, a_host), "d2h_gbs": best(y_host, y_dev),
            "how": "pinned host memory, one copy at a time, best of %d" % reps}


def source_stamp() -> str:
    """Hash of the kernel sources' code (comments and blank lines left out)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary of this kernel source."""
    stamp = source_stamp()
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        # "bench-key k=v" lines: one key per line (one record per file), or a
        # whole record of space-separated k=v pairs on one line
        records, single = [], {}
        with open(path) as f:
            for line in f:
                if not line.startswith("bench-key "):
                    continue
                pairs = [kv.partition("=") for kv in line[len("bench-key "):].split()]
                rec = {k.strip(): v.strip() for k, _, v in pairs if k}
                (records.append(rec) if len(rec) > 1 else single.update(rec))
        for fields in records + [single]:
            if (fields.get("kernel") == kernel and fields.get("workload") == workload
                    and fields.get("source_stamp") == stamp and "dram_bytes_per_launch" in fields):
                return float(fields["dram_bytes_per_launch"]), os.path.relpath(path, ROOT)
    return None, None


# ------------------------------------------------------------ distributed ----

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world: int):
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


def aggregate(flops_per_step: int, steps: int, seconds_max: float, world: int) -> float:
    """Whole-job TFLOP/s: all ranks' work over the slowest rank's time."""
    return world * flops_per_step * steps / seconds_max / 1e12


# ---------------------------------------------------------------- clocks ----

CLOCK_FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
                "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing runs."""

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        ident = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.cmd = ["nvidia-smi", "-i", ident, "--query-gpu=" + ",".join(CLOCK_FIELDS),
                    "--format=csv,noheader,nounits", "-lms", "100"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi gave no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- our arm ----

@dataclasses.dataclass
class Prepared:
    """One workload on the device: rotating operand copies and the forward call."""
    w: Workload
    fp8: bool
    down: bool
    flops: int
    alg_bytes: int
    copies: int
    plan: str
    kernel: str
    fwd: object            # fwd(j, stream=None): one forward on rotation slot j
    out_cols: int
    w_bytes: int
    a_cpu: object          # the step's activations (CPU), for the e2e leg
    host: dict             # CPU inputs kept for the oracle legs
    dev_state: dict        # device tensors (dropped by release())

    def release(self):
        self.dev_state.clear()
        self.fwd = None


def prepare(args, sg, w: Workload, dev) -> Prepared:
    """Inputs, packed weights and rotating copies for workload `w` on `dev`."""
    M, K, N = w.M, w.K, w.N
    mx = args.dtype == "mxfp8"
    fp8 = args.dtype == "fp8" or mx
    down = args.op == "down"
    if down and fp8:
        raise SystemExit("--op down runs in bf16 only")
    elem = 1 if fp8 else 2
    flops = w.flops
    alg_bytes = elem * M * K + 2 * elem * K * N + 2 * M * N  # A, W1 and W2 once, Y (bf16)
    if mx:  # one scale byte per 32 values of A, W1 and W2
        alg_bytes += (M * K + 2 * K * N) // 32
    host = {}
    SAs = None
    if down:
        # Out [M, H] = Y [M, N] x W3 [N, H] + R at this workload's MLP shape (H = K)
        H = K
        flops = 2 * M * N * H
        alg_bytes = 2 * M * N + 2 * N * H + 2 * 2 * M * H  # Y, W3 once, R read, Out written
        y_cpu, w3_cpu, _ = make_inputs(M, N, H, w.seed)
        r_cpu = make_inputs(M, H, 8, w.seed + 1)[0]
        wp0 = sg.swiglu_pack_down_weights(w3_cpu.to(dev))
        a_cpu = y_cpu
    elif mx:
        a_cpu, sa_cpu, w1_cpu, s1_cpu, w2_cpu, s2_cpu = make_inputs_mxfp8(M, K, N, w.seed)
        wp0 = sg.swiglu_pack_weights_mxfp8(w1_cpu.to(dev), s1_cpu.to(dev), w2_cpu.to(dev),
                                           s2_cpu.to(dev))
        sat0 = sg.swiglu_pack_act_scales_mxfp8(sa_cpu.to(dev))
        host["sat"] = sat0.cpu()
    elif fp8:
        a_cpu, w1_cpu, w2_cpu, scales = make_inputs_fp8(M, K, N, w.seed)
        wp0 = sg.swiglu_pack_weights_fp8(w1_cpu.to(dev), w2_cpu.to(dev))
    else:
        a_cpu, w1_cpu, w2_cpu = make_workload_inputs(w)
        wp0 = sg.swiglu_pack_weights(w1_cpu.to(dev), w2_cpu.to(dev))
        host.update(a=a_cpu, w1=w1_cpu, w2=w2_cpu)
    torch.cuda.synchronize()
    w_bytes = wp0.numel() * wp0.element_size()
    # Inputs larger than L2 between consecutive steps: rotate copies of the
    # packed weight (and of A and Y) so no step finds its operands in L2.
    # Between two uses of one copy the other copies stream at least 32 x L2
    # bytes: the decode kernel stages weight tiles in L2 ahead of its pipeline,
    # and those lines were measured to outlive several x L2 of evict-first
    # streaming, so a shallow rotation would let a step find some of its
    # weights still cached from the previous use of the same copy.
    copies = 1 + max(1, math.ceil(32 * L2_BYTES / max(alg_bytes, 1)))
    if args.rotate:
        copies = max(2, args.rotate)
    copies = min(copies, 64)
    wps = [wp0] + [wp0.clone() for _ in range(copies - 1)]
    a0 = a_cpu.to(dev)
    As = [a0] + [a0.clone() for _ in range(copies - 1)]
    out_cols = K if down else N
    Ys = [torch.empty(M, out_cols, dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    Rs = None
    if mx:
        SAs = [sat0] + [sat0.clone() for _ in range(copies - 1)]
    if down:
        r0 = r_cpu.to(dev)
        Rs = [r0] + [r0.clone() for _ in range(copies - 1)]
    variant = VARIANTS[args.variant]
    # down-projection: a workspace lets the decode kernel split K across
    # clusters; one per stream of calls (the timed graph is one stream)
    down_ws = down and args.down_workspace == "on"
    ws = sg.swiglu_down_workspace(M, N, K, dev) if down_ws else None
    plan = ((sg.swiglu_down_plan_string_ws if down_ws else sg.swiglu_down_plan_string)(M, N, K)
            if down else
            sg.swiglu_plan_string_mxfp8(M, K, N) if mx else
            sg.swiglu_plan_string_fp8(M, K, N) if fp8 else
            sg.swiglu_plan_string(M, K, N, variant))
    base = plan.split(" ", 1)[1] if plan.startswith(("down ", "fp8 ", "mxfp8 ")) else plan
    kernel = ("fused_small_m_kernel" if base.startswith("small_m") else
              "fused_large_m_pair_kernel" if base.startswith("large_m_pair") else
              "fused_sequential_kernel" if base.startswith("sequential") else
              "fused_split_k_kernel" if base.startswith("split_k") else
              "fused_resident_pair_kernel" if base.startswith("resident_pair") else
              "fused_large_m_kernel")
    if down or fp8:  # the template instance: <fp8> E4M3, <mxfp8> block-scaled, <down>
        kernel += "<down>" if down else "<mxfp8>" if mx else "<fp8>"

    def fwd(j, s=None):
        """One forward on rotation slot j (on stream s, default the current stream)."""
        if down:
            sg.swiglu_down_forward(As[j], wps[j], K, R=Rs[j], Out=Ys[j], stream=s, workspace=ws)
        elif mx:
            sg.swiglu_forward_mxfp8(As[j], SAs[j], wps[j], N, Y=Ys[j], stream=s)
        elif fp8:
            sg.swiglu_forward_fp8(As[j], wps[j], N, *scales, Y=Ys[j], stream=s)
        else:
            sg.swiglu_forward_variant(As[j], wps[j], N, variant, Y=Ys[j], stream=s)

    if fp8 and not mx:
        host["scales"] = scales
    return Prepared(w=w, fp8=fp8, down=down, flops=flops, alg_bytes=alg_bytes, copies=copies,
                    plan=plan, kernel=kernel, fwd=fwd, out_cols=out_cols, w_bytes=w_bytes,
                    a_cpu=a_cpu, host=host,
                    dev_state={"wps": wps, "As": As, "Ys": Ys, "Rs": Rs, "SAs": SAs,
                               "down_ws": down_ws})


def time_steps(args, sg, pr: Prepared, steps: int, world: int, dev, stream):
    """W eager warm-up steps, then exactly `steps` steps timed with CUDA events.

    Returns (steps, seconds on this rank, max over ranks, launch note, clocks).
    """
    copies = pr.copies

    def step(i):
        pr.fwd(i % copies, stream)

    for i in range(args.warmup):
        step(i)
    sg.swiglu_check_device_status(stream=stream)

    if steps <= 0:  # auto: about two seconds of timed work
        for i in range(2 * copies):
            step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(4 * copies):
            step(i)
        torch.cuda.synchronize()
        est = (time.perf_counter() - t0) / (4 * copies)
        steps = int(min(max(50, 2.0 / max(est, 1e-6)), 200000))

    # The timed steps replay from CUDA graphs captured from the same forward
    # calls (one kernel node per step), so consecutive launches overlap through
    # programmatic dependent launch as they do in a model's step, and the
    # host's per-call cost does not pace microsecond-scale kernels.
    run_steps, note = eager_runner(step), "eager launches, one host call per step"
    if not args.eager:
        try:
            run_steps = graph_runner(pr.fwd, copies, stream, steps)
            note = (f"CUDA graph replay of exactly {steps} steps: "
                    f"{run_steps.block_replays} replay(s) of a {run_steps.block_steps}-step graph"
                    + (f" + one {run_steps.tail_steps}-step graph" if run_steps.tail_steps else "")
                    + "; one kernel node per step, steps rotate over the operand copies")
        except Exception as exc:  # capture refused: keep eager launches, say so
            note = f"eager launches (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize()
    run_steps.warm() if hasattr(run_steps, "warm") else run_steps(min(steps, 2 * copies))
    torch.cuda.synchronize()

    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        t_begin.record(stream)
        run_steps(steps)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    sg.swiglu_check_device_status(stream=stream)
    elapsed = t_begin.elapsed_time(t_end) * 1e-3
    return steps, elapsed, max_over_ranks(elapsed, world), note, sampler.summary()


def roofline(pr: Prepared, avg_launch: float, peaks: dict, peak_src: str) -> dict:
    """The fused kernel's achieved rate per launch against the measured peaks."""
    # FP8 tensor peak: the measured bf16 figures times the nominal fp8/bf16
    # ratio (4.5 / 2.25 PFLOP/s dense).
    tensor_peak = peaks["bf16_tflops"] * (2.0 if pr.fp8 else 1.0)
    tensor_sus = peaks.get("bf16_tflops_sustained")
    tensor_sus = tensor_sus * (2.0 if pr.fp8 else 1.0) if tensor_sus else None
    hbm_bound = pr.flops / pr.alg_bytes < tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    traffic, traffic_src = profiled_traffic(pr.kernel, pr.w.name)
    if hbm_bound:
        achieved = pr.alg_bytes / avg_launch / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes": pr.alg_bytes}
    else:
        achieved = pr.flops / avg_launch / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(tensor_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / tensor_peak, 4),
                "traffic": traffic, "algorithmic_flops": pr.flops,
                "algorithmic_bytes": pr.alg_bytes,
                "peak_sustained": round(tensor_sus, 1) if tensor_sus else None,
                "frac_sustained": round(achieved / tensor_sus, 4) if tensor_sus else None}
    roof.update({"kernel": pr.kernel, "plan": pr.plan, "avg_launch_us": round(avg_launch * 1e6, 3),
                 "peak_source": peak_src + (
                     ", copy bandwidth" if hbm_bound else
                     ", bf16 burst x 2 (nominal fp8/bf16 ratio)" if pr.fp8 else ", burst"),
                 "traffic_source": traffic_src})
    return roof


def l2_note(pr: Prepared) -> str:
    return (f"inputs larger than L2: {pr.copies} rotating copies of "
            f"{'Y, packed W3, R and Out' if pr.down else 'A, packed W and Y'} "
            f"({pr.copies * pr.alg_bytes / 2**20:.0f} MiB; "
            f"{(pr.copies - 1) * pr.alg_bytes / 2**20:.0f} MiB of other copies "
            f"between two uses of one)")


def run_ours(args, w: Workload, world: int, rank: int, local: int):
    import swiglu_gated_mlp_gb300 as sg
    from swiglu_gated_mlp_gb300 import build as _build
    _build.build_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    M, K, N = w.M, w.K, w.N
    peaks, peak_src = load_peaks()

    pr = prepare(args, sg, w, dev)
    fp8, down, out_cols = pr.fp8, pr.down, pr.out_cols
    steps, elapsed, elapsed_max, graph_note, clocks = time_steps(args, sg, pr, args.steps, world,
                                                                 dev, stream)
    value = aggregate(pr.flops, steps, elapsed_max, world)
    # One fused-kernel launch per step and nothing else in the timed region, so
    # the average launch duration is the region's CUDA-event time over the
    # launches (events between launches would block the launch overlap).
    avg_launch = elapsed / steps
    roof = roofline(pr, avg_launch, peaks, peak_src)

    # ---- end to end through the public API: host activations in, host output out
    a_cpu = pr.a_cpu
    wps = pr.dev_state["wps"]
    Rs = pr.dev_state["Rs"]
    copies = pr.copies
    a_host = [a_cpu.pin_memory()] + [a_cpu.clone().pin_memory() for _ in range(min(copies, 4) - 1)]
    y_host = [torch.empty(M, out_cols, dtype=torch.bfloat16).pin_memory()
              for _ in range(len(a_host))]
    # Two streams, each with its own device staging buffers, take alternate
    # steps (as a serving loop would): one step's host copies overlap the
    # neighbouring steps' kernels, and every step's copies stay in the region.
    e2e_streams = [stream, torch.cuda.Stream(device=dev)]
    a_dev = [torch.empty(*a_cpu.shape, dtype=a_cpu.dtype, device=dev) for _ in e2e_streams]
    y_dev = [torch.empty(M, out_cols, dtype=torch.bfloat16, device=dev) for _ in e2e_streams]
    # down-projection with a workspace: one per stream, as the streams overlap
    e2e_ws = [sg.swiglu_down_workspace(M, N, K, dev) if pr.dev_state.get("down_ws") else None
              for _ in e2e_streams]
    mx = "sat" in pr.host
    if mx:  # A's block scales travel with A every step
        sa_host = [pr.host["sat"].pin_memory() for _ in a_host]
        sa_dev = [torch.empty_like(pr.host["sat"], device=dev) for _ in e2e_streams]
    e2e_steps = steps
    copy_rates = host_copy_rates(a_host[0], a_dev[0], y_dev[0], y_host[0], stream)

    def e2e_step(i):
        j = i % len(a_host)
        b = i % len(e2e_streams)
        st = e2e_streams[b]
        if down:  # host copies through torch around the down-projection call
            with torch.cuda.stream(st):
                a_dev[b].copy_(a_host[j], non_blocking=True)
                sg.swiglu_down_forward(a_dev[b], wps[i % copies], K, R=Rs[i % copies],
                                       Out=y_dev[b], stream=st, workspace=e2e_ws[b])
                y_host[j].copy_(y_dev[b], non_blocking=True)
        elif mx:  # host copies through torch around the block-scaled call
            with torch.cuda.stream(st):
                a_dev[b].copy_(a_host[j], non_blocking=True)
                sa_dev[b].copy_(sa_host[j], non_blocking=True)
                sg.swiglu_forward_mxfp8(a_dev[b], sa_dev[b], wps[i % copies], N, Y=y_dev[b],
                                        stream=st)
                y_host[j].copy_(y_dev[b], non_blocking=True)
        elif fp8:  # host copies through torch around the FP8 call
            with torch.cuda.stream(st):
                a_dev[b].copy_(a_host[j], non_blocking=True)
                sg.swiglu_forward_fp8(a_dev[b], wps[i % copies], N, *pr.host["scales"],
                                      Y=y_dev[b], stream=st)
                y_host[j].copy_(y_dev[b], non_blocking=True)
        else:
            sg.swiglu_forward_from_host(a_host[j], wps[i % copies], N, y_host[j], a_dev[b],
                                        y_dev[b], stream=st)

    for i in range(max(3, args.warmup // 10)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)

    def compute(i, b, st):  # the step's kernel on device buffers, as in e2e_step
        if down:
            sg.swiglu_down_forward(a_dev[b], wps[i % copies], K, R=Rs[i % copies], Out=y_dev[b],
                                   stream=st, workspace=e2e_ws[b])
        elif mx:
            sg.swiglu_forward_mxfp8(a_dev[b], sa_dev[b], wps[i % copies], N, Y=y_dev[b], stream=st)
        elif fp8:
            sg.swiglu_forward_fp8(a_dev[b], wps[i % copies], N, *pr.host["scales"], Y=y_dev[b],
                                  stream=st)
        else:
            sg.swiglu_forward(a_dev[b], wps[i % copies], N, Y=y_dev[b], stream=st)

    # Where an end-to-end step's time goes: a few more steps on the same two
    # streams and buffers, after the timed region, with events between the
    # host-to-device copy, the kernel and the device-to-host copy. A phase's
    # time includes any wait behind the other stream's work (copy engines, SMs).
    phase_ev = []
    for i in range(4):
        b, j = i % len(e2e_streams), i % len(a_host)
        st = e2e_streams[b]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        with torch.cuda.stream(st):
            ev[0].record(st)
            a_dev[b].copy_(a_host[j], non_blocking=True)
            if mx:
                sa_dev[b].copy_(sa_host[j], non_blocking=True)
            ev[1].record(st)
            compute(i, b, st)
            ev[2].record(st)
            y_host[j].copy_(y_dev[b], non_blocking=True)
            ev[3].record(st)
        phase_ev.append(ev)
    torch.cuda.synchronize()

    def phase_ms(k):
        return round(sum(e[k].elapsed_time(e[k + 1]) for e in phase_ev) / len(phase_ev), 3)
    phases = {"h2d_ms": phase_ms(0), "kernel_ms": phase_ms(1), "d2h_ms": phase_ms(2),
              "steps": len(phase_ev),
              "how": "4 steps after the timed region on the same two streams, CUDA events "
                     "between the phases; each includes waits behind the other stream"}
    sg.swiglu_check_device_status(stream=stream)
    e2e = {"value": round(aggregate(pr.flops, e2e_steps, e2e_s, world), 3), "unit": "TFLOP/s",
           "h2d_bytes_per_step": a_cpu.numel() * a_cpu.element_size() + (
               pr.host["sat"].numel() if mx else 0),
           "d2h_bytes_per_step": 2 * M * out_cols,
           "steps": e2e_steps, "streams": len(e2e_streams), "copy_rates": copy_rates,
           "phases": phases,
           "api": ("pinned-host copies + swiglu_down_forward" if down else
                   "pinned-host copies (A and its block scales) + swiglu_forward_mxfp8" if mx else
                   "pinned-host copies + swiglu_forward_fp8" if fp8 else
                   "swiglu_forward_from_host")}
    del a_dev, y_dev, a_host, y_host, wps, Rs, e2e_step, compute, phase_ev

    tensor_peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    out = {
        "metric": METRIC_DOWN if down else METRIC, "value": round(value, 3), "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(elapsed_max / steps * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("mxfp8-e4m3 (UE8M0 scale per 32 K, fp32 accumulate, bf16 out)" if args.dtype == "mxfp8"
                  else "fp8-e4m3 (fp32 accumulate, bf16 out)" if fp8 else "bf16"),
        "data": "synthetic",
        "config": {"workload": w.name, "M": M, "K": K, "N": N, "seed": w.seed,
                   "variant": args.variant, "inputs": args.dtype, "op": args.op,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": graph_note,
                   "l2": l2_note(pr),
                   "note": (f"down-projection Out[M,H] = Y[M,N] W3[N,H] + R at this workload's "
                            f"MLP shape, H = {K}" if down else w.note)},
        "pct_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 3),
        "pct_of_dtype_peak": round(100 * value / world / tensor_peak, 3),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": steps,
        "clocks": clocks,
        "packed_weight_bytes": pr.w_bytes,
    }
    if args.compare_unfused and not (fp8 or down):
        out["unfused"] = unfused_comparison(w, pr.dev_state["As"], pr.host["w1"].to(dev),
                                            pr.host["w2"].to(dev), copies, steps, elapsed / steps,
                                            peaks)
    y_check = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not (down or fp8):
        # the timed output itself (every rotation slot holds the same inputs) is
        # compared with the oracle values the baseline computes anyway
        y_check = bf16_bits(pr.dev_state["Ys"][0].cpu())
    host = pr.host
    pr.release()
    del pr
    torch.cuda.empty_cache()

    # ---- secondary records: other workloads, same timing path, device-timed only
    secondary = []
    if args.secondary and not (down or fp8 or args.m or args.variant != "auto"):
        for name in [s for s in args.secondary.split(",") if s and s != w.name]:
            ws = workload_by_name(name)
            ps = prepare(args, sg, ws, dev)
            s_steps, s_el, s_max, s_note, s_clocks = time_steps(args, sg, ps, args.steps, world,
                                                                dev, stream)
            secondary.append({
                "workload": ws.name, "M": ws.M, "K": ws.K, "N": ws.N, "seed": ws.seed,
                "value": round(aggregate(ps.flops, s_steps, s_max, world), 3), "unit": "TFLOP/s",
                "steps": s_steps, "ms_per_step": round(s_max / s_steps * 1e3, 6),
                "gpu_launches": s_steps, "launch": s_note, "l2": l2_note(ps),
                "roofline": roofline(ps, s_el / s_steps, peaks, peak_src), "clocks": s_clocks,
                "note": ws.note})
            ps.release()
            del ps
            torch.cuda.empty_cache()
    if secondary:
        out["secondary"] = secondary

    if rank == 0 and world == 1 and not args.no_cpu_baseline and not (down or fp8):
        out["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds, y_gpu_bits=y_check,
                                           inputs=(host["a"], host["w1"], host["w2"]))
    return out


# ------------------------------------------------------------ step runners ----

def eager_runner(step):
    def run(n):
        for i in range(n):
            step(i)
    return run


def graph_runner(fwd, copies, stream, steps, max_block=512):
    """Captures exactly `steps` forward steps into CUDA graphs.

    Up to `max_block` steps: one graph of exactly `steps` kernel nodes, so the
    whole timed region is one replay and every launch after the first overlaps
    its predecessor. More steps: a graph of whole turns of the rotation
    (about 256 steps), replayed, plus one graph of the remainder; both start at
    rotation slot 0, so slots keep their order across replays.
    """
    if steps <= max_block:
        block_steps, tail_steps = steps, 0
    else:
        block_steps = copies * max(1, 256 // copies)
        tail_steps = steps % block_steps
    replays = steps // block_steps
    side = torch.cuda.Stream(stream.device)
    side.wait_stream(stream)
    graphs = []
    with torch.cuda.stream(side):
        for n in (block_steps, tail_steps):
            if n == 0:
                graphs.append(None)
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    fwd(i % copies)
            graphs.append(g)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    block, tail = graphs

    def run(n):
        assert n == steps, "the graphs hold exactly the timed step count"
        for _ in range(replays):
            block.replay()
        if tail is not None:
            tail.replay()

    def warm():
        # first replays upload the graphs; not part of the timed region
        block.replay()
        if tail is not None:
            tail.replay()

    run.block_steps, run.tail_steps, run.block_replays, run.warm = block_steps, tail_steps, replays, warm
    return run


# ------------------------------------------------------ unfused comparator ----

def unfused_comparison(w: Workload, As, w1, w2, copies: int, steps: int, fused_s: float, peaks):
    """The unfused path the pages compare against, timed on the same GPU.

    PyTorch eager: two cuBLAS GEMMs that write bf16 Gate and Up to HBM, then
    SiLU and the product as separate kernels ("Tile-Level Activation Overlap
    for Efficient LLM Inference", gist.science, sections "Problem Statement"
    and "Results": speedup over PyTorch eager, fusion efficiency, arithmetic
    intensity). Timed like the fused path: rotating inputs, CUDA events over
    the region. Derived metrics follow the pages' model, in which fusion
    removes four intermediate HBM operations (write and read of Gate and Up,
    8*M*N bytes): theoretical speedup = t_unfused / (t_unfused - 8MN / HBM
    peak); fusion efficiency = actual speedup / theoretical speedup.
    """
    M, K, N = w.M, w.K, w.N
    n = max(3, min(steps, int(2.0 / max(fused_s * 2, 1e-6))))

    # the same rotation of inputs larger than L2 as the fused path
    W1s = [w1] + [w1.clone() for _ in range(copies - 1)]
    W2s = [w2] + [w2.clone() for _ in range(copies - 1)]

    def step(i):
        j = i % copies
        g = As[j] @ W1s[j]
        u = As[j] @ W2s[j]
        return torch.nn.functional.silu(g) * u

    for i in range(5):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(n):
        step(i)
    t1.record()
    torch.cuda.synchronize()
    t_unf = t0.elapsed_time(t1) * 1e-3 / n
    extra = 8 * M * N
    t_theory = max(t_unf - extra / (peaks["hbm_gbs"] * 1e9), 1e-12)
    speedup = t_unf / fused_s
    theoretical = t_unf / t_theory
    ai_fused = w.flops / w.algorithmic_bytes
    ai_unfused = w.flops / (w.algorithmic_bytes + 2 * M * K + extra)  # A read by both GEMMs
    return {"impl": "torch eager: cuBLAS GEMM x2 (bf16 Gate, Up in HBM) + silu + mul",
            "steps": n, "us_per_step": round(t_unf * 1e6, 3),
            "fused_us_per_step": round(fused_s * 1e6, 3),
            "tflops": round(w.flops / t_unf / 1e12, 3), "speedup": round(speedup, 4),
            "theoretical_speedup": round(theoretical, 4),
            "fusion_efficiency": round(speedup / theoretical, 4),
            "ai_fused": round(ai_fused, 2), "ai_unfused": round(ai_unfused, 2),
            "ai_increase_pct": round(100 * (ai_fused / ai_unfused - 1), 2),
            "intermediate_bytes_removed": extra}


# ---------------------------------------------------------- oracle timing ----

def _oracle_sample_call(a_bits, w1_bits, w2_bits, cols):
    from oracle.swiglu_ref import swiglu_f64
    return swiglu_f64(a_bits, w1_bits[:, cols], w2_bits[:, cols])


def cpu_baseline(w: Workload, budget_s: float = 12.0, y_gpu_bits=None, inputs=None,
                 max_rows: int = 512):
    """The float64 CPU oracle, as it stands, on a bounded sample of the workload.

    Up to `max_rows` rows are kept (all of them for small M; else a seeded
    subset that includes rows 0 and M-1), and a contiguous block of output
    columns is taken so that one call costs about a quarter of the budget.
    Returns TFLOP/s counted like the GPU metric (4 * rows * K * cols per
    call) and the time a whole step would take at that rate (extrapolated).
    With `y_gpu_bits` (the GPU's Y as bf16 bits), the oracle values of every
    call are also compared with it, outside the timed calls ("parity").
    """
    a, w1, w2 = inputs if inputs is not None else make_workload_inputs(w)
    rows = sample_rows(w.M, max_rows, seed=w.seed)
    a_bits = bf16_bits(a)[rows]
    w1_bits, w2_bits = bf16_bits(w1), bf16_bits(w2)
    # calibrate on a small block
    probe_cols = max(8, min(w.N, 256))
    t0 = time.perf_counter()
    _oracle_sample_call(a_bits, w1_bits, w2_bits, slice(0, probe_cols))
    t_probe = max(time.perf_counter() - t0, 1e-4)
    per_col = t_probe / probe_cols
    target = min(budget_s / 4, 3.0)
    cols = int(max(8, min(w.N, target / per_col)))
    calls, total_t, flops = 0, 0.0, 0
    checked = []  # (GPU bits, oracle values) per checked column block
    t_start = time.perf_counter()
    while True:
        c0 = (calls * cols) % max(w.N - cols + 1, 1)
        t0 = time.perf_counter()
        ref = _oracle_sample_call(a_bits, w1_bits, w2_bits, slice(c0, c0 + cols))
        total_t += time.perf_counter() - t0
        if y_gpu_bits is not None and calls < 4:
            checked.append((y_gpu_bits[rows][:, c0:c0 + cols], ref))
        flops += 4 * len(rows) * w.K * cols
        calls += 1
        if time.perf_counter() - t_start > budget_s:
            break
    rate = flops / total_t
    row_text = (f"all {w.M} rows" if len(rows) == w.M else
                f"{len(rows)} of {w.M} rows (seeded subset with rows 0 and {w.M - 1})")
    out = {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": _CORES,
           "kind": "oracle",
           "sample": f"{calls} call(s) of the float64 oracle on {row_text} x {cols} of "
                     f"{w.N} columns (K={w.K}), {total_t:.1f} s of CPU time",
           "full_step_s_extrapolated": round(w.flops / rate, 1),
           "threads_env": os.environ.get("OPENBLAS_NUM_THREADS")}
    if checked:
        from oracle import compare
        rep = compare.report(np.concatenate([c[0] for c in checked], axis=1),
                             np.concatenate([c[1] for c in checked], axis=1))
        out["parity"] = {"outputs": int(sum(c[1].size for c in checked)),
                         "rule": "|y - ref| <= 1e-2 |ref| + 1e-3",
                         "tolerance_pass": bool(rep["tolerance_pass"]),
                         "mismatch_rate": rep["mismatch_rate"],
                         "bf16_ulp_gt1_rate": rep["bf16_ulp_gt1_rate"],
                         "max_abs_err": rep["max_abs_err"], "nonfinite": rep["nonfinite"]}
    return out


def run_reference(args, w: Workload, world: int, rank: int):
    """Reference arm: the CPU oracle timed on bounded samples of the workload."""
    if rank != 0:
        return None
    steps = args.steps if args.steps > 0 else 20
    warm = max(args.warmup, 0)
    per_step = max(0.001, min(2.0, 90.0 / (steps + warm)))
    a, w1, w2 = make_workload_inputs(w)
    a_bits, w1_bits, w2_bits = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    probe_cols = max(8, min(w.N, 256))
    t0 = time.perf_counter()
    _oracle_sample_call(a_bits, w1_bits, w2_bits, slice(0, probe_cols))
    per_col = max(time.perf_counter() - t0, 1e-4) / probe_cols
    cols = int(max(8, min(w.N, per_step / per_col)))
    for i in range(warm):
        _oracle_sample_call(a_bits, w1_bits, w2_bits, slice(0, cols))
    t0 = time.perf_counter()
    for i in range(steps):
        c0 = (i * cols) % max(w.N - cols + 1, 1)
        _oracle_sample_call(a_bits, w1_bits, w2_bits, slice(c0, c0 + cols))
    t = time.perf_counter() - t0
    value = 4 * w.M * w.K * cols * steps / t / 1e12
    sample = (f"each step: the float64 oracle on all {w.M} rows x {cols} of {w.N} columns "
              f"(K={w.K})")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(t / steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "seed": w.seed,
                   "note": "no runnable implementation accompanies the method; the CPU "
                           "float64 oracle stands in as the reference arm"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _CORES,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def library_peak(kind: str, n: int = 8192, seconds: float = 4.0) -> dict:
    """cuBLAS(Lt) GEMM throughput on this GPU, as context for the roofline peaks.

    bf16: torch.matmul of two n x n bf16 matrices. fp8: torch._scaled_mm of two
    n x n E4M3 matrices (unit scales, bf16 output). FLOPs 2 n^3 per call.
    Burst: the best of 10 single calls (CUDA events); sustained: calls back to
    back for `seconds`, which on this part runs at the power cap.
    """
    dev = torch.device("cuda", torch.cuda.current_device())
    if kind == "fp8":
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()  # column-major operand
        one = torch.tensor(1.0, device=dev)

        def fn():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    else:
        a = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
        b = torch.randn(n, n, device=dev, dtype=torch.bfloat16)

        def fn():
            return a @ b
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    sampler = ClockSampler(dev.index)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    calls = 0
    with sampler:
        t0 = time.perf_counter()
        e0.record()
        while time.perf_counter() - t0 < seconds:
            for _ in range(20):
                fn()
            calls += 20
            torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
    flop = 2.0 * n ** 3
    return {"library_peak": "torch._scaled_mm (E4M3)" if kind == "fp8" else "torch.matmul (bf16)",
            "n": n, "unit": "TFLOP/s", "burst": round(flop / best / 1e12, 1),
            "sustained": round(flop * calls / (e0.elapsed_time(e1) * 1e-3) / 1e12, 1),
            "sustained_seconds": seconds, "clocks": sampler.summary()}


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0, help="timed steps (0: about 2 s of work)")
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--secondary", default=DEFAULT_SECONDARY,
                   help="comma-separated workloads timed after the main one, reported under "
                        "'secondary' (device-timed value and roofline); '' for none")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--rotate", type=int, default=0,
                   help="rotating copies of the operands (0: enough that 32 x L2 bytes of "
                        "other copies are read between two uses of one)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--down-workspace", choices=["on", "off"], default="on",
                   help="--op down: pass a workspace (K split across clusters allowed) or not")
    p.add_argument("--op", choices=["swiglu", "down"], default="swiglu",
                   help="swiglu: the fused gate/up projection (default); down: Out = Y W3 + R")
    p.add_argument("--dtype", choices=["bf16", "fp8", "mxfp8"], default="bf16",
                   help="input type: bf16 (the metric's), E4M3 with per-tensor scales, or "
                        "block-scaled E4M3 (one UE8M0 scale per 32 K values)")
    p.add_argument("--variant", choices=sorted(VARIANTS), default="auto",
                   help="kernel to time (default: the automatic choice)")
    p.add_argument("--eager", action="store_true",
                   help="time per-call launches instead of CUDA graph replay")
    p.add_argument("--compare-unfused", action="store_true",
                   help="also time the unfused PyTorch eager path and report the derived metrics")
    p.add_argument("--library-peak", choices=["bf16", "fp8"], default=None,
                   help="instead of the op: the library GEMM's throughput for context "
                        "(bf16: torch.matmul; fp8: torch._scaled_mm, E4M3), 8192^3, burst "
                        "(best of 10) and sustained (4 s back to back), with clocks")
    p.add_argument("--m", type=int, default=0,
                   help="token count in place of the workload's M (same K, N and seed; the "
                        "workload name gets an @M= suffix)")
    args = p.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    if args.library_peak:
        print(json.dumps(library_peak(args.library_peak)), flush=True)
        return
    w = workload_by_name(args.workload)
    if args.m > 0:
        w = dataclasses.replace(w, name=f"{w.name}@M={args.m}", M=args.m,
                                note=f"{w.note}; M set to {args.m}")
    if args.impl == "reference":
        # rank 0 alone runs the CPU reference; other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        out = run_reference(args, w, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    out = run_ours(args, w, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
