#!/usr/bin/env python3
"""Benchmark: bf16 GEMM TFLOP/s (2*M*N*K / time) on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config s4k|s8k|edge|skinny|s256]

A step is one C = alpha*A*B + beta*C over the configured workload (default:
M = N = K = 4096, bf16 inputs, fp32 accumulation, bf16 output, A row-major,
B and C column-major, N(0,1) inputs — the H100 work log's headline shape).

Timing: W untimed warm-up steps, then K timed steps between a barrier plus
torch.cuda.synchronize() on both sides.  The 96 MiB working set of the 4096
case fits in the 126 MiB L2, so a 512 MiB buffer is written between timed
steps (untimed) and each GEMM is timed alone with CUDA events on its stream.
The other large workloads (8192^3 with beta = 0.5, the 4000x4100x4104 edge
shape, the 64x8192x8192 skinny shape) are timed the same way after the main
line and reported under "subrecords", each with its own roofline and clocks.

With N > 1 (torchrun), the default (--multi slabs) splits one GEMM N times
wider than the workload into N contiguous column slabs of B and C, A
replicated: rank g computes C[:, g*N:(g+1)*N] (weak scaling, no collective on
the data path).  --multi replicas gives every rank its own copy of the
workload instead.  The max over ranks is taken and `value` is the aggregate
over all ranks.

`--impl reference` times the CPU oracle (the plain C definition) on a bounded
column slab of the same workload, on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bf16 GEMM TFLOP/s (2MNK/t) at 4096³/8192³ on 1 GB300; % of dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ("tensor_core_matmul_gb300/csrc/gemm_kernel.cuh", "tensor_core_matmul_gb300/csrc/ptx.cuh",
                  "tensor_core_matmul_gb300/csrc/tcgemm.cu")


def code_only(text: str) -> str:
    """C++ source without its comments and blank or trailing space, so that
    a change to a comment does not count as a change to the kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """sha256[:16] over the kernel sources' code (comments stripped)."""
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profile_traffic(kernel_tag: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None if the kernel's code changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel_tag and parts[1] == src:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float) -> float:
    """The largest x over all ranks (identity without a process group).  Every
    rank times its own independent problem; the job takes as long as the
    slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of `flops_per_step`
    (weak scaling), and the job lasted as long as the slowest rank."""
    return world * flops_per_step * steps / max_seconds / 1e12


EPILOGUES = {"none": (False, "none"), "bias": (True, "none"), "bias_relu": (True, "relu"),
             "bias_gelu": (True, "gelu"), "bias_gelu_tanh": (True, "gelu_tanh")}


def make_bias(args, N: int):
    """The fused epilogue's bias: N(0,1) fp32, one value per column of C
    (fixed seed), or None."""
    import torch
    if not EPILOGUES[args.epilogue][0]:
        return None
    return torch.randn(N, generator=torch.Generator().manual_seed(9001), dtype=torch.float32)


def flush_buffers(dev):
    import torch
    return (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev),
            torch.ones(FLUSH_BYTES // 8, dtype=torch.int64, device=dev))


def make_flush(bufs):
    flush, flush_rd = bufs

    def flush_l2(i: int, read: bool = True):
        # Write a buffer larger than L2 (evicts A, B and C), then read a
        # second one, so that L2 is left holding clean lines: the write-back
        # of the first buffer's dirty lines then happens here, untimed,
        # instead of inside the next timed call.
        flush.fill_(i & 0xFF)
        if read:
            flush_rd.sum()
    return flush_l2


def time_steps(gemm, flush_l2, stream, steps: int, dev, pg=None, sample_clocks: bool = True):
    """K timed steps, each one GEMM between its own CUDA events on `stream`
    after an untimed L2 flush; a barrier and a synchronize on both sides.
    Returns per-step milliseconds, the wall time of the loop, the library's
    kernel launches inside it and the sampled clocks."""
    import torch

    import tensor_core_matmul_gb300 as tc
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if sample_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.25)  # let the sampler take a first reading
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    n_launch0 = tc.launch_count()
    wall0 = time.perf_counter()
    for i in range(steps):
        flush_l2(i)                    # evict A, B, C from L2 (untimed)
        starts[i].record(stream)
        gemm()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if pg:
        pg.barrier()
    launches = tc.launch_count() - n_launch0
    clocks = sampler.stop() if sampler else None
    st, where = tc.check_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region (role {where})")
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], wall, launches, clocks


def gemm_call(args, case, A, B, C, stream, bias=None, act="none", row_scale=None, variant=0):
    """The public entry point this workload's options name, bound to its buffers."""
    import tensor_core_matmul_gb300 as tc
    M, N, K = case.M, case.N, case.K

    def gemm():
        if args.quant:
            tc.gemm_quant_i8(A, B, C, case.alpha, row_scale=row_scale, zero_point=0, bias=bias, activation=act, M=M,
                             N=N, K=K, stream=stream, variant=variant)
        elif case.in_format != "bf16":
            tc.gemm_fp8(A, B, C, case.alpha, case.beta, M=M, N=N, K=K, stream=stream, variant=variant)
        elif case.a_col or case.b_row:
            tc.gemm_bf16_layout(A, B, C, case.alpha, case.beta, a_col=case.a_col, b_row=case.b_row, M=M, N=N, K=K,
                                stream=stream, variant=variant)
        elif bias is None and act == "none":
            tc.gemm_bf16(A, B, C, case.alpha, case.beta, M=M, N=N, K=K, stream=stream, variant=variant)
        else:
            tc.gemm_bf16_bias_act(A, B, C, case.alpha, case.beta, bias=bias, activation=act, M=M, N=N, K=K,
                                  stream=stream, variant=variant)
    return gemm


def device_buffers(case, dev):
    import torch
    A = case.A.to(dev)
    B = case.B.to(dev)
    C = (case.C_in.to(dev) if case.C_in is not None
         else torch.zeros((case.N, case.ldc), dtype=case.out_torch_dtype(), device=dev))
    return A, B, C


def sub_record(args, name: str, dev, stream, flush_l2, world: int, pg, peaks, peak_src, sms: int) -> dict:
    """Another workload, plain bf16 GEMM through gemm_bf16, timed with the
    main line's protocol (flushed L2, CUDA events per call, clocks sampled):
    its own TFLOP/s, roofline and clocks.  Same slab rule as the main line."""
    import tensor_core_matmul_gb300 as tc
    sub_args = argparse.Namespace(**{**vars(args), "config": name, "in_format": "bf16", "layout": "tn",
                                     "epilogue": "none", "quant": False})
    case = bench_case(sub_args, world, dist_setup()[1])
    A, B, C = device_buffers(case, dev)
    gemm = gemm_call(sub_args, case, A, B, C, stream, variant=args.variant)
    for _ in range(args.warmup):
        flush_l2(1)
        gemm()
    times_ms, wall, launches, clocks = time_steps(gemm, flush_l2, stream, args.steps, dev, pg)
    total_s = max_over_ranks(sum(times_ms) / 1e3)
    variant = args.variant or tc.pick_variant(case.M, case.N, case.K, sms)
    plan = tc.plan(case.M, case.N, case.K, variant, sms)
    traffic = profile_traffic(f"gemm_{name}_full")
    del A, B, C
    return {
        "value": round(job_throughput(case.flops, args.steps, world, total_s), 2), "unit": "TFLOP/s",
        "ms_per_step": round(total_s / args.steps * 1e3, 5),
        "ms_per_step_median": round(float(sorted(times_ms)[len(times_ms) // 2]), 5),
        "steps": args.steps, "warmup": args.warmup, "gpu_launches": int(launches),
        "config": {"workload": workload_text(case, name), "M": case.M, "N": case.N, "K": case.K,
                   "kernel": {"variant": variant, **plan}},
        "roofline": roofline(case, total_s / args.steps, peaks, peak_src, traffic, sms=sms, clocks=clocks),
        "clocks": clocks,
    }


def workload_text(case, name: str) -> str:
    return (f"gemm {name}: M={case.M} N={case.N} K={case.K}, {case.in_format} A row-major x B col-major, "
            f"fp32 accumulate, {'bf16' if case.out_dtype else 'fp32'} C col-major, "
            f"alpha={case.alpha} beta={case.beta}, N(0,1) inputs")


def run_ours(args) -> None:
    import torch

    import tensor_core_matmul_gb300 as tc

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    case = bench_case(args, world, rank)
    M, N, K = case.M, case.N, case.K
    if args.quant:
        # int8 output of the quantising epilogue: written only, beta = 0.
        if case.beta != 0.0:
            raise SystemExit("--quant needs a workload with beta = 0")
        A, B = case.A.to(dev), case.B.to(dev)
        C = torch.zeros((N, (M + 15) // 16 * 16), dtype=torch.int8, device=dev)
        row_scale = (torch.rand(M, generator=torch.Generator().manual_seed(9002)) * 60 + 4).to(dev)
    else:
        A, B, C = device_buffers(case, dev)
        row_scale = None
    flush_bufs = flush_buffers(dev)
    flush, _ = flush_bufs
    flush_l2 = make_flush(flush_bufs)
    stream = torch.cuda.current_stream(dev)
    bias_cpu = make_bias(args, N)
    act = EPILOGUES[args.epilogue][1]
    bias = None if bias_cpu is None else bias_cpu.to(dev)

    if args.in_format != "bf16" and args.epilogue != "none" and not args.quant:
        raise SystemExit("--epilogue with 8-bit operands needs --quant")
    gemm = gemm_call(args, case, A, B, C, stream, bias=bias, act=act, row_scale=row_scale, variant=args.variant)

    tuned = None
    if args.autotune:
        if args.quant or args.epilogue != "none":
            raise SystemExit("--autotune times the plain GEMM (no --quant / --epilogue)")
        v, us = tc.autotune(A, B, C, case.alpha, case.beta, a_col=case.a_col, b_row=case.b_row, M=M, N=N, K=K,
                            iters=10, flush=flush, stream=stream)
        tuned = {"variant": v, "us_flushed": round(us, 2)}
    for _ in range(args.warmup):
        flush_l2(1)
        gemm()
    torch.cuda.synchronize(dev)
    st, where = tc.check_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} during warm-up (role {where})")

    times_ms, wall, launches, clocks = time_steps(gemm, flush_l2, stream, args.steps, dev, pg)
    total_s = max_over_ranks(sum(times_ms) / 1e3)
    # The work log's own protocol times back-to-back calls without flushing
    # L2 between them; reported beside the flushed number (same work).
    nf_steps = max(3, min(args.steps, 200))
    nf0 = torch.cuda.Event(enable_timing=True)
    nf1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    nf0.record(stream)
    for _ in range(nf_steps):
        gemm()
    nf1.record(stream)
    torch.cuda.synchronize(dev)
    nf_s = max_over_ranks(nf0.elapsed_time(nf1) / 1e3)
    # Same steps after a write-only flush (the dirty lines it leaves in L2
    # are written back during the timed call).
    wo = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i, (s0, s1) in enumerate(wo):
        flush_l2(i, read=False)
        s0.record(stream)
        gemm()
        s1.record(stream)
    torch.cuda.synchronize(dev)
    wo_s = max_over_ranks(sum(s0.elapsed_time(s1) for s0, s1 in wo) / 1e3)
    flops = case.flops
    value = job_throughput(flops, args.steps, world, total_s)
    ms_per_step = total_s / args.steps * 1e3

    peaks, peak_src = load_peaks()
    tag = (f"gemm_{args.config}_full" + ("" if args.epilogue == "none" else f"_{args.epilogue}")
           + ("" if args.in_format == "bf16" else f"_{args.in_format}") + ("_quant" if args.quant else "")
           + ("" if args.layout == "tn" else f"_{args.layout}"))
    traffic = profile_traffic(tag)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    variant = args.variant or (tuned["variant"] if tuned else tc.pick_variant(M, N, K, sms))
    plan = tc.plan(M, N, K, variant, sms, in_kind=0 if args.in_format == "bf16" else 1, a_col=case.a_col,
                   b_row=case.b_row)

    e2e = None
    if not args.no_e2e and not args.quant and args.layout == "tn":
        e2e = measure_e2e(args, case, dev, stream, bias_cpu, act, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quant and args.layout == "tn":
        cpu = cpu_baseline(case, target_s=args.cpu_seconds, bias=bias_cpu, act=act)

    subs = {}
    names = [n for n in (args.subrecords.split(",") if args.subrecords else []) if n and n != args.config]
    if names:
        del A, B, C, gemm
        torch.cuda.empty_cache()
        for name in names:
            subs[name] = sub_record(args, name, dev, stream, flush_l2, world, pg, peaks, peak_src, sms)
            torch.cuda.empty_cache()

    if rank == 0:
        slab = args.multi == "slabs" and world > 1
        out = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "ms_per_step_median": round(float(sorted(times_ms)[len(times_ms) // 2]), 5),
            "ms_per_step_min": round(float(min(times_ms)), 5),
            "no_flush": {"value": round(job_throughput(flops, nf_steps, world, nf_s), 2), "unit": "TFLOP/s",
                         "steps": nf_steps, "ms_per_step": round(nf_s / nf_steps * 1e3, 5),
                         "note": "back-to-back calls, L2 not flushed (the work log's protocol)"},
            "write_only_flush": {"value": round(job_throughput(flops, args.steps, world, wo_s), 2), "unit": "TFLOP/s",
                                 "ms_per_step": round(wo_s / args.steps * 1e3, 5),
                                 "note": "L2 flushed by the 512 MiB write alone: its dirty lines are written "
                                         "back inside the timed call"},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if args.in_format == "bf16" else f"fp8_{args.in_format}",
            "data": "synthetic",
            "config": {
                "workload": workload_text(case, args.config)
                            + ("" if args.epilogue == "none" else
                               f", fused epilogue C = {act}(alpha*A*B + beta*C + bias[j]), fp32 N(0,1) bias"),
                "M": M, "N": N, "K": K,
                "epilogue": args.epilogue,
                "in_format": args.in_format,
                "layout": {"tn": "A row-major, B column-major", "nn": "A column-major, B column-major",
                           "tt": "A row-major, B row-major", "nt": "A column-major, B row-major"}[args.layout],
                "output": "int8 (per-row quantisation)" if args.quant else ("bf16" if case.out_dtype else "fp32"),
                "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MiB written, then another "
                      f"{FLUSH_BYTES >> 20} MiB read, untimed: inputs evicted, L2 left clean)",
                "kernel": {"variant": {1: "1cta", 2: "2cta"}.get(variant, str(variant)), **plan},
                "autotuned": tuned,
                "parallelism": (f"one M x (N*{world}) x K GEMM in {world} contiguous column slabs of B and C, "
                                f"A replicated, no collective on the data path" if slab else
                                f"independent problem per GPU x{world}"),
                "wall_s_timed_loop": round(wall, 3),
            },
            "roofline": roofline(case, total_s / args.steps, peaks, peak_src, traffic,
                                 extra_bytes=(0 if bias_cpu is None else 4 * N)
                                 + (4 * M - M * N * (4 if case.out_dtype == 0 else 2) + M * N if args.quant else 0),
                                 sms=sms, clocks=clocks),
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "cpu_baseline": cpu,
        }
        if subs:
            out["subrecords"] = subs
        print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


def bench_case(args, world: int = 1, rank: int = 0):
    """The workload named by --config (shape, alpha/beta, output type, seed),
    with 8-bit operands when --in-format asks for them (same shapes, seeds and
    distribution).  Under --multi slabs with more than one rank, this rank's
    contiguous column slab of one GEMM `world` times wider (A replicated; the
    slabs are the column ranges gemm_inputs.slab_bounds gives)."""
    import gemm_inputs as gi
    c = gi.CONFIGS[args.config]
    if world > 1 and args.multi == "slabs":
        if args.in_format != "bf16" or args.layout != "tn":
            raise SystemExit("--multi slabs uses bf16 operands in the tn layout")
        n0, n1 = gi.slab_bounds(c["N"] * world, world, rank, align=c["N"])
        assert (n0, n1) == (rank * c["N"], (rank + 1) * c["N"])
        return gi.column_slab_case(args.config, world, rank)
    case = gi.make_case(args.config, c["M"], c["N"], c["K"], alpha=c["alpha"], beta=c["beta"],
                        out_dtype=c["out_dtype"], seed=c["seed"], in_format=args.in_format)
    if args.layout != "tn":
        # nn: A column-major; tt: B row-major; nt: both (the same logical matrices).
        case = gi.relayout(case, a_col=args.layout in ("nn", "nt"), b_row=args.layout in ("tt", "nt"))
    return case


def algorithmic_bytes(case) -> int:
    """Bytes a GEMM must move at least once: A and B read, C written, and C
    read too when beta != 0."""
    esz = 4 if case.out_dtype == 0 else 2
    isz = 2 if case.in_format == "bf16" else 1
    c = case.M * case.N * esz
    return isz * case.M * case.K + isz * case.N * case.K + c + (c if case.beta != 0.0 else 0)


# Dense bf16 tensor-core rate of one Blackwell SM taken by the formula peak
# SMs x rate x clock: 8192 FLOP (4096 multiply-adds) per clock; 8-bit
# operands at twice that.  Reported beside the measured cuBLAS peak.
BF16_FLOP_PER_CLK_SM = 8192


def formula_peak_tflops(sms: int, mhz: float, fp8: bool = False) -> float:
    return sms * BF16_FLOP_PER_CLK_SM * (2 if fp8 else 1) * mhz * 1e6 / 1e12


def roofline(case, t_launch: float, peaks: dict, peak_src: str, traffic, extra_bytes: int = 0, sms: int = 152,
             clocks: dict | None = None) -> dict:
    """Dominant kernel (the GEMM itself) against its bound: the tensor cores
    for the square / edge shapes, HBM for the skinny shape (intensity
    2MNK / bytes far below the ridge point).  extra_bytes: the fused
    epilogue's bias vector.  Tensor-bound lines also carry the formula peak
    SMs x 8192 FLOP/clk x clock, at the maximum SM clock and at the median
    clock sampled during the timed region."""
    flops = case.flops
    nbytes = algorithmic_bytes(case) + extra_bytes
    peak_flops = float(peaks["bf16_tflops"])
    fp8 = case.in_format != "bf16"
    if fp8:
        # No measured FP8 peak: the measured bf16 peak times the nominal
        # dense FP8 / BF16 ratio (4.5 / 2.25 PFLOP/s).
        peak_flops *= 2.0
    ridge = peak_flops * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    src = "measured" if peak_src == "measured" else "fallback"
    if flops / nbytes < ridge:
        achieved = nbytes / t_launch / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "algorithmic_bytes": nbytes, "tflops": round(flops / t_launch / 1e12, 2),
                "peak_source": f"{src} hbm_gbs (copy bandwidth)"}
    achieved = flops / t_launch / 1e12
    max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    med_mhz = (clocks or {}).get("sm_mhz") or None
    formula = formula_peak_tflops(sms, max_mhz, fp8)
    out = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_flops, "unit": "TFLOP/s",
           "frac": round(achieved / peak_flops, 4), "traffic": traffic, "algorithmic_bytes": nbytes,
           "peak_source": (f"{src} bf16_tflops (cuBLAS bf16 8192^3 burst)" if not fp8 else
                           f"{src} bf16_tflops x 2 (nominal dense fp8/bf16 ratio 4.5/2.25)"),
           "formula_peak": {"tflops": round(formula, 1), "sm_mhz": max_mhz,
                            "rule": f"{sms} SMs x {BF16_FLOP_PER_CLK_SM * (2 if fp8 else 1)} FLOP/clk x max SM clock",
                            "frac": round(achieved / formula, 4)}}
    if med_mhz:
        f_med = formula_peak_tflops(sms, float(med_mhz), fp8)
        out["formula_peak_at_median_clock"] = {"tflops": round(f_med, 1), "sm_mhz": med_mhz,
                                               "frac": round(achieved / f_med, 4)}
    return out


def measure_e2e(args, case, dev, stream, bias_cpu=None, act="none", world: int = 1) -> dict:
    """Same metric through the public API with host buffers: every step copies
    A and B (and C when beta != 0) from pinned host memory to the device, runs
    the GEMM and copies C back to pinned host memory.  For the plain GEMM that
    is one call of the C ABI's host-buffer entry point (gemm_bf16_host), which
    does the copies itself; the fused-epilogue and 8-bit workloads copy with
    torch around the device entry points.  Steps alternate between two streams
    with their own buffers, so one step's host-to-device copies overlap the
    previous step's GEMM and device-to-host copy (the copy engines run both
    directions at once); the timed region spans all steps on both streams."""
    import torch

    import tensor_core_matmul_gb300 as tc
    steps = max(4, min(args.steps, args.e2e_steps))
    nbuf = 2
    has_beta = case.beta != 0.0
    C0 = (case.C_in if case.C_in is not None
          else torch.zeros((case.N, case.ldc), dtype=case.out_torch_dtype()))
    hA = [case.A.pin_memory() for _ in range(nbuf)]
    hB = [case.B.pin_memory() for _ in range(nbuf)]
    hC_in = [C0.pin_memory() for _ in range(nbuf)]
    hC = [C0.clone().pin_memory() for _ in range(nbuf)]
    hbias = [None if bias_cpu is None else bias_cpu.pin_memory() for _ in range(nbuf)]
    dbias = [None if bias_cpu is None else torch.empty_like(bias_cpu, device=dev) for _ in range(nbuf)]
    dA = [torch.empty_like(case.A, device=dev) for _ in range(nbuf)]
    dB = [torch.empty_like(case.B, device=dev) for _ in range(nbuf)]
    dC = [torch.empty_like(C0, device=dev) for _ in range(nbuf)]
    streams = [torch.cuda.Stream(dev) for _ in range(nbuf)]

    host_entry = case.in_format == "bf16" and bias_cpu is None and act == "none"

    def step(i):
        b = i % nbuf
        s = streams[b]
        if host_entry:
            tc.gemm_bf16_host(hA[b], hB[b], hC[b], case.alpha, case.beta, M=case.M, N=case.N, K=case.K, stream=s)
            return
        with torch.cuda.stream(s):
            dA[b].copy_(hA[b], non_blocking=True)
            dB[b].copy_(hB[b], non_blocking=True)
            if has_beta:
                dC[b].copy_(hC_in[b], non_blocking=True)
            if case.in_format != "bf16":
                tc.gemm_fp8(dA[b], dB[b], dC[b], case.alpha, case.beta, M=case.M, N=case.N, K=case.K, stream=s,
                            variant=args.variant)
            elif bias_cpu is None and act == "none":
                tc.gemm_bf16(dA[b], dB[b], dC[b], case.alpha, case.beta, M=case.M, N=case.N, K=case.K, stream=s,
                             variant=args.variant)
            else:
                if bias_cpu is not None:
                    dbias[b].copy_(hbias[b], non_blocking=True)
                tc.gemm_bf16_bias_act(dA[b], dB[b], dC[b], case.alpha, case.beta, bias=dbias[b], activation=act,
                                      M=case.M, N=case.N, K=case.K, stream=s, variant=args.variant)
            hC[b].copy_(dC[b], non_blocking=True)

    for i in range(4):
        step(i)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(streams[0])
    for s in streams[1:]:
        s.wait_event(start)
    for i in range(steps):
        step(i)
    for s in streams[1:]:
        streams[0].wait_stream(s)
    end.record(streams[0])
    torch.cuda.synchronize(dev)
    t = start.elapsed_time(end) / 1e3
    h2d = (case.A.numel() * case.A.element_size() + case.B.numel() * case.B.element_size()
           + (C0.numel() * C0.element_size() if has_beta else 0))
    h2d += 0 if bias_cpu is None else bias_cpu.numel() * 4
    d2h = C0.numel() * C0.element_size()
    t = max_over_ranks(t)
    return {"value": round(world * case.flops * steps / t / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(t / steps * 1e3, 4), "streams": nbuf,
            "api": "gemm_bf16_host (C ABI, host buffers)" if host_entry else "torch copies + device entry point",
            "link_gbs": round((h2d + d2h) * steps / t / 1e9, 1)}


def oracle_slab(case, ncols: int, threads: int = 0, bias=None, act: str = "none") -> float:
    """Seconds for the oracle to compute columns [0, ncols) of C (with the
    fused epilogue when a bias or an activation is given)."""
    import numpy as np

    import gemm_inputs as gi
    import oracle
    o = oracle.get()
    A = gi.as_bits(case.A)
    B = gi.as_bits(case.B)[:ncols]
    fmt = None if case.in_format == "bf16" else case.in_format
    cin = None
    if case.C_in is not None:
        cin = case.C_in[:ncols]
        cin = gi.as_u16(cin) if cin.dtype.is_floating_point and cin.element_size() == 2 else cin.numpy()
    b = None if bias is None else bias[:ncols].numpy()
    t0 = time.perf_counter()
    if b is None and act == "none":
        o.gemm_f64(case.M, ncols, case.K, A, np.ascontiguousarray(B), cin, case.alpha, case.beta, threads=threads,
                   in_format=fmt)
    else:
        o.gemm_epi_f64(case.M, ncols, case.K, A, np.ascontiguousarray(B), cin, case.alpha, case.beta, bias=b,
                       act=act, threads=threads)
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 'model name', or the Arm
    implementer / part codes), else the platform string."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.processor() or platform.machine()
    for key in ("model name", "Model"):
        for line in info:
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in info:
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            if k in ("CPU implementer", "CPU part") and k not in parts:
                parts[k] = v
    if parts:
        return f"{platform.machine()} implementer {parts.get('CPU implementer')} part {parts.get('CPU part')}"
    return platform.machine()


def cpu_baseline(case, target_s: float, bias=None, act: str = "none") -> dict:
    import oracle
    cores = oracle.get().threads(0)
    ncal = max(1, min(case.N, cores))
    t = oracle_slab(case, ncal, bias=bias, act=act)
    per_col = t / ncal
    ncols = int(max(1, min(case.N, round(target_s / max(per_col, 1e-9)))))
    ncols = max(ncols, min(case.N, cores))
    t = oracle_slab(case, ncols, bias=bias, act=act)
    flops = 2 * case.M * ncols * case.K
    # One core: a slab of a few columns, for a per-core figure.
    n1 = max(1, min(case.N, int(round(1.0 / max(per_col * cores, 1e-9)))))
    t1 = oracle_slab(case, n1, threads=1, bias=bias, act=act)
    per_core = 2 * case.M * n1 * case.K / t1 / 1e9
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "per_core_gflops": round(per_core, 3),
            "sample": f"columns 0..{ncols - 1} of C ({case.M}x{ncols}x{case.K}, {flops / 1e9:.1f} GFLOP), "
                      f"{t:.1f} s on {cores} threads; fp64 k-ascending definition"}


def run_reference(args) -> None:
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle

    case = bench_case(args)
    bias = make_bias(args, case.N)
    act = EPILOGUES[args.epilogue][1]
    cores = oracle.get().threads(0)
    # Size each step's column slab so the whole run takes about args.ref_seconds.
    ncal = max(1, min(case.N, cores))
    per_col = oracle_slab(case, ncal, bias=bias, act=act) / ncal
    total_steps = args.steps + args.warmup
    ncols = int(max(1, min(case.N, round(args.ref_seconds / total_steps / max(per_col, 1e-9)))))
    for _ in range(args.warmup):
        oracle_slab(case, ncols, bias=bias, act=act)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_slab(case, ncols, bias=bias, act=act)
    flops = 2 * case.M * ncols * case.K
    value = flops * args.steps / t / 1e12
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"gemm {args.config}: M={case.M} N={case.N} K={case.K}; each step computes "
                               f"columns 0..{ncols - 1} of C with the CPU oracle"
                               + ("" if args.epilogue == "none" else f", fused epilogue {args.epilogue}"),
                   "M": case.M, "N": case.N, "K": case.K, "epilogue": args.epilogue,
                   "in_format": args.in_format},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{ncols} columns of C per step ({case.M}x{ncols}x{case.K})"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="s4k", choices=["s256", "s4k", "s8k", "edge", "skinny"])
    ap.add_argument("--variant", type=int, default=0, help="0 auto, 1 one-CTA, 2 CTA-pair kernel")
    ap.add_argument("--in-format", default="bf16", choices=["bf16", "e4m3", "e5m2"],
                    help="operand type: bf16 (gemm_bf16) or 8-bit floats (gemm_fp8)")
    ap.add_argument("--epilogue", default="none", choices=sorted(EPILOGUES),
                    help="fused epilogue: bias and/or activation (gemm_bf16_bias_act)")
    ap.add_argument("--layout", default="tn", choices=["tn", "nn", "tt", "nt"],
                    help="operand storage, first letter A (t row-major, n column-major), second B (n "
                         "column-major, t row-major): tn is the pages' layout; others use gemm_bf16_layout")
    ap.add_argument("--autotune", action="store_true",
                    help="time every variant first (tcgemm_autotune) and let the automatic choice use the fastest")
    ap.add_argument("--quant", action="store_true",
                    help="int8 output through the per-row quantising epilogue (gemm_quant_i8)")
    ap.add_argument("--subrecords", default="s8k,edge,skinny",
                    help="other workloads timed the same way (plain bf16 GEMM) and reported under 'subrecords' "
                         "(comma-separated; empty for none)")
    ap.add_argument("--multi", default="slabs", choices=["slabs", "replicas"],
                    help="with N > 1 ranks: 'slabs' splits one GEMM N times wider into contiguous column slabs "
                         "of B and C (A replicated); 'replicas' gives every rank its own copy of the workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
