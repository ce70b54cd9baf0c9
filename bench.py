#!/usr/bin/env python
"""Benchmark of the SmoothQuant W8A8 linear-layer hot path on B300.

One step = the whole path over one layer's synthetic inputs: per-channel
absmax of X and W, smoothing factors, fold + INT8 quantization of W, fused
X*S^-1 + per-token INT8 quantization, and the INT8 GEMM with its bf16
epilogue.  The step is replayed as two CUDA graphs (steps 1-4, then the
GEMM, whose duration gives the roofline figure).  Inputs are resident in
HBM before the timed region; L2 is flushed (a 256 MiB write, then a 256 MiB
read so no dirty flush lines remain, outside the per-step events) before
every step.  Each kernel is also timed alone, L2
flushed before it, for its HBM fraction.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead, on a bounded sample of the same workload.  Under torchrun each rank
runs an independent replica (the one-layer path has no exchange between
ranks); the reported time is the max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W8A8 GEMM TOPS (% int8 tensor peak); act-quant GB/s (% HBM peak)"
DEFAULT_WORKLOAD = "prefill_upgate_2048x4096x11008"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--codes", choices=["auto", "i8", "bf16"], default="auto",
                    help="storage of the INT8 codes: one byte each (i8), the same integers as exact "
                         "bf16 values (bf16), or the library's choice (auto: one byte each)")
    ap.add_argument("--i8-gemm", choices=["widened", "onchip"], default="widened",
                    help="1-byte codes above 64 tokens: widen both operands to fp16 in the GEMM's "
                         "workspace first (widened), or give the GEMM no workspace so it widens the "
                         "codes in shared memory as it goes (onchip)")
    ap.add_argument("--act-scale", choices=["dynamic", "static", "norm"], default="dynamic",
                    help="per-token scales (default), one calibrated scale per tensor, or per-token "
                         "scales after an RMS normalization whose gain absorbs S^-1 (the workload's X "
                         "then stands for the normalization's input)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("SQ_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="sq_clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, v in enumerate(flags)
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- the oracle arm
def blas_threads() -> int:
    """BLAS threads of this process: threadpoolctl's count where it is
    installed, else the OpenBLAS thread variable the parent set."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except ImportError:
        return int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0) or host_cores()


def oracle_sample_case(case, tokens: int):
    from w8a8_post_quantization_02_b300 import synth
    x = case.x[:tokens]
    return synth.Case(name=case.name + f"[:{tokens}]", dtype=case.dtype, tokens=tokens, cin=case.cin,
                      cout=case.cout, alpha=case.alpha, x=x, w=case.w, splits=case.splits)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_child(case_name: str, budget_s: float, sample_tokens: int, max_steps: int) -> dict:
    """Body of the oracle timing process (see time_oracle)."""
    from oracle import sq_oracle as O
    from w8a8_post_quantization_02_b300 import synth
    case = synth.workload(case_name)
    sc = oracle_sample_case(case, sample_tokens)
    x, w = sc.x_f32(), sc.w_f32()
    times = []
    t_start = time.perf_counter()
    while len(times) < max_steps:
        t0 = time.perf_counter()
        O.run_path(x, w, sc.alpha)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    return {"times": times, "ops": 2 * sample_tokens * case.cin * case.cout, "threads": blas_threads()}


def time_oracle(case_name: str, budget_s: float, sample_tokens: int, max_steps: int,
                threads: int | None = None):
    """Run the oracle's whole path on a token sample of the layer (full W)
    until ``max_steps`` runs or ``budget_s`` seconds are used, with the BLAS
    library (the oracle's one multi-threaded primitive, the accumulator
    matmul) on ``threads`` threads (default: every core this process may
    use).  It runs in a fresh interpreter whose thread count is fixed by the
    environment before numpy loads, so the limit holds without a runtime
    thread-control package and the oracle never shares a process with CUDA.
    Returns (times, ops, threads used)."""
    n = str(threads or host_cores())
    env = dict(os.environ, OPENBLAS_NUM_THREADS=n, OMP_NUM_THREADS=n, MKL_NUM_THREADS=n)
    code = ("import json, bench; print(json.dumps(bench.oracle_child(%r, %r, %d, %d)))"
            % (case_name, float(budget_s), sample_tokens, max_steps))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle timing process failed:\n" + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["times"], d["ops"], d["threads"]


def run_reference(args, case_name):
    from w8a8_post_quantization_02_b300 import synth
    rank, world, _ = dist_setup()
    if rank != 0:
        return 0
    case = synth.workload(case_name)
    sample_tokens = min(case.tokens, 256)
    # one untimed run first (warm-up), then the timed steps within a few minutes
    times, ops, cores = time_oracle(case_name, 150.0, sample_tokens, args.steps + 1)
    times = times[1:] or times
    sec = sum(times)
    value = ops * len(times) / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": sec / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(case, "oracle"),
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": f"whole path on the first {sample_tokens} tokens with the full "
                                   f"{case.cin}x{case.cout} weight, {len(times)} runs"},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(case, codes):
    return {"workload": case.name, "tokens": case.tokens, "cin": case.cin, "cout": case.cout,
            "alpha": case.alpha, "input_dtype": case.dtype, "codes": codes,
            "splits": list(case.splits) or None,
            "l2": "flushed before every step (256 MiB write, then 256 MiB read, outside the step events)"}


# ----------------------------------------------------------------- our arm
def to_device(case, torch):
    def conv(a):
        if case.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a))
    return conv(case.x), conv(case.w)


# DRAM bytes per launch read back from one ncu capture of the same kernel
# on the same workload (dram__bytes_read.sum + dram__bytes_write.sum), or
# absent when the kernel changed after the capture.
NCU_TRAFFIC_BYTES = {
    # 107.96 MB read + 26.16 MB written (the rest of Y still dirty in L2)
    ("k_gemm_bf16c", "prefill_upgate_2048x4096x11008"): 134.12e6,
    # 107.91 MB read (the widened fp16 operands) + 23.49 MB written
    ("k_gemm_bf16c<fp16>", "prefill_upgate_2048x4096x11008"): 131.40e6,
    # (--i8-gemm onchip) 53.87 MB read (the int8 codes of X and W, once) + 9.99 MB written
    ("k_gemm_i8c", "prefill_upgate_2048x4096x11008"): 63.86e6,
    # 16.88 MB read (the int8 weight codes and X codes), nothing written back yet
    ("k_gemm_dec", "decode_7b_16x4096x4096"): 16.88e6,
}


def run_ours(args, case_name):
    import torch
    from w8a8_post_quantization_02_b300 import pipeline, sq, synth
    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    sq.check_device(local)
    peaks, peaks_kind = load_peaks()
    case = synth.workload(case_name)
    x_host, w_host = to_device(case, torch)
    layer = pipeline.Layer.for_case(case, codes=None if args.codes == "auto" else args.codes,
                                    act_scale=args.act_scale, gemm_workspace=args.i8_gemm == "widened")
    layer.load(x_host.cuda(), w_host.cuda())
    stream = torch.cuda.current_stream()
    st = sq._stream(stream)
    stages = layer.stages()
    names = [n for n, _, _ in stages]
    # L2 flush: write one buffer larger than L2, then read a second one, so
    # the L2 holds only clean lines of the second buffer when a timed region
    # starts (after a write alone, up to the L2's size of the flush's dirty
    # lines would be written back to HBM inside the timed kernels)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush_l2():
        flush.zero_()
        flush_rd.sum()

    # one eager step (library set-up), then the step as two CUDA graphs:
    # steps 1-4 and the GEMM, so the GEMM's own duration is timed live
    layer.step()
    torch.cuda.synchronize()
    g_pre, g_gemm = layer.capture()

    def one_step(ev=None):
        flush_l2()
        if ev is not None:
            ev[0].record(stream)
        g_pre.replay()
        if ev is not None:
            ev[1].record(stream)
        g_gemm.replay()
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        one_step()
    torch.cuda.synchronize()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        one_step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    step_ms = np.array([e[0].elapsed_time(e[2]) for e in evs])
    gemm_ms = np.array([e[1].elapsed_time(e[2]) for e in evs])
    total_ms = max_over_ranks(float(step_ms.sum()), world)
    ops = layer.gemm_ops()
    value = world * K * ops / (total_ms * 1e-3) / 1e12
    gemm_tops = ops / (float(gemm_ms.mean()) * 1e-3) / 1e12
    if int(layer.flags.item()) != 0:
        raise RuntimeError(f"device flags raised during the timed steps: {int(layer.flags.item())}")

    # each kernel alone, L2 flushed before it: its HBM roofline fraction
    nbytes = layer.algorithmic_bytes()
    sbytes = layer.storage_bytes()
    hbm = float(peaks["hbm_gbs"])
    iso = {}
    reps = 20
    for name, _, fn in stages:
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in e:
            flush_l2()
            # hold the stream for ~0.5 ms so the host has enqueued the
            # kernel before the start event fires (no host gap is timed;
            # with a 50 us hold the X-absmax figure ran 9 us above the
            # profiler's time for the same launch)
            torch.cuda._sleep(1000000)
            a.record(stream)
            fn(st)
            b.record(stream)
        torch.cuda.synchronize()
        # the mean, not the median: event timestamps on this GPU come in
        # steps of about 2 us, and the mean of many samples with a random
        # phase is unbiased where the median stays on a step
        us = float(np.mean([a.elapsed_time(b) for a, b in e])) * 1e3
        gbs = nbytes[name] / (us * 1e-6) / 1e9
        iso[name] = {"us": round(us, 3), "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)}
        if sbytes[name] != nbytes[name]:  # codes stored as bf16: the bytes actually moved
            iso[name]["storage_gbs"] = round(sbytes[name] / (us * 1e-6) / 1e9, 1)
    iso["gemm"]["tops"] = round(ops / (iso["gemm"]["us"] * 1e-6) / 1e12, 2)
    act_stage = {"dynamic": "quant_act", "static": "quant_act_static",
                 "norm": "rmsnorm_quant_act"}[args.act_scale]

    bf16_peak = float(peaks["bf16_tflops"])
    if layer.codes == "bf16" or layer.tokens > pipeline.I8_TENSOR_MIN_TOKENS:
        if layer.codes == "bf16":
            kern, what = "k_gemm_bf16c", "tcgen05 kind::f16 on bf16-coded int8"
        elif not layer.gemm_workspace:
            kern, what = "k_gemm_i8c", "int8 codes widened to fp16 on chip, tcgen05 kind::f16"
        else:
            # the timed GEMM call is two kernels: k_widen_codes (the codes to
            # fp16 in the workspace, ~23 us here) and the fp16 form of the GEMM
            kern, what = "k_gemm_bf16c<fp16>", ("int8 codes widened to fp16 by k_widen_codes, "
                                                 "then tcgen05 kind::f16; both kernels timed")
        roofline = {"bound": "tensor", "achieved": gemm_tops, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": gemm_tops / bf16_peak,
                    "traffic": NCU_TRAFFIC_BYTES.get((kern, case.name)),
                    "kernel": f"{kern} (sq_w8a8_gemm, {what})",
                    "peak_source": f"bf16 dense burst, {peaks_kind} (fp16 runs at the same rate)"}
    else:
        if layer.tokens <= 16:
            kern, what = "k_gemm_dec", "weight-streaming decode kernel, mma.sync f16 on widened codes"
        else:
            kern, what = "k_gemm_i8_mma", "mma.sync s8"
        gbs = nbytes["gemm"] / (float(gemm_ms.mean()) * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": NCU_TRAFFIC_BYTES.get((kern, case.name)),
                    "kernel": f"{kern} (sq_w8a8_gemm, {what})",
                    "peak_source": f"HBM copy, {peaks_kind}"}
    launches = layer.kernel_count() * K
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": dict(workload_config(case, layer.codes), act_scale=args.act_scale,
                       **({"i8_gemm": args.i8_gemm}
                          if layer.codes == "i8" and layer.tokens > pipeline.I8_TENSOR_MIN_TOKENS else {})),
        "gemm_tops": gemm_tops,
        "act_quant_gbs": iso[act_stage]["gbs"],
        "act_quant_hbm_frac": iso[act_stage]["hbm_frac"],
        "stages_isolated": iso,
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clocks,
        "parallelism": f"replicas x{world}",
    }
    if not args.no_e2e:
        if args.act_scale == "dynamic":
            layers = [layer, pipeline.Layer.for_case(case, codes=layer.codes,
                                                     gemm_workspace=layer.gemm_workspace)]
            line["e2e"] = run_e2e(layers, x_host, w_host, args.e2e_steps, ops, world, torch)
    if rank == 0 and not args.no_cpu_baseline:
        nt = min(case.tokens, 256)
        times, o_ops, cores = time_oracle(case.name, 20.0, nt, 3)
        t1, _, _ = time_oracle(case.name, 20.0, nt, 2, threads=1)
        line["cpu_baseline"] = {"value": o_ops * len(times) / sum(times) / 1e12, "unit": "TOPS",
                                "cores": cores, "kind": "oracle",
                                "value_one_thread": o_ops * len(t1) / sum(t1) / 1e12,
                                "sample": f"whole path on the first {nt} tokens with the full "
                                          f"{case.cin}x{case.cout} weight, {len(times)} runs on "
                                          f"{cores} BLAS threads ({len(t1)} on one)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def gpu_local_cpus(torch, device):
    """The CPUs of the GPU's NUMA node (from sysfs) that this process may
    use, or None when that cannot be read."""
    try:
        p = torch.cuda.get_device_properties(device)
        path = (f"/sys/bus/pci/devices/{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:"
                f"{p.pci_device_id:02x}.0/local_cpulist")
        cpus = set()
        for part in open(path).read().strip().split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except (OSError, ValueError, AttributeError):
        return None


def run_e2e(layers, x_host, w_host, steps, ops, world, torch):
    """Same metric through the C ABI with host buffers: every step is one
    sq_linear_host call (X and W copied in from pinned host memory, the whole
    path, Y copied out to pinned host memory).  Steps alternate between two
    streams, each with its own device buffers and host Y, so one step's
    copies overlap the other step's copies in the opposite direction and its
    kernels."""
    # page-locked host buffers on the GPU's NUMA node: the pages are placed
    # where the pinning thread runs, and copies from a far node were measured
    # at less than half the near node's rate
    local = gpu_local_cpus(torch, torch.cuda.current_device())
    saved = os.sched_getaffinity(0)
    if local:
        os.sched_setaffinity(0, local)
    xh, wh = x_host.pin_memory(), w_host.pin_memory()
    yh = [torch.empty(layers[0].y.shape, dtype=torch.bfloat16).pin_memory() for _ in layers]
    streams = [torch.cuda.Stream() for _ in layers]
    bufs = [lay.linear_buffers() for lay in layers]

    def step(i):
        j = i % len(layers)
        layers[j].run_host(xh, wh, yh[j], stream=streams[j], bufs=bufs[j])

    for i in range(2 * len(layers)):
        step(i)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(main)
    for st in streams:
        st.wait_event(e0)
    for i in range(steps):
        step(i)
    for st in streams:
        main.wait_stream(st)
    e1.record(main)
    torch.cuda.synchronize()
    for lay in layers:
        if int(lay.flags.item()) != 0:
            raise RuntimeError(f"device flags raised during the end-to-end steps: {int(lay.flags.item())}")
    if local:
        os.sched_setaffinity(0, saved)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    return {"value": world * steps * ops / (ms * 1e-3) / 1e12, "unit": "TOPS",
            "host_buffers": ("page-locked, on the GPU's NUMA node" if local else "page-locked"),
            "h2d_bytes_per_step": xh.numel() * xh.element_size() + wh.numel() * wh.element_size(),
            "d2h_bytes_per_step": yh[0].numel() * yh[0].element_size(),
            "api": "sq_linear_host (C ABI, host buffers), two streams alternating"}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args, args.workload)
    return run_ours(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
