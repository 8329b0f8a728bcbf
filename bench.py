"""NVFP4 GEMM benchmark on GB300.

Headline workload: the square NVFP4 linear layer y = x . W^T, M = N = K = 8192
(x ~ N(0,1) with 0.1% outliers x20, W ~ N(0, 0.02), both quantised per 16-K
block to E2M1 + E4M3 scales + an FP32 global scale), bf16 output. One step is one
nvfp4_gemm call on operands already resident in HBM; the timed loop rotates over
4 distinct input/output sets (302 MB of operands > the 129 MB L2). The pages
exclude quantisation from their GEMM timings ("Blackwell NVFP4 GEMM" case page,
What is this?), so does the headline; the quantiser is timed on its own in the
breakdown, next to the decode, MoE-grouped and prefill workloads.

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle instead
(bounded row samples of the same workload on the host cores).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM TFLOPS & % of GB300 dense FP4 peak; decode/grouped weight GB/s vs HBM"
WORKLOAD = "square NVFP4 linear M=N=K=8192 (x N(0,1)+0.1% x20, W N(0,0.02)), bf16 out"
SQ = 8192
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio (fp4 13.5 PF vs bf16 2.25 PF)
NOMINAL_FP4_TFLOPS = 13500.0  # GB300 dense FP4, vendor figure
NOMINAL_HBM_GBS = 8000.0      # ~8 TB/s HBM3e
MIN_CLOCK_SAMPLES = 20        # a median clock from fewer samples is flagged


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sustained-seconds", type=float, default=3.0)
    ap.add_argument("--only", choices=["square", "decode", "moe", "prefill", "tiny", "sparse"], default=None,
                    help="run only this breakdown workload (for profiling) and print its numbers")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            def pick(keys):
                for k in keys:
                    if k in d and isinstance(d[k], (int, float)):
                        return float(d[k])
                return None
            hbm = pick(["hbm_gbs", "hbm_GBs"])
            bf16 = pick(["bf16_tflops"])
            bf16s = pick(["bf16_tflops_sustained"])
            if hbm and bf16:
                return {"hbm": hbm, "bf16": bf16, "bf16_sustained": bf16s or bf16, "source": "measured"}
        except Exception:
            pass
    return {"hbm": FALLBACK_HBM_GBS, "bf16": FALLBACK_BF16_TFLOPS, "bf16_sustained": 1700.0,
            "source": "fallback"}


class NvmlSampler:
    """SM clock and clock-event (throttle) reasons of this process's GPU, read through
    NVML every 2 ms by a background thread while running (read-only queries)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        import threading
        self.ct, self.threading = ctypes, threading
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        import torch
        props = torch.cuda.get_device_properties(torch_device)
        ok = False
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            ok = self.nvml.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(self.h)) == 0
        if not ok and hasattr(props, "pci_bus_id"):
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            ok = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        if not ok:
            raise RuntimeError("no NVML handle for this device")
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples, self.reason_bits, self.stop_flag, self.thread = [], 0, False, None
        self.period_s = 0.0002

    def _run(self):
        ct = self.ct
        mhz, bits = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag:
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if self.reasons_fn(self.h, ct.byref(bits)) == 0:
                self.reason_bits |= bits.value
            time.sleep(self.period_s)

    def start(self):
        self.thread = self.threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag = True
        self.thread.join()
        smax = self.ct.c_uint()
        self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(smax))
        reasons = sorted(n for b, n in self.REASONS.items() if self.reason_bits & b)
        n = len(self.samples)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": smax.value or None, "reasons": reasons, "samples": n,
                "sampler": f"nvml, every {self.period_s * 1e3:g} ms", "few_samples": n < MIN_CLOCK_SAMPLES}


def clock_sampler(torch_device, index):
    try:
        return NvmlSampler(torch_device)
    except Exception:
        return ClockSampler(index)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"nvfp4_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0, "sampler": "none", "few_samples": True}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        busy = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm), "sampler": "nvidia-smi, every 100 ms",
                "few_samples": len(sm) < MIN_CLOCK_SAMPLES}


# Sources each profiled kernel is built from: a recorded DRAM traffic figure stays valid
# only while these files are unchanged.
KERNEL_SOURCES = {
    "k_gemm_dense_pair": ["gemm_dense.cu", "ptx.cuh", "kernels.h"],
}


def kernel_src_hash(kernel: str):
    h = hashlib.sha256()
    d = os.path.join(ROOT, "moe_nvfp4_gemm_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json), if it
    was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent or ent.get("src_hash") != kernel_src_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------------------------
# CPU oracle arm


def cpu_oracle_gemm_rate(target_s: float):
    """Times the float64 oracle on a bounded row sample of the square workload."""
    import oracle
    import synth
    K = SQ
    MX = 2048
    x = synth.normal_bf16((MX, K), 2 * 1, 1.0, 1e-3)
    w = synth.normal_bf16((SQ, K), 2 * 1 + 1, 0.02)
    qa, sfa, ga = oracle.quantize(x)
    qb, sfb, gb = oracle.quantize(w)
    nt = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.gemm(qa, sfa, ga, qb, sfb, gb, MX, SQ, K, rows=list(range(nt)))
    t1 = (time.perf_counter() - t0) / nt  # seconds per row with all threads busy
    rows = int(max(nt, min(MX, target_s / max(t1, 1e-6))))
    t0 = time.perf_counter()
    oracle.gemm(qa, sfa, ga, qb, sfb, gb, MX, SQ, K, rows=list(range(rows)))
    dt = time.perf_counter() - t0
    tflops = 2.0 * rows * SQ * K / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} full output rows of the 8192^3 GEMM ({rows}x8192 outputs, K=8192), "
                      f"{dt:.1f} s"}


def run_reference(args):
    rank, local, world = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    K = SQ
    rows_per_step = oracle.num_threads()  # one output row per host thread per step
    MX = 4 * rows_per_step
    x = synth.normal_bf16((MX, K), 2, 1.0, 1e-3)
    w = synth.normal_bf16((SQ, K), 3, 0.02)
    qa, sfa, ga = oracle.quantize(x)
    qb, sfb, gb = oracle.quantize(w)
    sample = lambda i: [((i % 4) * rows_per_step + r) for r in range(rows_per_step)]
    for i in range(args.warmup):
        oracle.gemm(qa, sfa, ga, qb, sfb, gb, MX, SQ, K, rows=sample(i))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm(qa, sfa, ga, qb, sfb, gb, MX, SQ, K, rows=sample(i))
    dt = time.perf_counter() - t0
    tflops = 2.0 * rows_per_step * SQ * K * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "sample": f"{rows_per_step} output rows (x 8192 outputs, K=8192) per step"},
            "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{rows_per_step} output rows of the square GEMM per step"},
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# GPU arm


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import moe_nvfp4_gemm_gb300 as m
    import synth

    dev = torch.device("cuda", local)
    if args.only and args.only != "square":
        stream = torch.cuda.current_stream()
        peaks = load_peaks()

        def to_dev_only(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)

        def quantize_only(bf16_dev):
            amax, g = m.nvfp4_amax(bf16_dev)
            q, sf = m.nvfp4_quantize(bf16_dev, g)
            return q, sf, g

        out = run_breakdown(m, synth, dev, stream, to_dev_only, quantize_only, peaks,
                            peaks["bf16"] * FP4_OVER_BF16, only=args.only)
        print(json.dumps({"only": args.only, "breakdown": out}), flush=True)
        return
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    fp4_peak = peaks["bf16"] * FP4_OVER_BF16  # TFLOP/s

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    def quantize_dev(bf16_dev):
        amax, g = m.nvfp4_amax(bf16_dev)
        q, sf = m.nvfp4_quantize(bf16_dev, g)
        return q, sf, g

    # ---- square workload: 4 rotating sets --------------------------------------------------
    xb, wb = synth.dense_inputs(SQ, SQ, SQ, 1, 1.0, 1e-3, 0.02)
    xa, sfa, ga = quantize_dev(to_dev(xb))
    wq, sfb, gb = quantize_dev(to_dev(wb))
    del xb, wb
    R = 4
    sets = [(xa.clone(), sfa.clone(), ga.clone(), wq.clone(), sfb.clone(), gb.clone(),
             torch.empty((SQ, SQ), dtype=torch.bfloat16, device=dev)) for _ in range(R)]
    op_bytes = sum(t.numel() * t.element_size() for t in sets[0][:6])
    flops = 2.0 * SQ ** 3

    def gemm(i):
        a, sa, g1, b, sb, g2, y = sets[i % R]
        m.nvfp4_gemm(a, sa, g1, b, sb, g2, SQ, SQ, SQ, y=y)
        return m.nvfp4_last_launch_count()

    sampler = clock_sampler(dev, local)
    for i in range(args.warmup):
        gemm(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    torch.cuda.synchronize()
    sampler.start()
    t_all0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        launches += gemm(i)
        ends[i].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_all0.elapsed_time(t_all1)
    total_ms = reduce_max_over_ranks(total_ms, world, dev)
    per_launch_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms_per_step = total_ms / args.steps
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    if args.only == "square":
        print(json.dumps({"only": "square", "TFLOP/s": value, "per_launch_us": per_launch_ms * 1e3,
                          "clocks": clocks}), flush=True)
        return

    # ---- end to end through the C ABI with host buffers ------------------------------------
    # Every step copies its inputs in from pinned host memory and its result out to pinned
    # host memory. Serial (the reported value): copy in, GEMM, copy out on one stream.
    # Pipelined (reported beside it): two buffer sets, the copies in on one stream, the
    # GEMMs on the launching stream, the copies out on a third, so step i's GEMM overlaps
    # step i+1's copy in and step i-1's copy out; its throughput has varied by 2x between
    # runs (host copies in both directions at once), so it does not stand for the value.
    host_in = [t.cpu().pin_memory() for t in sets[0][:6]]
    host_out = [torch.empty((SQ, SQ), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dev_in = [[t.clone() for t in sets[0][:6]] for _ in range(2)]
    y_e2e = [torch.empty((SQ, SQ), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_steps = max(4, min(args.steps, 20))

    def e2e_serial(n):
        for _ in range(n):
            for d, h in zip(dev_in[0], host_in):
                d.copy_(h, non_blocking=True)
            m.nvfp4_gemm(*dev_in[0], SQ, SQ, SQ, y=y_e2e[0])
            host_out[0].copy_(y_e2e[0], non_blocking=True)

    def e2e_pipelined(n):
        landed = [torch.cuda.Event() for _ in range(n)]
        computed = [torch.cuda.Event() for _ in range(n)]
        copied_out = [torch.cuda.Event() for _ in range(n)]
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[i - 2])  # buffer set b is free again
                for d, h in zip(dev_in[b], host_in):
                    d.copy_(h, non_blocking=True)
                landed[i].record(s_in)
            stream.wait_event(landed[i])
            if i >= 2:
                stream.wait_event(copied_out[i - 2])  # y[b] has left the device
            m.nvfp4_gemm(*dev_in[b], SQ, SQ, SQ, y=y_e2e[b], stream=stream)
            computed[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                host_out[b].copy_(y_e2e[b], non_blocking=True)
                copied_out[i].record(s_out)
        stream.wait_event(copied_out[n - 1])
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)

    def timed_e2e(fn):
        fn(2)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        return reduce_max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    e2e_serial_ms = timed_e2e(e2e_serial)
    e2e_ms = timed_e2e(e2e_pipelined)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    sustained = None
    if args.sustained_seconds > 0 and not args.no_breakdown:
        sustained = run_sustained(m, dev, stream, gemm, peaks["bf16_sustained"] * FP4_OVER_BF16,
                                  args.sustained_seconds, local)

    # ---- breakdown of the other workloads ---------------------------------------------------
    breakdown = {}
    if not args.no_breakdown and rank == 0:
        del sets, dev_in, host_in, host_out, y_e2e
        torch.cuda.empty_cache()
        breakdown = run_breakdown(m, synth, dev, stream, to_dev, quantize_dev, peaks, fp4_peak)

    achieved = flops / (per_launch_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": SQ, "N": SQ, "K": SQ,
                   "l2": f"rotating {R} input/output sets ({R * op_bytes / 1e6:.0f} MB of operands > 129 MB L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp4_peak, "traffic": profiled_traffic("k_gemm_dense_pair"),
                     "kernel": "k_gemm_dense_pair",
                     "peak_source": f"{peaks['source']} bf16 {peaks['bf16']:.0f} TFLOP/s x {FP4_OVER_BF16:g} (nominal fp4/bf16)",
                     "frac_vs_nominal_13p5PF": achieved / NOMINAL_FP4_TFLOPS},
        "sustained": sustained,
        "e2e": {"value": flops / (e2e_serial_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_serial_ms,
                "pipelined_value": flops / (e2e_ms * 1e-3) / 1e12,
                "pipelined": "2 buffer sets; copies in, GEMMs and copies out on three streams"},
        "gpu_launches": launches,
        "clocks": clocks,
        "breakdown": breakdown,
    }
    if rank == 0 and world == 1 or rank == 0:
        try:
            line["cpu_baseline"] = cpu_oracle_gemm_rate(args.cpu_seconds) if world == 1 else None
            if line["cpu_baseline"] is not None:
                line["cpu_baseline"]["tiny"] = cpu_oracle_tiny()
        except Exception as ex:  # the baseline is reported, never required
            line["cpu_baseline"] = {"error": str(ex)}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def time_launches(fn, n, stream, warm=3):
    """Median device time (ms) of fn() over n launches, CUDA events on the launching stream."""
    import torch
    for i in range(warm):
        fn(i)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(ev):
        a.record(stream)
        fn(i)
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def time_graph(fn, calls, reps, stream, trials=3):
    """Device time (ms) per fn() call: `calls` calls captured in one CUDA graph, replayed
    `reps` times between two events (host launch overhead excluded); the median of
    `trials` such loops, so that one loop whose replays the host enqueued late (the
    events then time an idle GPU) does not decide the figure."""
    import torch
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(calls):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    per_call = []
    for _ in range(trials):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        per_call.append(a.elapsed_time(b) / (calls * reps))
    return statistics.median(per_call)


def run_breakdown(m, synth, dev, stream, to_dev, quantize_dev, peaks, fp4_peak, only=None):
    import torch
    out = {}
    hbm = peaks["hbm"]
    if only in (None, "decode"):
        run_decode(m, synth, dev, stream, to_dev, quantize_dev, hbm, out)
        run_decode_batched(m, synth, dev, stream, to_dev, quantize_dev, hbm, out)
    if only in (None, "decode", "sparse"):
        run_decode_sparse(m, synth, dev, stream, to_dev, hbm, out)
    if only in (None, "moe"):
        run_moe(m, synth, dev, stream, to_dev, quantize_dev, hbm, out)
    if only in (None, "moe", "sparse"):
        run_moe_sparse(m, synth, dev, stream, to_dev, hbm, out)
    if only in (None, "prefill"):
        run_prefill(m, synth, dev, stream, to_dev, quantize_dev, hbm, fp4_peak, out)
    if only in (None, "tiny"):
        run_tiny(m, synth, dev, stream, to_dev, quantize_dev, out)
    return out


def run_decode(m, synth, dev, stream, to_dev, quantize_dev, hbm, out):
    import torch
    # decode: M in {1, 16, 32}, N = K = 8192; 8 rotating weight copies (302 MB > L2)
    w_bits = synth.normal_bf16((SQ, SQ), 2 * 2 + 1, 0.02)
    wq, sfw, gw = quantize_dev(to_dev(w_bits))
    del w_bits
    copies = [(wq.clone(), sfw.clone()) for _ in range(8)]
    wbytes = wq.numel() + sfw.numel()
    for M in (1, 16, 32):
        x = synth.normal_bf16((M, SQ), 2 * 2, 1.0, 1e-3)
        xa, sfa, ga = quantize_dev(to_dev(x))
        y = torch.empty((M, SQ), dtype=torch.bfloat16, device=dev)
        fn = lambda i: m.nvfp4_gemm(xa, sfa, ga, copies[i % 8][0], copies[i % 8][1], gw, M, SQ, SQ, y=y)
        ms = time_graph(fn, 16, 20, stream)  # library default: set-up-only programmatic launch
        ms_eager = time_launches(fn, 100, stream)
        m.nvfp4_tune(m.NVFP4_TUNE_PDL, 1)
        ms_pdl = time_graph(fn, 16, 20, stream)
        m.nvfp4_tune(m.NVFP4_TUNE_PDL, -1)
        ms_plain = time_graph(fn, 16, 20, stream)
        m.nvfp4_tune(m.NVFP4_TUNE_PDL, 0)
        gbs = wbytes / (ms * 1e-3) / 1e9
        gbs_pdl = wbytes / (ms_pdl * 1e-3) / 1e9
        out[f"decode_M{M}"] = {"us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm,
                               "hbm_frac_vs_8TBps": gbs / NOMINAL_HBM_GBS,
                               "bytes": wbytes, "timing": "CUDA graph of 16 calls over 8 weight copies",
                               "us_eager_per_launch_events": ms_eager * 1e3,
                               "us_pdl": ms_pdl * 1e3, "weight_GBps_pdl": gbs_pdl,
                               "hbm_frac_pdl": gbs_pdl / hbm,
                               "pdl_note": "us: default (set-up overlaps the previous call, always ordered); "
                                           "us_pdl: weights also requested before the wait (static weights); "
                                           "us_plain_stream_order: no overlap",
                               "us_plain_stream_order": ms_plain * 1e3}
        if M in (1, 16):
            # L2 retention: one hot weight (the original matrix) called between four calls on
            # the rotating copies (151 MB streamed per step); hot-call time = step - cold-only step
            def step(i, keep):
                if keep is not None:
                    m.nvfp4_tune(m.NVFP4_TUNE_WEIGHT_L2, keep)
                    m.nvfp4_gemm(xa, sfa, ga, wq, sfw, gw, M, SQ, SQ, y=y)
                m.nvfp4_tune(m.NVFP4_TUNE_WEIGHT_L2, 0)
                for j in range(4):
                    c = copies[(4 * i + j) % 8]
                    m.nvfp4_gemm(xa, sfa, ga, c[0], c[1], gw, M, SQ, SQ, y=y)
            ms_cold = time_graph(lambda i: step(i, None), 8, 20, stream)
            ms_streamed = time_graph(lambda i: step(i, 0), 8, 20, stream) - ms_cold
            ms_kept = time_graph(lambda i: step(i, 1), 8, 20, stream) - ms_cold
            out[f"decode_l2_kept_M{M}"] = {
                "us_hot_call_kept": ms_kept * 1e3, "us_hot_call_streamed": ms_streamed * 1e3,
                "us_cold_step": ms_cold * 1e3,
                "timing": "CUDA graph of 8 steps; a step = hot-weight call + 4 calls on rotating copies; "
                          "hot-call time = step time - cold-only step time",
                "note": "kept: hot weight loaded L2 evict_last (NVFP4_TUNE_WEIGHT_L2=1), cold ones evict_first"}
    del copies, wq, sfw


def run_decode_batched(m, synth, dev, stream, to_dev, quantize_dev, hbm, out):
    """Eight independent decode GEMMs (N = K = 8192, M rows each, their own inputs and
    outputs) in one nvfp4_gemm_batched launch; two rotating sets of eight weight copies
    (604 MB > L2); graph of 6 launches. GB/s of the eight matrices' packed weights + scales."""
    import torch
    E = 8
    w_bits = synth.normal_bf16((SQ, SQ), 2 * 2 + 1, 0.02)
    wq, sfw, gw = quantize_dev(to_dev(w_bits))
    del w_bits
    copies = [(wq.clone(), sfw.clone()) for _ in range(2 * E)]
    wbytes = E * (wq.numel() + sfw.numel())
    for M in (1, 16, 32):
        xs = [quantize_dev(to_dev(synth.normal_bf16((M, SQ), 2 * 2 + 100 + e, 1.0, 1e-3))) for e in range(E)]
        ys = [torch.empty((M, SQ), dtype=torch.bfloat16, device=dev) for _ in range(E)]
        fn = lambda i: m.nvfp4_gemm_batched([(xs[e][0], xs[e][1], xs[e][2], copies[(i % 2) * E + e][0],
                                              copies[(i % 2) * E + e][1], gw, ys[e]) for e in range(E)], M)
        ms = time_graph(fn, 6, 10, stream)
        gbs = wbytes / (ms * 1e-3) / 1e9
        single = out.get(f"decode_M{M}")
        out[f"decode_batched_M{M}"] = {
            "us": ms * 1e3, "us_per_matrix": ms * 1e3 / E, "weight_GBps": gbs, "hbm_frac": gbs / hbm,
            "hbm_frac_vs_8TBps": gbs / NOMINAL_HBM_GBS, "bytes": wbytes, "matrices": E,
            "speedup_vs_single_calls": single["us"] * E / (ms * 1e3) if single else None,
            "timing": "CUDA graph of 6 launches over 2 sets of 8 weight copies"}
    del copies, wq, sfw


def run_decode_sparse(m, synth, dev, stream, to_dev, hbm, out):
    """Decode M = 1/16/32, N = K = 8192 with pair-wise 2:4 sparse weights: the decode
    workload's weight pruned, compressed and quantised on the GPU (values [N, K/2] as NVFP4,
    tiled metadata), activations in 32-element blocks; 8 rotating copies, graph of 16 calls."""
    import torch
    w_bits = synth.normal_bf16((SQ, SQ), 2 * 2 + 1, 0.02)
    wd = to_dev(w_bits)
    c, meta = m.nvfp4_prune_pairs(wd)
    _, g_c = m.nvfp4_amax(c)
    cq, csf = m.nvfp4_quantize(c, g_c)
    del wd, c
    scopies = [(cq.clone(), csf.clone(), meta.clone()) for _ in range(8)]
    sbytes = cq.numel() + csf.numel() + meta.numel()
    for M in (1, 16, 32):
        xd = to_dev(synth.normal_bf16((M, SQ), 2 * 2, 1.0, 1e-3))
        _, gx = m.nvfp4_amax(xd)
        xq, xsf = m.nvfp4_quantize_b32(xd, gx)
        y = torch.empty((M, SQ), dtype=torch.bfloat16, device=dev)
        fn = lambda i: m.nvfp4_sparse_gemm(xq, xsf, gx, scopies[i % 8][0], scopies[i % 8][1], scopies[i % 8][2], g_c,
                                           M, SQ, SQ, y=y)
        ms = time_graph(fn, 16, 20, stream)
        gbs = sbytes / (ms * 1e-3) / 1e9
        dense = out.get(f"decode_M{M}")
        out[f"decode_sparse_M{M}"] = {
            "us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm, "bytes": sbytes,
            "bytes_dense": 37748736, "speedup_vs_dense": dense["us"] / (ms * 1e3) if dense else None,
            "format": "pair-wise 2:4 (2 of 4 pairs per 8 K): values [N, K/2] NVFP4 + 4-bit metadata per 8 K; "
                      "activations in 32-element blocks",
            "timing": "CUDA graph of 16 calls over 8 weight copies"}
    del scopies, cq, csf, meta




def run_moe(m, synth, dev, stream, to_dev, quantize_dev, hbm, out):
    import torch
    # MoE grouped: 256 experts, 512 tokens top-8 (~16 rows/expert), K = 6144, N = 4096;
    # the same weights then routed with Zipf(1) expert popularity (skewed variant)
    E, N, K = 256, 4096, 6144
    a_rows, off, tok = synth.moe_tokens(512, E, 8, K, 3)
    Mt = int(off[-1])
    qa, sfa, ga = quantize_dev(to_dev(a_rows))
    qb = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
    sfb_bytes = m.nvfp4_scale_bytes(N, K)
    sfb = torch.empty((E, sfb_bytes), dtype=torch.uint8, device=dev)
    gb = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        wq, ws, g = quantize_dev(to_dev(synth.moe_expert_weight(e, N, K, 3)))
        qb[e].copy_(wq)
        sfb[e].copy_(ws)
        gb[e:e + 1].copy_(g)
    off_d = to_dev(off)
    y = torch.empty((Mt, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = m.nvfp4_grouped_gemm_workspace_bytes(E, Mt, N, K)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ms = time_graph(lambda i: m.nvfp4_grouped_gemm(qa, sfa, ga, qb, sfb, gb, off_d, E, Mt, N, K,
                                                   y=y, workspace=wsp), 4, 5, stream)
    hit = int((np.diff(off) > 0).sum())
    mbytes = hit * (N * K // 2 + sfb_bytes)
    gbs = mbytes / (ms * 1e-3) / 1e9
    out["moe_grouped"] = {"us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm, "experts_hit": hit,
                          "hbm_frac_vs_8TBps": gbs / NOMINAL_HBM_GBS,
                          "bytes": mbytes, "tflops": 2.0 * Mt * N * K / (ms * 1e-3) / 1e12}
    # the same tokens quantised once (512 rows) and gathered by routed row: copied out by the
    # preparation kernel (default workspace), or fetched by the GEMM's load stage (plain-size
    # workspace)
    xq_t, sf_t, g_t = quantize_dev(to_dev(synth.normal_bf16((512, K), 2 * 3, 1.0)))
    tok_d = torch.from_numpy(np.ascontiguousarray(tok.astype(np.int32))).to(dev)
    wsg = torch.empty(m.nvfp4_grouped_gemm_gather_workspace_bytes(E, Mt, N, K), dtype=torch.uint8, device=dev)
    ms = time_graph(lambda i: m.nvfp4_grouped_gemm_gather(xq_t, sf_t, g_t, qb, sfb, gb, off_d, tok_d, E, 512, Mt,
                                                          N, K, y=y, workspace=wsg), 4, 5, stream)
    ms_ls = time_graph(lambda i: m.nvfp4_grouped_gemm_gather(xq_t, sf_t, g_t, qb, sfb, gb, off_d, tok_d, E, 512, Mt,
                                                             N, K, y=y, workspace=wsp), 4, 5, stream)
    del wsg
    gbs = mbytes / (ms * 1e-3) / 1e9
    out["moe_grouped_gather"] = {"us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm, "experts_hit": hit,
                                 "bytes": mbytes, "tokens_quantised": 512, "routed_rows": Mt,
                                 "tflops": 2.0 * Mt * N * K / (ms * 1e-3) / 1e12,
                                 "rows": "copied out by the preparation kernel",
                                 "us_load_stage_gather4": ms_ls * 1e3}
    # the same weights read as interleaved gate/up rows, SwiGLU fused into the epilogue
    y_act = torch.empty((Mt, N // 2), dtype=torch.bfloat16, device=dev)
    ms = time_graph(lambda i: m.nvfp4_grouped_gemm_swiglu(qa, sfa, ga, qb, sfb, gb, off_d, E, Mt, N, K,
                                                          y=y_act, workspace=wsp), 4, 5, stream)
    gbs = mbytes / (ms * 1e-3) / 1e9
    ms_gu = ms
    out["moe_gate_up_swiglu"] = {"us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm, "experts_hit": hit,
                                 "bytes": mbytes, "out": f"bf16 [{Mt}, {N // 2}] = silu(gate) * up",
                                 "tflops": 2.0 * Mt * N * K / (ms * 1e-3) / 1e12}
    # down projection over the same routing: the SwiGLU output (I = N / 2 = 2048) quantised on
    # the GPU (amax + block quantise), then the grouped GEMM K = 2048 -> N = 6144
    I, Nd = N // 2, 6144
    qd = torch.empty((E, Nd, I // 2), dtype=torch.uint8, device=dev)
    sd_bytes = m.nvfp4_scale_bytes(Nd, I)
    sd = torch.empty((E, sd_bytes), dtype=torch.uint8, device=dev)
    gd = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        wq, ws, g = quantize_dev(to_dev(synth.moe_expert_weight(e, Nd, I, 5)))
        qd[e].copy_(wq)
        sd[e].copy_(ws)
        gd[e:e + 1].copy_(g)
    amax_a = torch.empty(1, dtype=torch.float32, device=dev)
    g_a = torch.empty(1, dtype=torch.float32, device=dev)
    q_a = torch.empty((Mt, I // 2), dtype=torch.uint8, device=dev)
    sf_a = torch.empty(m.nvfp4_scale_bytes(Mt, I), dtype=torch.uint8, device=dev)
    aws = torch.empty(m.nvfp4_amax_workspace_bytes(Mt * I), dtype=torch.uint8, device=dev)
    y_dn = torch.empty((Mt, Nd), dtype=torch.bfloat16, device=dev)
    wsd = torch.empty(m.nvfp4_grouped_gemm_workspace_bytes(E, Mt, Nd, I), dtype=torch.uint8, device=dev)

    def act_quantize(i):
        m.nvfp4_amax(y_act, amax_a, g_a, aws)
        m.nvfp4_quantize(y_act, g_a, q_a, sf_a)

    def down(i):
        m.nvfp4_grouped_gemm(q_a, sf_a, g_a, qd, sd, gd, off_d, E, Mt, Nd, I, y=y_dn, workspace=wsd)

    def layer(i):
        m.nvfp4_grouped_gemm_swiglu(qa, sfa, ga, qb, sfb, gb, off_d, E, Mt, N, K, y=y_act, workspace=wsp)
        act_quantize(i)
        down(i)

    act_quantize(0)
    ms_q = time_graph(act_quantize, 4, 5, stream)
    ms_dn = time_graph(down, 4, 5, stream)
    ms_layer = time_graph(layer, 2, 5, stream)
    dbytes = hit * (Nd * I // 2 + sd_bytes)
    gbs = dbytes / (ms_dn * 1e-3) / 1e9
    out["moe_down"] = {"us": ms_dn * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm,
                       "hbm_frac_vs_8TBps": gbs / NOMINAL_HBM_GBS, "experts_hit": hit, "bytes": dbytes,
                       "shape": f"per expert K = {I} -> N = {Nd}, {Mt} routed rows",
                       "tflops": 2.0 * Mt * Nd * I / (ms_dn * 1e-3) / 1e12,
                       "act_amax_quantize_us": ms_q * 1e3,
                       "layer_us": ms_layer * 1e3,
                       "layer": "gate/up + SwiGLU, amax + quantise of the activation, down projection (one graph)",
                       "layer_weight_GBps": (mbytes + dbytes) / (ms_layer * 1e-3) / 1e9,
                       "layer_hbm_frac": (mbytes + dbytes) / (ms_layer * 1e-3) / 1e9 / hbm}

    # The same layer with the gate/up epilogue emitting NVFP4 for the down projection, the
    # activation's global scale given (calibrated once: the value the amax above produced).
    def gate_up_nvfp4(i):
        m.nvfp4_grouped_gemm_swiglu_quantize_out(qa, sfa, ga, qb, sfb, gb, off_d, E, Mt, N, K, g_a, q_out=q_a,
                                                 sf_out=sf_a, workspace=wsp)

    def layer_nvfp4(i):
        gate_up_nvfp4(i)
        down(i)

    ms_guq = time_graph(gate_up_nvfp4, 4, 5, stream)
    ms_layer_q = time_graph(layer_nvfp4, 2, 5, stream)
    out["moe_layer_nvfp4_act"] = {
        "gate_up_swiglu_nvfp4_us": ms_guq * 1e3,
        "gate_up_swiglu_nvfp4_hbm_frac": mbytes / (ms_guq * 1e-3) / 1e9 / hbm,
        "layer_us": ms_layer_q * 1e3,
        "layer_weight_GBps": (mbytes + dbytes) / (ms_layer_q * 1e-3) / 1e9,
        "layer_hbm_frac": (mbytes + dbytes) / (ms_layer_q * 1e-3) / 1e9 / hbm,
        "layer": "gate/up + SwiGLU emitting NVFP4 (given activation scale), down projection (one graph)"}
    del y_act, qd, sd, y_dn
    a_s, off_s, _ = synth.moe_tokens(512, E, 8, K, 3, zipf_s=1.0)
    qs, sfs, gs = quantize_dev(to_dev(a_s))
    off_sd = to_dev(off_s)
    ms = time_graph(lambda i: m.nvfp4_grouped_gemm(qs, sfs, gs, qb, sfb, gb, off_sd, E, Mt, N, K,
                                                   y=y, workspace=wsp), 4, 5, stream)
    hit = int((np.diff(off_s) > 0).sum())
    mbytes = hit * (N * K // 2 + sfb_bytes)
    gbs = mbytes / (ms * 1e-3) / 1e9
    out["moe_grouped_skewed"] = {"us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm, "experts_hit": hit,
                                 "hbm_frac_vs_8TBps": gbs / NOMINAL_HBM_GBS,
                                 "max_rows_per_expert": int(np.diff(off_s).max()), "routing": "Zipf(1) popularity",
                                 "bytes": mbytes, "tflops": 2.0 * Mt * N * K / (ms * 1e-3) / 1e12}
    del qb, sfb, wsp
    torch.cuda.empty_cache()


def run_moe_sparse(m, synth, dev, stream, to_dev, hbm, out):
    """The MoE workload with pair-wise 2:4 sparse experts: each expert's weight pruned,
    compressed and quantised on the GPU, the routed rows quantised in 32-element blocks."""
    import torch
    E, N, K = 256, 4096, 6144
    a_rows, off, _ = synth.moe_tokens(512, E, 8, K, 3)
    Mt = int(off[-1])
    off_d = to_dev(off)
    hit = int((np.diff(off) > 0).sum())
    y = torch.empty((Mt, N), dtype=torch.bfloat16, device=dev)
    wsp = torch.empty(m.nvfp4_grouped_gemm_workspace_bytes(E, Mt, N, K), dtype=torch.uint8, device=dev)
    cqs = torch.empty((E, N, K // 4), dtype=torch.uint8, device=dev)
    csb = m.nvfp4_scale_bytes(N, K // 2)
    csfs = torch.empty((E, csb), dtype=torch.uint8, device=dev)
    gws = torch.empty(E, dtype=torch.float32, device=dev)
    mb = m.nvfp4_sparse_meta_bytes(N, K)
    metas = torch.empty((E, mb), dtype=torch.uint8, device=dev)
    for e in range(E):
        c, meta = m.nvfp4_prune_pairs(to_dev(synth.moe_expert_weight(e, N, K, 3)))
        _, g_c = m.nvfp4_amax(c)
        cq, csf = m.nvfp4_quantize(c, g_c)
        cqs[e].copy_(cq)
        csfs[e].copy_(csf)
        gws[e:e + 1].copy_(g_c)
        metas[e].copy_(meta)
    a_d = to_dev(a_rows)
    _, gxs = m.nvfp4_amax(a_d)
    xq32, xsf32 = m.nvfp4_quantize_b32(a_d, gxs)
    del a_d
    ms = time_graph(lambda i: m.nvfp4_grouped_sparse_gemm(xq32, xsf32, gxs, cqs, csfs, metas, gws, off_d, E, Mt, N,
                                                          K, y=y, workspace=wsp), 4, 5, stream)
    sbytes = hit * (N * K // 4 + csb + mb)
    gbs = sbytes / (ms * 1e-3) / 1e9
    out["moe_grouped_sparse"] = {"us": ms * 1e3, "weight_GBps": gbs, "hbm_frac": gbs / hbm, "experts_hit": hit,
                                 "bytes": sbytes, "bytes_dense": hit * (N * K // 2 + m.nvfp4_scale_bytes(N, K)),
                                 "speedup_vs_dense": (out["moe_grouped"]["us"] / (ms * 1e3)
                                                      if "moe_grouped" in out else None),
                                 "tflops_dense_equivalent": 2.0 * Mt * N * K / (ms * 1e-3) / 1e12,
                                 "format": "pair-wise 2:4 experts (values [N, K/2] NVFP4 + 4-bit metadata per 8 K); "
                                           "routed rows in 32-element blocks"}
    del cqs, csfs, metas, xq32, xsf32
    del y, wsp
    torch.cuda.empty_cache()


def run_prefill(m, synth, dev, stream, to_dev, quantize_dev, hbm, fp4_peak, out):
    import torch
    # prefill: quantize x (4096 x 8192) on the GPU, GEMM against pre-quantised W (28672 x 8192).
    # The quantiser and amax read their input from HBM: 4 rotating activation buffers
    # (4 x 67 MB in, 4 x 19 MB out: 344 MB > the 129 MB L2), so no call finds its input in L2.
    Mp, Np, Kp = 4096, 28672, 8192
    RQ = 4
    x0 = to_dev(synth.normal_bf16((Mp, Kp), 2 * 4, 1.0, 1e-3))
    xs = [x0] + [x0.clone() for _ in range(RQ - 1)]
    wq, sfw, gw = quantize_dev(to_dev(synth.normal_bf16((Np, Kp), 2 * 4 + 1, 0.02)))
    wcopies = [(wq, sfw), (wq.clone(), sfw.clone())]
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    qs = [torch.empty((Mp, Kp // 2), dtype=torch.uint8, device=dev) for _ in range(RQ)]
    sfs = [torch.empty(m.nvfp4_scale_bytes(Mp, Kp), dtype=torch.uint8, device=dev) for _ in range(RQ)]
    q, sf = qs[0], sfs[0]
    aws = torch.empty(m.nvfp4_amax_workspace_bytes(Mp * Kp), dtype=torch.uint8, device=dev)
    yp = torch.empty((Mp, Np), dtype=torch.bfloat16, device=dev)
    m.nvfp4_amax(x0, amax, g, aws)
    ms_q = time_graph(lambda i: m.nvfp4_quantize(xs[i % RQ], g, qs[i % RQ], sfs[i % RQ]), 12, 10, stream)
    ms_amax = time_graph(lambda i: m.nvfp4_amax(xs[i % RQ], amax, g, aws), 12, 10, stream)
    # the same calls repeated on one buffer (input resident in L2), for comparison
    ms_q_l2 = time_graph(lambda i: m.nvfp4_quantize(x0, g, q, sf), 10, 10, stream)
    ms_amax_l2 = time_graph(lambda i: m.nvfp4_amax(x0, amax, g, aws), 10, 10, stream)
    m.nvfp4_quantize(x0, g, q, sf)
    ms_g = time_launches(lambda i: m.nvfp4_gemm(q, sf, g, wcopies[i % 2][0], wcopies[i % 2][1], gw,
                                                Mp, Np, Kp, y=yp), 20, stream)

    def together(i):
        x, qq, ss = xs[i % RQ], qs[i % RQ], sfs[i % RQ]
        m.nvfp4_amax(x, amax, g, aws)
        m.nvfp4_quantize(x, g, qq, ss)
        m.nvfp4_gemm(qq, ss, g, wcopies[i % 2][0], wcopies[i % 2][1], gw, Mp, Np, Kp, y=yp)

    ms_t = time_launches(together, 20, stream)
    # layer chain: the GEMM's output as the next layer's NVFP4 input, with a given global
    # scale: quantised in the GEMM epilogue vs bf16 out + a separate quantize pass
    g_y = torch.full((1,), 2.0 ** -6, dtype=torch.float32, device=dev)
    qy = torch.empty((Mp, Np // 2), dtype=torch.uint8, device=dev)
    sfy = torch.empty(m.nvfp4_scale_bytes(Mp, Np), dtype=torch.uint8, device=dev)
    ms_gq = time_launches(lambda i: m.nvfp4_gemm_quantize_out(q, sf, g, wcopies[i % 2][0], wcopies[i % 2][1], gw,
                                                              g_y, Mp, Np, Kp, q_out=qy, sf_out=sfy), 20, stream)

    def gemm_then_quantize(i):
        m.nvfp4_gemm(q, sf, g, wcopies[i % 2][0], wcopies[i % 2][1], gw, Mp, Np, Kp, y=yp)
        m.nvfp4_quantize(yp, g_y, qy, sfy)

    ms_gtq = time_launches(gemm_then_quantize, 20, stream)
    qbytes = Mp * Kp * 2 + Mp * Kp // 2 + m.nvfp4_scale_bytes(Mp, Kp)
    abytes = Mp * Kp * 2
    gemm_tf = 2.0 * Mp * Np * Kp / (ms_g * 1e-3) / 1e12
    out["prefill"] = {
        "quantize_us": ms_q * 1e3, "quantize_GBps": qbytes / (ms_q * 1e-3) / 1e9,
        "quantize_hbm_frac": qbytes / (ms_q * 1e-3) / 1e9 / hbm,
        "quantize_hbm_frac_vs_8TBps": qbytes / (ms_q * 1e-3) / 1e9 / NOMINAL_HBM_GBS, "quantize_bytes": qbytes,
        "amax_us": ms_amax * 1e3, "amax_GBps": abytes / (ms_amax * 1e-3) / 1e9,
        "amax_hbm_frac": abytes / (ms_amax * 1e-3) / 1e9 / hbm,
        "quantize_amax_input": f"from HBM: {RQ} rotating activation buffers ({RQ * (qbytes) / 1e6:.0f} MB)",
        "quantize_us_input_in_l2": ms_q_l2 * 1e3, "amax_us_input_in_l2": ms_amax_l2 * 1e3,
        "gemm_us": ms_g * 1e3, "gemm_tflops": gemm_tf, "gemm_frac": gemm_tf / fp4_peak,
        "gemm_frac_vs_nominal_13p5PF": gemm_tf / NOMINAL_FP4_TFLOPS,
        "together_us": ms_t * 1e3,
        "together": "amax + quantize (rotating activations) + GEMM, per step",
        "gemm_nvfp4_out_us": ms_gq * 1e3, "gemm_nvfp4_out_tflops": 2.0 * Mp * Np * Kp / (ms_gq * 1e-3) / 1e12,
        "gemm_then_quantize_us": ms_gtq * 1e3}


def run_tiny(m, synth, dev, stream, to_dev, quantize_dev, out):
    """The tiny workload (128 x 128 x 256, x and W ~ N(0,1), seed 0) on the GPU: both
    operands quantised by nvfp4_quantize, then the GEMM; per-launch event times. Its
    parity is a test case; the oracle's time for it is reported with the CPU baseline."""
    import torch
    M, N, K = 128, 128, 256
    xb, wb = synth.dense_inputs(M, N, K, 0)
    xd, wd = to_dev(xb), to_dev(wb)
    ms_q = time_launches(lambda i: quantize_dev(xd), 50, stream)
    xa, sa, g1 = quantize_dev(xd)
    wa, sw, g2 = quantize_dev(wd)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ms = time_launches(lambda i: m.nvfp4_gemm(xa, sa, g1, wa, sw, g2, M, N, K, y=y), 50, stream)
    out["tiny"] = {"gpu_gemm_us": ms * 1e3, "gpu_amax_quantize_us": ms_q * 1e3,
                   "note": "128 x 128 x 256; per-launch CUDA events; oracle ms in cpu_baseline.tiny"}


def cpu_oracle_tiny():
    """The oracle on the tiny workload, in ms: quantising x and W, and the float64 GEMM."""
    import oracle
    import synth
    M, N, K = 128, 128, 256
    xb, wb = synth.dense_inputs(M, N, K, 0)
    reps = 20
    t0 = time.perf_counter()
    for _ in range(reps):
        qa, sfa, ga = oracle.quantize(xb)
        qb, sfb, gb = oracle.quantize(wb)
    tq = (time.perf_counter() - t0) / reps
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.gemm(qa, sfa, ga, qb, sfb, gb, M, N, K)
    tg = (time.perf_counter() - t0) / reps
    return {"oracle_gemm_ms": tg * 1e3, "oracle_quantize_x_and_w_ms": tq * 1e3, "cores": oracle.num_threads(),
            "workload": "tiny 128 x 128 x 256, seed 0 (float64 on the host cores)"}


def run_sustained(m, dev, stream, gemm, fp4_peak_sustained, seconds, local):
    """The headline GEMM back to back for `seconds` under the power cap (rotating input
    sets), clocks sampled throughout; TFLOP/s over the whole loop."""
    import torch
    flops = 2.0 * SQ ** 3
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(50):
        gemm(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    per = ev0.elapsed_time(ev1) / 50 * 1e-3
    n = max(100, int(seconds / per))
    sampler = clock_sampler(dev, local)
    sampler.period_s = 0.002 if isinstance(sampler, NvmlSampler) else 0.1
    sampler.start()
    ev0.record(stream)
    for i in range(n):
        gemm(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    tf = flops * n / (ms * 1e-3) / 1e12
    return {"launches": n, "seconds": ms * 1e-3, "TFLOP/s": tf, "peak_sustained": fp4_peak_sustained,
            "frac_of_sustained_peak": tf / fp4_peak_sustained, "frac_vs_nominal_13p5PF": tf / NOMINAL_FP4_TFLOPS,
            "peak_source": "measured bf16_tflops_sustained x 6 (nominal fp4/bf16)", "clocks": clocks}


if __name__ == "__main__":
    main()
