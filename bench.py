#!/usr/bin/env python
"""Benchmark of the fused quantize -> INT8 GEMM -> dequant linear layer on B300.

Workload (one "step"): the W8A8 per-channel linear layer at M = 4096 tokens,
N = 10240 outputs, K = 2560 inputs (the shape and token count of the Cider
README's operator-latency table, "Shape [N=10240, K=2560]", row M = 4096):
per-token INT8 quantization of x, the INT8 x INT8 -> INT32 product on the
tensor cores, the fused fp32 dequant to fp16. Inputs are synthetic (seeded,
N(0,1) activations with 4 outlier channels x20, N(0,0.02) weights), resident
in HBM; weight quantization is offline and untimed. Steps rotate over
independent input sets (x, weights, y) whose total exceeds 3x L2, so each
step reads its operands from HBM, as consecutive linears of a prefill do; the
same step after a 512 MiB L2-flush write is reported beside it.

Prints ONE JSON line (rank 0). `value` is whole-job TOPS (2*M*N*K per step,
all ranks); `e2e` is the same metric through the public C-ABI call with the
inputs copied from pinned host memory and the output copied back inside the
timed region (steps pipelined as a serving loop runs them: copy-in, layer and
copy-out of consecutive steps overlap on three streams); `gemv` is the M = 1 decode GEMV in HBM GB/s; `roofline` is the
dominant kernel (the tensor-core GEMM) against the measured dense bf16 peak
(fp16 has the same nominal rate); `cpu_baseline` is the CPU oracle timed on a
bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cider|reference]

With N > 1 it runs under torchrun, one process per GPU, as independent
replicas (the layer needs no exchange between GPUs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M, N, K = 4096, 10240, 2560
METRIC = "W8A8 GEMM TOPS & % INT8 peak at M=4096; M=1 INT8 GEMV HBM GB/s"
WORKLOAD = "w8a8_per_channel_linear_M4096_N10240_K2560"
FLUSH_BYTES = 512 << 20
# DRAM bytes (read + write) of one launch of the pair GEMM at this workload,
# from its ncu capture; reset to None whenever the kernel changes until it
# is captured again.
GEMM_DRAM_BYTES_PER_LAUNCH = 127.63e6  # 74.08 MB read + 53.54 MB written
# dram__bytes_read.sum + dram__bytes_write.sum of one cold gemv_kernel<8, false> launch at
# N10240 K2560 (ncu; the algorithmic bytes are 26.28 MB).
GEMV_DRAM_BYTES_PER_LAUNCH = 26.30e6


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("cider", "reference"), default="cider")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back steps for the sustained figure")
    ap.add_argument("--gemv-only", action="store_true",
                    help="run only the M = 1 GEMV leg (a small command for profilers)")
    ap.add_argument("--step-only", action="store_true",
                    help="run only the M = 4096 step (a small command for profilers)")
    ap.add_argument("--small-step", action="store_true",
                    help="run only the few-token per-channel call (M = 128: the SM-pair "
                         "few-token engine, or the single-SM one with CIDER_GEMM_ENGINE=single): "
                         "a small command for profilers")
    ap.add_argument("--layer", type=int, nargs=5, metavar=("M", "N", "K", "BITS", "GS"),
                    help="run only the public layer call of this shape (seeded inputs made "
                         "on the GPU): a small command for profilers")
    ap.add_argument("--configs", action="store_true",
                    help="time every workload of the config list (M sweeps, per-group, W4A8, "
                         "decoder layer) through the public calls; one JSON line")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave the per-config sweep out of the headline line")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1800.0, 6400.0, "fallback"


def cpu_model() -> str:
    """The host CPU's model name (for the CPU-baseline record)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, polled through
    NVML (the library nvidia-smi reads; called with ctypes, so no Python
    NVML package is needed) every 2 ms from a thread while the timed region
    runs. Reason bits are NVML's documented clocks-event-reason masks."""
    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8),
               ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40),
               ("hw_power_brake_slowdown", 0x80))
    NVML_CLOCK_SM = 1

    def __init__(self, torch_device_index: int):
        self.idx = torch_device_index
        self.samples = []
        self.error = None
        self._stop = None
        self._thread = None

    def _open(self):
        import ctypes
        import torch
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        # the PCI address is the key that survives CUDA_VISIBLE_DEVICES renumbering
        pr = torch.cuda.get_device_properties(self.idx)
        bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        h = ctypes.c_void_p()
        if nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError(f"no NVML handle for PCI {bus}")
        smax = ctypes.c_uint()
        nvml.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(smax))
        reasons_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        return nvml, h, int(smax.value), reasons_fn

    def start(self):
        import ctypes
        import threading
        try:
            nvml, h, self._smax, reasons_fn = self._open()
        except Exception as exc:  # no NVML: report why instead of clocks
            self.error = f"{type(exc).__name__}: {exc}"
            return
        self._stop = threading.Event()

        def poll():
            clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while True:
                if nvml.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0 \
                        and reasons_fn(h, ctypes.byref(rs)) == 0:
                    self.samples.append((int(clk.value), int(rs.value)))
                if self._stop.wait(0.002):
                    break

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 1.0:  # first sample before the region
            time.sleep(0.001)

    def stop(self):
        if self._thread is None:
            return {"error": self.error} if self.error else None
        self._stop.set()
        self._thread.join()
        reasons = set()
        for _, rs in self.samples:
            for name, bit in self.REASONS:
                if rs & bit:
                    reasons.add(name)
        sm = [s for s, _ in self.samples]
        if not sm:
            return {"error": "no NVML samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self._smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(info, low_frac: float = 0.9) -> bool:
    """True when a clock record disqualifies its timed region: a hardware
    or thermal slowdown was active, or the median SM clock sat below
    low_frac of the maximum with no reason active (a clock held low by
    someone else). sw_power_cap alone is kept. A missing record (no NVML)
    rejects nothing."""
    if not info or "sm_mhz" not in info:
        return False
    reasons = set(info.get("reasons", ()))
    if reasons & set(REJECT_REASONS):
        return True
    return not reasons and info["sm_mhz"] < low_frac * info["sm_max_mhz"]


def replica_max(v: float, world: int, device=None) -> float:
    """The slowest replica's time: the whole job's step time when N
    independent replicas run one per GPU (max over ranks of the process
    group; the identity for a single process)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_replica: float, seconds: float, world: int, device=None) -> float:
    """Whole-job throughput of N replicas: all ranks' work over the slowest
    rank's time (weak scaling: each replica does the same fixed work)."""
    return world * work_per_replica / replica_max(seconds, world, device)


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_tops(x_np, wq, s_w, rows: int):
    import oracle
    t0 = time.perf_counter()
    oracle.w8a8_linear(x_np[:rows], wq, s_w, 0)
    dt = time.perf_counter() - t0
    return 2.0 * rows * N * K / dt / 1e12, dt


def size_oracle_sample(x_np, wq, s_w, target_s: float) -> int:
    """Rows of the workload the oracle processes in about target_s seconds
    (calibrated on enough rows to keep every oracle thread busy)."""
    import oracle
    cal = max(16, 2 * oracle.get_threads())
    _, dt = oracle_tops(x_np, wq, s_w, cal)
    per_row = dt / cal
    return int(max(cal, min(M, target_s / max(per_row, 1e-9))))


def cpu_inputs():
    import oracle
    import synth
    li = synth.linear_inputs(M, N, K, n_out=4, seed=0)
    x_np = li.x.numpy()
    wq, s_w = oracle.quantize_weight_int8(li.w.numpy(), 0)
    return x_np, wq, s_w


def run_reference(args):
    """The CPU oracle, as it stands, on bounded samples of the workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    x_np, wq, s_w = cpu_inputs()
    per_step_target = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    rows = size_oracle_sample(x_np, wq, s_w, per_step_target)
    for _ in range(args.warmup):
        oracle_tops(x_np, wq, s_w, rows)
    times = [oracle_tops(x_np, wq, s_w, rows)[1] for _ in range(args.steps)]
    t = statistics.mean(times)
    value = 2.0 * rows * N * K / t / 1e12
    sample = f"{rows} of {M} token rows per step, full N={N}, K={K}"
    cores = oracle.get_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "mode": "per-channel",
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CUDA path
# ---------------------------------------------------------------------------

def gemv_leg(args, x, wq, s_w, y_row0, stream):
    """M = 1 decode GEMV on the workload's weights. Cold weights, as in decode
    (every other layer's weights pass through L2 between two reads of this
    one): the launches cycle through enough copies of wq that together exceed
    3x L2, so each read comes from HBM. Two measurements:
      standalone - each launch bracketed by its own events;
      sequence   - a CUDA graph of back-to-back GEMVs (one per weight copy,
                   as the linears of a decode step follow each other),
                   replayed and timed as a whole, divided by the launches.
    Returns (standalone s, sequence s, number of weight copies)."""
    import torch
    import w4a8_quantized_gemm_int8_b300 as cider
    dev = x.device
    x1 = x[0].contiguous()
    y1 = torch.empty((N,), dtype=torch.float16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_copies = (3 * l2) // (N * K) + 2
    wq_copies = [wq.clone() for _ in range(n_copies)]
    for i in range(max(args.warmup, n_copies)):
        cider.int8_gemv(x1, wq_copies[i % n_copies], s_w, 8, 0, out=y1)
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    # Keep the GPU busy while the host enqueues the timed launches, so the
    # events bracket back-to-back kernels and not host launch gaps.
    torch.cuda._sleep(int(2e5 * args.steps))
    for i, (a, b) in enumerate(gev):
        a.record(stream)
        cider.int8_gemv(x1, wq_copies[i % n_copies], s_w, 8, 0, out=y1)
        b.record(stream)
    torch.cuda.synchronize()
    if y_row0 is not None:
        assert torch.equal(y1.view(torch.int16), y_row0.view(torch.int16)), "GEMV != GEMM row"
    standalone = statistics.mean([a.elapsed_time(b) for a, b in gev]) / 1e3

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    ys = [torch.empty((N,), dtype=torch.float16, device=dev) for _ in range(n_copies)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        cider.int8_gemv(x1, wq_copies[0], s_w, 8, 0, out=ys[0])
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for i in range(n_copies):
                cider.int8_gemv(x1, wq_copies[i], s_w, 8, 0, out=ys[i])
    torch.cuda.synchronize()
    reps = max(3, args.steps // n_copies)
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    sequence = a.elapsed_time(b) / 1e3 / (reps * n_copies)
    if y_row0 is not None:
        for t in ys:
            assert torch.equal(t.view(torch.int16), y_row0.view(torch.int16)), "graph GEMV"
    # The same two measurements of a plain streaming read of the same bytes
    # (a measurement kernel launched as the GEMV is): the ceiling a GEMV of
    # this size can reach with this timing.
    sink = torch.empty(4096, dtype=torch.int32, device=dev)
    for i in range(n_copies):
        cider.read_bytes(wq_copies[i], sink)
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e5 * args.steps))
    for i, (a, b) in enumerate(rev):
        a.record(stream)
        cider.read_bytes(wq_copies[i % n_copies], sink)
        b.record(stream)
    torch.cuda.synchronize()
    read_standalone = statistics.mean([a.elapsed_time(b) for a, b in rev]) / 1e3
    rgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        cider.read_bytes(wq_copies[0], sink)
        side.synchronize()
        with torch.cuda.graph(rgraph, stream=side):
            for i in range(n_copies):
                cider.read_bytes(wq_copies[i], sink)
    torch.cuda.synchronize()
    rgraph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        rgraph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    read_sequence = a.elapsed_time(b) / 1e3 / (reps * n_copies)
    del wq_copies
    return standalone, sequence, n_copies, read_standalone, read_sequence


def gemv_sequence(args, N_, K_, dev, stream, seed=1):
    """CUDA-graph decode sequence of per-channel INT8 GEMVs of one shape over
    weight copies that together exceed 3x L2: mean time per launch (s)."""
    import torch
    import w4a8_quantized_gemm_int8_b300 as cider
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_copies = (3 * l2) // (N_ * K_) + 2
    x1 = (torch.randn(K_, generator=gen, device=dev)).half()
    ws = [torch.randint(-127, 128, (N_, K_), generator=gen, device=dev, dtype=torch.int8)
          for _ in range(n_copies)]
    s_w = torch.rand(N_, generator=gen, device=dev) * 0.01 + 1e-3
    ys = [torch.empty((N_,), dtype=torch.float16, device=dev) for _ in range(n_copies)]
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        cider.int8_gemv(x1, ws[0], s_w, 8, 0, out=ys[0])
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for i in range(n_copies):
                cider.int8_gemv(x1, ws[i], s_w, 8, 0, out=ys[i])
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    reps = max(3, args.steps // n_copies)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    del ws
    return a.elapsed_time(b) / 1e3 / (reps * n_copies), n_copies


def int8_mma_rate(dev, stream) -> float:
    """INT8 tensor rate (TOPS) of a register-only loop of the legacy
    mma.sync.m16n8k32 s8 instruction on every SM (a measurement kernel of the
    library): the "% INT8 peak" denominator (sm_103a has no integer kind of
    tcgen05.mma). Best of three timed launches."""
    import torch
    import w4a8_quantized_gemm_int8_b300 as cider
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = 8 * sms, 2048
    ops = blocks * 4 * 8 * iters * 8192
    cider.int8_mma_loop(blocks, 64)
    best = float("inf")
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        cider.int8_mma_loop(blocks, iters)
        b.record(stream)
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) / 1e3)
    return ops / best / 1e12


def config_sweep(args, check: bool):
    """Every workload shape of the operator configs, timed through the public
    calls (quant + GEMM + dequant per call; the GEMV for M = 1). Inputs are
    drawn on the GPU from a seeded generator (timing does not depend on the
    values), in sets rotated so that together they exceed 3x L2. Times are
    CUDA-event means over `steps` calls after `warmup`.

    Returns (results, samples): with `check`, samples holds, per case, a few
    token rows of x and 64 sampled output channels (their weight rows and
    scales, and the GPU's outputs there), for the CPU-baseline leg to
    recompute with the oracle (check_samples)."""
    import torch
    import w4a8_quantized_gemm_int8_b300 as cider
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    bf16_peak, hbm_peak, _ = peaks()
    samples = []

    def inputs(M, N, K, bits, gs, n_out):
        x = torch.randn(M, K, generator=gen, device=dev)
        x[:, torch.randperm(K, generator=gen, device=dev)[:n_out]] *= 20.0
        w = (torch.randn(N, K, generator=gen, device=dev) * 0.02).half()
        x = x.half()
        if bits == 8:
            wq, s = cider.quantize_weight_int8(w, gs)
        else:
            wq, s = cider.pack_weight_int4(w, gs)
        return x, wq, s

    def time_case(key, M, N, K, bits, gs, n_out=4, a16=False):
        wbytes = N * K if bits == 8 else N * K // 2
        per_set = 2 * M * K + wbytes + 2 * M * N
        n_sets = max(1, min(8, -(-3 * l2 // per_set) + 1))
        sets = []
        for _ in range(n_sets):
            x, wq, s = inputs(M, N, K, bits, gs, n_out)
            sets.append((x, wq, s, torch.empty((M, N), dtype=torch.float16, device=dev)))
        ws = torch.empty(max(1, cider.workspace_bytes(M, N, K, group_size=gs, bits=bits)),
                         dtype=torch.uint8, device=dev)

        def call(i):
            x, wq, s, y = sets[i % n_sets]
            if M == 1 and a16:
                cider.a16_gemv(x[0], wq, s, bits, gs, out=y[0])
            elif M == 1:
                cider.int8_gemv(x[0], wq, s, bits, gs, out=y[0])
            elif bits == 8:
                cider.w8a8_linear(x, wq, s, gs, out=y, ws=ws)
            else:
                cider.w4a8_linear(x, wq, s, gs, out=y, ws=ws)

        for i in range(max(args.warmup, n_sets)):
            call(i)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e5 * args.steps))
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            call(i)
            b.record(stream)
        torch.cuda.synchronize()
        t = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
        st, site = cider.device_status()
        assert st == cider.CIDER_OK, f"device status {st} at {site:#x}"
        G = 1 if gs == 0 else K // gs
        res = {"M": M, "N": N, "K": K, "bits": bits, "gs": gs, "us": round(t * 1e6, 2),
               "TOPS": round(2.0 * M * N * K / t / 1e12, 1)}
        if a16:
            res["mode"] = "a16"
        if M == 1:  # HBM-bound: algorithmic bytes over the measured copy bandwidth
            res["GB/s"] = round((wbytes + 4 * N * G + 2 * K + 2 * N) / t / 1e9, 1)
            res["frac"] = round(res["GB/s"] / hbm_peak, 3)
        else:  # tensor-bound: the whole call's flops over the measured dense f16 rate
            res["frac"] = round(res["TOPS"] / bf16_peak, 3)
        if check:
            # the last call's set: rows first, middle, last; 64 seeded channels
            x, wq, s, y = sets[(max(args.warmup, n_sets) + args.steps - 1) % n_sets]
            rows = sorted({0, M // 2, M - 1})
            cols = torch.randperm(N, generator=gen, device=dev)[:min(64, N)].sort().values
            samples.append({"key": key, "case": res, "a16": a16, "bits": bits, "gs": gs,
                            "x": x[rows].cpu(), "w": wq[cols].cpu(), "s": s[cols].cpu(),
                            "y": y[rows][:, cols].cpu()})
        del sets, ws
        return res

    out = {"per_channel_N10240_K2560": [time_case("per_channel_N10240_K2560", m, 10240, 2560,
                                                  8, 0) for m in (1, 128, 1024, 4096, 8192)]}
    for gs in (64, 128):
        key = f"per_group{gs}_N2560_K10240"
        out[key] = [time_case(key, m, 2560, 10240, 8, gs) for m in (1, 128, 1024, 4096, 8192)]
    for (n, k) in ((10240, 2560), (2560, 10240)):
        key = f"w4a8_gs128_N{n}_K{k}"
        out[key] = [time_case(key, m, n, k, 4, 128) for m in (1, 1024, 8192)]
    # The A16 decode product (activations unquantized, weights dequantized).
    out["a16_decode_M1"] = [time_case("a16_decode_M1", 1, n, k, b, g, a16=True)
                            for (n, k, b, g) in ((10240, 2560, 8, 0), (2560, 10240, 8, 64),
                                                 (10240, 2560, 4, 128))]
    import synth
    layer = []
    for name, K_, N_ in synth.DECODER_LAYER:
        r = time_case("decoder_layer", 2048, N_, K_, 8, 0, n_out=max(1, round(K_ * 0.01)))
        r["linear"] = name
        layer.append(r)
    tot_us = sum(r["us"] for r in layer)
    tot_ops = sum(2.0 * r["M"] * r["N"] * r["K"] for r in layer)
    # The same layer with the linears that share an input fused into one call
    # each (weights concatenated along N at prep time): q|k|v and gate|up.
    fused = []
    for name, K_, N_ in (("qkv", 4096, 6144), ("o", 4096, 4096), ("gate_up", 4096, 24576),
                         ("down", 12288, 4096)):
        r = time_case("decoder_layer_fused", 2048, N_, K_, 8, 0, n_out=max(1, round(K_ * 0.01)))
        r["linear"] = name
        fused.append(r)
    fused_us = sum(r["us"] for r in fused)
    out["decoder_layer_M2048"] = {"linears": layer, "total_us": round(tot_us, 2),
                                  "TOPS": round(tot_ops / (tot_us * 1e-6) / 1e12, 1),
                                  "frac": round(tot_ops / (tot_us * 1e-6) / 1e12 / bf16_peak, 3),
                                  "fused": {"linears": fused, "total_us": round(fused_us, 2),
                                            "TOPS": round(tot_ops / (fused_us * 1e-6) / 1e12, 1)}}
    return out, samples


def check_samples(samples) -> dict:
    """CPU-baseline leg: the oracle recomputes each sampled block of outputs
    from the same inputs and codes. Quantized layers must be bit-identical;
    the A16 product (a floating-point sum) must lie within its derived error
    bound. Marks each case with "oracle": "match" / "MISMATCH"; returns a
    summary."""
    import numpy as np
    import oracle
    n_match = n = 0
    for sm in samples:
        x = sm["x"].numpy()
        w, s = sm["w"].numpy(), sm["s"].numpy()
        y = sm["y"].numpy()
        if sm["a16"]:
            K = x.shape[1]
            G = 1 if sm["gs"] == 0 else K // sm["gs"]
            ref = oracle.a16_gemv(x[0], w, s, sm["bits"], sm["gs"])
            codes = (w.astype(np.float64) if sm["bits"] == 8
                     else oracle.unpack_int4(w, K).astype(np.float64))
            sc = np.repeat(np.abs(s.astype(np.float64).reshape(len(w), G)), K // G, axis=1)
            E = (K + 2) * 2.0 ** -24 * ((np.abs(codes) * sc) @ np.abs(x[0].astype(np.float64)))
            mag = np.maximum(np.abs(ref) + E, 2.0 ** -14)
            ulp = 2.0 ** (np.floor(np.log2(mag)) - 10)
            ok = bool(np.all(np.abs(y[0].astype(np.float64) - ref) <= 0.5 * ulp + E))
        else:
            fn = oracle.w8a8_linear if sm["bits"] == 8 else oracle.w4a8_linear
            ref = fn(x, w, s, sm["gs"])
            ok = bool(np.array_equal(ref.view(np.uint16), y.view(np.uint16)))
        sm["case"]["oracle"] = "match" if ok else "MISMATCH"
        n += 1
        n_match += ok
    return {"cases": n, "match": n_match,
            "sample": "per case: token rows first, middle, last x 64 seeded output channels"}


def run_configs(args):
    """The config sweep alone: one JSON line."""
    import torch
    import w4a8_quantized_gemm_int8_b300 as cider
    torch.cuda.set_device(0)
    cider.load_library()
    bf16_peak, hbm_peak, peak_src = peaks()
    out, samples = config_sweep(args, check=not args.no_cpu_baseline)
    summary = check_samples(samples) if samples else None
    print(json.dumps({"configs": out, "oracle_check": summary, "steps": args.steps,
                      "warmup": args.warmup,
                      "timing": "CUDA events per call, inputs rotating over sets > 3x L2",
                      "frac": f"of {peak_src} peaks: {bf16_peak} TFLOP/s dense bf16/fp16 "
                              f"(M > 1), {hbm_peak} GB/s HBM copy (M = 1)"}))


def run_cider(args):
    import torch
    import torch.distributed as dist

    import synth
    import w4a8_quantized_gemm_int8_b300 as cider

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    cider.load_library()

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        return replica_max(v, world, dev)

    li = synth.linear_inputs(M, N, K, n_out=4, seed=0)
    x = li.x.to(dev)
    wq, s_w = cider.quantize_weight_int8(li.w.to(dev), 0)  # offline prep, untimed
    stream = torch.cuda.current_stream()
    if args.gemv_only:
        gemv_s, gemv_seq_s, n_copies, _, _ = gemv_leg(args, x, wq, s_w, None, stream)
        if rank == 0:
            nb = N * K + 4 * N + 2 * K + 2 * N
            print(json.dumps({"gemv_us": gemv_s * 1e6, "sequence_us": gemv_seq_s * 1e6,
                              "copies": n_copies, "GB/s": nb / gemv_s / 1e9,
                              "sequence_GB/s": nb / gemv_seq_s / 1e9}))
        return
    a_img = torch.empty((M, K), dtype=torch.float16, device=dev)
    s_a = torch.empty((M,), dtype=torch.float32, device=dev)
    b_img = torch.empty((N, K), dtype=torch.float16, device=dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    y_staged = torch.empty_like(y)
    ws = torch.empty(cider.workspace_bytes(M, N, K, group_size=0, bits=8), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        # The public call: per-token quant + weight image (one launch), then
        # the tensor-core GEMM with the fused dequant epilogue.
        cider.w8a8_linear(x, wq, s_w, 0, out=y, ws=ws)

    def staged():
        cider.act_image(x, a_img, s_a)
        cider.weight_image(wq, K, 8, b_img)
        cider.gemm_images(a_img, s_a, b_img, s_w, 0, y_staged)

    # The staged calls run the same arithmetic kernel by kernel: same bits.
    step()
    staged()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_staged.view(torch.int16)), "staged != fused"

    # Inputs rotate over independent sets (activations, weights, outputs), as
    # the linears of a prefill follow each other, so that a set's data has
    # left L2 before it comes back: together the sets exceed 3x L2.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_set = 2 * M * K + N * K + 2 * M * N
    n_sets = max(2, -(-3 * l2 // per_set) + 1)
    sets = [(x, wq, s_w, y)] + [(x.clone(), wq.clone(), s_w.clone(), torch.empty_like(y))
                                for _ in range(n_sets - 1)]

    def step_i(i):
        xs, wqs, sws, ys = sets[i % n_sets]
        cider.w8a8_linear(xs, wqs, sws, 0, out=ys, ws=ws)

    for i in range(max(args.warmup, n_sets)):
        step_i(i)
    torch.cuda.synchronize()

    def timed_region():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
        clocks = ClockSampler(local)
        barrier()
        torch.cuda.synchronize()
        clocks.start()
        torch.cuda._sleep(int(2e5 * args.steps))  # host runs ahead of the GPU (see the GEMV leg)
        for i in range(args.steps):
            evs[i][0].record(stream)
            step_i(i)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        info = clocks.stop()
        barrier()
        return [e[0].elapsed_time(e[1]) for e in evs], info

    step_ms, clock_info = timed_region()
    # A region that saw a hardware or thermal slowdown, or clocks held low
    # with no reason given, is measured once more (every rank together).
    if max_over_ranks(1.0 if clocks_rejected(clock_info) else 0.0) > 0:
        first = clock_info
        step_ms, clock_info = timed_region()
        clock_info = dict(clock_info or {}, remeasured_after=first)
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at {site:#x}"

    # The same step after an L2 flush (a 512 MiB write) instead: every step
    # then also pays for writing back the flush buffer's dirty lines.
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e5 * args.steps))
    for i in range(args.steps):
        flush.zero_()
        fev[i][0].record(stream)
        step()
        fev[i][1].record(stream)
    torch.cuda.synchronize()
    flushed_ms = [e[0].elapsed_time(e[1]) for e in fev]

    # Per-kernel breakdown (kernels timed one by one with events between them,
    # so they do not overlap as in the step): the GEMM kernel's average launch
    # duration is the roofline's denominator.
    def staged_i(i, e=None):
        xs, wqs, sws, ys = sets[i % n_sets]
        if e is not None:
            e[0].record(stream)
        cider.act_image(xs, a_img, s_a)
        if e is not None:
            e[1].record(stream)
        cider.weight_image(wqs, K, 8, b_img)
        if e is not None:
            e[2].record(stream)
        cider.gemm_images(a_img, s_a, b_img, sws, 0, ys)
        if e is not None:
            e[3].record(stream)

    for i in range(max(args.warmup, n_sets)):
        staged_i(i)
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e5 * args.steps))
    for i in range(args.steps):
        staged_i(i, bev[i])
    torch.cuda.synchronize()
    quant_ms = [e[0].elapsed_time(e[1]) for e in bev]
    widen_ms = [e[1].elapsed_time(e[2]) for e in bev]
    gemm_ms = [e[2].elapsed_time(e[3]) for e in bev]

    if args.step_only:
        if rank == 0:
            print(json.dumps({"step_ms": statistics.mean(step_ms),
                              "act_quant_ms": statistics.mean(quant_ms),
                              "weight_image_ms": statistics.mean(widen_ms),
                              "gemm_ms": statistics.mean(gemm_ms)}))
        return
    flops = 2.0 * M * N * K
    mean_step_s = statistics.mean(step_ms) / 1e3
    mean_step_s = max_over_ranks(mean_step_s)

    gemm_s = statistics.mean(gemm_ms) / 1e3
    bf16_peak, hbm_peak, peak_src = peaks()
    achieved = flops / gemm_s / 1e12

    # ---- M = 1 decode GEMV on the same weights (HBM stream) ----------------
    gemv_s, gemv_seq_s, n_copies, read_s, read_seq_s = gemv_leg(args, x, wq, s_w, y[0], stream)
    gemv_bytes = N * K + 4 * N + 2 * K + 2 * N
    gemv_gbs = gemv_bytes / gemv_s / 1e9
    gemv_seq_gbs = gemv_bytes / gemv_seq_s / 1e9
    # The fused gate|up projection of an 8B-class decoder (K 4096 -> 12288 + 12288).
    gu_N, gu_K = 24576, 4096
    gu_s, gu_copies = gemv_sequence(args, gu_N, gu_K, dev, stream)
    gu_bytes = gu_N * gu_K + 4 * gu_N + 2 * gu_K + 2 * gu_N

    # ---- end to end through the public call, host buffers ------------------
    # Steps run as a serving loop runs them: the copy-in of step i + 1 and the
    # copy-out of step i - 1 overlap the layer of step i (three streams,
    # double-buffered device tensors). Every step's input crosses PCIe from
    # pinned host memory and its output back inside the timed region; L2 is
    # flushed before every layer.
    x_h = li.x.pin_memory()
    y_h = [torch.empty((M, N), dtype=torch.float16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    y_d = [torch.empty_like(y) for _ in range(2)]
    ws = torch.empty(cider.workspace_bytes(M, N, K, group_size=0, bits=8), dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def ev():
        return torch.cuda.Event()

    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        for i in range(n):
            k = i % 2
            if i >= 2:
                s_in.wait_event(ev_done[k])   # x_d[k] read by step i - 2's layer
            with torch.cuda.stream(s_in):
                x_d[k].copy_(x_h, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_out[k])  # y_d[k] copied out by step i - 2
            flush.zero_()
            cider.w8a8_linear(x_d[k], wq, s_w, 0, out=y_d[k], ws=ws)
            ev_done[k].record(stream)
            s_out.wait_event(ev_done[k])
            with torch.cuda.stream(s_out):
                y_h[k].copy_(y_d[k], non_blocking=True)
                ev_out[k].record(s_out)
        stream.wait_event(ev_out[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(ev_out[(n - 2) % 2])
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3 / n

    e2e_run(max(2, args.warmup))
    e2e_s = max_over_ranks(e2e_run(args.steps))
    e2e_value = world * flops / e2e_s / 1e12
    assert torch.equal(y_h[(args.steps - 1) % 2].view(torch.int16), y.cpu().view(torch.int16))

    # ---- sustained: the same step back to back for about 2 s ---------------
    # (the power cap can lower the SM clock of a long dense run below the
    # short timed region's). Run after the GEMV and end-to-end legs so that
    # their timings do not follow two seconds at the power cap.
    n_sus = max(args.steps, int(args.sustain_s / mean_step_s))
    sus_clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sus_clocks.start()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(n_sus):
        step_i(i)
    s1.record(stream)
    torch.cuda.synchronize()
    sus_clock_info = sus_clocks.stop()
    sus_s = max_over_ranks(s0.elapsed_time(s1) / 1e3 / n_sus)
    value = world * flops / mean_step_s / 1e12
    # ---- the INT8 tensor rate of this GPU (the "% INT8 peak" denominator) ---
    int8_rate = int8_mma_rate(dev, stream)

    # ---- every workload of the config list (compact) -----------------------
    sweep = (None if (args.no_configs or rank != 0)
             else config_sweep(args, check=not args.no_cpu_baseline))

    if rank != 0:
        return

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        x_np, wq_np, sw_np = cpu_inputs()
        rows = size_oracle_sample(x_np, wq_np, sw_np, args.cpu_seconds)
        # A host fast enough to finish the whole workload well inside the
        # target repeats it (at most 16 passes), so the figure rests on about
        # cpu_seconds of CPU work either way.
        passes, cpu_dt = 0, 0.0
        while passes == 0 or (passes < 16 and cpu_dt < 0.8 * args.cpu_seconds):
            cpu_dt += oracle_tops(x_np, wq_np, sw_np, rows)[1]
            passes += 1
        cpu_tops = 2.0 * passes * rows * N * K / cpu_dt / 1e12
        reps = f", {passes} passes" if passes > 1 else ""
        cpu = {"value": cpu_tops, "unit": "TOPS", "cores": oracle.get_threads(), "kind": "oracle",
               "sample": f"{rows} of {M} token rows, full N={N}, K={K}{reps} ({cpu_dt:.1f} s)",
               "cpu": cpu_model()}
        # The same leg recomputes the sampled outputs of every config case.
        if sweep is not None:
            cpu["config_check"] = check_samples(sweep[1])

    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_ms), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "mode": "per-channel",
                   "tensor_engine": "tcgen05 kind::f16 on exact fp16 integer codes",
                   "l2": f"inputs rotate over {n_sets} sets of x, wq, y ({n_sets * per_set >> 20} MiB > 3x L2); no flush",
                   "parallelism": f"replicas x{world}"},
        "step_ms_l2_flushed": statistics.mean(flushed_ms),
        "breakdown_ms": {"act_quant": statistics.mean(quant_ms),
                         "weight_image": statistics.mean(widen_ms),
                         "gemm": statistics.mean(gemm_ms),
                         "note": "kernels timed one by one; in the step the quant and weight "
                                 "image share one launch and the GEMM prologue overlaps it"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak,
                     "unit": "TFLOP/s", "frac": achieved / bf16_peak,
                     "traffic": GEMM_DRAM_BYTES_PER_LAUNCH,
                     "traffic_source": (
                         "ncu dram__bytes_read.sum + dram__bytes_write.sum, one cold-cache "
                         "launch of `python bench.py --step-only`"
                         if GEMM_DRAM_BYTES_PER_LAUNCH is not None else
                         "none: the kernel changed after its last ncu capture"),
                     "kernel": "gemm_tc2_kernel<kPcF16> (SM pairs, cta_group::2)",
                     "peak_source": f"{peak_src} dense bf16 burst; fp16 nominal rate equal"},
        "int8_peak": {"value": int8_rate, "unit": "TOPS",
                      "source": "register-only loop of mma.sync.m16n8k32 s8 on every SM, run "
                                "by this bench (sm_103a has no integer tcgen05.mma kind)",
                      "value_pct": 100.0 * value / int8_rate},
        "gemv": {"value": gemv_gbs, "unit": "GB/s", "us": gemv_s * 1e6, "M": 1, "N": N, "K": K,
                 "bytes": gemv_bytes, "kernel": "gemv_kernel<8, false>",
                 "l2": f"cold: {n_copies} rotating weight copies ({n_copies * N * K >> 20} MiB > 3x L2)",
                 "timing": "standalone launch, events around each",
                 "roofline": {"bound": "hbm", "achieved": gemv_gbs, "peak": hbm_peak,
                              "unit": "GB/s", "frac": gemv_gbs / hbm_peak,
                              "traffic": GEMV_DRAM_BYTES_PER_LAUNCH,
                              "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write."
                                                "sum, one cold launch of `python bench.py "
                                                "--gemv-only`"},
                 "sequence": {"value": gemv_seq_gbs, "unit": "GB/s", "us": gemv_seq_s * 1e6,
                              "timing": f"CUDA graph of {n_copies} back-to-back GEMVs (one per "
                                        "weight copy), total time / launches",
                              "frac": gemv_seq_gbs / hbm_peak},
                 "read_ceiling": {
                     "standalone_us": read_s * 1e6, "sequence_us": read_seq_s * 1e6,
                     "standalone_GB/s": N * K / read_s / 1e9,
                     "sequence_GB/s": N * K / read_seq_s / 1e9,
                     "what": "a plain streaming read of the same weight copies, launched and "
                             "timed like the GEMV (standalone and CUDA-graph sequence)"},
                 "gate_up_decode": {
                     "N": gu_N, "K": gu_K, "us": gu_s * 1e6, "GB/s": gu_bytes / gu_s / 1e9,
                     "frac": gu_bytes / gu_s / 1e9 / hbm_peak,
                     "timing": f"CUDA graph of {gu_copies} back-to-back GEMVs of the fused "
                               "gate|up projection (K 4096 -> 2 x 12288), total / launches"}},
        "sustained": {"value": world * flops / sus_s / 1e12, "unit": "TOPS",
                      "seconds": sus_s * n_sus, "steps": n_sus, "ms_per_step": sus_s * 1e3,
                      "clocks": sus_clock_info},
        "e2e": {"value": e2e_value, "unit": "TOPS", "h2d_bytes_per_step": M * K * 2,
                "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_s * 1e3,
                "timing": "steps pipelined on three streams (copy-in, layer, copy-out), "
                          "total time / steps"},
        "cpu_baseline": cpu,
        "configs": sweep[0] if sweep is not None else None,
        "gpu_launches": 2 * args.steps,
        "clocks": clock_info,
        "impl": "cider",
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_layer(args, m, n, k, bits, gs):
    """One public layer call of shape (m, n, k, bits, gs) alone: seeded codes,
    scales and activations made on the GPU, `warmup` calls, then `steps`
    calls timed with CUDA events. Prints the mean call time. Small enough to
    run under a profiler (--small-step: m = 128 per channel at N10240 K2560,
    the few-token engine)."""
    import torch
    import w4a8_quantized_gemm_int8_b300 as cider
    torch.cuda.set_device(0)
    cider.load_library()
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    G = 1 if gs == 0 else k // gs
    x = torch.randn(m, k, generator=gen, device=dev).half()
    w = torch.randint(-127, 128, (n, k if bits == 8 else k // 2), generator=gen, device=dev,
                      dtype=torch.int8)
    if bits == 4:
        w = w.view(torch.uint8)
    s_w = torch.rand((n, G) if gs else (n,), generator=gen, device=dev) * 0.01 + 0.001
    y = torch.empty(m, n, dtype=torch.float16, device=dev)
    ws = torch.empty(max(1, cider.workspace_bytes(m, n, k, group_size=gs, bits=bits)),
                     dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        cider.linear(x, w, s_w, bits, gs, out=y, ws=ws)
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        cider.linear(x, w, s_w, bits, gs, out=y, ws=ws)
        b.record(stream)
    torch.cuda.synchronize()
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at {site:#x}"
    us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    print(json.dumps({"layer_us": us, "M": m, "N": n, "K": k, "bits": bits, "gs": gs,
                      "TOPS": 2.0 * m * n * k / (us * 1e-6) / 1e12}))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.configs:
        run_configs(args)
    elif args.small_step:
        run_layer(args, 128, N, K, 8, 0)
    elif args.layer:
        run_layer(args, *args.layer)
    else:
        run_cider(args)


if __name__ == "__main__":
    main()
