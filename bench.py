"""Benchmark of the NVFP4 hot path on B300: one step = quantize the activations
(1D blocks, RNE, tensor amax computed), quantize the weights (2D 16x16
blocks), and the block-scaled GEMM, for the Llama-3-8B-shaped MLP fprop
(X 8192x4096, W 14336x4096, BF16 in, BF16 out) by default.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line.  Under torchrun (N > 1) every rank runs an independent
replica of the workload on its own GPU (weak scaling, no data-path
collective); time is the max over ranks.  ``--impl reference`` times the CPU
oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "quantize HBM GB/s and NVFP4 GEMM TFLOPS, each as % of B300 roofline"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 : BF16 tensor ratio of B300
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# workload name -> (M, N, K, X dtype, builder, description)
WORKLOADS = {
    "llama8b": dict(M=8192, N=14336, K=4096, desc="Llama-3-8B MLP fprop: X 8192x4096 bf16 N(0,1) + 0.1% channels x20 "
                                                 "(1D, RNE, max-6), W 14336x4096 bf16 N(0,0.02) (2D 16x16), "
                                                 "GEMM 8192x14336x4096 BF16 out"),
    "llama405b": dict(M=8192, N=53248, K=16384, desc="Llama-3.1-405B MLP fprop: X 8192x16384 bf16 N(0,1) (1D), "
                                                     "W 53248x16384 bf16 N(0,0.01) (2D), GEMM BF16 out"),
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK if k in d}, "measured"
    return dict(FALLBACK), "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "nvfp4_bit_block_02_b300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs:
    NVML polled every ~2 ms from a thread (read-only queries), else
    nvidia-smi at 100 ms."""

    NAMES = (("hw_slowdown", "nvmlClocksEventReasonHwSlowdown"),
             ("hw_thermal_slowdown", "nvmlClocksEventReasonHwThermalSlowdown"),
             ("sw_thermal_slowdown", "nvmlClocksEventReasonSwThermalSlowdown"),
             ("sw_power_cap", "nvmlClocksEventReasonSwPowerCap"))
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []   # (sm_mhz, reasons set)
        self.max_mhz = None
        self.stop_flag = threading.Event()
        self.thread = None
        self.proc = None
        self.source = None

    def start(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = float(pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM))
            masks = [(n, getattr(pynvml, a)) for n, a in self.NAMES]
            getr = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                pynvml.nvmlDeviceGetCurrentClocksThrottleReasons

            def poll():
                while not self.stop_flag.is_set():
                    mhz = float(pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM))
                    r = getr(h)
                    self.samples.append((mhz, {n for n, m in masks if r & m}))
                    time.sleep(0.002)

            self.source = "nvml"
            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            return
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi"

        def read():
            for line in self.proc.stdout:
                r = [c.strip() for c in line.split(",")]
                if len(r) >= 8 and r[0].replace(".", "").isdigit():
                    self.max_mhz = float(r[1]) if r[1].replace(".", "").isdigit() else self.max_mhz
                    self.samples.append((float(r[0]), {n for i, (n, _) in enumerate(self.NAMES) if r[4 + i] == "Active"}))

        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm = [m for m, _ in self.samples]
        reasons = sorted(set().union(*[r for _, r in self.samples])) if self.samples else []
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm), "source": self.source}


def encode_rates(nv, x, w, dev, reps=24):
    """Encode kernels alone (tensor amax supplied), back to back over copies
    whose total exceeds L2, replayed from a CUDA graph: microseconds per
    launch for X (1D) and W (2D)."""
    out = {}
    for name, src, copies, kw in (("X", x, 4, {}), ("W", w, 3, {"block": "2d"})):
        xs = [src.clone() for _ in range(copies)]
        qs = [nv.quantize(t, **kw) for t in xs]
        am = qs[0].amax.clone()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            for i in range(copies):
                nv.quantize(xs[i], out=qs[i], amax=am, **kw)
            with torch.cuda.graph(g, stream=side):
                for r in range(reps):
                    nv.quantize(xs[r % copies], out=qs[r % copies], amax=am, **kw)
        torch.cuda.current_stream(dev).wait_stream(side)
        g.replay()
        torch.cuda.synchronize(dev)
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(5):
            st.record()
            g.replay()
            en.record()
            torch.cuda.synchronize(dev)
            ts.append(st.elapsed_time(en) / reps)
        out[name] = {"us": statistics.median(ts) * 1e3, "elems": src.numel(), "launches": 5 * reps}
        del xs, qs, g
    torch.cuda.synchronize(dev)
    return out


# --------------------------------------------------------------------------
# our implementation
# --------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import nvfp4_bit_block_02_b300 as nv
    import synthetic

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfgw = WORKLOADS[args.workload]
    M, N, K = cfgw["M"], cfgw["N"], cfgw["K"]
    if args.workload == "llama8b":
        wl = synthetic.llama8b_fprop()
    else:
        wl = synthetic.llama405b_fprop()
    x_h = wl.tensors["X"].pin_memory()
    w_h = wl.tensors["W"].pin_memory()
    x = x_h.to(dev)
    w = w_h.to(dev)
    qx = nv.NVFP4Tensor.empty(M, K, device=dev)
    qw = nv.NVFP4Tensor.empty(N, K, device=dev)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    launches_per_step = 5  # amax + encode for X and W, GEMM

    def step(stream=None):
        nv.quantize(x, out=qx, stream=stream)
        nv.quantize(w, block="2d", out=qw, stream=stream)
        nv.gemm(qx, qw, out=d, stream=stream)

    # The step and each of its components are captured once as CUDA graphs
    # and replayed, so the device timeline carries no host-side launch gaps.
    for _ in range(args.warmup):
        step()
    nv.sync_check()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g_step = torch.cuda.CUDAGraph()
    parts = [torch.cuda.CUDAGraph() for _ in range(3)]
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_step, stream=side):
            step()
        with torch.cuda.graph(parts[0], stream=side):
            nv.quantize(x, out=qx)
        with torch.cuda.graph(parts[1], stream=side):
            nv.quantize(w, block="2d", out=qw)
        with torch.cuda.graph(parts[2], stream=side):
            nv.gemm(qx, qw, out=d)
    torch.cuda.current_stream(dev).wait_stream(side)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        g_step.replay()
        for g in parts:
            g.replay()
    nv.sync_check(stream)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    for i in range(args.steps):
        flush.zero_()          # L2 flush between steps (outside the timed events)
        ev[i][0].record(stream)
        g_step.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    nv.sync_check(stream)
    step_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    # component breakdown: the same step as three graphs with events between them
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        for j, g in enumerate(parts):
            evc[i][j].record(stream)
            g.replay()
        evc[i][3].record(stream)
    torch.cuda.synchronize(dev)
    t_qx = [evc[i][0].elapsed_time(evc[i][1]) for i in range(args.steps)]
    t_qw = [evc[i][1].elapsed_time(evc[i][2]) for i in range(args.steps)]
    t_gm = [evc[i][2].elapsed_time(evc[i][3]) for i in range(args.steps)]
    enc = encode_rates(nv, x, w, dev) if rank == 0 else None
    # end to end through the public API from pinned host buffers, D read back
    d_h = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    e2e_steps = max(2, min(args.steps, 5))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x.copy_(x_h, non_blocking=True)
        w.copy_(w_h, non_blocking=True)
        step()
        d_h.copy_(d, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps

    stats = torch.tensor([step_ms, e2e_s], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(stats, op=torch.distributed.ReduceOp.MAX)
    step_ms, e2e_s = float(stats[0]), float(stats[1])
    if rank != 0:
        return None

    pk, pk_src = peaks()
    flops = 2.0 * M * N * K
    ms_per_step = step_ms / args.steps
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    gemm_ms = statistics.mean(t_gm)
    qx_ms, qw_ms = statistics.mean(t_qx), statistics.mean(t_qw)
    # algorithmic bytes of the quantizer (BF16 in): 2 B read + 0.5 B codes + 1/16 B scales per element,
    # plus the second read of the tensor amax pass
    qbytes = lambda n: n * (2 + 0.5 + 1 / 16)
    amax_bytes = lambda n: n * 2
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    traffic = ncu_traffic("k_gemm", source_hash("gemm.cu", "gemm.h"))
    q_traffic = ncu_traffic("k_quant_rows", source_hash("quantize.cu", "nvfp4_device.cuh"))
    hbm = pk["hbm_gbs"]
    enc_line = {}
    if enc:
        for nm, e in enc.items():
            gbs = qbytes(e["elems"]) / (e["us"] * 1e-6) / 1e9
            enc_line[nm] = {"us_per_launch": round(e["us"], 2), "GB_s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4)}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4(e2m1)+e4m3 scales, fp32 accumulate; bf16 in/out",
        "data": "synthetic (seeded numpy draws, the pages' shapes; no model weights)",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "desc": cfgw["desc"],
                   "l2": "256 MiB flush write between steps (outside the timed events); inputs 176 MiB > L2",
                   "timing": "the step (and, for the component breakdown, each component) captured once as a CUDA "
                             "graph and replayed between CUDA events on the launching stream",
                   "value_is": "2*M*N*K / (quantize X + quantize W + GEMM) step time, summed over ranks"},
        "components": {
            "quantize_X": {"ms": round(qx_ms, 4), "GB_s": round((qbytes(M * K) + amax_bytes(M * K)) / (qx_ms * 1e-3) / 1e9, 1),
                           "encode_bytes_per_elem": 2.5625, "amax_pass_bytes_per_elem": 2.0},
            "quantize_W_2d": {"ms": round(qw_ms, 4), "GB_s": round((qbytes(N * K) + amax_bytes(N * K)) / (qw_ms * 1e-3) / 1e9, 1)},
            "gemm": {"ms": round(gemm_ms, 4), "TFLOP_s": round(gemm_tflops, 1),
                     "frac_of_fp4_peak": round(gemm_tflops / fp4_peak, 4)},
            # the encode kernel alone (tensor amax supplied), the quantizer's roofline figure
            "roofline_quantize": ({"bound": "hbm", "kernel": "k_quant_rows (X 1D RNE)",
                                   "achieved": enc_line["X"]["GB_s"], "peak": hbm, "unit": "GB/s",
                                   "frac": enc_line["X"]["frac_of_hbm"], "traffic": q_traffic,
                                   "algorithmic_bytes_per_elem": 2.5625,
                                   "per_tensor": enc_line,
                                   "timing": "CUDA events over a graph of 24 back-to-back encodes cycling "
                                             "through copies larger than L2 (X x4, W x3)",
                                   "peak_source": f"{pk_src} copy bandwidth"} if enc_line else None),
        },
        "roofline": {"bound": "tensor", "kernel": "k_gemm (tcgen05 mxf4nvf4 block-scaled)",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp4_peak, 4), "traffic": traffic,
                     "peak_source": f"{pk_src} bf16 burst {pk['bf16_tflops']} TFLOP/s x {FP4_OVER_BF16} "
                                    "(nominal FP4:BF16 dense ratio)"},
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(x_h.numel() * 2 + w_h.numel() * 2),
                "d2h_bytes_per_step": int(d_h.numel() * 2)},
        "gpu_launches": launches_per_step * args.steps * world,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    return line


# --------------------------------------------------------------------------
# the oracle on the host cores (the reference arm and the cpu_baseline key)
# --------------------------------------------------------------------------
def cpu_baseline(workload: str, budget_rows=(2048, 3584, 256)):
    """Time the oracle on a bounded sample of one step and extrapolate to the
    whole step: quantize the first rx rows of X and rw rows of W, GEMM (fp64)
    of rg output rows against the quantized W slice's columns scaled to N."""
    import oracle
    import synthetic
    oracle.build()
    cfgw = WORKLOADS[workload]
    M, N, K = cfgw["M"], cfgw["N"], cfgw["K"]
    rx, rw, rg = budget_rows
    wl = synthetic.llama8b_fprop() if workload == "llama8b" else synthetic.llama405b_fprop()
    X = wl.tensors["X"][:rx].to(torch.float32).numpy()
    W = wl.tensors["W"][:rw].to(torch.float32).numpy()
    t0 = time.perf_counter()
    qx = oracle.quantize(X)
    t1 = time.perf_counter()
    qw = oracle.quantize(W, block2d=True)
    t2 = time.perf_counter()
    oracle.gemm_reference(qx, qw, rows=np.arange(rg))
    t3 = time.perf_counter()
    t_step = (t1 - t0) * M / rx + (t2 - t1) * N / rw + (t3 - t2) * (M / rg) * (N / rw)
    return {"value": round(2.0 * M * N * K / t_step / 1e12, 6), "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"oracle quantize of X[:{rx}] (1D) and W[:{rw}] (2D), fp64 GEMM of {rg} rows x {rw} cols; "
                      f"times scaled to the full {M}x{N}x{K} step",
            "sample_seconds": round(t3 - t0, 2), "extrapolated_step_seconds": round(t_step, 2)}


def run_reference(args):
    t_steps = []
    cb = None
    for _ in range(args.warmup):
        pass
    for _ in range(max(1, args.steps)):
        cb = cpu_baseline(args.workload, budget_rows=(512, 896, 64))
        t_steps.append(cb["extrapolated_step_seconds"])
    cfgw = WORKLOADS[args.workload]
    M, N, K = cfgw["M"], cfgw["N"], cfgw["K"]
    t = statistics.mean(t_steps)
    value = 2.0 * M * N * K / t / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32/fp64 (CPU oracle)", "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K, "desc": cfgw["desc"]},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
