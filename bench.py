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

# workload name -> GEMM shape and description (the step of each is built in make_plan)
WORKLOADS = {
    "pr1": dict(M=256, N=256, K=256, desc="PR1: A, B 256x256 f32 N(0,1) with 1% of entries x50 (seeds 0, 1), "
                                         "1D RNE max-6, GEMM 256x256x256 FP32 out"),
    "wgrad": dict(M=14336, N=4096, K=8192, desc="Llama-3-8B MLP wgrad: dY 8192x14336 bf16 1e-3*t(4) (RHT along the "
                                               "tokens + SR seed 1, transposed), X 8192x4096 bf16 (RHT, transposed), "
                                               "rht_seed 1, GEMM 14336x4096x8192 FP32 out"),
    "llama8b": dict(M=8192, N=14336, K=4096, desc="Llama-3-8B MLP fprop: X 8192x4096 bf16 N(0,1) + 0.1% channels x20 "
                                                 "(1D, RNE, max-6), W 14336x4096 bf16 N(0,0.02) (2D 16x16), "
                                                 "GEMM 8192x14336x4096 BF16 out"),
    "llama405b": dict(M=8192, N=53248, K=16384, desc="Llama-3.1-405B MLP fprop: X 8192x16384 bf16 N(0,1) (1D), "
                                                     "W 53248x16384 bf16 N(0,0.01) (2D), GEMM BF16 out"),
    "moe": dict(E=64, M=512, N=1536, K=4096, desc="MoE experts: 64 x W_e 4096x1536 bf16 0.02*t(3) quantized as W_e^T "
                                                   "(1D along K=4096, Four-over-Six), 64 x X_e 512x4096 bf16 N(0,1) "
                                                   "(1D, max-6), grouped GEMM 64 x (512x1536x4096) BF16 out"),
    "w4a16": dict(L=8, M=4, N=14336, K=4096, desc="W4A16 decode: 8 layers' Llama-3-8B MLP up-projection weights "
                                                  "14336x4096 (bf16 N(0,0.02), quantized once with 2D blocks), "
                                                  "X 4x4096 bf16 N(0,1) + 0.1% channels x20, BF16 out"),
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


def ncu_traffic(kernel: str, src_hash: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and on this workload's launch."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    entries = d.get(kernel) or []
    for e in entries if isinstance(entries, list) else [entries]:
        if e.get("source_hash") == src_hash and e.get("bench_workload") == workload:
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs:
    NVML (read-only queries through libnvidia-ml) polled every ~2 ms from a
    thread, else nvidia-smi at 100 ms."""

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
        self.error = None

    def _uuid(self):
        try:
            u = str(torch.cuda.get_device_properties(self.index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    @staticmethod
    def _nvml_ctypes():
        """A minimal read-only NVML binding (libnvidia-ml ships with the driver;
        the Python wrapper may be absent): clock and clock-event queries."""
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")

        class N:
            NVML_CLOCK_SM = 1
            masks = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
                     "sw_power_cap": 0x4}

            @staticmethod
            def handle(uuid, index):
                h = ctypes.c_void_p()
                rc = (lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) if uuid else
                      lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)))
                if rc != 0:
                    raise RuntimeError(f"nvmlDeviceGetHandle rc={rc}")
                return h

            @staticmethod
            def clock(h, maximum=False):
                v = ctypes.c_uint()
                fn = lib.nvmlDeviceGetMaxClockInfo if maximum else lib.nvmlDeviceGetClockInfo
                if fn(h, ctypes.c_int(1), ctypes.byref(v)) != 0:
                    raise RuntimeError("clock query failed")
                return float(v.value)

            @staticmethod
            def reasons(h):
                v = ctypes.c_ulonglong()
                fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                    lib.nvmlDeviceGetCurrentClocksThrottleReasons
                if fn(h, ctypes.byref(v)) != 0:
                    raise RuntimeError("reason query failed")
                return int(v.value)
        return N

    def start(self):
        uuid = self._uuid()   # the CUDA device's NVML identity (CUDA_VISIBLE_DEVICES may renumber)
        try:
            N = self._nvml_ctypes()
            h = N.handle(uuid, self.index)
            self.max_mhz = N.clock(h, maximum=True)

            def poll():
                try:
                    while not self.stop_flag.is_set():
                        mhz = N.clock(h)
                        r = N.reasons(h)
                        self.samples.append((mhz, {n for n, m in N.masks.items() if r & m}))
                        time.sleep(0.002)
                except Exception as e:
                    self.error = f"nvml poll: {type(e).__name__}: {e}"

            self.source = "nvml"
            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            return
        except Exception as e:
            self.error = f"nvml: {type(e).__name__}: {e}"
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", uuid or str(self.index), f"--query-gpu={self.FIELDS}",
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
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(sm), "source": self.source}
        if self.error:
            out["note"] = self.error
        return out


def max_over_ranks(values, world: int) -> list:
    """Element-wise max of per-rank floats over all ranks (one all-reduce;
    on the GPU for NCCL, on the CPU for gloo)."""
    dev = "cpu"
    if world > 1 and torch.distributed.get_backend() == "nccl":
        dev = torch.device("cuda", torch.cuda.current_device())
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


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


L2_BYTES = 126 * 2**20


def _qbytes(q):
    return q.codes.numel() + q.scales.numel()


def operand_copies(per_set: int) -> int:
    """Operand sets to cycle through so that their total exceeds L2: one if a
    set alone does, else one more than L2 / set."""
    if per_set >= L2_BYTES:
        return 1
    return -(-L2_BYTES // per_set) + 1


def back_to_back_us(fns, dev, reps):
    """Per-launch microseconds of a kernel launched `reps` times back to back
    in one CUDA graph, cycling through the callables `fns` (each on its own
    operand copy), timed between CUDA events on the launching stream; median
    of 5 replays."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for f in fns:
            f()
        with torch.cuda.graph(g, stream=side):
            for r in range(reps):
                fns[r % len(fns)]()
    torch.cuda.current_stream(dev).wait_stream(side)
    g.replay()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(5):
        st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.record()
        g.replay()
        en.record()
        torch.cuda.synchronize(dev)
        ts.append(st.elapsed_time(en) * 1e3 / reps)
    del g
    torch.cuda.synchronize(dev)
    return statistics.median(ts)


def gemm_rate(nv, qa, qb, d, dev, reps=12):
    """The GEMM kernel alone, back to back over operand copies whose total
    exceeds L2 (so every launch streams its operands from DRAM): per-launch
    microseconds and the timing note, or None when more than 8 copies would
    be needed (a latency-bound shape, reported by its in-step time)."""
    per_set = _qbytes(qa) + _qbytes(qb)
    copies = operand_copies(per_set)
    if copies > 8:
        return None
    sets = [(qa, qb)] + [(qa.clone(), qb.clone()) for _ in range(copies - 1)]
    fns = [(lambda a=a, b=b: nv.gemm(a, b, out=d)) for a, b in sets]
    reps = max(reps, copies)
    us = back_to_back_us(fns, dev, reps)
    note = (f"CUDA events over a graph of {reps} back-to-back GEMMs cycling through {copies} operand "
            f"cop{'ies' if copies > 1 else 'y'} ({copies * per_set / 2**20:.0f} MiB of codes and scales, L2 "
            f"{L2_BYTES / 2**20:.0f} MiB); per launch")
    del sets, fns
    return us, note


def next_input_rates(nv, qa, qb, d, dev, flush, reps=10):
    """GEMM -> the next layer's NVFP4 input (its BF16 output quantized 1D,
    RNE, max-6 with the producer amax), three ways, each a CUDA graph timed
    between events with an L2 flush before every replay: the GEMM with the
    producer amax then the quantizer over D; the GEMM with the encoding in
    its epilogue and D not stored; the same with D stored."""
    M, N = qa.rows, qb.rows
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    amax_next = torch.zeros(1, dtype=torch.float32, device=dev)
    nv.gemm_amax(qa, qb, out=d, amax_out=amax)
    qd = nv.NVFP4Tensor.empty(M, N, device=dev)
    variants = {
        "gemm_amax_then_quantize": lambda: (nv.gemm_amax(qa, qb, out=d, amax_out=amax_next),
                                            nv.quantize(d, amax=amax_next, out=qd)),
        "gemm_quantize_fused": lambda: nv.gemm_quantize(qa, qb, amax, out=qd),
        "gemm_quantize_fused_with_d": lambda: nv.gemm_quantize(qa, qb, amax, out=qd, d=d),
    }
    out = {}
    side = torch.cuda.Stream(dev)
    for name, fn in variants.items():
        side.wait_stream(torch.cuda.current_stream(dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()
            with torch.cuda.graph(g, stream=side):
                fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        ts = []
        for _ in range(reps + 2):
            flush.zero_()
            st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            st.record()
            g.replay()
            en.record()
            torch.cuda.synchronize(dev)
            ts.append(st.elapsed_time(en))
        out[name] = {"us": round(statistics.median(ts[2:]) * 1e3, 2)}
        del g
    nv.sync_check()
    return out


# --------------------------------------------------------------------------
# our implementation
# --------------------------------------------------------------------------
def make_plan(workload: str, nv, synthetic, dev):
    """The step of a workload: its host inputs, device inputs, components
    (name, call, elements quantized, input bytes per element) with the GEMM
    last, the output D and the launches of our kernels per step."""
    c = WORKLOADS[workload]
    M, N, K = c["M"], c["N"], c["K"]
    if workload == "pr1":
        wl = synthetic.pr1()
        a_h, b_h = wl.tensors["A"], wl.tensors["B"]
    elif workload == "wgrad":
        wl = synthetic.wgrad()
        a_h, b_h = wl.tensors["dY"], wl.tensors["X"]
    else:
        wl = synthetic.llama8b_fprop() if workload == "llama8b" else synthetic.llama405b_fprop()
        a_h, b_h = wl.tensors["X"], wl.tensors["W"]
    a_h, b_h = a_h.pin_memory(), b_h.pin_memory()
    a, b = a_h.to(dev), b_h.to(dev)
    qa = nv.NVFP4Tensor.empty(M, K, device=dev)
    qb = nv.NVFP4Tensor.empty(N, K, device=dev)
    out_dtype = torch.float32 if workload in ("pr1", "wgrad") else torch.bfloat16
    d = torch.empty((M, N), dtype=out_dtype, device=dev)
    es = a.element_size()

    def qcalls(a, b):  # the two operand quantizations reading the device inputs a, b
        if workload == "wgrad":
            return [("quantize_dYT_rht_sr", lambda: nv.rht_quantize(a, rht_seed=1, transpose=True,
                                                                    rounding="stochastic", seed=1, out=qa),
                     a.numel(), es),
                    ("quantize_XT_rht", lambda: nv.rht_quantize(b, rht_seed=1, transpose=True, out=qb), b.numel(), es)]
        if workload == "pr1":
            return [("quantize_A", lambda: nv.quantize(a, out=qa), a.numel(), es),
                    ("quantize_B", lambda: nv.quantize(b, out=qb), b.numel(), es)]
        return [("quantize_X", lambda: nv.quantize(a, out=qa), a.numel(), es),
                ("quantize_W_2d", lambda: nv.quantize(b, block="2d", out=qb), b.numel(), es)]

    parts = qcalls(a, b)
    parts.append(("gemm", lambda: nv.gemm(qa, qb, out=d), None, None))
    # RHT: an amax-only pass of the transform and the encode; plain: amax + encode; GEMM: 1
    return dict(inputs_h=[a_h, b_h], inputs=[a, b], parts=parts, out=d, M=M, N=N, K=K, launches=5, fwd=(a, b),
                q=(qa, qb), qcalls=qcalls, gemm_into=lambda dd: nv.gemm(qa, qb, out=dd))


def run_ours(args, rank, world, local_rank):
    import nvfp4_bit_block_02_b300 as nv
    import synthetic

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfgw = WORKLOADS[args.workload]
    plan = make_plan(args.workload, nv, synthetic, dev)
    M, N, K = plan["M"], plan["N"], plan["K"]
    x_h, w_h = plan["inputs_h"]
    x, w = plan["inputs"]
    d = plan["out"]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    launches_per_step = plan["launches"]

    # The two operand quantizations are independent: the step forks them onto
    # two streams and joins before the GEMM (both HBM-bound; running together
    # they fill each other's launch gaps and latency-bound tails).
    fork_stream = torch.cuda.Stream(dev)

    def step():
        main = torch.cuda.current_stream(dev)
        fork_stream.wait_stream(main)
        plan["parts"][0][1]()
        with torch.cuda.stream(fork_stream):
            plan["parts"][1][1]()
        main.wait_stream(fork_stream)
        plan["parts"][2][1]()

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
        for g, (_, fn, _, _) in zip(parts, plan["parts"]):
            with torch.cuda.graph(g, stream=side):
                fn()
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
    t_parts = [[evc[i][j].elapsed_time(evc[i][j + 1]) for i in range(args.steps)] for j in range(3)]
    t_gm = t_parts[2]
    enc = encode_rates(nv, x, w, dev) if rank == 0 and args.workload in ("llama8b", "llama405b") else None
    # back-to-back timing only where a launch is short enough (< 1 ms) for its launch gap to matter; a longer
    # GEMM run back to back settles into the power-capped regime, which the step's own clocks decide about
    gr = gemm_rate(nv, *plan["q"], d, dev) if rank == 0 and statistics.mean(t_gm) < 1.0 else None
    nxt = next_input_rates(nv, *plan["q"], d, dev, flush) if rank == 0 and args.workload in ("llama8b",) else None
    # end to end through the public API from pinned host buffers, D read back.
    # Every step uploads its X and W and reads back all of D, with two device
    # copies of the inputs and of D so that neighbouring steps overlap on the
    # two directions of the host link: step i uploads into set i % 2 on an
    # upload stream once step i - 2 has quantized from that set, quantizes and
    # multiplies on the main stream, and reads D back on a download stream;
    # the GEMM into a set waits only for that set's previous read-back.
    d_h = torch.empty((M, N), dtype=d.dtype, pin_memory=True)
    xs, ws, ds = [x, torch.empty_like(x)], [w, torch.empty_like(w)], [d, torch.empty_like(d)]
    qsets = [plan["qcalls"](xs[k], ws[k]) for k in range(2)]
    up_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_steps = max(3, min(args.steps, 10))
    inputs_free, d_free = [None, None], [None, None]
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        k = i % 2
        main = torch.cuda.current_stream(dev)
        with torch.cuda.stream(up_stream):
            if inputs_free[k] is not None:
                up_stream.wait_event(inputs_free[k])
            xs[k].copy_(x_h, non_blocking=True)
            ws[k].copy_(w_h, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(up_stream)
        main.wait_event(loaded)
        fork_stream.wait_stream(main)
        qsets[k][0][1]()
        with torch.cuda.stream(fork_stream):
            qsets[k][1][1]()
        main.wait_stream(fork_stream)
        inputs_free[k] = torch.cuda.Event()
        inputs_free[k].record(main)
        if d_free[k] is not None:
            main.wait_event(d_free[k])
        plan["gemm_into"](ds[k])
        d2h_stream.wait_stream(main)
        with torch.cuda.stream(d2h_stream):
            d_h.copy_(ds[k], non_blocking=True)
            d_free[k] = torch.cuda.Event()
            d_free[k].record(d2h_stream)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    del xs, ws, ds, qsets

    step_ms, e2e_s = max_over_ranks([step_ms, e2e_s], world)
    if rank != 0:
        return None

    pk, pk_src = peaks()
    flops = 2.0 * M * N * K
    ms_per_step = step_ms / args.steps
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    gemm_ms = statistics.mean(t_gm)
    # algorithmic bytes of the quantizer: in-bytes read + 0.5 B codes + 1/16 B scales per element, plus the
    # second read of the tensor amax pass
    qbytes = lambda n, es=2: n * (es + 0.5 + 1 / 16)
    amax_bytes = lambda n, es=2: n * es
    comps = {}
    for j, (name, _, elems, es) in enumerate(plan["parts"][:2]):
        ms = statistics.mean(t_parts[j])
        comps[name] = {"ms": round(ms, 4), "GB_s": round((qbytes(elems, es) + amax_bytes(elems, es)) / (ms * 1e-3) / 1e9, 1),
                       "bytes_per_elem": f"{es} read + 0.5625 written (encode) + {es} read (amax pass)"}
    # a timed region that ran power-capped is a sustained regime: its denominator is the sustained peak
    sustained = bool(clocks and "sw_power_cap" in (clocks.get("reasons") or []))
    fp4_burst = pk["bf16_tflops"] * FP4_OVER_BF16
    fp4_peak = (pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]) * FP4_OVER_BF16
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    # the roofline's per-launch duration: back to back over operand copies > L2 (else the in-step time)
    roof_tflops = flops / (gr[0] * 1e-6) / 1e12 if gr else gemm_tflops
    roof_timing = gr[1] if gr else ("CUDA events around the GEMM's graph replay inside the component "
                                    "breakdown (L2 flushed before each step; used for launches of 1 ms or more "
                                    "and for shapes whose operands would need more than 8 copies to exceed L2)")
    traffic = ncu_traffic("k_gemm", source_hash("gemm.cu", "gemm.h"), args.workload)
    q_traffic = ncu_traffic("k_quant_rows", source_hash("quantize.cu", "nvfp4_device.cuh"), args.workload)
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
        "dtype": f"fp4(e2m1)+e4m3 scales, fp32 accumulate; {str(x.dtype).replace('torch.', '')} in, "
                 f"{str(d.dtype).replace('torch.', '')} out",
        "data": "synthetic (seeded numpy draws, the pages' shapes; no model weights)",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "desc": cfgw["desc"],
                   "l2": f"256 MiB flush write between steps (outside the timed events); inputs "
                         f"{(x.numel() * x.element_size() + w.numel() * w.element_size()) / 2**20:.0f} MiB",
                   "timing": "the step (and, for the component breakdown, each component) captured once as a CUDA "
                             "graph and replayed between CUDA events on the launching stream",
                   "value_is": "2*M*N*K / step time, summed over ranks; the step quantizes both operands "
                               "concurrently on two streams, then runs the GEMM"},
        "components": {
            **comps,
            "gemm": {"ms": round(gemm_ms, 4), "TFLOP_s": round(gemm_tflops, 1),
                     "frac_of_fp4_peak": round(gemm_tflops / fp4_peak, 4)},
            # GEMM -> next layer's NVFP4 input (D quantized with the producer amax): unfused vs fused epilogue
            "next_layer_input": nxt,
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
                     "achieved": round(roof_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(roof_tflops / fp4_peak, 4), "traffic": traffic,
                     "frac_of_burst_peak": round(roof_tflops / fp4_burst, 4),
                     "us_per_launch": round(flops / (roof_tflops * 1e12) * 1e6, 2),
                     "timing": roof_timing,
                     "peak_source": (f"{pk_src} bf16 {'sustained' if sustained else 'burst'} "
                                     f"{pk['bf16_tflops_sustained'] if sustained else pk['bf16_tflops']} TFLOP/s x "
                                     f"{FP4_OVER_BF16} (nominal FP4:BF16 dense ratio)"
                                     + ("; sustained because the timed region ran under sw_power_cap" if sustained
                                        else ""))},
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(x_h.numel() * x_h.element_size() + w_h.numel() * w_h.element_size()),
                "d2h_bytes_per_step": int(d_h.numel() * d_h.element_size())},
        "gpu_launches": launches_per_step * args.steps * world,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    return line


def run_moe(args, rank, world, local_rank):
    """The MoE configuration: per step, Four-over-Six quantization of the 64
    expert weights (W_e^T, K = 4096), max-6 quantization of the 64 routed
    token blocks, and one grouped GEMM launch; plus the Four-over-Six vs
    max-6 weight MSE over all experts."""
    import nvfp4_bit_block_02_b300 as nv
    import synthetic

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    c = WORKLOADS["moe"]
    E, M, N, K = c["E"], c["M"], c["N"], c["K"]
    wl = synthetic.moe(E, M, K, N)
    w_h = wl.tensors["W"].pin_memory()   # [E][K][N]
    x_h = wl.tensors["X"].pin_memory()   # [E][M][K]
    w, x = w_h.to(dev), x_h.to(dev)
    qw = [nv.NVFP4Tensor.empty(N, K, device=dev) for _ in range(E)]
    qx = [nv.NVFP4Tensor.empty(M, K, device=dev) for _ in range(E)]
    d = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(E)]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    w_list = [w[e] for e in range(E)]
    x_list = [x[e] for e in range(E)]

    def quant_w():   # one amax + one encode launch for the 64 experts
        nv.quantize_grouped(w_list, transpose=True, scaling="four_over_six", out=qw)

    def quant_x():
        nv.quantize_grouped(x_list, out=qx)

    def grouped():
        nv.gemm_grouped(qx, qw, out=d)

    fork_stream = torch.cuda.Stream(dev)

    def step():   # the two quantizations run concurrently (independent), then the grouped GEMM
        main = torch.cuda.current_stream(dev)
        fork_stream.wait_stream(main)
        quant_w()
        with torch.cuda.stream(fork_stream):
            quant_x()
        main.wait_stream(fork_stream)
        grouped()

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
        for g, fn in zip(parts, (quant_w, quant_x, grouped)):
            with torch.cuda.graph(g, stream=side):
                fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        g_step.replay()
        for g in parts:
            g.replay()
    nv.sync_check(stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        g_step.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    nv.sync_check(stream)
    step_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        for j, g in enumerate(parts):
            evc[i][j].record(stream)
            g.replay()
        evc[i][3].record(stream)
    torch.cuda.synchronize(dev)
    t = [[evc[i][j].elapsed_time(evc[i][j + 1]) for i in range(args.steps)] for j in range(3)]
    # weight MSE of Four-over-Six against max-6 (a measurement beside the path)
    q6 = [nv.quantize(w[e], transpose=True) for e in range(E)]
    se46 = se6 = 0.0
    for e in range(E):
        ref = w[e].t().float()
        se46 += float(((nv.dequantize(qw[e]) - ref) ** 2).double().sum())
        se6 += float(((nv.dequantize(q6[e]) - ref) ** 2).double().sum())
    nv.sync_check()
    # end to end: H2D of every expert's W and X from pinned memory, D2H of
    # every D, with two device copies of the inputs and of D (as in the other
    # workloads): step i uploads into set i % 2 on an upload stream once step
    # i - 2 has quantized from it and reads D back on a download stream; the
    # grouped GEMM into a set waits only for that set's previous read-back
    d_h = torch.empty((E, M, N), dtype=torch.bfloat16, pin_memory=True)
    ws2, xs2 = [w, torch.empty_like(w)], [x, torch.empty_like(x)]
    ds2 = [d, [torch.empty_like(t) for t in d]]
    up_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_steps = 4
    inputs_free, d_free = [None, None], [None, None]
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        k = i % 2
        main = torch.cuda.current_stream(dev)
        with torch.cuda.stream(up_stream):
            if inputs_free[k] is not None:
                up_stream.wait_event(inputs_free[k])
            ws2[k].copy_(w_h, non_blocking=True)
            xs2[k].copy_(x_h, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(up_stream)
        main.wait_event(loaded)
        fork_stream.wait_stream(main)
        nv.quantize_grouped([ws2[k][e] for e in range(E)], transpose=True, scaling="four_over_six", out=qw)
        with torch.cuda.stream(fork_stream):
            nv.quantize_grouped([xs2[k][e] for e in range(E)], out=qx)
        main.wait_stream(fork_stream)
        inputs_free[k] = torch.cuda.Event()
        inputs_free[k].record(main)
        if d_free[k] is not None:
            main.wait_event(d_free[k])
        nv.gemm_grouped(qx, qw, out=ds2[k])
        d2h_stream.wait_stream(main)
        with torch.cuda.stream(d2h_stream):
            for e in range(E):
                d_h[e].copy_(ds2[k][e], non_blocking=True)
            d_free[k] = torch.cuda.Event()
            d_free[k].record(d2h_stream)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    del ws2, xs2, ds2
    # the roofline's per-launch duration: the grouped GEMM back to back (its
    # operands, 268 MB of codes, exceed L2 on their own)
    g_us = back_to_back_us([lambda: nv.gemm_grouped(qx, qw, out=d)], dev, 6) if rank == 0 else None
    step_ms, e2e_s = max_over_ranks([step_ms, e2e_s], world)
    if rank != 0:
        return None
    pk, pk_src = peaks()
    flops = 2.0 * E * M * N * K
    ms_per_step = step_ms / args.steps
    gm_ms = statistics.mean(t[2])
    # grouped GEMM algorithmic bytes: codes and scales of A and B once, D once
    gbytes = E * (M * K // 2 + N * K // 2 + nv.scales_bytes(M, K) + nv.scales_bytes(N, K) + M * N * 2)
    g_gbs = gbytes / (g_us * 1e-6) / 1e9
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    q_elems = E * (N * K + M * K)
    line = {
        "metric": METRIC, "value": round(world * flops / (ms_per_step * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp4(e2m1)+e4m3 scales, fp32 accumulate; bf16 in/out",
        "data": "synthetic (seeded numpy draws, the pages' shapes; no model weights)",
        "config": {"workload": "moe", "experts": E, "tokens_per_expert": M, "N": N, "K": K, "desc": c["desc"],
                   "l2": "256 MiB flush write between steps (outside the timed events); inputs 1.07 GB > L2",
                   "timing": "the step captured once as a CUDA graph and replayed between CUDA events",
                   "value_is": "2*E*M*N*K / step time; the step quantizes W and X concurrently on two streams, "
                               "then runs the grouped GEMM"},
        "components": {
            "quantize_W_four_over_six": {"ms": round(statistics.mean(t[0]), 4),
                                         "GB_s": round(E * N * K * 4.5625 / (statistics.mean(t[0]) * 1e-3) / 1e9, 1)},
            "quantize_X": {"ms": round(statistics.mean(t[1]), 4),
                           "GB_s": round(E * M * K * 4.5625 / (statistics.mean(t[1]) * 1e-3) / 1e9, 1)},
            "grouped_gemm": {"ms": round(gm_ms, 4), "TFLOP_s": round(flops / (gm_ms * 1e-3) / 1e12, 1),
                             "frac_of_fp4_peak": round(flops / (gm_ms * 1e-3) / 1e12 / fp4_peak, 4)},
            "weight_mse": {"four_over_six": se46, "max6": se6, "ratio": round(se46 / se6, 5),
                           "context": "the Nemotron 3 Ultra story reports -16.4% expert-weight MSE on real weights"},
            "quantize_bytes_per_elem": "2.5625 encode + 2 amax read",
        },
        "roofline": {"bound": "hbm", "kernel": "k_gemm_grouped (64 experts, one launch)",
                     "achieved": round(g_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(g_gbs / pk["hbm_gbs"], 4),
                     "traffic": ncu_traffic("k_gemm_grouped", source_hash("gemm.cu", "gemm.h"), "moe"),
                     "algorithmic_bytes_per_launch": gbytes, "us_per_launch": round(g_us, 2),
                     "timing": "CUDA events over a graph of 6 back-to-back grouped GEMMs (operands 268 MB > L2); "
                               "per launch",
                     "peak_source": f"{pk_src} copy bandwidth"},
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(w_h.numel() * 2 + x_h.numel() * 2),
                "d2h_bytes_per_step": int(d_h.numel() * 2)},
        "gpu_launches": 7 * args.steps * world,   # (zero amax, amax, encode) x 2 + grouped GEMM
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline("moe")
    return line


def run_w4a16(args, rank, world, local_rank):
    """The weight-only decode configuration: per step, M tokens through L
    layers' NVFP4 weights (one W4A16 launch per layer, each on its own copy
    of the weight, so no launch finds its weight in L2).  Weights are
    quantized once, outside the step, as a serving deployment does."""
    import nvfp4_bit_block_02_b300 as nv
    import synthetic

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    c = WORKLOADS["w4a16"]
    L, M, N, K = c["L"], c["M"], c["N"], c["K"]
    wl = synthetic.llama8b_fprop(m=M, n=N, k=K)
    x_h = wl.tensors["X"].pin_memory()
    x = x_h.to(dev)
    w_bf16 = wl.tensors["W"].to(dev)
    q0 = nv.quantize(w_bf16, block="2d")
    qs = [nv.NVFP4Tensor(q0.codes.clone(), q0.scales.clone(), q0.global_scale.clone(), q0.amax.clone(), N, K)
          for _ in range(L)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    nv.sync_check()

    def step(xm, outs):
        for l in range(L):
            nv.w4a16_gemm(xm, qs[l], out=outs[l])

    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)

    def graph_of(fn):
        for _ in range(args.warmup):
            fn()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn()
        stream.wait_stream(side)
        for _ in range(args.warmup):
            g.replay()
        return g

    def timed(g, steps):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [e[0].elapsed_time(e[1]) for e in ev]

    g_step = graph_of(lambda: step(x, ys))
    nv.sync_check(stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    t_step = timed(g_step, args.steps)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    nv.sync_check(stream)
    step_ms = sum(t_step)
    # other decode batch sizes, and a BF16 GEMM of the same shape (cuBLAS, for context)
    comps = {}
    for m in (1, 4, 16):
        xm = synthetic.llama8b_fprop(m=m, n=16, k=K).tensors["X"].to(dev)
        outs = [torch.empty((m, N), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        ms = statistics.mean(timed(graph_of(lambda: step(xm, outs)), max(10, args.steps // 4))) / L
        b = N * K // 2 + nv.scales_bytes(N, K) + m * K * 2 + m * N * 2
        comps[f"w4a16_M{m}"] = {"us_per_launch": round(ms * 1e3, 2), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                                "TFLOP_s": round(2.0 * m * N * K / (ms * 1e-3) / 1e12, 2)}
    w_layers = [w_bf16.clone() for _ in range(L)]
    yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ms_bf16 = statistics.mean(timed(graph_of(lambda: [torch.matmul(x, wl_.t(), out=yb) for wl_ in w_layers]),
                                    max(10, args.steps // 4))) / L
    comps["bf16_cublas_same_shape"] = {"us_per_launch": round(ms_bf16 * 1e3, 2),
                                       "GB_s": round((N * K * 2 + M * K * 2 + M * N * 2) / (ms_bf16 * 1e-3) / 1e9, 1),
                                       "note": "torch.matmul on the BF16 weight (context, not the path)"}
    del w_layers
    # end to end: H2D of the step's activations, D2H of every layer's output
    y_h = torch.empty((L, M, N), dtype=torch.bfloat16, pin_memory=True)
    e2e_steps = 20
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x.copy_(x_h, non_blocking=True)
        step(x, ys)
        for l in range(L):
            y_h[l].copy_(ys[l], non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    step_ms, e2e_s = max_over_ranks([step_ms, e2e_s], world)
    if rank != 0:
        return None
    pk, pk_src = peaks()
    flops = 2.0 * L * M * N * K
    ms_per_step = step_ms / args.steps
    abytes = N * K // 2 + nv.scales_bytes(N, K) + M * K * 2 + M * N * 2
    gbs = abytes / (ms_per_step / L * 1e-3) / 1e9
    line = {
        "metric": "W4A16 decode TFLOP/s (weight-stream GB/s as % of B300 HBM roofline)",
        "value": round(world * flops / (ms_per_step * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 activations x fp4(e2m1)+e4m3 weights decoded to bf16, fp32 accumulate; bf16 out",
        "data": "synthetic (seeded numpy draws, the pages' shapes; no model weights)",
        "config": {"workload": "w4a16", "layers": L, "tokens": M, "N": N, "K": K, "desc": c["desc"],
                   "l2": f"256 MiB flush write between steps (outside the timed events); {L} weight copies "
                         f"of {abytes / 1e6:.1f} MB each",
                   "timing": "the step (one launch per layer) captured once as a CUDA graph, replayed between "
                             "CUDA events",
                   "value_is": "2*L*M*N*K / step time"},
        "components": comps,
        "roofline": {"bound": "hbm", "kernel": "k_w4a16 (one layer)", "achieved": round(gbs, 1),
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                     "traffic": ncu_traffic("k_w4a16", source_hash("w4a16.cu", "nvfp4_device.cuh"), "w4a16"),
                     "algorithmic_bytes_per_launch": abytes, "peak_source": f"{pk_src} copy bandwidth"},
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(x_h.numel() * 2), "d2h_bytes_per_step": int(y_h.numel() * 2)},
        "gpu_launches": L * args.steps * world,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline("w4a16")
    return line


# --------------------------------------------------------------------------
# the oracle on the host cores (the reference arm and the cpu_baseline key)
# --------------------------------------------------------------------------
def _oracle_inputs(workload: str):
    import synthetic
    if workload == "w4a16":
        c = WORKLOADS["w4a16"]
        wl = synthetic.llama8b_fprop(m=c["M"], n=c["N"], k=c["K"])
        return wl.tensors["X"].to(torch.float32).numpy(), wl.tensors["W"].to(torch.float32).numpy()
    if workload == "moe":
        c = WORKLOADS["moe"]
        wl = synthetic.moe(1, c["M"], c["K"], c["N"])
        return wl.tensors["X"][0].to(torch.float32).numpy(), wl.tensors["W"][0].to(torch.float32).numpy()
    if workload == "pr1":
        wl = synthetic.pr1()
        return wl.tensors["A"].numpy(), wl.tensors["B"].numpy()
    if workload == "wgrad":
        wl = synthetic.wgrad()
        return wl.tensors["dY"].to(torch.float32).numpy(), wl.tensors["X"].to(torch.float32).numpy()
    wl = synthetic.llama8b_fprop() if workload == "llama8b" else synthetic.llama405b_fprop()
    return wl.tensors["X"].to(torch.float32).numpy(), wl.tensors["W"].to(torch.float32).numpy()


def _flops(workload: str) -> float:
    c = WORKLOADS[workload]
    return 2.0 * c.get("E", 1) * c.get("L", 1) * c["M"] * c["N"] * c["K"]


def _linear_fit(n1: int, t1: float, n2: int, t2: float):
    """t(n) = a + b * n through two timed sizes: (fixed seconds, seconds per unit)."""
    b = max((t2 - t1) / (n2 - n1), 0.0)
    return max(t1 - b * n1, 0.0), b


# Oracle timing.  llama8b, wgrad and pr1 run the whole step (a few seconds on the host cores); llama405b, and the
# 1-core figure of every fprop/wgrad workload, time slices and extrapolate: per workload (X rows, W rows, GEMM
# output rows, GEMM output columns) at all cores; the 1-core figure divides the sizes by _ONE_CORE_DIV.
_FULL_STEP = ("llama8b", "wgrad", "pr1")
_ORACLE_SLICES = {"llama8b": (2048, 3584, 1024, 2048), "llama405b": (512, 1024, 512, 2048),
                  "wgrad": (1024, 512, 1024, 1024), "pr1": (128, 128, 128, 128)}
_ONE_CORE_DIV = 4


def _time(fn):
    t0 = time.perf_counter()
    r = fn()
    return time.perf_counter() - t0, r


def _oracle_step(workload: str, X, W, div: int = 1) -> dict:
    """Time the oracle, as it stands, on one step of the workload.

    Whole step (llama8b, wgrad, pr1 at all cores): quantize both operands and
    the fp64 GEMM reference, no extrapolation.  MoE times one whole expert
    (scaled to 64), W4A16 one whole layer (scaled to 8): the step's own
    repeated unit.  Otherwise slices, each part extrapolated separately:
    every quantization is timed at two sizes n and 2n and fit as a + b*n (the
    fixed cost a is charged once); the GEMM reference is timed on a block of
    output rows and columns, and its operand conversions (oracle.exact_values
    of the A rows and of the B rows) are timed on their own, so that the
    products' cost per output is separated from the per-row and per-column
    conversion costs before each is scaled to the whole step."""
    import oracle
    c = WORKLOADS[workload]
    M, N = c["M"], c["N"]
    if workload == "w4a16":
        qw = oracle.quantize(W, block2d=True)      # quantized once, outside the step (as on the GPU)
        t, _ = _time(lambda: oracle.w4a16_reference(X, qw))
        return {"step_s": c["L"] * t, "spent_s": t, "parts": {"w4a16_layer_s": round(t, 4)},
                "work": f"one whole layer (W {N}x{c['K']}, {c['M']} tokens), x{c['L']} layers"}
    if workload == "moe":
        tw, qw = _time(lambda: oracle.quantize(W, transpose=True, four_over_six=True))
        tx, qx = _time(lambda: oracle.quantize(X))
        tg, _ = _time(lambda: oracle.gemm_reference(qx, qw))
        t = tw + tx + tg
        return {"step_s": c["E"] * t, "spent_s": t,
                "parts": {"quantize_w_s": round(tw, 4), "quantize_x_s": round(tx, 4), "gemm_s": round(tg, 4)},
                "work": f"one whole expert (W_e^T Four-over-Six, X_e, GEMM {c['M']}x{N}x{c['K']}), x{c['E']}"}
    if workload == "wgrad":
        qa_fn = lambda n: oracle.quantize(np.ascontiguousarray(X[:, :n]), transpose=True, rht=True, stochastic=True,
                                          seed=1, rht_seed=1)
        qb_fn = lambda n: oracle.quantize(np.ascontiguousarray(W[:, :n]), transpose=True, rht=True, rht_seed=1)
        n_a, n_b = X.shape[1], W.shape[1]
    else:
        qa_fn = lambda n: oracle.quantize(X[:n])
        qb_fn = lambda n: oracle.quantize(W[:n], block2d=workload != "pr1")
        n_a, n_b = X.shape[0], W.shape[0]
    if div == 1 and workload in _FULL_STEP:
        ta, qa = _time(lambda: qa_fn(n_a))
        tb, qb = _time(lambda: qb_fn(n_b))
        tg, _ = _time(lambda: oracle.gemm_reference(qa, qb))
        t = ta + tb + tg
        return {"step_s": t, "spent_s": t,
                "parts": {"quantize_a_s": round(ta, 3), "quantize_b_s": round(tb, 3), "gemm_reference_s": round(tg, 3)},
                "work": "the whole step (both quantizations and the full fp64 GEMM reference), no extrapolation"}
    rx, rw, rg, rc = (max(1, v // div) for v in _ORACLE_SLICES[workload])
    ta1, _ = _time(lambda: qa_fn(rx))
    ta2, qa = _time(lambda: qa_fn(2 * rx))
    tb1, _ = _time(lambda: qb_fn(rw))
    tb2, qb = _time(lambda: qb_fn(2 * rw))
    fa, fb = _linear_fit(rx, ta1, 2 * rx, ta2), _linear_fit(rw, tb1, 2 * rw, tb2)
    rg, rc = min(rg, qa.R), min(rc, qb.R)
    qbc = oracle.Quantized(qb.codes[:rc], qb.scales[:rc], qb.amax, qb.g, None, None, rc, qb.K)
    qag = oracle.Quantized(qa.codes[:rg], qa.scales[:rg], qa.amax, qa.g, None, None, rg, qa.K)
    tg, _ = _time(lambda: oracle.gemm_reference(qag, qbc))
    tca, _ = _time(lambda: oracle.exact_values(qag.codes, qag.scales, qag.g))
    tcb, _ = _time(lambda: oracle.exact_values(qbc.codes, qbc.scales, qbc.g))
    prod = max(tg - tca - tcb, 0.0)
    t_gemm = tca * M / rg + tcb * N / rc + prod * (M / rg) * (N / rc)
    step = (fa[0] + fa[1] * M) + (fb[0] + fb[1] * N) + t_gemm
    spent = ta1 + ta2 + tb1 + tb2 + tg + tca + tcb
    parts = {name: {"fixed_s": round(a_, 5), "per_unit_us": round(b_ * 1e6, 4), "fixed_frac_at_n": round(a_ / t_, 4)}
             for name, (a_, b_), t_ in (("quantize_a", fa, ta1), ("quantize_b", fb, tb1))}
    parts["gemm"] = {"block": [rg, rc], "block_s": round(tg, 4), "convert_a_rows_s": round(tca, 4),
                     "convert_b_rows_s": round(tcb, 4), "products_per_output_ns": round(prod / (rg * rc) * 1e9, 3),
                     "whole_step_s": round(t_gemm, 3)}
    unit = "columns" if workload == "wgrad" else "rows"
    return {"step_s": step, "spent_s": spent, "parts": parts,
            "work": (f"extrapolated: quantize A {unit} [0,{rx}) and [0,{2 * rx}), B {unit} [0,{rw}) and [0,{2 * rw}) "
                     f"(each fit as a + b*n); fp64 GEMM reference on a {rg} x {rc} output block with its operand "
                     f"conversions timed apart; each part scaled to the whole step")}


def _set_threads(n: int | None):
    """Threads of the oracle's OpenMP loops and of numpy's BLAS (None: all)."""
    import ctypes
    try:
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(n or len(os.sched_getaffinity(0)))
    except OSError:
        pass
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(limits=n)
    except ImportError:
        return None


def cpu_baseline(workload: str):
    """The oracle as it stands on the host cores: all cores, then one core on
    slices 1/8 the size, each extrapolated to one whole step (labelled)."""
    import oracle
    oracle.build()
    X, W = _oracle_inputs(workload)
    cores = len(os.sched_getaffinity(0))
    _set_threads(None)
    r = _oracle_step(workload, X, W)
    r1 = None
    if workload in _ORACLE_SLICES:   # MoE and W4A16 time a whole expert / layer: no 1-core run of that size
        lim = _set_threads(1)
        r1 = _oracle_step(workload, X, W, div=_ONE_CORE_DIV)
        if lim is not None:
            lim.restore_original_limits()
        _set_threads(None)
    flops = _flops(workload)
    out = {"value": round(flops / r["step_s"] / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": r["work"], "extrapolated": workload not in _FULL_STEP,
           "extrapolated_step_seconds": round(r["step_s"], 3), "sample_seconds": round(r["spent_s"], 2),
           "parts": r["parts"]}
    if r1 is not None:
        out["one_core"] = {"value": round(flops / r1["step_s"] / 1e12, 6), "cores": 1,
                           "extrapolated_step_seconds": round(r1["step_s"], 3),
                           "sample_seconds": round(r1["spent_s"], 2), "sample": r1["work"]}
    return out


def run_reference(args):
    """The base contract's reference arm for a method with no installable
    code: the oracle, timed on the host cores.  Each step runs the same work
    as the cpu_baseline key: the whole step where it finishes in seconds
    (llama8b, Wgrad, PR1), otherwise a bounded sample extrapolated to the
    whole step with the same model; ms_per_step is the time the work took."""
    import oracle
    oracle.build()
    _set_threads(None)
    X, W = _oracle_inputs(args.workload)
    for _ in range(args.warmup):
        _oracle_step(args.workload, X, W)
    runs = [_oracle_step(args.workload, X, W) for _ in range(max(1, args.steps))]
    t_full = statistics.mean(r["step_s"] for r in runs)
    t_sample = statistics.mean(r["spent_s"] for r in runs)
    value = _flops(args.workload) / t_full / 1e12
    c = WORKLOADS[args.workload]
    cfg = {"workload": args.workload, **{k: v for k, v in c.items() if k != "desc"}, "desc": c["desc"]}
    cores = len(os.sched_getaffinity(0))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_sample * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32/fp64 (CPU oracle)",
            "data": "synthetic", "config": cfg,
            "value_is": ("2*M*N*K / the time of the whole oracle step, timed as it is; ms_per_step is that time"
                         if args.workload in _FULL_STEP else
                         "2*M*N*K / the whole step's oracle time, extrapolated from the timed sample (each part fit "
                         "as a + b*n at two sizes); ms_per_step is the time the sample itself took"),
            "extrapolated_step_ms": round(t_full * 1e3, 1),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: " + runs[0]["work"],
                             "extrapolated": args.workload not in _FULL_STEP},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_oracle_full_gemm():
    """One-off: the oracle's fp64 GEMM reference of the whole Llama-3-8B fprop
    (8192 x 14336 x 4096) on the host cores, with its wall time."""
    import oracle
    oracle.build()
    _set_threads(None)
    X, W = _oracle_inputs("llama8b")
    tq, (qa, qb) = _time(lambda: (oracle.quantize(X), oracle.quantize(W, block2d=True)))
    tg, _ = _time(lambda: oracle.gemm_reference(qa, qb))
    return {"oracle_full_gemm": "llama8b", "M": 8192, "N": 14336, "K": 4096, "cores": len(os.sched_getaffinity(0)),
            "quantize_both_s": round(tq, 2), "gemm_reference_s": round(tg, 2),
            "gemm_tflops_fp64": round(2 * 8192 * 14336 * 4096 / tg / 1e12, 4)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-full-gemm", action="store_true",
                    help="time the oracle's full Llama-3-8B fp64 GEMM once on the host cores and exit")
    args = ap.parse_args()
    if args.oracle_full_gemm:
        print(json.dumps(run_oracle_full_gemm()), flush=True)
        return
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
    run = {"moe": run_moe, "w4a16": run_w4a16}.get(args.workload, run_ours)
    line = run(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
