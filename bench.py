"""Benchmark of the GB300 ROCmFP4 library.

Default workload ("layer"): one dense decoder layer's four dual-scale ROCmFP4
matrices -- [N, K] = [7168, 5120] (fused QKV), [5120, 6144] (O), [34816, 5120]
(fused gate+up), [5120, 17408] (down) -- each multiplied by a batch-1 fp16
activation vector ~ N(0, 1).  One step = the four GEMVs, one launch each,
replayed as a CUDA graph (programmatic dependent launch between them).  Steps
rotate over enough resident copies of the layer that the working set is far
larger than L2, so every step streams its weights from HBM.

Metric: weight-streaming GB/s = (packed weight bytes + activation bytes +
output bytes) per step / step time.  The roofline object is that of the
dominant kernel (the streaming GEMV) against the measured HBM copy bandwidth.
The same line carries the W4A16 prefill GEMM ("prefill": X bf16 [M, K],
M in {512, 4096, 23552}, over the four layer shapes) in TFLOP/s against the
measured bf16 tensor peak.

Other workloads (--workload):
  single   N=256, K=1024 dual GEMV (latency; L2 flushed between iterations)
  sweep    the four shapes x {dual, single-scale} x M in {1, 2, 4, 8}
  model    64 layers x the four matrices + LM head [152064, 5120] (12.5 GB),
           one CUDA graph of 257 GEMVs per token
  prefill  the prefill GEMM alone

--impl reference times the CPU oracle (the fp64 C implementation under
oracle/) on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYER = [("qkv", 7168, 5120), ("o", 5120, 6144), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
LM_HEAD = ("lm_head", 152064, 5120)
ROLES = ("qkv", "o", "gate_up", "down", "lm_head")
N_LAYERS = 64
PREFILL_M = (512, 4096, 23552)
L2_BYTES = 129 * 1024 * 1024
METRIC = "ROCmFP4 GEMV weight GB/s (% of HBM peak); W4A16 GEMM TFLOP/s (% peak)"
DATA = "synthetic (seeded SplitMix64 weight bytes, Box-Muller N(0,1) activations)"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemv_stream_layer_dual_m1.md")
# the kernel and the host code that sizes its grid: the traffic record holds while both are unchanged
GEMV_SOURCES = (os.path.join(ROOT, "gemm_rocmfp4_dequant_gb300", "csrc", "gemv.cu"),
                os.path.join(ROOT, "gemm_rocmfp4_dequant_gb300", "csrc", "api.cu"))


def peaks():
    """(HBM GB/s, bf16 TF/s burst, bf16 TF/s sustained, 'measured' | 'fallback')."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def block_bytes(variant):
    return 18 if variant == 0 else 17


def matrix_bytes(N, K, variant=0):
    return N * (K // 32) * block_bytes(variant)


def step_bytes(mats, variant=0, M=1):
    """Algorithmic bytes of one pass: packed weights + activations (2 B) + outputs (4 B)."""
    return sum(matrix_bytes(N, K, variant) + 2 * M * K + 4 * M * N for _, N, K in mats)


def weight_bytes(mats, variant=0):
    return sum(matrix_bytes(N, K, variant) for _, N, K in mats)


def gemv_traffic():
    """DRAM bytes per launch of the streaming GEMV on the layer shapes, from the
    committed ncu summary, if that capture was taken on the current kernel and
    launch-sizing source (the sha256 of both files is recorded in the summary);
    else None."""
    try:
        text = open(TRAFFIC_FILE).read()
        src = hashlib.sha256(b"".join(open(f, "rb").read() for f in GEMV_SOURCES)).hexdigest()
    except OSError:
        return None
    m = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    t = re.search(r"dram_bytes_per_launch:\s*(.+)", text)
    if not m or not t or m.group(1) != src:
        return None
    out = {}
    for part in t.group(1).split(","):
        k, v = part.strip().split("=")
        out[k.strip()] = int(v)
    return out


# ---- clocks -------------------------------------------------------------------------

class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region: NVML through
    ctypes every 2 ms (so short regions still get samples), else nvidia-smi every
    200 ms."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: int = 0):
        self.device = device
        self.samples: list[tuple[float, int]] = []
        self.max_mhz = None
        self.kind = None
        self._stop = threading.Event()
        self._nvml = None
        self._handle = None
        self._proc = None

    def _open_nvml(self):
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return False
        props = torch.cuda.get_device_properties(self.device)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self._reasons_fn = None
        for name in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
            try:
                self._reasons_fn = getattr(lib, name)
                break
            except AttributeError:
                continue
        self._nvml, self._handle = lib, h
        return True

    def _sample_nvml(self):
        lib, h = self._nvml, self._handle
        clk, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        while True:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = 0
                if self._reasons_fn is not None and self._reasons_fn(h, ctypes.byref(reasons)) == 0:
                    r = reasons.value
                self.samples.append((float(clk.value), int(r)))
            if self._stop.wait(0.002):
                break

    def _read_smi(self):
        for ln in self._proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.max_mhz = mx
            bits = 0
            for bit, v in zip((0x8, 0x40, 0x20, 0x4), parts[2:6]):
                if v.lower() == "active":
                    bits |= bit
            self.samples.append((sm, bits))

    def __enter__(self):
        try:
            ok = self._open_nvml()
        except Exception:
            ok = False
        if ok:
            self.kind = "nvml"
            self._t = threading.Thread(target=self._sample_nvml, daemon=True)
            self._t.start()
            return self
        try:
            fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                      "clocks_event_reasons.sw_power_cap")
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device}", f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.kind = "nvidia-smi"
            self._t = threading.Thread(target=self._read_smi, daemon=True)
            self._t.start()
        except Exception:
            self.kind = None
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self.kind == "nvml":
            self._t.join(timeout=1)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": self.kind}
        sm = [s for s, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(name for bit, name in self.REASONS.items() if bits & bit)
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "source": self.kind}


# ---- distributed plumbing (replicas only) -----------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- CPU oracle baseline ------------------------------------------------------------------

def cpu_oracle_rate(mats, variant=0, M=1, budget_s=12.0, act=0, rows=None):
    """Times the oracle on row samples of each matrix; returns (GB/s of the metric,
    cores, sample text, seconds).  The sample size comes from a short probe so that
    the timed run takes about budget_s seconds; the metric counts the sampled rows'
    packed bytes plus their share of activation and output bytes."""
    import oracle
    import synth
    cores = os.cpu_count() or 1
    inputs = []
    for idx, (name, N, K) in enumerate(mats):
        inputs.append((N, K, synth.activations(M, K, act, seed=0, stream=synth.act_stream(0, idx))))

    cache = {}

    def run(rows_per, passes=1):
        nbytes, secs = 0.0, 0.0
        for idx, (N, K, Xh) in enumerate(inputs):
            n = min(rows_per, N)
            if (idx, n) not in cache:
                cache[(idx, n)] = synth.weights(N, K, variant, seed=0, stream=synth.weight_stream(0, idx),
                                                rows=np.arange(n))
            Wr = cache[(idx, n)]
            for _ in range(passes):
                t0 = time.perf_counter()
                oracle.gemm(Wr, Xh, n, K, variant, act=act, nthreads=cores)
                secs += time.perf_counter() - t0
                rb = (K // 32) * block_bytes(variant)
                nbytes += n * (rb + 4 * M) + 2 * M * K * n / N
        return nbytes, secs

    passes = 1
    if rows is None:
        # grow a probe until it takes a quarter of the budget (small probes are
        # dominated by fixed costs), then scale to the budget
        nmax = max(N for _, N, _ in mats)
        rows = 2 * cores
        b, t = run(rows)
        while t < budget_s / 4 and rows < nmax:
            rows = min(nmax, rows * 4)
            b, t = run(rows)
        if rows < nmax:
            rows = int(min(nmax, rows * budget_s / max(t, 1e-3)))
        else:  # whole matrices are quicker than the budget: repeat them
            passes = max(1, int(budget_s / max(t, 1e-3)))
    rows_per = rows
    b, t = run(rows_per, passes)
    desc = (f"{passes} pass(es) over {rows_per if rows_per < max(N for _, N, _ in mats) else 'all'} rows of each of "
            f"the {len(mats)} matrices (M={M}), oracle threaded over rows on {cores} cores")
    return b / t / 1e9, cores, desc, t


def cpu_oracle_flops(mats, M, budget_s=8.0, act=1, rows=None):
    """Oracle TFLOP/s of the prefill product on a sample of rows x tokens."""
    import oracle
    import synth
    cores = os.cpu_count() or 1
    toks = min(M, 64)

    def run(rows_per):
        flops, secs = 0.0, 0.0
        for idx, (name, N, K) in enumerate(mats):
            rows = np.arange(min(rows_per, N))
            Wr = synth.weights(N, K, 0, seed=0, stream=synth.weight_stream(0, idx), rows=rows)
            Xh = synth.activations(toks, K, act, seed=0, stream=synth.act_stream(0, idx))
            t0 = time.perf_counter()
            oracle.gemm(Wr, Xh, len(rows), K, 0, act=act, nthreads=cores)
            secs += time.perf_counter() - t0
            flops += 2.0 * toks * len(rows) * K
        return flops, secs

    if rows is None:
        f, t = run(cores)
        rows = int(max(cores, min(5120, cores * budget_s / max(t, 1e-3))))
    rows_per = rows
    f, t = run(rows_per)
    return f / t / 1e12, cores, f"{rows_per} rows x {toks} tokens of each layer matrix, {cores} cores", t


# ---- timing helpers ---------------------------------------------------------------------------

def time_steps(step_fn, steps, warmup, world):
    """Seconds for `steps` calls of step_fn after `warmup`, between CUDA events on the
    current stream, with a device synchronisation and a barrier on both sides."""
    import torch
    for i in range(warmup):
        step_fn(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for i in range(steps):
        step_fn(warmup + i)
    b.record(s)
    b.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    return a.elapsed_time(b) / 1e3


def time_runs(run_fn, steps, warmup, world):
    """As time_steps, for a run_fn(n, first) that performs n consecutive steps."""
    import torch
    run_fn(warmup, 0)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    run_fn(steps, warmup)
    b.record(s)
    b.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    return a.elapsed_time(b) / 1e3


class L2Flush:
    """A buffer larger than L2; writing it evicts whatever an earlier call left in L2."""

    def __init__(self):
        import torch
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.buf.zero_()


# ---- batch-1 / small-batch GEMV workloads ---------------------------------------------------

class GemvStep:
    """R resident copies of a list of matrices; step i runs one product per matrix
    of copy i % R (one launch each), captured per copy as a CUDA graph."""

    def __init__(self, mats, variant, M, act, copies, seed0=0):
        import torch

        import gemm_rocmfp4_dequant_gb300 as rf4
        import synth
        import synth.device
        self.rf4, self.mats, self.variant, self.M, self.act = rf4, mats, variant, M, act
        dt = torch.float16 if act == 0 else torch.bfloat16
        self.W, self.X, self.Y = [], [], []
        for r in range(copies):
            Wc, Xc, Yc = [], [], []
            for m, (name, N, K) in enumerate(mats):
                w = torch.empty(N * rf4.row_bytes(K, variant), dtype=torch.uint8, device="cuda")
                synth.device.fill_weights(w, N, K, variant, seed=seed0 + r, stream=synth.weight_stream(m // 5, m % 5))
                x = torch.empty((M, K), dtype=torch.int16, device="cuda")
                synth.device.fill_act(x, act, seed=seed0 + r, stream=synth.act_stream(m // 5, m % 5))
                Wc.append(w)
                Xc.append(x.view(dt))
                Yc.append(torch.empty((M, N), dtype=torch.float32, device="cuda"))
            self.W.append(Wc)
            self.X.append(Xc)
            self.Y.append(Yc)
        torch.cuda.synchronize()
        self.copies = copies
        self.graphs = None

    def run(self, r, stream=None):
        for m, (name, N, K) in enumerate(self.mats):
            self.rf4.gemm(self.W[r][m], self.X[r][m], N, K, self.variant, Y=self.Y[r][m], stream=stream)

    def capture(self):
        import torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run(0, s)  # the first call on the device does the library's one-time set-up
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graphs = []
        for r in range(self.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.run(r)
            self.graphs.append(g)
        # one pass per resident copy in one graph, as an engine captures many layers per token
        self.multi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.multi):
            for r in range(self.copies):
                self.run(r)
        torch.cuda.synchronize()

    def run_steps(self, n, first):
        """n consecutive passes starting at pass `first` (copy first % copies): whole
        rotations from the multi-pass graph, the rest from single-pass graphs."""
        i = 0
        while i < n:
            r = (first + i) % self.copies
            if r == 0 and i + self.copies <= n:
                self.multi.replay()
                i += self.copies
            else:
                self.graphs[r].replay()
                i += 1

    def launches_per_step(self):
        return len(self.mats)


def copies_for(mats, variant):
    """Resident copies so that a rotation streams more than four times the L2."""
    return max(2, int(np.ceil(4 * L2_BYTES / weight_bytes(mats, variant))) + 1)


def per_matrix_kernel_times(L: GemvStep, reps=None, ceilings=None):
    """Average device time of each matrix's kernel: a CUDA graph of `reps` launches
    of that matrix's product is replayed between CUDA events on the launching
    stream.  The launches rotate over copies of the matrix whose total exceeds
    four times the L2 (the resident layer copies plus extra copies for small
    matrices), so every launch streams its weights from HBM.  If `ceilings` is
    a list, it receives per matrix the device time of a plain read of the same
    bytes (ceiling/read.cu: bulk copies into shared memory and an XOR checksum
    of every word, no decode), in the same graph shape over the same copies,
    the fastest of ceiling.CONFIGS: what one launch of that size reaches
    without any decode or arithmetic."""
    import torch

    import synth
    import synth.device
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = []
    for m, (name, N, K) in enumerate(L.mats):
        nbytes = N * L.rf4.row_bytes(K, L.variant)
        ncopies = max(L.copies, int(np.ceil(4 * L2_BYTES / nbytes)) + 1)
        Ws = [L.W[r][m] for r in range(L.copies)]
        for r in range(L.copies, ncopies):
            w = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            synth.device.fill_weights(w, N, K, L.variant, seed=1000 + r, stream=synth.weight_stream(0, m))
            Ws.append(w)
        n = reps or max(50, 2 * ncopies)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                r = i % ncopies
                L.rf4.gemm(Ws[r], L.X[r % L.copies][m], N, K, L.variant, Y=L.Y[r % L.copies][m])
        g.replay()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(3):
            g.replay()
        e1.record(s)
        e1.synchronize()
        out.append(e0.elapsed_time(e1) / 1e3 / (3 * n))
        del g
        if ceilings is not None and nbytes % 16 == 0:
            import ceiling
            sink = torch.zeros(2, dtype=torch.int32, device="cuda")
            best = None
            for cfg in ceiling.CONFIGS:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(n):
                        ceiling.read(Ws[i % ncopies], sink, cfg, sms)
                g.replay()
                torch.cuda.synchronize()
                e0.record(s)
                for _ in range(3):
                    g.replay()
                e1.record(s)
                e1.synchronize()
                t = e0.elapsed_time(e1) / 1e3 / (3 * n)
                best = t if best is None or t < best else best
                del g
            if int(sink[1].item()) != 0:
                raise RuntimeError("read ceiling kernel: a bounded wait gave up")
            ceilings.append(best)
            del sink
        del Ws
    torch.cuda.empty_cache()
    return out


def e2e_rate(L: GemvStep, steps, warmup, world, staged=True):
    """The metric through the public API with host buffers: every step copies the
    step's activations (all matrices', packed in one pinned host buffer) to the
    device, runs the products through the API and reads all outputs back into one
    pinned host buffer; weights stay resident.  staged: both transfers by the
    library's staging copy (rocmfp4_copy, a kernel in the chain of dependent
    launches); else by torch copies on the copy engines."""
    import torch
    xs = [x.numel() for x in L.X[0]]
    ys = [y.numel() for y in L.Y[0]]
    hx = [torch.cat([x.reshape(-1) for x in Xc]).cpu().pin_memory() for Xc in L.X]
    hy = [torch.empty(sum(ys), dtype=torch.float32).pin_memory() for _ in L.Y]
    dx_all = torch.empty(sum(xs), dtype=L.X[0][0].dtype, device="cuda")
    dy_all = torch.empty(sum(ys), dtype=torch.float32, device="cuda")
    dx = [v.view(x.shape) for v, x in zip(torch.split(dx_all, xs), L.X[0])]
    dy = [v.view(y.shape) for v, y in zip(torch.split(dy_all, ys), L.Y[0])]
    h2d = dx_all.numel() * dx_all.element_size()
    d2h = dy_all.numel() * 4

    def one(i):
        r = i % L.copies
        if staged:
            L.rf4.copy(dx_all, hx[r])
        else:
            dx_all.copy_(hx[r], non_blocking=True)
        for m, (name, N, K) in enumerate(L.mats):
            L.rf4.gemm(L.W[r][m], dx[m], N, K, L.variant, Y=dy[m])
        if staged:
            L.rf4.copy(hy[r], dy_all)
        else:
            hy[r].copy_(dy_all, non_blocking=True)

    t = time_steps(one, steps, warmup, world)
    return t, h2d, d2h


def run_gemv(args, world, hbm, mats, variant=0, M=1, act=0, with_e2e=True, with_ceiling=True):
    """Timed steps of the GEMV workload; returns the measurements of the JSON line."""
    import torch
    copies = copies_for(mats, variant)
    L = GemvStep(mats, variant, M, act, copies)
    L.capture()
    launches0 = L.rf4.launch_count()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t = time_runs(L.run_steps, args.steps, args.warmup, world)
    t = max_over_ranks(t, world)
    sb = step_bytes(mats, variant, M)
    ceil = []
    kt = per_matrix_kernel_times(L, ceilings=ceil if with_ceiling else None)
    algo = [matrix_bytes(N, K, variant) + 2 * M * K + 4 * M * N for _, N, K in mats]
    achieved = sum(algo) / sum(kt) / 1e9
    res = dict(
        value=world * sb * args.steps / t / 1e9, ms_per_step=t / args.steps * 1e3, clocks=clk.summary(),
        gpu_launches=L.launches_per_step() * args.steps, copies=copies,
        footprint_gb=round(copies * weight_bytes(mats, variant) / 1e9, 3),
        per_launch_us={n: round(x * 1e6, 2) for (n, _, _), x in zip(mats, kt)},
        achieved=achieved, algo_bytes={n: a for (n, _, _), a in zip(mats, algo)}, kernel_s=kt,
        read_ceiling_us={n: round(x * 1e6, 2) for (n, _, _), x in zip(mats, ceil)} if len(ceil) == len(mats) else None,
        read_ceiling_gbs={n: round(matrix_bytes(N, K, variant) / x / 1e9, 1) for (n, N, K), x in zip(mats, ceil)}
        if len(ceil) == len(mats) else None,
        graph_launch_check=L.rf4.launch_count() - launches0)
    if with_e2e:
        ne = max(10, args.steps // 4)
        te, h2d, d2h = e2e_rate(L, ne, args.warmup, world)
        te = max_over_ranks(te, world)
        tc, _, _ = e2e_rate(L, ne, args.warmup, world, staged=False)
        tc = max_over_ranks(tc, world)
        res["e2e"] = {"value": round(world * sb * ne / te / 1e9, 1), "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "transfers": "rocmfp4_copy (staging kernel in the chain of dependent launches) from and to "
                                   "pinned host buffers, every step",
                      "copy_engine_GB/s": round(world * sb * ne / tc / 1e9, 1)}
    del L
    torch.cuda.empty_cache()
    return res


# ---- fused gate/up GEMV -----------------------------------------------------------------------

GATE_UP = (17408, 5120)  # I, K of the layer's gate+up matrix (2I = 34816 rows)


def gate_up_bytes(I, K, variant=0, M=1):
    """Algorithmic bytes of one fused gate/up product: 2I weight rows, M activation
    rows in, M x I outputs."""
    return matrix_bytes(2 * I, K, variant) + 2 * M * K + 4 * M * I


def run_gate_up(hbm, reps=16):
    """Fused gate/up product (Y = SiLU(gate . x) * (up . x)) on the layer's gate+up
    matrix, batch 1, dual, x fp16: average device time per launch of a CUDA graph of
    `reps` launches rotating over resident copies (every launch streams from HBM),
    beside the plain GEMV of the same matrix (2I outputs, no epilogue)."""
    import torch

    import gemm_rocmfp4_dequant_gb300 as rf4
    import synth
    import synth.device
    I, K = GATE_UP
    copies = max(2, int(np.ceil(4 * L2_BYTES / matrix_bytes(2 * I, K))) + 1)
    W, X, Yf, Yp = [], [], [], []
    for r in range(copies):
        w = torch.empty(2 * I * rf4.row_bytes(K, 0), dtype=torch.uint8, device="cuda")
        synth.device.fill_weights(w, 2 * I, K, 0, seed=r, stream=synth.weight_stream(0, 2))
        x = torch.empty((1, K), dtype=torch.int16, device="cuda")
        synth.device.fill_act(x, 0, seed=r, stream=synth.act_stream(0, 2))
        W.append(w)
        X.append(x.view(torch.float16))
        Yf.append(torch.empty((1, I), dtype=torch.float32, device="cuda"))
        Yp.append(torch.empty((1, 2 * I), dtype=torch.float32, device="cuda"))
    rf4.gemv_gate_up(W[0], X[0], I, K, 0, Y=Yf[0])
    rf4.gemm(W[0], X[0], 2 * I, K, 0, Y=Yp[0])
    torch.cuda.synchronize()

    def per_launch(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                fn(i % copies)
        g.replay()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(5):
            g.replay()
        e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / (5 * reps)

    launches0 = rf4.launch_count()
    tf = per_launch(lambda r: rf4.gemv_gate_up(W[r], X[r], I, K, 0, Y=Yf[r]))
    tp = per_launch(lambda r: rf4.gemm(W[r], X[r], 2 * I, K, 0, Y=Yp[r]))
    assert rf4.launch_count() - launches0 == 2 * reps  # one launch per call while capturing
    b = gate_up_bytes(I, K)
    out = {"kernel": "gemv_stream_kernel, gate/up epilogue", "I": I, "K": K, "variant": "dual", "M": 1,
           "act": "fp16", "us": round(tf * 1e6, 2), "GB/s": round(b / tf / 1e9, 1), "peak": hbm,
           "frac": round(b / tf / 1e9 / hbm, 4), "algorithmic_bytes": b,
           "plain_gemv_us": round(tp * 1e6, 2), "copies": copies,
           "note": "plain_gemv_us: the same matrix as one GEMV of 2I outputs (SiLU*mul not applied)"}
    del W, X, Yf, Yp
    torch.cuda.empty_cache()
    return out


# ---- decode attention over a ROCmFP4 K/V cache ------------------------------------------------

ATTN_HEADS = (40, 8, 128)  # query heads, KV heads, head dim of the layer (5120 = 40 x 128; 1024 KV = 8 x 128)
ATTN_CASES = ((1, 32768), (16, 4096))  # (sequences, tokens each)


def attention_bytes(B, T, H=40, Hkv=8, D=128, variant=0):
    """Algorithmic bytes of one decode-attention call with every sequence T tokens
    long: the K and V rows read once, q in, out written."""
    return 2 * B * Hkv * T * (D // 32) * block_bytes(variant) + 2 * B * H * D + 4 * B * H * D


def run_attention(hbm, reps=16):
    """Decode attention (one query token per sequence, dual ROCmFP4 K/V, q fp16):
    device time per call of a CUDA graph of `reps` calls rotating over resident
    caches (every call streams its cache from HBM)."""
    import torch

    import gemm_rocmfp4_dequant_gb300 as rf4
    import synth.device
    H, Hkv, D = ATTN_HEADS
    out = {}
    for B, T in ATTN_CASES:
        kv = B * Hkv * T * rf4.row_bytes(D, 0)
        copies = max(2, int(np.ceil(4 * L2_BYTES / (2 * kv))) + 1)
        Ks, Vs, Qs, Os = [], [], [], []
        for r in range(copies):
            k = torch.empty(kv, dtype=torch.uint8, device="cuda")
            v = torch.empty(kv, dtype=torch.uint8, device="cuda")
            synth.device.fill_weights(k, B * Hkv * T, D, 0, seed=r, stream=synth.weight_stream(0, 5))
            synth.device.fill_weights(v, B * Hkv * T, D, 0, seed=r, stream=synth.weight_stream(0, 6))
            q = torch.empty((B, H, D), dtype=torch.int16, device="cuda")
            synth.device.fill_act(q, 0, seed=r, stream=synth.act_stream(0, 5))
            Ks.append(k)
            Vs.append(v)
            Qs.append(q.view(torch.float16))
            Os.append(torch.empty((B, H, D), dtype=torch.float32, device="cuda"))
        lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
        scale = 1.0 / np.sqrt(D)
        rf4.decode_attention(Qs[0], Ks[0], Vs[0], lens, Hkv, T, scale, 0, out=Os[0])
        torch.cuda.synchronize()
        launches0 = rf4.launch_count()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                r = i % copies
                rf4.decode_attention(Qs[r], Ks[r], Vs[r], lens, Hkv, T, scale, 0, out=Os[r])
        per_call = (rf4.launch_count() - launches0) / reps
        g.replay()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(5):
            g.replay()
        e1.record(st)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / (5 * reps)
        b = attention_bytes(B, T, H, Hkv, D)
        out[f"B={B} T={T}"] = {"us": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4),
                               "algorithmic_bytes": b, "launches_per_call": per_call, "copies": copies}
        del g, Ks, Vs, Qs, Os
        torch.cuda.empty_cache()
    return {"kernel": "attn_split_kernel + attn_combine_kernel", "heads": H, "kv_heads": Hkv, "head_dim": D,
            "variant": "dual", "act": "fp16", "peak": hbm, "cases": out}


# ---- quantiser -----------------------------------------------------------------------------------

def quantize_bytes(N, K, variant=0):
    """Algorithmic bytes of quantising N x K 16-bit values: read once, blocks written once."""
    return 2 * N * K + matrix_bytes(N, K, variant)


def run_quantize(hbm, reps=8):
    """bf16 -> dual ROCmFP4 of the layer's gate+up matrix [34816, 5120]: device
    time per call of a CUDA graph of `reps` calls over resident sources
    (356 MB each, larger than L2)."""
    import torch

    import gemm_rocmfp4_dequant_gb300 as rf4
    N, K = 34816, 5120
    copies = 2
    gen = torch.Generator(device="cuda").manual_seed(0)
    srcs = [torch.randn((N, K), dtype=torch.float32, device="cuda", generator=gen).to(torch.bfloat16)
            for _ in range(copies)]
    outs = [torch.empty(N * rf4.row_bytes(K, 0), dtype=torch.uint8, device="cuda") for _ in range(copies)]
    rf4.quantize(srcs[0], 0, W=outs[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            rf4.quantize(srcs[i % copies], 0, W=outs[i % copies])
    g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(3):
        g.replay()
    e1.record(st)
    e1.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / (3 * reps)
    b = quantize_bytes(N, K)
    del g, srcs, outs
    torch.cuda.empty_cache()
    return {"kernel": "quantize_kernel", "N": N, "K": K, "src": "bf16", "variant": "dual", "us": round(t * 1e6, 2),
            "GB/s": round(b / t / 1e9, 1), "peak": hbm, "frac": round(b / t / 1e9 / hbm, 4), "algorithmic_bytes": b}


# ---- prefill GEMM ---------------------------------------------------------------------------

def run_prefill(Ms, tflops_peak, reps_small=10, reps_large=3):
    """W4A16 prefill GEMM (dual weights, X bf16 [M, K] ~ N(0,1), Y fp32) over the four
    layer shapes for each M: every call is timed alone between CUDA events, with L2
    flushed before it (outside the events).  Returns per-M totals and per-shape times."""
    import torch

    import gemm_rocmfp4_dequant_gb300 as rf4
    import synth.device
    flush = L2Flush()
    out = {}
    launches = 0
    for M in Ms:
        tot_f, tot_t, shapes = 0.0, 0.0, {}
        for m, (name, N, K) in enumerate(LAYER):
            W = torch.empty(N * rf4.row_bytes(K, 0), dtype=torch.uint8, device="cuda")
            synth.device.fill_weights(W, N, K, 0, seed=0, stream=synth.weight_stream(0, m))
            X = torch.empty((M, K), dtype=torch.int16, device="cuda")
            synth.device.fill_act(X, 1, seed=0, stream=synth.act_stream(0, m))
            X = X.view(torch.bfloat16)
            Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            for _ in range(2):
                rf4.gemm(W, X, N, K, 0, Y=Y)
            reps = reps_small if M <= 4096 else reps_large
            s = torch.cuda.current_stream()
            times = []
            for _ in range(reps):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                rf4.gemm(W, X, N, K, 0, Y=Y)
                b.record(s)
                b.synchronize()
                times.append(a.elapsed_time(b) / 1e3)
            launches += reps + 2
            t = float(np.median(times))
            f = 2.0 * M * N * K
            shapes[name] = {"us": round(t * 1e6, 1), "tflops": round(f / t / 1e12, 1)}
            tot_f += f
            tot_t += t
            del W, X, Y
            torch.cuda.empty_cache()
        out[M] = {"tflops": round(tot_f / tot_t / 1e12, 1), "frac": round(tot_f / tot_t / 1e12 / tflops_peak, 4),
                  "layer_ms": round(tot_t * 1e3, 3), "per_shape": shapes}
    del flush
    torch.cuda.empty_cache()
    return out, launches


# ---- single GEMV latency (N=256, K=1024) ------------------------------------------------------

def run_single(args, world):
    import torch

    import gemm_rocmfp4_dequant_gb300 as rf4
    import synth.device
    N, K = 256, 1024
    W = torch.empty(N * rf4.row_bytes(K, 0), dtype=torch.uint8, device="cuda")
    synth.device.fill_weights(W, N, K, 0, seed=0, stream=0)
    x = torch.empty((1, K), dtype=torch.int16, device="cuda")
    synth.device.fill_act(x, 0, seed=0, stream=synth.act_stream(0, 0))
    x = x.view(torch.float16)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    flush = L2Flush()
    for _ in range(args.warmup):
        rf4.gemm(W, x, N, K, 0, Y=y)
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.current_stream()
    times = []
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            rf4.gemm(W, x, N, K, 0, Y=y)
            b.record(s)
            b.synchronize()
            times.append(a.elapsed_time(b) / 1e3)
    t = max_over_ranks(float(np.sum(times)), world)
    sb = step_bytes([("single", N, K)])
    return dict(value=world * sb * args.steps / t / 1e9, ms_per_step=t / args.steps * 1e3, clocks=clk.summary(),
                us_median=round(float(np.median(times)) * 1e6, 2), gpu_launches=args.steps, step_bytes=sb)


# ---- whole-model decode step (config: 64 layers x 4 matrices + LM head) --------------------------

def parse_layouts(text):
    """Block layout per tensor role, "role=dual|fast,..." over the roles qkv, o,
    gate_up, down, lm_head; roles not named are dual."""
    out = {r: 0 for r in ROLES}
    for item in filter(None, (text or "").split(",")):
        role, _, v = item.partition("=")
        if role not in out or v not in ("dual", "fast"):
            raise SystemExit(f"--layouts: bad item {item!r} (roles {', '.join(ROLES)}; layouts dual, fast)")
        out[role] = 0 if v == "dual" else 1
    return out


def role_of(name):
    return name.split(".")[-1]


class ModelStep:
    """All weights resident (12.5 GB all dual); one CUDA graph of 257 GEMV launches
    per token, each with its own activation vector (outputs are not chained).
    Each matrix takes the block layout that `layouts` gives its tensor role."""

    def __init__(self, layouts=None):
        import torch

        import gemm_rocmfp4_dequant_gb300 as rf4
        import synth
        import synth.device
        self.rf4 = rf4
        self.layouts = layouts or {r: 0 for r in ROLES}
        self.mats = [(f"l{l}.{n}", N, K) for l in range(N_LAYERS) for (n, N, K) in LAYER] + [LM_HEAD]
        self.variants = [self.layouts[role_of(n)] for n, _, _ in self.mats]
        self.W, self.X, self.Y = [], [], []
        for i, (name, N, K) in enumerate(self.mats):
            layer, m = (i // 4, i % 4) if i < 4 * N_LAYERS else (N_LAYERS, 4)
            variant = self.variants[i]
            w = torch.empty(N * rf4.row_bytes(K, variant), dtype=torch.uint8, device="cuda")
            synth.device.fill_weights(w, N, K, variant, seed=0, stream=synth.weight_stream(layer, m))
            x = torch.empty((1, K), dtype=torch.int16, device="cuda")
            synth.device.fill_act(x, 0, seed=0, stream=synth.act_stream(layer, m))
            self.W.append(w)
            self.X.append(x.view(torch.float16))
            self.Y.append(torch.empty((1, N), dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run()
        torch.cuda.synchronize()

    def run(self):
        for (name, N, K), v, w, x, y in zip(self.mats, self.variants, self.W, self.X, self.Y):
            self.rf4.gemm(w, x, N, K, v, Y=y)


def run_model(args, world):
    import torch
    S = ModelStep(parse_layouts(args.layouts))
    with ClockSampler(torch.cuda.current_device()) as clk:
        t = time_steps(lambda i: S.graph.replay(), args.steps, args.warmup, world)
    t = max_over_ranks(t, world)
    sb = sum(step_bytes([m], v) for m, v in zip(S.mats, S.variants))
    res = dict(value=world * sb * args.steps / t / 1e9, ms_per_step=t / args.steps * 1e3, clocks=clk.summary(),
               tok_s=world * args.steps / t, gpu_launches=len(S.mats) * args.steps, step_bytes=sb,
               launches_per_step=len(S.mats),
               weight_gb=round(sum(weight_bytes([m], v) for m, v in zip(S.mats, S.variants)) / 1e9, 3))
    del S
    torch.cuda.empty_cache()
    return res


def model_object(args, world, hbm, peak_kind):
    """The whole-model decode step (257 GEMVs, one CUDA graph per token) for the
    default line: equivalent decode tok/s and GB/s against the HBM copy peak."""
    r = run_model(argparse.Namespace(steps=args.steps, warmup=args.warmup, layouts=""), world)
    return {"kernel": "gemv_stream_kernel", "workload": "64 layers x [7168,5120] [5120,6144] [34816,5120] "
            "[5120,17408] + LM head [152064,5120], dual, batch 1, fresh x fp16 per GEMV",
            "tok_s": round(r["tok_s"], 1), "GB/s": round(r["value"], 1), "peak": hbm,
            "frac": round(r["value"] / hbm, 4), "frac_of": f"{peak_kind} HBM copy bandwidth",
            "ms_per_step": round(r["ms_per_step"], 4), "step_bytes": r["step_bytes"], "weight_gb": r["weight_gb"],
            "launches_per_step": r["launches_per_step"],
            "us_per_launch": round(r["ms_per_step"] * 1e3 / r["launches_per_step"], 3),
            "steps": args.steps, "clocks": r["clocks"]}


def run_sweep(args, world, hbm):
    """The four layer shapes x {dual, single-scale} x M in {1, 2, 4, 8}: GB/s of
    each variant's layer step (one graph of four launches)."""
    table = {}
    for variant in (0, 1):
        for M in (1, 2, 4, 8):
            r = run_gemv(argparse.Namespace(steps=max(20, args.steps // 10), warmup=args.warmup), world, hbm,
                         LAYER, variant=variant, M=M, with_e2e=False, with_ceiling=False)
            table[f"{'dual' if variant == 0 else 'fast'} M={M}"] = {
                "GB/s": round(r["value"], 1), "frac": round(r["value"] / hbm, 4),
                "kernel_GB/s": round(r["achieved"], 1), "per_launch_us": r["per_launch_us"]}
    return table


# ---- main -----------------------------------------------------------------------------------

def base_line(args, world, value, unit, ms, cfg, dtype, higher=True):
    return {"metric": METRIC, "value": round(value, 4 if value < 10 else 1), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": higher,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": DATA, "config": cfg,
            "parallelism": "replicas" if world > 1 else "single GPU"}


def reference_line(args, cfg):
    """The oracle, as it stands, on the host cores: each step a bounded sample."""
    t0 = time.perf_counter()
    # one probe sizes the sample so that all steps together take about 150 s
    per_step = 150.0 / (args.steps + args.warmup)
    cores = os.cpu_count() or 1
    if args.workload == "prefill":
        fn = lambda rows=None, b=1.0: cpu_oracle_flops(LAYER, 4096, budget_s=b, rows=rows)
    elif args.workload == "single":
        fn = lambda rows=None, b=1.0: cpu_oracle_rate([("single", 256, 1024)], budget_s=b, rows=rows)
    else:
        fn = lambda rows=None, b=1.0: cpu_oracle_rate(LAYER, budget_s=b, rows=rows)
    _, _, _, tp = fn(rows=cores)
    rows = max(1, int(cores * per_step / max(tp, 1e-4)))
    vals, desc = [], ""
    for _ in range(args.warmup + args.steps):
        v, cores, desc, _ = fn(rows=rows)
        vals.append(v)
    v = float(np.mean(vals[args.warmup:]))
    unit = "TFLOP/s" if args.workload == "prefill" else "GB/s"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": DATA, "config": dict(cfg, l2="host run"),
            "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t0, 1)}
    if unit == "GB/s":
        sb = step_bytes(LAYER if args.workload != "single" else [("single", 256, 1024)])
        line["ms_per_step"] = round(sb / (v * 1e9) * 1e3, 3)
    return line


def gemv_roofline(res, hbm, peak_kind, mats, variant, M):
    traffic = gemv_traffic() if (mats == LAYER and variant == 0 and M == 1) else None
    roof = {"bound": "hbm", "achieved": round(res["achieved"], 1), "peak": hbm, "unit": "GB/s",
            "frac": round(res["achieved"] / hbm, 4), "traffic": None,
            "kernel": "gemv_stream_kernel", "peak_kind": peak_kind, "frac_of": f"{peak_kind} HBM copy bandwidth",
            "per_launch_us": res["per_launch_us"],
            "algorithmic_bytes_per_launch": res["algo_bytes"]}
    if res.get("read_ceiling_us"):
        roof["read_ceiling"] = {"us": res["read_ceiling_us"], "GB/s": res["read_ceiling_gbs"],
                                "note": "a plain read of each matrix's bytes (ceiling/read.cu: bulk copies into shared "
                                        "memory, XOR checksum of every word; fastest of four grid shapes), same graph "
                                        "and copies: what one launch of that size reaches without decode or arithmetic"}
    if traffic and all(n in traffic for n, _, _ in mats):
        roof["traffic"] = int(round(sum(traffic[n] for n, _, _ in mats) / len(mats)))
        roof["traffic_per_launch"] = {n: traffic[n] for n, _, _ in mats}
        roof["traffic_note"] = "mean DRAM read+write bytes per launch over the four matrices (ncu)"
    return roof


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="layer",
                    choices=["layer", "single", "sweep", "model", "prefill", "gate_up", "attention", "quantize"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layouts", default="", help="model workload: block layout per tensor role, "
                    "e.g. qkv=dual,o=dual,gate_up=fast,down=fast,lm_head=dual (default: all dual)")
    ap.add_argument("--no-prefill", action="store_true", help="leave the prefill object out of the layer line")
    ap.add_argument("--no-model", action="store_true", help="leave the whole-model object out of the layer line")
    ap.add_argument("--no-sweep", action="store_true", help="leave the variant sweep out of the layer line")
    ap.add_argument("--prefill-m", type=str, default=",".join(str(m) for m in PREFILL_M),
                    help="comma-separated token counts of the prefill GEMM")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    hbm, bf16, bf16_s, peak_kind = peaks()
    cfgs = {
        "layer": {"workload": "layer sweep: batch-1 dual-scale GEMV, [N,K] = [7168,5120] [5120,6144] "
                              "[34816,5120] [5120,17408], x fp16 ~ N(0,1), one launch per matrix",
                  "variant": "dual", "M": 1, "act": "fp16"},
        "single": {"workload": "single dual-scale GEMV N=256 K=1024, x fp16 ~ N(0,1)", "variant": "dual", "M": 1,
                   "act": "fp16", "l2": "flushed (256 MB write) before every timed call"},
        "sweep": {"workload": "the four layer shapes x {dual, single-scale} x M in {1,2,4,8}, x fp16",
                  "act": "fp16"},
        "model": {"workload": "whole-model decode step: 64 layers x 4 matrices + LM head [152064,5120], dual, "
                              "batch 1, fresh x fp16 per GEMV, one CUDA graph of 257 launches per token",
                  "variant": "dual", "M": 1, "act": "fp16", "l2": "12.5 GB of weights per step > L2"},
        "prefill": {"workload": "W4A16 prefill GEMM, dual weights of the four layer shapes x X bf16 [M,K] ~ N(0,1), "
                                "M in {512, 4096, 23552}", "act": "bf16",
                    "l2": "flushed (256 MB write) before every timed call"},
        "gate_up": {"workload": "fused gate/up GEMV, [2 x 17408, 5120] dual, batch 1, x fp16 ~ N(0,1)",
                    "l2": "rotating resident copies larger than 4 x L2"},
        "attention": {"workload": "decode attention over a dual ROCmFP4 K/V cache, 40 heads / 8 KV heads / D 128, "
                                  "1 x 32768 and 16 x 4096 tokens, q fp16 ~ N(0,1)",
                      "l2": "rotating resident caches larger than 4 x L2"},
        "quantize": {"workload": "quantiser bf16 [34816, 5120] ~ N(0,1) -> dual ROCmFP4",
                     "l2": "two resident 356 MB sources, larger than L2"},
    }
    cfg = cfgs[args.workload]
    if args.workload == "model" and args.layouts:
        lay = parse_layouts(args.layouts)
        names = ",".join(f"{r}={'dual' if v == 0 else 'fast'}" for r, v in lay.items())
        cfg = dict(cfg, workload=cfg["workload"].replace(", dual,", f", layouts {names},"), variant="per role")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_line(args, cfg)))
        return

    import torch

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    import gemm_rocmfp4_dequant_gb300 as rf4

    if args.workload == "layer":
        res = run_gemv(args, world, hbm, LAYER)
        cfg["l2"] = (f"rotating {res['copies']} resident layer copies ({res['footprint_gb']} GB > 129 MB L2); "
                     "inputs larger than L2")
        cfg["graphs"] = (f"one CUDA graph holds one layer pass per resident copy ({res['copies']} passes, "
                         f"{4 * res['copies']} PDL launches); steps replay it")
        line = base_line(args, world, res["value"], "GB/s", res["ms_per_step"], cfg, "f16")
        line["roofline"] = gemv_roofline(res, hbm, peak_kind, LAYER, 0, 1)
        line["e2e"] = res["e2e"]
        line["gpu_launches"] = res["gpu_launches"]
        line["clocks"] = res["clocks"]
        line["frac_of_hbm_peak"] = round(res["value"] / hbm, 4)
        if not args.no_model:
            line["model"] = model_object(args, world, hbm, peak_kind)
        if not args.no_sweep:
            line["sweep"] = run_sweep(args, world, hbm)
        line["gate_up"] = run_gate_up(hbm)
        line["attention"] = run_attention(hbm)
        line["quantize"] = run_quantize(hbm)
        if not args.no_prefill:
            pre, _ = run_prefill([int(m) for m in args.prefill_m.split(",")], bf16)
            line["prefill"] = {"unit": "TFLOP/s", "dtype": "bf16", "peak": bf16, "peak_kind": f"{peak_kind} bf16 burst",
                               "kernel": "gemm_tc_kernel", "bound": "tensor",
                               "by_M": {str(m): v for m, v in pre.items()}}
        if rank == 0 and not args.no_cpu_baseline:
            v, cores, desc, tt = cpu_oracle_rate(LAYER, budget_s=12.0)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                    "sample": desc + f" ({tt:.1f} s)"}
    elif args.workload == "single":
        res = run_single(args, world)
        line = base_line(args, world, res["value"], "GB/s", res["ms_per_step"], cfg, "f16")
        line.update(us_median=res["us_median"], gpu_launches=res["gpu_launches"], clocks=res["clocks"])
    elif args.workload == "model":
        res = run_model(args, world)
        line = base_line(args, world, res["value"], "GB/s", res["ms_per_step"], cfg, "f16")
        line.update(tok_s=round(res["tok_s"], 1), gpu_launches=res["gpu_launches"], clocks=res["clocks"],
                    weight_gb=res["weight_gb"], frac_of_hbm_peak=round(res["value"] / hbm, 4))
    elif args.workload == "sweep":
        table = run_sweep(args, world, hbm)
        first = table["dual M=1"]
        line = base_line(args, world, first["GB/s"], "GB/s", 0.0, cfg, "f16")
        line["sweep"] = table
    elif args.workload in ("gate_up", "attention", "quantize"):
        launches0 = rf4.launch_count()
        if args.workload == "gate_up":
            r = run_gate_up(hbm)
            v, ms = r["GB/s"], r["us"] / 1e3
        elif args.workload == "attention":
            r = run_attention(hbm)
            head = r["cases"]["B=1 T=32768"]
            v, ms = head["GB/s"], head["us"] / 1e3
        else:
            r = run_quantize(hbm)
            v, ms = r["GB/s"], r["us"] / 1e3
        line = base_line(args, world, v, "GB/s", ms, cfg, "f16" if args.workload != "quantize" else "bf16")
        line["roofline"] = {"bound": "hbm", "achieved": v, "peak": hbm, "unit": "GB/s", "frac": round(v / hbm, 4),
                            "traffic": None, "peak_kind": peak_kind}
        line["detail"] = r
        line["gpu_launches"] = rf4.launch_count() - launches0
    else:  # prefill
        Ms = [int(m) for m in args.prefill_m.split(",")]
        pre, launches = run_prefill(Ms, bf16)
        head = 4096 if 4096 in pre else Ms[0]
        v = pre[head]["tflops"]
        line = base_line(args, world, v, "TFLOP/s", pre[head]["layer_ms"], dict(cfg, headline=f"M={head}"), "bf16")
        line["roofline"] = {"bound": "tensor", "achieved": v, "peak": bf16, "unit": "TFLOP/s",
                            "frac": round(v / bf16, 4), "traffic": None, "kernel": "gemm_tc_kernel",
                            "peak_kind": f"{peak_kind} bf16 burst"}
        line["by_M"] = {str(m): r for m, r in pre.items()}
        line["gpu_launches"] = launches
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
