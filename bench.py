"""Benchmark of the GB300 ROCmFP4 library.

Default workload ("layer"): one dense decoder layer's four dual-scale ROCmFP4
matrices -- [N, K] = [7168, 5120] (fused QKV), [5120, 6144] (O), [34816, 5120]
(fused gate+up), [5120, 17408] (down) -- each multiplied by a batch-1 fp16
activation vector ~ N(0, 1).  One step = the four GEMVs.  Steps rotate over
enough resident copies of the layer that the working set is far larger than
L2, so every step streams its weights from HBM.

Metric: weight-streaming GB/s = (packed weight bytes + activation bytes +
output bytes) per step / step time, with the roofline of the dominant kernel
against the measured HBM copy bandwidth.

Other workloads (--workload): single (N=256, K=1024), sweep (both layouts x
M in {1,2,4,8}), model (64 layers x 4 matrices + LM head [152064, 5120], one
CUDA graph per token), prefill (M in {512, 4096, 23552}).

--impl reference times the CPU oracle (the fp64 C implementation under
oracle/) on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYER = [("qkv", 7168, 5120), ("o", 5120, 6144), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
LM_HEAD = ("lm_head", 152064, 5120)
N_LAYERS = 64
L2_BYTES = 129 * 1024 * 1024
METRIC = "ROCmFP4 GEMV weight GB/s (% of HBM peak); W4A16 GEMM TFLOP/s (% peak)"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def step_bytes(mats, variant=0, M=1):
    bb = 18 if variant == 0 else 17
    return sum(N * (K // 32) * bb + 2 * M * K + 4 * M * N for _, N, K in mats)


def weight_bytes(mats, variant=0):
    bb = 18 if variant == 0 else 17
    return sum(N * (K // 32) * bb for _, N, K in mats)


# ---- clocks -------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


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

def cpu_oracle_rate(mats, variant, M, budget_s=12.0, act=0):
    """Times the oracle on row samples of each matrix; returns (GB/s of the metric, cores, sample text, seconds).

    The sample size is chosen from a short probe so that the timed run takes
    about budget_s seconds; the metric counts the sampled rows' packed bytes
    plus their share of activation and output bytes."""
    import oracle
    import synth
    cores = os.cpu_count() or 1
    inputs = []
    for idx, (name, N, K) in enumerate(mats):
        inputs.append((N, K, synth.activations(M, K, act, seed=0, stream=synth.act_stream(0, idx))))

    def run(rows_per):
        nbytes, secs = 0.0, 0.0
        for idx, (N, K, Xh) in enumerate(inputs):
            rows = np.arange(min(rows_per, N))
            Wr = synth.weights(N, K, variant, seed=0, stream=synth.weight_stream(0, idx), rows=rows)
            t0 = time.perf_counter()
            oracle.gemm(Wr, Xh, len(rows), K, variant, act=act, nthreads=cores)
            secs += time.perf_counter() - t0
            rb = (K // 32) * (18 if variant == 0 else 17)
            nbytes += len(rows) * (rb + 4 * M) + 2 * M * K * len(rows) / N
        return nbytes, secs

    probe_rows = 2 * cores
    b, t = run(probe_rows)
    rows_per = int(max(probe_rows, min(min(N for _, N, _ in mats), probe_rows * budget_s / max(t, 1e-3))))
    b, t = run(rows_per)
    desc = (f"{rows_per} rows of each of the {len(mats)} matrices (M={M}), "
            f"oracle threaded over rows on {cores} cores")
    return b / t / 1e9, cores, desc, t


# ---- GPU workloads -----------------------------------------------------------------------------

class LayerStep:
    """R resident copies of one layer (four matrices); step i runs the four GEMVs of copy i % R."""

    def __init__(self, mats, variant, M, act, copies):
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
                synth.device.fill_weights(w, N, K, variant, seed=r, stream=synth.weight_stream(0, m))
                x = torch.empty((M, K), dtype=torch.int16, device="cuda")
                synth.device.fill_act(x, act, seed=r, stream=synth.act_stream(0, m))
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
            self.run(0, s)  # first call on the device does the library's one-time set-up
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graphs = []
        for r in range(self.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.run(r)
            self.graphs.append(g)
        torch.cuda.synchronize()

    def launches_per_step(self):
        return len(self.mats) * ((self.M + 7) // 8)


def time_steps(step_fn, steps, warmup, world):
    import torch
    for i in range(warmup):
        step_fn(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(steps):
        step_fn(warmup + i)
    b.record()
    b.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    return a.elapsed_time(b) / 1e3


def per_matrix_kernel_times(L: LayerStep, reps=None):
    """Average device time of each matrix's kernel: a CUDA graph of `reps` launches
    of that matrix's product (rotating over the resident copies, so every launch
    streams from HBM) is replayed between CUDA events on the launching stream."""
    import torch
    reps = reps or max(8, 2 * L.copies)
    out = []
    for m, (name, N, K) in enumerate(L.mats):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                r = i % L.copies
                L.rf4.gemm(L.W[r][m], L.X[r][m], N, K, L.variant, Y=L.Y[r][m])
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s = torch.cuda.current_stream()
        e0.record(s)
        for _ in range(3):
            g.replay()
        e1.record(s)
        e1.synchronize()
        out.append(e0.elapsed_time(e1) / 1e3 / (3 * reps))
        del g
    return out


def e2e_rate(L: LayerStep, steps, warmup, world):
    """Same metric through the public API with host buffers: each step copies the four
    activation vectors from pinned host memory, runs the four products and reads the
    four outputs back into pinned host memory; weights stay resident."""
    import torch
    hx = [[x.cpu().pin_memory() for x in Xc] for Xc in L.X]
    hy = [[torch.empty(y.shape, dtype=torch.float32).pin_memory() for y in Yc] for Yc in L.Y]
    dx = [torch.empty_like(x) for x in L.X[0]]
    dy = [torch.empty_like(y) for y in L.Y[0]]
    h2d = sum(x.numel() * x.element_size() for x in dx)
    d2h = sum(y.numel() * 4 for y in dy)

    def one(i):
        r = i % L.copies
        for m, (name, N, K) in enumerate(L.mats):
            dx[m].copy_(hx[r][m], non_blocking=True)
            L.rf4.gemm(L.W[r][m], dx[m], N, K, L.variant, Y=dy[m])
            hy[r][m].copy_(dy[m], non_blocking=True)

    t = time_steps(one, steps, warmup, world)
    return t, h2d, d2h


def run_layer(args, world, rank, hbm, mats=None, variant=0, M=1, act=0, label="layer"):
    import torch
    mats = mats or LAYER
    per_copy = weight_bytes(mats, variant)
    copies = max(2, int(np.ceil(4 * L2_BYTES / per_copy)) + 1)
    L = LayerStep(mats, variant, M, act, copies)
    L.capture()
    launches0 = L.rf4.launch_count()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t = time_steps(lambda i: L.graphs[i % copies].replay(), args.steps, args.warmup, world)
    t = max_over_ranks(t, world)
    sb = step_bytes(mats, variant, M)
    value = world * sb * args.steps / t / 1e9
    kt = per_matrix_kernel_times(L)
    algo = [N * (K // 32) * (18 if variant == 0 else 17) + 2 * M * K + 4 * M * N for _, N, K in mats]
    achieved = sum(algo) / sum(kt) / 1e9
    te, h2d, d2h = e2e_rate(L, max(10, args.steps // 4), args.warmup, world)
    te = max_over_ranks(te, world)
    e2e = world * sb * max(10, args.steps // 4) / te / 1e9
    res = dict(
        value=value, ms_per_step=t / args.steps * 1e3, clocks=clk.summary(),
        gpu_launches=L.launches_per_step() * args.steps,
        graph_launches_check=L.rf4.launch_count() - launches0,
        roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                  "frac": round(achieved / hbm, 4), "traffic": None,
                  "per_launch_us": {n: round(x * 1e6, 2) for (n, _, _), x in zip(mats, kt)}},
        e2e={"value": round(e2e, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        copies=copies, footprint_gb=round(copies * per_copy / 1e9, 3),
    )
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="layer", choices=["layer"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    hbm, bf16, bf16_s, peak_kind = peaks()
    mats = LAYER
    cfg = {"workload": "layer: batch-1 dual-scale GEMV over [7168,5120] [5120,6144] [34816,5120] [5120,17408], "
                       "fp16 x ~ N(0,1)", "variant": "dual", "M": 1, "act": "fp16"}

    if args.impl == "reference":
        if rank != 0:
            return
        t0 = time.perf_counter()
        vals = []
        for _ in range(args.warmup + args.steps):
            v, cores, desc, _ = cpu_oracle_rate(mats, 0, 1, budget_s=min(10.0, 120.0 / (args.steps + args.warmup)))
            vals.append(v)
        v = float(np.mean(vals[args.warmup:]))
        sb = step_bytes(mats)
        line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sb / (v * 1e9) * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded SplitMix64 weights, Box-Muller activations)",
                "config": dict(cfg, l2="CPU run; no GPU L2"),
                "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": round(time.perf_counter() - t0, 1)}
        print(json.dumps(line))
        return

    import torch
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    res = run_layer(args, world, rank, hbm)
    cfg["l2"] = (f"rotating {res['copies']} resident layer copies ({res['footprint_gb']} GB > 129 MB L2); "
                 "inputs larger than L2")
    line = {"metric": METRIC, "value": round(res["value"], 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16 x e2m1 -> f32",
            "data": "synthetic (seeded SplitMix64 weights, Box-Muller activations)", "config": cfg,
            "parallelism": "replicas" if world > 1 else "single GPU",
            "roofline": dict(res["roofline"], peak_kind=peak_kind),
            "e2e": res["e2e"], "gpu_launches": res["gpu_launches"], "clocks": res["clocks"]}
    line["roofline"]["frac_of"] = f"{peak_kind} HBM copy bandwidth"
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, desc, tt = cpu_oracle_rate(mats, 0, 1, budget_s=12.0)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc + f" ({tt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
