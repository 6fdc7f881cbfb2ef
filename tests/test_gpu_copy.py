"""GPU tests of rocmfp4_copy, the staging copy between pinned host memory and
the device.

Bytes must arrive exactly, in every direction, at aligned and unaligned
addresses and ragged sizes.  Inside a chain of dependent launches the copy
must see what the preceding product wrote (it reads nothing before that
kernel has completed) and must not overwrite an input that the preceding
product still reads: a step loop with fresh inputs every step is compared,
output by output, with the same loop on copy-engine transfers, and with the
fp64 oracle.  Pageable host memory is refused on the host.
"""
import ctypes

import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
from gpu_util import assert_close, max_halfscale, torch, upload_w

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 16, 17, 4099, 67584, 208896, (1 << 20) + 5]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def pattern(n, seed):
    return np.random.default_rng(seed).integers(0, 256, size=n, dtype=np.uint8)


def buffer(n, where):
    t = torch()
    if where == "host":
        return t.zeros(n, dtype=t.uint8).pin_memory()
    return t.zeros(n, dtype=t.uint8, device="cuda")


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (0, 3), (5, 5)])
def test_bytes_arrive_exactly(direction, n, offsets):
    t = torch()
    so, do = offsets
    src_where, dst_where = {"h2d": ("host", "cuda"), "d2h": ("cuda", "host"), "d2d": ("cuda", "cuda")}[direction]
    data = pattern(n, seed=n + 7 * so + do)
    src = buffer(n + so, src_where)
    src[so:].copy_(t.from_numpy(data))
    dst = buffer(n + do + 8, dst_where)
    guard = 0xA5
    dst.fill_(guard)
    t.cuda.synchronize()
    rf4.copy(dst[do:do + n], src[so:])
    t.cuda.synchronize()
    got = dst.cpu().numpy()
    assert np.array_equal(got[do:do + n], data)
    assert (got[:do] == guard).all() and (got[do + n:] == guard).all()


def test_pageable_host_memory_is_refused():
    t = torch()
    L = rf4.load()
    pageable = np.zeros(64, dtype=np.uint8)
    dev = t.zeros(64, dtype=t.uint8, device="cuda")
    st = L.rocmfp4_copy(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(pageable.ctypes.data), 64, None)
    assert st == 1 and b"pageable" in L.rocmfp4_last_error()
    with pytest.raises(ValueError):
        rf4.copy(dev, t.zeros(64, dtype=t.uint8))


@pytest.mark.parametrize("variant", [rf4.DUAL, rf4.FAST])
def test_step_loop_with_staged_inputs_and_outputs(variant):
    """Steps of (copy in, three products, copy out) on one stream with fresh
    inputs each step: every step's outputs are its own, as with copy-engine
    transfers, and match the oracle."""
    t = torch()
    shapes = [(1000, 1024), (256, 2048), (4096, 512)]
    Ws, Wh = [], []
    for i, (N, K) in enumerate(shapes):
        h = synth.weights(N, K, variant, seed=5, stream=3000 + i)
        Wh.append(h)
        Ws.append(upload_w(h))
    xs = [K for N, K in shapes]
    ys = [N for N, K in shapes]
    steps = 6
    hx = []
    for s in range(steps):
        bits = np.concatenate([synth.activations(1, K, synth.ACT_F16, seed=100 + s, stream=3100 + i).reshape(-1)
                               for i, (N, K) in enumerate(shapes)])
        hx.append(t.from_numpy(bits.view(np.int16)).view(t.float16).pin_memory())
    dx = t.empty(sum(xs), dtype=t.float16, device="cuda")
    dy = t.empty(sum(ys), dtype=t.float32, device="cuda")
    xv = [v.view(1, K) for v, K in zip(t.split(dx, xs), xs)]
    yv = [v.view(1, N) for v, N in zip(t.split(dy, ys), ys)]

    def run(staged):
        out = [t.full((sum(ys),), float("nan"), dtype=t.float32).pin_memory() for _ in range(steps)]
        for s in range(steps):
            if staged:
                rf4.copy(dx, hx[s])
            else:
                dx.copy_(hx[s], non_blocking=True)
            for (N, K), W, x, y in zip(shapes, Ws, xv, yv):
                rf4.gemm(W, x, N, K, variant, Y=y)
            if staged:
                rf4.copy(out[s], dy)
            else:
                out[s].copy_(dy, non_blocking=True)
        t.cuda.synchronize()
        return [o.numpy().copy() for o in out]

    ref = run(False)
    got = run(True)
    for s in range(steps):
        assert np.array_equal(got[s], ref[s]), f"step {s}"
        xb = hx[s].view(t.int16).numpy().view(np.uint16)
        o = 0
        for i, (N, K) in enumerate(shapes):
            xo = sum(xs[:i])
            yref = oracle.gemm(Wh[i], xb[xo:xo + K].reshape(1, K), N, K, variant, act=synth.ACT_F16)
            assert_close(got[s][o:o + N].reshape(1, N), yref, K, max_halfscale(Wh[i], variant), f"step {s} product {i}")
            o += N


def test_step_captured_in_a_graph():
    """The same step (copy in, product, copy out) captured once in a CUDA graph
    and replayed with new host inputs: every replay sees its own inputs and
    hands back its own outputs."""
    t = torch()
    N, K, variant = 1000, 1024, rf4.DUAL
    Wh = synth.weights(N, K, variant, seed=9, stream=3200)
    W = upload_w(Wh)
    hx = t.empty(K, dtype=t.float16).pin_memory()
    hy = t.full((N,), float("nan"), dtype=t.float32).pin_memory()
    dx = t.empty((1, K), dtype=t.float16, device="cuda")
    dy = t.empty((1, N), dtype=t.float32, device="cuda")

    def step():
        rf4.copy(dx, hx)
        rf4.gemm(W, dx, N, K, variant, Y=dy)
        rf4.copy(hy, dy)

    s = t.cuda.Stream()
    s.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(s):
        step()  # the library's one-time set-up happens outside the capture
    t.cuda.current_stream().wait_stream(s)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g):
        step()
    for rep in range(3):
        bits = synth.activations(1, K, synth.ACT_F16, seed=200 + rep, stream=3300)
        hx.copy_(t.from_numpy(bits.reshape(-1).view(np.int16)).view(t.float16))
        hy.fill_(float("nan"))
        g.replay()
        t.cuda.synchronize()
        yref = oracle.gemm(Wh, bits, N, K, variant, act=synth.ACT_F16)
        assert_close(hy.numpy().reshape(1, N), yref, K, max_halfscale(Wh, variant), f"replay {rep}")
