"""GPU parity of the whole-model weight-streaming decode step against the oracle.

The workload: 64 decoder layers, each with the fused QKV [7168, 5120], O
[5120, 6144], fused gate+up [34816, 5120] and down [5120, 17408] matrices, and
an LM head [152064, 5120], all in the dual layout (12.5 GB resident); batch 1,
a fresh fp16 activation vector per product (outputs are not chained).  The
step is one CUDA graph of the 257 products, as the benchmark times it.

Weights and activations are filled on the device by the generator's CUDA
twin; on sampled rows of several layers and of the LM head, the device bytes
are compared with the host generator and the outputs with the fp64 oracle
(rel-L2 1e-5, max |err| <= 1e-3 * sqrt(K) * max half-scale).
"""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
import synth.device
from gpu_util import assert_close, max_halfscale, torch

pytestmark = pytest.mark.gpu

DUAL = rf4.DUAL
F16 = synth.ACT_F16
LAYER = [("qkv", 7168, 5120), ("o", 5120, 6144), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
LM_HEAD = ("lm_head", 152064, 5120)
N_LAYERS = 64


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def sample_rows(N, seed, n=40):
    """Both ends of the matrix, both edges of the first and last 32-row tiles, random rows."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 15, 16, 31, 32, N // 2, N - 33, N - 32, N - 17, N - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, N, n)]))


def fill(N, K, layer, m):
    t = torch()
    W = t.empty(N * synth.row_bytes(K, DUAL), dtype=t.uint8, device="cuda")
    synth.device.fill_weights(W, N, K, DUAL, seed=0, stream=synth.weight_stream(layer, m))
    X = t.empty((1, K), dtype=t.int16, device="cuda")
    synth.device.fill_act(X, F16, seed=0, stream=synth.act_stream(layer, m))
    return W, X


def check_rows(W, Y, N, K, layer, m, what):
    t = torch()
    rows = sample_rows(N, 1000 * layer + m)
    rb = synth.row_bytes(K, DUAL)
    Wrows = synth.weights(N, K, DUAL, seed=0, stream=synth.weight_stream(layer, m), rows=rows)
    assert np.array_equal(W.view(N, rb)[t.from_numpy(rows).cuda()].cpu().numpy(), Wrows), f"{what}: generator"
    xh = synth.activations(1, K, F16, seed=0, stream=synth.act_stream(layer, m))
    ref = oracle.gemm(Wrows, xh, len(rows), K, DUAL)
    assert_close(Y.view(1, N)[:, t.from_numpy(rows).cuda()].cpu().numpy(), ref, K, max_halfscale(Wrows, DUAL), what)


def test_lm_head_full_size_sampled_rows():
    """The largest matrix of the model, [152064, 5120] (4752 tiles of 32 rows),
    at M = 1 and, on the same rows, M = 2, 4, 8."""
    t = torch()
    name, N, K = LM_HEAD
    W, X = fill(N, K, N_LAYERS, 4)
    x = X.view(t.float16)
    Y = rf4.gemv(W, x.view(-1), N, K, DUAL)
    check_rows(W, Y, N, K, N_LAYERS, 4, "lm_head M=1")
    rows = sample_rows(N, 7)
    Wrows = synth.weights(N, K, DUAL, seed=0, stream=synth.weight_stream(N_LAYERS, 4), rows=rows)
    for M in (2, 4, 8):
        Xh = synth.activations(M, K, F16, seed=3, stream=synth.act_stream(N_LAYERS, 4))
        XM = t.from_numpy(Xh.view(np.int16)).cuda().view(t.float16)
        YM = rf4.gemm(W, XM, N, K, DUAL).cpu().numpy()
        assert_close(YM[:, rows], oracle.gemm(Wrows, Xh, len(rows), K, DUAL), K, max_halfscale(Wrows, DUAL),
                     f"lm_head M={M}")


def test_whole_model_step_in_one_graph_sampled_rows():
    """All 257 products resident and captured in one CUDA graph; sampled rows of
    every matrix of five layers and of the LM head against the oracle, after
    two replays (the second must repeat the first bitwise)."""
    t = torch()
    mats = [(f"l{l}.{n}", N, K, l, m) for l in range(N_LAYERS) for m, (n, N, K) in enumerate(LAYER)]
    mats.append((LM_HEAD[0], LM_HEAD[1], LM_HEAD[2], N_LAYERS, 4))
    Ws, Xs, Ys = [], [], []
    for name, N, K, l, m in mats:
        W, X = fill(N, K, l, m)
        Ws.append(W)
        Xs.append(X.view(t.float16))
        Ys.append(t.full((1, N), float("nan"), dtype=t.float32, device="cuda"))
    t.cuda.synchronize()

    def run():
        for (name, N, K, l, m), W, X, Y in zip(mats, Ws, Xs, Ys):
            rf4.gemm(W, X, N, K, DUAL, Y=Y)

    s = t.cuda.Stream()
    s.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(s):
        run()  # the first call does the library's one-time set-up outside the capture
    t.cuda.current_stream().wait_stream(s)
    t.cuda.synchronize()
    for Y in Ys:
        Y.fill_(float("nan"))
    g = t.cuda.CUDAGraph()
    launches = rf4.launch_count()
    with t.cuda.graph(g):
        run()
    assert rf4.launch_count() - launches == len(mats) == 257
    g.replay()
    t.cuda.synchronize()
    first = [Y.clone() for Y in Ys]
    g.replay()
    t.cuda.synchronize()
    for a, b in zip(first, Ys):
        assert bool(t.isfinite(b).all())
        assert t.equal(a.view(t.int32), b.view(t.int32))
    for i, (name, N, K, l, m) in enumerate(mats):
        if l in (0, 1, 31, 62, 63, N_LAYERS):
            check_rows(Ws[i], Ys[i], N, K, l, m, name)
