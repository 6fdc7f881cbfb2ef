"""GPU parity of the tensor-core W4A16 product (M > 8) against the fp64 oracle.

Shapes span several 128-row weight tiles and several token tiles, with ragged
tails in M and N.  The full prefill shapes (M = 512, 4096, 23552 over the
four layer matrices) are checked on sampled rows and tokens: weights and
activations are filled on the device by the generator's CUDA twin, whose
bytes are compared with the host generator on the sampled rows, and the
expected values come from the oracle on the host copies of those rows.
"""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
import synth.device
from gpu_util import assert_close, max_halfscale, torch, upload_w, upload_x

pytestmark = pytest.mark.gpu

DUAL, FAST = rf4.DUAL, rf4.FAST
F16, BF16 = synth.ACT_F16, synth.ACT_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def check(Wh, Xh, N, K, variant, act, what):
    Y = rf4.gemm(upload_w(Wh), upload_x(Xh, act), N, K, variant).cpu().numpy()
    ref = oracle.gemm(Wh, Xh, N, K, variant, act=act)
    assert_close(Y, ref, K, max_halfscale(Wh, variant), what)
    return Y


# token counts: one 16-wide tile, ragged tiles, exactly 256, balanced 2- and 3-tile splits
MS = [9, 16, 31, 100, 129, 256, 300, 513]
DUAL_NK = [(128, 256), (200, 1024), (384, 512), (1000, 2048)]
FAST_NK = [(128, 512), (200, 1024), (257, 1536)]


@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("M", MS)
@pytest.mark.parametrize("N,K", DUAL_NK)
def test_dual_matches_oracle(act, M, N, K):
    Wh = synth.weights(N, K, DUAL, seed=11, stream=1000 + N)
    Xh = synth.activations(M, K, act, seed=11, stream=1100 + K)
    check(Wh, Xh, N, K, DUAL, act, f"tc dual M={M} N={N} K={K}")


@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("M", MS)
@pytest.mark.parametrize("N,K", FAST_NK)
def test_fast_matches_oracle(act, M, N, K):
    Wh = synth.weights(N, K, FAST, seed=12, stream=1200 + N)
    Xh = synth.activations(M, K, act, seed=12, stream=1300 + K)
    check(Wh, Xh, N, K, FAST, act, f"tc fast M={M} N={N} K={K}")


@pytest.mark.parametrize("variant", [DUAL, FAST])
def test_single_weight_lands_in_its_row_and_column(variant):
    """One nonzero weight per matrix: Y[:, n] = w * X[:, k] exactly, every other output 0."""
    t = torch()
    N, K, M = 300, 1024, 40
    bb = synth.block_bytes(variant)
    rng = np.random.default_rng(7)
    Xh = synth.activations(M, K, BF16, seed=13, stream=1400)
    X = upload_x(Xh, BF16)
    xf = synth.bits_to_float(Xh, BF16)
    for n, k in ((0, 0), (127, 31), (128, 32), (299, 1023), (200, 517)) + tuple(
            (int(a), int(b)) for a, b in zip(rng.integers(0, N, 6), rng.integers(0, K, 6))):
        Wh = np.zeros((N, K // 32 * bb), dtype=np.uint8)
        blk, i = divmod(k, 32)
        j = i % 16
        Wh[n, blk * bb + j] = 0x3 if i < 16 else 0x30          # code 3 -> 3.0
        Wh[n, blk * bb + 16:(blk + 1) * bb] = 0x40              # E4M3 2.0 -> half-scale 1.0
        Y = rf4.gemm(upload_w(Wh), X, N, K, variant).cpu().numpy()
        expect = np.zeros((M, N))
        expect[:, n] = 3.0 * xf[:, k]
        assert np.array_equal(Y.astype(np.float64), expect), (n, k)
    assert t.cuda.is_available()


def test_zero_weights_give_zero_and_outputs_stay_in_bounds():
    t = torch()
    N, K, M = 250, 512, 77
    for variant in (DUAL, FAST):
        Wh = np.zeros((N, synth.row_bytes(K, variant)), dtype=np.uint8)
        Xh = synth.activations(M, K, F16, seed=14, stream=1500)
        guard = 8192
        buf = t.full((M * N + 2 * guard,), float("nan"), device="cuda")
        Y = buf[guard:guard + M * N]
        rf4.gemm(upload_w(Wh), upload_x(Xh, F16), N, K, variant, Y=Y)
        assert t.all(Y == 0)
        assert t.all(t.isnan(buf[:guard])) and t.all(t.isnan(buf[guard + M * N:]))


def test_repeat_is_bitwise_identical():
    t = torch()
    N, K, M = 700, 2048, 333
    for variant in (DUAL, FAST):
        Wh = synth.weights(N, K, variant, seed=15, stream=1600)
        Xh = synth.activations(M, K, BF16, seed=15, stream=1601)
        W, X = upload_w(Wh), upload_x(Xh, BF16)
        a = rf4.gemm(W, X, N, K, variant)
        b = rf4.gemm(W, X, N, K, variant)
        assert t.equal(a.view(t.int32), b.view(t.int32))


# ---- prefill shapes at full size, sampled rows and tokens ------------------------------

LAYER = {"qkv": (7168, 5120), "o": (5120, 6144), "gate_up": (34816, 5120), "down": (5120, 17408)}
MATRIX = {"qkv": 0, "o": 1, "gate_up": 2, "down": 3}


def prefill_case(name, M, variant=DUAL, act=BF16, nrows=48, ntok=24):
    t = torch()
    N, K = LAYER[name]
    m = MATRIX[name]
    rb = synth.row_bytes(K, variant)
    W = t.empty(N * rb, dtype=t.uint8, device="cuda")
    synth.device.fill_weights(W, N, K, variant, seed=0, stream=synth.weight_stream(0, m))
    X = t.empty((M, K), dtype=t.float16 if act == F16 else t.bfloat16, device="cuda")
    synth.device.fill_act(X.view(t.int16), act, seed=0, stream=synth.act_stream(0, m))
    Y = rf4.gemm(W, X, N, K, variant)
    rng = np.random.default_rng(1000 * m + M)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 129, N - 1], rng.integers(0, N, nrows)]))
    toks = np.unique(np.concatenate([[0, 15, 255, 256, M - 1], rng.integers(0, M, ntok)]))
    toks = toks[toks < M]
    Wrows = synth.weights(N, K, variant, seed=0, stream=synth.weight_stream(0, m), rows=rows)
    assert np.array_equal(W.view(N, rb)[t.from_numpy(rows).cuda()].cpu().numpy(), Wrows)
    Xt = synth.activations(M, K, act, seed=0, stream=synth.act_stream(0, m), rows=toks)
    assert np.array_equal(X.view(t.int16)[t.from_numpy(toks).cuda()].cpu().numpy().view(np.uint16), Xt)
    got = Y[t.from_numpy(toks).cuda()][:, t.from_numpy(rows).cuda()].cpu().numpy()
    ref = oracle.gemm(Wrows, Xt, len(rows), K, variant, act=act)
    assert_close(got, ref, K, max_halfscale(Wrows, variant), f"{name} M={M}")
    return Y


@pytest.mark.parametrize("name", sorted(LAYER))
@pytest.mark.parametrize("M", [512, 4096])
def test_prefill_layer_shapes_sampled(name, M):
    prefill_case(name, M)


@pytest.mark.slow
def test_prefill_largest_batch_sampled():
    """M = 23552 tokens over the fused gate+up matrix (3.3 GB of fp32 output)."""
    Y = prefill_case("gate_up", 23552, nrows=32, ntok=40)
    t = torch()
    assert bool(t.isfinite(Y).all())
    del Y
    t.cuda.empty_cache()


def test_prefill_fast_variant_and_fp16_sampled():
    prefill_case("o", 4096, variant=FAST, act=F16)


# ---- K split across CTAs -----------------------------------------------------------------
# Fewer tiles than SMs (or a partial last wave): each tile's K range is shared
# by consecutive CTAs whose partial tiles the last one to finish adds in
# chunk order.  One 128 x 16 tile over K = 8192 is cut into 8 parts; the
# results must match the oracle, repeat bit for bit (fixed order), and stay
# right on later launches (the hand-off counters reset themselves).

@pytest.mark.parametrize("variant,M,N,K", [(DUAL, 16, 128, 8192), (DUAL, 33, 250, 17408),
                                           (FAST, 20, 256, 16384), (DUAL, 600, 520, 4096)])
def test_split_k_matches_oracle_and_repeats(variant, M, N, K):
    t = torch()
    Wh = synth.weights(N, K, variant, seed=16, stream=1700 + N)
    Xh = synth.activations(M, K, BF16, seed=16, stream=1701)
    W, X = upload_w(Wh), upload_x(Xh, BF16)
    ref = oracle.gemm(Wh, Xh, N, K, variant, act=BF16)
    first = None
    for _ in range(3):
        Y = rf4.gemm(W, X, N, K, variant)
        assert_close(Y.cpu().numpy(), ref, K, max_halfscale(Wh, variant), f"split M={M} N={N} K={K}")
        if first is None:
            first = Y
        else:
            assert t.equal(first.view(t.int32), Y.view(t.int32))


def test_split_k_shapes_interleaved():
    """Split and unsplit launches back to back share the counters and workspace."""
    shapes = [(DUAL, 16, 128, 8192), (DUAL, 300, 4096, 1024), (FAST, 40, 128, 4096), (DUAL, 64, 384, 2048)]
    data = []
    for i, (v, M, N, K) in enumerate(shapes):
        Wh = synth.weights(N, K, v, seed=17, stream=1800 + i)
        Xh = synth.activations(M, K, F16, seed=17, stream=1900 + i)
        data.append((v, M, N, K, Wh, Xh, upload_w(Wh), upload_x(Xh, F16)))
    for _ in range(2):
        outs = [rf4.gemm(W, X, N, K, v) for v, M, N, K, _, _, W, X in data]
        for (v, M, N, K, Wh, Xh, _, _), Y in zip(data, outs):
            ref = oracle.gemm(Wh, Xh, N, K, v, act=F16)
            assert_close(Y.cpu().numpy(), ref, K, max_halfscale(Wh, v), f"interleaved M={M} N={N} K={K}")
