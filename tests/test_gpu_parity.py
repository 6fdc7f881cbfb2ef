"""GPU parity of the CUDA library against the fp64 oracle.

Every input is drawn by the seeded host generator (synth) -- or, for inputs
too large for the host, by its CUDA twin, whose bytes are checked against the
host generator on the sampled rows.  Expected values come only from the
oracle.  Bars: dequantisation bit-exact; products within rel-L2 1e-5 and
max |err| <= 1e-3 * sqrt(K) * max half-scale.
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


def run_gemm(Wh, Xh, N, K, variant, act):
    W = upload_w(Wh)
    X = upload_x(Xh, act)
    return rf4.gemm(W, X, N, K, variant).cpu().numpy()


# ---- dequantisation: bit-exact ---------------------------------------------------

@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("out", ["float32", "bfloat16", "float16"])
@pytest.mark.parametrize("N,K", [(1, 32), (37, 320), (256, 1024)])
def test_dequant_bit_exact(variant, out, N, K):
    t = torch()
    Wh = synth.weights(N, K, variant, seed=1, stream=101)
    got = rf4.dequant(upload_w(Wh), N, K, variant, out_dtype=getattr(t, out))
    ref = oracle.dequant(Wh, N, K, variant)
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(g, ref)
    assert not np.any(np.signbit(g[g == 0]))


@pytest.mark.parametrize("variant", [DUAL, FAST])
def test_dequant_every_code_and_scale(variant):
    """All 256 qs byte values against all 127 finite scale bytes, plus exponent-0 codes."""
    t = torch()
    bb = synth.block_bytes(variant)
    rows = []
    for s in range(0x7F):
        for base in range(0, 256, 16):
            blk = np.zeros(bb, dtype=np.uint8)
            blk[:16] = np.arange(base, base + 16, dtype=np.uint8)
            blk[16:] = s if variant == FAST else [s, (s * 37 + 11) % 0x7F]
            rows.append(blk)
    Wh = np.stack(rows)  # one block per row
    N = Wh.shape[0]
    ref = oracle.dequant(Wh, N, 32, variant)
    for out in (t.float32, t.bfloat16, t.float16):
        g = rf4.dequant(upload_w(Wh), N, 32, variant, out_dtype=out).float().cpu().numpy().astype(np.float64)
        assert np.array_equal(g, ref), out
        assert not np.any(np.signbit(g[g == 0]))


# ---- products on small and ragged shapes -------------------------------------------

SHAPES = [(1, 32), (3, 64), (17, 256), (33, 512), (256, 1024), (100, 288), (16, 5120), (5, 17408), (40, 1536)]


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_matches_oracle(variant, act, N, K):
    Wh = synth.weights(N, K, variant, seed=2, stream=200 + N)
    xh = synth.activations(1, K, act, seed=2, stream=300 + K)
    y = rf4.gemv(upload_w(Wh), upload_x(xh[0], act), N, K, variant).cpu().numpy()
    ref = oracle.gemv(Wh, xh[0], N, K, variant, act=act)
    assert_close(y, ref, K, max_halfscale(Wh, variant), f"gemv N={N} K={K}")


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 9, 17])
def test_small_batch_and_chunked_gemm(variant, act, M):
    N, K = 200, 1024
    Wh = synth.weights(N, K, variant, seed=3, stream=400)
    Xh = synth.activations(M, K, act, seed=3, stream=401)
    Y = run_gemm(Wh, Xh, N, K, variant, act)
    ref = oracle.gemm(Wh, Xh, N, K, variant, act=act)
    assert_close(Y, ref, K, max_halfscale(Wh, variant), f"gemm M={M}")


def test_k_zero_writes_zeros_and_empty_shapes():
    t = torch()
    Y = t.full((2, 5), 7.0, device="cuda")
    W = t.zeros(0, dtype=t.uint8, device="cuda")
    X = t.zeros((2, 0), dtype=t.float16, device="cuda")
    rf4.gemm(W, X, 5, 0, DUAL, Y=Y)
    assert t.all(Y == 0)
    out = rf4.gemm(t.zeros(2 * 18 * 4, dtype=t.uint8, device="cuda"), t.zeros((0, 128), dtype=t.float16, device="cuda"),
                   2, 128, DUAL)
    assert out.shape == (0, 2)


def test_unaligned_pointers_take_the_generic_path():
    t = torch()
    N, K = 24, 512
    for variant in (DUAL, FAST):
        Wh = synth.weights(N, K, variant, seed=4, stream=500)
        xh = synth.activations(1, K, F16, seed=4, stream=501)[0]
        raw = t.zeros(Wh.size + 1, dtype=t.uint8, device="cuda")
        raw[1:] = upload_w(Wh)
        xr = t.zeros(K + 1, dtype=t.float16, device="cuda")
        xr[1:] = upload_x(xh, F16)
        y = rf4.gemv(raw[1:], xr[1:], N, K, variant).cpu().numpy()
        assert_close(y, oracle.gemv(Wh, xh, N, K, variant), K, max_halfscale(Wh, variant), "unaligned")


def test_outputs_stay_inside_their_buffer_and_repeat_bitwise():
    t = torch()
    N, K, M = 1000, 2048, 3
    for variant in (DUAL, FAST):
        Wh = synth.weights(N, K, variant, seed=5, stream=600)
        Xh = synth.activations(M, K, F16, seed=5, stream=601)
        W, X = upload_w(Wh), upload_x(Xh, F16)
        guard = 4096
        buf = t.full((M * N + 2 * guard,), float("nan"), device="cuda")
        Y = buf[guard:guard + M * N]
        rf4.gemm(W, X, N, K, variant, Y=Y)
        first = Y.clone()
        rf4.gemm(W, X, N, K, variant, Y=Y)
        assert t.equal(first.view(t.int32), Y.view(t.int32))
        assert t.all(t.isnan(buf[:guard])) and t.all(t.isnan(buf[guard + M * N:]))


def test_validate_finds_first_bad_block():
    for variant in (DUAL, FAST):
        N, K = 50, 640
        Wh = synth.weights(N, K, variant, seed=6, stream=700).copy()
        assert rf4.validate(upload_w(Wh), N, K, variant) == -1
        flat = Wh.reshape(-1)
        bb = synth.block_bytes(variant)
        for blk, off, val in ((733, 16, 0x7F), (400, bb - 1, 0x80), (999, 16, 0xFF)):
            flat[blk * bb + off] = val
        expect = oracle.validate(Wh, N, K, variant)
        assert expect == 400
        assert rf4.validate(upload_w(Wh), N, K, variant) == expect


# ---- full-size layer shapes, sampled rows ----------------------------------------------

LAYER = {"qkv": (7168, 5120), "o": (5120, 6144), "gate_up": (34816, 5120), "down": (5120, 17408)}


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("name", sorted(LAYER))
def test_full_size_layer_matrix_sampled_rows(variant, name):
    t = torch()
    N, K = LAYER[name]
    m = sorted(LAYER).index(name)
    rb = synth.row_bytes(K, variant)
    W = t.empty(N * rb, dtype=t.uint8, device="cuda")
    synth.device.fill_weights(W, N, K, variant, seed=0, stream=synth.weight_stream(0, m))
    rng = np.random.default_rng(m)
    rows = np.unique(np.concatenate([[0, 15, 16, N - 17, N - 1], rng.integers(0, N, 120)]))
    Wrows = synth.weights(N, K, variant, seed=0, stream=synth.weight_stream(0, m), rows=rows)
    assert np.array_equal(W.view(N, rb)[t.from_numpy(rows).cuda()].cpu().numpy(), Wrows)
    for M in (1, 2, 4, 8):
        Xh = synth.activations(M, K, F16, seed=0, stream=synth.act_stream(0, m))
        Y = rf4.gemm(W, upload_x(Xh, F16), N, K, variant).cpu().numpy()
        ref = oracle.gemm(Wrows, Xh, len(rows), K, variant)
        assert_close(Y[:, rows], ref, K, max_halfscale(Wrows, variant), f"{name} M={M}")


def test_device_generator_matches_host():
    t = torch()
    for variant in (DUAL, FAST):
        N, K = 300, 1536
        W = t.empty(N * synth.row_bytes(K, variant), dtype=t.uint8, device="cuda")
        synth.device.fill_weights(W, N, K, variant, seed=9, stream=77)
        assert np.array_equal(W.cpu().numpy(), synth.weights(N, K, variant, seed=9, stream=77).reshape(-1))
    for act in (F16, BF16):
        X = t.empty(50000, dtype=t.int16, device="cuda")
        synth.device.fill_act(X, act, seed=9, stream=78, first=12345)
        host = synth.act_bits_at(np.arange(12345, 12345 + 50000), act, 9, 78)
        assert np.array_equal(X.cpu().numpy().view(np.uint16), host)
