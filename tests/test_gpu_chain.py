"""GPU tests of rocmfp4_gemv_chain: products run in order, one launch each.

Values are checked against the fp64 oracle; the chain must also give, bit for
bit, what one rocmfp4_gemm_ex call per product gives (the same kernel and
the same fixed summation order), including when a later product reads memory
that an earlier one writes.
"""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
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


def make_ops(shapes, M, variant, act, seed):
    t = torch()
    ops, host = [], []
    for i, (N, K) in enumerate(shapes):
        Wh = synth.weights(N, K, variant, seed=seed, stream=2000 + i)
        Xh = synth.activations(M, K, act, seed=seed, stream=2100 + i)
        Y = t.full((M, N), float("nan"), device="cuda")
        ops.append((upload_w(Wh), upload_x(Xh, act), Y, N, K))
        host.append((Wh, Xh))
    return ops, host


def check_ops(ops, host, variant, act):
    for (W, X, Y, N, K), (Wh, Xh) in zip(ops, host):
        ref = oracle.gemm(Wh, Xh, N, K, variant, act=act)
        assert_close(Y.cpu().numpy(), ref, K, max_halfscale(Wh, variant), f"chain N={N} K={K}")


# layer-like and ragged shapes; K = 288 and K = 640 (single-scale) are not
# multiples of the streaming unit and fall back to single calls in between
DUAL_SHAPES = [(700, 2048), (33, 256), (1000, 1024), (64, 288), (4096, 512), (130, 1536)]
FAST_SHAPES = [(700, 2048), (33, 512), (257, 640), (1000, 1024), (96, 1536)]


@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("act", [F16, BF16])
def test_chain_dual_matches_oracle(M, act):
    ops, host = make_ops(DUAL_SHAPES, M, DUAL, act, seed=21)
    rf4.gemv_chain(ops, DUAL)
    check_ops(ops, host, DUAL, act)


@pytest.mark.parametrize("M", [1, 2])
def test_chain_fast_matches_oracle(M):
    ops, host = make_ops(FAST_SHAPES, M, FAST, F16, seed=22)
    rf4.gemv_chain(ops, FAST)
    check_ops(ops, host, FAST, F16)


def test_long_chain_one_launch_per_product():
    """60 products of ragged sizes: one launch each, in order, and a second call gives the same."""
    rng = np.random.default_rng(5)
    shapes = [(int(rng.integers(1, 400)), int(rng.choice([256, 512, 1024]))) for _ in range(60)]
    ops, host = make_ops(shapes, 1, DUAL, F16, seed=23)
    launches = rf4.launch_count()
    rf4.gemv_chain(ops, DUAL)
    assert rf4.launch_count() - launches == 60
    check_ops(ops, host, DUAL, F16)
    rf4.gemv_chain(ops, DUAL)
    check_ops(ops, host, DUAL, F16)


@pytest.mark.parametrize("variant", [DUAL, FAST])
def test_chain_equals_single_calls_bitwise(variant):
    t = torch()
    shapes = [(7168, 5120), (5120, 6144), (900, 1024)]
    for M in (1, 4):
        ops, _ = make_ops(shapes, M, variant, F16, seed=24)
        rf4.gemv_chain(ops, variant)
        for W, X, Y, N, K in ops:
            single = rf4.gemm(W, X, N, K, variant)
            assert t.equal(single.view(t.int32), Y.view(t.int32))


def test_later_product_reads_earlier_output():
    """Product 1's activations are product 0's output memory (its fp32 bits seen
    as fp16 pairs).  Product 0 has codes in {0, +1, -1}, half-scale 1, K = 256
    and x = +-1, so its outputs are integers of magnitude <= 256: at most 8
    significant bits, hence zero low 16 bits, and the fp16 view is finite."""
    t = torch()
    K0, N0 = 256, 2048                   # product 0 writes 2048 fp32 = 4096 fp16
    N1, K1 = 300, 4096
    bb = synth.block_bytes(DUAL)
    rng = np.random.default_rng(25)
    nib = rng.choice(np.array([0, 1, 9], dtype=np.uint8), size=(N0 * K0 // 32, 16, 2))
    W0h = np.zeros((N0 * K0 // 32, bb), dtype=np.uint8)
    W0h[:, :16] = nib[:, :, 0] | (nib[:, :, 1] << 4)
    W0h[:, 16:] = 0x40                    # E4M3 2.0: half-scale 1.0
    W0h = W0h.reshape(N0, -1)
    x0 = np.where(synth.activations(1, K0, F16, seed=25, stream=2201) >= 0x8000, 0xBC00, 0x3C00).astype(np.uint16)
    W1h = synth.weights(N1, K1, DUAL, seed=25, stream=2202)
    W0, X0, W1 = upload_w(W0h), upload_x(x0, F16), upload_w(W1h)
    Y0 = t.empty((1, N0), dtype=t.float32, device="cuda")
    Y1 = t.empty((1, N1), dtype=t.float32, device="cuda")
    X1 = Y0.view(t.float16).view(1, K1)
    rf4.gemv_chain([(W0, X0, Y0, N0, K0), (W1, X1, Y1, N1, K1)], DUAL)
    ref0 = oracle.gemv(W0h, x0[0], N0, K0, DUAL)
    assert np.array_equal(Y0.cpu().numpy()[0].astype(np.float64), ref0)  # integer sums are exact
    assert bool(t.isfinite(X1).all())
    # product 1 equals its single call on the finished product 0, and the oracle
    single = rf4.gemm(W1, X1, N1, K1, DUAL)
    assert t.equal(single.view(t.int32), Y1.view(t.int32))
    ref1 = oracle.gemv(W1h, X1.cpu().numpy().view(np.uint16)[0], N1, K1, DUAL)
    assert_close(Y1.cpu().numpy()[0], ref1, K1, max_halfscale(W1h, DUAL), "dependent product")


def test_empty_and_degenerate_chains():
    t = torch()
    rf4.gemv_chain([], DUAL)
    ops, host = make_ops([(0, 256), (50, 512)], 1, DUAL, F16, seed=26)
    rf4.gemv_chain(ops, DUAL)
    check_ops(ops[1:], host[1:], DUAL, F16)
    Y = t.full((1, 5), 3.0, device="cuda")
    W = t.zeros(0, dtype=t.uint8, device="cuda")
    X = t.zeros((1, 0), dtype=t.float16, device="cuda")
    rf4.gemv_chain([(W, X, Y, 5, 0)], DUAL)  # K = 0 writes zeros
    assert t.all(Y == 0)
