"""GPU parity of the fused gate/up decode product (rocmfp4_gemv_gate_up)
against the fp64 oracle.

W packs 2I rows (the I gate rows, then the I up rows) and
Y[m][i] = SiLU(g) * u with g, u the gate and up row products.  Tolerance:
the two sums each carry the product bound tau = 1e-3 * sqrt(K) * max
half-scale, and |SiLU'| <= 1.1, so element-wise
    |dY| <= tau * (1.1 |u| + |SiLU(g)|) + 1.1 tau^2,
with the relative L2 bound of every product (1e-5) on the whole output.
"""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
from gpu_util import ABS_PER_SQRT_K, REL_L2, max_halfscale, torch, upload_w, upload_x

pytestmark = pytest.mark.gpu

DUAL, FAST = rf4.DUAL, rf4.FAST
F16, BF16 = synth.ACT_F16, synth.ACT_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def silu(g):
    with np.errstate(over="ignore"):  # exp(-g) = inf for very negative g gives the right 0
        return g / (1.0 + np.exp(-g))


def check_gate_up(Y, Wh, Xh, I, K, variant, act, what):
    Y = np.asarray(Y, dtype=np.float64)
    ref = oracle.gemv_gate_up(Wh, Xh, I, K, variant, act=act)
    GU = oracle.gemm(Wh, Xh, 2 * I, K, variant, act=act)
    G, U = GU[:, :I], GU[:, I:]
    assert Y.shape == ref.shape, (Y.shape, ref.shape)
    assert np.all(np.isfinite(Y)), f"{what}: non-finite outputs"
    err = np.abs(Y - ref)
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(Y - ref) / nref if nref > 0 else np.linalg.norm(Y - ref)
    tau = ABS_PER_SQRT_K * np.sqrt(K) * max_halfscale(Wh, variant)
    bound = tau * (1.1 * np.abs(U) + np.abs(silu(G))) + 1.1 * tau * tau
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), f"{what}: |err| {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e}"


def run_case(I, K, M, variant, act, seed):
    Wh = synth.weights(2 * I, K, variant, seed=seed, stream=3000 + I)
    Xh = synth.activations(M, K, act, seed=seed, stream=3100 + K)
    Y = rf4.gemv_gate_up(upload_w(Wh), upload_x(Xh, act), I, K, variant).cpu().numpy()
    check_gate_up(Y, Wh, Xh, I, K, variant, act, f"gate_up v={variant} act={act} M={M} I={I} K={K}")
    return Wh, Xh, Y


# ragged I (not a multiple of the 16-output tile), several tiles, several spans
DUAL_IK = [(16, 256), (50, 1024), (1000, 2048), (333, 5120)]
FAST_IK = [(16, 512), (50, 1024), (1000, 2048), (333, 5120)]


@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("I,K", DUAL_IK)
def test_dual_matches_oracle(act, M, I, K):
    run_case(I, K, M, DUAL, act, seed=31)


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("I,K", FAST_IK)
def test_fast_matches_oracle(M, I, K):
    run_case(I, K, M, FAST, F16, seed=32)


def test_layer_shape_m1():
    """The decoder layer's gate+up matrix, [2 x 17408, 5120], batch 1."""
    run_case(17408, 5120, 1, DUAL, F16, seed=33)


def test_gate_only_and_up_only_rows():
    """Zero up rows give zero outputs; up rows of +1 with gate rows of +1
    (one code-1 weight each, half-scale 1) give SiLU(x_0) * x_0 exactly
    at every output."""
    t = torch()
    I, K = 40, 256
    bb = synth.block_bytes(DUAL)
    Xh = synth.activations(2, K, F16, seed=34, stream=3200)
    x0 = synth.bits_to_float(Xh, F16)[:, 0]
    Wh = np.zeros((2 * I, K // 32 * bb), dtype=np.uint8)
    Wh[:, 0] = 0x1  # weight 0 of each row: code 1
    for b in range(K // 32):
        Wh[:, b * bb + 16:(b + 1) * bb] = 0x40  # half-scale 1.0
    Y = rf4.gemv_gate_up(upload_w(Wh), upload_x(Xh, F16), I, K, DUAL).cpu().numpy()
    want = (silu(x0) * x0)[:, None] * np.ones((1, I))
    assert np.allclose(Y, want, rtol=2e-6, atol=1e-30), np.max(np.abs(Y - want))
    Wz = Wh.copy()
    Wz[I:] = 0
    for b in range(K // 32):
        Wz[I:, b * bb + 16:(b + 1) * bb] = 0x40
    Y = rf4.gemv_gate_up(upload_w(Wz), upload_x(Xh, F16), I, K, DUAL).cpu().numpy()
    assert np.all(Y == 0)
    assert t.cuda.is_available()


def test_repeat_is_bitwise_identical_and_in_bounds():
    t = torch()
    I, K, M = 700, 2048, 3
    Wh = synth.weights(2 * I, K, DUAL, seed=35, stream=3300)
    Xh = synth.activations(M, K, BF16, seed=35, stream=3301)
    W, X = upload_w(Wh), upload_x(Xh, BF16)
    guard = 4096
    buf = t.full((M * I + 2 * guard,), float("nan"), device="cuda")
    Y = buf[guard:guard + M * I]
    rf4.gemv_gate_up(W, X, I, K, DUAL, Y=Y)
    a = Y.clone()
    rf4.gemv_gate_up(W, X, I, K, DUAL, Y=Y)
    assert t.equal(a.view(t.int32), Y.view(t.int32))
    assert t.all(t.isnan(buf[:guard])) and t.all(t.isnan(buf[guard + M * I:]))


def test_unsupported_and_degenerate():
    t = torch()
    I, K = 32, 256
    Wh = synth.weights(2 * I, K, DUAL, seed=36, stream=3400)
    W = upload_w(Wh)
    X9 = upload_x(synth.activations(9, K, F16, seed=36, stream=3401), F16)
    with pytest.raises(rf4.RocmFP4Error) as e:
        rf4.gemv_gate_up(W, X9, I, K, DUAL)
    assert e.value.status == 2  # ROCMFP4_ERR_UNSUPPORTED
    K2 = 288  # a multiple of 32 but not of the 256-weight streaming unit
    W2 = upload_w(synth.weights(2 * I, K2, DUAL, seed=36, stream=3402))
    X2 = upload_x(synth.activations(1, K2, F16, seed=36, stream=3403), F16)
    with pytest.raises(rf4.RocmFP4Error) as e:
        rf4.gemv_gate_up(W2, X2, I, K2, DUAL)
    assert e.value.status == 2  # ROCMFP4_ERR_UNSUPPORTED
    Y = t.full((1, 5), 3.0, device="cuda")
    rf4.gemv_gate_up(t.zeros(0, dtype=t.uint8, device="cuda"), t.zeros((1, 0), dtype=t.float16, device="cuda"),
                     5, 0, DUAL, Y=Y)
    assert t.all(Y == 0)  # K = 0: SiLU(0) * 0
