"""GPU tests of per-tensor block layouts in one chain (rocmfp4_gemv_chain_mixed).

"Feasibility Report: Porting ROCmFP4 to Atlas", section "Tensor-Aware Presets":
a preset mixes the 18- and 17-byte layouts across tensor roles, so the engine
applies a layout per tensor.  The pages list none of the six presets, so these
tests take layout maps of their own: every product must match the fp64 oracle
for its own layout, and give bit for bit what one rocmfp4_gemm_ex call with
that layout gives.
"""
import ctypes

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


def make_ops(shapes, variants, M, act, seed):
    t = torch()
    ops, host = [], []
    for i, ((N, K), v) in enumerate(zip(shapes, variants)):
        Wh = synth.weights(N, K, v, seed=seed, stream=2600 + i)
        Xh = synth.activations(M, K, act, seed=seed, stream=2700 + i)
        Y = t.full((M, N), float("nan"), device="cuda")
        ops.append((upload_w(Wh), upload_x(Xh, act), Y, N, K))
        host.append((Wh, Xh))
    return ops, host


# a layer's four roles at reduced size (several tiles and spans, ragged N):
# attention matrices in one layout, FFN matrices in the other, and a map
# that changes layout at every product
LAYER_SHAPES = [(700, 2048), (520, 1536), (1000, 2048), (520, 3072)]
MAPS = {
    "attention dual, FFN fast": [DUAL, DUAL, FAST, FAST],
    "attention fast, FFN dual": [FAST, FAST, DUAL, DUAL],
    "alternating": [DUAL, FAST, DUAL, FAST],
    "all fast": [FAST] * 4,
}


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("name", list(MAPS))
def test_mixed_chain_matches_oracle_and_single_calls(name, M):
    t = torch()
    variants = MAPS[name]
    act = F16 if M != 4 else BF16
    ops, host = make_ops(LAYER_SHAPES, variants, M, act, seed=61)
    rf4.gemv_chain(ops, variants)
    for (W, X, Y, N, K), (Wh, Xh), v in zip(ops, host, variants):
        ref = oracle.gemm(Wh, Xh, N, K, v, act=act)
        assert_close(Y.cpu().numpy(), ref, K, max_halfscale(Wh, v), f"{name} v={v} N={N} K={K} M={M}")
        single = rf4.gemm(W, X, N, K, v)
        assert t.equal(single.view(t.int32), Y.view(t.int32)), f"{name}: chain differs from a single call"


def test_later_product_of_other_layout_reads_earlier_output():
    """A dual product writes Y0; a single-scale product reads Y0's memory as its
    activations (fp16 view of integer-valued fp32, as in the single-layout test)."""
    t = torch()
    K0, N0 = 256, 2048
    bb = synth.block_bytes(DUAL)
    rng = np.random.default_rng(62)
    nib = rng.choice(np.array([0, 1, 9], dtype=np.uint8), size=(N0 * K0 // 32, 16, 2))
    W0h = np.zeros((N0 * K0 // 32, bb), dtype=np.uint8)
    W0h[:, :16] = nib[:, :, 0] | (nib[:, :, 1] << 4)
    W0h[:, 16:] = 0x40
    W0h = W0h.reshape(N0, -1)
    x0 = np.where(synth.activations(1, K0, F16, seed=62, stream=2801) >= 0x8000, 0xBC00, 0x3C00).astype(np.uint16)
    N1, K1 = 300, 4096
    W1h = synth.weights(N1, K1, FAST, seed=62, stream=2802)
    W0, X0, W1 = upload_w(W0h), upload_x(x0, F16), upload_w(W1h)
    Y0 = t.empty((1, N0), dtype=t.float32, device="cuda")
    Y1 = t.empty((1, N1), dtype=t.float32, device="cuda")
    X1 = Y0.view(t.float16).view(1, 2 * N0)[:, :K1]
    rf4.gemv_chain([(W0, X0, Y0, N0, K0), (W1, X1, Y1, N1, K1)], [DUAL, FAST])
    x1 = Y0.view(t.int16).cpu().numpy().view(np.uint16).reshape(1, -1)[:, :K1]
    assert np.all(np.isfinite(synth.bits_to_float(x1, F16)))
    ref1 = oracle.gemm(W1h, x1, N1, K1, FAST, act=F16)
    assert_close(Y1.cpu().numpy(), ref1, K1, max_halfscale(W1h, FAST), "second product")
    assert t.equal(rf4.gemm(W1, X1.contiguous(), N1, K1, FAST).view(t.int32), Y1.view(t.int32))


def test_errors_are_found_before_any_launch():
    """A bad layout (or shape) in the last product: nothing runs, the earlier
    outputs keep their NaN fill."""
    t = torch()
    ops, _ = make_ops(LAYER_SHAPES, [DUAL, FAST, DUAL, FAST], 1, F16, seed=63)
    launches = rf4.launch_count()
    with pytest.raises(rf4.RocmFP4Error) as e:
        rf4.gemv_chain(ops, [DUAL, FAST, DUAL, 7])
    assert e.value.status == 1  # ROCMFP4_ERR_INVALID_ARG
    # K not a multiple of 32 in the last product
    arr = (rf4.GemvOp * 4)()
    for i, (W, X, Y, N, K) in enumerate(ops):
        arr[i] = rf4.GemvOp(W.data_ptr(), X.data_ptr(), Y.data_ptr(), N, K + (33 if i == 3 else 0))
    varr = (ctypes.c_int * 4)(DUAL, FAST, DUAL, FAST)
    status = rf4.load().rocmfp4_gemv_chain_mixed(arr, varr, 4, 1, F16, None)
    assert status == 1  # ROCMFP4_ERR_INVALID_ARG
    assert rf4.launch_count() == launches
    for (_, _, Y, _, _) in ops:
        assert bool(t.isnan(Y).all())
    rf4.gemv_chain([], [])  # nothing to do


def test_mixed_and_single_layout_chains_agree():
    """One layout for every product through the mixed entry point is the
    single-layout chain, bit for bit."""
    t = torch()
    shapes = [(7168, 5120), (5120, 6144)]
    ops, _ = make_ops(shapes, [FAST, FAST], 2, F16, seed=64)
    rf4.gemv_chain(ops, [FAST, FAST])
    first = [Y.clone() for (_, _, Y, _, _) in ops]
    rf4.gemv_chain(ops, FAST)
    for a, (_, _, Y, _, _) in zip(first, ops):
        assert t.equal(a.view(t.int32), Y.view(t.int32))
