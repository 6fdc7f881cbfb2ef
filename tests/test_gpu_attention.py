"""GPU parity of decode attention over a ROCmFP4 K/V cache
(rocmfp4_decode_attention) against the fp64 oracle.

Tolerance, from the arithmetic of the kernel: a score is an fp32 sum of exact
products over D (at most 8 tensor-core steps, then one multiply by
scale * log2 e), so its error in base-2 units is at most
    dx = 16 * 2^-23 * scale * log2(e) * max_t sum_d |q_d k_{t,d}|   (+ 2^-24 |x|);
the softmax weights then carry a relative error of at most ln 2 * dx each (the
max is subtracted exactly), and the weighted sum adds a few 1e-7 relative
(P split into two fp16 parts, fp32 sums).  Each output element is a convex
combination of V rows, so
    |d out| <= (2 ln2 dx + 4e-6) * max |V|   (over the sequence's rows and D),
and the whole output is held to relative L2 error 1e-5, the bar of every
product here.
"""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
from gpu_util import REL_L2, torch, upload_w, upload_x

pytestmark = pytest.mark.gpu

DUAL, FAST = rf4.DUAL, rf4.FAST
F16, BF16 = synth.ACT_F16, synth.ACT_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def make_case(B, H, Hkv, D, Tmax, variant, act, seed):
    Kh = synth.weights(B * Hkv * Tmax, D, variant, seed=seed, stream=4000 + D)
    Vh = synth.weights(B * Hkv * Tmax, D, variant, seed=seed, stream=4100 + D)
    qh = synth.activations(B * H, D, act, seed=seed, stream=4200 + H).reshape(B, H, D)
    return Kh, Vh, qh


def bound(qh, Kh, Vh, lens, B, H, Hkv, D, Tmax, scale, variant, act):
    """Element-wise bound of the module docstring, per (b, h)."""
    G = H // Hkv
    Kd = oracle.dequant(Kh, B * Hkv * Tmax, D, variant).reshape(B, Hkv, Tmax, D)
    Vd = oracle.dequant(Vh, B * Hkv * Tmax, D, variant).reshape(B, Hkv, Tmax, D)
    qf = synth.bits_to_float(qh.reshape(-1), act).reshape(B, H, D)
    out = np.zeros((B, H, 1))
    for b in range(B):
        T = int(min(max(lens[b], 0), Tmax))
        if T == 0:
            continue
        for h in range(H):
            hk = h // G
            mag = np.abs(Kd[b, hk, :T]) @ np.abs(qf[b, h])
            dx = 16 * 2.0 ** -23 * abs(scale) * np.log2(np.e) * mag.max()
            x = np.abs(scale * (Kd[b, hk, :T] @ qf[b, h])) * np.log2(np.e)
            dx += 2.0 ** -24 * x.max()
            out[b, h, 0] = (2 * np.log(2) * dx + 4e-6) * np.abs(Vd[b, hk, :T]).max()
    return out


def run_and_check(B, H, Hkv, D, Tmax, lens, scale, variant, act, seed, what=""):
    t = torch()
    Kh, Vh, qh = make_case(B, H, Hkv, D, Tmax, variant, act, seed)
    lens = np.asarray(lens, dtype=np.int32)
    out = rf4.decode_attention(upload_x(qh.reshape(B, H, D), act), upload_w(Kh), upload_w(Vh),
                               t.from_numpy(lens).cuda(), Hkv, Tmax, scale, variant)
    got = out.cpu().numpy().astype(np.float64)
    ref = oracle.decode_attention(qh, Kh, Vh, lens, B, H, Hkv, D, Tmax, scale, variant, act=act)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    lim = bound(qh, Kh, Vh, lens, B, H, Hkv, D, Tmax, scale, variant, act)
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - lim), err.shape)
    assert np.all(err <= lim), f"{what}: |err| {err[worst]:.3e} > {lim[worst[0], worst[1], 0]:.3e} at {worst}"
    nref = np.linalg.norm(ref)
    if nref > 0:  # the relative L2 bar of every product in this library
        rel = np.linalg.norm(got - ref) / nref
        assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    return got, ref, err


# (B, H, Hkv, D, Tmax, lens): MHA and grouped heads, one to several chunks
# and splits, ragged lengths (0, partial chunks, full cache)
CASES = [
    (1, 8, 8, 128, 32, [32]),
    (1, 8, 8, 128, 96, [77]),
    (2, 40, 8, 128, 1024, [1024, 517]),
    (3, 16, 2, 64, 256, [0, 1, 255]),
    (1, 4, 1, 64, 2048, [2048]),
    (4, 8, 1, 128, 128, [5, 33, 64, 128]),
]


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_matches_oracle(case, act, variant):
    B, H, Hkv, D, Tmax, lens = CASES[case]
    for scale in (1.0 / np.sqrt(D), 0.01):
        run_and_check(B, H, Hkv, D, Tmax, lens, scale, variant, act, seed=40 + case,
                      what=f"case {case} v={variant} act={act} scale={scale:.3g}")


def test_long_context_split_and_combine():
    """A 16k-token cache for one sequence: many splits merged by the combine launch."""
    launches = rf4.launch_count()
    run_and_check(1, 40, 8, 128, 16384, [16000], 1.0 / np.sqrt(128), DUAL, F16, seed=50, what="16k")
    assert rf4.launch_count() - launches == 2


def test_rows_past_lengths_are_never_read_as_data():
    """Rows at or past lens[b] hold non-finite scale bytes (0xFF); the result is
    that of the oracle, which ignores them, and bitwise that of a cache whose
    rows past lens are zeros."""
    t = torch()
    B, H, Hkv, D, Tmax, variant = 2, 8, 2, 128, 128, DUAL
    lens = np.array([70, 3], dtype=np.int32)
    Kh, Vh, qh = make_case(B, H, Hkv, D, Tmax, variant, F16, seed=51)
    rb = synth.row_bytes(D, variant)
    K3 = Kh.reshape(B, Hkv, Tmax, rb).copy()
    V3 = Vh.reshape(B, Hkv, Tmax, rb).copy()
    Kz, Vz = K3.copy(), V3.copy()
    for b in range(B):
        K3[b, :, lens[b]:] = 0xFF
        V3[b, :, lens[b]:] = 0xFF
        Kz[b, :, lens[b]:] = 0
        Vz[b, :, lens[b]:] = 0
    q = upload_x(qh, F16)
    L = t.from_numpy(lens).cuda()
    a = rf4.decode_attention(q, upload_w(K3), upload_w(V3), L, Hkv, Tmax, 0.05, variant)
    z = rf4.decode_attention(q, upload_w(Kz), upload_w(Vz), L, Hkv, Tmax, 0.05, variant)
    assert bool(t.isfinite(a).all())
    assert t.equal(a.view(t.int32), z.view(t.int32))
    ref = oracle.decode_attention(qh, K3, V3, lens, B, H, Hkv, D, Tmax, 0.05, variant)
    assert np.allclose(a.cpu().numpy(), ref, rtol=1e-4, atol=1e-4)


def test_one_token_returns_its_value_row():
    """lens = 1: softmax of one score is 1, so out = V row 0 exactly."""
    t = torch()
    B, H, Hkv, D, Tmax = 2, 8, 4, 64, 32
    Kh, Vh, qh = make_case(B, H, Hkv, D, Tmax, DUAL, BF16, seed=52)
    out = rf4.decode_attention(upload_x(qh, BF16), upload_w(Kh), upload_w(Vh),
                               t.from_numpy(np.array([1, 1], dtype=np.int32)).cuda(), Hkv, Tmax, 0.3, DUAL)
    Vd = oracle.dequant(Vh, B * Hkv * Tmax, D, DUAL).reshape(B, Hkv, Tmax, D)
    for b in range(B):
        for h in range(H):
            assert np.array_equal(out[b, h].cpu().numpy().astype(np.float64), Vd[b, h // 2, 0]), (b, h)


def test_repeat_is_bitwise_identical():
    t = torch()
    B, H, Hkv, D, Tmax = 2, 40, 8, 128, 4096
    lens = np.array([4096, 1500], dtype=np.int32)
    Kh, Vh, qh = make_case(B, H, Hkv, D, Tmax, FAST, F16, seed=53)
    args = (upload_x(qh, F16), upload_w(Kh), upload_w(Vh), t.from_numpy(lens).cuda(), Hkv, Tmax, 0.088, FAST)
    a = rf4.decode_attention(*args)
    b = rf4.decode_attention(*args)
    assert t.equal(a.view(t.int32), b.view(t.int32))


def test_unsupported_and_degenerate():
    t = torch()
    B, H, Hkv, D, Tmax = 1, 16, 1, 128, 64  # 16 heads per KV head
    Kh, Vh, qh = make_case(B, H, Hkv, D, Tmax, DUAL, F16, seed=54)
    L = t.from_numpy(np.array([64], dtype=np.int32)).cuda()
    with pytest.raises(rf4.RocmFP4Error) as e:
        rf4.decode_attention(upload_x(qh, F16), upload_w(Kh), upload_w(Vh), L, Hkv, Tmax, 0.1, DUAL)
    assert e.value.status == 2  # ROCMFP4_ERR_UNSUPPORTED
    Kh, Vh, qh = make_case(1, 8, 8, 128, 40, DUAL, F16, seed=55)  # Tmax not a multiple of 32
    with pytest.raises(rf4.RocmFP4Error) as e:
        rf4.decode_attention(upload_x(qh, F16), upload_w(Kh), upload_w(Vh), L, 8, 40, 0.1, DUAL)
    assert e.value.status == 2
    # all lengths zero: zeros
    Kh, Vh, qh = make_case(2, 8, 8, 64, 32, DUAL, F16, seed=56)
    out = t.full((2, 8, 64), 7.0, device="cuda")
    rf4.decode_attention(upload_x(qh, F16), upload_w(Kh), upload_w(Vh), t.zeros(2, dtype=t.int32, device="cuda"),
                         8, 32, 0.1, DUAL, out=out)
    assert t.all(out == 0)
