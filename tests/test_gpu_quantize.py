"""GPU quantiser (rocmfp4_quantize): bit-exact against the oracle (codes and
scale bytes are integers, and every decision of the rule is exact in fp32),
and the round trip through the GPU dequantiser."""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
from gpu_util import torch

pytestmark = pytest.mark.gpu

DUAL, FAST = rf4.DUAL, rf4.FAST
F16, BF16 = synth.ACT_F16, synth.ACT_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def source(N, K, act, seed):
    """Values whose magnitudes span subnormal scales to saturation (per-block
    factors 2^-22 .. 2^14), with zeros, -0, NaN and +-Inf mixed in."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, K)) * np.exp2(rng.integers(-22, 15, size=(N, K // 32, 1))).repeat(32, axis=2).reshape(N, K)
    x[rng.random((N, K)) < 0.05] = 0.0
    special = rng.random((N, K))
    x[special < 0.002] = np.nan
    x[(special >= 0.002) & (special < 0.004)] = np.inf
    x[(special >= 0.004) & (special < 0.006)] = -np.inf
    x[(special >= 0.006) & (special < 0.010)] = -0.0
    if act == F16:
        with np.errstate(over="ignore"):  # values past fp16's range become +-Inf, which the rule counts as 0
            return x.astype(np.float16).view(np.uint16)
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # bf16 by truncation (any bits will do)


def to_device(bits, act):
    t = torch()
    return t.from_numpy(bits.view(np.int16)).cuda().view(t.float16 if act == F16 else t.bfloat16)


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("N,K", [(1, 32), (7, 96), (64, 1024), (33, 2080)])
def test_bit_exact_against_oracle(N, K, act, variant):
    bits = source(N, K, act, seed=60 + N)
    W = rf4.quantize(to_device(bits, act), variant).cpu().numpy().reshape(N, -1)
    ref = oracle.quantize(bits, N, K, variant, act=act)
    assert np.array_equal(W, ref), np.argwhere(W != ref)[:5]


def test_unaligned_source_takes_the_same_rule():
    t = torch()
    N, K = 16, 512
    bits = source(N, K, F16, seed=70)
    buf = t.empty(N * K + 1, dtype=t.int16, device="cuda")
    buf[1:] = t.from_numpy(bits.view(np.int16).reshape(-1)).cuda()
    src = buf[1:].view(t.float16).view(N, K)  # 2 bytes past a 16-byte boundary
    W = rf4.quantize(src, DUAL).cpu().numpy().reshape(N, -1)
    assert np.array_equal(W, oracle.quantize(bits, N, K, DUAL))


@pytest.mark.parametrize("variant", [DUAL, FAST])
def test_round_trip_through_dequant(variant):
    """Blocks with a code of magnitude 10 in every scale group and no code 8:
    quantize(dequant(W)) == W bit for bit, on the GPU."""
    t = torch()
    rng = np.random.default_rng(71)
    N, K = 128, 512
    bb = synth.block_bytes(variant)
    nb = N * K // 32
    codes = rng.choice(np.r_[0:8, 9:16], size=(nb, 32))
    ng = 2 if variant == DUAL else 1
    for g in range(ng):
        codes[np.arange(nb), g * (32 // ng) + rng.integers(0, 32 // ng, size=nb)] = rng.choice([7, 15], size=nb)
    Wh = np.zeros((nb, bb), dtype=np.uint8)
    Wh[:, :16] = codes[:, :16] | (codes[:, 16:] << 4)
    Wh[:, 16:] = rng.integers(0x01, 0x7F, size=(nb, bb - 16))
    W = t.from_numpy(Wh.reshape(-1)).cuda()
    dense = rf4.dequant(W, N, K, variant, out_dtype=t.float16)
    back = rf4.quantize(dense, variant)
    assert t.equal(back, W)


def test_layer_shape_sampled_rows():
    """The gate+up matrix [34816, 5120] from bf16 N(0,1) values: sampled rows bit-exact."""
    t = torch()
    N, K = 34816, 5120
    src = t.randn((N, K), dtype=t.float32, device="cuda", generator=t.Generator(device="cuda").manual_seed(5))
    src = src.to(t.bfloat16)
    W = rf4.quantize(src, DUAL).view(N, -1)
    rows = np.array([0, 1, 4095, 17407, 17408, 34815] + list(np.random.default_rng(72).integers(0, N, 20)))
    bits = src[t.from_numpy(rows).cuda()].view(t.int16).cpu().numpy().view(np.uint16)
    ref = oracle.quantize(bits, len(rows), K, DUAL, act=BF16)
    assert np.array_equal(W[t.from_numpy(rows).cuda()].cpu().numpy(), ref)
