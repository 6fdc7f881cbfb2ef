"""Every qs byte against every finite scale byte, through each product kernel.

The format ("Feasibility Report: Porting ROCmFP4 to Atlas", section "What is
ROCmFP4?", subsections "Block Layout", "Codebook10 Value Table" and "Scale
Format") decodes a weight as Codebook10[q] times half of an unsigned E4M3
scale byte.  The product kernels do not decode through a table: they convert
nibble pairs as OCP E2M1, clamp the magnitude to 5 and multiply by the E4M3
value of the scale byte (or apply it after a half-block sum).  This file runs
that route on all 256 qs byte values x all 127 finite scale bytes (exponent
field 0 -- the subnormal half-scales down to 2^-10 -- through 15, up to
half-scale 224), for both block layouts, in:

* the streaming GEMV at M = 1 (half-block sums scaled in fp32 afterwards) and
  M = 2, 4, 8 (scales applied to the weights before the products);
* the tensor-core GEMM (M > 8) with fp16 and with bf16 activations;
* the fused gate/up product;
* decode attention, V rows (one-token caches) and K rows.

Weights.  Matrix row r = (s, b) holds a single nonzero qs byte b, at block
(s + b) % nb, byte (7b + s) % 16; that block's first scale byte is s and, in
the dual layout, its second scale byte (37 s + 11 + b) % 127, so over all rows
each byte value meets every finite byte in either scale slot.  All other qs
bytes are 0.

Activations.  X rows are 0/1 masks of the first or the second 16 positions of
every block, times a power of two.  Every output is then one decoded weight
times a power of two plus exact zeros, so the kernels' results must equal the
fp64 oracle exactly, whatever the summation order.
"""
import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
from gpu_util import torch, upload_w, upload_x

pytestmark = pytest.mark.gpu

DUAL, FAST = rf4.DUAL, rf4.FAST
F16, BF16 = synth.ACT_F16, synth.ACT_BF16
NSCALE = 0x7F          # finite scale bytes 0x00 .. 0x7E
EXPS = [0, 0, -3, 2, 4, -1, 1, -2]  # power of two of X row m (m % 8)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert rf4.device_error_bits() == 0


def kmin(variant):
    """Smallest K that every product kernel takes for the layout."""
    return 256 if variant == DUAL else 512


def code_matrix(variant, K=None):
    """[127 * 256, row_bytes] blocks, row s * 256 + b as in the module docstring."""
    K = K or kmin(variant)
    bb = synth.block_bytes(variant)
    nb = K // 32
    s, b = np.meshgrid(np.arange(NSCALE), np.arange(256), indexing="ij")
    s, b = s.ravel(), b.ravel()
    N = s.size
    W = np.zeros((N, nb * bb), dtype=np.uint8)
    rng = np.random.default_rng(1234 + variant)
    # every scale byte of every block: any finite value (their codes are 0)
    for blk in range(nb):
        W[:, blk * bb + 16:(blk + 1) * bb] = rng.integers(0, NSCALE, (N, bb - 16), dtype=np.uint8)
    beta = (s + b) % nb
    j = (7 * b + s) % 16
    rows = np.arange(N)
    W[rows, beta * bb + j] = b
    W[rows, beta * bb + 16] = s
    if variant == DUAL:
        W[rows, beta * bb + 17] = (37 * s + 11 + b) % NSCALE
    return W


def pow2_bits(e, act):
    return (e + 15) << 10 if act == F16 else (e + 127) << 7


def mask_rows(M, K, act):
    """X [M, K] bits: row m is the mask of half m % 2 of every block times 2^EXPS[m % 8]."""
    X = np.zeros((M, K), dtype=np.uint16)
    half = (np.arange(K) % 32) >= 16
    for m in range(M):
        sel = half if m % 2 else ~half
        X[m, sel] = pow2_bits(EXPS[m % 8], act)
    return X


def assert_exact(Y, ref, what):
    Y = np.asarray(Y, dtype=np.float64)
    assert Y.shape == ref.shape
    bad = np.flatnonzero(Y.ravel() != ref.ravel())
    assert bad.size == 0, (f"{what}: {bad.size} outputs differ; first at {np.unravel_index(bad[0], Y.shape)}: "
                           f"{Y.flat[bad[0]]!r} vs {ref.flat[bad[0]]!r}")


def test_code_matrix_covers_every_byte_with_every_scale():
    """The construction itself: each (qs byte, scale byte) pair occurs in each scale slot."""
    for variant in (DUAL, FAST):
        W = code_matrix(variant)
        bb = synth.block_bytes(variant)
        nb = W.shape[1] // bb
        blocks = W.reshape(-1, nb, bb)
        nz = blocks[:, :, :16].any(axis=2)
        assert np.all(nz.sum(axis=1) <= 1)
        r, blk = np.nonzero(nz)
        qs = blocks[r, blk, :16]
        byte = qs.max(axis=1)
        lo = set(zip(byte.tolist(), blocks[r, blk, 16].tolist()))
        hi = set(zip(byte.tolist(), blocks[r, blk, 17 if variant == DUAL else 16].tolist()))
        assert len(lo) == 255 * NSCALE and len(hi) == 255 * NSCALE  # byte 0 leaves no trace
        assert oracle.validate(W, W.shape[0], nb * 32, variant) == -1


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_streaming_kernel_every_code_and_scale(variant, act, M):
    K = kmin(variant)
    Wh = code_matrix(variant, K)
    N = Wh.shape[0]
    W = upload_w(Wh)
    launches = rf4.launch_count()
    if M == 1:
        for m in range(2):  # both halves of every block through the column-split route
            Xh = mask_rows(2, K, act)[m]
            y = rf4.gemv(W, upload_x(Xh, act), N, K, variant).cpu().numpy()
            assert_exact(y, oracle.gemv(Wh, Xh, N, K, variant, act=act), f"gemv half {m} v={variant} act={act}")
        assert rf4.launch_count() - launches == 2
    else:
        Xh = mask_rows(M, K, act)
        Y = rf4.gemm(W, upload_x(Xh, act), N, K, variant).cpu().numpy()
        assert_exact(Y, oracle.gemm(Wh, Xh, N, K, variant, act=act), f"M={M} v={variant} act={act}")
        assert rf4.launch_count() - launches == 1


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
def test_tensor_core_kernel_every_code_and_scale(variant, act):
    K = kmin(variant)
    Wh = code_matrix(variant, K)
    N = Wh.shape[0]
    Xh = mask_rows(16, K, act)  # M = 16: the tensor-core kernel
    Y = rf4.gemm(upload_w(Wh), upload_x(Xh, act), N, K, variant).cpu().numpy()
    assert_exact(Y, oracle.gemm(Wh, Xh, N, K, variant, act=act), f"tc v={variant} act={act}")


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("M", [1, 4])
def test_gate_up_every_code_and_scale(variant, M):
    """Up rows are the code matrix; every gate row sums to exactly 1 under both
    masks (weights 1.0 at positions 0 and 16), so Y = S * u with S the kernel's
    SiLU(1).  S must be SiLU(1) to the fast exponential's accuracy, and every
    output the fp32 product of S and the oracle's exact up weight."""
    K = kmin(variant)
    up = code_matrix(variant, K)
    I = up.shape[0]
    bb = synth.block_bytes(variant)
    gate = np.zeros_like(up)
    gate[:, 0] = 0x22                 # codes 2, 2 at positions 0 and 16: Codebook10 2
    gate[:, 16:bb] = 0x38             # E4M3 1.0: half-scale 0.5, so both weights are 1.0
    Wh = np.concatenate([gate, up])
    Xh = np.zeros((M, K), dtype=np.uint16)
    half = (np.arange(K) % 32) >= 16
    for m in range(M):
        Xh[m, half if m % 2 else ~half] = pow2_bits(0, F16)
    Y = rf4.gemv_gate_up(upload_w(Wh), upload_x(Xh, F16), I, K, variant).cpu().numpy()
    U = oracle.gemm(up, Xh, I, K, variant)
    G = oracle.gemm(gate, Xh, I, K, variant)
    assert np.all(G == 1.0)
    silu1 = 1.0 / (1.0 + np.exp(-1.0))
    for m in range(M):
        ones = np.flatnonzero(U[m] == 1.0)
        assert ones.size > 0
        S = np.float32(Y[m, ones[0]])
        assert abs(float(S) - silu1) <= 4e-6 * silu1, (m, float(S), silu1)
        expect = (S * U[m].astype(np.float32)).astype(np.float64)
        assert_exact(Y[m], expect, f"gate/up v={variant} row {m}")


@pytest.mark.parametrize("variant", [DUAL, FAST])
@pytest.mark.parametrize("act", [F16, BF16])
def test_attention_value_rows_every_code_and_scale(variant, act):
    """One-token caches: softmax of one score is 1, so out[b, h] is V row 0 of
    KV head h / G, decoded.  Sequence b's V rows use scale byte b (dual: the
    second scale byte 37 b + 11 mod 127); KV head k of it holds the qs byte
    values 64k .. 64k + 63 in its four blocks."""
    t = torch()
    B, Hkv, G, D, Tmax = NSCALE, 4, 2, 128, 32
    H = Hkv * G
    bb = synth.block_bytes(variant)
    rb = synth.row_bytes(D, variant)
    V = synth.weights(B * Hkv * Tmax, D, variant, seed=60, stream=4300).reshape(B, Hkv, Tmax, rb).copy()
    V[:, :, 1:] = 0xFF  # rows past the length: never read as data
    for b in range(B):
        for k in range(Hkv):
            row = V[b, k, 0]
            for blk in range(D // 32):
                row[blk * bb:blk * bb + 16] = np.arange(16, dtype=np.uint8) + 64 * k + 16 * blk
                row[blk * bb + 16] = b
                if variant == DUAL:
                    row[blk * bb + 17] = (37 * b + 11) % NSCALE
    Kc = synth.weights(B * Hkv * Tmax, D, variant, seed=60, stream=4301)
    qh = synth.activations(B * H, D, act, seed=60, stream=4302).reshape(B, H, D)
    lens = np.ones(B, dtype=np.int32)
    out = rf4.decode_attention(upload_x(qh, act), upload_w(Kc), upload_w(V), t.from_numpy(lens).cuda(), Hkv, Tmax,
                               0.125, variant).cpu().numpy()
    Vd = oracle.dequant(V[:, :, 0].reshape(-1), B * Hkv, D, variant).reshape(B, Hkv, D)
    expect = np.repeat(Vd, G, axis=1)
    assert_exact(out, expect, f"attention V v={variant} act={act}")
    ref = oracle.decode_attention(qh, Kc, V, lens, B, H, Hkv, D, Tmax, 0.125, variant, act=act)
    assert_exact(out, ref, f"attention V vs oracle v={variant} act={act}")


@pytest.mark.parametrize("variant", [DUAL, FAST])
def test_attention_key_rows_every_code_and_scale(variant):
    """K rows over every qs byte and every finite scale byte (sequence b uses
    scale byte b), 32 tokens per sequence, against the oracle within the
    attention bound; V rows are ordinary blocks."""
    from test_gpu_attention import bound
    t = torch()
    B, Hkv, G, D, Tmax = NSCALE, 4, 2, 128, 32
    H = Hkv * G
    bb = synth.block_bytes(variant)
    rb = synth.row_bytes(D, variant)
    Kc = np.zeros((B, Hkv, Tmax, rb), dtype=np.uint8)
    vals = np.arange(Hkv * Tmax * (D // 32) * 16) % 256  # each byte value 32 times per sequence
    for b in range(B):
        blocks = Kc[b].reshape(Hkv * Tmax * (D // 32), bb)
        blocks[:, :16] = vals.reshape(-1, 16)
        blocks[:, 16] = b
        if variant == DUAL:
            blocks[:, 17] = (37 * b + 11) % NSCALE
    Kc = Kc.reshape(-1)
    Vh = synth.weights(B * Hkv * Tmax, D, variant, seed=61, stream=4310)
    qh = synth.activations(B * H, D, F16, seed=61, stream=4311).reshape(B, H, D)
    lens = np.full(B, Tmax, dtype=np.int32)
    scale = 1e-3
    out = rf4.decode_attention(upload_x(qh, F16), upload_w(Kc), upload_w(Vh), t.from_numpy(lens).cuda(), Hkv, Tmax,
                               scale, variant).cpu().numpy().astype(np.float64)
    ref = oracle.decode_attention(qh, Kc, Vh, lens, B, H, Hkv, D, Tmax, scale, variant)
    lim = bound(qh, Kc, Vh, lens, B, H, Hkv, D, Tmax, scale, variant, F16)
    err = np.abs(out - ref)
    worst = np.unravel_index(np.argmax(err - lim), err.shape)
    assert np.all(err <= lim), f"|err| {err[worst]:.3e} > {lim[worst[0], worst[1], 0]:.3e} at {worst}"
    # the scores of the large-scale sequences are far from uniform, so a wrong K decode shows
    Kd = oracle.dequant(Kc, B * Hkv * Tmax, D, variant).reshape(B, Hkv, Tmax, D)
    spread = max(np.ptp(scale * Kd[NSCALE - 1, h // G] @ synth.bits_to_float(qh[NSCALE - 1, h], F16))
                 for h in range(H))
    assert spread > 2  # some head's softmax weights spread over a factor e^2 or more
