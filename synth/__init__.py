"""Seeded synthetic inputs for the ROCmFP4 tests and benchmark.

This module holds none of the ROCmFP4 arithmetic: it only draws bytes and
activations.  The oracle and the CUDA library both consume what it produces.
The same generator is implemented twice, here in numpy and in ``synth.cu`` as a
CUDA fill kernel (for inputs too large to draw on the host), from one
definition, so that any row of a device-resident matrix can be re-drawn on
the host for the oracle.  The GPU tests check that both sides agree bit for
bit.

Definition
----------
* Counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014): with gamma =
  0x9E3779B97F4A7C15 and the published finaliser ``mix64``,
  ``key = mix64(seed + gamma*(stream+1))`` and the i-th draw of a stream is
  ``draw(i) = mix64(key + gamma*(i+1))`` (all mod 2^64) -- the i-th output of
  a SplitMix64 generator whose state starts at ``key``.
* Weight bytes of a packed matrix (N rows of K/32 blocks of B bytes, B = 18 for
  the dual-scale layout, 17 for the single-scale one): byte g draws r =
  draw(g).  Bytes at offsets 0..15 of a block (the packed nibbles) take r>>56,
  so every nibble is uniform over 0..15.  Scale bytes (offsets 16, 17) take
  exponent field E = 4 + floor((r>>32)*7 / 2^32) (uniform over 4..10) and
  mantissa M = (r>>29) & 7, byte = E<<3 | M.
* Activations ~ N(0, 1) by Box-Muller: element e of a stream uses pair
  p = e//2, u1 = ((draw(2p)>>11) + 1) * 2^-53 in (0, 1],
  u2 = (draw(2p+1)>>11) * 2^-53 in [0, 1); rho = sqrt(-2 ln u1);
  element 2p = rho*cos(2 pi u2), element 2p+1 = rho*sin(2 pi u2).  ln, sin and
  cos are evaluated from their power series with the hex-float coefficients
  below, using only correctly rounded IEEE fp64 +, -, *, /, sqrt in a fixed
  order, so that numpy and CUDA give identical bits.  The fp64 value is
  rounded to fp32 (nearest-even), then to fp16 or bf16 (nearest-even).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_U64 = np.uint64

DUAL, FAST = 0, 1
ACT_F16, ACT_BF16 = 0, 1

# 1/(2j+1), j = 0..13  (series of ln f = 2 atanh t)
LN_COEF = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "0x1.5555555555555p-2", "0x1.999999999999ap-3", "0x1.2492492492492p-3",
    "0x1.c71c71c71c71cp-4", "0x1.745d1745d1746p-4", "0x1.3b13b13b13b14p-4", "0x1.1111111111111p-4",
    "0x1.e1e1e1e1e1e1ep-5", "0x1.af286bca1af28p-5", "0x1.8618618618618p-5", "0x1.642c8590b2164p-5",
    "0x1.47ae147ae147bp-5", "0x1.2f684bda12f68p-5")]
# (-1)^j/(2j+1)!, j = 0..11
SIN_COEF = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "-0x1.5555555555555p-3", "0x1.1111111111111p-7", "-0x1.a01a01a01a01ap-13",
    "0x1.71de3a556c734p-19", "-0x1.ae64567f544e4p-26", "0x1.6124613a86d09p-33", "-0x1.ae7f3e733b81fp-41",
    "0x1.952c77030ad4ap-49", "-0x1.2f49b46814157p-57", "0x1.71b8ef6dcf572p-66", "-0x1.761b41316381ap-75")]
# (-1)^j/(2j)!, j = 0..11
COS_COEF = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "-0x1.0000000000000p-1", "0x1.5555555555555p-5", "-0x1.6c16c16c16c17p-10",
    "0x1.a01a01a01a01ap-16", "-0x1.27e4fb7789f5cp-22", "0x1.1eed8eff8d898p-29", "-0x1.93974a8c07c9dp-37",
    "0x1.ae7f3e733b81fp-45", "-0x1.6827863b97d97p-53", "0x1.e542ba4020225p-62", "-0x1.0ce396db7f853p-70")]
LN2 = float.fromhex("0x1.62e42fefa39efp-1")
HALF_PI = float.fromhex("0x1.921fb54442d18p+0")
SQRT_HALF = float.fromhex("0x1.6a09e667f3bcdp-1")

# Stream ids used by the tests and the benchmark (weights and activations of
# one matrix use different streams).
ACT_STREAM_BASE = 1 << 20


def weight_stream(layer: int, matrix: int) -> int:
    """Stream of the weight bytes of matrix `matrix` (0 QKV, 1 O, 2 gate+up, 3 down, 4 LM head) of layer `layer`."""
    return layer * 8 + matrix


def act_stream(layer: int, matrix: int) -> int:
    return ACT_STREAM_BASE + layer * 8 + matrix


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=_U64)
    z = (z ^ (z >> _U64(30))) * _M1
    z = (z ^ (z >> _U64(27))) * _M2
    return z ^ (z >> _U64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = _U64(seed & 0xFFFFFFFFFFFFFFFF) + GAMMA * _U64(stream + 1)
        return mix64(np.array([s], dtype=_U64))[0]


def draws(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """64-bit draws number idx (any integer array) of a stream."""
    key = stream_key(seed, stream)
    idx = np.asarray(idx, dtype=_U64)
    with np.errstate(over="ignore"):
        return mix64(key + GAMMA * (idx + _U64(1)))


def block_bytes(variant: int) -> int:
    return 18 if variant == DUAL else 17


def row_bytes(K: int, variant: int) -> int:
    return (K // 32) * block_bytes(variant)


def weight_bytes_at(g: np.ndarray, variant: int, seed: int, stream: int) -> np.ndarray:
    """Bytes at global byte offsets g of a packed matrix."""
    g = np.asarray(g, dtype=np.int64)
    r = draws(seed, stream, g.astype(_U64))
    bb = block_bytes(variant)
    pos = g % bb
    nib = (r >> _U64(56)).astype(np.uint8)
    e = _U64(4) + (((r >> _U64(32)) * _U64(7)) >> _U64(32))
    m = (r >> _U64(29)) & _U64(7)
    sc = ((e << _U64(3)) | m).astype(np.uint8)
    return np.where(pos < 16, nib, sc).astype(np.uint8)


def weights(N: int, K: int, variant: int, seed: int = 0, stream: int = 0,
            rows: np.ndarray | None = None) -> np.ndarray:
    """Packed matrix bytes, shape [len(rows) or N, row_bytes]; `rows` selects rows of the full matrix."""
    rb = row_bytes(K, variant)
    r_idx = np.arange(N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((r_idx.size, rb), dtype=np.uint8)
    col = np.arange(rb, dtype=np.int64)
    chunk = max(1, (1 << 22) // max(rb, 1))
    for i in range(0, r_idx.size, chunk):
        rr = r_idx[i:i + chunk]
        g = rr[:, None] * rb + col[None, :]
        out[i:i + chunk] = weight_bytes_at(g, variant, seed, stream)
    return out


# ---- activations -----------------------------------------------------------

def _ln(u: np.ndarray) -> np.ndarray:
    """ln u for u in (0, 1]: u = f*2^e, f in [sqrt(1/2), sqrt(2)), ln f = 2 atanh((f-1)/(f+1))."""
    f, e = np.frexp(u)  # exact: f in [0.5, 1)
    low = f < SQRT_HALF
    f = np.where(low, f * 2.0, f)
    e = np.where(low, e - 1, e).astype(np.float64)
    t = (f - 1.0) / (f + 1.0)
    t2 = t * t
    s = np.full_like(t, LN_COEF[-1])
    for c in reversed(LN_COEF[:-1]):
        s = s * t2
        s = s + c
    lnf = (t * 2.0) * s
    return e * LN2 + lnf


def _sincos_quarter(phi: np.ndarray):
    p2 = phi * phi
    s = np.full_like(phi, SIN_COEF[-1])
    c = np.full_like(phi, COS_COEF[-1])
    for k in reversed(SIN_COEF[:-1]):
        s = s * p2
        s = s + k
    for k in reversed(COS_COEF[:-1]):
        c = c * p2
        c = c + k
    return phi * s, c


def _sincos_turn(u: np.ndarray):
    """(sin, cos) of 2*pi*u for u in [0, 1)."""
    x = u * 4.0                      # exact
    q = np.floor(x)
    r = x - q                        # exact, in [0, 1)
    comp = r > 0.5
    rr = np.where(comp, 1.0 - r, r)  # exact
    phi = rr * HALF_PI               # in [0, pi/4]
    s0, c0 = _sincos_quarter(phi)
    # angle within the quadrant = r*pi/2; the complement swaps sin and cos
    s1 = np.where(comp, c0, s0)
    c1 = np.where(comp, s0, c0)
    qi = q.astype(np.int64) & 3
    sin = np.select([qi == 0, qi == 1, qi == 2, qi == 3], [s1, c1, -s1, -c1])
    cos = np.select([qi == 0, qi == 1, qi == 2, qi == 3], [c1, -s1, -c1, s1])
    return sin, cos


def normal_f64(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """fp64 N(0,1) values number idx of a stream (before rounding to 16 bits)."""
    idx = np.asarray(idx, dtype=np.int64)
    p = idx // 2
    r1 = draws(seed, stream, (2 * p).astype(_U64))
    r2 = draws(seed, stream, (2 * p + 1).astype(_U64))
    u1 = ((r1 >> _U64(11)) + _U64(1)).astype(np.float64) * (2.0 ** -53)
    u2 = (r2 >> _U64(11)).astype(np.float64) * (2.0 ** -53)
    rho = np.sqrt(_ln(u1) * -2.0)
    sin, cos = _sincos_turn(u2)
    return np.where(idx % 2 == 0, rho * cos, rho * sin)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit pattern (finite inputs)."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return (b >> np.uint64(16)).astype(np.uint16)


def act_bits_at(idx: np.ndarray, act: int, seed: int, stream: int) -> np.ndarray:
    v32 = normal_f64(seed, stream, idx).astype(np.float32)
    if act == ACT_F16:
        return v32.astype(np.float16).view(np.uint16)
    return f32_to_bf16_bits(v32)


def activations(M: int, K: int, act: int, seed: int = 0, stream: int = 0,
                rows: np.ndarray | None = None) -> np.ndarray:
    """uint16 bit patterns of an [M, K] activation matrix (or of the selected rows)."""
    r_idx = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((r_idx.size, K), dtype=np.uint16)
    col = np.arange(K, dtype=np.int64)
    chunk = max(1, (1 << 21) // max(K, 1))
    for i in range(0, r_idx.size, chunk):
        rr = r_idx[i:i + chunk]
        out[i:i + chunk] = act_bits_at(rr[:, None] * K + col[None, :], act, seed, stream)
    return out


def bits_to_float(bits: np.ndarray, act: int) -> np.ndarray:
    """fp16/bf16 bit patterns -> float32 values (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if act == ACT_F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
