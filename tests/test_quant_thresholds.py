"""CPU checks of the facts the GPU quantiser's packed comparisons rest on.

The quantiser picks, per value, the nearest Codebook10 magnitude by comparing
|x| with the midpoints (0.5, 1.5, 2.5, 3.5, 5, 7, 9) times the group's
half-scale ("Feasibility Report: Porting ROCmFP4 to Atlas", section "What is
ROCmFP4?": Codebook10 Value Table, Scale Format).  The kernel compares in the
source's own 16-bit format, two values at a time, which is the exact
comparison only if every threshold is exactly representable there; and it
counts in packed halves from 1024 (fp16) / 128 (bf16), which needs k + base
exact with k in the low bits.
"""
import numpy as np
import pytest

MIDPOINTS = (0.5, 1.5, 2.5, 3.5, 5.0, 7.0, 9.0)


def ue4m3(e):
    E, M = (e >> 3) & 15, e & 7
    return 2.0 ** (E - 7) * (1 + M / 8) if E else M / 512.0


def exact_in_f16(v):
    return float(np.float16(v)) == v


def exact_in_bf16(v):
    bits = np.array([v], dtype=np.float32).view(np.uint32)[0]
    return (bits & 0xFFFF) == 0 and float(np.float32(v)) == v


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_every_threshold_is_exact_in_the_source_format(fmt):
    exact = exact_in_f16 if fmt == "f16" else exact_in_bf16
    for e in range(0x7F):  # every finite scale byte
        hs = 0.5 * ue4m3(e)
        for m in MIDPOINTS:
            t = m * hs  # exact in fp64 (and fp32): at most 8 significant bits
            assert float(np.float32(t)) == t
            assert exact(t), (fmt, hex(e), m, t)
            if t > 0:
                # inside the normal range of the format (no subnormal thresholds)
                assert t >= (2.0 ** -14 if fmt == "f16" else 2.0 ** -126)
                assert t <= 2016.0


@pytest.mark.parametrize("fmt,base,base_bits", [("f16", 1024.0, 0x6400), ("bf16", 128.0, 0x4300)])
def test_packed_count_base(fmt, base, base_bits):
    for k in range(8):
        v = base + k
        if fmt == "f16":
            bits = int(np.array([v], dtype=np.float16).view(np.uint16)[0])
            assert exact_in_f16(v)
        else:
            assert exact_in_bf16(v)
            bits = int(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)
        assert bits == base_bits + k and bits & 7 == k


def test_comparison_in_the_source_format_equals_the_fp32_comparison():
    """Brute force over every fp16 value and a spread of bf16 values against
    the thresholds of a sample of scale bytes."""
    f16 = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)  # every finite non-negative fp16
    rng = np.random.default_rng(7)
    bf = (rng.integers(0, 0x7F80, size=20000).astype(np.uint32) << 16).view(np.float32)
    for e in (0x01, 0x07, 0x08, 0x38, 0x40, 0x55, 0x7E):
        hs = 0.5 * ue4m3(e)
        for m in MIDPOINTS:
            t = m * hs
            assert np.array_equal(f16 > np.float16(t), f16.astype(np.float32) > np.float32(t))
            tb = np.float32(t)
            assert np.array_equal(bf > tb, bf.astype(np.float64) > t)
