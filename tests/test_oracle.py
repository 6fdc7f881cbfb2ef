"""CPU tests of the oracle: pins to the pages, invariants, and planted mistakes."""
import os

import numpy as np
import pytest

import oracle
import synth
from oracle_pins import f16_bits, pin_failures

DUAL, FAST = oracle.DUAL, oracle.FAST


def test_oracle_meets_every_pin():
    assert pin_failures() == []


# Plausible mistakes, planted in a copy of the oracle source.  Each one must be
# caught by at least one pin (so a pin that passes means something).
MUTANTS = {
    "nibble pairs order": ("unsigned byte = qs[i % 16];\n  return (i < 16) ? (byte & 0xFu) : (byte >> 4);",
                           "unsigned byte = qs[i / 2];\n  return (i % 2 == 0) ? (byte & 0xFu) : (byte >> 4);"),
    "nibble halves swapped": ("return (i < 16) ? (byte & 0xFu) : (byte >> 4);",
                              "return (i < 16) ? (byte >> 4) : (byte & 0xFu);"),
    "half-scale factor dropped": ("return 0.5 * oracle_ue4m3_value(s);", "return oracle_ue4m3_value(s);"),
    "exponent bias 8": ("(int)e - 7);", "(int)e - 8);"),
    "mantissa /16": ("ldexp(1.0 + (double)m / 8.0", "ldexp(1.0 + (double)m / 16.0"),
    "subnormal as normal": ("if (e == 0) return ldexp((double)m / 8.0, -6);",
                            "if (e == 0) return ldexp(1.0 + (double)m / 8.0, -7);"),
    "first scale for both halves": ("blk[16 + i / 16]", "blk[16]"),
    "scale halves swapped": ("blk[16 + i / 16]", "blk[17 - i / 16]"),
    "codebook 12 kept": ("0, 1, 2, 3, 4, 6, 8, 10,\n", "0, 1, 2, 3, 4, 6, 8, 12,\n"),
    "sign dropped": ("0, -1, -2, -3, -4, -6, -8, -10,", "0, 1, 2, 3, 4, 6, 8, 10,"),
    "last term dropped": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k + 1 < K; ++k) {"),
    "activation row fixed": ("const uint16_t *xr = j->X + m * K;", "const uint16_t *xr = j->X;"),
    "output transposed": ("j->Y[m * j->N + n] = acc;", "j->Y[n * j->M + m] = acc;"),
    "fp16 exponent off by one": ("ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    "bf16 mantissa width": ("ldexp((double)(128 + m), e - 134)", "ldexp((double)(128 + m), e - 133)"),
    "validate misses second scale": ("(variant == ORACLE_DUAL) ? 2 : 1;", "1;"),
    "0x7F accepted": ("return s < 0x7Fu;", "return s < 0x80u;"),
    "fast block 18 bytes": ("if (variant == ORACLE_FAST) return 17;", "if (variant == ORACLE_FAST) return 18;"),
    "gate and up swapped": ("Y[m * I + i] = oracle_silu(g) * u;", "Y[m * I + i] = oracle_silu(u) * g;"),
    "sigmoid of -g": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    "up read from the gate row": ("const double u = gu[m * 2 * I + I + i];", "const double u = gu[m * 2 * I + i];"),
    "gate/up output transposed": ("Y[m * I + i] = oracle_silu(g) * u;", "Y[i * M + m] = oracle_silu(g) * u;"),
    "attention max not subtracted": ("const double p = exp(s[t] - smax);", "const double p = exp(s[t]);"),
    "kv head by modulo": ("const int64_t hk = h / G;", "const int64_t hk = h % Hkv;"),
    "lengths ignored": ("int64_t T = lens[b];", "int64_t T = Tmax;"),
    "scale dropped": ("s[t] = scale * acc;", "s[t] = acc;"),
    "values read from K": ("oracle_dequant(Vc + ((b * Hkv + hk) * Tmax + t) * rb", "oracle_dequant(Kc + ((b * Hkv + hk) * Tmax + t) * rb"),
    "denominator dropped": ("for (int64_t d = 0; d < D; ++d) o[d] /= denom;", "(void)denom;"),
    "quant ties to the larger": ("while (k < 7 && a > oracle_cb_mid[k] * hs) ++k;", "while (k < 7 && a >= oracle_cb_mid[k] * hs) ++k;"),
    "quant scale one too large": ("if (5.0 * oracle_ue4m3_value(e) >= amax) return e;", "if (5.0 * oracle_ue4m3_value(e) > amax) return e;"),
    "quant one scale for both halves": ("const int groups = variant == ORACLE_DUAL ? 2 : 1,", "const int groups = 1,"),
    "quant sign dropped": ("return x < 0.0 ? 8u + k : k;", "return k;"),
    "quant nibbles swapped": ("blk[j] = (uint8_t)(code[j] | (code[j + 16] << 4));", "blk[j] = (uint8_t)(code[j + 16] | (code[j] << 4));"),
    "quant midpoint 4.5": ("{0.5, 1.5, 2.5, 3.5, 5.0, 7.0, 9.0}", "{0.5, 1.5, 2.5, 3.5, 4.5, 7.0, 9.0}"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    L = oracle.bind(oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so")))
    assert pin_failures(L) != [], f"no pin catches: {name}"


# ---- invariants -------------------------------------------------------------

def _rand_blocks(n, variant, seed):
    return synth.weights(n, 32, variant, seed=seed, stream=99)


def test_fast_equals_dual_with_equal_scales():
    fast = _rand_blocks(64, FAST, 1)
    for row in fast:
        dual = np.concatenate([row[:16], [row[16], row[16]]]).astype(np.uint8)
        wf = oracle.decode_block(row, FAST)
        wd = oracle.decode_block(dual, DUAL)
        assert np.array_equal(wf.view(np.uint64), wd.view(np.uint64))


def test_sign_bit_negates_exactly():
    blocks = _rand_blocks(32, DUAL, 2)
    for blk in blocks:
        w = oracle.decode_block(blk, DUAL)
        flipped = blk.copy()
        flipped[:16] ^= 0x88  # bit 3 of both nibbles of every byte
        wf = oracle.decode_block(flipped, DUAL)
        nz = w != 0
        assert np.array_equal(wf[nz], -w[nz])
        assert np.all(wf[~nz] == 0) and not np.any(np.signbit(wf[~nz]))


def test_exponent_increment_doubles_its_half():
    blk = _rand_blocks(1, DUAL, 3)[0].copy()
    blk[16], blk[17] = 0x2B, 0x45
    w = oracle.decode_block(blk, DUAL)
    up = blk.copy()
    up[17] += 0x08  # E -> E+1 on the second half only
    wu = oracle.decode_block(up, DUAL)
    assert np.array_equal(wu[:16], w[:16])
    assert np.array_equal(wu[16:], 2 * w[16:])


def test_linearity_and_power_of_two_scaling():
    N, K = 7, 256
    W = synth.weights(N, K, DUAL, seed=5, stream=3)
    x = synth.activations(1, K, synth.ACT_F16, seed=5, stream=4)[0]
    xf = x.view(np.float16).astype(np.float64)
    y = oracle.gemv(W, x, N, K, DUAL)
    y4 = oracle.gemv(W, f16_bits(xf * 4), N, K, DUAL)
    assert np.array_equal(y4, 4 * y)
    x2 = synth.activations(1, K, synth.ACT_F16, seed=6, stream=4)[0]
    xs = f16_bits(xf + x2.view(np.float16).astype(np.float64))
    ys = oracle.gemv(W, xs, N, K, DUAL)
    dense = oracle.dequant(W, N, K, DUAL)
    ref = dense @ xs.view(np.float16).astype(np.float64)
    assert np.allclose(ys, ref, rtol=1e-14, atol=1e-12)


def test_gaussian_inputs_match_dense_fp64_matmul():
    for var, act in ((DUAL, synth.ACT_F16), (FAST, synth.ACT_BF16)):
        N, K, M = 33, 512, 4
        W = synth.weights(N, K, var, seed=9, stream=5)
        X = synth.activations(M, K, act, seed=9, stream=6)
        Y = oracle.gemm(W, X, N, K, var, act=act)
        xf = synth.bits_to_float(X, act).astype(np.float64)
        dense = oracle.dequant(W, N, K, var)
        assert np.all(np.abs(Y - xf @ dense.T) <= 1e-14 * (np.abs(xf) @ np.abs(dense).T) + 1e-300)


def test_thread_count_does_not_change_bits():
    N, K = 41, 320
    W = synth.weights(N, K, FAST, seed=1, stream=1)
    X = synth.activations(2, K, synth.ACT_F16, seed=1, stream=2)
    a = oracle.gemm(W, X, N, K, FAST, nthreads=1)
    b = oracle.gemm(W, X, N, K, FAST, nthreads=os.cpu_count() or 4)
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64))


def test_shape_errors_and_empty():
    W = np.zeros(18, dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.dequant(W, 1, 33, DUAL)
    assert oracle.gemm(np.zeros(0, np.uint8), np.zeros((1, 0), np.uint16), 0, 0, DUAL).shape == (1, 0)
    assert oracle.dequant(np.zeros(0, np.uint8), 0, 64, FAST).shape == (0, 64)
