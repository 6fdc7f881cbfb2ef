"""ROCmFP4 CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (``rocmfp4_oracle.c``) of what the ROCmFP4
block-quantised weight product computes, with a ctypes wrapper.  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package; the library under ``gemm_rocmfp4_dequant_gb300`` never
does, and this package imports nothing from it.

Definitions follow "Feasibility Report: Porting ROCmFP4 to Atlas", section
"What is ROCmFP4?" (subsections "Block Layout", "Codebook10 Value Table",
"Scale Format").  The readings R1-R6 taken where that text is silent are listed
at the top of the C file.  On-disk compatibility with files written by the
original implementation is parity unpinned (no such file or printed example
exists).

Every function takes an optional ``L`` (a library returned by :func:`bind`);
the tests use it to run the same pins against deliberately broken copies of
the oracle and check that the pins catch them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "rocmfp4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_rocmfp4.so")

DUAL, FAST = 0, 1
ACT_F16, ACT_BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc -O2, no fast-math, no contraction: the oracle's only build recipe."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build (skipped when up to date)."""
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)
    if fresh and not force:
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def bind(path: str) -> ctypes.CDLL:
    """Load an oracle library and declare its C signatures."""
    L = ctypes.CDLL(path)
    i64, c_int, c_dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    sigs = {
        "oracle_block_bytes": ([c_int], c_int),
        "oracle_codebook": ([c_int], c_int),
        "oracle_scale_is_valid": ([ctypes.c_uint], c_int),
        "oracle_ue4m3_value": ([ctypes.c_uint], c_dbl),
        "oracle_halfscale": ([ctypes.c_uint], c_dbl),
        "oracle_act_value": ([ctypes.c_uint16, c_int], c_dbl),
        "oracle_decode_block": ([vp, c_int, vp], None),
        "oracle_dequant": ([vp, i64, i64, c_int, vp], c_int),
        "oracle_validate": ([vp, i64, i64, c_int], i64),
        "oracle_gemm": ([vp, vp, c_int, vp, i64, i64, i64, c_int, c_int], c_int),
        "oracle_gemv_gate_up": ([vp, vp, c_int, vp, i64, i64, i64, c_int, c_int], c_int),
        "oracle_decode_attention": ([vp, c_int, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_dbl, c_int], c_int),
        "oracle_quantize": ([vp, c_int, vp, i64, i64, c_int], c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _L(L):
    return lib() if L is None else L


def block_bytes(variant: int, L=None) -> int:
    return _L(L).oracle_block_bytes(int(variant))


def row_bytes(K: int, variant: int, L=None) -> int:
    return (K // 32) * block_bytes(variant, L)


def codebook(q: int, L=None) -> int:
    return _L(L).oracle_codebook(int(q))


def scale_is_valid(s: int, L=None) -> bool:
    return bool(_L(L).oracle_scale_is_valid(int(s)))


def ue4m3(s: int, L=None) -> float:
    return _L(L).oracle_ue4m3_value(int(s))


def halfscale(s: int, L=None) -> float:
    return _L(L).oracle_halfscale(int(s))


def act_value(bits: int, act: int, L=None) -> float:
    return _L(L).oracle_act_value(int(bits), int(act))


def decode_block(blk, variant: int, L=None) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    assert blk.size >= block_bytes(variant, L)
    w = np.empty(32, dtype=np.float64)
    _L(L).oracle_decode_block(blk.ctypes.data, int(variant), w.ctypes.data)
    return w


def dequant(W, N: int, K: int, variant: int, L=None) -> np.ndarray:
    """fp64 [N, K] weights of a packed ROCmFP4 matrix."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= N * row_bytes(K, variant, L)
    out = np.empty((N, K), dtype=np.float64)
    rc = _L(L).oracle_dequant(W.ctypes.data, N, K, int(variant), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_dequant rejected N={N} K={K} variant={variant}")
    return out


def validate(W, N: int, K: int, variant: int, L=None) -> int:
    """Index (row-major over blocks) of the first block with a non-finite scale byte, or -1."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rc = _L(L).oracle_validate(W.ctypes.data, N, K, int(variant))
    if rc == -2:
        raise ValueError("oracle_validate: bad shape")
    return int(rc)


def gemm(W, X_bits, N: int, K: int, variant: int, act: int = ACT_F16,
         nthreads: int | None = None, L=None) -> np.ndarray:
    """fp64 Y[M, N] = X[M, K] . W[N, K]^T with X given as fp16/bf16 bit patterns (uint16)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    X = np.ascontiguousarray(X_bits, dtype=np.uint16)
    if X.ndim == 1:
        X = X.reshape(1, -1)
    M = X.shape[0]
    assert X.shape[1] == K, (X.shape, K)
    assert W.size >= N * row_bytes(K, variant, L)
    Y = np.empty((M, N), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _L(L).oracle_gemm(W.ctypes.data, X.ctypes.data, int(act), Y.ctypes.data, M, N, K,
                           int(variant), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_gemm failed with {rc}")
    return Y


def gemv(W, x_bits, N: int, K: int, variant: int, act: int = ACT_F16,
         nthreads: int | None = None, L=None) -> np.ndarray:
    """fp64 y[N] = W . x for one activation vector."""
    return gemm(W, np.asarray(x_bits).reshape(1, K), N, K, variant, act, nthreads, L)[0]


def gemv_gate_up(W, X_bits, I: int, K: int, variant: int, act: int = ACT_F16,
                 nthreads: int | None = None, L=None) -> np.ndarray:
    """fp64 Y[M, I] = SiLU(X . Wg^T) * (X . Wu^T), W holding 2I rows (the gate
    rows, then the up rows) and X given as fp16/bf16 bit patterns.  The formula
    is reading R11 of the "gemv_gate_up" kernel type ("Kernel System" section
    of the report); see the C source."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    X = np.ascontiguousarray(X_bits, dtype=np.uint16)
    if X.ndim == 1:
        X = X.reshape(1, -1)
    M = X.shape[0]
    assert X.shape[1] == K, (X.shape, K)
    assert W.size >= 2 * I * row_bytes(K, variant, L)
    Y = np.empty((M, I), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _L(L).oracle_gemv_gate_up(W.ctypes.data, X.ctypes.data, int(act), Y.ctypes.data, M, I, K,
                                   int(variant), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_gemv_gate_up failed with {rc}")
    return Y


def decode_attention(q_bits, Kc, Vc, lens, B: int, H: int, Hkv: int, D: int, Tmax: int, scale: float,
                     variant: int, act: int = ACT_F16, L=None) -> np.ndarray:
    """fp64 out[B, H, D] of single-token attention over a ROCmFP4 K/V cache
    (reading R12; see the C source): q [B, H, D] as fp16/bf16 bits, Kc and Vc
    [B, Hkv, Tmax] rows of D/32 blocks, lens [B] tokens per sequence."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16).reshape(B, H, D)
    Kc = np.ascontiguousarray(Kc, dtype=np.uint8).reshape(-1)
    Vc = np.ascontiguousarray(Vc, dtype=np.uint8).reshape(-1)
    lens = np.ascontiguousarray(lens, dtype=np.int32).reshape(B)
    need = B * Hkv * Tmax * row_bytes(D, variant, L)
    assert Kc.size >= need and Vc.size >= need, (Kc.size, Vc.size, need)
    out = np.empty((B, H, D), dtype=np.float64)
    rc = _L(L).oracle_decode_attention(q.ctypes.data, int(act), Kc.ctypes.data, Vc.ctypes.data, lens.ctypes.data,
                                       out.ctypes.data, B, H, Hkv, D, Tmax, float(scale), int(variant))
    if rc != 0:
        raise ValueError(f"oracle_decode_attention failed with {rc}")
    return out


def quantize(src_bits, N: int, K: int, variant: int, act: int = ACT_F16, L=None) -> np.ndarray:
    """ROCmFP4 blocks [N, row_bytes] of fp16/bf16 values (bit patterns, [N, K]),
    by the scale and rounding rules of reading R13 (see the C source)."""
    X = np.ascontiguousarray(src_bits, dtype=np.uint16).reshape(N, K)
    W = np.zeros((N, row_bytes(K, variant, L)), dtype=np.uint8)
    rc = _L(L).oracle_quantize(X.ctypes.data, int(act), W.ctypes.data, N, K, int(variant))
    if rc != 0:
        raise ValueError(f"oracle_quantize failed with {rc}")
    return W
