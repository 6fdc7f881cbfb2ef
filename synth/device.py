"""CUDA fill kernels of the seeded input generator (same definition as the numpy side).

Builds ``synth/_build/libsynth.so`` from ``synth.cu``; holds no ROCmFP4 arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "synth.cu")
LIB = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", SRC, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i64, u64, c_int, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
        L.synth_fill_weights.argtypes = [vp, i64, i64, c_int, u64, u64, vp]
        L.synth_fill_weights.restype = c_int
        L.synth_fill_act.argtypes = [vp, i64, i64, c_int, u64, u64, vp]
        L.synth_fill_act.restype = c_int
        _lib = L
    return _lib


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_weights(W, N: int, K: int, variant: int, seed: int, stream: int) -> None:
    """Fill a uint8 CUDA tensor with the packed matrix of (seed, stream)."""
    rc = lib().synth_fill_weights(ctypes.c_void_p(W.data_ptr()), N, K, variant, seed, stream, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_fill_weights failed: {rc}")


def fill_act(X, act: int, seed: int, stream: int, first: int = 0) -> None:
    """Fill a 16-bit CUDA tensor with activation elements first.. of (seed, stream)."""
    rc = lib().synth_fill_act(ctypes.c_void_p(X.data_ptr()), X.numel(), first, act, seed, stream, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_fill_act failed: {rc}")
