"""Plain-read ceiling kernel for the benchmark (measurement only, not part of the library).

Builds ``ceiling/_build/libreadceil.so`` from ``read.cu``: one kernel that
streams a device buffer into shared memory with bulk copies and folds every
word into an XOR checksum.  bench.py times it beside each weight product, on
copies of the same bytes, as the read ceiling of a launch of that size.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "read.cu")
LIB = os.path.join(_HERE, "_build", "libreadceil.so")
MAX_SMEM = 227 * 1024
# (chunk bytes, warps per CTA, CTAs per SM, stages): the configurations the
# benchmark tries per buffer; it keeps the fastest.
CONFIGS = [(4608, 4, 4, 2), (9216, 4, 2, 2), (18432, 4, 1, 2), (9216, 8, 1, 2)]
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
                    "-Xcompiler", "-fPIC", "-shared", SRC, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.readceil_launch.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        L.readceil_launch.restype = ctypes.c_int
        L.readceil_prepare.argtypes = [ctypes.c_int]
        L.readceil_prepare.restype = ctypes.c_int
        L.readceil_smem.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.readceil_smem.restype = ctypes.c_size_t
        rc = L.readceil_prepare(MAX_SMEM)
        if rc != 0:
            raise RuntimeError(f"readceil_prepare failed: {rc}")
        _lib = L
    return _lib


def read(buf, sink, config, sms: int, stream=None) -> None:
    """Launch one read of the uint8 CUDA tensor `buf` (its whole storage) with
    `config` = (chunk, warps, ctas_per_sm, stages); `sink` is a 2-word int32
    CUDA tensor (checksum, gave-up flag)."""
    import torch
    chunk, warps, per_sm, stages = config
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = lib().readceil_launch(ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size(), chunk, warps,
                               per_sm * sms, stages, ctypes.c_void_p(sink.data_ptr()), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"readceil_launch failed: {rc}")
