"""CPU tests of the C ABI: the library loads, exports every declared entry
point, and rejects bad arguments on the host without touching a GPU."""
import ctypes
import os
import re

import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
from gemm_rocmfp4_dequant_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rocmfp4.h")


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return rf4.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rocmfp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("rocmfp4_gemv", "rocmfp4_gemm", "rocmfp4_gemv_ex", "rocmfp4_gemm_ex", "rocmfp4_dequant",
                     "rocmfp4_validate", "rocmfp4_block_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert missing == []
    assert set(declared_functions()) <= set(rf4.EXPORTS) | {"rocmfp4_device_error_bits"}


def test_block_and_row_bytes(L):
    assert rf4.block_bytes(rf4.DUAL) == 18 and rf4.block_bytes(rf4.FAST) == 17
    assert rf4.block_bytes(7) == 0
    assert rf4.row_bytes(5120, rf4.DUAL) == 2880 and rf4.row_bytes(5120, rf4.FAST) == 2720
    assert rf4.row_bytes(33, rf4.DUAL) == 0 and rf4.row_bytes(-32, rf4.DUAL) == 0


def test_status_strings(L):
    for code, name in rf4.STATUS.items():
        assert L.rocmfp4_status_string(code).decode() == name


def _vp(v):
    return ctypes.c_void_p(v)


def test_host_argument_checks_return_invalid_arg(L):
    fake = _vp(0x1000)  # never dereferenced: every call below fails its host checks
    null = _vp(0)
    ok_stream = _vp(0)
    # K not a multiple of 32
    assert L.rocmfp4_gemv(fake, fake, fake, 4, 33, 0) == 1
    # unknown variant / activation type
    assert L.rocmfp4_gemv(fake, fake, fake, 4, 32, 5) == 1
    assert L.rocmfp4_gemv_ex(fake, fake, fake, 4, 32, 0, 9, ok_stream) == 1
    # negative sizes
    assert L.rocmfp4_gemm(fake, fake, fake, -1, 4, 32, 0) == 1
    assert L.rocmfp4_gemm(fake, fake, fake, 1, -4, 32, 0) == 1
    # NULL pointers with a non-empty shape
    assert L.rocmfp4_gemm(null, fake, fake, 1, 4, 32, 0) == 1
    assert L.rocmfp4_gemm(fake, null, fake, 1, 4, 32, 0) == 1
    assert L.rocmfp4_gemm(fake, fake, null, 1, 4, 32, 0) == 1
    assert L.rocmfp4_dequant(fake, null, 0, 4, 32, 0, ok_stream) == 1
    assert L.rocmfp4_dequant(fake, fake, 7, 4, 32, 0, ok_stream) == 1
    assert L.rocmfp4_validate(fake, 4, 40, 0, None, ok_stream) == 1
    assert b"multiple of 32" in L.rocmfp4_last_error() or L.rocmfp4_last_error() != b""
    # staging copy: negative size, NULL pointers, overlapping ranges
    assert L.rocmfp4_copy(fake, _vp(0x9000), -1, ok_stream) == 1
    assert L.rocmfp4_copy(null, fake, 16, ok_stream) == 1
    assert L.rocmfp4_copy(fake, null, 16, ok_stream) == 1
    assert L.rocmfp4_copy(_vp(0x1000), _vp(0x1008), 16, ok_stream) == 1
    assert L.rocmfp4_copy(_vp(0x1008), _vp(0x1000), 16, ok_stream) == 1
    assert b"overlapping" in L.rocmfp4_last_error()


def test_empty_shapes_are_no_ops(L):
    null = _vp(0)
    assert L.rocmfp4_gemm(null, null, null, 0, 8, 64, 0) == 0
    assert L.rocmfp4_gemm(null, null, null, 3, 0, 64, 0) == 0
    assert L.rocmfp4_dequant(null, null, 0, 0, 64, 1, null) == 0
    assert L.rocmfp4_copy(null, null, 0, null) == 0
    first = ctypes.c_int64(5)
    assert L.rocmfp4_validate(null, 0, 64, 0, ctypes.byref(first), null) == 0 and first.value == -1
