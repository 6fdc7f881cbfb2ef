"""GPU test of rocmfp4_gemm_noalloc, the entry point for callers that cannot
allocate device memory (an engine whose memory all belongs to its own pool,
code running during CUDA graph capture, or a host that forbids allocation
after start-up).  It must give the same products as rocmfp4_gemm_ex, within
the tolerance every product test here uses, on consecutive calls that share
its fixed scratch array.

This file is named so that pytest collects it last; it also passes alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import synth
import synth.device
from gpu_util import assert_close, max_halfscale, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return rf4.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch().cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("variant", [rf4.DUAL, rf4.FAST])
@pytest.mark.parametrize("N,K,M", [(1000, 2048, 1), (777, 1536, 3), (34816, 5120, 1), (5120, 17408, 8)])
def test_noalloc_matches_allocating_entry_point_twice(L, variant, N, K, M):
    t = torch()
    rb = rf4.row_bytes(K, variant)
    W = t.empty(N * rb, dtype=t.uint8, device="cuda")
    synth.device.fill_weights(W, N, K, variant, seed=11, stream=3)
    X = t.empty((M, K), dtype=t.int16, device="cuda")
    synth.device.fill_act(X, synth.ACT_F16, seed=11, stream=4)
    ref = t.empty((M, N), dtype=t.float32, device="cuda")
    st = L.rocmfp4_gemm_ex(_p(W), _p(X), _p(ref), M, N, K, variant, rf4.ACT_F16, _stream())
    assert st == 0, L.rocmfp4_last_error()
    max_hs = max_halfscale(W[: min(N, 64) * rb].cpu().numpy(), variant)
    for call in range(2):
        Y = t.full((M, N), float("nan"), dtype=t.float32, device="cuda")
        st = L.rocmfp4_gemm_noalloc(_p(W), _p(X), _p(Y), M, N, K, variant, rf4.ACT_F16, _stream())
        assert st == 0, L.rocmfp4_last_error()
        t.cuda.synchronize()
        assert_close(Y.cpu().numpy(), ref.cpu().numpy().astype(np.float64), K, max_hs, f"noalloc call {call}")
    assert rf4.device_error_bits() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    t = torch()
    W = t.zeros(18 * 8 * 32, dtype=t.uint8, device="cuda")
    X = t.zeros((9, 256), dtype=t.float16, device="cuda")
    Y = t.zeros((9, 32), dtype=t.float32, device="cuda")
    st = L.rocmfp4_gemm_noalloc(_p(W), _p(X), _p(Y), 9, 32, 256, rf4.DUAL, rf4.ACT_F16, _stream())
    assert st == 2  # ROCMFP4_ERR_UNSUPPORTED
    assert b"M > 8" in L.rocmfp4_last_error()
