"""GPU tests of rocmfp4_gemm_noalloc, the product for callers that cannot
allocate device memory where they run it: an inference engine that hands all
device memory to its own pool at start-up, a host with a rule against
allocating after initialisation, or a plug-in that must not touch its host
process's allocator.  Its scratch is a fixed array inside the library, shared
by every call.

Checked here, through the C ABI:
  * two calls in a row give the fp64 oracle's products (rel-L2 1e-5, max |err|
    <= 1e-3 * sqrt(K) * max half-scale), the same bits both times, and the
    products of rocmfp4_gemm_ex within that tolerance (called afterwards);
  * in a fresh process that never calls an allocating entry point, free
    device memory does not change across calls after the first (which looks
    up the array and zeroes its counters), nor across the error query;
  * sizes beyond the array's limit are rejected before any launch.

This file is named so that pytest collects it last; it also passes alone in a
fresh process.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import gemm_rocmfp4_dequant_gb300 as rf4
import oracle
import synth
import synth.device
from gpu_util import assert_close, max_halfscale, torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return rf4.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch().cuda.current_stream().cuda_stream)


# (N, K, M): ragged small shapes (whole oracle), then full-size layer matrices
# whose splits reach the cross-CTA level of the reduction (sampled rows)
CASES = [(1000, 2048, 1), (777, 1536, 3), (200, 1024, 8), (34816, 5120, 1), (5120, 17408, 8), (5120, 17408, 2)]


@pytest.mark.parametrize("variant", [rf4.DUAL, rf4.FAST])
@pytest.mark.parametrize("N,K,M", CASES)
def test_noalloc_twice_matches_oracle_and_allocating_entry_point(L, variant, N, K, M):
    t = torch()
    rb = rf4.row_bytes(K, variant)
    W = t.empty(N * rb, dtype=t.uint8, device="cuda")
    synth.device.fill_weights(W, N, K, variant, seed=11, stream=3)
    Xh = synth.activations(M, K, synth.ACT_F16, seed=11, stream=4)
    X = t.from_numpy(Xh.view(np.int16)).cuda()
    rows = np.arange(N) if N <= 1000 else np.unique(
        np.concatenate([[0, 31, 32, N - 1], np.random.default_rng(N + M).integers(0, N, 96)]))
    Wrows = synth.weights(N, K, variant, seed=11, stream=3, rows=rows)
    ref = oracle.gemm(Wrows, Xh, len(rows), K, variant)
    max_hs = max_halfscale(Wrows, variant)
    outs = []
    for call in range(2):
        Y = t.full((M, N), float("nan"), dtype=t.float32, device="cuda")
        st = L.rocmfp4_gemm_noalloc(_p(W), _p(X), _p(Y), M, N, K, variant, rf4.ACT_F16, _stream())
        assert st == 0, L.rocmfp4_last_error()
        t.cuda.synchronize()
        assert_close(Y.cpu().numpy()[:, rows], ref, K, max_hs, f"noalloc call {call}")
        outs.append(Y)
    assert t.equal(outs[0].view(t.int32), outs[1].view(t.int32))
    assert L.rocmfp4_device_error_bits(_stream()) == 0
    ex = t.empty((M, N), dtype=t.float32, device="cuda")
    st = L.rocmfp4_gemm_ex(_p(W), _p(X), _p(ex), M, N, K, variant, rf4.ACT_F16, _stream())
    assert st == 0, L.rocmfp4_last_error()
    assert_close(outs[1].cpu().numpy(), ex.cpu().numpy().astype(np.float64), K, max_hs, "noalloc vs gemm_ex")


FRESH = r"""
import ctypes, sys
import numpy as np
import torch
sys.path[:0] = [ROOT, HERE]
import gemm_rocmfp4_dequant_gb300 as rf4
import oracle, synth
from gpu_util import assert_close, max_halfscale
L = rf4.load()
N, K, M, v = 5000, 17408, 2, rf4.DUAL
Wh = synth.weights(N, K, v, seed=21, stream=1)
Xh = synth.activations(M, K, synth.ACT_F16, seed=21, stream=2)
W = torch.from_numpy(Wh.reshape(-1)).cuda()
X = torch.from_numpy(Xh.view(np.int16)).cuda()
Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
ref = oracle.gemm(Wh, Xh, N, K, v)
hs = max_halfscale(Wh, v)
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
p = lambda t: ctypes.c_void_p(t.data_ptr())

def call(i):
    Y.fill_(float("nan"))
    st = L.rocmfp4_gemm_noalloc(p(W), p(X), p(Y), M, N, K, v, rf4.ACT_F16, s)
    assert st == 0, L.rocmfp4_last_error()
    torch.cuda.synchronize()
    got = Y.cpu().numpy()
    assert_close(got, ref, K, hs, f"fresh-process call {i}")
    return got

first = call(0)  # set-up: the array's address, its counters zeroed
free0 = torch.cuda.mem_get_info()[0]
for i in range(1, 4):
    assert np.array_equal(call(i).view(np.int32), first.view(np.int32))
free1 = torch.cuda.mem_get_info()[0]
assert L.rocmfp4_device_error_bits(s) == 0
free2 = torch.cuda.mem_get_info()[0]
assert free1 == free0, ("noalloc calls changed free device memory", free0, free1)
assert free2 == free1, ("the error query changed free device memory", free1, free2)
print("FRESH_OK", free0, free1, free2)
"""


def test_noalloc_in_a_fresh_process_allocates_nothing(L):
    code = FRESH.replace("sys.path[:0] = [ROOT, HERE]", f"sys.path[:0] = [{ROOT!r}, {HERE!r}]")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "FRESH_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    t = torch()
    W = t.zeros(18 * 8 * 32, dtype=t.uint8, device="cuda")
    X = t.zeros((9, 256), dtype=t.float16, device="cuda")
    Y = t.zeros((9, 32), dtype=t.float32, device="cuda")
    launches = rf4.launch_count()
    st = L.rocmfp4_gemm_noalloc(_p(W), _p(X), _p(Y), 9, 32, 256, rf4.DUAL, rf4.ACT_F16, _stream())
    assert st == 2  # ROCMFP4_ERR_UNSUPPORTED
    assert b"M > 8" in L.rocmfp4_last_error()
    assert rf4.launch_count() == launches
