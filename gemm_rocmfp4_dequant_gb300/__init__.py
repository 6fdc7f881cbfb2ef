"""Python binding of the GB300 ROCmFP4 library (``include/rocmfp4.h``).

Argument marshalling only: every step of dequantisation and of the products
runs in the CUDA kernels of ``_build/librocmfp4.so``.  There is no CPU
fallback: if the library is missing or no GPU is present, calls raise.

Entry points (names as in the C ABI, without the ``rocmfp4_`` prefix):
``gemv``, ``gemm``, ``dequant``, ``validate``, ``block_bytes``, ``row_bytes``.
Tensors are torch CUDA tensors; packed weights are ``uint8`` tensors holding
``N * row_bytes(K, variant)`` bytes; activations are ``float16`` or
``bfloat16``; outputs are ``float32``.  Calls are asynchronous on torch's
current CUDA stream unless a stream is given.
"""
from __future__ import annotations

import ctypes
import os

DUAL, FAST = 0, 1
ACT_F16, ACT_BF16 = 0, 1
OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2
STATUS = {0: "ROCMFP4_OK", 1: "ROCMFP4_ERR_INVALID_ARG", 2: "ROCMFP4_ERR_UNSUPPORTED",
          3: "ROCMFP4_ERR_INVALID_SCALE", 4: "ROCMFP4_ERR_CUDA"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librocmfp4.so")
EXPORTS = ("rocmfp4_block_bytes", "rocmfp4_row_bytes", "rocmfp4_gemv", "rocmfp4_gemv_ex", "rocmfp4_gemm",
           "rocmfp4_gemm_ex", "rocmfp4_gemm_noalloc", "rocmfp4_gemv_gate_up", "rocmfp4_decode_attention", "rocmfp4_quantize", "rocmfp4_gemv_chain", "rocmfp4_gemv_chain_mixed", "rocmfp4_dequant", "rocmfp4_copy", "rocmfp4_validate", "rocmfp4_device_error_bits",
           "rocmfp4_status_string", "rocmfp4_last_error", "rocmfp4_launch_count", "rocmfp4_shutdown")

_lib = None


class GemvOp(ctypes.Structure):
    """rocmfp4_gemv_op: one product of a chain."""
    _fields_ = [("W", ctypes.c_void_p), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class RocmFP4Error(RuntimeError):
    def __init__(self, status: int, where: str, message: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} {message}".strip())


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (build it first with ``build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"ROCmFP4 CUDA library not built: {path} is missing (run __graft_entry__.build())")
    L = ctypes.CDLL(path)
    vp, i64, c_int, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
    sig = {
        "rocmfp4_block_bytes": ([c_int], ctypes.c_size_t),
        "rocmfp4_row_bytes": ([i64, c_int], ctypes.c_size_t),
        "rocmfp4_gemv": ([vp, vp, vp, i64, i64, c_int], c_int),
        "rocmfp4_gemv_ex": ([vp, vp, vp, i64, i64, c_int, c_int, vp], c_int),
        "rocmfp4_gemm": ([vp, vp, vp, i64, i64, i64, c_int], c_int),
        "rocmfp4_gemm_ex": ([vp, vp, vp, i64, i64, i64, c_int, c_int, vp], c_int),
        "rocmfp4_gemm_noalloc": ([vp, vp, vp, i64, i64, i64, c_int, c_int, vp], c_int),
        "rocmfp4_gemv_gate_up": ([vp, vp, vp, i64, i64, i64, c_int, c_int, vp], c_int),
        "rocmfp4_decode_attention": ([vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_float, c_int, c_int, vp],
                                     c_int),
        "rocmfp4_quantize": ([vp, c_int, vp, i64, i64, c_int, vp], c_int),
        "rocmfp4_gemv_chain": ([ctypes.POINTER(GemvOp), c_int, i64, c_int, c_int, vp], c_int),
        "rocmfp4_gemv_chain_mixed": ([ctypes.POINTER(GemvOp), ctypes.POINTER(c_int), c_int, i64, c_int, vp], c_int),
        "rocmfp4_dequant": ([vp, vp, c_int, i64, i64, c_int, vp], c_int),
        "rocmfp4_copy": ([vp, vp, i64, vp], c_int),
        "rocmfp4_validate": ([vp, i64, i64, c_int, ctypes.POINTER(i64), vp], c_int),
        "rocmfp4_device_error_bits": ([vp], u32),
        "rocmfp4_status_string": ([c_int], ctypes.c_char_p),
        "rocmfp4_last_error": ([], ctypes.c_char_p),
        "rocmfp4_launch_count": ([], ctypes.c_uint64),
        "rocmfp4_shutdown": ([], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(status: int, where: str) -> None:
    if status != 0:
        msg = load().rocmfp4_last_error().decode(errors="replace")
        raise RocmFP4Error(status, where, msg)


_torch_mod = None
_raw_stream = None  # (current device, raw current stream of a device), when torch exposes them


def _torch():
    global _torch_mod
    if _torch_mod is None:
        import torch
        _torch_mod = torch
    return _torch_mod


def _current_stream() -> int:
    """Handle of torch's current CUDA stream on the current device.  The public
    torch.cuda.current_stream() builds a Stream object per call (about 3 us on
    the host); torch's raw accessors give the same handle without it."""
    global _raw_stream
    torch = _torch()
    if _raw_stream is None:
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream = (get_dev, get_raw) if get_dev and get_raw else False
    if _raw_stream:
        return _raw_stream[1](_raw_stream[0]())
    return torch.cuda.current_stream().cuda_stream


def _stream(stream):
    if stream is None:
        return _current_stream()
    torch = _torch()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _act_of(t) -> int:
    torch = _torch()
    dt = t.dtype
    if dt == torch.float16:
        return ACT_F16
    if dt == torch.bfloat16:
        return ACT_BF16
    raise TypeError(f"activations must be float16 or bfloat16, got {dt}")


def _ptr(t) -> int:
    return t.data_ptr() if t is not None and t.numel() > 0 else 0


def block_bytes(variant: int) -> int:
    return int(load().rocmfp4_block_bytes(variant))


def row_bytes(K: int, variant: int) -> int:
    return int(load().rocmfp4_row_bytes(K, variant))


def _row_bytes_fast(K: int, variant: int) -> int:
    # the layouts' arithmetic (18- or 17-byte blocks of 32 weights); anything
    # else goes to the library, which rejects it
    if (variant == DUAL or variant == FAST) and K >= 0 and K % 32 == 0:
        return (K // 32) * (18 if variant == DUAL else 17)
    return row_bytes(K, variant)


def _check_w(W, N: int, K: int, variant: int):
    torch = _torch()
    if W.dtype != torch.uint8 or not W.is_cuda or not W.is_contiguous():
        raise TypeError("W must be a contiguous uint8 CUDA tensor")
    if W.numel() < N * _row_bytes_fast(K, variant):
        raise ValueError("W holds fewer than N * row_bytes bytes")


def gemm(W, X, N: int, K: int, variant: int = DUAL, Y=None, stream=None):
    """Y[M, N] = X[M, K] . W^T in fp32 (X fp16 or bf16, on the GPU)."""
    torch = _torch()
    _check_w(W, N, K, variant)
    if X.dim() == 1:
        X = X.view(1, -1)
    if not X.is_cuda or not X.is_contiguous() or X.shape[1] != K:
        raise ValueError("X must be a contiguous [M, K] CUDA tensor")
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    elif Y.dtype != torch.float32 or not Y.is_contiguous() or Y.numel() < M * N:
        raise ValueError("Y must be a contiguous float32 tensor with M*N elements")
    _check(load().rocmfp4_gemm_ex(_ptr(W), _ptr(X), _ptr(Y), M, N, K, variant, _act_of(X), _stream(stream)),
           "rocmfp4_gemm_ex")
    return Y


def gemv(W, x, N: int, K: int, variant: int = DUAL, y=None, stream=None):
    """y[N] = W . x in fp32 (x fp16 or bf16, length K)."""
    torch = _torch()
    _check_w(W, N, K, variant)
    if not x.is_cuda or not x.is_contiguous() or x.numel() != K:
        raise ValueError("x must be a contiguous CUDA tensor of K elements")
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=x.device)
    _check(load().rocmfp4_gemv_ex(_ptr(W), _ptr(x), _ptr(y), N, K, variant, _act_of(x), _stream(stream)),
           "rocmfp4_gemv_ex")
    return y


def gemv_gate_up(W, X, I: int, K: int, variant: int = DUAL, Y=None, stream=None):
    """Y[M, I] = SiLU(X . Wg^T) * (X . Wu^T) in fp32, where W packs 2I rows:
    the I gate rows, then the I up rows (X fp16 or bf16 [M, K], M <= 8)."""
    torch = _torch()
    _check_w(W, 2 * I, K, variant)
    if X.dim() == 1:
        X = X.view(1, -1)
    if not X.is_cuda or not X.is_contiguous() or X.shape[1] != K:
        raise ValueError("X must be a contiguous [M, K] CUDA tensor")
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, I), dtype=torch.float32, device=X.device)
    elif Y.dtype != torch.float32 or not Y.is_contiguous() or Y.numel() < M * I:
        raise ValueError("Y must be a contiguous float32 tensor with M*I elements")
    _check(load().rocmfp4_gemv_gate_up(_ptr(W), _ptr(X), _ptr(Y), M, I, K, variant, _act_of(X), _stream(stream)),
           "rocmfp4_gemv_gate_up")
    return Y


def decode_attention(q, K, V, lens, Hkv: int, Tmax: int, scale: float, variant: int = DUAL, out=None,
                     stream=None):
    """out[B, H, D] (fp32) of single-token attention over a ROCmFP4 K/V cache:
    q [B, H, D] fp16 or bf16, K and V uint8 holding [B, Hkv, Tmax] rows of D/32
    blocks, lens int32 [B] (tokens per sequence), all on the GPU."""
    torch = _torch()
    if q.dim() != 3 or not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous [B, H, D] CUDA tensor")
    B, H, D = q.shape
    rb = row_bytes(D, variant)
    for t, name in ((K, "K"), (V, "V")):
        if not t.is_cuda or t.dtype != torch.uint8 or not t.is_contiguous() or t.numel() < B * Hkv * Tmax * rb:
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor of B*Hkv*Tmax rows")
    if not lens.is_cuda or lens.dtype != torch.int32 or lens.numel() < B:
        raise ValueError("lens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float32, device=q.device)
    elif out.dtype != torch.float32 or not out.is_contiguous() or out.numel() < B * H * D:
        raise ValueError("out must be a contiguous float32 tensor with B*H*D elements")
    _check(load().rocmfp4_decode_attention(_ptr(q), _ptr(K), _ptr(V), _ptr(lens), _ptr(out), B, H, Hkv, D, Tmax,
                                           float(scale), variant, _act_of(q), _stream(stream)),
           "rocmfp4_decode_attention")
    return out


def gemv_chain(ops, variant=DUAL, stream=None):
    """Runs products in order, as gemm() for each: ops is a list of (W, X, Y, N, K)
    with X [M, K] (all float16 or all bfloat16, one M) and Y [M, N] float32.
    variant is one block layout for every product, or a sequence with one per
    product (rocmfp4_gemv_chain_mixed)."""
    torch = _torch()
    if not ops:
        return
    mixed = not isinstance(variant, int)
    variants = [int(v) for v in variant] if mixed else [variant] * len(ops)
    if len(variants) != len(ops):
        raise ValueError("one variant per product")
    M = ops[0][1].shape[0] if ops[0][1].dim() == 2 else 1
    act = _act_of(ops[0][1])
    arr = (GemvOp * len(ops))()
    for i, (W, X, Y, N, K) in enumerate(ops):
        _check_w(W, N, K, variants[i])
        Xm = X.view(1, -1) if X.dim() == 1 else X
        if not Xm.is_cuda or not Xm.is_contiguous() or tuple(Xm.shape) != (M, K) or _act_of(Xm) != act:
            raise ValueError(f"product {i}: X must be a contiguous [M, K] CUDA tensor of the chain's dtype")
        if Y.dtype != torch.float32 or not Y.is_contiguous() or Y.numel() < M * N:
            raise ValueError(f"product {i}: Y must be a contiguous float32 tensor with M*N elements")
        arr[i] = GemvOp(W.data_ptr(), Xm.data_ptr(), Y.data_ptr(), N, K)
    if mixed:
        varr = (ctypes.c_int * len(ops))(*variants)
        _check(load().rocmfp4_gemv_chain_mixed(arr, varr, len(ops), M, act, _stream(stream)), "rocmfp4_gemv_chain_mixed")
    else:
        _check(load().rocmfp4_gemv_chain(arr, len(ops), M, variant, act, _stream(stream)), "rocmfp4_gemv_chain")


def copy(dst, src, stream=None):
    """Copies src into dst (the same number of bytes) on the stream by a kernel
    (rocmfp4_copy): each is a contiguous CUDA tensor or a pinned CPU tensor.  It
    runs after the stream's preceding kernel and lets the next one begin early."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src must hold the same number of bytes")
    if nbytes == 0:
        return
    _check(load().rocmfp4_copy(dst.data_ptr(), src.data_ptr(), nbytes, _stream(stream)), "rocmfp4_copy")


def quantize(src, variant: int = DUAL, W=None, stream=None):
    """ROCmFP4 blocks (uint8, N * row_bytes) of a [N, K] float16 / bfloat16 CUDA tensor."""
    torch = _torch()
    if src.dim() != 2 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous [N, K] CUDA tensor")
    N, K = src.shape
    if W is None:
        W = torch.empty(N * row_bytes(K, variant), dtype=torch.uint8, device=src.device)
    elif W.dtype != torch.uint8 or not W.is_contiguous() or W.numel() < N * row_bytes(K, variant):
        raise ValueError("W must be a contiguous uint8 tensor of N * row_bytes bytes")
    _check(load().rocmfp4_quantize(_ptr(src), _act_of(src), _ptr(W), N, K, variant, _stream(stream)),
           "rocmfp4_quantize")
    return W


def dequant(W, N: int, K: int, variant: int = DUAL, out_dtype=None, out=None, stream=None):
    """Dense [N, K] weights (float32 by default, or bfloat16 / float16), exact."""
    torch = _torch()
    _check_w(W, N, K, variant)
    dt = out_dtype or (out.dtype if out is not None else torch.float32)
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16, torch.float16: OUT_F16}[dt]
    if out is None:
        out = torch.empty((N, K), dtype=dt, device=W.device)
    _check(load().rocmfp4_dequant(_ptr(W), _ptr(out), code, N, K, variant, _stream(stream)), "rocmfp4_dequant")
    return out


def validate(W, N: int, K: int, variant: int = DUAL, stream=None) -> int:
    """-1 if every scale byte is finite, else the index of the first bad block."""
    _check_w(W, N, K, variant)
    first = ctypes.c_int64(-1)
    st = load().rocmfp4_validate(_ptr(W), N, K, variant, ctypes.byref(first), _stream(stream))
    if st not in (0, 3):
        _check(st, "rocmfp4_validate")
    return int(first.value)


def device_error_bits(stream=None) -> int:
    return int(load().rocmfp4_device_error_bits(_stream(stream)))


def launch_count() -> int:
    return int(load().rocmfp4_launch_count())
