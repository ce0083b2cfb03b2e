"""Thin Python binding of libw8a8 (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors that already live on the current CUDA device, checks their dtype and
contiguity, passes raw pointers, sizes and the current stream to the library,
and raises ``W8A8Error`` on a nonzero status.  All arithmetic runs in the
library's kernels; there is no fallback of any kind: if the library is not
built, or the device is not a compute-capability 10.3 GPU, the call fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libw8a8.so")

_lock = threading.Lock()
_lib = None

STATUS = {0: "ok", 1: "invalid argument", 2: "misaligned pointer or K",
          3: "unsupported device", 4: "CUDA error", 5: "device-side wait timed out",
          6: "workspace too small or misaligned"}

# every symbol that include/w8a8.h declares
EXPORTS = ("w8a8_is_available", "w8a8_status_string", "w8a8_check_status",
           "quantize_weight_int8", "pack_weight_int4", "quantize_act_per_token",
           "w8a8_gemm", "w8a8_mv", "w4a8_gemm", "quantize_act_per_token_h", "w8a8_gemm_h",
           "w8a8_linear_workspace_bytes", "linear", "linear_noalloc", "w8a8_gemm_i32",
           "w8a8_test_set_fault", "weight_only_gemm")


class W8A8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({STATUS.get(status, 'unknown')})")
        self.status = status


def load(path: str | None = None):
    """Load libw8a8.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libw8a8 is not built ({p} missing): run "
                               "w4a8_int8_quantized_gb300.build.build() first")
        lib = ctypes.CDLL(p)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "w8a8_is_available": ([], I),
            "w8a8_status_string": ([I], ctypes.c_char_p),
            "w8a8_check_status": ([P], I),
            "quantize_weight_int8": ([P, I, I, I, P, P, P], I),
            "pack_weight_int4": ([P, I, I, P, P, P], I),
            "quantize_act_per_token": ([P, I, I, I, P, P, P], I),
            "w8a8_gemm": ([P, P, P, P, I, I, I, I, P, P], I),
            "w8a8_mv": ([P, P, P, P, I, I, I, I, P, P], I),
            "w4a8_gemm": ([P, P, P, P, I, I, I, P, P], I),
            "quantize_act_per_token_h": ([P, I, I, I, P, P, P], I),
            "w8a8_gemm_h": ([P, P, P, P, I, I, I, I, I, P, P], I),
            "w8a8_linear_workspace_bytes": ([I, I, I], Z),
            "linear": ([P, P, P, I, I, I, I, I, P, Z, P, P], I),
            "linear_noalloc": ([P, P, P, I, I, I, I, I, P, P], I),
            "w8a8_gemm_i32": ([P, P, I, I, I, I, I, P, P], I),
            "w8a8_test_set_fault": ([ctypes.c_longlong, I], I),
            "weight_only_gemm": ([P, P, P, I, I, I, I, I, P, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check(status: int, what: str):
    if status != 0:
        raise W8A8Error(status, what)


def _groups(K: int, group_size: int) -> int:
    return 1 if group_size == 0 else K // group_size


def w8a8_is_available() -> bool:
    return bool(load().w8a8_is_available())


def w8a8_status_string(status: int) -> str:
    return load().w8a8_status_string(int(status)).decode()


def w8a8_check_status() -> int:
    return load().w8a8_check_status(_stream())


def quantize_weight_int8(W: torch.Tensor, group_size: int = 0, Wq=None, scale_w=None):
    """fp16 W [N, K] -> (int8 Wq [N, K], fp32 scale_w [N, G])."""
    _need(W, torch.float16, "W")
    N, K = W.shape
    G = _groups(K, group_size)
    Wq = torch.empty((N, K), dtype=torch.int8, device=W.device) if Wq is None else Wq
    scale_w = (torch.empty((N, G), dtype=torch.float32, device=W.device)
               if scale_w is None else scale_w)
    _need(Wq, torch.int8, "Wq", (N, K))
    _need(scale_w, torch.float32, "scale_w", (N, G))
    _check(load().quantize_weight_int8(_ptr(W), N, K, group_size, _ptr(Wq), _ptr(scale_w),
                                       _stream()), "quantize_weight_int8")
    return Wq, scale_w


def pack_weight_int4(W: torch.Tensor, Wp=None, scale_w=None):
    """fp16 W [N, K] -> (uint8 Wp [N, K/2], fp32 scale_w [N, 1])."""
    _need(W, torch.float16, "W")
    N, K = W.shape
    Wp = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device) if Wp is None else Wp
    scale_w = (torch.empty((N, 1), dtype=torch.float32, device=W.device)
               if scale_w is None else scale_w)
    _need(Wp, torch.uint8, "Wp", (N, K // 2))
    _need(scale_w, torch.float32, "scale_w", (N, 1))
    _check(load().pack_weight_int4(_ptr(W), N, K, _ptr(Wp), _ptr(scale_w), _stream()),
           "pack_weight_int4")
    return Wp, scale_w


def quantize_act_per_token(x: torch.Tensor, group_size: int = 0, xq=None, scale_a=None):
    """fp16 x [M, K] -> (int8 xq [M, K], fp32 scale_a [M, G])."""
    _need(x, torch.float16, "x")
    M, K = x.shape
    G = _groups(K, group_size)
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    scale_a = (torch.empty((M, G), dtype=torch.float32, device=x.device)
               if scale_a is None else scale_a)
    _need(xq, torch.int8, "xq", (M, K))
    _need(scale_a, torch.float32, "scale_a", (M, G))
    _check(load().quantize_act_per_token(_ptr(x), M, K, group_size, _ptr(xq), _ptr(scale_a),
                                         _stream()), "quantize_act_per_token")
    return xq, scale_a


def _gemm_args(xq, scale_a, Wq, scale_w, group_size, wdtype, kdiv):
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    G = _groups(K, group_size)
    _need(Wq, wdtype, "Wq")
    N = Wq.shape[0]
    if Wq.shape[1] * kdiv != K:
        raise ValueError("Wq inner dimension does not match K")
    _need(scale_a, torch.float32, "scale_a", (M, G))
    _need(scale_w, torch.float32, "scale_w", (N, G))
    return M, N, K


def w8a8_gemm(xq, scale_a, Wq, scale_w, group_size: int = 0, y=None):
    """int8 xq [M, K] x int8 Wq [N, K]^T with fused dequant -> fp16 y [M, N]."""
    M, N, K = _gemm_args(xq, scale_a, Wq, scale_w, group_size, torch.int8, 1)
    y = torch.empty((M, N), dtype=torch.float16, device=xq.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().w8a8_gemm(_ptr(xq), _ptr(scale_a), _ptr(Wq), _ptr(scale_w), M, N, K,
                            group_size, _ptr(y), _stream()), "w8a8_gemm")
    return y


def w8a8_mv(xq, scale_a, Wq, scale_w, group_size: int = 0, y=None):
    """Decode matrix-vector product; xq must have one row."""
    M, N, K = _gemm_args(xq, scale_a, Wq, scale_w, group_size, torch.int8, 1)
    y = torch.empty((M, N), dtype=torch.float16, device=xq.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().w8a8_mv(_ptr(xq), _ptr(scale_a), _ptr(Wq), _ptr(scale_w), M, N, K,
                          group_size, _ptr(y), _stream()), "w8a8_mv")
    return y


def w4a8_gemm(xq, scale_a, Wp, scale_w, y=None):
    """int8 xq [M, K] x packed int4 Wp [N, K/2]^T with fused dequant."""
    M, N, K = _gemm_args(xq, scale_a, Wp, scale_w, 0, torch.uint8, 2)
    y = torch.empty((M, N), dtype=torch.float16, device=xq.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().w4a8_gemm(_ptr(xq), _ptr(scale_a), _ptr(Wp), _ptr(scale_w), M, N, K,
                            _ptr(y), _stream()), "w4a8_gemm")
    return y


def quantize_act_per_token_h(x: torch.Tensor, group_size: int = 0, xq_h=None, scale_a=None):
    """fp16 x [M, K] -> (INT8 codes as fp16 xq_h [M, K], fp32 scale_a [M, G])."""
    _need(x, torch.float16, "x")
    M, K = x.shape
    G = _groups(K, group_size)
    xq_h = torch.empty((M, K), dtype=torch.float16, device=x.device) if xq_h is None else xq_h
    scale_a = (torch.empty((M, G), dtype=torch.float32, device=x.device)
               if scale_a is None else scale_a)
    _need(xq_h, torch.float16, "xq_h", (M, K))
    _need(scale_a, torch.float32, "scale_a", (M, G))
    _check(load().quantize_act_per_token_h(_ptr(x), M, K, group_size, _ptr(xq_h),
                                           _ptr(scale_a), _stream()), "quantize_act_per_token_h")
    return xq_h, scale_a


def w8a8_gemm_h(xq_h, scale_a, Wq, scale_w, group_size: int = 0, wbits: int = 8, y=None):
    """GEMM with the activation codes given as fp16 values (wbits 8: int8 Wq
    [N, K]; wbits 4: packed Wq [N, K/2])."""
    _need(xq_h, torch.float16, "xq_h")
    M, K = xq_h.shape
    G = _groups(K, group_size)
    wdtype = torch.int8 if wbits == 8 else torch.uint8
    _need(Wq, wdtype, "Wq")
    N = Wq.shape[0]
    if Wq.shape[1] * (1 if wbits == 8 else 2) != K:
        raise ValueError("Wq inner dimension does not match K")
    _need(scale_a, torch.float32, "scale_a", (M, G))
    _need(scale_w, torch.float32, "scale_w", (N, G))
    y = torch.empty((M, N), dtype=torch.float16, device=xq_h.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().w8a8_gemm_h(_ptr(xq_h), _ptr(scale_a), _ptr(Wq), _ptr(scale_w), M, N, K,
                              group_size, wbits, _ptr(y), _stream()), "w8a8_gemm_h")
    return y


def w8a8_linear_workspace_bytes(M: int, K: int, group_size: int = 0) -> int:
    return int(load().w8a8_linear_workspace_bytes(M, K, group_size))


def linear(x, Wq, scale_w, group_size: int = 0, wbits: int = 8, workspace=None, y=None):
    """The whole layer: per-token quantization of x, then GEMM (M > 1) or
    matrix-vector (M == 1) with the fused dequant.  Wq is int8 [N, K]
    (wbits 8) or packed uint8 [N, K/2] (wbits 4)."""
    _need(x, torch.float16, "x")
    M, K = x.shape
    wdtype = torch.int8 if wbits == 8 else torch.uint8
    _need(Wq, wdtype, "Wq")
    N = Wq.shape[0]
    _need(scale_w, torch.float32, "scale_w", (N, _groups(K, group_size)))
    need = w8a8_linear_workspace_bytes(M, K, group_size)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _need(workspace, torch.uint8, "workspace")
    y = torch.empty((M, N), dtype=torch.float16, device=x.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().linear(_ptr(x), _ptr(Wq), _ptr(scale_w), M, N, K, group_size, wbits,
                         _ptr(workspace), workspace.numel(), _ptr(y), _stream()), "linear")
    return y


def linear_noalloc(x, Wq, scale_w, group_size: int = 0, wbits: int = 8, y=None):
    """linear() without a workspace: the library's fixed 8 MiB device array
    serves as the workspace, so the C call allocates nothing (the output is
    allocated here if not given).  Problems that do not fit raise W8A8Error
    (status 6).  Calls on streams that overlap on the GPU race on the array."""
    _need(x, torch.float16, "x")
    M, K = x.shape
    wdtype = torch.int8 if wbits == 8 else torch.uint8
    _need(Wq, wdtype, "Wq")
    N = Wq.shape[0]
    _need(scale_w, torch.float32, "scale_w", (N, _groups(K, group_size)))
    y = torch.empty((M, N), dtype=torch.float16, device=x.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().linear_noalloc(_ptr(x), _ptr(Wq), _ptr(scale_w), M, N, K, group_size, wbits,
                                 _ptr(y), _stream()), "linear_noalloc")
    return y


def weight_only_gemm(x, Wq, scale_w, group_size: int = 0, wbits: int = 8, y=None):
    """Weight-only product (W8A16 / W4A16): fp16 x [M, K] times the dequantized
    weights (int8 Wq [N, K], or packed uint8 [N, K/2] with wbits 4)."""
    _need(x, torch.float16, "x")
    M, K = x.shape
    wdtype = torch.int8 if wbits == 8 else torch.uint8
    _need(Wq, wdtype, "Wq")
    N = Wq.shape[0]
    if Wq.shape[1] * (1 if wbits == 8 else 2) != K:
        raise ValueError("Wq inner dimension does not match K")
    _need(scale_w, torch.float32, "scale_w", (N, _groups(K, group_size)))
    y = torch.empty((M, N), dtype=torch.float16, device=x.device) if y is None else y
    _need(y, torch.float16, "y", (M, N))
    _check(load().weight_only_gemm(_ptr(x), _ptr(Wq), _ptr(scale_w), M, N, K, group_size, wbits,
                                   _ptr(y), _stream()), "weight_only_gemm")
    return y


def w8a8_gemm_i32(xq, Wq, group_size: int = 0, wbits: int = 8, acc=None):
    """Exact INT32 (per-group) sums acc [M, N, G] of the tensor-core contraction."""
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    wdtype = torch.int8 if wbits == 8 else torch.uint8
    _need(Wq, wdtype, "Wq")
    N = Wq.shape[0]
    G = _groups(K, group_size)
    acc = torch.empty((M, N, G), dtype=torch.int32, device=xq.device) if acc is None else acc
    _need(acc, torch.int32, "acc", (M, N, G))
    _check(load().w8a8_gemm_i32(_ptr(xq), _ptr(Wq), M, N, K, group_size, wbits, _ptr(acc),
                                _stream()), "w8a8_gemm_i32")
    return acc


def w8a8_test_set_fault(wait_limit_cycles: int = 0, skip_first_copy: bool = False) -> None:
    """Test hook: the GEMM's bounded-wait limit (cycles, 0 = default) and
    whether its first weight-staging copy per CTA is left unissued, for the
    launches that follow."""
    _check(load().w8a8_test_set_fault(int(wait_limit_cycles), int(bool(skip_first_copy))),
           "w8a8_test_set_fault")
