"""CPU oracle for the W8A8 / W4A8 quantized linear layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does; the two share no code.

The arithmetic lives in ``w8a8_oracle.c`` (plain loops, one IEEE fp32
operation per step, built with ``-O2 -ffp-contract=off``).  This module only
compiles that file with gcc and marshals numpy arrays to it.  The method it
restates is described on two web pages about the Cider SDK:

* "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다", section
  "INT8 TensorOps 커널 설계" (the four-step pipeline: absmax scales, fp16 ->
  INT8, INT8 GEMM with INT32 accumulation, rescale to fp16) and section
  "입도(Granularity)" (per-group scales);
* "cider 소개", section "cider의 양자화 모드와 적용 가능한 영역" (W8A8 and
  W4A8 modes, per-channel / gs=128 / gs=64) and "cider 설치와 사용법"
  (quantize_weight_int8, pack_weight_int4).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w8a8_oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liboracle_w8a8.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fopenmp", "-std=c11", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/lib/liboracle_w8a8.so."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, L, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_int
        lib.oracle_quant_rows.argtypes = [P, L, L, L, I, P, P]
        lib.oracle_pack_int4.argtypes = [P, L, L, P]
        lib.oracle_unpack_int4.argtypes = [P, L, L, P]
        lib.oracle_int_gemm.argtypes = [P, P, L, L, L, L, P]
        lib.oracle_dequant.argtypes = [P, P, P, L, L, L, P]
        lib.oracle_sampled_outputs.argtypes = [P, P, P, P, L, L, L, L, P, P, L, P, P]
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_weight_only.argtypes = [P, P, P, L, L, L, L, P]
        for f in (lib.oracle_quant_rows, lib.oracle_pack_int4, lib.oracle_unpack_int4,
                  lib.oracle_int_gemm, lib.oracle_dequant, lib.oracle_sampled_outputs,
                  lib.oracle_num_threads, lib.oracle_weight_only):
            f.restype = ctypes.c_int
        lib.oracle_set_threads.restype = None
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        names = {1: "bad argument", 2: "non-finite input", 3: "int32 overflow"}
        raise OracleError(f"{what}: {names.get(rc, rc)}")


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def quant_rows(x: np.ndarray, group_size: int = 0, qmax: int = 127):
    """Symmetric per-row (per-group) quantization of fp16 rows.

    Returns (q int8 [R, K], s float32 [R, G]).  Used for per-token
    activations (qmax 127), per-channel / per-group INT8 weights (qmax 127)
    and per-channel INT4 weights (qmax 7)."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    R, K = x.shape
    G = 1 if group_size == 0 else K // group_size
    q = np.empty((R, K), dtype=np.int8)
    s = np.empty((R, G), dtype=np.float32)
    _check(_load().oracle_quant_rows(_ptr(x.view(np.uint16)), R, K, group_size,
                                     qmax, _ptr(q), _ptr(s)), "quant_rows")
    return q, s


def pack_int4(q4: np.ndarray) -> np.ndarray:
    q4 = np.ascontiguousarray(q4, dtype=np.int8)
    N, K = q4.shape
    out = np.empty((N, K // 2), dtype=np.uint8)
    _check(_load().oracle_pack_int4(_ptr(q4), N, K, _ptr(out)), "pack_int4")
    return out


def unpack_int4(packed: np.ndarray, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    out = np.empty((N, K), dtype=np.int8)
    _check(_load().oracle_unpack_int4(_ptr(packed), N, K, _ptr(out)), "unpack_int4")
    return out


def int_gemm(a: np.ndarray, w: np.ndarray, group_size: int = 0) -> np.ndarray:
    """Exact INT32 partials acc [M, N, G] of a [M, K] x w [N, K]^T."""
    a = np.ascontiguousarray(a, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    M, K = a.shape
    N = w.shape[0]
    assert w.shape[1] == K
    G = 1 if group_size == 0 else K // group_size
    acc = np.empty((M, N, G), dtype=np.int32)
    _check(_load().oracle_int_gemm(_ptr(a), _ptr(w), M, N, K, group_size, _ptr(acc)),
           "int_gemm")
    return acc


def dequant(acc: np.ndarray, sa: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """fp16 y [M, N] from acc [M, N, G], sa [M, G], sw [N, G]."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    M, N, G = acc.shape
    sa = np.ascontiguousarray(sa, dtype=np.float32).reshape(M, G)
    sw = np.ascontiguousarray(sw, dtype=np.float32).reshape(N, G)
    y = np.empty((M, N), dtype=np.float16)
    _check(_load().oracle_dequant(_ptr(acc), _ptr(sa), _ptr(sw), M, N, G,
                                  _ptr(y.view(np.uint16))), "dequant")
    return y


def sampled_outputs(a, sa, w, sw, rows, cols, group_size: int = 0):
    """(acc [count, G], y fp16 [count]) at output positions (rows[i], cols[i])."""
    a = np.ascontiguousarray(a, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    M, K = a.shape
    N = w.shape[0]
    G = 1 if group_size == 0 else K // group_size
    sa = np.ascontiguousarray(sa, dtype=np.float32).reshape(M, G)
    sw = np.ascontiguousarray(sw, dtype=np.float32).reshape(N, G)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    cnt = rows.shape[0]
    acc = np.empty((cnt, G), dtype=np.int32)
    y = np.empty((cnt,), dtype=np.float16)
    _check(_load().oracle_sampled_outputs(_ptr(a), _ptr(sa), _ptr(w), _ptr(sw), M, N, K,
                                          group_size, _ptr(rows), _ptr(cols), cnt,
                                          _ptr(acc), _ptr(y.view(np.uint16))),
           "sampled_outputs")
    return acc, y


def weight_only(x: np.ndarray, q: np.ndarray, sw: np.ndarray, group_size: int = 0) -> np.ndarray:
    """Weight-only product y = x . (q * s_w)^T rounded once to fp16: fp16 x
    [M, K], integer weight codes q int8 [N, K] (INT8, or INT4 unpacked),
    s_w [N, G]."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    M, K = x.shape
    N = q.shape[0]
    assert q.shape[1] == K
    G = 1 if group_size == 0 else K // group_size
    sw = np.ascontiguousarray(sw, dtype=np.float32).reshape(N, G)
    y = np.empty((M, N), dtype=np.float16)
    _check(_load().oracle_weight_only(_ptr(x.view(np.uint16)), _ptr(q), _ptr(sw), M, N, K,
                                      group_size, _ptr(y.view(np.uint16))), "weight_only")
    return y


# ---- composites: the whole layer, step by step -----------------------------

def quantize_weight_int8(W: np.ndarray, group_size: int = 0):
    """Offline INT8 weight quantization: per output channel (group_size 0) or
    per group along K."""
    return quant_rows(W, group_size, 127)


def pack_weight_int4(W: np.ndarray):
    """Offline INT4 weight quantization (per output channel, [-7, 7]) and
    packing, two nibbles per byte, low nibble = even k."""
    q4, s4 = quant_rows(W, 0, 7)
    return pack_int4(q4), s4


def quantize_act_per_token(x: np.ndarray, group_size: int = 0):
    return quant_rows(x, group_size, 127)


def linear(x: np.ndarray, wq: np.ndarray, sw: np.ndarray, group_size: int = 0,
           wbits: int = 8) -> np.ndarray:
    """y = dequant(int_gemm(quant(x), w)): the layer's forward pass.

    wq is int8 [N, K] for wbits 8 or packed uint8 [N, K/2] for wbits 4."""
    xq, sa = quantize_act_per_token(x, group_size)
    K = x.shape[1]
    w = unpack_int4(wq, K) if wbits == 4 else wq
    return dequant(int_gemm(xq, w, group_size), sa, sw)


def linear_weight_only(x: np.ndarray, wq: np.ndarray, sw: np.ndarray, group_size: int = 0,
                       wbits: int = 8) -> np.ndarray:
    """The W8A16 / W4A16 layer: fp16 x times the dequantized weights; wq is
    int8 [N, K] (wbits 8, per channel or per group) or packed uint8 [N, K/2]
    (wbits 4, per channel)."""
    K = x.shape[1]
    w = unpack_int4(wq, K) if wbits == 4 else wq
    return weight_only(x, w, sw, group_size)
