"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every function include/w8a8.h declares; argument errors are
reported before any device work; the workspace size rule."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from w4a8_int8_quantized_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[a-z_][a-z0-9_ \t]*?\**\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.w8a8_status_string(0) == b"ok"
    for code in range(1, 7):
        assert lib.w8a8_status_string(code) not in (b"ok", b"unknown status")
    assert lib.w8a8_status_string(99) == b"unknown status"


def test_workspace_bytes(lib):
    f = lib.w8a8_linear_workspace_bytes
    # int8 activations then fp32 scales, each region rounded up to 256 bytes
    # codes: fp16 values for M > 1 (the GEMM operand), int8 for M == 1
    assert f(4096, 2560, 0) == 2 * 4096 * 2560 + 4096 * 4
    assert f(1, 2560, 0) == 2560 + 256
    assert f(3, 512, 128) == 2 * 1536 + 256
    assert f(4516, 4096, 64) == 2 * 4516 * 4096 + ((4516 * 64 * 4 + 255) // 256) * 256
    assert f(-1, 16, 0) == 0
    assert f(4, 100, 64) == 0


A16 = ctypes.c_void_p(1 << 20)     # 16-byte aligned fake addresses: never dereferenced,
B16 = ctypes.c_void_p(2 << 20)     # the calls below fail their host checks first
C16 = ctypes.c_void_p(3 << 20)
D16 = ctypes.c_void_p(4 << 20)
ODD = ctypes.c_void_p((5 << 20) + 8)
NUL = ctypes.c_void_p(0)
S0 = ctypes.c_void_p(0)


def test_argument_errors_before_any_launch(lib):
    INV, MIS, WS = 1, 2, 6
    q = lib.quantize_act_per_token
    assert q(A16, -1, 64, 0, B16, C16, S0) == INV        # negative M
    assert q(A16, 4, 0, 0, B16, C16, S0) == INV          # K <= 0
    assert q(A16, 4, 64, 32, B16, C16, S0) == INV        # group size not 0/64/128
    assert q(A16, 4, 192, 128, B16, C16, S0) == INV      # K % group size
    assert q(A16, 4, 40, 0, B16, C16, S0) == MIS         # K % 16
    assert q(A16, 4, 65536, 0, B16, C16, S0) == INV      # K above the maximum
    assert q(NUL, 4, 64, 0, B16, C16, S0) == INV         # null input
    assert q(ODD, 4, 64, 0, B16, C16, S0) == MIS         # misaligned input
    assert q(A16, 0, 64, 0, NUL, NUL, S0) == 0           # empty problem: no-op
    g = lib.w8a8_gemm
    assert g(A16, C16, B16, C16, 8, 8, 64, 0, NUL, S0) == INV
    assert g(A16, C16, ODD, C16, 8, 8, 64, 0, D16, S0) == MIS
    assert g(A16, C16, B16, C16, 0, 8, 64, 0, NUL, S0) == 0
    assert g(A16, C16, B16, C16, 8, 0, 64, 0, NUL, S0) == 0
    assert lib.w8a8_mv(A16, C16, B16, C16, 2, 8, 64, 0, D16, S0) == INV   # M must be 1
    assert lib.w4a8_gemm(A16, C16, B16, C16, 2, 8, 48, D16, S0) == MIS    # K % 32
    lin = lib.linear
    assert lin(A16, B16, C16, 4, 8, 64, 0, 3, D16, 1 << 20, D16, S0) == INV   # wbits
    assert lin(A16, B16, C16, 4, 8, 64, 64, 4, D16, 1 << 20, D16, S0) == INV  # W4 per group
    assert lin(A16, B16, C16, 4, 8, 64, 0, 8, D16, 16, D16, S0) == WS         # too small
    assert lin(A16, B16, C16, 4, 8, 64, 0, 8, ODD, 1 << 20, D16, S0) == WS    # misaligned
    assert lin(A16, B16, C16, 4, 8, 64, 0, 8, NUL, 1 << 20, D16, S0) == WS    # missing
    gh = lib.w8a8_gemm_h
    assert gh(A16, C16, B16, C16, 4, 8, 64, 0, 5, D16, S0) == INV      # wbits
    assert gh(A16, C16, B16, C16, 4, 8, 64, 64, 4, D16, S0) == INV     # W4 per group
    assert gh(ODD, C16, B16, C16, 4, 8, 64, 0, 8, D16, S0) == MIS
    assert lib.quantize_act_per_token_h(A16, 4, 40, 0, B16, C16, S0) == MIS
    wo = lib.weight_only_gemm
    assert wo(A16, B16, C16, 4, 8, 64, 0, 5, D16, S0) == INV      # wbits
    assert wo(A16, B16, C16, 4, 8, 64, 64, 4, D16, S0) == INV     # W4 per group
    assert wo(A16, B16, C16, 4, 8, 48, 0, 4, D16, S0) == MIS      # K % 32 for INT4
    assert wo(ODD, B16, C16, 4, 8, 64, 0, 8, D16, S0) == MIS
    assert wo(A16, B16, C16, 0, 8, 64, 0, 8, D16, S0) == 0        # empty problem
    i32 = lib.w8a8_gemm_i32
    assert i32(A16, B16, 4, 8, 64, 0, 5, C16, S0) == INV
    assert i32(A16, B16, 4, 8, 64, 64, 4, C16, S0) == INV


def test_binding_raises_without_touching_device():
    import torch
    with pytest.raises(TypeError):
        binding.quantize_act_per_token(torch.zeros(4, 64, dtype=torch.float32))
    with pytest.raises(ValueError):
        binding.quantize_act_per_token(torch.zeros(4, 64, dtype=torch.float16))  # CPU tensor


NO_DEVICE_SCRIPT = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from w4a8_int8_quantized_gb300 import binding
lib = binding.load()
P = ctypes.c_void_p
assert lib.w8a8_is_available() == 0
# aligned fake addresses: the device check refuses before any launch
assert lib.quantize_act_per_token(P(1 << 20), 4, 64, 0, P(2 << 20), P(3 << 20), P(0)) == 3
assert lib.w8a8_gemm(P(1 << 20), P(3 << 20), P(2 << 20), P(3 << 20), 4, 8, 64, 0, P(4 << 20),
                     P(0)) == 3
assert lib.linear_noalloc(P(1 << 20), P(2 << 20), P(3 << 20), 4, 8, 64, 0, 8, P(4 << 20),
                          P(0)) == 3
assert lib.w8a8_test_set_fault(-1, 0) == 1 and lib.w8a8_test_set_fault(0, 2) == 1
assert lib.w8a8_test_set_fault(0, 0) == 0
print("no-device ok")
"""


def test_no_visible_device_is_unsupported(lib):
    """With no CUDA device visible (CUDA_VISIBLE_DEVICES empty), the library
    still loads, w8a8_is_available() is 0 and every compute call returns
    W8A8_ERR_UNSUPPORTED_DEVICE after its host checks, launching nothing (the
    analogue of the SDK's is_available() gate, "cider 설치와 사용법")."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", NO_DEVICE_SCRIPT, ROOT], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "no-device ok" in r.stdout
