"""linear_noalloc: the layer for callers that cannot allocate device memory.

Such callers (a serving runtime's per-request path where cudaMalloc may
synchronize the device and fail under memory pressure; a plugin whose host
framework owns all device memory and offers no allocator) call
linear_noalloc, whose workspace is a fixed 8 MiB array in the library.  This
test calls it through the C ABI twice in a row per case -- the second call
reuses the array as the first left it -- and after a call that nearly fills
the array, and compares each result with linear() given an ordinary
workspace, within the tolerance the parity tests use.  It also checks that a problem too large for the array is refused
without touching the output.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20
WORKSPACE_ERROR = 6


def _tol_ok(y, ref):
    y = y.astype(np.float64)
    r = ref.astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    tol = 2e-3 * (np.abs(r).max() if r.size else 0.0) + ulp
    return bool(np.all(np.abs(y - r) <= tol))


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from w4a8_int8_quantized_gb300 import build
    build.build()
    import w4a8_int8_quantized_gb300 as w8
    from w4a8_int8_quantized_gb300 import synth
    lib = w8.load()
    assert w8.w8a8_is_available()
    return w8, synth, lib


# (M, N, K, group_size, wbits): prefill shapes (M > 1, whose quantized
# activations live in the array) that fit in 8 MiB, and one decode call
# (M == 1 quantizes inside the matrix-vector kernel and leaves the array
# alone)
CASES = [(300, 1000, 2560, 0, 8), (257, 520, 4096, 128, 8), (130, 700, 4096, 0, 4),
         (1600, 384, 2560, 0, 8), (64, 256, 14336, 64, 8), (1, 4096, 2560, 0, 8)]


def _problem(w8, synth, M, N, K, gs, wbits):
    x = torch.from_numpy(synth.activations(M, K, seed=M + K, n_outliers=4,
                                           outlier_scale=40.0)).cuda()
    W = torch.from_numpy(synth.weights(N, K, seed=N)).cuda()
    if wbits == 8:
        wq, sw = w8.quantize_weight_int8(W, gs)
    else:
        wq, sw = w8.pack_weight_int4(W)
    ref = w8.linear(x, wq, sw, gs, wbits)
    torch.cuda.synchronize()
    return x, wq, sw, ref.cpu().numpy()


def _call_noalloc(lib, x, wq, sw, M, N, K, gs, wbits):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = ctypes.c_void_p
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    st = lib.linear_noalloc(P(x.data_ptr()), P(wq.data_ptr()), P(sw.data_ptr()), M, N, K, gs,
                            wbits, P(y.data_ptr()), stream)
    assert st == 0, lib.w8a8_status_string(st)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("M,N,K,gs,wbits", CASES)
def test_noalloc_matches_linear_twice(ctx, M, N, K, gs, wbits):
    w8, synth, lib = ctx
    assert w8.w8a8_linear_workspace_bytes(M, K, gs) <= SCRATCH_BYTES
    x, wq, sw, ref_h = _problem(w8, synth, M, N, K, gs, wbits)
    for _ in range(2):
        assert _tol_ok(_call_noalloc(lib, x, wq, sw, M, N, K, gs, wbits), ref_h)
    assert lib.w8a8_check_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0


def test_noalloc_after_a_larger_call(ctx):
    """The array keeps what the last call left: a call that nearly fills it
    (1600 x 2560 fp16 codes) followed by smaller calls with another K and
    group size (their codes and scales land at other offsets than the stale
    ones) must each still match linear()."""
    w8, synth, lib = ctx
    seq = [(1600, 384, 2560, 0, 8), (37, 300, 4096, 64, 8), (5, 129, 512, 128, 8),
           (130, 257, 4096, 0, 4), (1600, 384, 2560, 0, 8)]
    assert w8.w8a8_linear_workspace_bytes(1600, 2560, 0) > SCRATCH_BYTES * 0.9
    probs = [_problem(w8, synth, *c) for c in seq]
    for c, (x, wq, sw, ref_h) in zip(seq, probs):
        assert _tol_ok(_call_noalloc(lib, x, wq, sw, *c), ref_h), c


def test_noalloc_refuses_oversized_problem(ctx):
    w8, synth, lib = ctx
    M, N, K = 4096, 64, 2560  # fp16 codes alone need 20 MiB
    assert w8.w8a8_linear_workspace_bytes(M, K, 0) > SCRATCH_BYTES
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    wq = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    sw = torch.zeros((N, 1), dtype=torch.float32, device="cuda")
    y = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    P = ctypes.c_void_p
    st = lib.linear_noalloc(P(x.data_ptr()), P(wq.data_ptr()), P(sw.data_ptr()), M, N, K, 0, 8,
                            P(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == WORKSPACE_ERROR
    torch.cuda.synchronize()
    assert bool(torch.all(y == 7.0))
