"""Parity of the CUDA path (called through the C ABI via the binding) against
the CPU oracle, on the same seeded inputs.

The bar: INT8 codes, INT4 packed bytes, fp32 scales and INT32 sums
bit-exact; fp16 outputs within |dy| <= 2e-3 * max|y_ref| + ulp_fp16(y_ref)
element by element.  Where the kernel evaluates the dequant in the oracle's
operation order (per channel everywhere, per group on the GEMM) the fp16
output is also checked bit-exact.

Method: "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다", section "INT8
TensorOps 커널 설계" (steps 1-4) and section "입도(Granularity)"; "cider 소개",
sections "cider의 양자화 모드와 적용 가능한 영역" and "cider 설치와 사용법".
"""
import numpy as np
import pytest

import oracle
from w4a8_int8_quantized_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import w4a8_int8_quantized_gb300 as w8


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def fp16_tol(ref):
    r = ref.astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    return 2e-3 * (np.abs(r).max() if r.size else 0.0) + ulp


def assert_fp16_close(y, ref):
    assert y.shape == ref.shape
    err = np.abs(y.astype(np.float64) - ref.astype(np.float64))
    tol = fp16_tol(ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{len(bad)} outputs out of tolerance, first {bad[:3]}"


def assert_bits(y, ref):
    np.testing.assert_array_equal(y.view(np.uint16), ref.view(np.uint16))


def act(M, K, seed=0, zero_rows=(), **kw):
    x = synth.activations(M, K, seed=seed, **kw)
    for r in zero_rows:
        if r < M:
            x[r] = 0
    return x


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w8.load()
    assert w8.w8a8_is_available(), "the current device is not a GB300 (compute 10.3)"


# ------------------------------------------------------- quantization ----

QUANT_CASES = [(1, 16, 0), (3, 48, 0), (37, 512, 0), (130, 2560, 0), (257, 4096, 0),
               (5, 14336, 0), (9, 32768, 0), (33, 512, 64), (130, 2560, 128), (7, 4096, 64),
               (65, 14336, 128)]


@pytest.mark.parametrize("M,K,gs", QUANT_CASES)
def test_act_quant_bit_exact(M, K, gs):
    x = act(M, K, seed=M + K, zero_rows=(0, M // 2), n_outliers=max(1, K // 100),
            outlier_scale=40.0)
    if M > 2:
        x[1] = synth.activations(1, K, seed=1, heavy_rows=True)[0] * np.float16(50)
    xq, sa = w8.quantize_act_per_token(dev(x), gs)
    rq, rs = oracle.quantize_act_per_token(x, gs)
    np.testing.assert_array_equal(host(xq), rq)
    np.testing.assert_array_equal(host(sa), rs)


def _all_fp16_upto(amax):
    bits = np.arange(0, 0x7C00, dtype=np.uint16)
    pos = bits.view(np.float16)
    pos = pos[pos.astype(np.float32) <= np.float32(amax)]
    return np.concatenate([pos, -pos[1:]])


@pytest.mark.parametrize("amax", [127.0, 100.0, 3.140625, 0.0999755859375, 65504.0,
                                  1000.5, 2.0 ** -20, 6.103515625e-05])
def test_act_quant_exhaustive_fp16(amax):
    """Every finite fp16 value up to a fixed absmax, laid out in rows that
    each contain +-absmax (so every row has the same scale): the GPU's
    reciprocal fast path with its near-tie fallback must give exactly the
    codes of one IEEE division and round-half-even, for all of them."""
    vals = _all_fp16_upto(amax)
    K = 4096
    per_row = K - 2
    rows = -(-vals.size // per_row)
    x = np.zeros((rows, K), np.float16)
    flat = np.resize(vals, rows * per_row).reshape(rows, per_row)
    x[:, 0] = np.float16(amax)
    x[:, 1] = -np.float16(amax)
    x[:, 2:] = flat
    for gs in (0, 128):
        xq, sa = w8.quantize_act_per_token(dev(x), gs)
        rq, rs = oracle.quantize_act_per_token(x, gs)
        np.testing.assert_array_equal(host(xq), rq)
        np.testing.assert_array_equal(host(sa), rs)
    xh, sh = w8.quantize_act_per_token_h(dev(x))
    rq, rs = oracle.quantize_act_per_token(x)
    np.testing.assert_array_equal(host(xh), rq.astype(np.float16))
    np.testing.assert_array_equal(host(sh), rs)


@pytest.mark.parametrize("M,K,gs", [(3, 48, 0), (130, 2560, 128), (257, 4096, 64), (5, 14336, 0)])
def test_act_quant_half_codes(M, K, gs):
    """quantize_act_per_token_h writes exactly the INT8 codes, as fp16."""
    x = act(M, K, seed=K + 1, zero_rows=(0,), n_outliers=3, outlier_scale=40.0)
    xh, sa = w8.quantize_act_per_token_h(dev(x), gs)
    rq, rs = oracle.quantize_act_per_token(x, gs)
    np.testing.assert_array_equal(host(xh), rq.astype(np.float16))
    np.testing.assert_array_equal(host(sa), rs)


@pytest.mark.parametrize("N,K,gs", [(1, 16, 0), (257, 512, 0), (130, 2560, 64),
                                    (64, 4096, 128), (33, 14336, 0)])
def test_weight_quant_bit_exact(N, K, gs):
    W = synth.weights(N, K, seed=N)
    W[0, :] = 0
    wq, sw = w8.quantize_weight_int8(dev(W), gs)
    rq, rs = oracle.quantize_weight_int8(W, gs)
    np.testing.assert_array_equal(host(wq), rq)
    np.testing.assert_array_equal(host(sw), rs)


@pytest.mark.parametrize("N,K", [(1, 32), (257, 512), (130, 4096), (17, 14336)])
def test_int4_pack_bit_exact(N, K):
    W = synth.weights(N, K, seed=K)
    W[-1, :] = 0
    wp, s4 = w8.pack_weight_int4(dev(W))
    rp, rs = oracle.pack_weight_int4(W)
    np.testing.assert_array_equal(host(wp), rp)
    np.testing.assert_array_equal(host(s4), rs)


# ----------------------------------------------------- INT32 contraction ----

I32_CASES = [  # (M, N, K, gs, wbits): several tiles and ragged tails
    (2, 1, 16, 0, 8), (130, 257, 192, 0, 8), (257, 130, 2560, 0, 8), (1, 300, 512, 0, 8),
    (300, 129, 4096, 0, 8), (129, 131, 48, 0, 8), (130, 257, 512, 64, 8),
    (257, 200, 2560, 128, 8), (3, 129, 1024, 64, 8), (130, 257, 512, 0, 4),
    (257, 64, 4096, 0, 4), (1, 33, 96, 0, 4)]


@pytest.mark.parametrize("M,N,K,gs,wbits", I32_CASES)
def test_int32_sums_bit_exact(M, N, K, gs, wbits):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    if wbits == 8:
        w = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
        wdev = dev(w)
    else:
        w = rng.integers(-7, 8, size=(N, K), dtype=np.int8)
        wdev = dev(oracle.pack_int4(w))
    acc = w8.w8a8_gemm_i32(dev(a), wdev, gs, wbits)
    np.testing.assert_array_equal(host(acc), oracle.int_gemm(a, w, gs))


def test_int32_worst_case_magnitudes():
    """All-extreme operands: every product is +-127^2 and the sums reach
    127^2 * K, the largest magnitude the format allows at K = 32768."""
    K = 32768
    a = np.full((3, K), 127, np.int8)
    a[1] = -127
    a[2, ::2] = -127
    w = np.full((5, K), 127, np.int8)
    w[1] = -127
    w[3, 1::2] = -127
    w[4, : K // 2] = 1
    acc = w8.w8a8_gemm_i32(dev(a), dev(w))
    np.testing.assert_array_equal(host(acc), oracle.int_gemm(a, w))
    assert host(acc).max() == 127 * 127 * K


# ------------------------------------------------------ fused dequant ----

GEMM_CASES = [(130, 257, 512, 0), (257, 130, 2560, 0), (64, 96, 4096, 64),
              (200, 257, 2560, 128), (2, 3, 16, 0), (129, 520, 14336, 0)]


@pytest.mark.parametrize("M,N,K,gs", GEMM_CASES)
def test_w8a8_gemm_output(M, N, K, gs):
    x = act(M, K, seed=K, n_outliers=4, outlier_scale=40.0, zero_rows=(M - 1,))
    W = synth.weights(N, K, seed=N)
    xq, sa = oracle.quantize_act_per_token(x, gs)
    wq, sw = oracle.quantize_weight_int8(W, gs)
    ref = oracle.dequant(oracle.int_gemm(xq, wq, gs), sa, sw)
    y = host(w8.w8a8_gemm(dev(xq), dev(sa), dev(wq), dev(sw), gs))
    assert_fp16_close(y, ref)
    assert_bits(y, ref)


@pytest.mark.parametrize("M,N,K,gs,wbits", [
    (130, 257, 512, 0, 8), (257, 130, 2560, 0, 8), (1, 300, 2560, 0, 8), (64, 96, 4096, 64, 8),
    (200, 257, 2560, 128, 8), (2, 3, 16, 0, 8), (129, 520, 14336, 0, 8), (300, 257, 4096, 0, 4),
    (1, 129, 512, 0, 4), (400, 300, 1024, 64, 8), (577, 129, 4096, 128, 8)])
def test_gemm_with_half_codes(M, N, K, gs, wbits):
    """The GEMM fed with fp16 activation codes (the path linear uses for
    M > 1) gives the oracle's outputs bit for bit."""
    x = act(M, K, seed=K + 7, n_outliers=4, outlier_scale=40.0, zero_rows=(M - 1,))
    W = synth.weights(N, K, seed=N + 7)
    xq, sa = oracle.quantize_act_per_token(x, gs)
    if wbits == 8:
        wq, sw = oracle.quantize_weight_int8(W, gs)
        ref = oracle.dequant(oracle.int_gemm(xq, wq, gs), sa, sw)
    else:
        wq, sw = oracle.pack_weight_int4(W)
        ref = oracle.dequant(oracle.int_gemm(xq, oracle.unpack_int4(wq, K)), sa, sw)
    y = host(w8.w8a8_gemm_h(dev(xq.astype(np.float16)), dev(sa), dev(wq), dev(sw), gs, wbits))
    assert_fp16_close(y, ref)
    assert_bits(y, ref)


@pytest.mark.parametrize("N,K,gs", [(257, 512, 0), (10240, 2560, 0), (130, 2560, 64),
                                    (300, 4096, 128), (4096, 14336, 0), (1, 16, 0),
                                    (700, 48, 0), (5, 32768, 0), (33, 64, 64), (9, 32768, 64),
                                    (3000, 32768, 64), (1001, 640, 128)])
def test_w8a8_mv_output(N, K, gs):
    x = act(1, K, seed=N + 1, n_outliers=2, outlier_scale=30.0)
    W = synth.weights(N, K, seed=N + 2)
    xq, sa = oracle.quantize_act_per_token(x, gs)
    wq, sw = oracle.quantize_weight_int8(W, gs)
    ref = oracle.dequant(oracle.int_gemm(xq, wq, gs), sa, sw)
    y = host(w8.w8a8_mv(dev(xq), dev(sa), dev(wq), dev(sw), gs))
    assert_fp16_close(y, ref)
    if gs == 0:
        assert_bits(y, ref)


@pytest.mark.parametrize("M,N,K", [(1, 257, 512), (1, 14336, 4096), (130, 257, 512),
                                   (257, 129, 4096), (2, 64, 32), (1, 700, 32), (1, 7, 32768)])
def test_w4a8_gemm_output(M, N, K):
    x = act(M, K, seed=M + 5)
    W = synth.weights(N, K, seed=N + 5)
    xq, sa = oracle.quantize_act_per_token(x)
    wp, s4 = oracle.pack_weight_int4(W)
    ref = oracle.dequant(oracle.int_gemm(xq, oracle.unpack_int4(wp, K)), sa, s4)
    y = host(w8.w4a8_gemm(dev(xq), dev(sa), dev(wp), dev(s4)))
    assert_fp16_close(y, ref)
    assert_bits(y, ref)


# --------------------------------------------------------- whole layer ----

@pytest.mark.parametrize("M,N,K,gs,wbits", [
    (1, 512, 512, 0, 8), (128, 512, 512, 0, 8), (5, 300, 2560, 128, 8), (1, 300, 2560, 64, 8),
    (300, 257, 4096, 0, 4), (1, 257, 4096, 0, 4), (1, 40, 32768, 64, 8), (1, 1000, 16, 0, 8),
    (1, 333, 96, 0, 4)])
def test_linear_matches_oracle(M, N, K, gs, wbits):
    x = act(M, K, seed=3, n_outliers=4, outlier_scale=40.0)
    W = synth.weights(N, K, seed=4)
    if wbits == 8:
        wq, sw = oracle.quantize_weight_int8(W, gs)
    else:
        wq, sw = oracle.pack_weight_int4(W)
    ref = oracle.linear(x, wq, sw, gs, wbits)
    y = host(w8.linear(dev(x), dev(wq), dev(sw), gs, wbits))
    assert_fp16_close(y, ref)
    if gs == 0 or M > 1:
        assert_bits(y, ref)


def test_small_workload_end_to_end():
    """W8A8 per-channel linear, M=128 tokens, K=512, N=512, seed 0: x ~ N(0,1)
    with 4 of the 512 K-channels scaled x40; weights N(0, 0.02) quantized
    per output channel on the GPU; activations quantized per token."""
    cfg = synth.WORKLOADS["pc_small"]
    M, N, K = cfg["Ms"][0], cfg["N"], cfg["K"]
    x = synth.activations(M, K, seed=0, **cfg["act"])
    W = synth.weights(N, K, seed=0)
    wq, sw = w8.quantize_weight_int8(dev(W))
    rq, rs = oracle.quantize_weight_int8(W)
    np.testing.assert_array_equal(host(wq), rq)
    np.testing.assert_array_equal(host(sw), rs)
    y = host(w8.linear(dev(x), wq, sw))
    ref = oracle.linear(x, rq, rs)
    assert_fp16_close(y, ref)
    assert_bits(y, ref)


# ------------------------------------------------------------ edge cases ----

def test_empty_problems_are_noops():
    x = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    xq, sa = w8.quantize_act_per_token(x)
    assert xq.shape == (0, 64) and sa.shape == (0, 1)
    wq = torch.empty((0, 64), dtype=torch.int8, device="cuda")
    sw = torch.empty((0, 1), dtype=torch.float32, device="cuda")
    xq1, sa1 = w8.quantize_act_per_token(torch.ones((3, 64), dtype=torch.float16, device="cuda"))
    assert w8.w8a8_gemm(xq1, sa1, wq, sw).shape == (3, 0)
    assert w8.linear(x, wq, sw).shape == (0, 0)


def test_misaligned_pointer_is_rejected():
    buf = torch.zeros(4 * 64 + 8, dtype=torch.float16, device="cuda")
    x = buf[4:4 + 4 * 64].view(4, 64)  # 8-byte offset
    with pytest.raises(w8.W8A8Error) as e:
        w8.quantize_act_per_token(x)
    assert e.value.status == 2


def test_outputs_outside_the_problem_are_untouched():
    """Guard bytes around y: the kernels write exactly M x N outputs."""
    M, N, K = 130, 257, 512
    x = act(M, K, seed=11)
    W = synth.weights(N, K, seed=11)
    wq, sw = oracle.quantize_weight_int8(W)
    for m in (M, 1):
        big = torch.full((m * N + 64,), 12345, dtype=torch.int16, device="cuda")
        y = big[32:32 + m * N].view(torch.float16).view(m, N)
        w8.linear(dev(x[:m]), dev(wq), dev(sw), y=y)
        g = host(big)
        assert np.all(g[:32] == 12345) and np.all(g[32 + m * N:] == 12345)


def test_device_status_clean_after_calls():
    assert w8.w8a8_check_status() == 0
