"""Parity of the CUDA path (called through the C ABI via the binding) against
the CPU oracle, on the same seeded inputs.

The bar: INT8 codes, INT4 packed bytes, fp32 scales and INT32 sums
bit-exact; fp16 outputs within |dy| <= 2e-3 * max|y_ref| + ulp_fp16(y_ref)
element by element.  Where the kernel evaluates the dequant in the oracle's
operation order (per channel, on every path) the fp16 output is also checked
bit-exact; the per-group GEMM accumulates the rescaled group partials with
fused multiply-adds (the order of the dequant is not fixed by the method), so
its outputs are held to the tolerance.

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


@pytest.mark.parametrize("M,K,gs", [(3, 48, 0), (130, 2560, 128), (257, 4096, 64), (5, 14336, 0),
                                   (3001, 2560, 0), (2999, 4096, 128), (1801, 1024, 64),
                                   (4099, 256, 0), (2500, 8192, 0)])
def test_act_quant_half_codes(M, K, gs):
    """quantize_act_per_token_h writes exactly the INT8 codes, as fp16.  The
    larger M make every row team of the persistent kernel take several rows
    (with its next row loaded while the current one is quantized), with a
    ragged last round; K from 256 (one vector per thread) to 8192 (four)."""
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


# ---------------------------------- exactness of the fp32 tensor-core sums ----
#
# The contraction runs on kind::f16 tensor cores with an fp32 accumulator
# that is drained every K-chunk (1024 for INT8 weights, 16384 for INT4).  It
# is exact only if the accumulator keeps every bit of an integer below 2^24
# while each 16-deep MMA adds an integer of any parity.  These inputs drive
# the running sum of every chunk of every (token, channel) pair into
# [2^23, 2^24), with per-MMA increments of random parity and runs of +-1
# products added to an accumulator already near 2^24; a tensor core that
# aligned its addends with fewer than 24 significant bits would lose low
# bits here.

CHUNK = {8: 1024, 4: 16384}


def _large_partial_operands(M, N, K, wbits, seed):
    """a [M, K], w [N, K] with a[m, k] w[n, k] >= 0 almost everywhere: a is
    +-127 with one sign pattern s(k) shared by all rows, w is s(k) times a
    magnitude drawn from the top of the range; every chunk then sums to
    between 2^23 and 2^24.  Row variants: a tail of each chunk with +-1
    activations (small increments on a large accumulator), weights whose
    chunk tails are +-1, a few perturbed activations, and all-negative
    products (negative accumulators)."""
    rng = np.random.default_rng(seed)
    qmax = 127 if wbits == 8 else 7
    lo = 100 if wbits == 8 else 5
    chunk = CHUNK[wbits]
    s = np.where(rng.random(K) < 0.5, -1, 1).astype(np.int64)
    kin = np.arange(K) % chunk
    a = np.tile(127 * s, (M, 1))
    for m in range(M):
        kind = m % 4
        if kind == 1:      # the last 1/8 of every chunk: +-1 activations
            tail = kin >= chunk - chunk // 8
            a[m, tail] = s[tail]
        elif kind == 2:    # a few perturbed magnitudes (odd and even)
            idx = rng.choice(K, size=min(K, 40), replace=False)
            a[m, idx] = s[idx] * rng.integers(1, 128, size=idx.size)
        elif kind == 3:    # negative products: the accumulator runs to -2^24
            a[m] = -a[m]
    w = s * rng.integers(lo, qmax + 1, size=(N, K))
    for n in range(0, N, 3):  # every third channel: +-1 weights at chunk tails
        tail = kin >= chunk - chunk // 16
        w[n, tail] = s[tail]
    return a.astype(np.int8), w.astype(np.int8)


def _chunk_partials(a, w, chunk):
    """Exact running partial of every chunk at its end, [M, N, K / chunk]."""
    a64, w64 = a.astype(np.int64), w.astype(np.int64)
    K = a.shape[1]
    return np.stack([a64[:, c:c + chunk] @ w64[:, c:c + chunk].T for c in range(0, K, chunk)],
                    axis=-1)


@pytest.mark.parametrize("M,N,K,wbits", [(130, 257, 4096, 8), (257, 130, 2048, 8),
                                         (130, 96, 32768, 4), (3, 33, 16384, 4)])
def test_int32_sums_exact_at_large_partials(M, N, K, wbits):
    a, w = _large_partial_operands(M, N, K, wbits, seed=K + M)
    part = np.abs(_chunk_partials(a, w, CHUNK[wbits]))
    # the inputs do what they are for: most chunk partials in [2^23, 2^24)
    assert part.max() < 2 ** 24
    assert np.mean(part >= 2 ** 23) > 0.5
    wdev = dev(w) if wbits == 8 else dev(oracle.pack_int4(w))
    acc = w8.w8a8_gemm_i32(dev(a), wdev, 0, wbits)
    np.testing.assert_array_equal(host(acc), oracle.int_gemm(a, w))


def _cancelling_operands(M, N, wbits, seed):
    """K = two chunks; the second chunk holds the products of the first with
    the opposite sign, in a different order along K, plus a few activations
    one or two below full scale.  Each chunk partial is near 2^24 while the
    exact total is small (|total| < 2048), so the fp16 output y = total (unit
    scales) shows any bit a chunk lost."""
    rng = np.random.default_rng(seed)
    chunk = CHUNK[wbits]
    qmax = 127 if wbits == 8 else 7
    lo = 100 if wbits == 8 else 5
    s = np.where(rng.random(chunk) < 0.5, -1, 1).astype(np.int64)
    v = rng.integers(lo, qmax + 1, size=(N, chunk))
    perm = rng.permutation(chunk)
    a1 = 127 * s
    a = np.empty((M, 2 * chunk), np.int64)
    a[:, :chunk] = a1
    a[:, chunk + perm] = a1
    w = np.empty((N, 2 * chunk), np.int64)
    w[:, :chunk] = s * v
    w[:, chunk + perm] = -(s * v)
    for m in range(M):  # perturb a few activations: total = -sum d * v
        half = m % 2
        idx = rng.choice(chunk, size=rng.integers(0, 8), replace=False)
        d = rng.integers(1, 3, size=idx.size)
        cols = idx if half == 0 else chunk + perm[idx]
        a[m, cols] = (127 - d) * s[idx]
    return a.astype(np.int8), w.astype(np.int8)


@pytest.mark.parametrize("M,N,wbits", [(130, 257, 8), (300, 129, 8), (130, 64, 4)])
def test_fp16_output_exact_at_large_partials(M, N, wbits):
    """Through the layer's own GEMM (fp16 codes, w8a8_gemm_h): with unit
    scales the fp16 output is the exact integer total, which stays below
    2048 although every chunk partial is near 2^24."""
    a, w = _cancelling_operands(M, N, wbits, seed=M + N)
    K = a.shape[1]
    part = np.abs(_chunk_partials(a, w, CHUNK[wbits]))
    assert part.min() >= 2 ** 22 and part.max() < 2 ** 24
    ref_acc = oracle.int_gemm(a, w)
    assert np.abs(ref_acc).max() < 2048
    sa = np.ones((M, 1), np.float32)
    sw = np.ones((N, 1), np.float32)
    ref = oracle.dequant(ref_acc, sa, sw)
    wdev = dev(w) if wbits == 8 else dev(oracle.pack_int4(w))
    y = host(w8.w8a8_gemm_h(dev(a.astype(np.float16)), dev(sa), wdev, dev(sw), 0, wbits))
    assert_bits(y, ref)
    acc = host(w8.w8a8_gemm_i32(dev(a), wdev, 0, wbits))
    np.testing.assert_array_equal(acc, ref_acc)
    assert K == 2 * CHUNK[wbits]


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
    if gs == 0:
        assert_bits(y, ref)


@pytest.mark.parametrize("M,N,K,gs,wbits", [
    (130, 257, 512, 0, 8), (257, 130, 2560, 0, 8), (1, 300, 2560, 0, 8), (64, 96, 4096, 64, 8),
    (200, 257, 2560, 128, 8), (2, 3, 16, 0, 8), (129, 520, 14336, 0, 8), (300, 257, 4096, 0, 4),
    (1, 129, 512, 0, 4), (400, 300, 1024, 64, 8), (577, 129, 4096, 128, 8)])
def test_gemm_with_half_codes(M, N, K, gs, wbits):
    """The GEMM fed with fp16 activation codes (the path linear uses for
    M > 1) gives the oracle's outputs, bit for bit per channel."""
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
    if gs == 0:
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


# ------------------------------------- few-row products (M = 2..16) ----
#
# Two to eight activation rows run on the weight stream of the matrix-vector
# kernel (one weight load, one dp4a per activation row) when their codes fit
# its shared memory, more rows on the tensor-core GEMM; the outputs are
# those of the oracle bit for bit on either side of that boundary.  ("cider 소개", section "cider의 동작 방식과 자동 경로 선택": the
# seq_len rule leaves the choice open between one token and a GEMM tile.)

SKINNY_CASES = [(2, 257, 512, 8), (3, 1000, 2560, 8), (4, 130, 4096, 8), (5, 300, 2560, 8),
                (8, 10240, 2560, 8), (13, 129, 4096, 8), (16, 520, 4096, 8), (16, 64, 256, 8),
                (2, 33, 32768, 8), (7, 100, 8192, 8), (2, 300, 1024, 4), (6, 129, 4096, 4),
                (16, 14336, 4096, 4), (9, 77, 8192, 4)]


@pytest.mark.parametrize("M,N,K,wbits", SKINNY_CASES)
def test_few_row_products_bit_exact(M, N, K, wbits):
    x = act(M, K, seed=M * 3 + K, n_outliers=4, outlier_scale=40.0, zero_rows=(M - 1,))
    W = synth.weights(N, K, seed=N + M)
    xq, sa = oracle.quantize_act_per_token(x)
    if wbits == 8:
        wq, sw = oracle.quantize_weight_int8(W)
        ref = oracle.dequant(oracle.int_gemm(xq, wq), sa, sw)
        y = host(w8.w8a8_gemm(dev(xq), dev(sa), dev(wq), dev(sw)))
    else:
        wq, sw = oracle.pack_weight_int4(W)
        ref = oracle.dequant(oracle.int_gemm(xq, oracle.unpack_int4(wq, K)), sa, sw)
        y = host(w8.w4a8_gemm(dev(xq), dev(sa), dev(wq), dev(sw)))
    assert_fp16_close(y, ref)
    assert_bits(y, ref)
    # the whole layer: the INT8 quantizer, then the same kernel
    yl = host(w8.linear(dev(x), dev(wq), dev(sw), 0, wbits))
    assert_bits(yl, oracle.linear(x, wq, sw, 0, wbits))


def test_few_row_products_extreme_codes():
    """All-+-127 activations and weights: the int32 sums reach 127^2 K."""
    M, N, K = 16, 96, 4096
    a = np.full((M, K), 127, np.int8)
    a[1::2] = -127
    w = np.full((N, K), 127, np.int8)
    w[::3, ::2] = -127
    sa = np.full((M, 1), 2.0 ** -7, np.float32)
    sw = np.full((N, 1), 2.0 ** -10, np.float32)
    ref = oracle.dequant(oracle.int_gemm(a, w), sa, sw)
    y = host(w8.w8a8_gemm(dev(a), dev(sa), dev(w), dev(sw)))
    assert_bits(y, ref)


# ------------------------------- weight-only W8A16 / W4A16 (the baseline) ----
#
# fp16 activations times the dequantized weights, float accumulation on the
# tensor cores; against the oracle's exact product rounded once, within the
# fp16 tolerance ("Apple Silicon의 AI 한계치는 …", MLX weight-only section;
# "cider 소개", W8A16 / W4A16 rows of the mode table).

WONLY_CASES = [(130, 257, 512, 0, 8), (257, 130, 2560, 128, 8), (300, 129, 4096, 64, 8),
               (129, 520, 14336, 0, 8), (2, 3, 16, 0, 8), (1, 300, 2560, 0, 8),
               (300, 257, 4096, 0, 4), (5, 1000, 2560, 0, 4), (513, 384, 2560, 64, 8),
               (64, 64, 32768, 0, 8)]


@pytest.mark.parametrize("M,N,K,gs,wbits", WONLY_CASES)
def test_weight_only_matches_oracle(M, N, K, gs, wbits):
    x = act(M, K, seed=K + M, n_outliers=4, outlier_scale=40.0, zero_rows=(M - 1,))
    W = synth.weights(N, K, seed=N + 11)
    if wbits == 8:
        wq, sw = oracle.quantize_weight_int8(W, gs)
    else:
        wq, sw = oracle.pack_weight_int4(W)
    ref = oracle.linear_weight_only(x, wq, sw, gs, wbits)
    y = host(w8.weight_only_gemm(dev(x), dev(wq), dev(sw), gs, wbits))
    assert_fp16_close(y, ref)
    assert np.all(y[M - 1] == 0)  # a zero row gives zero outputs


def test_weight_only_exact_cases():
    """Integer x with power-of-two scales: every product, sum and scaling is
    exact in fp32, so the output equals the oracle bit for bit."""
    rng = np.random.default_rng(21)
    M, N, K = 130, 257, 1024
    x = rng.integers(-8, 9, size=(M, K)).astype(np.float16)
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    sw = (2.0 ** -rng.integers(10, 14, size=(N, 1))).astype(np.float32)
    ref = oracle.weight_only(x, q, sw)
    y = host(w8.weight_only_gemm(dev(x), dev(q), dev(sw)))
    assert_bits(y, ref)


# --------------------------------------------------------- whole layer ----

@pytest.mark.parametrize("M,N,K,gs,wbits", [
    (1, 512, 512, 0, 8), (128, 512, 512, 0, 8), (5, 300, 2560, 128, 8), (1, 300, 2560, 64, 8),
    (300, 257, 4096, 0, 4), (1, 257, 4096, 0, 4), (1, 40, 32768, 64, 8), (1, 1000, 16, 0, 8),
    (1, 333, 96, 0, 4),
    # decode with part of each warp's weight segment staged in shared memory
    # and the rest streamed through registers
    (1, 4096, 14336, 128, 8), (1, 28672, 4096, 0, 4), (1, 3000, 8192, 0, 8)])
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
    if gs == 0:
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


def test_bounded_wait_gives_up_and_reports_timeout():
    """Failure detection without a fault: with the test hook, every CTA of
    the GEMM leaves its first weight-staging copy unissued and the role waits
    are limited to ~1 ms, so the converters' wait for that stage runs out.
    The kernel must return (abort flag, in-flight copies and MMAs allowed to
    land, TMEM freed), w8a8_check_status must report W8A8_ERR_TIMEOUT, and
    the context must stay usable: the next call is exact and the status
    clean."""
    M, N, K = 130, 257, 512
    rng = np.random.default_rng(5)
    a = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    w = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    ref = oracle.int_gemm(a, w)
    ad, wd = dev(a), dev(w)
    assert w8.w8a8_check_status() == 0
    try:
        w8.w8a8_test_set_fault(2_000_000, True)
        w8.w8a8_gemm_i32(ad, wd)
        status = w8.w8a8_check_status()
    finally:
        w8.w8a8_test_set_fault(0, False)
    assert status == 5, w8.w8a8_status_string(status)
    assert w8.w8a8_check_status() == 0  # read-and-clear
    acc = w8.w8a8_gemm_i32(ad, wd)
    np.testing.assert_array_equal(host(acc), ref)
    assert w8.w8a8_check_status() == 0
