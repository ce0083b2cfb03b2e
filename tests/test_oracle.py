"""Pins for the CPU oracle: each test checks it against something other than
itself (hand-worked examples, exhaustive fp16 sweeps with brute-force
rounding, exact rational bounds, numpy's integer matmul, closed forms and
invariants).  No GPU needed.

Method sources: "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다",
section "INT8 TensorOps 커널 설계" (four-step pipeline) and section
"입도(Granularity)"; "cider 소개", section "cider의 양자화 모드와 적용 가능한
영역" (W8A8 / W4A8 modes, per-channel and per-group).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from golden_io import act_quant_cases, int4_cases, linear_cases, weight_only_cases
from w4a8_int8_quantized_gb300 import synth


# ---------------------------------------------------------------- golden ----

@pytest.mark.parametrize("case", act_quant_cases(), ids=lambda c: c["name"])
def test_golden_act_quant(case):
    q, s = oracle.quant_rows(case["x"][None, :], case["gs"])
    np.testing.assert_array_equal(q[0], case["q"])
    np.testing.assert_array_equal(s[0], case["s"])


def test_golden_int4():
    packs, quants = int4_cases()
    for q4, packed in packs:
        np.testing.assert_array_equal(oracle.pack_int4(q4[None, :])[0], packed)
        np.testing.assert_array_equal(oracle.unpack_int4(packed[None, :], q4.size)[0], q4)
    for w, s4, q4, packed in quants:
        p, s = oracle.pack_weight_int4(w[None, :])
        assert s[0, 0] == s4
        np.testing.assert_array_equal(p[0], packed)
        np.testing.assert_array_equal(oracle.unpack_int4(p, w.size)[0], q4)


@pytest.mark.parametrize("case", linear_cases(), ids=lambda c: c["name"])
def test_golden_linear(case):
    gs = case["gs"]
    M, K = case["x"].shape
    N = case["W"].shape[0]
    G = 1 if gs == 0 else K // gs
    xq, sa = oracle.quantize_act_per_token(case["x"], gs)
    wq, sw = oracle.quantize_weight_int8(case["W"], gs)
    np.testing.assert_array_equal(xq, case["xq"])
    np.testing.assert_array_equal(wq, case["wq"])
    np.testing.assert_array_equal(sa.reshape(-1), case["sa"].reshape(-1))
    np.testing.assert_array_equal(sw.reshape(-1), case["sw"].reshape(-1))
    acc = oracle.int_gemm(xq, wq, gs)
    np.testing.assert_array_equal(acc.reshape(-1), case["acc"].reshape(-1))
    y = oracle.dequant(acc, sa, sw)
    np.testing.assert_array_equal(y.reshape(-1), case["y"].reshape(-1))
    np.testing.assert_array_equal(oracle.linear(case["x"], wq, sw, gs).reshape(-1),
                                  case["y"].reshape(-1))
    assert acc.shape == (M, N, G)


# ------------------------------------------- exhaustive fp16 quant sweeps ----

def _finite_fp16_upto(a):
    bits = np.arange(0, 0x7C00, dtype=np.uint16)  # +0 .. largest finite
    pos = bits.view(np.float16)
    pos = pos[pos.astype(np.float32) <= np.float32(a)]
    return np.concatenate([pos, -pos[1:]])


def _nearest_even(t):
    """Brute-force nearest integer in [-127, 127], ties to the even one."""
    cand = np.arange(-127, 128, dtype=np.float64)
    d = np.abs(t.astype(np.float64)[:, None] - cand[None, :])
    best = d.min(axis=1, keepdims=True)
    is_best = d == best
    # among tied candidates prefer the even one
    even = (cand.astype(np.int64) % 2 == 0)[None, :]
    pick = np.where((is_best & even).any(axis=1, keepdims=True), is_best & even, is_best)
    return cand[pick.argmax(axis=1)].astype(np.int64)


@pytest.mark.parametrize("amax", [127.0, 1.0, 3.140625, 0.0999755859375, 65504.0,
                                  6.103515625e-05, 1000.5, 2.0 ** -20])
def test_exhaustive_fp16_rounding(amax):
    """For one fixed absmax, every finite fp16 x with |x| <= absmax: q is the
    integer nearest to the fp32 quotient x/s (ties to even), the real-number
    error |x - q*s| is at most s/2 (up to the fp32 rounding of x/s), and
    +-absmax maps to +-127."""
    xs = _finite_fp16_upto(amax)
    row = np.concatenate([[np.float16(amax)], xs]).astype(np.float16)
    q, s = oracle.quant_rows(row[None, :])
    q = q[0].astype(np.int64)
    s = np.float32(s[0, 0])
    assert s == np.float32(np.float16(amax)) / np.float32(127)
    t = row.astype(np.float32) / s  # the fp32 quotient the reading specifies
    np.testing.assert_array_equal(q, _nearest_even(t))
    assert q[0] == 127 and np.all(np.abs(q) <= 127)
    neg = np.where(row == -np.float16(amax))[0]
    assert np.all(q[neg] == -127)
    # exact rational error bound on a strided subset (Fractions are slow)
    sf = Fraction(float(s))
    for i in range(0, row.size, max(1, row.size // 2000)):
        err = abs(Fraction(float(row[i])) - q[i] * sf)
        assert err <= sf / 2 * (1 + Fraction(1, 2 ** 20)), (row[i], q[i])


def test_quant_invariants():
    x = synth.activations(64, 256, seed=3, n_outliers=3, outlier_scale=40.0)
    q, s = oracle.quant_rows(x)
    # sign symmetry
    qn, sn = oracle.quant_rows(-x)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sn, s)
    # power-of-two scaling leaves q unchanged and scales s exactly
    for k in (-1, 1, 3):
        xk = (x.astype(np.float32) * np.float32(2.0 ** k)).astype(np.float16)
        exact = np.all(xk.astype(np.float32) == x.astype(np.float32) * np.float32(2.0 ** k))
        assert exact
        qk, sk = oracle.quant_rows(xk)
        np.testing.assert_array_equal(qk, q)
        np.testing.assert_array_equal(sk, s * np.float32(2.0 ** k))
    # the row maximum maps to +-127
    idx = np.abs(x.astype(np.float32)).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(64), idx]) == 127)
    # -128 never appears
    assert q.min() >= -127


def test_zero_rows_and_groups():
    x = synth.activations(4, 256, seed=1)
    x[1] = 0
    x[2, 128:] = 0
    q, s = oracle.quant_rows(x, 128)
    assert np.all(q[1] == 0) and np.all(s[1] == 0)
    assert np.all(q[2, 128:] == 0) and s[2, 1] == 0 and s[2, 0] > 0
    qp, sp = oracle.quant_rows(x)
    assert sp[1, 0] == 0 and np.all(qp[1] == 0)


def test_nonfinite_rejected():
    x = np.zeros((1, 8), np.float16)
    x[0, 3] = np.inf
    with pytest.raises(oracle.OracleError):
        oracle.quant_rows(x)


# ----------------------------------------------------- integer contraction ----

def test_int_gemm_matches_numpy_int64():
    rng = np.random.default_rng(7)
    for (M, N, K, gs) in [(5, 7, 64, 0), (3, 9, 128, 64), (17, 13, 256, 128), (1, 33, 96, 32)]:
        a = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
        w = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
        acc = oracle.int_gemm(a, w, gs)
        G = 1 if gs == 0 else K // gs
        g = K if gs == 0 else gs
        ref = np.einsum("mgk,ngk->mng", a.astype(np.int64).reshape(M, G, g),
                        w.astype(np.int64).reshape(N, G, g))
        np.testing.assert_array_equal(acc, ref)


def test_int_gemm_brute_force_tiny():
    rng = np.random.default_rng(11)
    for _ in range(20):
        M, N = rng.integers(1, 6, size=2)
        K = int(rng.integers(1, 9))
        a = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
        w = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
        acc = oracle.int_gemm(a, w)
        # k-outer accumulation in Python integers: a different loop order
        ref = [[0] * N for _ in range(M)]
        for k in range(K):
            for n in range(N):
                for m in range(M):
                    ref[m][n] += int(a[m, k]) * int(w[n, k])
        np.testing.assert_array_equal(acc[:, :, 0], np.array(ref))


def test_int_gemm_worst_case_and_overflow():
    K = 14336
    a = np.full((1, K), 127, np.int8)
    w = np.full((1, K), -127, np.int8)
    assert oracle.int_gemm(a, w)[0, 0, 0] == -127 * 127 * K
    K = 133200  # 127^2 * K > 2^31 - 1
    with pytest.raises(oracle.OracleError):
        oracle.int_gemm(np.full((1, K), 127, np.int8), np.full((1, K), 127, np.int8))


def test_group_partials_sum_to_per_channel():
    rng = np.random.default_rng(5)
    a = rng.integers(-127, 128, size=(6, 256), dtype=np.int8)
    w = rng.integers(-127, 128, size=(5, 256), dtype=np.int8)
    pc = oracle.int_gemm(a, w)[:, :, 0]
    for gs in (64, 128, 32):
        np.testing.assert_array_equal(oracle.int_gemm(a, w, gs).sum(axis=2), pc)


def test_group_size_k_equals_per_channel():
    x = synth.activations(8, 128, seed=2, n_outliers=2, outlier_scale=30.0)
    W = synth.weights(12, 128, seed=2)
    wq0, sw0 = oracle.quantize_weight_int8(W, 0)
    wqK, swK = oracle.quantize_weight_int8(W, 128)
    np.testing.assert_array_equal(wq0, wqK)
    np.testing.assert_array_equal(sw0, swK)
    np.testing.assert_array_equal(oracle.linear(x, wq0, sw0, 0), oracle.linear(x, wqK, swK, 128))


# ------------------------------------------------------------- int4 pack ----

def test_int4_pack_bijection_all_bytes():
    allbytes = np.arange(256, dtype=np.uint8).reshape(1, 256)
    q4 = oracle.unpack_int4(allbytes, 512)
    assert q4.min() == -8 and q4.max() == 7
    np.testing.assert_array_equal(oracle.pack_int4(q4), allbytes)
    # two's complement nibbles, low nibble first
    lo = allbytes[0].astype(np.int64) & 0xF
    hi = allbytes[0].astype(np.int64) >> 4
    np.testing.assert_array_equal(q4[0, 0::2], np.where(lo >= 8, lo - 16, lo))
    np.testing.assert_array_equal(q4[0, 1::2], np.where(hi >= 8, hi - 16, hi))


def test_int4_weight_range_and_error():
    W = synth.weights(32, 256, seed=4)
    p, s4 = oracle.pack_weight_int4(W)
    q4 = oracle.unpack_int4(p, 256)
    assert q4.min() >= -7 and q4.max() <= 7
    err = np.abs(W.astype(np.float64) - q4 * s4.astype(np.float64))
    assert np.all(err <= s4.astype(np.float64) / 2 * (1 + 2 ** -20))


# ---------------------------------------------------------------- dequant ----

def test_dequant_exact_with_power_of_two_scales():
    acc = np.array([[[12035], [-16193], [1 << 20]]], np.int32)
    sa = np.array([[0.5]], np.float32)
    sw = np.array([[2.0 ** -7], [2.0 ** -6], [2.0 ** -12]], np.float32)
    y = oracle.dequant(acc, sa, sw)
    # 12035/256 = 47.01171875 -> fp16 (ulp 2^-5) 47.0; -16193/128 = -126.5078125
    # -> (ulp 2^-4) -126.5; 2^20/2^13 = 128 exactly.
    np.testing.assert_array_equal(y[0], np.array([47.0, -126.5, 128.0], np.float16))


def test_dequant_error_bound_random():
    rng = np.random.default_rng(9)
    acc = rng.integers(-2 ** 26, 2 ** 26, size=(7, 9, 1)).astype(np.int32)
    sa = rng.uniform(1e-4, 1e-1, size=(7, 1)).astype(np.float32)
    sw = rng.uniform(1e-5, 1e-2, size=(9, 1)).astype(np.float32)
    y = oracle.dequant(acc, sa, sw).astype(np.float64)
    exact = acc[:, :, 0].astype(np.float64) * sa.astype(np.float64) * sw.astype(np.float64).T
    # three fp32 roundings (float(acc), sa*sw, the product) then one fp16
    ulp16 = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(y - exact) <= ulp16 / 2 + np.abs(exact) * 3 * 2 ** -24)


def test_identity_weight_recovers_x():
    K = 256
    x = synth.activations(16, K, seed=6)
    W = np.eye(K, dtype=np.float16)
    wq, sw = oracle.quantize_weight_int8(W)
    assert np.all(wq == 127 * np.eye(K, dtype=np.int8))
    y = oracle.linear(x, wq, sw).astype(np.float64)
    _, sa = oracle.quantize_act_per_token(x)
    tol = sa.astype(np.float64) / 2 * (1 + 1e-6) + np.spacing(np.abs(x).astype(np.float16)) + 1e-7
    assert np.all(np.abs(y - x.astype(np.float64)) <= tol)


def test_sampled_matches_full():
    x = synth.activations(33, 192, seed=8, heavy_rows=True)
    W = synth.weights(47, 192, seed=8)
    for gs in (0, 64):
        xq, sa = oracle.quantize_act_per_token(x, gs)
        wq, sw = oracle.quantize_weight_int8(W, gs)
        acc = oracle.int_gemm(xq, wq, gs)
        y = oracle.dequant(acc, sa, sw)
        rows = np.array([0, 32, 5, 17]); cols = np.array([0, 46, 23, 1])
        acc_s, y_s = oracle.sampled_outputs(xq, sa, wq, sw, rows, cols, gs)
        np.testing.assert_array_equal(acc_s, acc[rows, cols])
        np.testing.assert_array_equal(y_s, y[rows, cols])


def test_w4a8_linear_equals_unpacked_w8_path():
    x = synth.activations(9, 128, seed=10)
    W = synth.weights(10, 128, seed=10)
    p, s4 = oracle.pack_weight_int4(W)
    q4 = oracle.unpack_int4(p, 128)
    np.testing.assert_array_equal(oracle.linear(x, p, s4, 0, wbits=4),
                                  oracle.linear(x, q4, s4, 0, wbits=8))


# ------------------------------------------ weight-only (W8A16 / W4A16) ----
#
# The baseline the method is measured against: fp16 activations times the
# integer weights dequantized with their scales ("Apple Silicon의 AI 한계치는
# …", the section on MLX's weight-only quantization; "cider 소개", mode table
# and the w8a16 / w4a16 latency columns).

@pytest.mark.parametrize("case", weight_only_cases(), ids=lambda c: c["name"])
def test_golden_weight_only(case):
    y = oracle.weight_only(case["x"], case["q"], case["sw"], case["gs"])
    np.testing.assert_array_equal(y.view(np.uint16), case["y"].view(np.uint16))


def test_weight_only_unit_rows_pick_one_weight():
    """x = e_k (one 1 per row) selects column k: y[m, n] = fp16(q[n, k] * s_w[n, g(k)]),
    rounded by numpy's own float64 -> float16 conversion."""
    rng = np.random.default_rng(11)
    K, N = 256, 37
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    for gs in (0, 64, 128):
        G = 1 if gs == 0 else K // gs
        sw = (rng.random((N, G)) * 0.05).astype(np.float32)
        ks = rng.choice(K, size=20, replace=False)
        x = np.zeros((ks.size, K), np.float16)
        x[np.arange(ks.size), ks] = 1
        y = oracle.weight_only(x, q, sw, gs)
        g = ks // (K if gs == 0 else gs)
        want = (q[:, ks].T.astype(np.float64) * sw[:, g].T.astype(np.float64)).astype(np.float16)
        np.testing.assert_array_equal(y.view(np.uint16), want.view(np.uint16))


def test_weight_only_matches_float64_matmul():
    """Against numpy's float64 matmul of x with the dequantized weights (a
    different summation order): within one fp16 ulp everywhere, and bit-equal
    except where the exact value sits within 2^-35 (relative) of a rounding
    boundary."""
    rng = np.random.default_rng(12)
    M, N, K = 33, 65, 512
    x = synth.activations(M, K, seed=3, n_outliers=3, outlier_scale=30.0)
    for gs, wbits in ((0, 8), (64, 8), (128, 8), (0, 4)):
        W = synth.weights(N, K, seed=4 + gs)
        if wbits == 8:
            q, sw = oracle.quantize_weight_int8(W, gs)
        else:
            p, sw = oracle.pack_weight_int4(W)
            q = oracle.unpack_int4(p, K)
        G = sw.shape[1]
        deq = q.astype(np.float64) * np.repeat(sw.astype(np.float64), K // G, axis=1)
        ref64 = x.astype(np.float64) @ deq.T
        ref = ref64.astype(np.float16)
        y = oracle.weight_only(x, q, sw, gs)
        ulp = np.spacing(np.abs(ref)).astype(np.float64)
        assert np.all(np.abs(y.astype(np.float64) - ref.astype(np.float64)) <= ulp)
        assert np.mean(y.view(np.uint16) == ref.view(np.uint16)) > 0.999
        if wbits == 4:
            np.testing.assert_array_equal(
                oracle.linear_weight_only(x, p, sw, 0, 4).view(np.uint16), y.view(np.uint16))


def test_weight_only_quantization_error_bound():
    """|y - x . W^T| <= sum_k |x_k| s_w / 2 + half an fp16 ulp of y: the only
    errors are the weight rounding (at most half a step each) and the final
    fp16 rounding (per channel, INT8 and INT4)."""
    M, N, K = 17, 40, 1024
    x = synth.activations(M, K, seed=5, n_outliers=4, outlier_scale=40.0)
    W = synth.weights(N, K, seed=6)
    exact = x.astype(np.float64) @ W.astype(np.float64).T
    xs = np.abs(x.astype(np.float64)).sum(axis=1)
    for wbits in (8, 4):
        if wbits == 8:
            q, sw = oracle.quantize_weight_int8(W)
            y = oracle.weight_only(x, q, sw)
        else:
            p, sw = oracle.pack_weight_int4(W)
            y = oracle.linear_weight_only(x, p, sw, 0, 4)
        bound = xs[:, None] * sw[:, 0][None, :].astype(np.float64) / 2 * (1 + 1e-6)
        bound += np.spacing(np.abs(y)).astype(np.float64) / 2
        assert np.all(np.abs(y.astype(np.float64) - exact) <= bound)


def test_weight_only_special_cases():
    """gs = K equals per channel; x -> -x gives y -> -y; integer x with
    power-of-two scales equals the exact W8A8 path (s_a = 1, every step
    exact); zero weights give zero."""
    rng = np.random.default_rng(13)
    M, N, K = 9, 21, 256
    x = synth.activations(M, K, seed=7)
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    sw = (rng.random((N, 1)) * 0.05).astype(np.float32)
    a = oracle.weight_only(x, q, sw, 0)
    b = oracle.weight_only(x, q, sw, K)
    np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))
    np.testing.assert_array_equal((-a).view(np.uint16), oracle.weight_only(-x, q, sw).view(np.uint16))
    xi = rng.integers(-127, 128, size=(M, K)).astype(np.float16)
    xi[:, 0] = 127  # row absmax 127: the activation scale is exactly 1
    sp = (2.0 ** -rng.integers(6, 12, size=(N, 1))).astype(np.float32)
    xq, sa = oracle.quantize_act_per_token(xi)
    assert np.all(sa == 1) and np.array_equal(xq, xi.astype(np.int8))
    w8a8 = oracle.dequant(oracle.int_gemm(xq, q), sa, sp)
    np.testing.assert_array_equal(oracle.weight_only(xi, q, sp).view(np.uint16), w8a8.view(np.uint16))
    assert np.all(oracle.weight_only(x, np.zeros_like(q), sw) == 0)
