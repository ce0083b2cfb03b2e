/*
 * CPU oracle for the W8A8 / W4A8 quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or constant table
 * with the CUDA library.
 *
 * It is deliberately plain: every step is the textbook definition written as
 * straight loops, in the order the method describes it, with no blocking,
 * no fusion and no reordering.  Compile with -O2 -ffp-contract=off and never
 * with -ffast-math, so that each float operation below is one IEEE fp32
 * operation rounded to nearest-even.
 *
 * Sources (web pages on the Cider W8A8 SDK; cited by title and section):
 *   [P1] "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다" (molayo1419.me),
 *        section "INT8 TensorOps 커널 설계", the four-step kernel pipeline:
 *        (1) dynamic min/max reduction for scales, (2) fp16 -> INT8 mapping,
 *        (3) INT8 GEMM with INT32 accumulation, (4) rescale of the INT32
 *        result by the product of activation and weight scales to fp16.
 *        Section "입도(Granularity)": per-group scales (group 64 or 128)
 *        need grouped dequantization during accumulation.
 *   [P2] "cider 소개" (discuss.pytorch.kr), section "cider의 양자화 모드와
 *        적용 가능한 영역": W8A8 = symmetric INT8 weights x per-token INT8
 *        activations; W4A8 = INT4 weights packed in uint8, unpacked before the
 *        INT8 matmul; per-channel = one scale per output channel, per-group
 *        gs=128 / gs=64.  Section "cider 설치와 사용법": quantize_weight_int8
 *        and pack_weight_int4 return (integer tensor, scale).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   - symmetric scale s = absmax / qmax in fp32 (qmax = 127 for INT8,
 *     7 for INT4); the quotient x / s is one IEEE fp32 division and is
 *     rounded half-to-even (rintf under the default rounding mode), then
 *     clamped to [-qmax, qmax]; -128 is never produced;
 *   - a group whose absmax is 0 gets s = 0 and q = 0;
 *   - a per-group scale applies to both operands along K; group_size 0 means
 *     one group spanning K (per-token activations, per-channel weights);
 *   - INT4 nibbles are two's complement, the low nibble holds the even k;
 *   - per-channel dequant: y = half((float)acc * (s_a * s_w)), the scale
 *     product first; per-group: f accumulates (float)acc_g * (s_a,g * s_w,g)
 *     over g in ascending order, then y = half(f).
 *
 * Parity pins: tests/test_oracle.py (exhaustive fp16 sweeps, brute force on
 * tiny shapes, closed forms and invariants); hand-computed worked examples
 * in tests/golden/.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NONFINITE 2
#define ORACLE_OVERFLOW 3

/* binary16 <-> binary32 through the compiler's _Float16 type: widening is
 * exact, narrowing rounds to nearest-even (IEEE 754 conversion). */
static float half_to_float(uint16_t bits) {
    _Float16 h;
    memcpy(&h, &bits, sizeof h);
    return (float)h;
}

static uint16_t float_to_half(float f) {
    _Float16 h = (_Float16)f;
    uint16_t bits;
    memcpy(&bits, &h, sizeof bits);
    return bits;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Symmetric quantization of each row of x [rows, K] (fp16 bits), one scale
 * per group of `group_size` consecutive elements along K (group_size 0: one
 * group per row).  [P1] pipeline steps 1-2; [P2] mode table.
 *   q: int8 [rows, K];  s: fp32 [rows, G] with G = K / group_size (or 1). */
int oracle_quant_rows(const uint16_t *x, long rows, long K, long group_size,
                      int qmax, int8_t *q, float *s) {
    if (!x || !q || !s || rows < 0 || K <= 0 || qmax <= 0 || qmax > 127)
        return ORACLE_BAD_ARG;
    long gs = group_size == 0 ? K : group_size;
    if (gs <= 0 || K % gs != 0) return ORACLE_BAD_ARG;
    long G = K / gs;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        for (long g = 0; g < G; ++g) {
            const uint16_t *xg = x + r * K + g * gs;
            int8_t *qg = q + r * K + g * gs;
            /* step 1: absmax of the group (exact in fp32) */
            float amax = 0.0f;
            for (long k = 0; k < gs; ++k) {
                float v = half_to_float(xg[k]);
                if (!isfinite(v)) {
                    status = ORACLE_NONFINITE;
                }
                float a = fabsf(v);
                if (a > amax) amax = a;
            }
            /* scale = absmax / qmax, one fp32 division */
            float scale = amax / (float)qmax;
            s[r * G + g] = amax == 0.0f ? 0.0f : scale;
            /* step 2: q = clamp(rint(x / scale), -qmax, qmax) */
            for (long k = 0; k < gs; ++k) {
                if (amax == 0.0f) {
                    qg[k] = 0;
                    continue;
                }
                float t = half_to_float(xg[k]) / scale;
                float rq = rintf(t);
                if (rq > (float)qmax) rq = (float)qmax;
                if (rq < (float)-qmax) rq = (float)-qmax;
                qg[k] = (int8_t)rq;
            }
        }
    }
    return status;
}

/* Two INT4 values per byte along K: byte j of row n holds q4[n, 2j] in the
 * low nibble and q4[n, 2j+1] in the high nibble, both two's complement.
 * [P2] mode table (W4A8: INT4 packed in uint8). */
int oracle_pack_int4(const int8_t *q4, long N, long K, uint8_t *packed) {
    if (!q4 || !packed || N < 0 || K <= 0 || K % 2 != 0) return ORACLE_BAD_ARG;
    for (long n = 0; n < N; ++n) {
        for (long j = 0; j < K / 2; ++j) {
            int lo = q4[n * K + 2 * j];
            int hi = q4[n * K + 2 * j + 1];
            if (lo < -8 || lo > 7 || hi < -8 || hi > 7) return ORACLE_BAD_ARG;
            packed[n * (K / 2) + j] = (uint8_t)((lo & 0xF) | ((hi & 0xF) << 4));
        }
    }
    return ORACLE_OK;
}

/* Inverse of oracle_pack_int4: sign-extend each nibble back to int8.
 * [P2] mode table (W4A8: unpack before the INT8 matmul). */
int oracle_unpack_int4(const uint8_t *packed, long N, long K, int8_t *q4) {
    if (!q4 || !packed || N < 0 || K <= 0 || K % 2 != 0) return ORACLE_BAD_ARG;
    for (long n = 0; n < N; ++n) {
        for (long j = 0; j < K / 2; ++j) {
            uint8_t b = packed[n * (K / 2) + j];
            int lo = b & 0xF;
            int hi = (b >> 4) & 0xF;
            q4[n * K + 2 * j] = (int8_t)(lo >= 8 ? lo - 16 : lo);
            q4[n * K + 2 * j + 1] = (int8_t)(hi >= 8 ? hi - 16 : hi);
        }
    }
    return ORACLE_OK;
}

/* Exact integer contraction, [P1] pipeline step 3: for every output (m, n)
 * and K-group g, acc[m, n, g] = sum over k in g of a[m, k] * w[n, k], summed
 * in int64 and checked to fit INT32.  a: [M, K], w: [N, K], both int8. */
int oracle_int_gemm(const int8_t *a, const int8_t *w, long M, long N, long K,
                    long group_size, int32_t *acc) {
    if (!a || !w || !acc || M < 0 || N < 0 || K <= 0) return ORACLE_BAD_ARG;
    long gs = group_size == 0 ? K : group_size;
    if (gs <= 0 || K % gs != 0) return ORACLE_BAD_ARG;
    long G = K / gs;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < M; ++m) {
        for (long n = 0; n < N; ++n) {
            for (long g = 0; g < G; ++g) {
                int64_t sum = 0;
                for (long k = g * gs; k < (g + 1) * gs; ++k)
                    sum += (int64_t)a[m * K + k] * (int64_t)w[n * K + k];
                if (sum > INT32_MAX || sum < INT32_MIN) status = ORACLE_OVERFLOW;
                acc[(m * N + n) * G + g] = (int32_t)sum;
            }
        }
    }
    return status;
}

/* Dequantization, [P1] pipeline step 4 and section "입도(Granularity)":
 *   f = 0;  for g = 0..G-1:  f = f + (float)acc[m,n,g] * (sa[m,g] * sw[n,g]);
 *   y[m, n] = half(f).
 * With G == 1 this is half((float)acc * (sa * sw)), the per-channel rule
 * (0 + v is exactly v). */
int oracle_dequant(const int32_t *acc, const float *sa, const float *sw, long M,
                   long N, long G, uint16_t *y) {
    if (!acc || !sa || !sw || !y || M < 0 || N < 0 || G <= 0) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (long m = 0; m < M; ++m) {
        for (long n = 0; n < N; ++n) {
            float f = 0.0f;
            for (long g = 0; g < G; ++g) {
                float scale = sa[m * G + g] * sw[n * G + g];
                float term = (float)acc[(m * N + n) * G + g] * scale;
                f = f + term;
            }
            y[m * N + n] = float_to_half(f);
        }
    }
    return ORACLE_OK;
}

/* The same contraction and dequant evaluated only at `count` chosen output
 * positions (rows[i], cols[i]); used to check full-size runs one output at a
 * time.  acc_out (optional) receives the per-group int32 partials [count, G]. */
int oracle_sampled_outputs(const int8_t *a, const float *sa, const int8_t *w,
                           const float *sw, long M, long N, long K,
                           long group_size, const long *rows, const long *cols,
                           long count, int32_t *acc_out, uint16_t *y_out) {
    if (!a || !sa || !w || !sw || !rows || !cols || !y_out || K <= 0)
        return ORACLE_BAD_ARG;
    long gs = group_size == 0 ? K : group_size;
    if (gs <= 0 || K % gs != 0) return ORACLE_BAD_ARG;
    long G = K / gs;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < count; ++i) {
        long m = rows[i], n = cols[i];
        if (m < 0 || m >= M || n < 0 || n >= N) {
            status = ORACLE_BAD_ARG;
            continue;
        }
        float f = 0.0f;
        for (long g = 0; g < G; ++g) {
            int64_t sum = 0;
            for (long k = g * gs; k < (g + 1) * gs; ++k)
                sum += (int64_t)a[m * K + k] * (int64_t)w[n * K + k];
            if (sum > INT32_MAX || sum < INT32_MIN) status = ORACLE_OVERFLOW;
            if (acc_out) acc_out[i * G + g] = (int32_t)sum;
            float scale = sa[m * G + g] * sw[n * G + g];
            float term = (float)(int32_t)sum * scale;
            f = f + term;
        }
        y_out[i] = float_to_half(f);
    }
    return status;
}

/* Weight-only product, the W8A16 / W4A16 baselines the method is measured
 * against: fp16 activations times the weights dequantized from their integer
 * codes, What[n, k] = q[n, k] * s_w[n, g(k)].  [P1] section on MLX's
 * weight-only quantization (the weights are dequantized to fp16 on the fly
 * and multiplied with fp16 activations); [P2] mode table (W8A16 / W4A16:
 * fp16 activations, MLX's GEMM) and the latency table's w8a16 / w4a16
 * columns.
 * Reading: the result is the real product y = x . What^T, rounded once to
 * fp16.  It is evaluated in double: every x * q product is exact, the group
 * sums carry a relative error below 2^-40 at K <= 32768, and the last step
 * rounds double -> fp16 directly.
 *   y[m, n] = half( sum over g of s_w[n, g] * (sum over k in g of x[m, k] * q[n, k]) )
 * x: fp16 bits [M, K]; q: int8 codes [N, K]; s_w: fp32 [N, G]; y: fp16 [M, N]. */
int oracle_weight_only(const uint16_t *x, const int8_t *q, const float *sw, long M,
                       long N, long K, long group_size, uint16_t *y) {
    if (!x || !q || !sw || !y || M < 0 || N < 0 || K <= 0) return ORACLE_BAD_ARG;
    long gs = group_size == 0 ? K : group_size;
    if (gs <= 0 || K % gs != 0) return ORACLE_BAD_ARG;
    long G = K / gs;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (long m = 0; m < M; ++m) {
        for (long n = 0; n < N; ++n) {
            double total = 0.0;
            for (long g = 0; g < G; ++g) {
                double part = 0.0;
                for (long k = g * gs; k < (g + 1) * gs; ++k) {
                    double xv = (double)half_to_float(x[m * K + k]);
                    if (!isfinite(xv)) status = ORACLE_NONFINITE;
                    part += xv * (double)q[n * K + k];
                }
                total += (double)sw[n * G + g] * part;
            }
            _Float16 h = (_Float16)total;
            memcpy(&y[m * N + n], &h, sizeof h);
        }
    }
    return status;
}
