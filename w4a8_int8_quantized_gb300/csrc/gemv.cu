// Decode-path matrix-vector kernels (M == 1): W8A8 per channel / per group,
// and W4A8 per channel; optionally fused with the activation quantization.
//
// Method: "cider 소개", section "cider의 성능 측정 결과" (CiderLinear picks
// the INT8 MV kernel when seq_len == 1) and the kernel list in the same page
// (w8a8_int8_mv, pergroup_int8_mv); "Apple Silicon의 AI 한계치는 당신의
// 생각보다 높습니다", section "INT8 TensorOps 커널 설계", steps 1-4.
//
// Design (HBM-bound: the weight matrix is streamed once).  One persistent CTA
// per SM owns a contiguous range of weight rows, which is one contiguous
// range of bytes, and streams it through a 4-stage shared-memory ring with
// bulk asynchronous copies (cp.async.bulk, 32 KB stages holding whole rows),
// so each SM keeps up to 128 KB of weights in flight without spending
// registers on it.  The quantized activation row sits in shared memory: the
// fused kernel quantizes the fp16 row itself (every CTA redundantly; the row
// is a few KB from L2) with the same rule as the row quantizer, the plain
// kernel copies the INT8 codes.  Each warp takes whole rows of a stage: lane
// l reads 16-byte chunks l, l + 32, ... (conflict-free), dp4a sums exactly in
// int32, a shuffle reduction finishes the row, and the dequant is one fp32
// scale product, one multiply and one fp16 rounding, as on the GEMM path.
// Waits on the ring are bounded; a wait that gives up records a code in the
// device error word and the CTA returns after its copies land.
#include "common.cuh"
#include "quant_rule.cuh"

namespace w8a8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
#ifndef W8A8_MV_STAGES
constexpr int kStages = 4;
#else
constexpr int kStages = W8A8_MV_STAGES;
#endif
#ifndef W8A8_MV_STAGE_KB
constexpr int kStageBytes = 32 * 1024;
#else
constexpr int kStageBytes = W8A8_MV_STAGE_KB * 1024;
#endif
constexpr long long kTimeoutCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) return false;
  }
  return true;
}

// bulk copy of `bytes` contiguous bytes global -> shared, completing on `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ int dot16(const uint4 &w, const uint4 &a, int acc) {
  acc = __dp4a(static_cast<int>(w.x), static_cast<int>(a.x), acc);
  acc = __dp4a(static_cast<int>(w.y), static_cast<int>(a.y), acc);
  acc = __dp4a(static_cast<int>(w.z), static_cast<int>(a.z), acc);
  acc = __dp4a(static_cast<int>(w.w), static_cast<int>(a.w), acc);
  return acc;
}

// signed a (4 x s8) . unsigned b (4 x u8) + c
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// W4A8 chunk: 16 packed bytes = 32 consecutive k (element 2i in the low
// nibble of byte i) against the 32 INT8 activations a[0..7] (4 per word).
// A nibble v in [-8, 7] is read as the unsigned u = v + 8 (top bit flipped):
// sum_k a_k v_k = sum_k a_k u_k - 8 sum_k a_k, all exact in int32; the even
// nibbles of a word meet (a0 a2 a4 a6), the odd ones (a1 a3 a5 a7).
__device__ __forceinline__ void dot32_w4(const uint4 &w, const uint32_t (&a)[8], int &acc,
                                         int &asum) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t ev = __byte_perm(a[2 * j], a[2 * j + 1], 0x6420);
    const uint32_t od = __byte_perm(a[2 * j], a[2 * j + 1], 0x7531);
    const uint32_t wx = ww[j] ^ 0x88888888u;
    acc = dp4a_su(ev, wx & 0x0f0f0f0fu, acc);
    acc = dp4a_su(od, (wx >> 4) & 0x0f0f0f0fu, acc);
    asum = __dp4a(static_cast<int>(a[2 * j]), 0x01010101, asum);
    asum = __dp4a(static_cast<int>(a[2 * j + 1]), 0x01010101, asum);
  }
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Shared memory: [barriers (2 x kStages x 8 bytes, padded to 256)][kStages x
// kStageBytes ring][K codes][G scales].  Every region starts aligned: the
// barriers at 0 (mbarriers need 8 bytes), the ring and the codes at multiples
// of 16 (bulk copies and 16-byte loads; K % 16 == 0), the scales at 4.
constexpr int kBarBytes = 256;
inline size_t mv_smem_bytes(int K, int G) {
  return kBarBytes + static_cast<size_t>(kStages) * kStageBytes + K + 4 * G;
}

// FUSED: xin is fp16 x [K] and the CTA quantizes it (scales in shared
// memory); otherwise xin is int8 codes [K] with scales sa_in [G].
// y[n] = fp16(float(sum_k q_k w_nk) * (s_a * s_w[n]))            (gs == 0)
// y[n] = fp16(sum_g float(acc_g) * (s_a[g] * s_w[n, g]))          (gs > 0)
template <int WBITS, bool PERGROUP, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) mv_kernel(
    const void *__restrict__ xin, const float *__restrict__ sa_in,
    const uint8_t *__restrict__ W, const float *__restrict__ sw, int N, int K, int gs,
    __half *__restrict__ y, unsigned int *err) {
  extern __shared__ __align__(128) uint8_t smem[];
  static_assert(2 * kStages * 8 <= kBarBytes, "barrier block");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = PERGROUP ? K / gs : 1;
  uint8_t *ring = smem + kBarBytes;
  int8_t *xs = reinterpret_cast<int8_t *>(ring + kStages * kStageBytes);
  float *ss = reinterpret_cast<float *>(ring + kStages * kStageBytes + K);
  const uint32_t bar0 = smem_u32(smem);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };

  const int row_bytes = WBITS == 8 ? K : K / 2;
  const int rps = kStageBytes / row_bytes;  // whole rows per stage (>= 1: K <= 32768)
  const long r0 = static_cast<long>(blockIdx.x) * N / gridDim.x;
  const long r1 = static_cast<long>(blockIdx.x + 1) * N / gridDim.x;
  const int nst = static_cast<int>((r1 - r0 + rps - 1) / rps);

  int issued = 0;  // stages whose copy thread 0 has started
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full(s)));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty(s)), "r"(kWarps));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // start streaming before the activation row is ready
    for (int st = 0; st < nst && st < kStages; ++st) {
      issued = st + 1;
      const long rr = r0 + static_cast<long>(st) * rps;
      const long cnt = r1 - rr < rps ? r1 - rr : rps;
      bulk_load(smem_u32(ring + st * kStageBytes), W + rr * row_bytes,
                static_cast<uint32_t>(cnt * row_bytes), full(st));
    }
  }

  // ---- the activation row: INT8 codes (and scales) into shared memory ----
  if (FUSED) {
    const uint4 *xv = static_cast<const uint4 *>(xin);
    const int nvec = K >> 3;
    __shared__ float red[kWarps];
    float amax_row = 0.f;
    if (!PERGROUP) {
      for (int v = tid; v < nvec; v += kThreads) amax_row = fmaxf(amax_row, absmax8(__ldg(xv + v)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        amax_row = fmaxf(amax_row, __shfl_xor_sync(0xffffffffu, amax_row, o));
      if (lane == 0) red[warp] = amax_row;
      __syncthreads();
      amax_row = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) amax_row = fmaxf(amax_row, red[w]);
    }
    const float s_row = __fdiv_rn(amax_row, 127.f);
    const float rcp_row = amax_row == 0.f ? 0.f : __frcp_rn(s_row);
    if (!PERGROUP && tid == 0) ss[0] = s_row;
    // a group of gs is gs / 8 consecutive vectors, i.e. consecutive lanes
    for (int v0 = 0; v0 < nvec; v0 += kThreads) {
      const int v = v0 + tid;
      const uint4 xvv = v < nvec ? __ldg(xv + v) : make_uint4(0, 0, 0, 0);
      float s = s_row, rcp = rcp_row;
      if (PERGROUP) {
        float m = absmax8(xvv);
        for (int o = (gs >> 4); o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        s = __fdiv_rn(m, 127.f);
        rcp = m == 0.f ? 0.f : __frcp_rn(s);
        if (v < nvec && (tid & ((gs >> 3) - 1)) == 0) ss[(v << 3) / gs] = s;
      }
      if (v < nvec) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&xvv);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(h[j]);
          const uint32_t b = (static_cast<uint32_t>(quant1(f.x, s, rcp, 127)) & 0xffu) |
                             ((static_cast<uint32_t>(quant1(f.y, s, rcp, 127)) & 0xffu) << 8);
          if (j < 2)
            lo |= b << (16 * j);
          else
            hi |= b << (16 * (j - 2));
        }
        reinterpret_cast<uint2 *>(xs)[v] = make_uint2(lo, hi);
      }
    }
  } else {
    const uint4 *xv = static_cast<const uint4 *>(xin);
    for (int v = tid; v < (K >> 4); v += kThreads) reinterpret_cast<uint4 *>(xs)[v] = __ldg(xv + v);
    for (int g = tid; g < G; g += kThreads) ss[g] = __ldg(sa_in + g);
  }
  __syncthreads();

  // ---- stream the rows ----
  const int nchunk = row_bytes >> 4;  // 16-byte weight chunks per row
  const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
  bool ok = true;
  for (int st = 0; st < nst && ok; ++st) {
    const int s = st % kStages;
    const uint32_t par = (st / kStages) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(full(s), par))) {
      if (lane == 0) atomicCAS(err, 0u, static_cast<unsigned>(kDevErrFullBarrier));
      ok = false;
      break;
    }
    const long rr = r0 + static_cast<long>(st) * rps;
    const int cnt = static_cast<int>(r1 - rr < rps ? r1 - rr : rps);
    const uint8_t *stage = ring + s * kStageBytes;
    for (int i = warp; i < cnt; i += kWarps) {
      const uint4 *wrow = reinterpret_cast<const uint4 *>(stage + i * row_bytes);
      const long n = rr + i;
      int acc = 0, asum = 0;
      float f = 0.f;
      // every lane runs the same trip count (the group shuffles need all 32)
      for (int c0 = 0; c0 < nchunk; c0 += 32) {
        const int c = c0 + lane;
        const bool in = c < nchunk;
        const uint4 w = in ? wrow[c] : make_uint4(0, 0, 0, 0);
        if (WBITS == 8) {
          const uint4 a = in ? xs4[c] : make_uint4(0, 0, 0, 0);
          if (!PERGROUP) {
            acc = dot16(w, a, acc);
          } else {
            // the cpg lanes of one group reduce their exact partial; the
            // group's first lane rescales it
            const int cpg = gs >> 4;
            int pp = dot16(w, a, 0);
            for (int o = cpg >> 1; o > 0; o >>= 1) pp += __shfl_xor_sync(0xffffffffu, pp, o);
            if (in && (lane & (cpg - 1)) == 0) {
              const int g = c / cpg;
              const float sc = __fmul_rn(ss[g], __ldg(sw + n * G + g));
              f = __fadd_rn(f, __fmul_rn(static_cast<float>(pp), sc));
            }
          }
        } else if (in) {
          const uint4 a0 = xs4[2 * c], a1 = xs4[2 * c + 1];
          const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          dot32_w4(w, av, acc, asum);
        }
      }
      if (!PERGROUP) {
        const int tot = warp_sum(acc) - (WBITS == 4 ? 8 * warp_sum(asum) : 0);
        if (lane == 0)
          y[n] = __float2half_rn(
              __fmul_rn(static_cast<float>(tot), __fmul_rn(ss[0], __ldg(sw + n))));
      } else {
        const float tot = warp_sumf(f);
        if (lane == 0) y[n] = __float2half_rn(tot);
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty(s)) : "memory");
    // refill this stage once every warp is done with it
    if (tid == 0 && st + kStages < nst) {
      if (!mbar_wait(empty(s), par)) {
        atomicCAS(err, 0u, static_cast<unsigned>(kDevErrEmptyBarrier));
        ok = false;
      } else {
        const long rn = r0 + static_cast<long>(st + kStages) * rps;
        const long cn = r1 - rn < rps ? r1 - rn : rps;
        bulk_load(smem_u32(ring + s * kStageBytes), W + rn * row_bytes,
                  static_cast<uint32_t>(cn * row_bytes), full(s));
        issued = st + kStages + 1;
      }
    }
  }
  // the copies this CTA started must land before it exits (normally they
  // have all been consumed already)
  if (tid == 0) {
    for (int st = issued - kStages > 0 ? issued - kStages : 0; st < issued; ++st)
      mbar_wait(full(st % kStages), (st / kStages) & 1u);
  }
}

template <int WBITS, bool PERGROUP, bool FUSED>
int launch_mv(const void *xin, const float *sa, const void *W, const float *sw, int N, int K,
              int gs, __half *y, cudaStream_t s) {
  static bool attr_set[64] = {};
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return W8A8_ERR_CUDA;
  const int G = PERGROUP ? K / gs : 1;
  const size_t smem = mv_smem_bytes(K, G);
  if (!attr_set[dev]) {
    // the largest plan (K = 32768, group size 64) sets the attribute once
    if (cudaFuncSetAttribute(mv_kernel<WBITS, PERGROUP, FUSED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(mv_smem_bytes(kMaxK, kMaxK / 64))) != cudaSuccess)
      return W8A8_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return W8A8_ERR_CUDA;
    attr_set[dev] = true;
  }
  unsigned int *err = device_error_word();
  if (err == nullptr) return W8A8_ERR_CUDA;
  const int grid = N < sms[dev] ? N : sms[dev];
  mv_kernel<WBITS, PERGROUP, FUSED><<<grid, kThreads, smem, s>>>(
      xin, sa, static_cast<const uint8_t *>(W), sw, N, K, gs, y, err);
  return launch_status();
}

}  // namespace

int launch_gemv_w8a8(const int8_t *xq, const float *sa, const int8_t *Wq,
                     const float *sw, int N, int K, int group_size, __half *y,
                     cudaStream_t s) {
  if (group_size != 0) return launch_mv<8, true, false>(xq, sa, Wq, sw, N, K, group_size, y, s);
  return launch_mv<8, false, false>(xq, sa, Wq, sw, N, K, 0, y, s);
}

int launch_gemv_w4a8(const int8_t *xq, const float *sa, const uint8_t *Wp,
                     const float *sw, int N, int K, __half *y, cudaStream_t s) {
  return launch_mv<4, false, false>(xq, sa, Wp, sw, N, K, 0, y, s);
}

int launch_linear_mv(const __half *x, const void *W, const float *sw, int N, int K,
                     int group_size, int wbits, __half *y, cudaStream_t s) {
  if (wbits == 4) return launch_mv<4, false, true>(x, nullptr, W, sw, N, K, 0, y, s);
  if (group_size != 0) return launch_mv<8, true, true>(x, nullptr, W, sw, N, K, group_size, y, s);
  return launch_mv<8, false, true>(x, nullptr, W, sw, N, K, 0, y, s);
}

}  // namespace w8a8
