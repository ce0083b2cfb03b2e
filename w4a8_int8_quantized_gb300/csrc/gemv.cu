// Decode-path matrix-vector kernels (M == 1): W8A8 per channel / per group,
// and W4A8 per channel.
//
// Method: "cider 소개", section "cider의 성능 측정 결과" (CiderLinear picks
// the INT8 MV kernel when seq_len == 1) and the kernel list in the same page
// (w8a8_int8_mv, pergroup_int8_mv); "Apple Silicon의 AI 한계치는 당신의
// 생각보다 높습니다", section "INT8 TensorOps 커널 설계", steps 3-4 (INT32
// accumulation, rescale by s_a * s_w).
//
// Design (HBM-bound: the weight matrix is streamed once): one warp per
// weight row.  Lane l reads 16-byte chunks l, l + 32, ... of the row, so
// every warp load is a coalesced 512-byte transaction, and issues up to
// kUnroll of them before the first use (the whole row for K <= 4096) to keep
// enough bytes in flight; weight loads bypass L1 allocation.  The quantized
// activation row is read through the read-only cache (every warp of the
// grid reads the same K bytes).  Products are summed exactly in int32 with
// dp4a and reduced across the warp with shuffles; the dequant is one fp32
// scale product, one multiply and one fp16 rounding, as on the GEMM path.
// Few registers per thread keep many warps resident per SM.
#include "common.cuh"

namespace w8a8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

// y[n] = fp16(float(sum_k xq[k] Wq[n,k]) * (sa * sw[n]))            (gs == 0)
// y[n] = fp16(sum_g float(acc_g) * (sa[g] * sw[n,g]))                (gs > 0)
__global__ void __launch_bounds__(kThreads) gemv_w8a8_kernel(
    const int8_t *__restrict__ xq, const float *__restrict__ sa,
    const int8_t *__restrict__ Wq, const float *__restrict__ sw, int N, int K,
    int gs, __half *__restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int nchunk = K >> 4;
  const int G = gs == 0 ? 1 : K / gs;
  const int cpg = gs >> 4;  // 16-byte chunks per group (4 or 8)
  const uint4 *xv = reinterpret_cast<const uint4 *>(xq);
  for (long n = static_cast<long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); n < N;
       n += static_cast<long>(gridDim.x) * kWarps) {
    const uint4 *wrow = reinterpret_cast<const uint4 *>(Wq + n * K);
    int acc = 0;
    float f = 0.f;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        w[u] = c < nchunk ? ld_stream(wrow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        const uint4 a = c < nchunk ? __ldg(xv + c) : make_uint4(0, 0, 0, 0);
        if (gs == 0) {
          acc = dot16(w[u], a, acc);
        } else {
          // the cpg lanes of one group reduce their exact partial, then the
          // group's first lane rescales it
          int p = dot16(w[u], a, 0);
          for (int o = cpg >> 1; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
          if ((lane & (cpg - 1)) == 0 && c < nchunk) {
            const int g = c / cpg;
            const float s = __fmul_rn(__ldg(sa + g), __ldg(sw + n * G + g));
            f = __fadd_rn(f, __fmul_rn(static_cast<float>(p), s));
          }
        }
      }
    }
    if (gs == 0) {
      const int tot = warp_sum(acc);
      if (lane == 0)
        y[n] = __float2half_rn(
            __fmul_rn(static_cast<float>(tot), __fmul_rn(__ldg(sa), __ldg(sw + n))));
    } else {
      const float tot = warp_sumf(f);
      if (lane == 0) y[n] = __float2half_rn(tot);
    }
  }
}

// W4A8: weights packed two nibbles per byte along K (low nibble = even k).
// A packed 32-bit word holds 8 consecutive k; its even nibbles meet the
// activations (a0 a2 a4 a6) and its odd nibbles (a1 a3 a5 a7) in one dp4a
// each.  A nibble v in [-8, 7] is read as the unsigned u = v + 8 (its top
// bit flipped), so sum_k a_k v_k = sum_k a_k u_k - 8 sum_k a_k, all exact in
// int32.
__global__ void __launch_bounds__(kThreads) gemv_w4a8_kernel(
    const int8_t *__restrict__ xq, const float *__restrict__ sa,
    const uint8_t *__restrict__ Wp, const float *__restrict__ sw, int N, int K,
    __half *__restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int nchunk = K >> 5;  // 16-byte chunks of packed weights (32 k each)
  const int rowbytes = K >> 1;
  const uint4 *xv = reinterpret_cast<const uint4 *>(xq);
  for (long n = static_cast<long>(blockIdx.x) * kWarps + (threadIdx.x >> 5); n < N;
       n += static_cast<long>(gridDim.x) * kWarps) {
    const uint4 *wrow = reinterpret_cast<const uint4 *>(Wp + n * rowbytes);
    int acc = 0, asum = 0;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        w[u] = c < nchunk ? ld_stream(wrow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c >= nchunk) continue;
        // chunk c covers k in [32c, 32c + 32): activations 32c .. 32c + 31
        const uint4 a0 = __ldg(xv + 2 * c), a1 = __ldg(xv + 2 * c + 1);
        const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // activations of k = 8j .. 8j + 7 of the chunk: even and odd lanes
          const uint32_t ev = __byte_perm(av[2 * j], av[2 * j + 1], 0x6420);
          const uint32_t od = __byte_perm(av[2 * j], av[2 * j + 1], 0x7531);
          const uint32_t wx = ww[j] ^ 0x88888888u;
          acc = dp4a_su(ev, wx & 0x0f0f0f0fu, acc);
          acc = dp4a_su(od, (wx >> 4) & 0x0f0f0f0fu, acc);
          asum = __dp4a(static_cast<int>(av[2 * j]), 0x01010101, asum);
          asum = __dp4a(static_cast<int>(av[2 * j + 1]), 0x01010101, asum);
        }
      }
    }
    const int tot = warp_sum(acc) - 8 * warp_sum(asum);
    if (lane == 0)
      y[n] = __float2half_rn(
          __fmul_rn(static_cast<float>(tot), __fmul_rn(__ldg(sa), __ldg(sw + n))));
  }
}

int gemv_grid(int N) { return (N + kWarps - 1) / kWarps; }

}  // namespace

int launch_gemv_w8a8(const int8_t *xq, const float *sa, const int8_t *Wq,
                     const float *sw, int N, int K, int group_size, __half *y,
                     cudaStream_t s) {
  gemv_w8a8_kernel<<<gemv_grid(N), kThreads, 0, s>>>(xq, sa, Wq, sw, N, K, group_size, y);
  return launch_status();
}

int launch_gemv_w4a8(const int8_t *xq, const float *sa, const uint8_t *Wp,
                     const float *sw, int N, int K, __half *y, cudaStream_t s) {
  gemv_w4a8_kernel<<<gemv_grid(N), kThreads, 0, s>>>(xq, sa, Wp, sw, N, K, y);
  return launch_status();
}

}  // namespace w8a8
