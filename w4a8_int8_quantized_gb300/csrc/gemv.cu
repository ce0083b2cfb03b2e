// Decode-path matrix-vector kernels (M == 1): W8A8 per channel / per group,
// and W4A8 per channel.
//
// Method: "cider 소개", section "cider의 성능 측정 결과" (CiderLinear picks
// the INT8 MV kernel when seq_len == 1) and the kernel list in the same page
// (w8a8_int8_mv, pergroup_int8_mv); "Apple Silicon의 AI 한계치는 당신의
// 생각보다 높습니다", section "INT8 TensorOps 커널 설계", steps 3-4 (INT32
// accumulation, rescale by s_a * s_w).
//
// Design (HBM-bound: the weight matrix is streamed once): each CTA stages the
// quantized activation row in shared memory; each warp owns ROWS weight rows
// at a time and its lanes read consecutive 16-byte chunks of each row
// (coalesced 512-byte warp loads, non-allocating in L1), with UNROLL chunks
// per row in flight.  Products are summed exactly with dp4a into int32 and
// reduced across the warp with shuffles; the dequant is one fp32 scale
// product, one multiply and one fp16 rounding, as on the GEMM path.
#include "common.cuh"

namespace w8a8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 2;
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
  extern __shared__ uint4 xs[];
  const int nchunk = K >> 4;
  for (int i = threadIdx.x; i < nchunk; i += kThreads)
    xs[i] = __ldg(reinterpret_cast<const uint4 *>(xq) + i);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarps;
  const int G = gs == 0 ? 1 : K / gs;
  const int cpg = gs >> 4;  // 16-byte chunks per group (4 or 8)

  for (long n0 = static_cast<long>(warp) * kRows; n0 < N;
       n0 += static_cast<long>(nwarps) * kRows) {
    int acc[kRows];
    float f[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) { acc[r] = 0; f[r] = 0.f; }
    const uint4 *wrow[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      long n = n0 + r < N ? n0 + r : N - 1;  // clamp: duplicate row, not stored
      wrow[r] = reinterpret_cast<const uint4 *>(Wq + n * K);
    }
    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {
      uint4 w[kRows][kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
#pragma unroll
        for (int r = 0; r < kRows; ++r)
          w[r][u] = c < nchunk ? ld_stream(wrow[r] + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        const uint4 a = c < nchunk ? xs[c] : make_uint4(0, 0, 0, 0);
        if (gs == 0) {
#pragma unroll
          for (int r = 0; r < kRows; ++r) acc[r] = dot16(w[r][u], a, acc[r]);
        } else {
          // the cpg lanes of one group reduce their exact partial, then the
          // group's first lane rescales it
          const int g = (c < nchunk ? c : nchunk - 1) / cpg;
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            int p = dot16(w[r][u], a, 0);
            for (int o = cpg >> 1; o > 0; o >>= 1)
              p += __shfl_xor_sync(0xffffffffu, p, o);
            if ((lane & (cpg - 1)) == 0 && c < nchunk) {
              const long n = n0 + r < N ? n0 + r : N - 1;
              const float s = __fmul_rn(sa[g], sw[n * G + g]);
              f[r] = __fadd_rn(f[r], __fmul_rn(static_cast<float>(p), s));
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const long n = n0 + r;
      if (gs == 0) {
        const int tot = warp_sum(acc[r]);
        if (lane == 0 && n < N)
          y[n] = __float2half_rn(
              __fmul_rn(static_cast<float>(tot), __fmul_rn(sa[0], sw[n])));
      } else {
        const float tot = warp_sumf(f[r]);
        if (lane == 0 && n < N) y[n] = __float2half_rn(tot);
      }
    }
  }
}

// W4A8: weights packed two nibbles per byte along K (low nibble = even k).
// Shared memory holds the activations re-ordered per block of 8 elements as
// (a0 a2 a4 a6)(a1 a3 a5 a7), so that the even / odd nibbles of a 32-bit
// weight word meet their activations in one dp4a each.  A nibble v in
// [-8, 7] is read as the unsigned u = v + 8 (its top bit flipped), so
// sum_k a_k v_k = sum_k a_k u_k - 8 sum_k a_k, all exact in int32.
__global__ void __launch_bounds__(kThreads) gemv_w4a8_kernel(
    const int8_t *__restrict__ xq, const float *__restrict__ sa,
    const uint8_t *__restrict__ Wp, const float *__restrict__ sw, int N, int K,
    __half *__restrict__ y) {
  extern __shared__ uint4 xs[];
  __shared__ int s_sum;
  uint2 *xs2 = reinterpret_cast<uint2 *>(xs);
  if (threadIdx.x == 0) s_sum = 0;
  __syncthreads();
  int part = 0;
  for (int b = threadIdx.x; b < (K >> 3); b += kThreads) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(xq) + b);
    // bytes a0..a7 -> (a0 a2 a4 a6), (a1 a3 a5 a7)
    const uint32_t ev = __byte_perm(v.x, v.y, 0x6420);
    const uint32_t od = __byte_perm(v.x, v.y, 0x7531);
    xs2[b] = make_uint2(ev, od);
    part = __dp4a(static_cast<int>(v.x), 0x01010101, part);
    part = __dp4a(static_cast<int>(v.y), 0x01010101, part);
  }
  part = warp_sum(part);
  if ((threadIdx.x & 31) == 0) atomicAdd(&s_sum, part);
  __syncthreads();
  const int sum_a = s_sum;

  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarps;
  const int nchunk = K >> 5;  // 16-byte chunks of packed weights (32 k each)
  const int rowbytes = K >> 1;

  for (long n0 = static_cast<long>(warp) * kRows; n0 < N;
       n0 += static_cast<long>(nwarps) * kRows) {
    int acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[r] = 0;
    const uint4 *wrow[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      long n = n0 + r < N ? n0 + r : N - 1;
      wrow[r] = reinterpret_cast<const uint4 *>(Wp + n * rowbytes);
    }
    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {
      uint4 w[kRows][kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
#pragma unroll
        for (int r = 0; r < kRows; ++r)
          w[r][u] = c < nchunk ? ld_stream(wrow[r] + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c >= nchunk) continue;
        // chunk c covers k in [32c, 32c + 32): four 8-element blocks
        const uint4 a0 = xs[2 * c], a1 = xs[2 * c + 1];
        const uint32_t ae[4] = {a0.x, a0.z, a1.x, a1.z};
        const uint32_t ao[4] = {a0.y, a0.w, a1.y, a1.w};
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const uint32_t ww[4] = {w[r][u].x, w[r][u].y, w[r][u].z, w[r][u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t wx = ww[j] ^ 0x88888888u;
            acc[r] = dp4a_su(ae[j], wx & 0x0f0f0f0fu, acc[r]);
            acc[r] = dp4a_su(ao[j], (wx >> 4) & 0x0f0f0f0fu, acc[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const long n = n0 + r;
      const int tot = warp_sum(acc[r]) - 8 * sum_a;
      if (lane == 0 && n < N)
        y[n] = __float2half_rn(
            __fmul_rn(static_cast<float>(tot), __fmul_rn(sa[0], sw[n])));
    }
  }
}

int gemv_grid(int N) {
  const int per_block = kWarps * kRows;
  return (N + per_block - 1) / per_block;
}

}  // namespace

int launch_gemv_w8a8(const int8_t *xq, const float *sa, const int8_t *Wq,
                     const float *sw, int N, int K, int group_size, __half *y,
                     cudaStream_t s) {
  const size_t smem = static_cast<size_t>(K);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(gemv_w8a8_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return W8A8_ERR_CUDA;
  }
  gemv_w8a8_kernel<<<gemv_grid(N), kThreads, smem, s>>>(xq, sa, Wq, sw, N, K,
                                                        group_size, y);
  return launch_status();
}

int launch_gemv_w4a8(const int8_t *xq, const float *sa, const uint8_t *Wp,
                     const float *sw, int N, int K, __half *y, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(K);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(gemv_w4a8_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return W8A8_ERR_CUDA;
  }
  gemv_w4a8_kernel<<<gemv_grid(N), kThreads, smem, s>>>(xq, sa, Wp, sw, N, K,
                                                        y);
  return launch_status();
}

}  // namespace w8a8
