// INT8 x INT8 -> INT32 GEMM on the warp-level integer MMA
// (mma.sync m16n8k32 s8.s8.s32), with the dequant epilogue fused.
//
// Method: "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다", section
// "INT8 TensorOps 커널 설계", steps 3-4 (INT8 GEMM accumulating in INT32,
// rescale by s_a * s_w into fp16) and section "입도(Granularity)" (per-group
// scales need grouped dequantization during accumulation: the INT32
// accumulator is rescaled and cleared at every group boundary); "cider
// 소개", mode table (W4A8: INT4 weights unpacked before the INT8 matmul).
//
// sm_103a has no INT8 form of tcgen05.mma, so this warp-level MMA is the one
// exact INT8 tensor instruction on the chip.  Layout: CTA tile 128 x 128 x 64
// bytes, 8 warps in a 2 x 4 grid (64 x 32 each), a 4-stage cp.async ring of
// A / B tiles in shared memory with the 16-byte chunks of each 64-byte row
// XOR-swizzled so that ldmatrix reads are bank-conflict free.  W4A8 stages
// the packed weight tile and sign-extends its nibbles into the INT8 B tile
// in shared memory before the MMAs read it.
#include "common.cuh"

namespace w8a8 {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, P_BYTES = BN * BK / 2;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of 16-byte chunk c (0..3) of row r in a swizzled 64-byte-row tile
__device__ __forceinline__ int swz(int r, int c) {
  return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src,
                                           bool pred) {
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "r"(n));
}

__device__ __forceinline__ void cp_commit() {
  asm volatile("cp.async.commit_group;");
}

template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0,
                                        uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4],
                                       uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 8 two's-complement nibbles (element 2i in the low nibble of byte i) ->
// 8 sign-extended int8 in element order.
__device__ __forceinline__ uint2 unpack8(uint32_t w) {
  uint32_t lo = w & 0x0f0f0f0fu, hi = (w >> 4) & 0x0f0f0f0fu;
  lo |= (lo & 0x08080808u) * 0x1eu;
  hi |= (hi & 0x08080808u) * 0x1eu;
  return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

template <int WBITS>
__global__ void __launch_bounds__(THREADS) gemm_mma_kernel(
    const int8_t *__restrict__ A, const float *__restrict__ sa,
    const uint8_t *__restrict__ B, const float *__restrict__ sw, int M, int N,
    int K, int gs, __half *__restrict__ y, int32_t *__restrict__ acc_out) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sA = smem;                          // STAGES x A_BYTES
  uint8_t *sB = smem + STAGES * A_BYTES;       // STAGES x B_BYTES (W8)
  uint8_t *sP = sB;                            // STAGES x P_BYTES (W4)
  uint8_t *sBu = sB + STAGES * P_BYTES;        // one unpacked B tile (W4)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int warp_m = warp >> 2, warp_n = warp & 3;
  const long m0 = static_cast<long>(blockIdx.y) * BM;
  const long n0 = static_cast<long>(blockIdx.x) * BN;
  const int ktiles = (K + BK - 1) / BK;
  const int G = gs == 0 ? 1 : K / gs;
  const int tiles_per_group = gs == 0 ? ktiles : gs / BK;

  auto load_tile = [&](int kt, int slot) {
    const int k0 = kt * BK;
    // A: 128 rows x 4 chunks, two per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + i * THREADS;
      const int r = idx >> 2, c = idx & 3;
      const long gm = m0 + r;
      const int gk = k0 + c * 16;
      const bool p = gm < M && gk < K;
      const int8_t *src = A + (p ? gm * K + gk : 0);
      cp_async16(smem_u32(sA + slot * A_BYTES + swz(r, c)), src, p);
    }
    if (WBITS == 8) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int idx = tid + i * THREADS;
        const int r = idx >> 2, c = idx & 3;
        const long gn = n0 + r;
        const int gk = k0 + c * 16;
        const bool p = gn < N && gk < K;
        const uint8_t *src = B + (p ? gn * K + gk : 0);
        cp_async16(smem_u32(sB + slot * B_BYTES + swz(r, c)), src, p);
      }
    } else {
      // packed tile: 128 rows x 32 bytes, one 16-byte chunk per thread
      const int r = tid >> 1, c = tid & 1;
      const long gn = n0 + r;
      const int gk = k0 + c * 32;  // first k of the chunk
      const bool p = gn < N && gk < K;
      const uint8_t *src = B + (p ? gn * (K / 2) + gk / 2 : 0);
      cp_async16(smem_u32(sP + slot * P_BYTES + r * 32 + c * 16), src, p);
    }
  };

  int acc[4][4][4];
  float facc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) { acc[i][j][e] = 0; facc[i][j][e] = 0.f; }

  // output coordinates owned by this thread
  auto row_of = [&](int mi, int h) {
    return m0 + warp_m * 64 + mi * 16 + (lane >> 2) + h * 8;
  };
  auto col_of = [&](int ni, int e) {
    return n0 + warp_n * 32 + ni * 8 + (lane & 3) * 2 + e;
  };

  // per-group: rescale the exact int32 partial of group g and clear it
  auto fold_group = [&](int g) {
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long r = row_of(mi, h);
        const float sar = (acc_out == nullptr && r < M) ? sa[r * G + g] : 0.f;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const long c = col_of(ni, e);
            int &a = acc[mi][ni][h * 2 + e];
            if (acc_out != nullptr) {
              if (r < M && c < N) acc_out[(r * N + c) * G + g] = a;
            } else {
              const float swc = c < N ? sw[c * G + g] : 0.f;
              float &f = facc[mi][ni][h * 2 + e];
              f = __fadd_rn(f, __fmul_rn(static_cast<float>(a),
                                         __fmul_rn(sar, swc)));
            }
            a = 0;
          }
      }
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ktiles) load_tile(s, s);
    cp_commit();
  }

  for (int kt = 0; kt < ktiles; ++kt) {
    cp_wait<STAGES - 2>();
    __syncthreads();
    const int slot = kt % STAGES;
    const uint8_t *tB;
    if (WBITS == 4) {
      // sign-extend the staged nibbles into the INT8 tile: one 16-byte
      // packed chunk (32 k) per thread -> two swizzled 16-byte INT8 chunks
      const int r = tid >> 1, c = tid & 1;
      const uint4 pk =
          *reinterpret_cast<const uint4 *>(sP + slot * P_BYTES + r * 32 + c * 16);
      const uint2 u0 = unpack8(pk.x), u1 = unpack8(pk.y);
      const uint2 u2 = unpack8(pk.z), u3 = unpack8(pk.w);
      *reinterpret_cast<uint4 *>(sBu + swz(r, 2 * c)) =
          make_uint4(u0.x, u0.y, u1.x, u1.y);
      *reinterpret_cast<uint4 *>(sBu + swz(r, 2 * c + 1)) =
          make_uint4(u2.x, u2.y, u3.x, u3.y);
      __syncthreads();
      tB = sBu;
    } else {
      tB = sB + slot * B_BYTES;
    }
    // refill the slot that was consumed one iteration ago
    {
      const int nk = kt + STAGES - 1;
      if (nk < ktiles) load_tile(nk, nk % STAGES);
      cp_commit();
    }
    const uint8_t *tA = sA + slot * A_BYTES;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {  // two k32 steps per 64-byte tile
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int r = warp_m * 64 + mi * 16 + (lane & 15);
        const int c = kk * 2 + (lane >> 4);
        ldsm_x4(smem_u32(tA + swz(r, c)), af[mi][0], af[mi][1], af[mi][2],
                af[mi][3]);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int r = warp_n * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kk * 2 + ((lane >> 3) & 1);
        ldsm_x4(smem_u32(tB + swz(r, c)), bf[2 * np][0], bf[2 * np][1],
                bf[2 * np + 1][0], bf[2 * np + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_s8(acc[mi][ni], af[mi], bf[ni][0], bf[ni][1]);
    }
    if (gs != 0 && (kt + 1) % tiles_per_group == 0) fold_group(kt / tiles_per_group);
  }
  cp_wait<0>();

  if (gs == 0 && acc_out != nullptr) {
    fold_group(0);
    return;
  }
  if (acc_out != nullptr) return;

  // epilogue: per channel y = fp16(float(acc) * (sa * sw)); per group the
  // fp32 sum of the rescaled partials
  const bool even_n = (N & 1) == 0;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long r = row_of(mi, h);
      if (r >= M) continue;
      const float sar = gs == 0 ? sa[r] : 0.f;
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const long c = col_of(ni, e);
          if (gs == 0) {
            const float swc = c < N ? sw[c] : 0.f;
            v[e] = __fmul_rn(static_cast<float>(acc[mi][ni][h * 2 + e]),
                             __fmul_rn(sar, swc));
          } else {
            v[e] = facc[mi][ni][h * 2 + e];
          }
        }
        const long c0 = col_of(ni, 0);
        if (even_n && c0 + 1 < N) {
          *reinterpret_cast<__half2 *>(y + r * N + c0) =
              __halves2half2(__float2half_rn(v[0]), __float2half_rn(v[1]));
        } else {
          if (c0 < N) y[r * N + c0] = __float2half_rn(v[0]);
          if (c0 + 1 < N) y[r * N + c0 + 1] = __float2half_rn(v[1]);
        }
      }
    }
}

template <int WBITS>
int launch_t(const int8_t *xq, const float *sa, const void *W, const float *sw,
             int M, int N, int K, int gs, __half *y, int32_t *acc_out,
             cudaStream_t s) {
  const size_t smem = WBITS == 8
                          ? STAGES * (A_BYTES + B_BYTES)
                          : STAGES * (A_BYTES + P_BYTES) + B_BYTES;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_mma_kernel<WBITS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return W8A8_ERR_CUDA;
    attr_set[dev] = true;
  }
  dim3 grid(ceil_div(N, BN), ceil_div(M, BM));
  if (grid.y > 65535) return W8A8_ERR_INVALID_ARG;
  gemm_mma_kernel<WBITS><<<grid, THREADS, smem, s>>>(
      xq, sa, static_cast<const uint8_t *>(W), sw, M, N, K, gs, y, acc_out);
  return launch_status();
}

}  // namespace

int launch_gemm_mma(const int8_t *xq, const float *sa, const void *W,
                    const float *sw, int M, int N, int K, int group_size,
                    int wbits, __half *y, int32_t *acc_out, cudaStream_t s) {
  if (wbits == 4)
    return launch_t<4>(xq, sa, W, sw, M, N, K, group_size, y, acc_out, s);
  return launch_t<8>(xq, sa, W, sw, M, N, K, group_size, y, acc_out, s);
}

}  // namespace w8a8
