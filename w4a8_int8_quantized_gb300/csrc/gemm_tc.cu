// W8A8 / W4A8 GEMM on the 5th-generation tensor cores (tcgen05), exact.
//
// Method: "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다", section
// "INT8 TensorOps 커널 설계", steps 3-4 (INT8 x INT8 GEMM accumulating in
// INT32, then a rescale by s_a * s_w into fp16) and section
// "입도(Granularity)" (per-group scales: each group's partial sum is
// rescaled during accumulation); "cider 소개", mode table (W4A8: INT4
// weights unpacked before the INT8 matmul).
//
// sm_103a has no integer form of tcgen05.mma, so the contraction runs on
// kind::f16 and is kept exact by construction:
//   * every INT8 code (|q| <= 127) and INT4 code (|q| <= 7) is an fp16 value
//     exactly, and every product (|p| <= 16129 < 2^14) is exact in fp32;
//   * the fp32 accumulator in tensor memory (TMEM) holds an integer exactly
//     while every partial sum stays below 2^24 in magnitude.  A K-chunk of
//     1024 bounds it by 1024 * 127^2 = 16,516,096 < 2^24 (W4A8: a chunk of
//     16384 gives 16384 * 127 * 7 < 2^24), so the accumulator is drained at
//     least every chunk: the epilogue converts it to int32 (exact) and adds
//     it to an int32 running sum in registers.  Per-group scales drain at
//     every group (64 or 128 of K) and rescale each exact partial in fp32.
//
// Kernel layout (persistent, one CTA of 16 warps per SM, 128 x 256 output
// tiles, 64-deep K blocks):
//   warp 0      TMA producer: INT8 (or packed INT4) A / B tiles into a
//               4-stage staging ring in shared memory;
//   warp 1      allocates TMEM and issues the MMAs (one thread): four
//               128x256x16 tcgen05.mma per K block into one of two TMEM
//               accumulators (ping-pong per chunk);
//   warps 2-7   converters: INT8 / INT4 codes -> fp16, written in the
//               128-byte-swizzled K-major layout the MMA reads (2 stages);
//   warps 8-15  epilogue: drain TMEM (tcgen05.ld), exact int32 sums or fp32
//               per-group rescale, then the fp16 output.
// Stages hand over through mbarriers; every wait is bounded, and a wait that
// gives up records a code in the device error word, raises an abort flag
// seen by every role, lets in-flight copies and MMAs land, frees TMEM and
// returns.
#include <cuda.h>

#include "common.cuh"

namespace w8a8 {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int S8 = 4, S16 = 2;
constexpr int NUM_THREADS = 512;
constexpr int CONV_WARPS = 6, EPI_WARPS = 8;
constexpr int A8_BYTES = BM * BK;        // INT8 A stage
constexpr int B8_BYTES = BN * BK;        // INT8 B stage (packed INT4 uses half)
constexpr int A16_BYTES = BM * BK * 2;   // fp16 A stage, 128-byte rows
constexpr int B16_BYTES = BN * BK * 2;   // fp16 B stage
constexpr int OFF_A8 = 0;
constexpr int OFF_B8 = OFF_A8 + S8 * A8_BYTES;
constexpr int OFF_A16 = OFF_B8 + S8 * B8_BYTES;
constexpr int OFF_B16 = OFF_A16 + S16 * A16_BYTES;
constexpr int OFF_BAR = OFF_B16 + S16 * B16_BYTES;
constexpr int NUM_BARS = 2 * S8 + 2 * S16 + 2 + 2 + 1;
constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16 + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr long long kTimeoutCycles = 4000000000LL;  // about 2 s at 2 GHz

// instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// N = 256, M = 128
constexpr uint32_t IDESC = (1u << 4) | (0u << 7) | (0u << 10) |
                           (static_cast<uint32_t>(BN >> 3) << 17) |
                           (static_cast<uint32_t>(BM >> 4) << 24);

struct TcParams {
  int M, N, K, gs, G, nkb, chunk_kb, mblocks, ntiles;
  const float *sa;
  const float *sw;
  __half *y;
  int32_t *acc_out;
  unsigned int *err;
};

// ---------------------------------------------------------------- PTX ----

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map,
                                            uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accum));
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (rows are 128 bytes), descriptor version 1
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3ffff) >> 4);      // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                    // version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
        "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
        "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// Ordered global accesses for the epilogue: as volatile asm they keep their
// program order, so a fully unrolled loop does not hoist all of its loads
// ahead of its stores (which would need one register per load).
__device__ __forceinline__ float ldg_f32(const float *ptr) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
  return v;
}

__device__ __forceinline__ void stg_v4(void *ptr, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void stg_b16(void *ptr, __half v) {
  asm volatile("st.global.b16 [%0], %1;" ::"l"(ptr), "h"(__half_as_ushort(v)) : "memory");
}

__device__ __forceinline__ void stg_b32(void *ptr, int v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait.  Returns false if the CTA is aborting or the wait gave up
// (then it records `code` and raises the abort flag).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity,
                                         volatile int *abort_flag, unsigned int code,
                                         unsigned int *err) {
#pragma unroll 1
  for (int i = 0; i < 32; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kTimeoutCycles) {
      if (err != nullptr) atomicCAS(err, 0u, code);
      *abort_flag = 1;
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag (teardown: let own work land).
__device__ __forceinline__ void wait_bar_teardown(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) return;
  }
}

// 4 INT8 (one 32-bit word) -> 4 fp16, exactly: bytes b become halves with
// bits 0x64 | (b ^ 0x80), i.e. 1024 + b + 128, then 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_h(uint32_t w, uint32_t &h01, uint32_t &h23) {
  const uint32_t x = w ^ 0x80808080u;
  h01 = __byte_perm(x, 0x64646464u, 0x5140);
  h23 = __byte_perm(x, 0x64646464u, 0x7362);
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
  __half2 a = __hsub2(*reinterpret_cast<__half2 *>(&h01), bias);
  __half2 b = __hsub2(*reinterpret_cast<__half2 *>(&h23), bias);
  h01 = *reinterpret_cast<uint32_t *>(&a);
  h23 = *reinterpret_cast<uint32_t *>(&b);
}

// 8 two's-complement nibbles (element 2i in the low nibble of byte i) -> 8
// fp16 in element order: a nibble v becomes 1024 + (v + 8), minus 1032.
__device__ __forceinline__ uint4 i4x8_to_h(uint32_t w) {
  const uint32_t x = w ^ 0x88888888u;
  const uint32_t lo = x & 0x0f0f0f0fu, hi = (x >> 4) & 0x0f0f0f0fu;
  const uint32_t p0 = __byte_perm(lo, hi, 0x5140);  // u0 u1 u2 u3
  const uint32_t p1 = __byte_perm(lo, hi, 0x7362);  // u4 u5 u6 u7
  uint32_t h[4] = {__byte_perm(p0, 0x64646464u, 0x5140), __byte_perm(p0, 0x64646464u, 0x7362),
                   __byte_perm(p1, 0x64646464u, 0x5140), __byte_perm(p1, 0x64646464u, 0x7362)};
  const __half2 bias = __half2half2(__ushort_as_half(0x6408));  // 1032
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 t = __hsub2(*reinterpret_cast<__half2 *>(&h[i]), bias);
    h[i] = *reinterpret_cast<uint32_t *>(&t);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// byte offset of 16-byte chunk j of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128_off(int r, int j) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

// ------------------------------------------------------------- kernel ----

template <int WBITS, bool PERGROUP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = base + OFF_BAR;
  auto full8 = [&](int s) { return bar0 + 8u * s; };
  auto empty8 = [&](int s) { return bar0 + 8u * (S8 + s); };
  auto full16 = [&](int s) { return bar0 + 8u * (2 * S8 + s); };
  auto empty16 = [&](int s) { return bar0 + 8u * (2 * S8 + S16 + s); };
  auto accfull = [&](int r) { return bar0 + 8u * (2 * S8 + 2 * S16 + r); };
  auto accempty = [&](int r) { return bar0 + 8u * (2 * S8 + 2 * S16 + 2 + r); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S8 + 2 * S16 + 4);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S8; ++s) {
      mbar_init(full8(s), 1);
      mbar_init(empty8(s), CONV_WARPS);
    }
    for (int s = 0; s < S16; ++s) {
      mbar_init(full16(s), CONV_WARPS);
      mbar_init(empty16(s), 1);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(accfull(r), 1);
      mbar_init(accempty(r), EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int nkb = p.nkb, chunk_kb = p.chunk_kb;

  // Register split per warpgroup (launch: 512 threads x 128 registers):
  // warpgroups 2-3 (epilogue) rise to 184, warpgroups 0-1 (producer, MMA,
  // converters) drop to 72; 256 * 184 + 256 * 72 = 65536 = 512 * 128.  Each
  // side's code sits inside the branch of its own setmaxnreg, so the compiler
  // allocates registers to that limit.
  if (warp >= 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    // ------------------------------------------------------ epilogue ----
    const int q = warp & 3;             // TMEM lane quadrant of this warp
    const int half = (warp - 8) >> 2;   // which 128 of the 256 columns
    const int row = q * 32 + lane;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t cc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
      const int mb = tile % p.mblocks, nb = tile / p.mblocks;
      const long m = static_cast<long>(mb) * BM + row;
      const long n0 = static_cast<long>(nb) * BN + half * 128;
      uint32_t acc[128];  // int32 sums (per channel) or fp32 totals (per group)
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0u;
      const int nchunks = (nkb + chunk_kb - 1) / chunk_kb;
      for (int c = 0; c < nchunks; ++c) {
        const uint32_t r = cc & 1u;
        bool w = wait_bar(accfull(r), (cc >> 1) & 1u, abort_flag, kDevErrAccumBarrier, p.err);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sa_g = 0.f;
        if (PERGROUP && p.acc_out == nullptr && m < p.M) sa_g = p.sa[m * p.G + c];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t v[16];
          tmem_ld16(tq + r * BN + half * 128 + j * 16, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float f = __uint_as_float(v[i]);
            const int idx = j * 16 + i;
            if (PERGROUP) {
              const long n = n0 + idx;
              if (p.acc_out != nullptr) {
                if (m < p.M && n < p.N)
                  stg_b32(p.acc_out + (m * p.N + n) * p.G + c, __float2int_rn(f));
              } else {
                const float swv = n < p.N ? ldg_f32(p.sw + n * p.G + c) : 0.f;
                acc[idx] = __float_as_uint(__fadd_rn(__uint_as_float(acc[idx]),
                                                     __fmul_rn(f, __fmul_rn(sa_g, swv))));
              }
            } else {
              acc[idx] = static_cast<uint32_t>(static_cast<int>(acc[idx]) + __float2int_rn(f));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accempty(r));
        ++cc;
      }
      if (!ok) break;
      if (m >= p.M) continue;
      if (p.acc_out != nullptr) {
        if (!PERGROUP) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (n0 + i < p.N) stg_b32(p.acc_out + m * p.N + n0 + i, static_cast<int>(acc[i]));
        }
        continue;
      }
      const float sam = PERGROUP ? 0.f : p.sa[m];
      __half *yr = p.y + m * p.N;
      const bool vec = (p.N & 7) == 0;
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        const long nb8 = n0 + c8 * 8;
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int idx = c8 * 8 + i;
          if (PERGROUP) {
            o[i] = __uint_as_float(acc[idx]);
          } else {
            const long n = nb8 + i;
            const float swv = n < p.N ? ldg_f32(p.sw + n) : 0.f;
            o[i] = __fmul_rn(static_cast<float>(static_cast<int>(acc[idx])),
                             __fmul_rn(sam, swv));
          }
        }
        if (vec && nb8 + 8 <= p.N) {
          uint4 h;
          __half2 t0 = __floats2half2_rn(o[0], o[1]), t1 = __floats2half2_rn(o[2], o[3]);
          __half2 t2 = __floats2half2_rn(o[4], o[5]), t3 = __floats2half2_rn(o[6], o[7]);
          h.x = *reinterpret_cast<uint32_t *>(&t0);
          h.y = *reinterpret_cast<uint32_t *>(&t1);
          h.z = *reinterpret_cast<uint32_t *>(&t2);
          h.w = *reinterpret_cast<uint32_t *>(&t3);
          stg_v4(yr + nb8, h);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (nb8 + i < p.N) stg_b16(yr + nb8 + i, __float2half_rn(o[i]));
        }
      }
    }
    tc_fence_before();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
    if (warp == 0) {
      // ---------------------------------------------------- TMA producer --
      if (lane == 0) {
        int s = 0;
        uint32_t ph = 0;
        uint32_t pending = 0, pend_ph = 0;  // bit i: stage i issued / its parity
        const uint32_t bytes = A8_BYTES + (WBITS == 8 ? B8_BYTES : B8_BYTES / 2);
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
          const int mb = tile % p.mblocks, nb = tile / p.mblocks;
          bool ok = true;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bar(empty8(s), ph ^ 1u, abort_flag, kDevErrEmptyBarrier, p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full8(s), bytes);
            tma_load_2d(base + OFF_A8 + s * A8_BYTES, &tmA, full8(s), kb * BK, mb * BM);
            tma_load_2d(base + OFF_B8 + s * B8_BYTES, &tmB, full8(s),
                        WBITS == 8 ? kb * BK : kb * (BK / 2), nb * BN);
            pending |= 1u << s;
            pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
            if (++s == S8) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
        }
        // every copy this thread issued has landed before the CTA can exit
        for (int i = 0; i < S8; ++i)
          if ((pending >> i) & 1u) wait_bar_teardown(full8(i), (pend_ph >> i) & 1u);
      }
    } else if (warp == 1) {
      // ---------------------------------------------------- MMA issuer ----
      if (lane == 0) {
        int s = 0;
        uint32_t ph = 0, cc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
          for (int kb = 0; kb < nkb; ++kb) {
            const bool first = (kb % chunk_kb) == 0;
            const uint32_t r = cc & 1u;
            if (first) {
              if (!wait_bar(accempty(r), ((cc >> 1) & 1u) ^ 1u, abort_flag, kDevErrTmemEmpty,
                            p.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!wait_bar(full16(s), ph, abort_flag, kDevErrFullBarrier, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + r * BN;
            const uint32_t a_base = base + OFF_A16 + s * A16_BYTES;
            const uint32_t b_base = base + OFF_B16 + s * B16_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              tc_mma(d, sw128_desc(a_base + k * 32), sw128_desc(b_base + k * 32),
                     (first && k == 0) ? 0u : 1u);
            }
            tc_commit(empty16(s));
            if ((kb % chunk_kb) == chunk_kb - 1 || kb == nkb - 1) {
              tc_commit(accfull(r));
              ++cc;
            }
            if (++s == S16) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        // all MMAs issued here have completed before TMEM is freed
        tc_commit(drain_bar);
        wait_bar_teardown(drain_bar, 0);
      }
    } else if (warp < 2 + CONV_WARPS) {
      // ---------------------------------------------------- converters ----
      const int ct = (warp - 2) * 32 + lane;
      int s8 = 0, s16 = 0;
      uint32_t ph8 = 0, ph16 = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb) {
          bool w = wait_bar(full8(s8), ph8, abort_flag, kDevErrFullBarrier, p.err);
          w = w && wait_bar(empty16(s16), ph16 ^ 1u, abort_flag, kDevErrEmptyBarrier, p.err);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          const uint8_t *a8 = sm + OFF_A8 + s8 * A8_BYTES;
          const uint8_t *b8 = sm + OFF_B8 + s8 * B8_BYTES;
          uint8_t *a16 = sm + OFF_A16 + s16 * A16_BYTES;
          uint8_t *b16 = sm + OFF_B16 + s16 * B16_BYTES;
          // A: 128 rows x 8 units of 8 elements
#pragma unroll 1
          for (int u = ct; u < BM * 8; u += CONV_WARPS * 32) {
            const int r = u >> 3, j = u & 7;
            const uint2 v = *reinterpret_cast<const uint2 *>(a8 + r * 64 + j * 8);
            uint4 o;
            i8x4_to_h(v.x, o.x, o.y);
            i8x4_to_h(v.y, o.z, o.w);
            *reinterpret_cast<uint4 *>(a16 + sw128_off(r, j)) = o;
          }
          // B: 256 rows x 8 units
#pragma unroll 1
          for (int u = ct; u < BN * 8; u += CONV_WARPS * 32) {
            const int r = u >> 3, j = u & 7;
            uint4 o;
            if (WBITS == 8) {
              const uint2 v = *reinterpret_cast<const uint2 *>(b8 + r * 64 + j * 8);
              i8x4_to_h(v.x, o.x, o.y);
              i8x4_to_h(v.y, o.z, o.w);
            } else {
              o = i4x8_to_h(*reinterpret_cast<const uint32_t *>(b8 + r * 32 + j * 4));
            }
            *reinterpret_cast<uint4 *>(b16 + sw128_off(r, j)) = o;
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(full16(s16));
            mbar_arrive(empty8(s8));
          }
          if (++s8 == S8) {
            s8 = 0;
            ph8 ^= 1u;
          }
          if (++s16 == S16) {
            s16 = 0;
            ph16 ^= 1u;
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

// ------------------------------------------------------------ host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D UINT8 tensor map over a row-major [rows, cols] byte matrix with a
// box of [box_rows, box_cols] (no swizzle; out-of-range elements read 0).
bool make_map(CUtensorMap *map, const void *ptr, long rows, long cols, int box_rows,
              int box_cols) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int WBITS, bool PERGROUP>
int launch_t(const CUtensorMap &ta, const CUtensorMap &tb, const TcParams &p, cudaStream_t s) {
  static bool attr_set[64] = {};
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return W8A8_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<WBITS, PERGROUP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return W8A8_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return W8A8_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int grid = p.ntiles < sms[dev] ? p.ntiles : sms[dev];
  gemm_tc_kernel<WBITS, PERGROUP><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ta, tb, p);
  return launch_status();
}

}  // namespace

int launch_gemm_tc(const int8_t *xq, const float *sa, const void *W, const float *sw, int M,
                   int N, int K, int group_size, int wbits, __half *y, int32_t *acc_out,
                   cudaStream_t s) {
  CUtensorMap ta, tb;
  if (!make_map(&ta, xq, M, K, BM, BK)) return W8A8_ERR_CUDA;
  if (wbits == 8) {
    if (!make_map(&tb, W, N, K, BN, BK)) return W8A8_ERR_CUDA;
  } else {
    if (!make_map(&tb, W, N, K / 2, BN, BK / 2)) return W8A8_ERR_CUDA;
  }
  unsigned int *err = device_error_word();
  if (err == nullptr) return W8A8_ERR_CUDA;
  TcParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.gs = group_size;
  p.G = groups_of(K, group_size);
  p.nkb = (K + BK - 1) / BK;
  // K blocks per exact fp32 chunk (see the header comment)
  if (group_size != 0)
    p.chunk_kb = group_size / BK;
  else
    p.chunk_kb = wbits == 8 ? 1024 / BK : 16384 / BK;
  p.mblocks = (M + BM - 1) / BM;
  const long nblocks = (N + BN - 1) / BN;
  const long ntiles = static_cast<long>(p.mblocks) * nblocks;
  if (ntiles > 0x7fffffffL) return W8A8_ERR_INVALID_ARG;
  p.ntiles = static_cast<int>(ntiles);
  p.sa = sa;
  p.sw = sw;
  p.y = y;
  p.acc_out = acc_out;
  p.err = err;
  if (wbits == 4) return launch_t<4, false>(ta, tb, p, s);
  if (group_size != 0) return launch_t<8, true>(ta, tb, p, s);
  return launch_t<8, false>(ta, tb, p, s);
}

}  // namespace w8a8
