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
// Operand roles: the weights are the MMA's A operand (128 output channels
// per tile, the TMEM lanes) and the activations its B operand (BT = 256 or
// 128 tokens per tile, the TMEM columns), so the operand that has to be
// converted from INT8 / INT4 codes to fp16 in shared memory is the smaller
// 128-row one.  The activations arrive either as fp16 codes, which TMA
// places directly in the MMA's layout, or as INT8 codes, converted too.
//
// Kernel layout (persistent, one CTA of 16 warps per SM; a pipeline stage
// holds KS 64-deep K blocks, KS = 2 per channel with fp16 codes, else 1):
//   warp 0      TMA producer: INT8 / packed INT4 weight tiles into a staging
//               ring; activation tiles into the staging ring (INT8) or
//               straight into the MMA operand stage (fp16 codes, 128-byte
//               swizzle, K-major);
//   warp 1      allocates TMEM and issues the MMAs (one thread): four
//               128 x BT x 16 tcgen05.mma per K block into one of two TMEM
//               accumulators (ping-pong per chunk);
//   warps 2-7   converters: INT8 / INT4 codes -> fp16, written in the
//               128-byte-swizzled K-major layout the MMA reads, one K block
//               of a stage at a time, each announced on its own barrier so
//               that the MMAs start on a stage's first block;
//   warps 8-15  epilogue: drain TMEM (tcgen05.ld), exact int32 sums or fp32
//               per-group rescale, then the fp16 output; each thread owns
//               one output channel and BT / 2 tokens, so a warp's store
//               writes 32 consecutive channels of one token.  The
//               activation scales of the tile are staged in shared memory.
// The kernel is launched as a programmatic dependent of the previous one on
// the stream: its set-up (barriers, TMEM) may overlap that kernel's tail,
// and griddepcontrol.wait precedes every read of an input.
// Stages hand over through mbarriers; every wait is bounded, and a wait that
// gives up records a code in the device error word, raises an abort flag
// seen by every role, lets in-flight copies and MMAs land, frees TMEM and
// returns.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace w8a8 {
namespace {

constexpr int BW = 128, BK = 64;  // weight rows (output channels) per tile, K block
constexpr int NUM_THREADS = 512;
constexpr int EPI_WARPS = 8, EPI_THREADS = EPI_WARPS * 32;
// Limit of every bounded wait, in SM clock cycles (about 2 s at 2 GHz).  The
// role waits take theirs from the launch (TcParams::wait_limit, this value
// unless a test shortened it); the teardown waits always use this one.
constexpr long long kTimeoutCycles = 4000000000LL;

// Shared-memory plan.  XH: activations arrive as fp16 codes (TMA straight
// into the operand layout); BT: tokens per tile (activations as INT8 codes
// use BT = 128); KS: 64-wide K blocks per stage.  Two rings: the INT8 / INT4
// staging ring (TMA -> converters) and the operand stages, each holding KS
// K blocks of fp16 weights (written by the converters) and fp16 activations
// (written by TMA, or by the converters), as KS 64-wide sub-tiles of
// 128-byte swizzled rows per operand.  Operand stages are released REL at a
// time (one MMA commit per REL stages).
//
// Every stage costs the same hand-offs between the roles (staging copy ->
// converters -> MMA -> release), so KS = 2 (two K blocks behind one
// hand-off, two stages of 96 KB) halves that cost per FLOP; single-K-block
// stages, even four of them, measured slower.  What bounds the two-stage
// ring (clock64 trace of one CTA at M = 8192): a stage's activation copy is
// issued ~675 cycles after the last MMA of the stage whose slot it refills
// (MMA completion, commit, wake-up) and lands ~2000 cycles later, against
// ~1000 cycles of MMAs in the other stage, so the tensor pipe waits ~40 % of
// the time.  The plan needs the full 227 KB, with no room for aligning the
// dynamic shared memory by hand: the kernel checks that its base is 1 KB
// aligned instead.
template <bool XH, int BT, int KS>
struct Plan {
  static constexpr int KB = BK * KS;                // K per stage
  static constexpr int W8_BYTES = BW * KB;          // INT8 weight stage (INT4 uses half)
  static constexpr int X8_BYTES = XH ? 0 : BT * KB;
  static constexpr int W16_SUB = BW * BK * 2;       // one fp16 sub-tile, 128-byte rows
  static constexpr int X16_SUB = BT * BK * 2;
  static constexpr int W16_BYTES = W16_SUB * KS;
  static constexpr int X16_BYTES = X16_SUB * KS;
  static constexpr int STAGE_BYTES = W16_BYTES + X16_BYTES;
  // S: operand stages.  With KS = 1 a fourth measured no faster, and three
  // leave more of the SM's L1 to the per-group epilogue's scale loads.
  // S8: weight staging stages.  128-token tiles of two K blocks have room
  // for a third (M = 128: 19.3 -> 17.9 us; a fourth gained nothing more,
  // and a third operand stage in its place gained nothing).
  static constexpr int S8 = KS == 1 ? 3 : (BT == 128 ? 3 : 2), S = KS == 1 ? 3 : 2;
  static constexpr int REL = 1;                    // stages released per commit
  // warp roles: 0 producers (lane 0 staging, lane 1 fp16 activations), 1
  // MMA, 2-7 converters, 8-15 epilogue
  static constexpr int CONV_WARPS = 6;
  static constexpr int CONV_WARP0 = 2;
  static constexpr int CONV_THREADS = CONV_WARPS * 32;
  static constexpr int OFF_W8 = 0;
  static constexpr int OFF_X8 = OFF_W8 + S8 * W8_BYTES;
  static constexpr int OFF_ST = OFF_X8 + S8 * X8_BYTES;    // stage s: W16, then X16
  static constexpr int OFF_SA = OFF_ST + S * STAGE_BYTES;  // 2 x BT fp32 scales
  static constexpr int OFF_BAR = OFF_SA + 2 * BT * 4;
  static constexpr int NUM_BARS = 2 * S8 + S * KS + S / REL + 2 + 2 + 2 + 1;  // full: one per sub-tile
  static constexpr int ALIGN_SLACK = KS == 1 ? 1024 : 0;
  static constexpr int SMEM_BYTES = OFF_BAR + NUM_BARS * 8 + 16 + ALIGN_SLACK;
  static constexpr uint32_t TMEM_COLS = 2 * BT;  // two accumulators of BT fp32 columns
  static_assert(OFF_ST % 1024 == 0 && W16_SUB % 1024 == 0 && X16_SUB % 1024 == 0 &&
                    STAGE_BYTES % 1024 == 0,
                "swizzled stages need 1 KB alignment");
  static_assert(S % REL == 0, "stages are released in groups of REL");
};
static_assert(Plan<true, 256, 1>::SMEM_BYTES <= 232448, "shared memory plan too large");
static_assert(Plan<true, 256, 2>::SMEM_BYTES <= 232448, "shared memory plan too large");
static_assert(Plan<true, 128, 2>::SMEM_BYTES <= 232448, "shared memory plan too large");
static_assert(Plan<false, 128, 1>::SMEM_BYTES <= 232448, "shared memory plan too large");

// instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// M = 128 (weights), N = BT (tokens)
template <int BT>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(BT >> 3) << 17) |
         (static_cast<uint32_t>(BW >> 4) << 24);
}

struct TcParams {
  int M, N, K, gs, G, nkb, chunk_kb, nblocks, ntiles;
  const float *sa;
  const float *sw;
  __half *y;
  int32_t *acc_out;
  unsigned int *err;
  long long wait_limit;  // role waits give up after this many cycles
  int skip_first_copy;   // test only: leave the first staging copy of each CTA unissued
};

// ---------------------------------------------------------------- PTX ----

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

// HINT: the waiting thread re-checks at least every 100 ns instead of
// after the system-dependent suspend time (measured on GB300: the per
// channel kernels ~2 % faster, the per-group ones ~4 % slower, so only the
// former pass it).
template <bool HINT = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if (HINT)
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(100)
        : "memory");
  else
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
                                       uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum));
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

// Ordered memory accesses for the epilogue: as volatile asm they keep their
// program order, so a fully unrolled loop does not hoist all of its loads
// ahead of its stores (which would need one register per load).
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void stg_b16(void *ptr, __half v) {
  asm volatile("st.global.b16 [%0], %1;" ::"l"(ptr), "h"(__half_as_ushort(v)) : "memory");
}

__device__ __forceinline__ void stg_b32(void *ptr, int v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Bounded wait.  Returns false if the CTA is aborting or the wait gave up
// (then it records `code` and raises the abort flag).
template <bool HINT = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity,
                                         volatile int *abort_flag, unsigned int code,
                                         unsigned int *err, long long limit) {
#pragma unroll 1
  for (int i = 0; i < 32; ++i)
    if (mbar_try_wait<HINT>(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait<HINT>(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
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

__device__ __forceinline__ uint4 i8x8_to_h(uint2 v) {
  uint4 o;
  i8x4_to_h(v.x, o.x, o.y);
  i8x4_to_h(v.y, o.z, o.w);
  return o;
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

// Two scale products s_i * w with one paired fp32 multiply (each half an
// IEEE multiply rounded to nearest).
__device__ __forceinline__ void mul2(float s0, float s1, float w, float &p0, float &p1) {
  asm("{\n.reg .b64 a, b, c;\n"
      "mov.b64 a, {%2, %3};\n"
      "mov.b64 b, {%4, %4};\n"
      "mul.rn.f32x2 c, a, b;\n"
      "mov.b64 {%0, %1}, c;\n}\n"
      : "=f"(p0), "=f"(p1)
      : "f"(s0), "f"(s1), "f"(w));
}

// f_i = fma(v_i, s_i, f_i) for two lanes with one paired fused multiply-add
// (f and v are fp32 bit patterns held in integer registers).
__device__ __forceinline__ void fma2(uint32_t &f0, uint32_t &f1, uint32_t v0, uint32_t v1,
                                     float s0, float s1) {
  asm("{\n.reg .b64 a, b, c, d;\n"
      "mov.b64 a, {%2, %3};\n"
      "mov.b64 b, {%4, %5};\n"
      "mov.b64 c, {%0, %1};\n"
      "fma.rn.f32x2 d, a, b, c;\n"
      "mov.b64 {%0, %1}, d;\n}\n"
      : "+r"(f0), "+r"(f1)
      : "r"(v0), "r"(v1), "f"(s0), "f"(s1));
}

// Converts sub-tile `sub` (codes 64 sub .. 64 sub + 63 of each of ROWS rows)
// of a staged tile of ROWS x (64 KS) codes into its swizzled fp16 operand
// sub-tile (ROWS x 64, 128-byte rows; sub-tiles ROWS * 128 bytes apart).
// Unit u = (row u / 4, codes 16 (u % 4) .. +16 of the sub-tile): one 16-byte
// load (8 bytes of packed INT4) and two 16-byte stores into the swizzled
// chunks 2 (u % 4) and 2 (u % 4) + 1 of its row.  A warp covers 8 whole
// rows; each 8-thread store phase writes two rows' even (or odd) chunks,
// which the 128-byte swizzle puts in disjoint banks.  All of a thread's
// units (UPT of them) are loaded before any is converted, so a sub-tile
// costs one shared-memory round trip per thread, not one per unit.
template <bool INT4, int NT, int ROWS, int KS>
__device__ __forceinline__ void convert_sub(const uint8_t *src, uint8_t *dst, int ct, int sub) {
  constexpr int units = ROWS * 4;
  constexpr int UPT = (units + NT - 1) / NT;  // units per thread
  constexpr int SRC_ROW = INT4 ? 32 * KS : 64 * KS;
  uint4 v[UPT];
#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = ct + i * NT;
    v[i] = make_uint4(0, 0, 0, 0);
    if (u < units) {
      const int r = u >> 2, c = sub * 4 + (u & 3);
      if (INT4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(src + r * SRC_ROW + c * 8);
        v[i].x = w.x;
        v[i].y = w.y;
      } else {
        v[i] = *reinterpret_cast<const uint4 *>(src + r * SRC_ROW + c * 16);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = ct + i * NT;
    if (u < units) {
      const int r = u >> 2, c4 = u & 3;
      uint4 lo, hi;
      if (INT4) {
        lo = i4x8_to_h(v[i].x);
        hi = i4x8_to_h(v[i].y);
      } else {
        lo = i8x8_to_h(make_uint2(v[i].x, v[i].y));
        hi = i8x8_to_h(make_uint2(v[i].z, v[i].w));
      }
      uint8_t *row = dst + sub * (ROWS * 128) + (r >> 3) * 1024 + (r & 7) * 128;
      const int x = r & 7;
      *reinterpret_cast<uint4 *>(row + (((2 * c4) ^ x) << 4)) = lo;
      *reinterpret_cast<uint4 *>(row + (((2 * c4 + 1) ^ x) << 4)) = hi;
    }
  }
}

// 32 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
        "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
        "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
        "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
        "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// Waits for this thread's TMEM loads; the loaded registers pass through the
// statement, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// Epilogue of the tensor-core GEMM (warps 8-15): drains the TMEM
// accumulators chunk by chunk and writes fp16 y.  The accumulator of a tile
// holds 128 output channels (TMEM lanes) x BT tokens (columns); warp 8 + 4h
// + q owns lane quadrant q and tokens [h BT/2, (h+1) BT/2).  Tiles are
// tile0, tile0 + tile_step, ...; tile t covers channels (t % nblocks) *
// ch_block + ch_off + [0, 128) and tokens (t / nblocks) * BT + [0, BT).
// Each warp arrives on accempty0 (+8 per accumulator) when its share of a
// chunk is drained.  The columns of a chunk are read 32 at a time, each
// slice finished before the next is loaded (one slice live keeps the
// register count within the epilogue's share; loading the next slice early,
// 16 columns at a time, measured slower per group).  Modes:
//   exact per channel: each chunk is converted to int32 (exact) and summed
//     in integer; y = fp16(float(sum) * (s_a * s_w));
//   per group: each group's exact partial is rescaled and accumulated in
//     ascending order, f = fma(acc_g, s_a,g * s_w,g, f), two lanes per
//     instruction (paired multiply for the scale products, paired fused
//     multiply-add); the fused form skips the rounding of each product
//     (at most half an ulp of acc_g * s per group), far inside the fp16
//     tolerance, and halves the drain's instructions; y = fp16(f);
//   weight-only (WONLY, fp16 activations): one float accumulation over K,
//     y = fp16(acc * s_w), or per group f = fma(acc_g, s_w,g, f).
template <bool PERGROUP, bool WONLY, int BT>
__device__ __forceinline__ void epilogue_role(const TcParams &p, uint32_t tmem, uint32_t base,
                                              uint8_t *sm, int off_sa, int warp, int lane,
                                              int tile0, int tile_step, int nblocks, int ch_block,
                                              int ch_off, uint32_t accfull0, uint32_t accempty0,
                                              uint32_t saready0, volatile int *abort_flag) {
  constexpr int CPT = BT / 2;  // token columns per epilogue thread
  // activation scales are staged per tile (per channel) or per group
  constexpr bool STAGE_SA = !WONLY;
  const int nkb = p.nkb, chunk_kb = p.chunk_kb;
  auto accfull = [&](uint32_t r) { return accfull0 + 8u * r; };
  auto accempty = [&](uint32_t r) { return accempty0 + 8u * r; };
  auto saready = [&](uint32_t b) { return saready0 + 8u * b; };
  const int q = warp & 3;             // TMEM lane quadrant of this warp
  const int et = (warp - 8) * 32 + lane;
  const int half = (warp - 8) >> 2;   // which half of the BT token columns
  const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
  const uint32_t sas = base + off_sa;
  float *sas_ptr = reinterpret_cast<float *>(sm + off_sa);
  const bool want_y = p.acc_out == nullptr;
  uint32_t cc = 0, su = 0;  // chunks drained, scale buffers used
  bool ok = true;
  for (int tile = tile0; tile < p.ntiles && ok; tile += tile_step) {
    const int nb = tile % nblocks, tb = tile / nblocks;
    // this thread's channel
    const long n = static_cast<long>(nb) * ch_block + ch_off + q * 32 + lane;
    const long mtile = static_cast<long>(tb) * BT;
    const long m0 = mtile + half * CPT;                           // its first token
    // per channel: stage the tile's BT activation scales now, used at the end
    uint32_t sb = 0, sph = 0;
    float swn = 0.f;
    if (!PERGROUP && want_y) {
      if (STAGE_SA) {
        sb = su & 1u;
        sph = (su >> 1) & 1u;
        ++su;
        if (et < BT) {
          const long m = mtile + et;
          sas_ptr[sb * BT + et] = m < p.M ? __ldg(p.sa + m) : 0.f;
        }
        mbar_arrive(saready(sb));
      }
      if (n < p.N) swn = __ldg(p.sw + n);
    }
    uint32_t acc[CPT];  // int32 sums (exact per channel) or fp32 totals
#pragma unroll
    for (int i = 0; i < CPT; ++i) acc[i] = 0u;
    const int nchunks = (nkb + chunk_kb - 1) / chunk_kb;
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t r = cc & 1u;
      float sw_g = 0.f;
      uint32_t gb = 0, gph = 0;
      if (PERGROUP && want_y) {
        if (STAGE_SA) {
          // stage group c's activation scales for the BT tokens
          gb = su & 1u;
          gph = (su >> 1) & 1u;
          ++su;
          if (et < BT) {
            const long m = mtile + et;
            sas_ptr[gb * BT + et] = m < p.M ? __ldg(p.sa + m * p.G + c) : 0.f;
          }
          mbar_arrive(saready(gb));
        }
        if (n < p.N) sw_g = __ldg(p.sw + n * p.G + c);
      }
      bool w = wait_bar<!PERGROUP>(accfull(r), (cc >> 1) & 1u, abort_flag, kDevErrAccumBarrier, p.err,
                        p.wait_limit);
      if (PERGROUP && want_y && STAGE_SA)
        w = w && wait_bar<!PERGROUP>(saready(gb), gph, abort_flag, kDevErrAccumBarrier, p.err, p.wait_limit);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t col0 = tq + r * BT + half * CPT;
#pragma unroll
      for (int j = 0; j < CPT / 32; ++j) {
        uint32_t v[32];
        tmem_ld32(col0 + j * 32, v);
        tmem_wait_ld32(v);
        if (PERGROUP) {
          if (want_y) {
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              float sc[4];
              if (WONLY) {
                sc[0] = sc[1] = sc[2] = sc[3] = sw_g;
              } else {
                const float4 s4 = lds_f32x4(sas + (gb * BT + half * CPT + j * 32 + i4 * 4) * 4);
                mul2(s4.x, s4.y, sw_g, sc[0], sc[1]);  // s_a * s_w first, as in the dequant rule
                mul2(s4.z, s4.w, sw_g, sc[2], sc[3]);
              }
              const int idx = j * 32 + i4 * 4;
              fma2(acc[idx], acc[idx + 1], v[i4 * 4], v[i4 * 4 + 1], sc[0], sc[1]);
              fma2(acc[idx + 2], acc[idx + 3], v[i4 * 4 + 2], v[i4 * 4 + 3], sc[2], sc[3]);
            }
          } else if (n < p.N) {
            // export of the exact group partials; sequential addresses
            int32_t *ap = p.acc_out + ((m0 + j * 32) * p.N + n) * p.G + c;
            const long step = static_cast<long>(p.N) * p.G;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (m0 + j * 32 + i < p.M) stg_b32(ap, __float2int_rn(__uint_as_float(v[i])));
              ap += step;
              asm volatile("" : "+l"(ap));
            }
          }
        } else if (WONLY) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int idx = j * 32 + i;
            acc[idx] = __float_as_uint(__fadd_rn(__uint_as_float(acc[idx]), __uint_as_float(v[i])));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int idx = j * 32 + i;
            acc[idx] = static_cast<uint32_t>(static_cast<int>(acc[idx]) +
                                             __float2int_rn(__uint_as_float(v[i])));
          }
        }
        // finish this slice before the next TMEM load (keeps one slice live)
#pragma unroll
        for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(acc[j * 32 + i]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty(r));
      ++cc;
    }
    if (!ok) break;
    if (!want_y) {
      if (!PERGROUP && n < p.N) {
        int32_t *ap = p.acc_out + m0 * p.N + n;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          if (m0 + i < p.M) stg_b32(ap, static_cast<int>(acc[i]));
          ap += p.N;
          asm volatile("" : "+l"(ap));
        }
      }
      continue;
    }
    if (!PERGROUP && STAGE_SA) {
      bool w = wait_bar<!PERGROUP>(saready(sb), sph, abort_flag, kDevErrAccumBarrier, p.err, p.wait_limit);
      if (!__all_sync(0xffffffffu, w)) break;
    }
    if (n >= p.N) continue;
    // y[m, n] for this thread's channel n and tokens m0 .. m0 + CPT - 1: a
    // warp store covers 32 consecutive channels (64 contiguous bytes).  The
    // row pointer advances by N per token; the empty asm keeps the compiler
    // from precomputing all CPT addresses at once.
    __half *yp = p.y + m0 * p.N + n;
    const int mcount = static_cast<int>(min(static_cast<long>(CPT), p.M - m0));
#pragma unroll
    for (int i4 = 0; i4 < CPT / 4; ++i4) {
      float sv[4] = {0.f, 0.f, 0.f, 0.f};
      if (!PERGROUP && !WONLY) {
        const float4 s4 = lds_f32x4(sas + (sb * BT + half * CPT + i4 * 4) * 4);
        sv[0] = s4.x;
        sv[1] = s4.y;
        sv[2] = s4.z;
        sv[3] = s4.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = i4 * 4 + e;
        if (i < mcount) {
          float o;
          if (PERGROUP)
            o = __uint_as_float(acc[i]);
          else if (WONLY)
            o = __fmul_rn(__uint_as_float(acc[i]), swn);
          else
            o = __fmul_rn(static_cast<float>(static_cast<int>(acc[i])), __fmul_rn(sv[e], swn));
          stg_b16(yp, __float2half_rn(o));
        }
        yp += p.N;
        asm volatile("" : "+l"(yp));
      }
    }
  }
  tc_fence_before();
}

// ------------------------------------------------------------- kernel ----

template <int WBITS, bool PERGROUP, bool XH, int BT, int KS, bool WONLY>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmW, const TcParams p) {
  using PL = Plan<XH, BT, KS>;
  constexpr int S8 = PL::S8, S = PL::S;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  if (PL::ALIGN_SLACK == 0 && (raw & 1023u) != 0) {
    // the plan has no slack for aligning by hand: report and do nothing
    if (threadIdx.x == 0 && p.err != nullptr) atomicCAS(p.err, 0u, static_cast<unsigned>(kDevErrSmemAlign));
    return;
  }
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sm = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = base + PL::OFF_BAR;
  auto full8 = [&](int s) { return bar0 + 8u * s; };
  auto empty8 = [&](int s) { return bar0 + 8u * (S8 + s); };
  // full(s, j): sub-tile j of stage s is in place (its converters and its
  // activation copy), so the MMAs of a stage start on its first sub-tile
  auto full = [&](int s, int j) { return bar0 + 8u * (2 * S8 + s * KS + j); };
  constexpr int REL = PL::REL;
  auto empty = [&](int g) { return bar0 + 8u * (2 * S8 + S * KS + g); };  // per release group
  constexpr int B_ACC = 2 * S8 + S * KS + S / REL;
  auto accfull = [&](int r) { return bar0 + 8u * (B_ACC + r); };
  auto accempty = [&](int r) { return bar0 + 8u * (B_ACC + 2 + r); };
  auto saready = [&](int b) { return bar0 + 8u * (B_ACC + 4 + b); };
  const uint32_t drain_bar = bar0 + 8u * (B_ACC + 6);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + PL::OFF_BAR + PL::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto w16 = [&](int s) { return base + PL::OFF_ST + s * PL::STAGE_BYTES; };  // + j W16_SUB
  auto x16 = [&](int s) { return base + PL::OFF_ST + s * PL::STAGE_BYTES + PL::W16_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S8; ++s) {
      mbar_init(full8(s), 1);
      mbar_init(empty8(s), PL::CONV_WARPS);
    }
    for (int s = 0; s < S; ++s)
      for (int j = 0; j < KS; ++j) mbar_init(full(s, j), PL::CONV_WARPS + (XH ? 1 : 0));
    for (int g = 0; g < S / REL; ++g) mbar_init(empty(g), 1);
    for (int r = 0; r < 2; ++r) {
      mbar_init(accfull(r), 1);
      mbar_init(accempty(r), EPI_WARPS);
      mbar_init(saready(r), EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(PL::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as a programmatic dependent: the set-up above may overlap the
  // previous kernel on the stream; every read of an input comes after this
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int nkb = p.nkb, chunk_kb = p.chunk_kb;

  // Register split per warpgroup (launch: 512 threads x 128 registers):
  // warpgroups 2-3 (epilogue) rise to 184, warpgroups 0-1 (producer, MMA,
  // converters) drop to 72; 256 * 184 + 256 * 72 = 65536 = 512 * 128.  The
  // per-group kernels, bound by their epilogue, give it 200 and the others
  // 56 (256 * 200 + 256 * 56 = 65536; measured ~1 % faster, and the
  // converters still fit).  Each side's code sits inside the branch of its
  // own setmaxnreg, so the compiler allocates registers to that limit.
  if (warp >= 8) {
    if (PERGROUP)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    epilogue_role<PERGROUP, WONLY, BT>(p, tmem, base, sm, PL::OFF_SA, warp, lane, blockIdx.x,
                                       gridDim.x, p.nblocks, BW, 0, accfull(0), accempty(0),
                                       saready(0), abort_flag);
    tc_fence_before();
  } else {
    if (PERGROUP)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
    if (warp == 0) {
      // ------------------------------------------- staging TMA producer --
      if (lane == 0) {
        int s8 = 0;
        uint32_t ph8 = 0;
        uint32_t pend = 0, pph = 0;  // bit i: stage i has a copy issued / its parity
        const uint32_t bytes8 = (WBITS == 8 ? PL::W8_BYTES : PL::W8_BYTES / 2) + PL::X8_BYTES;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
          const int nb = tile % p.nblocks, tb = tile / p.nblocks;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bar<!PERGROUP>(empty8(s8), ph8 ^ 1u, abort_flag, kDevErrEmptyBarrier, p.err, p.wait_limit)) {
              ok = false;
              break;
            }
            // (test only) a stage left unissued: its full barrier never
            // completes, so the converters' bounded wait on it runs out
            if (!(p.skip_first_copy && tile == static_cast<int>(blockIdx.x) && kb == 0)) {
              mbar_arrive_expect_tx(full8(s8), bytes8);
              tma_load_2d(base + PL::OFF_W8 + s8 * PL::W8_BYTES, &tmW, full8(s8),
                          WBITS == 8 ? kb * PL::KB : kb * (PL::KB / 2), nb * BW);
              if (!XH)
                tma_load_2d(base + PL::OFF_X8 + s8 * PL::X8_BYTES, &tmX, full8(s8),
                            kb * PL::KB, tb * BT);
              pend |= 1u << s8;
              pph = (pph & ~(1u << s8)) | (ph8 << s8);
            }
            if (++s8 == S8) {
              s8 = 0;
              ph8 ^= 1u;
            }
          }
        }
        // every copy this thread issued has landed before the CTA can exit
        for (int i = 0; i < S8; ++i)
          if ((pend >> i) & 1u) wait_bar_teardown(full8(i), (pph >> i) & 1u);
      } else if (XH && lane == 1) {
        // ----------------------------- activation (fp16 codes) producer --
        int s = 0;
        uint32_t ph = 0, pend = 0, pph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
          const int tb = tile / p.nblocks;
          for (int kb = 0; kb < nkb; ++kb) {
            // a release group is refilled once the MMAs of its last use are done
            if ((s % REL) == 0 &&
                !wait_bar<!PERGROUP>(empty(s / REL), ph ^ 1u, abort_flag, kDevErrEmptyBarrier, p.err, p.wait_limit)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < KS; ++j) {
              mbar_arrive_expect_tx(full(s, j), PL::X16_SUB);
              tma_load_2d(x16(s) + j * PL::X16_SUB, &tmX, full(s, j), kb * PL::KB + j * BK,
                          tb * BT);
            }
            pend |= 1u << s;
            pph = (pph & ~(1u << s)) | (ph << s);
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        for (int i = 0; i < S; ++i)
          if ((pend >> i) & 1u)
            for (int j = 0; j < KS; ++j) wait_bar_teardown(full(i, j), (pph >> i) & 1u);
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
              if (!wait_bar<!PERGROUP>(accempty(r), ((cc >> 1) & 1u) ^ 1u, abort_flag, kDevErrTmemEmpty,
                            p.err, p.wait_limit)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d = tmem + r * BT;
#pragma unroll
            for (int j = 0; j < KS; ++j) {
              if (!wait_bar<!PERGROUP>(full(s, j), ph, abort_flag, kDevErrFullBarrier, p.err, p.wait_limit)) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                tc_mma(d, sw128_desc(w16(s) + j * PL::W16_SUB + k * 32),
                       sw128_desc(x16(s) + j * PL::X16_SUB + k * 32), idesc<BT>(),
                       (first && j == 0 && k == 0) ? 0u : 1u);
              }
            }
            if (!ok) break;
            if ((s % REL) == REL - 1) tc_commit(empty(s / REL));
            if ((kb % chunk_kb) == chunk_kb - 1 || kb == nkb - 1) {
              tc_commit(accfull(r));
              ++cc;
            }
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        // release a partly used last group, then let every MMA land before TMEM is freed
        if ((s % REL) != 0) tc_commit(empty(s / REL));
        tc_commit(drain_bar);
        wait_bar_teardown(drain_bar, 0);
      }
    } else {
      // ---------------------------------------------------- converters ----
      constexpr int NT = PL::CONV_THREADS;
      const int ct = (warp - PL::CONV_WARP0) * 32 + lane;
      int s8 = 0, s = 0;
      uint32_t ph8 = 0, ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb) {
          bool w = wait_bar<!PERGROUP>(full8(s8), ph8, abort_flag, kDevErrFullBarrier, p.err, p.wait_limit);
          if ((s % REL) == 0)
            w = w && wait_bar<!PERGROUP>(empty(s / REL), ph ^ 1u, abort_flag, kDevErrEmptyBarrier, p.err, p.wait_limit);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int j = 0; j < KS; ++j) {
            convert_sub<WBITS == 4, NT, BW, KS>(sm + PL::OFF_W8 + s8 * PL::W8_BYTES,
                                                sm + (w16(s) - base), ct, j);
            if (!XH)
              convert_sub<false, NT, BT, KS>(sm + PL::OFF_X8 + s8 * PL::X8_BYTES,
                                             sm + (x16(s) - base), ct, j);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(full(s, j));
          }
          if (lane == 0) mbar_arrive(empty8(s8));
          if (++s8 == S8) {
            s8 = 0;
            ph8 ^= 1u;
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
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
                 "r"(PL::TMEM_COLS));
  }
}

// ------------------------------------------------------------ host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
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

// Role-wait limit and test switch for the next launches (w8a8_test_set_fault).
std::atomic<long long> g_wait_limit{kTimeoutCycles};
std::atomic<int> g_skip_first_copy{0};

// 2-D tensor map over a row-major [rows, cols] matrix of 1- or 2-byte
// elements, box [box_rows, box_cols]; out-of-range elements read 0.  2-byte
// maps use the 128-byte swizzle (box rows of exactly 128 bytes): the
// K-major layout the MMA reads.
bool make_map(CUtensorMap *map, const void *ptr, long rows, long cols, int elem_bytes,
              int box_rows, int box_cols) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const bool h = elem_bytes == 2;
  return enc(map, h ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             h ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int WBITS, bool PERGROUP, bool XH, int BT, int KS, bool WONLY = false>
int launch_t(const CUtensorMap &tx, const CUtensorMap &tw, const TcParams &p, cudaStream_t s) {
  // per device: the shared-memory attribute set once, and the SM count
  static bool attr_set[64] = {};
  static int sms[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W8A8_ERR_CUDA;
  constexpr int smem = Plan<XH, BT, KS>::SMEM_BYTES;
  int nsm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(gemm_tc_kernel<WBITS, PERGROUP, XH, BT, KS, WONLY>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return W8A8_ERR_CUDA;
      if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return W8A8_ERR_CUDA;
      attr_set[dev] = true;
    }
    nsm = sms[dev];
  }
  const int grid = p.ntiles < nsm ? p.ntiles : nsm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemm_tc_kernel<WBITS, PERGROUP, XH, BT, KS, WONLY>, tx, tw, p) !=
      cudaSuccess) {
    cudaGetLastError();
    return W8A8_ERR_CUDA;
  }
  return launch_status();
}

template <bool XH, int BT>
int launch_modes(const CUtensorMap &tx, const CUtensorMap &tw, const TcParams &p, int wbits,
                 cudaStream_t s) {
  if (wbits == 4) return launch_t<4, false, XH, BT, 1>(tx, tw, p, s);
  if (p.gs != 0) return launch_t<8, true, XH, BT, 1>(tx, tw, p, s);
  return launch_t<8, false, XH, BT, 1>(tx, tw, p, s);
}

// X (activations) is int8 codes [M, K] (x_half false), the same codes as
// fp16 values (x_half true) or, for the weight-only product (wonly), the
// fp16 activations themselves.  256-token tiles for fp16 operands with M >
// 128, else 128; per channel with fp16 operands, a stage holds two K blocks.
int launch_gemm_any(const void *X, bool x_half, bool wonly, const float *sa, const void *W,
                    const float *sw, int M, int N, int K, int group_size, int wbits, __half *y,
                    int32_t *acc_out, cudaStream_t s) {
  // INT8 activation codes are converted in the kernel too: 128-token tiles
  const int bt = (M <= 128 || !x_half) ? 128 : 256;
  const int ks = (x_half && group_size == 0) ? 2 : 1;
  const int kb = BK * ks;  // K per stage
  CUtensorMap tx, tw;
  if (!make_map(&tx, X, M, K, x_half ? 2 : 1, bt, BK)) return W8A8_ERR_CUDA;
  if (wbits == 8) {
    if (!make_map(&tw, W, N, K, 1, BW, kb)) return W8A8_ERR_CUDA;
  } else {
    if (!make_map(&tw, W, N, K / 2, 1, BW, kb / 2)) return W8A8_ERR_CUDA;
  }
  unsigned int *err = device_error_word();
  if (err == nullptr) return W8A8_ERR_CUDA;
  TcParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.gs = group_size;
  p.G = groups_of(K, group_size);
  p.nkb = (K + kb - 1) / kb;  // stages per tile
  // stages per accumulator drain: per group, every group; exact per
  // channel, every chunk that keeps the fp32 sums exact (see the header
  // comment); weight-only per channel, once (float accumulation)
  if (group_size != 0)
    p.chunk_kb = group_size / kb;
  else if (wonly)
    p.chunk_kb = p.nkb;
  else
    p.chunk_kb = wbits == 8 ? 1024 / kb : 16384 / kb;
  p.nblocks = (N + BW - 1) / BW;
  const long tblocks = (M + bt - 1) / bt;
  const long ntiles = static_cast<long>(p.nblocks) * tblocks;
  if (ntiles > 0x7fffffffL) return W8A8_ERR_INVALID_ARG;
  p.ntiles = static_cast<int>(ntiles);
  p.sa = sa;
  p.sw = sw;
  p.y = y;
  p.acc_out = acc_out;
  p.err = err;
  p.wait_limit = g_wait_limit.load();
  p.skip_first_copy = g_skip_first_copy.load();
  if (wonly) {
    if (ks == 2) {
      if (bt == 128)
        return wbits == 4 ? launch_t<4, false, true, 128, 2, true>(tx, tw, p, s)
                          : launch_t<8, false, true, 128, 2, true>(tx, tw, p, s);
      return wbits == 4 ? launch_t<4, false, true, 256, 2, true>(tx, tw, p, s)
                        : launch_t<8, false, true, 256, 2, true>(tx, tw, p, s);
    }
    if (bt == 128) return launch_t<8, true, true, 128, 1, true>(tx, tw, p, s);
    return launch_t<8, true, true, 256, 1, true>(tx, tw, p, s);
  }
  if (x_half) {
    if (ks == 2) {
      if (bt == 128)
        return wbits == 4 ? launch_t<4, false, true, 128, 2>(tx, tw, p, s)
                          : launch_t<8, false, true, 128, 2>(tx, tw, p, s);
      return wbits == 4 ? launch_t<4, false, true, 256, 2>(tx, tw, p, s)
                        : launch_t<8, false, true, 256, 2>(tx, tw, p, s);
    }
    if (bt == 128) return launch_t<8, true, true, 128, 1>(tx, tw, p, s);
    return launch_t<8, true, true, 256, 1>(tx, tw, p, s);
  }
  return launch_modes<false, 128>(tx, tw, p, wbits, s);
}

}  // namespace

int launch_gemm_tc(const void *X, bool x_half, const float *sa, const void *W, const float *sw,
                   int M, int N, int K, int group_size, int wbits, __half *y,
                   int32_t *acc_out, cudaStream_t s) {
  return launch_gemm_any(X, x_half, false, sa, W, sw, M, N, K, group_size, wbits, y, acc_out, s);
}

int launch_gemm_weight_only(const __half *x, const void *W, const float *sw, int M, int N, int K,
                            int group_size, int wbits, __half *y, cudaStream_t s) {
  return launch_gemm_any(x, true, true, nullptr, W, sw, M, N, K, group_size, wbits, y, nullptr,
                         s);
}

}  // namespace w8a8

extern "C" int w8a8_test_set_fault(long long wait_limit_cycles, int skip_first_copy) {
  if (wait_limit_cycles < 0 || (skip_first_copy != 0 && skip_first_copy != 1))
    return W8A8_ERR_INVALID_ARG;
  w8a8::g_wait_limit.store(wait_limit_cycles == 0 ? w8a8::kTimeoutCycles : wait_limit_cycles);
  w8a8::g_skip_first_copy.store(skip_first_copy);
  return W8A8_OK;
}
