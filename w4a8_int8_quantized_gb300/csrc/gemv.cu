// Matrix-vector kernels for decode (M == 1) and few-row products (M = 2..8):
// W8A8 per channel / per group and W4A8 per channel; for M == 1 optionally
// fused with the activation quantization.
//
// Method: "cider 소개", section "cider의 동작 방식과 자동 경로 선택"
// (CiderLinear picks the INT8 MV kernel when seq_len == 1; the kernel list
// names a per-channel and a per-group MV kernel); "Apple Silicon의 AI
// 한계치는 당신의 생각보다 높습니다", section "INT8 TensorOps 커널 설계",
// steps 1-4.  The few-row variant fills the gap the seq_len rule leaves
// between one token and a full GEMM tile: it is the same weight stream,
// with the dot products of MR activation rows per weight load.
//
// Design (HBM-bound: the weight matrix is read once, as a flat stream).
//  * Each CTA owns a contiguous range of weight rows -- one contiguous range
//    of bytes, cut into 16-byte chunks -- and each of its warps a contiguous
//    segment of that range (a multiple of 32 chunks).  Step j of a warp reads
//    chunks seg + 32 j + lane: 512 contiguous bytes per warp load, and
//    consecutive steps are adjacent, so the row and column of the next step
//    follow from the last by one add and one compare.  Rows need not line up
//    with warps: every warp streams the same number of bytes (to within one
//    step) for any K.
//  * Loads go straight into registers (16-byte non-caching loads): each lane
//    keeps the loads of the next U steps in flight in a rolling register
//    pipeline -- a step's registers are consumed, then reloaded with the step
//    U ahead -- so an SM has 2 CTAs x 256 threads x U x 16 bytes in flight
//    (96 KB at U = 12).  Measured on GB300 this streams at least as fast as
//    shared-memory rings filled by cp.async or by bulk copies.  The unrolled
//    loop body must stay one basic block: a branch between a load and its
//    use makes the compiler wait for the loads in flight where the paths
//    merge (measured: half the bandwidth), so loads and shared-memory adds
//    are predicated in place and the row walk is selects.
//  * When a row is a whole number of 32-chunk steps (K a multiple of 512 for
//    INT8 weights, 1024 for INT4 -- every workload here), each step lies in
//    one row: each lane adds its exact int32 dot products (dp4a) with the
//    activation codes over the steps of a row, and when the row (or the
//    warp's segment) ends the warp reduces them (redux.sync) and lane 0 adds
//    the sum to the row's accumulator in shared memory (with 4 or 8
//    activation rows, every step is reduced: the per-row partials would
//    take the registers the loads need).  Per group, the 4 or 8 lanes of each
//    K-group are reduced with xor shuffles and the group's first lane stores
//    the sum.  Other row lengths take a general walk (a step may meet two or
//    more rows).  int32 sums are exact, so the order of the additions is
//    free.
//  * The dequant runs once the CTA's range is done: y = fp16(float(acc) *
//    (s_a * s_w)) per channel, or the groups rescaled and summed in
//    ascending order per group -- the rounding order of the GEMM path.
//  * The quantized activation rows sit in shared memory.  The fused kernel
//    (M == 1) quantizes the fp16 row itself (every CTA redundantly; the row
//    is a few KB, read from L2) with the same rule as the row quantizer.  It
//    fetches the row with one bulk copy (cp.async.bulk): per-thread loads of
//    x would queue behind the weight loads the SM already has in flight.
//  * Programmatic dependent launch: the kernel lets the next launch on the
//    stream start as soon as all its CTAs run, and each CTA issues its first
//    U loads per lane before griddepcontrol.wait.  Only reads of Wq come
//    before the wait; x, the scales and every write come after it.  Wq must
//    therefore not be written by a kernel that lets this one start early
//    (one that executes griddepcontrol.launch_dependents); the library's
//    kernels that write weights do not.
#include <mutex>

#include "common.cuh"
#include "quant_rule.cuh"

namespace w8a8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCtasPerSm = 2;
constexpr int kAccBytesMax = 32 * 1024;  // per-row (per-group) state per CTA

// Loads in flight per lane: fewer with more activation rows (their partials
// take the registers).  Measured at one activation row, 12 beat 8 and 16
// (26 MB layer back to back: 7.7 / 8.0 / 8.9 us per call).
template <int MR>
constexpr int pipe_depth() {
  return MR <= 4 ? 12 : 8;
}

// Row walks of a warp's segment: kWalkAligned when a row is a whole number
// of 32-chunk steps (every step lies in one row and is full), kWalkWide for
// other rows of at least 32 chunks (a step meets at most two rows),
// kWalkNarrow for shorter rows.
enum Walk { kWalkAligned = 0, kWalkWide = 1, kWalkNarrow = 2 };

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The predicated forms below are single predicated instructions (no branch
// around them), so the unrolled streaming loop stays one basic block.
__device__ __forceinline__ void ldg_stream_if(const uint4 *p, uint4 &v, bool pred) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
      "@p ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n}\n"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "l"(p), "r"(static_cast<int>(pred)));
}

__device__ __forceinline__ void red_shared_if(uint32_t addr, int v, bool pred) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n"
      "@p red.shared.add.s32 [%0], %1;\n}\n" ::"r"(addr),
      "r"(v), "r"(static_cast<int>(pred))
      : "memory");
}

// When `pred` (uniform over the warp): the warp's sum of v, added to the
// shared int32 at addr by the lane with `lane0`.
__device__ __forceinline__ void redux_red_if(uint32_t addr, int v, bool pred, bool lane0) {
  asm volatile(
      "{\n.reg .pred p, q;\n.reg .s32 t;\n"
      "setp.ne.b32 p, %2, 0;\n"
      "@p redux.sync.add.s32 t, %1, 0xffffffff;\n"
      "setp.ne.and.b32 q, %3, 0, p;\n"
      "@q red.shared.add.s32 [%0], t;\n}\n" ::"r"(addr),
      "r"(v), "r"(static_cast<int>(pred)), "r"(static_cast<int>(lane0))
      : "memory");
}

__device__ __forceinline__ void st_shared_if(uint32_t addr, int v, bool pred) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n"
      "@p st.shared.b32 [%0], %1;\n}\n" ::"r"(addr),
      "r"(v), "r"(static_cast<int>(pred))
      : "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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

// Bounded wait for phase 0 of `bar` (the bulk copy of the activation row):
// false after about `limit` cycles.
__device__ __forceinline__ bool wait_copy(uint32_t bar, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, 0u)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ int dot16(const uint4 &w, const uint4 &a) {
  int acc = __dp4a(static_cast<int>(w.x), static_cast<int>(a.x), 0);
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
// nibble of byte i) against the 32 INT8 activations a0, a1 (4 per word).  A
// nibble v in [-8, 7] is read as the unsigned u = v + 8 (top bit flipped), so
// this returns sum_k a_k u_k = sum_k a_k v_k + 8 sum_k a_k; the caller
// subtracts 8 sum_k a_k once per row.  The even nibbles of a word meet
// (a0 a2 a4 a6), the odd ones (a1 a3 a5 a7).
__device__ __forceinline__ int dot32_w4u(const uint4 &w, const uint4 &a0, const uint4 &a1) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  const uint32_t a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  int acc = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t ev = __byte_perm(a[2 * j], a[2 * j + 1], 0x6420);
    const uint32_t od = __byte_perm(a[2 * j], a[2 * j + 1], 0x7531);
    const uint32_t wx = ww[j] ^ 0x88888888u;
    acc = dp4a_su(ev, wx & 0x0f0f0f0fu, acc);
    acc = dp4a_su(od, (wx >> 4) & 0x0f0f0f0fu, acc);
  }
  return acc;
}

// Shared memory: [fused: the fp16 activation row, 2K bytes][MR x K codes]
// [MR x G activation scales][acc: rows x G x MR int32 (rows x G per
// group)][per group: the CTA's weight scales, rows x G fp32].  K is a
// multiple of 16, so the row and the codes are 16-byte aligned and the rest
// 4-byte.
inline size_t mv_state_bytes(int K, int G, int rows, bool pergroup, int mr, bool fused) {
  return (fused ? 2u * K : 0u) + static_cast<size_t>(mr) * K + 4u * mr * G +
         static_cast<size_t>(rows) * G * 4u * (pergroup ? 2 : mr);
}

// Cycles a CTA waits for the bulk copy of its activation row before it
// records a device error (the outputs of that call are then undefined).
constexpr long long kCopyWaitCycles = 2000000000LL;

// FUSED (MR == 1): xin is fp16 x [K] and the CTA quantizes it; otherwise
// xin is int8 codes [M, K] (M <= MR) with scales sa_in [M, G].  WALK is the
// row walk (enum Walk); each walk is its own instantiation, which keeps the
// unrolled loop short.
// y[m, n] = fp16(float(sum_k q_mk w_nk) * (s_a[m] * s_w[n]))        (gs == 0)
// y[n] = fp16(sum_g float(acc_g) * (s_a[g] * s_w[n, g]))              (gs > 0, MR == 1)
template <int WBITS, bool PERGROUP, bool FUSED, int MR, int WALK>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) mv_kernel(
    const void *__restrict__ xin, const float *__restrict__ sa_in,
    const uint8_t *__restrict__ W, const float *__restrict__ sw, int M, int N, int K, int gs,
    __half *__restrict__ y, unsigned int *err) {
  static_assert(!(PERGROUP && MR > 1), "per group: one row");
  // the fused single row is staged by one bulk copy; fused rows of a
  // few-row product are read by one warp each
  constexpr bool STAGED = FUSED && MR == 1;
  constexpr int U = pipe_depth<MR>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int red_i[kWarps][MR];
  __shared__ float red_f[kWarps];
  __shared__ __align__(8) unsigned long long xbar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = PERGROUP ? K / gs : 1;
  const long r0 = static_cast<long>(blockIdx.x) * N / gridDim.x;
  const int rows = static_cast<int>(static_cast<long>(blockIdx.x + 1) * N / gridDim.x - r0);
  const int row_bytes = WBITS == 8 ? K : K / 2;
  const int cpr = row_bytes >> 4;   // chunks per row
  const int nchunk = rows * cpr;     // rows <= 8192: < 2^28
  // this warp's segment [sb, se) of the CTA's chunks
  const int seg = ((nchunk + kWarps - 1) / kWarps + 31) & ~31;
  const int sb = min(warp * seg, nchunk), se = min(sb + seg, nchunk);
  const int nsteps = (se - sb + 31) >> 5;
  const int nseg = se - sb;
  const uint4 *wg = reinterpret_cast<const uint4 *>(W + r0 * row_bytes) + sb + lane;
  const __half *xrow = reinterpret_cast<const __half *>(smem);  // staged fp16 row
  int8_t *xs = reinterpret_cast<int8_t *>(smem + (STAGED ? 2 * K : 0));
  float *ss = reinterpret_cast<float *>(xs + static_cast<size_t>(MR) * K);
  int *acc = reinterpret_cast<int *>(ss + MR * G);
  float *sws = reinterpret_cast<float *>(acc + rows * G * (PERGROUP ? 1 : MR));

  // step j of this lane: chunk sb + 32 j + lane, if inside the segment
  auto load = [&](int j) -> uint4 {
    return 32 * j + lane < nseg ? ldg_stream(wg + 32 * j) : make_uint4(0, 0, 0, 0);
  };

  if (STAGED) {
    if (tid == 0) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&xbar)));
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
  }
  asm volatile("griddepcontrol.launch_dependents;");
  // ---- before the wait: reads of Wq only ----
  uint4 buf[U];
#pragma unroll
  for (int u = 0; u < U; ++u) buf[u] = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (WALK == kWalkAligned)
      ldg_stream_if(wg + 32 * u, buf[u], u < nsteps);
    else
      buf[u] = load(u);
  }
  // everything below may read what the previous kernel on the stream wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (STAGED && tid == 0) {
    // the fp16 row by one bulk copy: it does not queue behind the weight
    // loads this SM has in flight, as per-thread loads of x would
    const uint32_t bytes = 2u * static_cast<uint32_t>(K);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&xbar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem)),
        "l"(xin), "r"(bytes), "r"(smem_u32(&xbar))
        : "memory");
  }

  for (int i = tid; i < rows * G * (PERGROUP ? 1 : MR); i += kThreads) {
    acc[i] = 0;
    if (PERGROUP) sws[i] = __ldg(sw + r0 * G + i);
  }

  // ---- the activation rows: INT8 codes (and scales) into shared memory ----
  const uint4 *xv = static_cast<const uint4 *>(xin);  // fused: the staged row (below)
  int asum[MR];  // W4: this thread's share of sum_k q_mk
#pragma unroll
  for (int m = 0; m < MR; ++m) asum[m] = 0;
  if (FUSED && !STAGED) {
    // each warp quantizes whole rows m = warp, warp + 8, ... (one scale per
    // row: the absmax is a warp reduction, no block barrier); rows m >= M
    // get zero codes and scale 0
    const int nvec = K >> 3;
    for (int m = warp; m < MR; m += kWarps) {
      const uint4 *xr = xv + static_cast<long>(m) * nvec;
      float amax = 0.f;
      if (m < M)
        for (int v = lane; v < nvec; v += 32) amax = fmaxf(amax, absmax8(__ldg(xr + v)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float sm_ = __fdiv_rn(amax, 127.f);
      const float rcp = amax == 0.f ? 0.f : __frcp_rn(sm_);
      if (lane == 0) ss[m] = m < M ? sm_ : 0.f;
      int as = 0;
      for (int v = lane; v < nvec; v += 32) {
        float q[8];
        quant_vec8(m < M ? __ldg(xr + v) : make_uint4(0, 0, 0, 0), sm_, rcp, q);
#pragma unroll
        for (int j = 0; j < 8; ++j) as += __float2int_rn(q[j]);
        reinterpret_cast<uint2 *>(xs + static_cast<long>(m) * K)[v] = pack_i8x8(q);
      }
#pragma unroll
      for (int mm = 0; mm < MR; ++mm)
        if (mm == m) asum[mm] += as;
    }
  } else if (FUSED) {
    if (!wait_copy(smem_u32(&xbar), kCopyWaitCycles)) {
      // record the failure; still let the copy land before going on
      if (err != nullptr) atomicCAS(err, 0u, static_cast<unsigned>(kDevErrRowCopy));
      wait_copy(smem_u32(&xbar), kCopyWaitCycles);
    }
    xv = reinterpret_cast<const uint4 *>(xrow);
    const int nvec = K >> 3;
    float amax_row = 0.f;
    if (!PERGROUP) {
      for (int v = tid; v < nvec; v += kThreads) amax_row = fmaxf(amax_row, absmax8(xv[v]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        amax_row = fmaxf(amax_row, __shfl_xor_sync(0xffffffffu, amax_row, o));
      if (lane == 0) red_f[warp] = amax_row;
      __syncthreads();
      amax_row = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) amax_row = fmaxf(amax_row, red_f[w]);
    }
    const float s_row = __fdiv_rn(amax_row, 127.f);
    const float rcp_row = amax_row == 0.f ? 0.f : __frcp_rn(s_row);
    if (!PERGROUP && tid == 0) ss[0] = s_row;
    // a group of gs is gs / 8 consecutive vectors, i.e. consecutive lanes
    for (int v0 = 0; v0 < nvec; v0 += kThreads) {
      const int v = v0 + tid;
      const uint4 xvv = v < nvec ? xv[v] : make_uint4(0, 0, 0, 0);
      float s = s_row, rcp = rcp_row;
      if (PERGROUP) {
        float m = absmax8(xvv);
        for (int o = (gs >> 4); o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        s = __fdiv_rn(m, 127.f);
        rcp = m == 0.f ? 0.f : __frcp_rn(s);
        if (v < nvec && (tid & ((gs >> 3) - 1)) == 0) ss[(v << 3) / gs] = s;
      }
      if (v < nvec) {
        float q[8];
        quant_vec8(xvv, s, rcp, q);
#pragma unroll
        for (int j = 0; j < 8; ++j) asum[0] += __float2int_rn(q[j]);
        reinterpret_cast<uint2 *>(xs)[v] = pack_i8x8(q);
      }
    }
  } else {
    // rows m >= M are zero codes (their partials stay 0 and are not stored)
    const int kvec = K >> 4;
    for (int i = tid; i < MR * kvec; i += kThreads) {
      const int m = i / kvec;
      const uint4 q = m < M ? __ldg(xv + i) : make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4 *>(xs)[i] = q;
      if (WBITS == 4) {
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) {
          if (mm == m) {
            asum[mm] = __dp4a(static_cast<int>(q.x), 0x01010101, asum[mm]);
            asum[mm] = __dp4a(static_cast<int>(q.y), 0x01010101, asum[mm]);
            asum[mm] = __dp4a(static_cast<int>(q.z), 0x01010101, asum[mm]);
            asum[mm] = __dp4a(static_cast<int>(q.w), 0x01010101, asum[mm]);
          }
        }
      }
    }
    for (int i = tid; i < M * G; i += kThreads) ss[i] = __ldg(sa_in + i);
  }
  if (WBITS == 4) {
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      asum[m] = __reduce_add_sync(0xffffffffu, asum[m]);
      if (lane == 0) red_i[warp][m] = asum[m];
    }
  }
  __syncthreads();
  int asum_row[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    asum_row[m] = 0;
    if (WBITS == 4) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) asum_row[m] += red_i[w][m];
    }
  }

  // ---- the dot products of this warp's segment ----
  const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
  const int kv = K >> 4;                       // 16-byte code vectors per activation row
  int crow = sb / cpr, ckc = sb - crow * cpr;  // row and column of lane 0's chunk
  const int q32 = 32 / cpr, r32 = 32 % cpr;    // one step = 32 chunks
  constexpr bool wide = WALK == kWalkWide;     // a step meets at most two rows
  int R = crow;                                // partials of rows R and R + 1
  int accA[MR], accB[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) accA[m] = accB[m] = 0;
  auto step = [&](int j, const uint4 &w) {
    const bool in = 32 * j + lane < nseg;
    int rl = crow, kl = ckc + lane;
    if (wide) {
      if (kl >= cpr) {
        kl -= cpr;
        ++rl;
      }
    } else {
      rl += kl / cpr;
      kl -= (kl / cpr) * cpr;
    }
    int d[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      d[m] = 0;
      if (in) {
        if (WBITS == 8)
          d[m] = dot16(w, xs4[m * kv + kl]);
        else
          d[m] = dot32_w4u(w, xs4[m * kv + 2 * kl], xs4[m * kv + 2 * kl + 1]);
      }
    }
    if (PERGROUP) {
      // groups are aligned runs of cpg lanes (segments and cpr are multiples of cpg)
      const int cpg = gs >> 4;
      int dd = d[0];
      for (int o = cpg >> 1; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
      if (in && (lane & (cpg - 1)) == 0) atomicAdd(acc + rl * G + kl / cpg, dd);
    } else if (wide) {
      if (crow != R) {  // the warp has left row R (crow == R + 1)
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const int t = __reduce_add_sync(0xffffffffu, accA[m]);
          if (lane == 0) atomicAdd(acc + R * MR + m, t);
          accA[m] = accB[m];
          accB[m] = 0;
        }
        R = crow;
      }
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        if (rl == R)
          accA[m] += d[m];
        else
          accB[m] += d[m];
      }
    } else {
      const int rlast = min(__shfl_sync(0xffffffffu, rl, 31), rows - 1);
      for (int r = crow; r <= rlast; ++r) {
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const int t = __reduce_add_sync(0xffffffffu, rl == r ? d[m] : 0);
          if (lane == 0) atomicAdd(acc + r * MR + m, t);
        }
      }
    }
    crow += q32;
    ckc += r32;
    if (ckc >= cpr) {
      ckc -= cpr;
      ++crow;
    }
  };

  // rolling pipeline: consume step j from its registers, reload them with
  // step j + U (the loads of U steps stay in flight)
  if (WALK == kWalkAligned) {
    // Every step is 32 whole chunks of one row.  The unrolled body has no
    // branch: a conditional block between a load and its use makes the
    // compiler wait for the loads in flight where the paths merge, which
    // took the prefetch depth down to about one load per lane (measured:
    // half the bandwidth).  So the loads and the shared-memory adds are
    // predicated in place, the row walk is selects, and each step's dot
    // products are reduced over the warp (one redux per activation row)
    // and added to the row's accumulator by lane 0.  Per group, each
    // K-group is an aligned run of cpg lanes of one step: its sum (xor
    // shuffles) is stored by the run's first lane, and by no other step.
    int row = crow, col = ckc;
    const uint32_t acc_s = smem_u32(acc);
    // per channel with one or two activation rows, each lane sums its dot
    // products over the steps of a row and the warp reduces once per row
    // (when the row ends, or the segment); with more rows (their partials
    // would take the registers) the warp reduces every step
    constexpr bool ROWSUM = MR <= 2;
    int racc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) racc[m] = 0;
    for (int j0 = 0; j0 < nsteps; j0 += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u;
        const bool valid = j < nsteps;  // uniform over the warp
        const int kl = col + lane;      // in [0, cpr) whatever j is
        const int c2 = col + 32;
        const bool wrap = c2 == cpr;    // this step ends its row
        if (PERGROUP) {
          const int cpg = gs >> 4;
          int d = dot16(buf[u], xs4[kl]);
          for (int o = cpg >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          st_shared_if(acc_s + 4u * static_cast<uint32_t>(row * G + kl / cpg), d,
                       valid && (lane & (cpg - 1)) == 0);
        } else {
#pragma unroll
          for (int m = 0; m < MR; ++m) {
            const int d = WBITS == 8 ? dot16(buf[u], xs4[m * kv + kl])
                                     : dot32_w4u(buf[u], xs4[m * kv + 2 * kl],
                                                 xs4[m * kv + 2 * kl + 1]);
            if (ROWSUM) {
              racc[m] += valid ? d : 0;
              redux_red_if(acc_s + 4u * static_cast<uint32_t>(row * MR + m), racc[m],
                           valid && wrap, lane == 0);
              racc[m] = valid && wrap ? 0 : racc[m];
            } else {
              const int t = __reduce_add_sync(0xffffffffu, d);
              red_shared_if(acc_s + 4u * static_cast<uint32_t>(row * MR + m), t,
                            valid && lane == 0);
            }
          }
        }
        ldg_stream_if(wg + 32 * (j + U), buf[u], j + U < nsteps);
        col = valid ? (wrap ? 0 : c2) : col;
        row += valid && wrap ? 1 : 0;
      }
    }
    // the row the segment ends in, when it ends inside one
    if (!PERGROUP && ROWSUM) {
#pragma unroll
      for (int m = 0; m < MR; ++m)
        redux_red_if(acc_s + 4u * static_cast<uint32_t>(row * MR + m), racc[m], row < rows,
                     lane == 0);
    }
  } else {
    for (int j0 = 0; j0 < nsteps; j0 += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u;
        if (j < nsteps) step(j, buf[u]);
        buf[u] = load(j + U);
      }
    }
  }
  if (!PERGROUP && wide && nsteps > 0) {
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      const int ta = __reduce_add_sync(0xffffffffu, accA[m]);
      const int tb = __reduce_add_sync(0xffffffffu, accB[m]);
      if (lane == 0) {
        atomicAdd(acc + R * MR + m, ta);
        if (R + 1 < rows) atomicAdd(acc + (R + 1) * MR + m, tb);
      }
    }
  }
  __syncthreads();

  // ---- dequant ----
  for (int r = tid; r < rows; r += kThreads) {
    const long n = r0 + r;
    if (!PERGROUP) {
      const float swn = __ldg(sw + n);
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        if (m < M) {
          const int tot = acc[r * MR + m] - (WBITS == 4 ? 8 * asum_row[m] : 0);
          y[static_cast<long>(m) * N + n] =
              __float2half_rn(__fmul_rn(static_cast<float>(tot), __fmul_rn(ss[m], swn)));
        }
      }
    } else {
      float f = 0.f;
      for (int g = 0; g < G; ++g)
        f = __fadd_rn(f, __fmul_rn(static_cast<float>(acc[r * G + g]), __fmul_rn(ss[g], sws[r * G + g])));
      y[n] = __float2half_rn(f);
    }
  }
}

template <int WBITS, bool PERGROUP, bool FUSED, int MR, int WALK>
int launch_mv_t(const void *xin, const float *sa, const void *W, const float *sw, int M, int N,
                int K, int gs, __half *y, cudaStream_t s) {
  // per device: the shared-memory attribute set once, and the SM count
  static bool attr_set[64] = {};
  static int sms[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W8A8_ERR_CUDA;
  const int G = PERGROUP ? K / gs : 1;
  const int per_row = G * 4 * (PERGROUP ? 2 : MR);  // shared bytes per weight row
  int nsm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      const size_t most = MR == 1 ? mv_state_bytes(kMaxK, kMaxK / 64, 0, PERGROUP, 1, FUSED)
                                  : static_cast<size_t>(kSkinnyMaxCodeBytes) + 4 * MR;  // not staged
      if (cudaFuncSetAttribute(mv_kernel<WBITS, PERGROUP, FUSED, MR, WALK>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(most + kAccBytesMax)) != cudaSuccess)
        return W8A8_ERR_CUDA;
      if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return W8A8_ERR_CUDA;
      attr_set[dev] = true;
    }
    nsm = sms[dev];
  }
  // kCtasPerSm CTAs per SM, more when a CTA's rows would not fit its shared
  // state (at most kAccBytesMax bytes)
  const long rows_cap = kAccBytesMax / per_row;
  long grid = static_cast<long>(kCtasPerSm) * nsm;
  const long need = (N + rows_cap - 1) / rows_cap;
  if (grid < need) grid = need;
  if (grid > N) grid = N;
  const int rows_max = static_cast<int>((N + grid - 1) / grid);
  const size_t smem = mv_state_bytes(K, G, rows_max, PERGROUP, MR, FUSED && MR == 1);
  unsigned int *err = device_error_word();
  if (err == nullptr) return W8A8_ERR_CUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mv_kernel<WBITS, PERGROUP, FUSED, MR, WALK>, xin, sa,
                         static_cast<const uint8_t *>(W), sw, M, N, K, gs, y, err) != cudaSuccess) {
    cudaGetLastError();
    return W8A8_ERR_CUDA;
  }
  return launch_status();
}

// the row walk from the row length in 16-byte chunks
template <int WBITS, bool PERGROUP, bool FUSED, int MR>
int launch_mv(const void *xin, const float *sa, const void *W, const float *sw, int M, int N,
              int K, int gs, __half *y, cudaStream_t s) {
  const int cpr = (WBITS == 8 ? K : K / 2) >> 4;
  if (cpr % 32 == 0)
    return launch_mv_t<WBITS, PERGROUP, FUSED, MR, kWalkAligned>(xin, sa, W, sw, M, N, K, gs, y, s);
  if (cpr >= 32)
    return launch_mv_t<WBITS, PERGROUP, FUSED, MR, kWalkWide>(xin, sa, W, sw, M, N, K, gs, y, s);
  return launch_mv_t<WBITS, PERGROUP, FUSED, MR, kWalkNarrow>(xin, sa, W, sw, M, N, K, gs, y, s);
}

template <int WBITS, int MR>
int launch_rows(const int8_t *xq, const float *sa, const void *W, const float *sw, int M, int N,
                int K, __half *y, cudaStream_t s) {
  return launch_mv<WBITS, false, false, MR>(xq, sa, W, sw, M, N, K, 0, y, s);
}

template <int WBITS, int MR>
int launch_rows_fused(const __half *x, const void *W, const float *sw, int M, int N, int K,
                      __half *y, cudaStream_t s) {
  return launch_mv<WBITS, false, true, MR>(x, nullptr, W, sw, M, N, K, 0, y, s);
}

}  // namespace

int launch_gemv_w8a8(const int8_t *xq, const float *sa, const int8_t *Wq,
                     const float *sw, int N, int K, int group_size, __half *y,
                     cudaStream_t s) {
  if (group_size != 0)
    return launch_mv<8, true, false, 1>(xq, sa, Wq, sw, 1, N, K, group_size, y, s);
  return launch_mv<8, false, false, 1>(xq, sa, Wq, sw, 1, N, K, 0, y, s);
}

int launch_gemv_w4a8(const int8_t *xq, const float *sa, const uint8_t *Wp,
                     const float *sw, int N, int K, __half *y, cudaStream_t s) {
  return launch_mv<4, false, false, 1>(xq, sa, Wp, sw, 1, N, K, 0, y, s);
}

int launch_linear_mv(const __half *x, const void *W, const float *sw, int N, int K,
                     int group_size, int wbits, __half *y, cudaStream_t s) {
  if (wbits == 4) return launch_mv<4, false, true, 1>(x, nullptr, W, sw, 1, N, K, 0, y, s);
  if (group_size != 0)
    return launch_mv<8, true, true, 1>(x, nullptr, W, sw, 1, N, K, group_size, y, s);
  return launch_mv<8, false, true, 1>(x, nullptr, W, sw, 1, N, K, 0, y, s);
}

int skinny_rows(int M) { return M <= 2 ? 2 : M <= 4 ? 4 : 8; }

bool skinny_supported(int M, int K, int group_size) {
  return M >= 2 && M <= kSkinnyMaxM && group_size == 0 &&
         static_cast<long>(skinny_rows(M)) * K <= kSkinnyMaxCodeBytes;
}

int launch_skinny(const int8_t *xq, const float *sa, const void *W, const float *sw, int M, int N,
                  int K, int wbits, __half *y, cudaStream_t s) {
  switch (skinny_rows(M)) {
    case 2:
      return wbits == 4 ? launch_rows<4, 2>(xq, sa, W, sw, M, N, K, y, s)
                        : launch_rows<8, 2>(xq, sa, W, sw, M, N, K, y, s);
    case 4:
      return wbits == 4 ? launch_rows<4, 4>(xq, sa, W, sw, M, N, K, y, s)
                        : launch_rows<8, 4>(xq, sa, W, sw, M, N, K, y, s);
    default:
      return wbits == 4 ? launch_rows<4, 8>(xq, sa, W, sw, M, N, K, y, s)
                        : launch_rows<8, 8>(xq, sa, W, sw, M, N, K, y, s);
  }
}

int launch_linear_rows(const __half *x, const void *W, const float *sw, int M, int N, int K,
                       int wbits, __half *y, cudaStream_t s) {
  switch (skinny_rows(M)) {
    case 2:
      return wbits == 4 ? launch_rows_fused<4, 2>(x, W, sw, M, N, K, y, s)
                        : launch_rows_fused<8, 2>(x, W, sw, M, N, K, y, s);
    case 4:
      return wbits == 4 ? launch_rows_fused<4, 4>(x, W, sw, M, N, K, y, s)
                        : launch_rows_fused<8, 4>(x, W, sw, M, N, K, y, s);
    default:
      return wbits == 4 ? launch_rows_fused<4, 8>(x, W, sw, M, N, K, y, s)
                        : launch_rows_fused<8, 8>(x, W, sw, M, N, K, y, s);
  }
}

}  // namespace w8a8
