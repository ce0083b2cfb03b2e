// Decode-path matrix-vector kernels (M == 1): W8A8 per channel / per group,
// and W4A8 per channel; optionally fused with the activation quantization.
//
// Method: "cider 소개", section "cider의 동작 방식과 자동 경로 선택"
// (CiderLinear picks the INT8 MV kernel when seq_len == 1; the kernel list
// names a per-channel and a per-group MV kernel); "Apple Silicon의 AI
// 한계치는 당신의 생각보다 높습니다", section "INT8 TensorOps 커널 설계",
// steps 1-4.
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
//  * Loads go global -> shared memory by per-thread asynchronous copies
//    (cp.async, 16 bytes each): a stage is kU steps of a warp, each lane
//    copies and later reads its own 16 bytes of each step (no cross-lane
//    hand-off), and kD stages are in flight per thread, so an SM keeps
//    kCtasPerSm * kThreads * kD * kU * 16 bytes in flight without holding
//    registers for them, and the dot products of one stage overlap the
//    copies of the next ones.  The first kD stages are issued before
//    griddepcontrol.wait (see below).
//  * Per channel (rows of 32 chunks or more), a warp load meets at most two
//    rows: each lane adds its chunk's exact int32 dot product (dp4a) with the
//    activation codes into one of two register partials (this row, next
//    row), and when the warp moves past a row the partial of that row is
//    reduced over the warp (redux.sync) and added to the row's int32
//    accumulator in shared memory -- one reduction per row and warp.  Per
//    group, each step reduces the 4 or 8 lanes of every K-group (xor
//    shuffles) and adds the group sums to the row-and-group accumulators.
//    int32 sums are exact, so the order of these additions is free.
//  * The dequant runs once the CTA's range is done: y = fp16(float(acc) *
//    (s_a * s_w)) per channel, or the groups rescaled and summed in
//    ascending order per group -- the rounding order of the GEMM path.
//  * The quantized activation row sits in shared memory.  The fused kernel
//    quantizes the fp16 row itself (every CTA redundantly; the row is a few
//    KB, read from L2) with the same rule as the row quantizer.
//  * Programmatic dependent launch: the kernel lets the next launch on the
//    stream start as soon as all its CTAs run, and two kernels' CTAs fit on
//    an SM together.  Only reads of Wq come before griddepcontrol.wait; x,
//    the scales and every write come after it.  Wq must therefore not be
//    written by a kernel that lets this one start early (one that executes
//    griddepcontrol.launch_dependents); the library's kernels that write
//    weights do not.
#include <mutex>

#include "common.cuh"
#include "quant_rule.cuh"

namespace w8a8 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
#ifndef W8A8_MV_STAGE_STEPS
constexpr int kU = 4;  // warp steps (32 chunks of 16 bytes) per stage
#else
constexpr int kU = W8A8_MV_STAGE_STEPS;
#endif
#ifndef W8A8_MV_STAGES
constexpr int kD = 3;  // stages in flight per thread
#else
constexpr int kD = W8A8_MV_STAGES;
#endif
#ifndef W8A8_MV_CTAS_PER_SM
constexpr int kCtasPerSm = 2;
#else
constexpr int kCtasPerSm = W8A8_MV_CTAS_PER_SM;
#endif
constexpr int kAccBytesMax = 32 * 1024;  // per-row (per-group) state per CTA
constexpr int kRingBytes = kThreads * kD * kU * 16;  // per CTA

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (L2 only), and its groups
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

// Shared memory: [ring: kRingBytes][K codes][G activation scales][acc: rows
// x G int32][per group: the CTA's weight scales, rows x G fp32].  The ring
// and K are multiples of 16, so the ring and the codes are 16-byte aligned
// and the rest 4-byte.
inline size_t mv_state_bytes(int K, int G, int rows, bool pergroup) {
  return static_cast<size_t>(K) + 4u * G + static_cast<size_t>(rows) * G * 4u * (pergroup ? 2 : 1);
}

// FUSED: xin is fp16 x [K] and the CTA quantizes it; otherwise xin is int8
// codes [K] with scales sa_in [G].
// y[n] = fp16(float(sum_k q_k w_nk) * (s_a * s_w[n]))            (gs == 0)
// y[n] = fp16(sum_g float(acc_g) * (s_a[g] * s_w[n, g]))          (gs > 0)
template <int WBITS, bool PERGROUP, bool FUSED>
__global__ void __launch_bounds__(kThreads, 2 * kCtasPerSm) mv_kernel(
    const void *__restrict__ xin, const float *__restrict__ sa_in,
    const uint8_t *__restrict__ W, const float *__restrict__ sw, int N, int K, int gs,
    __half *__restrict__ y) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int red_i[kWarps];
  __shared__ float red_f[kWarps];
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
  const int nst = (nsteps + kU - 1) / kU;  // stages
  const uint4 *wg = reinterpret_cast<const uint4 *>(W + r0 * row_bytes) + sb;
  // this warp's kD stage buffers; step u of a stage is 512 bytes, lane-major
  uint8_t *ring = smem + warp * (kD * kU * 512);
  int8_t *xs = reinterpret_cast<int8_t *>(smem + kRingBytes);
  float *ss = reinterpret_cast<float *>(xs + K);
  int *acc = reinterpret_cast<int *>(ss + G);
  float *sws = reinterpret_cast<float *>(acc + rows * G);

  // stage t: this lane's chunk of steps t * kU + u; a group is committed
  // even when empty, so that "all but the newest kD - 1 groups" is stage t
  auto issue = [&](int t) {
    if (t < nst) {
      const uint32_t b = smem_u32(ring + (t % kD) * (kU * 512) + lane * 16);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = 32 * (t * kU + u) + lane;
        if (sb + c < se) cp_async16(b + u * 512, wg + c);
      }
    }
    cp_async_commit();
  };

  asm volatile("griddepcontrol.launch_dependents;");
  // ---- before the wait: reads of Wq only ----
#pragma unroll
  for (int t = 0; t < kD; ++t) issue(t);
  // everything below may read what the previous kernel on the stream wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int i = tid; i < rows * G; i += kThreads) {
    acc[i] = 0;
    if (PERGROUP) sws[i] = __ldg(sw + r0 * G + i);
  }

  // ---- the activation row: INT8 codes (and scales) into shared memory ----
  const uint4 *xv = static_cast<const uint4 *>(xin);
  int asum = 0;  // W4: this thread's share of sum_k q_k
  if (FUSED) {
    const int nvec = K >> 3;
    float amax_row = 0.f;
    if (!PERGROUP) {
      for (int v = tid; v < nvec; v += kThreads) amax_row = fmaxf(amax_row, absmax8(__ldg(xv + v)));
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
        float q[8];
        quant_vec8(xvv, s, rcp, q);
#pragma unroll
        for (int j = 0; j < 8; ++j) asum += __float2int_rn(q[j]);
        reinterpret_cast<uint2 *>(xs)[v] = pack_i8x8(q);
      }
    }
  } else {
    for (int v = tid; v < (K >> 4); v += kThreads) {
      const uint4 q = __ldg(xv + v);
      reinterpret_cast<uint4 *>(xs)[v] = q;
      if (WBITS == 4) {
        asum = __dp4a(static_cast<int>(q.x), 0x01010101, asum);
        asum = __dp4a(static_cast<int>(q.y), 0x01010101, asum);
        asum = __dp4a(static_cast<int>(q.z), 0x01010101, asum);
        asum = __dp4a(static_cast<int>(q.w), 0x01010101, asum);
      }
    }
    for (int g = tid; g < G; g += kThreads) ss[g] = __ldg(sa_in + g);
  }
  if (WBITS == 4) {
    asum = __reduce_add_sync(0xffffffffu, asum);
    if (lane == 0) red_i[warp] = asum;
  }
  __syncthreads();
  int asum_row = 0;
  if (WBITS == 4) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) asum_row += red_i[w];
  }

  // ---- the dot products of this warp's segment ----
  const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
  int crow = sb / cpr, ckc = sb - crow * cpr;  // row and column of lane 0's chunk
  const int q32 = 32 / cpr, r32 = 32 % cpr;   // one step = 32 chunks
  const bool wide = cpr >= 32;                // a step meets at most two rows
  int R = crow, accA = 0, accB = 0;           // partials of rows R and R + 1
  auto step = [&](int j, const uint4 &w) {
    const bool in = sb + 32 * j + lane < se;
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
    int d = 0;
    if (in) {
      if (WBITS == 8)
        d = dot16(w, xs4[kl]);
      else
        d = dot32_w4u(w, xs4[2 * kl], xs4[2 * kl + 1]);
    }
    if (PERGROUP) {
      // groups are aligned runs of cpg lanes (segments and cpr are multiples of cpg)
      const int cpg = gs >> 4;
      for (int o = cpg >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (in && (lane & (cpg - 1)) == 0) atomicAdd(acc + rl * G + kl / cpg, d);
    } else if (wide) {
      if (crow != R) {  // the warp has left row R (crow == R + 1)
        accA = __reduce_add_sync(0xffffffffu, accA);
        if (lane == 0) atomicAdd(acc + R, accA);
        accA = accB;
        accB = 0;
        R = crow;
      }
      if (rl == R)
        accA += d;
      else
        accB += d;
    } else {
      const int rlast = min(__shfl_sync(0xffffffffu, rl, 31), rows - 1);
      for (int r = crow; r <= rlast; ++r) {
        const int s = __reduce_add_sync(0xffffffffu, rl == r ? d : 0);
        if (lane == 0) atomicAdd(acc + r, s);
      }
    }
    crow += q32;
    ckc += r32;
    if (ckc >= cpr) {
      ckc -= cpr;
      ++crow;
    }
  };

  for (int t = 0; t < nst; ++t) {
    cp_async_wait<kD - 1>();  // this lane's copies of stage t have landed
    const uint4 *b = reinterpret_cast<const uint4 *>(ring + (t % kD) * (kU * 512)) + lane;
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (t * kU + u < nsteps) step(t * kU + u, b[u * 32]);
    issue(t + kD);  // into the buffer just read (by this lane only)
  }
  cp_async_wait<0>();
  if (!PERGROUP && wide && nsteps > 0) {
    accA = __reduce_add_sync(0xffffffffu, accA);
    accB = __reduce_add_sync(0xffffffffu, accB);
    if (lane == 0) {
      atomicAdd(acc + R, accA);
      if (R + 1 < rows) atomicAdd(acc + R + 1, accB);
    }
  }
  __syncthreads();

  // ---- dequant ----
  for (int r = tid; r < rows; r += kThreads) {
    const long n = r0 + r;
    if (!PERGROUP) {
      const int tot = acc[r] - (WBITS == 4 ? 8 * asum_row : 0);
      y[n] = __float2half_rn(__fmul_rn(static_cast<float>(tot), __fmul_rn(ss[0], __ldg(sw + n))));
    } else {
      float f = 0.f;
      for (int g = 0; g < G; ++g)
        f = __fadd_rn(f, __fmul_rn(static_cast<float>(acc[r * G + g]), __fmul_rn(ss[g], sws[r * G + g])));
      y[n] = __float2half_rn(f);
    }
  }
}

template <int WBITS, bool PERGROUP, bool FUSED>
int launch_mv(const void *xin, const float *sa, const void *W, const float *sw, int N, int K,
              int gs, __half *y, cudaStream_t s) {
  // per device: the shared-memory attribute set once, and the SM count
  static bool attr_set[64] = {};
  static int sms[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W8A8_ERR_CUDA;
  const int G = PERGROUP ? K / gs : 1;
  const int per_row = G * 4 * (PERGROUP ? 2 : 1);  // shared bytes per weight row
  int nsm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(mv_kernel<WBITS, PERGROUP, FUSED>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kRingBytes + kMaxK + 4 * (kMaxK / 64) + kAccBytesMax) !=
          cudaSuccess)
        return W8A8_ERR_CUDA;
      if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return W8A8_ERR_CUDA;
      attr_set[dev] = true;
    }
    nsm = sms[dev];
  }
  // kCtasPerSm CTAs per SM, more when a CTA's rows would not fit its shared
  // state (at most kAccBytesMax bytes, i.e. at most 8192 rows)
  const long rows_cap = kAccBytesMax / per_row;
  long grid = static_cast<long>(kCtasPerSm) * nsm;
  const long need = (N + rows_cap - 1) / rows_cap;
  if (grid < need) grid = need;
  if (grid > N) grid = N;
  const int rows_max = static_cast<int>((N + grid - 1) / grid);
  const size_t state = mv_state_bytes(K, G, rows_max, PERGROUP);
  const size_t smem = kRingBytes + state;

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
  if (cudaLaunchKernelEx(&cfg, mv_kernel<WBITS, PERGROUP, FUSED>, xin, sa,
                         static_cast<const uint8_t *>(W), sw, N, K, gs, y) != cudaSuccess) {
    cudaGetLastError();
    return W8A8_ERR_CUDA;
  }
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
