// Row quantization kernels: online per-token activation quantization and the
// offline INT8 / INT4 weight quantizers share one kernel.
//
// Method: "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다", section
// "INT8 TensorOps 커널 설계", steps 1-2 (a fast min/max reduction gives each
// row -- or each group of 64 / 128 elements, section "입도(Granularity)" --
// its scale; one streaming pass maps fp16 to INT8); "cider 소개", section
// "cider의 양자화 모드와 적용 가능한 영역" (symmetric INT8 per token; INT4
// weights packed two per uint8 for W4A8).
//
// Design (HBM-bound, one streaming pass): a team of T threads (32 to 256,
// so that each thread caches at most 4 vectors where K allows) owns a row.
// Activation codes (INT8 or fp16, K <= 8192) and INT8 weights run on a
// persistent grid whose teams take row after row, each loading its next row
// while it quantizes the current one (row_quant_rows); INT4 weights and
// longer rows launch one team per row (row_quant_kernel).  Each thread
// loads its V 16-byte vectors (8 fp16 each) once into registers, the team
// reduces absmax with warp shuffles (and shared memory when T > 32), and the
// same registers are quantized and stored.  Vector i of thread t covers
// elements [8 (i T + t), 8 (i T + t) + 8): consecutive lanes read consecutive
// 16-byte chunks, so every warp load is one coalesced 512-byte transaction,
// and a group of 64 / 128 elements is 8 / 16 consecutive lanes of one warp,
// reduced with xor shuffles inside the warp.
//
// Outputs: INT8 codes (8-byte stores), the same codes as fp16 values (16-byte
// stores; the operand format of the tensor-core GEMM, every code being an
// fp16 integer exactly), or INT4 codes packed two per byte.
//
// Rounding: see quant_rule.cuh.
#include <mutex>

#include "common.cuh"
#include "quant_rule.cuh"

namespace w8a8 {
namespace {

enum OutMode { kOutInt8 = 0, kOutHalf = 1, kOutInt4 = 2 };

// Resident CTAs per SM to aim for: the loads in flight (the only latency
// hiding this one-pass kernel has) scale with it.  Five CTAs (<= 51
// registers) measured best where each thread holds at most 4 vectors; more
// vectors keep the register count they need.
template <int V>
constexpr int quant_min_blocks() {
  return V <= 4 ? 5 : V <= 7 ? 3 : V <= 14 ? 2 : 1;
}

template <int V, int MODE>
__global__ void __launch_bounds__(256, quant_min_blocks<V>()) row_quant_kernel(
    const uint4 *__restrict__ x, long R, int K, int gs, int qmax, int T,
    void *__restrict__ out, float *__restrict__ scale) {
  // activation codes for the GEMM: let it launch now and run its prologue
  // while this grid finishes (it waits for this grid before reading any
  // input); the weight quantizers (other modes) never start dependents early
  if (MODE == kOutHalf) asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float red[8];
  const int nvec = K >> 3;
  const int t = threadIdx.x % T;
  const int team = threadIdx.x / T;
  const long r = static_cast<long>(blockIdx.x) * (blockDim.x / T) + team;
  const bool active = r < R;
  const int G = gs == 0 ? 1 : K / gs;

  uint4 v[V];
  float vmax[V];
  const uint4 *xr = x + r * nvec;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int vi = i * T + t;
    if (active && vi < nvec) {
      v[i] = __ldcs(xr + vi);
    } else {
      v[i] = make_uint4(0, 0, 0, 0);
    }
    vmax[i] = absmax8(v[i]);
  }

  float amax_row = 0.f;
  if (gs == 0) {
#pragma unroll
    for (int i = 0; i < V; ++i) amax_row = fmaxf(amax_row, vmax[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      amax_row = fmaxf(amax_row, __shfl_xor_sync(0xffffffffu, amax_row, o));
    if (T > 32) {
      const int warp = threadIdx.x >> 5;
      if ((threadIdx.x & 31) == 0) red[warp] = amax_row;
      __syncthreads();
      const int w0 = team * (T >> 5);
      amax_row = 0.f;
      for (int w = 0; w < (T >> 5); ++w) amax_row = fmaxf(amax_row, red[w0 + w]);
    }
  } else {
    // a group is gs/8 consecutive lanes of one warp
    const int width = gs >> 3;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      for (int o = width >> 1; o > 0; o >>= 1)
        vmax[i] = fmaxf(vmax[i], __shfl_xor_sync(0xffffffffu, vmax[i], o));
    }
  }
  if (!active) return;

  const float fq = static_cast<float>(qmax);
  const float s_row = __fdiv_rn(amax_row, fq);
  const float rcp_row = amax_row == 0.f ? 0.f : __frcp_rn(s_row);
  if (gs == 0 && t == 0) scale[r] = s_row;

#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int vi = i * T + t;
    if (vi >= nvec) continue;
    float s = s_row, rcp = rcp_row;
    if (gs != 0) {
      s = __fdiv_rn(vmax[i], fq);
      rcp = vmax[i] == 0.f ? 0.f : __frcp_rn(s);
      const int g = (vi << 3) / gs;
      if ((t & ((gs >> 3) - 1)) == 0) scale[r * G + g] = s;
    }
    // a zero row or group has s = 0 and rcp = 0: t = 0 and every code is 0
    float q[8];
    quant_vec8(v[i], s, rcp, q);
    if (MODE == kOutInt8) {
      reinterpret_cast<uint2 *>(static_cast<int8_t *>(out) + r * K)[vi] = pack_i8x8(q);
    } else if (MODE == kOutHalf) {
      // integral codes of magnitude <= 127 are fp16 values exactly
      reinterpret_cast<uint4 *>(static_cast<__half *>(out) + r * K)[vi] = pack_h8(q);
    } else {
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) w |= (static_cast<uint32_t>(__float2int_rn(q[j])) & 0xfu) << (4 * j);
      static_cast<uint32_t *>(out)[r * (K >> 3) + vi] = w;
    }
  }
}

// Activation quantization (INT8 codes, or the same codes as fp16 values) as
// a persistent grid: team g of T
// threads owns rows g, g + nteams, ... and loads its next row while it
// quantizes the current one, so every SM keeps two rows per team in flight
// and no CTA is launched per row.  Per token, the team's absmax goes through
// a named barrier of its own T threads (teams leave the loop independently),
// with the shared partials double-buffered by row parity; per group (gs > 0)
// a group is gs / 8 consecutive lanes of one warp, reduced with shuffles.
template <int V, bool PG, int MODE>
__global__ void __launch_bounds__(256, V <= 2 ? 4 : 3) row_quant_rows(const uint4 *__restrict__ x, long R,
                                                        int K, int gs, int T,
                                                        void *__restrict__ out,
                                                        float *__restrict__ scale) {
  static_assert(MODE == kOutHalf || MODE == kOutInt8, "activation modes");
  // fp16 codes feed the GEMM: let it launch now (it waits for this grid
  // before reading any input); the INT8 mode never starts dependents early
  if (MODE == kOutHalf) asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float red[2][8];
  const int nvec = K >> 3;
  const int G = gs == 0 ? 1 : K / gs;
  const int t = threadIdx.x % T, team = threadIdx.x / T, teams = blockDim.x / T;
  const int warp = threadIdx.x >> 5, wpt = T >> 5;
  const long nteams = static_cast<long>(gridDim.x) * teams;
  long r = static_cast<long>(blockIdx.x) * teams + team;
  auto load = [&](long row, uint4 (&v)[V]) {
    const uint4 *xr = x + row * nvec;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int vi = i * T + t;
      v[i] = (row < R && vi < nvec) ? __ldcs(xr + vi) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 cur[V], nxt[V];
  load(r, cur);
  for (int it = 0; r < R; r += nteams, ++it) {
    load(r + nteams, nxt);
    float vmax[V];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      vmax[i] = absmax8(cur[i]);
      amax = fmaxf(amax, vmax[i]);
    }
    if (!PG) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (T > 32) {
        if ((threadIdx.x & 31) == 0) red[it & 1][warp] = amax;
        asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(T) : "memory");
        amax = 0.f;
        for (int w = 0; w < wpt; ++w) amax = fmaxf(amax, red[it & 1][team * wpt + w]);
      }
    } else {
      const int width = gs >> 3;
#pragma unroll
      for (int i = 0; i < V; ++i)
        for (int o = width >> 1; o > 0; o >>= 1)
          vmax[i] = fmaxf(vmax[i], __shfl_xor_sync(0xffffffffu, vmax[i], o));
    }
    const float s_row = __fdiv_rn(amax, 127.f);
    const float rcp_row = amax == 0.f ? 0.f : __frcp_rn(s_row);
    if (!PG && t == 0) scale[r] = s_row;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int vi = i * T + t;
      if (vi < nvec) {
        float sc = s_row, rc = rcp_row;
        if (PG) {
          sc = __fdiv_rn(vmax[i], 127.f);
          rc = vmax[i] == 0.f ? 0.f : __frcp_rn(sc);
          if ((t & ((gs >> 3) - 1)) == 0) scale[r * G + (vi << 3) / gs] = sc;
        }
        float q[8];
        quant_vec8(cur[i], sc, rc, q);
        if (MODE == kOutHalf)
          reinterpret_cast<uint4 *>(static_cast<__half *>(out) + r * K)[vi] = pack_h8(q);
        else
          reinterpret_cast<uint2 *>(static_cast<int8_t *>(out) + r * K)[vi] = pack_i8x8(q);
      }
      cur[i] = nxt[i];
    }
  }
}

template <int V, bool PG, int MODE>
int launch_rows(const __half *x, long R, int K, int gs, int T, void *out, float *scale,
                cudaStream_t s) {
  static int blocks[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W8A8_ERR_CUDA;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (blocks[dev] == 0) {
      int nsm = 0, occ = 0;
      if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, row_quant_rows<V, PG, MODE>, 256, 0) !=
              cudaSuccess || occ < 1)
        return W8A8_ERR_CUDA;
      blocks[dev] = nsm * occ;
    }
    per_sm = blocks[dev];
  }
  const int teams = 256 / T;
  const long need = (R + teams - 1) / teams;
  const long grid = need < per_sm ? need : per_sm;
  row_quant_rows<V, PG, MODE><<<static_cast<unsigned>(grid), 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), R, K, gs, T, out, scale);
  return launch_status();
}

template <int V, int MODE>
int launch_v(const __half *x, long R, int K, int gs, int qmax, int T, void *out,
             float *scale, cudaStream_t s) {
  const int block = 256;
  const int rows_per_block = block / T;
  const long grid = (R + rows_per_block - 1) / rows_per_block;
  row_quant_kernel<V, MODE><<<static_cast<unsigned>(grid), block, 0, s>>>(
      reinterpret_cast<const uint4 *>(x), R, K, gs, qmax, T, out, scale);
  return launch_status();
}

template <int MODE>
int launch_mode(const __half *x, int R, int K, int group_size, int qmax, void *out,
                float *scale, cudaStream_t s) {
  const int nvec = K >> 3;
  // enough threads per row that each caches at most 4 vectors (more warps
  // resident per SM), up to 256; beyond that up to 16 vectors per thread
  int T = 32;
  while (T < 256 && (nvec + T - 1) / T > 4) T <<= 1;
  const int V = (nvec + T - 1) / T;
  if ((MODE == kOutHalf || MODE == kOutInt8) && qmax == 127 && V <= 4) {
    constexpr int AM = MODE == kOutInt4 ? kOutInt8 : MODE;  // (INT4 never gets here)
    if (group_size != 0) {
      switch (V) {
        case 1: return launch_rows<1, true, AM>(x, R, K, group_size, T, out, scale, s);
        case 2: return launch_rows<2, true, AM>(x, R, K, group_size, T, out, scale, s);
        case 3: return launch_rows<3, true, AM>(x, R, K, group_size, T, out, scale, s);
        default: return launch_rows<4, true, AM>(x, R, K, group_size, T, out, scale, s);
      }
    }
    switch (V) {
      case 1: return launch_rows<1, false, AM>(x, R, K, 0, T, out, scale, s);
      case 2: return launch_rows<2, false, AM>(x, R, K, 0, T, out, scale, s);
      case 3: return launch_rows<3, false, AM>(x, R, K, 0, T, out, scale, s);
      default: return launch_rows<4, false, AM>(x, R, K, 0, T, out, scale, s);
    }
  }
  switch (V) {
#define W8A8_CASE(n) \
  case n:            \
    return launch_v<n, MODE>(x, R, K, group_size, qmax, T, out, scale, s);
    W8A8_CASE(1) W8A8_CASE(2) W8A8_CASE(3) W8A8_CASE(4) W8A8_CASE(5)
    W8A8_CASE(6) W8A8_CASE(7) W8A8_CASE(8) W8A8_CASE(9) W8A8_CASE(10)
    W8A8_CASE(11) W8A8_CASE(12) W8A8_CASE(13) W8A8_CASE(14) W8A8_CASE(15)
    W8A8_CASE(16)
#undef W8A8_CASE
    default:
      return W8A8_ERR_INVALID_ARG;  // K > 32768
  }
}

}  // namespace

int launch_row_quant(const __half *x, int R, int K, int group_size, int qmax,
                     int8_t *q, uint8_t *packed, float *scale, cudaStream_t s) {
  if (R == 0) return W8A8_OK;
  if (packed != nullptr)
    return launch_mode<kOutInt4>(x, R, K, group_size, qmax, packed, scale, s);
  return launch_mode<kOutInt8>(x, R, K, group_size, qmax, q, scale, s);
}

int launch_row_quant_half(const __half *x, int R, int K, int group_size, __half *qh,
                          float *scale, cudaStream_t s) {
  if (R == 0) return W8A8_OK;
  return launch_mode<kOutHalf>(x, R, K, group_size, 127, qh, scale, s);
}

}  // namespace w8a8
