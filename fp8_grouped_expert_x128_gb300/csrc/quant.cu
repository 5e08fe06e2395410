// 1x128 activation quantisation, 128x128 weight quantisation and the fused
// SwiGLU + requantisation.  All three are HBM-bound streaming kernels: 16-byte
// vector loads, one half-warp per 128-element block (8 elements per lane), the
// block amax reduced with shuffles inside the half-warp, IEEE fp32 divisions
// (so the bytes match the definition exactly), and a saturating
// round-to-nearest-even E4M3 conversion in hardware.
//
// Definition: per 128-element block, s = fp32(max(amax, 1e-4) / 448) and
// q = e4m3(fp32(x / s)); the scale array is "packed" MN-major (see moe_fp8.h).
// The FP8 GEMM of "Deploying DeepSeek on GB200 NVL72 with PD and Large Scale
// EP (Part I)", section "Implementation details" (DeepGEMM bullet), consumes
// exactly these quantised inputs with their packed scales.
#include "common.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- a1
// One warp covers 256 columns of one row: lanes 0-15 block 2w, 16-31 block 2w+1.
// kUE8M0: power-of-two block scales (block_scale_ue8m0), their exponent bytes
// also stored to e8 when it is given.
template <bool kUE8M0>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const uint16_t* __restrict__ x,
                                                          int64_t M, int64_t KB, int64_t ldx,
                                                          uint8_t* __restrict__ q, int64_t ldq,
                                                          float* __restrict__ s, int64_t s_ld,
                                                          uint8_t* __restrict__ e8) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t warps_per_row = (KB + 1) / 2;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t m = gw / warps_per_row;
  if (m >= M) return;
  const int64_t kb = (gw % warps_per_row) * 2 + (lane >> 4);
  const bool active = kb < KB;
  float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int64_t col = kb * 128 + (lane & 15) * 8;
  if (active) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + m * ldx + col));
    unpack_bf16x8(u, f);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  amax = half_warp_max(amax);
  if (!active) return;
  uint8_t byte = 0;
  const float sc = kUE8M0 ? block_scale_ue8m0(amax, &byte) : block_scale(amax);
  *reinterpret_cast<uint2*>(q + m * ldq + col) = kUE8M0 ? quant8_pow2(f, sc, byte) : quant8(f, sc);
  if ((lane & 15) == 0) {
    s[kb * s_ld + m] = sc;
    if (kUE8M0 && e8 != nullptr) e8[kb * s_ld + m] = byte;
  }
}

// ---------------------------------------------------------------- a3
// One CTA of 256 threads per 128x128 tile; thread t covers columns
// (t % 16) * 8 .. +7 of rows t/16 + 16 i, i = 0..7.  kUE8M0: power-of-two
// tile scales (block_scale_ue8m0), their exponent bytes also stored to e8.
template <bool kUE8M0>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const uint16_t* __restrict__ w,
                                                            int64_t N, int64_t K,
                                                            uint8_t* __restrict__ q,
                                                            float* __restrict__ s,
                                                            uint8_t* __restrict__ e8) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t tile = blockIdx.x;  // over E * NB * KB
  const int64_t e = tile / (NB * KB);
  const int64_t nb = (tile / KB) % NB;
  const int64_t kb = tile % KB;
  const int t = threadIdx.x;
  const int c8 = t & 15, r0 = t >> 4;
  const uint16_t* base = w + (e * N + nb * 128) * K + kb * 128 + c8 * 8;
  float f[8][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(base + (r0 + 16 * i) * K));
    unpack_bf16x8(u, f[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[i][j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[8];
  if ((t & 31) == 0) red[t >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  uint8_t byte = 0;
  const float sc = kUE8M0 ? block_scale_ue8m0(amax, &byte) : block_scale(amax);
  uint8_t* qb = q + (e * N + nb * 128) * K + kb * 128 + c8 * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    *reinterpret_cast<uint2*>(qb + (r0 + 16 * i) * K) = kUE8M0 ? quant8_pow2(f[i], sc, byte) : quant8(f[i], sc);
  if (t == 0) {
    s[(e * NB + nb) * KB + kb] = sc;
    if (kUE8M0 && e8 != nullptr) e8[(e * NB + nb) * KB + kb] = byte;
  }
}

// ---------------------------------------------------------------- a5
// h = silu(g) * u in fp32, quantised by the a1 rule (kUE8M0: with power-of-two
// scales).  A warp covers blocks 4w + h and 4w + h + 2 of one row (w = `part`,
// h = its half-warp), with all four 16-byte loads (g and u of both blocks)
// issued before any use.
template <bool kUE8M0>
__device__ __forceinline__ void swiglu_row_part(const uint16_t* __restrict__ y1, int64_t I, int64_t KB,
                                                int64_t r, int64_t part, int lane, uint8_t* __restrict__ q,
                                                const ScaleOut& so) {
  const int64_t kb0 = part * 4 + (lane >> 4);
  const uint16_t* row = y1 + r * 2 * I;
  uint4 gv[2], uv[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int64_t kb = kb0 + 2 * j;
    const int64_t col = kb * 128 + (lane & 15) * 8;
    gv[j] = kb < KB ? __ldg(reinterpret_cast<const uint4*>(row + col)) : make_uint4(0, 0, 0, 0);
    uv[j] = kb < KB ? __ldg(reinterpret_cast<const uint4*>(row + I + col)) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int64_t kb = kb0 + 2 * j;
    const bool active = kb < KB;
    const int64_t col = kb * 128 + (lane & 15) * 8;
    float h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (active) {
      float g[8], u[8];
      unpack_bf16x8(gv[j], g);
      unpack_bf16x8(uv[j], u);
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = __fdiv_rn(g[i], 1.0f + expf(-g[i])) * u[i];
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
    amax = half_warp_max(amax);
    if (active) {
      uint8_t byte = 0;
      const float sc = kUE8M0 ? block_scale_ue8m0(amax, &byte) : block_scale(amax);
      *reinterpret_cast<uint2*>(q + r * I + col) = kUE8M0 ? quant8_pow2(h, sc, byte) : quant8(h, sc);
      if ((lane & 15) == 0) so.put(r, kb, KB, sc, byte);
    }
  }
}

// Contiguous layout (rows selected by m_indices, or all rows): one warp per
// (row, part), the grid covering every row.
template <bool kUE8M0>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(
    const uint16_t* __restrict__ y1, int64_t rows, int64_t I, const int32_t* __restrict__ m_indices,
    uint8_t* __restrict__ q, const ScaleOut so) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t KB = I / 128;
  const int64_t warps_per_row = (KB + 3) / 4;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t r = gw / warps_per_row;
  if (r >= rows) return;
  if (m_indices != nullptr && __ldg(m_indices + r) < 0) return;
  swiglu_row_part<kUE8M0>(y1, I, KB, r, gw % warps_per_row, threadIdx.x & 31, q, so);
}

// Masked layout: only the rows below each expert's count hold tokens (a few
// hundred of E * max_m at decode).  A resident wave of CTAs walks the valid
// rows alone: each CTA turns the counts into a prefix over the experts in
// shared memory, and a warp task (valid row, part) finds its expert by binary
// search over the prefix.
constexpr int kSwMaxExperts = 1024;

template <bool kUE8M0>
__global__ void __launch_bounds__(256) swiglu_quant_masked_kernel(
    const uint16_t* __restrict__ y1, int64_t I, const int32_t* __restrict__ counts, int32_t E,
    int64_t max_m, uint8_t* __restrict__ q, const ScaleOut so) {
  __shared__ int32_t pre[kSwMaxExperts + 1];   // pre[e] = valid rows of the experts before e
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      // rows r of expert e with r < min(count, max_m), as the per-row rule reads
      const int c = e < E ? min(max(__ldg(counts + e), 0), static_cast<int>(max_m)) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) pre[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pre[E] = run;
  }
  __syncthreads();
  const int64_t KB = I / 128, warps_per_row = (KB + 3) / 4;
  const int64_t tasks = static_cast<int64_t>(pre[E]) * warps_per_row;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t task = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp; task < tasks;
       task += nwarps) {
    const int vr = static_cast<int>(task / warps_per_row);
    int lo = 0, hi = E - 1;   // the last expert e with pre[e] <= vr (it has rows: pre[e + 1] > vr)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= vr) lo = mid;
      else hi = mid - 1;
    }
    const int64_t r = static_cast<int64_t>(lo) * max_m + (vr - pre[lo]);
    swiglu_row_part<kUE8M0>(y1, I, KB, r, task % warps_per_row, lane, q, so);
  }
}

inline unsigned grid_for_warps(int64_t warps) {
  return static_cast<unsigned>((warps * 32 + 255) / 256);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_quant_fp8(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                             int64_t ldq, float* s, int64_t s_ld, int32_t flags, int32_t* err, void* stream) {
  (void)err;
  MOE_CHECK_ARG((flags & ~MOE_QUANT_UE8M0) == 0);
  if (flags & MOE_QUANT_UE8M0) return moe_quant_fp8_ue8m0(x, M, K, ldx, q, ldq, s, nullptr, s_ld, err, stream);
  MOE_CHECK_ARG(M >= 0 && K > 0 && K % 128 == 0);
  if (M == 0) return MOE_OK;
  MOE_CHECK_ARG(x && q && s && aligned16(x) && aligned16(q) && aligned16(s));
  MOE_CHECK_ARG(ldx >= K && ldx % 8 == 0 && ldq >= K && ldq % 16 == 0 && s_ld >= M);
  if (int st = check_device()) return st;
  const int64_t warps = M * ((K / 128 + 1) / 2);
  return launch_pdl(quant_1x128_kernel<false>, grid_for_warps(warps), 256, 0, as_stream(stream), x, M,
                    K / 128, ldx, q, ldq, s, s_ld, static_cast<uint8_t*>(nullptr));
}

extern "C" int moe_quant_fp8_ue8m0(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                   int64_t ldq, float* s, uint8_t* e8, int64_t s_ld, int32_t* err,
                                   void* stream) {
  (void)err;
  MOE_CHECK_ARG(M >= 0 && K > 0 && K % 128 == 0);
  if (M == 0) return MOE_OK;
  MOE_CHECK_ARG(x && q && s && aligned16(x) && aligned16(q) && aligned16(s));
  MOE_CHECK_ARG(ldx >= K && ldx % 8 == 0 && ldq >= K && ldq % 16 == 0 && s_ld >= M);
  if (int st = check_device()) return st;
  const int64_t warps = M * ((K / 128 + 1) / 2);
  return launch_pdl(quant_1x128_kernel<true>, grid_for_warps(warps), 256, 0, as_stream(stream), x, M,
                    K / 128, ldx, q, ldq, s, s_ld, e8);
}

extern "C" float moe_ue8m0_scale(float amax, uint8_t* byte_out) {
  uint8_t byte = 0;
  const float s = block_scale_ue8m0(amax, &byte);
  if (byte_out != nullptr) *byte_out = byte;
  return s;
}

extern "C" int moe_quant_weight_fp8(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint8_t* q,
                                    float* s, void* stream) {
  MOE_CHECK_ARG(E >= 0 && N > 0 && K > 0 && N % 128 == 0 && K % 128 == 0);
  if (E == 0) return MOE_OK;
  MOE_CHECK_ARG(w && q && s && aligned16(w) && aligned16(q));
  MOE_CHECK_ARG((reinterpret_cast<uintptr_t>(s) & 3u) == 0);  // scalar scale stores
  if (int st = check_device()) return st;
  const int64_t tiles = E * (N / 128) * (K / 128);
  MOE_CHECK_ARG(tiles < (1ll << 31));
  return launch_pdl(quant_128x128_kernel<false>, static_cast<unsigned>(tiles), 256, 0, as_stream(stream), w,
                    N, K, q, s, static_cast<uint8_t*>(nullptr));
}

extern "C" int moe_quant_weight_fp8_ue8m0(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint8_t* q,
                                          float* s, uint8_t* e8, void* stream) {
  MOE_CHECK_ARG(E >= 0 && N > 0 && K > 0 && N % 128 == 0 && K % 128 == 0);
  if (E == 0) return MOE_OK;
  MOE_CHECK_ARG(w && q && s && aligned16(w) && aligned16(q));
  MOE_CHECK_ARG((reinterpret_cast<uintptr_t>(s) & 3u) == 0);
  if (int st = check_device()) return st;
  const int64_t tiles = E * (N / 128) * (K / 128);
  MOE_CHECK_ARG(tiles < (1ll << 31));
  return launch_pdl(quant_128x128_kernel<true>, static_cast<unsigned>(tiles), 256, 0, as_stream(stream), w,
                    N, K, q, s, e8);
}

namespace moe {

// Shared by moe_swiglu_quant and moe_ffn: the scales go to s (fp32, groups of
// G rows) or, with sf8, as exponent bytes into the packed UE8M0 layout.
int swiglu_launch(const uint16_t* Y1, int64_t rows, int32_t I, const int32_t* counts, int32_t max_m,
                  const int32_t* m_indices, uint8_t* q, float* s, int64_t s_ld, bool ue8m0, uint8_t* sf8,
                  cudaStream_t st) {
  MOE_CHECK_ARG(rows >= 0 && I > 0 && I % 128 == 0);
  if (rows == 0) return MOE_OK;
  MOE_CHECK_ARG(Y1 && q && (s || sf8) && aligned16(Y1) && aligned16(q) && aligned16(s) && aligned16(sf8));
  MOE_CHECK_ARG(!sf8 || ue8m0);
  int64_t G;
  if (counts != nullptr) {
    MOE_CHECK_ARG(max_m > 0 && rows % max_m == 0);
    G = max_m;
  } else {
    MOE_CHECK_ARG(s_ld >= rows);
    G = s_ld;
  }
  if (int rc = check_device()) return rc;
  const ScaleOut so{s, sf8, G, static_cast<int32_t>((I / 128 + 3) / 4), static_cast<int32_t>((G + 127) / 128)};
  const int64_t warps = rows * ((I / 128 + 3) / 4);
  if (counts != nullptr) {
    const int64_t E = rows / max_m;
    MOE_CHECK_ARG(E <= kSwMaxExperts);
    // one resident wave at most (8 CTAs of 256 threads per SM), fewer when
    // even a full layout has fewer warp tasks
    const int64_t wave = static_cast<int64_t>(num_sms()) * 8;
    const int64_t need = grid_for_warps(warps);
    auto kern = ue8m0 ? swiglu_quant_masked_kernel<true> : swiglu_quant_masked_kernel<false>;
    return launch_pdl(kern, static_cast<unsigned>(need < wave ? need : wave), 256, 0, st, Y1,
                      static_cast<int64_t>(I), counts, static_cast<int32_t>(E), static_cast<int64_t>(max_m), q, so);
  }
  auto kern = ue8m0 ? swiglu_quant_kernel<true> : swiglu_quant_kernel<false>;
  return launch_pdl(kern, grid_for_warps(warps), 256, 0, st, Y1, rows, static_cast<int64_t>(I), m_indices, q, so);
}

}  // namespace moe

extern "C" int moe_swiglu_quant(const uint16_t* Y1, int64_t rows, int32_t I, const int32_t* counts,
                                int32_t max_m, const int32_t* m_indices, uint8_t* q, float* s,
                                int64_t s_ld, int32_t flags, int32_t* err, void* stream) {
  (void)err;
  MOE_CHECK_ARG((flags & ~MOE_QUANT_UE8M0) == 0 && s != nullptr);
  return swiglu_launch(Y1, rows, I, counts, max_m, m_indices, q, s, s_ld, (flags & MOE_QUANT_UE8M0) != 0, nullptr,
                       as_stream(stream));
}
