// Pieces shared by the grouped GEMM kernels (fp32-scale and block-scaled):
// tile and warp-role constants, the register split between warpgroups, the
// one-time launch preparation, and the device-built tile schedule over the
// per-expert row extents.
#pragma once

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;                         // epilogue = warps 4..11 (warpgroups 1, 2)
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);  // warps 2-3 only hold warpgroup 0 together
// Register split between warpgroups (setmaxnreg): warpgroup 0 (TMA + MMA
// issue) needs few registers, the epilogue holds 128 fp32 accumulators per
// thread.  The launch allocates kLaunchRegs to all 384 threads; warpgroup 0
// gives back down to kRegsLow and the two epilogue warpgroups take kRegsHigh:
// 128 * 40 + 256 * 232 = 64512 = 384 * 168, exactly the launch allocation, so
// the increase never waits on registers that do not exist.  The host refuses to
// launch a split kernel whose compiled register count differs from kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 40;
constexpr int kRegsHigh = 232;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs, "register split");
static_assert(kThreads * kLaunchRegs <= 65536, "register file");

__device__ __forceinline__ void regs_release_low() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
}
__device__ __forceinline__ void regs_acquire_high() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
}

// Per-device, per-kernel launch set-up done once: the dynamic shared-memory
// opt-in and, for kernels that split registers, the check that the launch
// register count equals kLaunchRegs.  Keyed by (device, kernel address).
template <typename F>
int prepare_kernel(F kernel, size_t smem, bool split_regs) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> prepared;  // -> smem opted in
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const auto key = std::make_pair(dev, reinterpret_cast<const void*>(kernel));
  std::lock_guard<std::mutex> lock(mu);
  auto it = prepared.find(key);
  if (it == prepared.end()) {
    if (split_regs) {
      cudaFuncAttributes attr;
      if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess) return MOE_ERR_CUDA;
      if (attr.numRegs != kLaunchRegs) return MOE_ERR_UNSUPPORTED;
    }
    it = prepared.emplace(key, 0).first;
  }
  if (smem > it->second) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    it->second = smem;
  }
  return MOE_OK;
}
constexpr uint32_t kTmemCols = 512;
// Output staging of the tokens-as-M epilogues: per epilogue warp, 32 rows x
// 32 bf16 columns (64 bytes per row), the row's 16-byte chunk c kept in slot
// c ^ ((row >> 1) & 3): conflict-free both when a lane writes its own row's
// chunks and when 8 lanes read two rows' four chunks.
constexpr uint32_t kOutStageBytes = 32 * 64;
__device__ __forceinline__ uint32_t out_stage_slot(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
constexpr size_t kMaxSmemPerBlock = 232448;   // 227 KB opt-in dynamic shared memory per block
constexpr int kMaxExperts = 1024;

// Token-side tensor maps: the same [E*max_m, K] matrix with boxes of 16 << i
// rows (a map whose box would exceed the matrix repeats the 16-row map; the
// kernel never picks a box taller than the tile's rows).
struct TokenMaps {
  CUtensorMap box[4];
};

struct Sched {
  int32_t* tile0;  // [E+1] first tile of each expert
  int32_t* rbase;  // [E]   first A/D row of each expert
  int32_t* rext;   // [E]   row extent (masked: kept count; contiguous: segment rows)
};

struct TileCursor {
  int e = 0;
  __device__ __forceinline__ void seek(const Sched& s, int t) {
    while (t >= s.tile0[e + 1]) ++e;
  }
};

// Warp 0 builds the tile schedule: each lane owns a contiguous chunk of experts;
// an expert's rows are cut into blocks of kRows (128, or 256 for a CTA pair).
// Args: the kernel's argument block (layout, counts / offsets, max_m,
// M_capacity, E, err).
template <int kRows = BM, class Args>
__device__ void build_schedule(const Args& p, const Sched& s, int n_tiles) {
  const int lane = threadIdx.x & 31;
  const int per = (p.E + 31) / 32;
  const int e0 = min(lane * per, p.E), e1 = min(e0 + per, p.E);
  int local = 0;
  bool overflow = false, bad = false;
  for (int e = e0; e < e1; ++e) {
    int rb, rx;
    if (p.layout == MOE_LAYOUT_MASKED) {
      int c = __ldcg(p.counts + e);   // from L2: may be read before the grid dependency wait
      if (c > p.max_m) { overflow = true; c = p.max_m; }
      if (c < 0) { bad = true; c = 0; }
      rb = e * p.max_m;
      rx = c;
    } else {
      rb = __ldcg(p.offsets + e);
      rx = __ldcg(p.offsets + e + 1) - rb;
      // a segment must start on a 128-row boundary and lie inside the
      // M_capacity rows of A, D and m_indices; otherwise it is skipped
      if (rb < 0 || (rb % BM) != 0 || rx < 0 || (rx % BM) != 0 ||
          static_cast<int64_t>(rb) + rx > p.M_capacity) {
        bad = true;
        rb = 0;
        rx = 0;
      }
    }
    s.rbase[e] = rb;
    s.rext[e] = rx;
    local += (rx + kRows - 1) / kRows * n_tiles;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int e = e0; e < e1; ++e) {
    s.tile0[e] = run;
    run += (s.rext[e] + kRows - 1) / kRows * n_tiles;
  }
  if (lane == 31) s.tile0[p.E] = incl;
  if (blockIdx.x == 0) {
    if (overflow) set_err(p.err, MOE_DEV_OVERFLOW);
    if (bad) set_err(p.err, MOE_DEV_BAD_INDEX);
  }
}

}  // namespace
}  // namespace moe
