// Permute token-order FP8 rows into the grouped expert layouts, and combine
// expert outputs back into token order.
//
// The grouped layouts are the inputs of the two grouped GEMMs of "Deploying
// DeepSeek with PD Disaggregation and Large-Scale Expert Parallelism on 96 H100
// GPUs", section "DeepGEMM integration": contiguous segments for prefill (after
// DeepEP's normal dispatch) and a fixed-capacity slab per expert with
// device-side counts for decode (after the CUDA-Graph-compatible low-latency
// dispatch; same page, section "Expert parallelism based on DeepEP").  Here the
// cross-GPU shuffle is absent: tokens are already resident, and the permute is
// the local half of a dispatch.
//
// permute: one CTA of 1024 threads assigns every routed row a destination in
// ascending assignment order (deterministic), counting with warp match masks
// and a per-warp table in shared memory; a second kernel copies the 1-byte
// rows (16-byte vectors, one warp per row) and gathers their fp32 scales, or --
// inside moe_ffn -- quantises the bf16 token rows straight into their slots.
// combine: a resident wave of CTAs over the tokens, fp32 accumulation over the
// k choices in order (then the optional shared-expert row).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kIdxThreads = 1024;
constexpr int kIdxWarps = kIdxThreads / 32;
constexpr int kIdxPer = 4;  // assignments per thread per ranking chunk
static_assert(kIdxWarps == 32, "the scan over warps runs one warp lane per warp");
constexpr int kMaxExperts = 1024;
static_assert(kMaxExperts <= kIdxThreads, "one expert per thread in the index pass");
constexpr size_t kIdxSmemLimit = 200 * 1024;

struct IndexParams {
  const int32_t* topk_ids;
  int64_t n_assign;  // T * k
  int32_t expert_begin, E, layout, max_m;
  int64_t rows_capacity;
  int32_t* counts;
  int32_t* offsets;
  int32_t* m_indices;
  int32_t* row_src;
  int32_t* dst_row;
  int32_t* err;
};

// dynamic smem: cnt[E] | base[E] | wc[kIdxWarps][E] | ids[n_assign] (when they fit)
// The routing ids are read from global memory once, into shared memory, so the
// ordered rank pass below runs at shared-memory latency.
__global__ void __launch_bounds__(kIdxThreads) permute_index_kernel(IndexParams p, int ids_in_smem) {
  extern __shared__ int32_t sm[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int E = p.E;
  int32_t* cnt = sm;
  int32_t* base = sm + E;
  int32_t* wc = sm + 2 * E;
  int32_t* ids = sm + 2 * E + kIdxWarps * E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto local_expert = [&](int64_t i) -> int {
    const int e = (ids_in_smem ? ids[i] : p.topk_ids[i]) - p.expert_begin;
    return (e >= 0 && e < E) ? e : -1;
  };

  // 1. stage ids, histogram (order-free; one atomic per distinct expert per warp)
  for (int e = tid; e < E; e += kIdxThreads) cnt[e] = 0;
  if (ids_in_smem) {
    // eight loads in flight per thread before their shared-memory stores
    for (int64_t i0 = 0; i0 < p.n_assign; i0 += 8 * kIdxThreads) {
      int32_t v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t i = i0 + j * kIdxThreads + tid;
        v[j] = i < p.n_assign ? __ldg(p.topk_ids + i) : 0;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t i = i0 + j * kIdxThreads + tid;
        if (i < p.n_assign) ids[i] = v[j];
      }
    }
  }
  __syncthreads();
  for (int64_t c0 = 0; c0 < p.n_assign; c0 += kIdxThreads) {
    const int64_t i = c0 + tid;
    const int e = i < p.n_assign ? local_expert(i) : -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (same & ((1u << lane) - 1u)) == 0) atomicAdd(&cnt[e], __popc(same));
  }
  __syncthreads();

  // 2. segment bases, counts, offsets, one expert per thread (E <= kIdxThreads);
  //    the contiguous offsets are a block-wide exclusive scan of the padded counts
  {
    __shared__ int64_t wsum[kIdxWarps];
    const int e = tid;
    const int c = e < E ? cnt[e] : 0;
    if (p.layout == MOE_LAYOUT_MASKED) {
      if (e < E) {
        base[e] = e * p.max_m;
        p.counts[e] = c < p.max_m ? c : p.max_m;
        if (c > p.max_m) set_err(p.err, MOE_DEV_OVERFLOW);
      }
    } else {
      const int64_t padded = (static_cast<int64_t>(c) + 127) / 128 * 128;
      int64_t incl = padded;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        const int64_t v = wsum[lane];
        int64_t w_incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t y = __shfl_up_sync(0xffffffffu, w_incl, o);
          if (lane >= o) w_incl += y;
        }
        wsum[lane] = w_incl - v;   // rows before this warp's experts
      }
      __syncthreads();
      const int64_t excl = wsum[warp] + incl - padded;
      if (e < E) {
        base[e] = static_cast<int32_t>(excl);
        p.offsets[e] = static_cast<int32_t>(excl);
        p.counts[e] = c;
      }
      if (e == E - 1) {
        const int64_t row = excl + padded;
        p.offsets[E] = static_cast<int32_t>(row);
        if (row > p.rows_capacity) set_err(p.err, MOE_DEV_BAD_INDEX);
      }
    }
  }
  __syncthreads();
  const int64_t map_rows =
      p.layout == MOE_LAYOUT_MASKED ? static_cast<int64_t>(E) * p.max_m : p.rows_capacity;
  for (int64_t r = tid; r < map_rows; r += kIdxThreads) {
    p.row_src[r] = -1;
    if (p.layout == MOE_LAYOUT_CONTIG) p.m_indices[r] = -1;
  }
  for (int e = tid; e < E; e += kIdxThreads) cnt[e] = 0;  // becomes the running rank
  __syncthreads();

  // 3. ranks in ascending assignment order, in chunks of kIdxThreads * kIdxPer:
  //    warp w owns the chunk's assignments [w, w+1) * 32 * kIdxPer, visited in
  //    kIdxPer rounds of 32 consecutive ones.
  const uint32_t lanes_below = (1u << lane) - 1u;
  for (int64_t c0 = 0; c0 < p.n_assign; c0 += static_cast<int64_t>(kIdxThreads) * kIdxPer) {
    for (int x = tid; x < kIdxWarps * E; x += kIdxThreads) wc[x] = 0;
    __syncthreads();
    // (a) per-warp count of each expert, and each assignment's rank in its warp
    int e_r[kIdxPer], rk_r[kIdxPer];
#pragma unroll
    for (int r = 0; r < kIdxPer; ++r) {
      const int64_t i = c0 + (static_cast<int64_t>(warp) * kIdxPer + r) * 32 + lane;
      const int e = i < p.n_assign ? local_expert(i) : -1;
      const uint32_t same = __match_any_sync(0xffffffffu, e);
      const int lower = __popc(same & lanes_below);
      const int before = e >= 0 ? wc[warp * E + e] : 0;   // this expert in earlier rounds
      __syncwarp();
      if (e >= 0 && lower == 0) wc[warp * E + e] = before + __popc(same);
      __syncwarp();
      e_r[r] = e;
      rk_r[r] = before + lower;
    }
    __syncthreads();
    // (b) per expert, exclusive scan over the warps (lane = warp), on top of
    //     the running count of earlier chunks
    for (int ee = warp; ee < E; ee += kIdxWarps) {
      const int v = wc[lane * E + ee];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int run = cnt[ee];
      __syncwarp();
      wc[lane * E + ee] = run + incl - v;
      if (lane == 31) cnt[ee] = run + incl;
    }
    __syncthreads();
    // (c) destinations
#pragma unroll
    for (int r = 0; r < kIdxPer; ++r) {
      const int64_t i = c0 + (static_cast<int64_t>(warp) * kIdxPer + r) * 32 + lane;
      const int e = e_r[r];
      if (e >= 0) {
        const int rank = wc[warp * E + e] + rk_r[r];
        int32_t dst = -1;
        if (p.layout == MOE_LAYOUT_CONTIG || rank < p.max_m) {
          const int64_t row = static_cast<int64_t>(base[e]) + rank;
          if (row < map_rows) {
            dst = static_cast<int32_t>(row);
            p.row_src[row] = static_cast<int32_t>(i);
            if (p.layout == MOE_LAYOUT_CONTIG) p.m_indices[row] = e;
          }
        }
        p.dst_row[i] = dst;
      } else if (i < p.n_assign) {
        p.dst_row[i] = -1;
      }
    }
    __syncthreads();
  }
}

// Large batches: the index pass over many CTAs, in two kernels.
// permute_chunk_rank_kernel: CTA c takes assignments [c, c+1) * kIdxChunk and
// ranks each among the chunk's assignments to the same expert (the ordered
// per-warp counting of the one-CTA pass), writing the rank (lrank) and the
// chunk's per-expert totals (chunk_hist[c][E]).
// permute_finalize_kernel: every CTA adds up the chunk totals -- each expert's
// count, segment base (masked: e * max_m; contiguous: exclusive scan of the
// counts padded to 128) and the total of the chunks before its own -- and for
// its assignments writes dst_row / row_src / m_indices exactly as the one-CTA
// pass does; all CTAs share the -1 fill of the rows no assignment uses, and
// CTA 0 writes counts, offsets and the error flags.
constexpr int kIdxChunk = kIdxThreads * kIdxPer;
constexpr int kFinThreads = 256;
static_assert(kIdxChunk == 4096, "permute_chunk_count sizes chunk_hist for 4096-id chunks");
static_assert(kIdxChunk % kFinThreads == 0, "a finalize CTA stays inside one chunk");

__global__ void __launch_bounds__(kIdxThreads, 1) permute_chunk_rank_kernel(IndexParams p, int32_t* lrank,
                                                                         int32_t* chunk_hist) {
  extern __shared__ int32_t sm[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int E = p.E;
  int32_t* cnt = sm;        // [E] running count inside the chunk
  int32_t* wc = sm + E;     // [kIdxWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kIdxChunk;
  for (int e = tid; e < E; e += kIdxThreads) cnt[e] = 0;
  for (int x = tid; x < kIdxWarps * E; x += kIdxThreads) wc[x] = 0;
  __syncthreads();
  const uint32_t lanes_below = (1u << lane) - 1u;
  int e_r[kIdxPer], rk_r[kIdxPer];
#pragma unroll
  for (int r = 0; r < kIdxPer; ++r) {
    const int64_t i = c0 + (static_cast<int64_t>(warp) * kIdxPer + r) * 32 + lane;
    int e = i < p.n_assign ? __ldg(p.topk_ids + i) - p.expert_begin : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int lower = __popc(same & lanes_below);
    const int before = e >= 0 ? wc[warp * E + e] : 0;
    __syncwarp();
    if (e >= 0 && lower == 0) wc[warp * E + e] = before + __popc(same);
    __syncwarp();
    e_r[r] = e;
    rk_r[r] = before + lower;
  }
  __syncthreads();
  for (int ee = warp; ee < E; ee += kIdxWarps) {
    const int v = wc[lane * E + ee];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncwarp();
    wc[lane * E + ee] = incl - v;
    if (lane == 31) cnt[ee] = incl;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kIdxPer; ++r) {
    const int64_t i = c0 + (static_cast<int64_t>(warp) * kIdxPer + r) * 32 + lane;
    if (i < p.n_assign) lrank[i] = e_r[r] >= 0 ? wc[warp * E + e_r[r]] + rk_r[r] : -1;
  }
  for (int e = tid; e < E; e += kIdxThreads) chunk_hist[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
}

__global__ void __launch_bounds__(kFinThreads) permute_finalize_kernel(IndexParams p, const int32_t* lrank,
                                                                       const int32_t* chunk_hist, int32_t n_chunks) {
  extern __shared__ int32_t fsm[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int E = p.E;
  int32_t* tot = fsm;           // [E] count over all chunks
  int32_t* pre = fsm + E;       // [E] count over the chunks before this CTA's
  int32_t* base = fsm + 2 * E;  // [E] segment base
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kFinThreads;
  const int my_chunk = static_cast<int>(i0 / kIdxChunk);
  for (int e = tid; e < E; e += kFinThreads) {
    int t = 0, b = 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int h = __ldg(chunk_hist + static_cast<int64_t>(c) * E + e);
      if (c < my_chunk) b += h;
      t += h;
    }
    tot[e] = t;
    pre[e] = b;
  }
  __syncthreads();
  if (p.layout == MOE_LAYOUT_MASKED) {
    for (int e = tid; e < E; e += kFinThreads) base[e] = e * p.max_m;
  } else if (tid < 32) {
    // exclusive scan of the padded counts over the experts, 32 at a time
    int64_t run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int64_t padded = e < E ? (static_cast<int64_t>(tot[e]) + 127) / 128 * 128 : 0;
      int64_t incl = padded;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) base[e] = static_cast<int32_t>(run + incl - padded);
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (blockIdx.x == 0 && lane == 0) {
      p.offsets[E] = static_cast<int32_t>(run);
      if (run > p.rows_capacity) set_err(p.err, MOE_DEV_BAD_INDEX);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += kFinThreads) {
      if (p.layout == MOE_LAYOUT_MASKED) {
        p.counts[e] = tot[e] < p.max_m ? tot[e] : p.max_m;
        if (tot[e] > p.max_m) set_err(p.err, MOE_DEV_OVERFLOW);
      } else {
        p.offsets[e] = base[e];
        p.counts[e] = tot[e];
      }
    }
  }
  const int64_t map_rows =
      p.layout == MOE_LAYOUT_MASKED ? static_cast<int64_t>(E) * p.max_m : p.rows_capacity;
  // this CTA's assignments
  const int64_t i = i0 + tid;
  if (i < p.n_assign) {
    const int lr = __ldg(lrank + i);
    int32_t dst = -1;
    if (lr >= 0) {
      int e = __ldg(p.topk_ids + i) - p.expert_begin;
      const int rank = pre[e] + lr;
      if (p.layout == MOE_LAYOUT_CONTIG || rank < p.max_m) {
        const int64_t row = static_cast<int64_t>(base[e]) + rank;
        if (row < map_rows) {
          dst = static_cast<int32_t>(row);
          p.row_src[row] = static_cast<int32_t>(i);
          if (p.layout == MOE_LAYOUT_CONTIG) p.m_indices[row] = e;
        }
      }
    }
    p.dst_row[i] = dst;
  }
  // the rows no assignment uses: each expert's rows past its count up to its
  // segment end, and (contiguous) the rows past the last segment
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kFinThreads;
  const int64_t gtid = i0 + tid;
  for (int e = 0; e < E; ++e) {
    const int64_t used = p.layout == MOE_LAYOUT_MASKED ? (tot[e] < p.max_m ? tot[e] : p.max_m) : tot[e];
    const int64_t seg = p.layout == MOE_LAYOUT_MASKED ? p.max_m : (static_cast<int64_t>(tot[e]) + 127) / 128 * 128;
    for (int64_t r = base[e] + used + gtid; r < base[e] + seg && r < map_rows; r += stride) {
      p.row_src[r] = -1;
      if (p.layout == MOE_LAYOUT_CONTIG) p.m_indices[r] = -1;
    }
  }
  if (p.layout == MOE_LAYOUT_CONTIG) {
    const int64_t end = static_cast<int64_t>(base[E - 1]) + (static_cast<int64_t>(tot[E - 1]) + 127) / 128 * 128;
    for (int64_t r = end + gtid; r < map_rows; r += stride) {
      p.row_src[r] = -1;
      p.m_indices[r] = -1;
    }
  }
}

// One warp per assignment: copy the FP8 row and gather its scales.
__global__ void __launch_bounds__(128) permute_scatter_kernel(
    const uint8_t* __restrict__ q, const float* __restrict__ s, int64_t s_ld,
    const int32_t* __restrict__ dst_row, int64_t n_assign, int32_t k, int64_t H,
    uint8_t* __restrict__ q_out, float* __restrict__ s_out, int64_t G) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= n_assign) return;
  const int32_t dst = __ldg(dst_row + i);
  if (dst < 0) return;
  const int64_t t = i / k;
  const uint4* src = reinterpret_cast<const uint4*>(q + t * H);
  uint4* out = reinterpret_cast<uint4*>(q_out + static_cast<int64_t>(dst) * H);
  const int64_t n16 = H / 16;
  for (int64_t v = lane; v < n16; v += 32) out[v] = __ldg(src + v);
  const int64_t KB = H / 128;
  const int64_t grp = dst / G, pos = dst - grp * G;
  for (int64_t kb = lane; kb < KB; kb += 32) s_out[(grp * KB + kb) * G + pos] = __ldg(s + kb * s_ld + t);
}

// Fused 1x128 quantisation + scatter for moe_ffn: one resident wave of CTAs
// walks the tokens (grid stride); the CTA's kQsWarps warps share the token's
// 128-column block pairs (a half-warp per block), loads issued before use,
// quantise the bf16 row once and write it into each of the token's local
// expert slots (the bytes equal moe_quant_fp8 followed by moe_permute: same
// helpers, same arithmetic).  The quantisation needs only x, so a CTA's first
// row is loaded and quantised before the kernel waits on the routing index
// kernel launched just before it (programmatic dependent launch): the index
// work hides behind the first row's loads.  Nothing the index kernel writes is
// read, and nothing is written, before that wait.
// Two shapes, both with a whole row's loads in flight (H <= 7168 in one pass):
// many tokens (prefill) take 4-warp CTAs, 7 block pairs per warp, ~6 CTAs per
// SM for the bytes in flight; a few hundred tokens (decode) take 8-warp CTAs,
// 4 pairs per warp, so each row finishes sooner.
// kUE8M0: power-of-two block scales, their exponent bytes written to the
// packed layout of the block-scaled GEMM (ScaleOut with sf8).
// kRank (masked layout, small batches, k <= kRankMaxK): the kernel also does the
// index pass's work, so no separate index kernel runs.  For its token t each CTA
// counts, over the assignments before each of the token's slots, those routed
// to the same expert -- the slot's rank in ascending assignment order, the
// index pass's definition -- with every thread scanning a strided share of the
// routing ids (four per 16-byte load, all loads of a pass in flight); CTA 0
// also builds the per-expert counts (clamped to max_m, overflow flagged).
// Unused slab rows' row_src entries are left as they are (moe_ffn reads
// row_src only for rows below a count).
constexpr int kRankMaxK = 16;
struct RankArgs {
  const int32_t* topk_ids;
  int32_t expert_begin, E, max_m;
  int32_t* counts;
  int32_t* row_src;
  int32_t* dst_row;
  int32_t* err;
};

template <int kQsWarps, int kQsPairs, bool kUE8M0, bool kRank = false>
__global__ void __launch_bounds__(32 * kQsWarps, kRank ? 2 : (kQsWarps == 4 ? 8 : 4)) quant_scatter_kernel(
    const uint16_t* __restrict__ x, int64_t ldx, const int32_t* __restrict__ dst_row,
    int64_t T, int32_t k, int64_t H, uint8_t* __restrict__ q_out, const ScaleOut so,
    uint16_t* __restrict__ zero_out, int64_t ldo, const RankArgs ra) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t KB = H / 128, NP = (KB + 1) / 2;
  bool waited = false;
  auto wait_index = [&]() {
    if (!waited) {
      grid_dependency_wait();
      grid_launch_dependents();
      waited = true;
    }
  };
  __shared__ int32_t s_dst[kRank ? kRankMaxK : 1];
  __shared__ int32_t s_rank[kRank ? kRankMaxK : 1];
  __shared__ int32_t s_sid[kRank ? kRankMaxK : 1];
  if constexpr (kRank) {
    // x and the routing ids may come from the kernel just before this one
    wait_index();
    if (blockIdx.x == 0) {
      // per-expert counts over all assignments (warp-aggregated shared atomics)
      __shared__ int32_t hist[kMaxExperts];
      for (int e = threadIdx.x; e < ra.E; e += blockDim.x) hist[e] = 0;
      __syncthreads();
      const int64_t n = T * k;
      for (int64_t i0 = 0; i0 < n; i0 += blockDim.x) {
        const int64_t i = i0 + threadIdx.x;
        int e = i < n ? __ldg(ra.topk_ids + i) - ra.expert_begin : -1;
        if (e < 0 || e >= ra.E) e = -1;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (same & ((1u << lane) - 1u)) == 0) atomicAdd(&hist[e], __popc(same));
      }
      __syncthreads();
      for (int e = threadIdx.x; e < ra.E; e += blockDim.x) {
        const int c = hist[e];
        ra.counts[e] = c < ra.max_m ? c : ra.max_m;
        if (c > ra.max_m) set_err(ra.err, MOE_DEV_OVERFLOW);
      }
    }
  }
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const uint16_t* xr = x + t * ldx;
    if constexpr (kRank) {
      // the token's slot ranks: assignments [0, t*k + j) routed like slot j
      if (threadIdx.x < k) {
        s_sid[threadIdx.x] = __ldg(ra.topk_ids + t * k + threadIdx.x);
        s_rank[threadIdx.x] = 0;
      }
      __syncthreads();
      int sid[kRankMaxK], c[kRankMaxK];
#pragma unroll
      for (int j = 0; j < kRankMaxK; ++j) {
        sid[j] = j < k ? s_sid[j] : INT32_MIN;
        c[j] = 0;
      }
      const int64_t first = t * k, lim = first + k;   // positions that can precede a slot
      for (int64_t p0 = static_cast<int64_t>(threadIdx.x) * 4; p0 < lim; p0 += static_cast<int64_t>(blockDim.x) * 4) {
        int v[4];
        if (p0 + 4 <= lim && (reinterpret_cast<uintptr_t>(ra.topk_ids + p0) & 15) == 0) {
          const int4 w = __ldg(reinterpret_cast<const int4*>(ra.topk_ids + p0));
          v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = p0 + q < lim ? __ldg(ra.topk_ids + p0 + q) : INT32_MIN;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t pos = p0 + q;
#pragma unroll
          for (int j = 0; j < kRankMaxK; ++j) c[j] += (v[q] == sid[j] && pos < first + j) ? 1 : 0;
        }
      }
#pragma unroll
      for (int j = 0; j < kRankMaxK; ++j) {
        if (j < k) {
          int cj = c[j];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) cj += __shfl_xor_sync(0xffffffffu, cj, o);
          if (lane == 0 && cj) atomicAdd(&s_rank[j], cj);
        }
      }
      __syncthreads();
      if (threadIdx.x < k) {
        const int j = threadIdx.x;
        const int e = s_sid[j] - ra.expert_begin;
        const int rank = s_rank[j];
        int32_t dst = -1;
        if (e >= 0 && e < ra.E && rank < ra.max_m) {
          dst = e * ra.max_m + rank;
          ra.row_src[dst] = static_cast<int32_t>(first + j);
        }
        ra.dst_row[first + j] = dst;
        s_dst[j] = dst;
      }
      __syncthreads();
    }
    for (int64_t p0 = warp; p0 < NP; p0 += static_cast<int64_t>(kQsWarps) * kQsPairs) {
      uint4 u[kQsPairs];
#pragma unroll
      for (int j = 0; j < kQsPairs; ++j) {
        const int64_t kb = (p0 + j * kQsWarps) * 2 + (lane >> 4);
        u[j] = kb < KB ? __ldg(reinterpret_cast<const uint4*>(xr + kb * 128 + (lane & 15) * 8))
                       : make_uint4(0, 0, 0, 0);
      }
      uint2 code[kQsPairs];
      float sc[kQsPairs];
      uint8_t e8b[kQsPairs];
#pragma unroll
      for (int j = 0; j < kQsPairs; ++j) {
        float f[8];
        unpack_bf16x8(u[j], f);
        float amax = 0.f;
#pragma unroll
        for (int v = 0; v < 8; ++v) amax = fmaxf(amax, fabsf(f[v]));
        amax = half_warp_max(amax);
        e8b[j] = 0;
        sc[j] = kUE8M0 ? block_scale_ue8m0(amax, &e8b[j]) : block_scale(amax);
        code[j] = kUE8M0 ? quant8_pow2(f, sc[j], e8b[j]) : quant8(f, sc[j]);
      }
      wait_index();
      // the token's routing slots, one per lane, with the k-independent part
      // of each slot's scale index
      int32_t dl = -1;
      if (lane < k) dl = kRank ? s_dst[lane] : __ldg(dst_row + t * k + lane);
      const int64_t sbl = dl >= 0 ? so.row_base(dl, KB) : 0;
      for (int j2 = 0; j2 < k; ++j2) {
        const int32_t dst = __shfl_sync(0xffffffffu, dl, j2);
        if (dst < 0) continue;
        const int64_t sb = __shfl_sync(0xffffffffu, sbl, j2);
        uint8_t* qr = q_out + static_cast<int64_t>(dst) * H;
#pragma unroll
        for (int j = 0; j < kQsPairs; ++j) {
          const int64_t kb = (p0 + j * kQsWarps) * 2 + (lane >> 4);
          if (kb < KB) {
            *reinterpret_cast<uint2*>(qr + kb * 128 + (lane & 15) * 8) = code[j];
            if ((lane & 15) == 0) so.put_at(sb, kb, sc[j], e8b[j]);
          }
        }
      }
    }
    if (zero_out != nullptr) {
      // one slot per token and it is not routed here: the token's output row
      // is zero (what the combine writes for a token without local slots)
      wait_index();
      if ((kRank ? s_dst[0] : __ldg(dst_row + t)) < 0)
        for (int64_t c = threadIdx.x; c < H / 8; c += blockDim.x)
          reinterpret_cast<uint4*>(zero_out + t * ldo)[c] = make_uint4(0, 0, 0, 0);
    }
  }
  wait_index();   // a CTA with no token still orders its exit after the index kernel
}

// A resident wave of CTAs walks the tokens (grid stride), one token at a
// time per CTA.  Warp 0 holds the token's routing slots: it compacts the valid
// ones (order kept) into shared memory and, while the CTA works on this token,
// already loads the next token's slots, so only the row loads sit on the
// per-token path.  For each slot a thread issues all of its 16-byte row loads
// (kCombVec chunks of 8 columns, strided by the block) before accumulating.
// Accumulation per element is fp32 fmaf in slot order.
constexpr int kCombThreads = 128;
constexpr int kCombVec = 8;

// Optional terms (both default off): with `accumulate` the sum starts from the
// output row's current value, and `shared` (a bf16 [T, H] row per token, row
// stride lds) is added with weight 1 after the slots -- the same fp32 steps as
// one more routing slot of weight 1, so the bits equal that formulation.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    f[2 * h] = __uint_as_float(x[h] << 16);
    f[2 * h + 1] = __uint_as_float(x[h] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(kCombThreads) combine_kernel(
    const uint16_t* __restrict__ y2, int64_t ldy, int64_t y_rows, const int32_t* __restrict__ dst_row,
    const float* __restrict__ topk_w, int32_t k, int64_t H, const uint16_t* __restrict__ shared, int64_t lds,
    int accumulate, uint16_t* __restrict__ out, int64_t ldo, int64_t T, int32_t* err) {
  grid_dependency_wait();
  grid_launch_dependents();
  __shared__ int32_t s_dst[32];
  __shared__ float s_w[32];
  __shared__ int s_n;
  const int tid = threadIdx.x;
  int32_t d_next = -1;
  float w_next = 0.f;
  if (tid < k && blockIdx.x < T) {
    d_next = __ldg(dst_row + static_cast<int64_t>(blockIdx.x) * k + tid);
    w_next = __ldg(topk_w + static_cast<int64_t>(blockIdx.x) * k + tid);
  }
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    if (tid < 32) {
      int32_t d = d_next;
      const float w = w_next;
      if (d >= y_rows) {
        set_err(err, MOE_DEV_BAD_INDEX);
        d = -1;
      }
      const uint32_t valid = __ballot_sync(0xffffffffu, d >= 0);
      if (d >= 0) {
        const int slot = __popc(valid & ((1u << tid) - 1u));
        s_dst[slot] = d;
        s_w[slot] = w;
      }
      if (tid == 0) s_n = __popc(valid);
      // the next token's slots load while this one is combined
      const int64_t tn = t + gridDim.x;
      d_next = -1;
      w_next = 0.f;
      if (tid < k && tn < T) {
        d_next = __ldg(dst_row + tn * k + tid);
        w_next = __ldg(topk_w + tn * k + tid);
      }
    }
    __syncthreads();
    const int n = s_n;
    for (int64_t base = 0; base < H; base += static_cast<int64_t>(kCombThreads) * 8 * kCombVec) {
      float acc[kCombVec][8];
#pragma unroll
      for (int v = 0; v < kCombVec; ++v) {
        const int64_t c = base + (static_cast<int64_t>(v) * kCombThreads + tid) * 8;
        if (accumulate && c < H) {
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(out + t * ldo + c), acc[v]);
        } else {
#pragma unroll
          for (int h = 0; h < 8; ++h) acc[v][h] = 0.f;
        }
      }
      for (int jj = 0; jj < n; ++jj) {
        const uint16_t* row = y2 + static_cast<int64_t>(s_dst[jj]) * ldy;
        const float w = s_w[jj];
        uint4 u[kCombVec];
#pragma unroll
        for (int v = 0; v < kCombVec; ++v) {
          const int64_t c = base + (static_cast<int64_t>(v) * kCombThreads + tid) * 8;
          u[v] = c < H ? __ldg(reinterpret_cast<const uint4*>(row + c)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int v = 0; v < kCombVec; ++v) {
          const uint32_t x[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            acc[v][2 * h] = fmaf(w, __uint_as_float(x[h] << 16), acc[v][2 * h]);
            acc[v][2 * h + 1] = fmaf(w, __uint_as_float(x[h] & 0xFFFF0000u), acc[v][2 * h + 1]);
          }
        }
      }
      if (shared != nullptr) {
#pragma unroll
        for (int v = 0; v < kCombVec; ++v) {
          const int64_t c = base + (static_cast<int64_t>(v) * kCombThreads + tid) * 8;
          if (c >= H) continue;
          float f[8];
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(shared + t * lds + c)), f);
#pragma unroll
          for (int h = 0; h < 8; ++h) acc[v][h] = fmaf(1.0f, f[h], acc[v][h]);
        }
      }
#pragma unroll
      for (int v = 0; v < kCombVec; ++v) {
        const int64_t c = base + (static_cast<int64_t>(v) * kCombThreads + tid) * 8;
        if (c >= H) continue;
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(acc[v][2 * h], acc[v][2 * h + 1]);
          o[h] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(out + t * ldo + c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncthreads();   // s_dst / s_w / s_n are rewritten for the next token
  }
}

// Latency shape for a few tokens (all-experts decode: up to 9 routing slots
// per token): one CTA of kCombLatThreads per token, each thread owning
// kCombLatVec chunks of 8 columns, with the row loads of kCombLatSlots slots
// in flight at once.  Same per-element arithmetic and slot order as above, so
// the bytes are the same.
constexpr int kCombLatThreads = 512;
constexpr int kCombLatVec = 2;
constexpr int kCombLatSlots = 4;

__global__ void __launch_bounds__(kCombLatThreads) combine_latency_kernel(
    const uint16_t* __restrict__ y2, int64_t ldy, int64_t y_rows, const int32_t* __restrict__ dst_row,
    const float* __restrict__ topk_w, int32_t k, int64_t H, const uint16_t* __restrict__ shared, int64_t lds,
    int accumulate, uint16_t* __restrict__ out, int64_t ldo, int32_t* err) {
  grid_dependency_wait();
  grid_launch_dependents();
  __shared__ int32_t s_dst[32];
  __shared__ float s_w[32];
  __shared__ int s_n;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < 32) {
    int32_t d = -1;
    float w = 0.f;
    if (tid < k) {
      d = __ldg(dst_row + t * k + tid);
      if (d >= y_rows) {
        set_err(err, MOE_DEV_BAD_INDEX);
        d = -1;
      }
      w = __ldg(topk_w + t * k + tid);
    }
    const uint32_t valid = __ballot_sync(0xffffffffu, d >= 0);
    if (d >= 0) {
      const int slot = __popc(valid & ((1u << tid) - 1u));
      s_dst[slot] = d;
      s_w[slot] = w;
    }
    if (tid == 0) s_n = __popc(valid);
  }
  __syncthreads();
  const int n = s_n;
  for (int64_t base = 0; base < H; base += static_cast<int64_t>(kCombLatThreads) * 8 * kCombLatVec) {
    float acc[kCombLatVec][8];
#pragma unroll
    for (int v = 0; v < kCombLatVec; ++v) {
      const int64_t c = base + (static_cast<int64_t>(v) * kCombLatThreads + tid) * 8;
      if (accumulate && c < H) {
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(out + t * ldo + c), acc[v]);
      } else {
#pragma unroll
        for (int h = 0; h < 8; ++h) acc[v][h] = 0.f;
      }
    }
    for (int j0 = 0; j0 < n; j0 += kCombLatSlots) {
      uint4 u[kCombLatSlots][kCombLatVec];
#pragma unroll
      for (int j = 0; j < kCombLatSlots; ++j) {
        const uint16_t* row = y2 + static_cast<int64_t>(j0 + j < n ? s_dst[j0 + j] : 0) * ldy;
#pragma unroll
        for (int v = 0; v < kCombLatVec; ++v) {
          const int64_t c = base + (static_cast<int64_t>(v) * kCombLatThreads + tid) * 8;
          u[j][v] = (j0 + j < n && c < H) ? __ldg(reinterpret_cast<const uint4*>(row + c)) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < kCombLatSlots; ++j) {
        if (j0 + j >= n) break;
        const float w = s_w[j0 + j];
#pragma unroll
        for (int v = 0; v < kCombLatVec; ++v) {
          const uint32_t x[4] = {u[j][v].x, u[j][v].y, u[j][v].z, u[j][v].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            acc[v][2 * h] = fmaf(w, __uint_as_float(x[h] << 16), acc[v][2 * h]);
            acc[v][2 * h + 1] = fmaf(w, __uint_as_float(x[h] & 0xFFFF0000u), acc[v][2 * h + 1]);
          }
        }
      }
    }
    if (shared != nullptr) {
#pragma unroll
      for (int v = 0; v < kCombLatVec; ++v) {
        const int64_t c = base + (static_cast<int64_t>(v) * kCombLatThreads + tid) * 8;
        if (c >= H) continue;
        float f[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(shared + t * lds + c)), f);
#pragma unroll
        for (int h = 0; h < 8; ++h) acc[v][h] = fmaf(1.0f, f[h], acc[v][h]);
      }
    }
#pragma unroll
    for (int v = 0; v < kCombLatVec; ++v) {
      const int64_t c = base + (static_cast<int64_t>(v) * kCombLatThreads + tid) * 8;
      if (c >= H) continue;
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[v][2 * h], acc[v][2 * h + 1]);
        o[h] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(out + t * ldo + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int64_t moe_contig_rows_bound(int64_t assignments, int32_t E) {
  if (assignments < 0 || E < 0) return -1;
  return (assignments + 127ll * E) / 128 * 128;
}

namespace moe {

// Shared by moe_permute and moe_ffn: validate, run the index pass, then either
// gather already-quantised rows (q, s) or, when x is given, quantise the bf16
// token rows straight into the grouped layout.
int permute_launch(const uint8_t* q, const float* s, int64_t s_ld, const uint16_t* x, int64_t ldx,
                   const int32_t* topk_ids, int64_t T, int32_t H, int32_t k,
                   int32_t expert_begin, int32_t E, int32_t layout, int32_t max_m,
                   uint8_t* q_out, float* s_out, int64_t s_out_ld, int32_t* counts,
                   int32_t* offsets, int32_t* m_indices, int32_t* row_src, int32_t* dst_row,
                   int64_t rows_capacity, int32_t* err, cudaStream_t st, uint16_t* zero_out,
                   int64_t ldo, uint8_t* sf8_out, bool fuse_index, int32_t* lrank, int32_t* chunk_hist) {
  // (defaults for zero_out .. chunk_hist are in common.cuh)
  MOE_CHECK_ARG(T >= 0 && H > 0 && H % 128 == 0 && k >= 1 && k <= 32);
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts);
  MOE_CHECK_ARG(layout == MOE_LAYOUT_MASKED || layout == MOE_LAYOUT_CONTIG);
  MOE_CHECK_ARG(counts && row_src && q_out && (s_out || sf8_out));
  MOE_CHECK_ARG(aligned16(q_out) && aligned16(s_out) && aligned16(sf8_out));
  int64_t G;
  if (layout == MOE_LAYOUT_MASKED) {
    MOE_CHECK_ARG(max_m > 0 && static_cast<int64_t>(E) * max_m < (1ll << 31));
    G = max_m;
  } else {
    MOE_CHECK_ARG(offsets && m_indices && rows_capacity >= 0 && rows_capacity < (1ll << 31));
    MOE_CHECK_ARG(rows_capacity >= moe_contig_rows_bound(T * k, E));
    MOE_CHECK_ARG(s_out_ld >= rows_capacity);
    G = s_out_ld;
  }
  if (T > 0) {
    MOE_CHECK_ARG(topk_ids && dst_row);
    if (x != nullptr)
      MOE_CHECK_ARG(aligned16(x) && ldx >= H && ldx % 8 == 0);
    else
      MOE_CHECK_ARG(q && s && aligned16(q) && s_ld >= T);
  }
  MOE_CHECK_ARG(T * k < (1ll << 31));
  if (int rc = check_device()) return rc;
  // the index pass inside the quant-scatter kernel: masked layout, bf16 rows
  // to quantise, a few slots per token
  fuse_index = fuse_index && T > 0 && x != nullptr && layout == MOE_LAYOUT_MASKED && k <= kRankMaxK;
  IndexParams p{topk_ids, T * k, expert_begin, E, layout, max_m, rows_capacity,
                counts, offsets, m_indices, row_src, dst_row, err};
  if (fuse_index) {
    const bool packed = sf8_out != nullptr;
    auto kern = packed ? quant_scatter_kernel<8, 4, true, true> : quant_scatter_kernel<8, 4, false, true>;
    const ScaleOut so{s_out, sf8_out, G, static_cast<int32_t>((H / 128 + 3) / 4), static_cast<int32_t>((G + 127) / 128)};
    static int per_sm[2][64] = {{0}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    int& occ = per_sm[packed ? 1 : 0][dev];
    if (occ == 0 && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 256, 0) != cudaSuccess || occ < 1))
      return MOE_ERR_CUDA;
    const int64_t wave = static_cast<int64_t>(num_sms()) * occ;
    const RankArgs ra{topk_ids, expert_begin, E, max_m, counts, row_src, dst_row, err};
    return launch_pdl(kern, static_cast<unsigned>(T < wave ? T : wave), 256, 0, st, x, ldx, dst_row, T, k,
                      static_cast<int64_t>(H), q_out, so, k == 1 ? zero_out : nullptr, ldo, ra);
  }
  if (lrank != nullptr && chunk_hist != nullptr && T * k > kIdxMultiMinIds) {
    // many assignments: the index pass over many CTAs (rank per chunk, then finalize)
    const int64_t n = T * k;
    const int n_chunks = static_cast<int>((n + kIdxChunk - 1) / kIdxChunk);
    const size_t rsmem = sizeof(int32_t) * static_cast<size_t>(E + kIdxWarps * E);
    if (rsmem > 48 * 1024)
      MOE_CUDA_TRY(cudaFuncSetAttribute(permute_chunk_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(rsmem)));
    if (int rc = launch_pdl(permute_chunk_rank_kernel, static_cast<unsigned>(n_chunks), kIdxThreads, rsmem, st, p,
                            lrank, chunk_hist))
      return rc;
    if (int rc = launch_pdl(permute_finalize_kernel, static_cast<unsigned>((n + kFinThreads - 1) / kFinThreads),
                            kFinThreads, sizeof(int32_t) * 3 * static_cast<size_t>(E), st, p,
                            static_cast<const int32_t*>(lrank), static_cast<const int32_t*>(chunk_hist), n_chunks))
      return rc;
  } else {
  size_t smem = sizeof(int32_t) * (2 * E + kIdxWarps * E);
  const size_t ids_bytes = sizeof(int32_t) * static_cast<size_t>(T * k);
  const int ids_in_smem = smem + ids_bytes <= kIdxSmemLimit ? 1 : 0;
  if (ids_in_smem) smem += ids_bytes;
  if (smem > 48 * 1024) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(permute_index_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
  }
  if (int rc = launch_pdl(permute_index_kernel, 1, kIdxThreads, smem, st, p, ids_in_smem)) return rc;
  }
  if (T == 0) return MOE_OK;
  const int64_t n = T * k;
  const unsigned grid = static_cast<unsigned>((n + 3) / 4);
  if (x != nullptr) {
    // many rows: throughput shape; decode batches: latency shape
    const bool many = T >= 16384;
    const bool packed = sf8_out != nullptr;
    auto kern = packed ? (many ? quant_scatter_kernel<4, 7, true> : quant_scatter_kernel<8, 4, true>)
                       : (many ? quant_scatter_kernel<4, 7, false> : quant_scatter_kernel<8, 4, false>);
    const ScaleOut so{s_out, sf8_out, G, static_cast<int32_t>((H / 128 + 3) / 4), static_cast<int32_t>((G + 127) / 128)};
    const int threads = many ? 128 : 256;
    static int per_sm[4][64] = {{0}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    int& occ = per_sm[(many ? 1 : 0) + (packed ? 2 : 0)][dev];
    if (occ == 0 && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, 0) != cudaSuccess || occ < 1))
      return MOE_ERR_CUDA;
    const int64_t wave = static_cast<int64_t>(num_sms()) * occ;
    return launch_pdl(kern, static_cast<unsigned>(T < wave ? T : wave), threads, 0, st, x, ldx, dst_row, T, k,
                      static_cast<int64_t>(H), q_out, so, k == 1 ? zero_out : nullptr, ldo, RankArgs{});
  }
  return launch_pdl(permute_scatter_kernel, grid, 128, 0, st, q, s, s_ld, dst_row, n, k, H, q_out,
                    s_out, G);
}

}  // namespace moe

extern "C" int moe_permute(const uint8_t* q, const float* s, int64_t s_ld, const int32_t* topk_ids,
                           int64_t T, int32_t H, int32_t k, int32_t expert_begin, int32_t E,
                           int32_t layout, int32_t max_m, uint8_t* q_out, float* s_out,
                           int64_t s_out_ld, int32_t* counts, int32_t* offsets,
                           int32_t* m_indices, int32_t* row_src, int32_t* dst_row,
                           int64_t rows_capacity, int32_t* err, void* stream) {
  return permute_launch(q, s, s_ld, nullptr, 0, topk_ids, T, H, k, expert_begin, E, layout, max_m,
                        q_out, s_out, s_out_ld, counts, offsets, m_indices, row_src, dst_row,
                        rows_capacity, err, as_stream(stream), nullptr, 0, nullptr, false);
}

extern "C" int moe_combine(const uint16_t* Y2, int64_t ldy, int64_t y_rows, const int32_t* dst_row,
                           const float* topk_w, int64_t T, int32_t k, int32_t H, const uint16_t* shared_or_null,
                           int64_t lds, int32_t flags, uint16_t* out, int64_t ldo, int32_t* err, void* stream) {
  MOE_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && H > 0 && H % 8 == 0);
  MOE_CHECK_ARG((flags & ~MOE_COMBINE_ACCUMULATE) == 0);
  if (T == 0) return MOE_OK;
  MOE_CHECK_ARG(Y2 && dst_row && topk_w && out && aligned16(Y2) && aligned16(out));
  MOE_CHECK_ARG(ldy >= H && ldy % 8 == 0 && ldo >= H && ldo % 8 == 0 && y_rows >= 0);
  if (shared_or_null != nullptr) MOE_CHECK_ARG(aligned16(shared_or_null) && lds >= H && lds % 8 == 0);
  MOE_CHECK_ARG(T < (1ll << 31));
  if (int st = check_device()) return st;
  const int acc = (flags & MOE_COMBINE_ACCUMULATE) ? 1 : 0;
  // a few tokens (up to one per SM): one wide CTA per token, slots' loads in flight together
  if (T <= num_sms())
    return launch_pdl(combine_latency_kernel, static_cast<unsigned>(T), kCombLatThreads, 0, as_stream(stream), Y2,
                      ldy, y_rows, dst_row, topk_w, k, static_cast<int64_t>(H), shared_or_null, lds, acc, out, ldo,
                      err);
  static int per_sm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (per_sm[dev] == 0 &&
      (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[dev], combine_kernel, kCombThreads, 0) != cudaSuccess ||
       per_sm[dev] < 1))
    return MOE_ERR_CUDA;
  const int64_t wave = static_cast<int64_t>(num_sms()) * per_sm[dev];
  return launch_pdl(combine_kernel, static_cast<unsigned>(T < wave ? T : wave), kCombThreads, 0,
                    as_stream(stream), Y2, ldy, y_rows, dst_row, topk_w, k, static_cast<int64_t>(H), shared_or_null,
                    lds, acc, out, ldo, T, err);
}
