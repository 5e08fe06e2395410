// Grouped FP8 GEMM with power-of-two (UE8M0) block scales applied by the
// tensor cores: tcgen05.mma kind::mxf8f6f4.block_scale, the scales staged in
// tensor memory with tcgen05.cp.
//
// The pages describe the Blackwell FP8 GEMM they deploy as built on UMMA with
// an API that quantises and packs the input scales ("Deploying DeepSeek on
// GB200 NVL72 with PD and Large Scale EP (Part I)", section "Implementation
// details", DeepGEMM bullet).  This file is the reading in which the packed
// scales are UE8M0 exponent bytes, four k-blocks per 32-bit word, consumed by
// the MMA itself.  With a power-of-two scale per 128-deep block the MMA
// applies sa * sb exactly, so the fp32 accumulator stays in TMEM across all
// k-blocks and the epilogue drains it once per tile (the fp32-scale kernel in
// gemm.cu must promote every 128-deep block in the epilogue instead).
//
// Scale-factor placement in TMEM (measured on sm_103a): for the M = 128 A
// operand, row m's word sits at lane m, column base + m / 32; for the B
// operand, column n's word at lane n % 32, column base + n / 32; the byte of
// the word is chosen by the instruction descriptor's scale-factor id.
// tcgen05.cp .32x128b.warpx4 writes source row i (16 bytes) to lanes i,
// 32 + i, 64 + i, 96 + i, columns 0..3, so:
//  * activation scales are stored in global memory as 512-byte chunks (128
//    rows, one k-group) whose word 4 * (i % 32) + i / 32 is row i's word, and
//    one copy puts every row where the MMA reads it;
//  * weight scales are per 128 x 128 block, the same word for 128 rows: a
//    128-byte record of 32 copies, copied with a core-matrix stride of 0 so all
//    32 lanes read it, gives the 4 columns of a 128-row block.
#include <cstring>

#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kBsStages = 4;
constexpr uint32_t kBsA = BM * BK;          // 16 KB of A rows
constexpr uint32_t kBsB = BN * BK;          // 32 KB of B rows
constexpr uint32_t kBsSfA = 512;            // one activation chunk: 128 words
constexpr uint32_t kBsSfB = 128;            // one weight block's word, 32 copies
constexpr uint32_t kBsOffSfA = kBsA + kBsB;
constexpr uint32_t kBsOffSfB0 = kBsOffSfA + kBsSfA;
constexpr uint32_t kBsOffSfB1 = kBsOffSfB0 + kBsSfB;
constexpr uint32_t kBsStage = kBsA + kBsB + 1024;   // scale records padded to keep stages 1 KB aligned
// TMEM: the fp32 accumulator in columns [0, 256); two scale-factor regions of
// 16 columns (A: 4, B: 8) from column 256, alternating per k-group.
constexpr uint32_t kSfCol0 = 256;
constexpr uint32_t kSfRegion = 16;
constexpr int kBsBars = 2 * kBsStages + 3;   // full, empty [stages]; tfull, tempty, drain

struct BsArgs {
  const uint32_t* sfA;   // packed activation scale words
  int64_t sf_G;          // rows per scale group (masked: max_m; contiguous: sfA_ld)
  int32_t sf_NC;         // 128-row chunks per group
  int32_t KG;            // k-groups (4 k-blocks each)
  const uint32_t* sfB;   // packed weight scale records
  const int32_t* counts;     // masked
  const int32_t* offsets;    // contiguous
  const int32_t* m_indices;  // contiguous
  int64_t M_capacity;        // contiguous
  uint16_t* D;
  int64_t ldd;
  int32_t E, N, K, max_m, layout;
  int32_t* err;
  uint64_t wait_limit_ns;
  int32_t flags;
  // one routing slot per token (tokens-as-M kernel): write out[token] =
  // bf16(w * bf16(D)) instead of D, the combine's arithmetic for one slot
  const int32_t* row_src;
  const float* topk_w;
  uint16_t* out;
  int64_t ldo;
  // plain D leaves through TMA stores (tmD) for warps whose 32 rows are all valid
  int32_t tma_store;
};

// Instruction descriptor, kind::mxf8f6f4 with block scaling: D fp32, A = B =
// E4M3 (format 0), both K-major, scale factors UE8M0, both operands' scale
// byte = sf_id.
__host__ __device__ constexpr uint32_t idesc_e4m3_ue8m0(int M, int N, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4)         // B scale-factor byte
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (1u << 23)                                // UE8M0 scale factors
         | (static_cast<uint32_t>(M >> 4) << 24)     // M / 16
         | (static_cast<uint32_t>(sf_id) << 29);     // A scale-factor byte
}

__device__ __forceinline__ void umma_e4m3_ue8m0(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t tmem_sfa, uint32_t tmem_sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tmem_sfa), "r"(tmem_sfb), "r"(accumulate)
      : "memory");
}

// 32 rows x 16 bytes of shared memory to TMEM lanes i, 32+i, 64+i, 96+i,
// 4 columns; issued by one thread, ordered with its MMAs.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory descriptor of an unswizzled tcgen05.cp source: 8-row core
// matrices of 16-byte rows, `sbo` bytes apart (128: 32 consecutive rows; 0:
// the same 8 rows for all 32).
__device__ __forceinline__ uint64_t sdesc_cp_src(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;   // descriptor version; no swizzle
  return d;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_ue8m0_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmD,   // bf16 D, when p.tma_store
                          const BsArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // output staging after the stages, 1 KB aligned: kEpiWarps x kOutStageBytes
  uint8_t* ostage = smem + kBsStages * kBsStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ostage + kEpiWarps * kOutStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBsBars);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int32_t* sched_mem = reinterpret_cast<int32_t*>(tmem_slot + 4);
  const Sched sched{sched_mem, sched_mem + p.E + 1, sched_mem + 2 * p.E + 1};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kBsStages;
  const uint32_t tfull = empty0 + 8 * kBsStages;   // the tile's accumulator is complete
  const uint32_t tempty = tfull + 8;                // the epilogue has drained it
  const uint32_t drain = tempty + 8;                // MMAs in flight on an abort
  const int n_tiles = (p.N + BN - 1) / BN;
  const int KB = p.K / BK;
  const int NB = p.N / 128;
  volatile int* abort = abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBsStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.tma_store) tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // the schedule reads the counts / offsets after waiting for the previous
  // kernel, or before it with MOE_GEMM_EARLY_WEIGHTS (then the producer also
  // issues its first stages' weight tiles and weight scales before waiting)
  const bool early = (p.flags & MOE_GEMM_EARLY_WEIGHTS) != 0;
  if (!early) {
    grid_dependency_wait();
    grid_launch_dependents();
  }
  if (warp == 0) build_schedule(p, sched, n_tiles);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool early_producer = early && warp == 0 && lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL);
  if (early && !early_producer) {
    grid_dependency_wait();
    grid_launch_dependents();
  }
  const uint32_t tmem_base = *tmem_slot;
  const int total = sched.tile0[p.E];
  // No register split here: the epilogue holds one tile's 128 fp32 values per
  // thread only while it stores them, so every warp fits the launch allocation.
  if (warp < kEpiWarp0) {
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL)) {
        uint32_t it = 0;
        TileCursor cur;
        bool ok = true;
        struct Tile {
          int a_row, b_row;
          const uint32_t* sfa;   // the tile's 128-row chunk of its scale group
          const uint32_t* sfb0;  // the one or two 128-row weight blocks of its columns
          const uint32_t* sfb1;
        };
        auto tile_of = [&](int t, TileCursor& c) {
          c.seek(sched, t);
          const int e = c.e;
          const int l = t - sched.tile0[e];
          const int mt = l / n_tiles, nt = l % n_tiles;
          const bool half = (nt == n_tiles - 1) && (p.N % BN) != 0;
          Tile tl;
          tl.a_row = sched.rbase[e] + mt * BM;
          tl.b_row = e * p.N + nt * BN;
          const int64_t grp = tl.a_row / p.sf_G, r_in = tl.a_row - grp * p.sf_G;
          tl.sfa = p.sfA + (grp * p.KG * p.sf_NC + r_in / BM) * 128;
          tl.sfb0 = p.sfB + (static_cast<int64_t>(e) * NB + 2 * nt) * p.KG * 32;
          tl.sfb1 = half ? tl.sfb0 : tl.sfb0 + static_cast<int64_t>(p.KG) * 32;
          return tl;
        };
        // a stage's weight half (the B tile and, every fourth k-block, the
        // weight scale records) with the stage's whole byte count expected ...
        auto issue_b = [&](uint32_t s, int kb, const Tile& tl) {
          const bool sf = (kb & 3) == 0;
          const uint32_t st = smem_u32(smem + s * kBsStage);
          mbar_arrive_expect_tx(full0 + 8 * s, kBsA + kBsB + (sf ? kBsSfA + 2 * kBsSfB : 0));
          tma_load_2d(st + kBsA, &tmB, full0 + 8 * s, kb * BK, tl.b_row);
          if (sf) {
            bulk_g2s(st + kBsOffSfB0, tl.sfb0 + (kb >> 2) * 32, kBsSfB, full0 + 8 * s);
            bulk_g2s(st + kBsOffSfB1, tl.sfb1 + (kb >> 2) * 32, kBsSfB, full0 + 8 * s);
          }
        };
        // ... and its activation half (the A tile and the activation scale chunk)
        auto issue_a = [&](uint32_t s, int kb, const Tile& tl) {
          const uint32_t st = smem_u32(smem + s * kBsStage);
          tma_load_2d(st, &tmA, full0 + 8 * s, kb * BK, tl.a_row);
          if ((kb & 3) == 0)
            bulk_g2s(st + kBsOffSfA, tl.sfa + static_cast<int64_t>(kb >> 2) * p.sf_NC * 128, kBsSfA, full0 + 8 * s);
        };
        uint32_t pre = 0;   // stages whose weight half went out before the wait
        if (early_producer) {
          TileCursor c0;
          for (int t = blockIdx.x; t < total && pre < static_cast<uint32_t>(kBsStages); t += gridDim.x) {
            const Tile tl = tile_of(t, c0);
            for (int kb = 0; kb < KB && pre < static_cast<uint32_t>(kBsStages); ++kb, ++pre) issue_b(pre, kb, tl);
          }
          grid_dependency_wait();
          grid_launch_dependents();
        }
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
          const Tile tl = tile_of(t, cur);
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t s = it % kBsStages, ph = (it / kBsStages) & 1;
            if (it >= pre) {
              if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, p.err, p.wait_limit_ns)) {
                ok = false;
                break;
              }
              issue_b(s, kb, tl);
            }
            issue_a(s, kb, tl);
          }
        }
        if (!ok) {
          // drain: let the copies already issued land before the CTA exits
          const uint32_t first = it > kBsStages ? it - kBsStages : 0;
          for (uint32_t j = first; j < it; ++j) {
            int dummy = 0;
            mbar_wait_bounded(full0 + 8 * (j % kBsStages), (j / kBsStages) & 1, &dummy, nullptr,
                              p.wait_limit_ns / 10);
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        uint32_t it = 0, tile_no = 0, kgroup = 0;
        bool ok = true, issued = false;
        TileCursor cur;
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++tile_no) {
          cur.seek(sched, t);
          const int nt = (t - sched.tile0[cur.e]) % n_tiles;
          const bool half = (nt == n_tiles - 1) && (p.N % BN) != 0;
          // the accumulator is free once the epilogue has read the previous tile
          if (!mbar_wait_bounded(tempty, (tile_no & 1) ^ 1, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t s = it % kBsStages, ph = (it / kBsStages) & 1;
            if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, p.err, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * kBsStage);
            if ((kb & 3) == 0 && kb > 0) ++kgroup;   // alternate the scale regions across k-groups and tiles
            const uint32_t sfa = tmem_base + kSfCol0 + (kgroup & 1) * kSfRegion;
            const uint32_t sfb = sfa + 4;
            if ((kb & 3) == 0) {
              tmem_cp_32x128b_x4(sfa, sdesc_cp_src(st + kBsOffSfA, 128));
              tmem_cp_32x128b_x4(sfb, sdesc_cp_src(st + kBsOffSfB0, 0));
              tmem_cp_32x128b_x4(sfb + 4, sdesc_cp_src(st + kBsOffSfB1, 0));
            }
            const uint64_t ad = sdesc_kmajor_sw128(st);
            const uint64_t bd = sdesc_kmajor_sw128(st + kBsA);
            const uint32_t idesc = idesc_e4m3_ue8m0(BM, half ? BN / 2 : BN, kb & 3);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)  // 32 bytes of K per MMA: +2 in the 16-byte address field
              umma_e4m3_ue8m0(tmem_base, ad + 2 * k, bd + 2 * k, idesc, sfa, sfb, (kb > 0 || k > 0) ? 1u : 0u);
            umma_commit(empty0 + 8 * s);
            issued = true;
          }
          if (ok) umma_commit(tfull);
          ++kgroup;
        }
        if (!ok && issued) {  // the MMAs in flight finish before TMEM is freed
          umma_commit(drain);
          int dummy = 0;
          mbar_wait_bounded(drain, 0, &dummy, nullptr, p.wait_limit_ns / 10);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int g = (warp - kEpiWarp0) >> 2;  // column half
    uint32_t tile_no = 0;
    TileCursor cur;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tile_no) {
      cur.seek(sched, t);
      const int e = cur.e;
      const int l = t - sched.tile0[e];
      const int mt = l / n_tiles, nt = l % n_tiles;
      const bool half = (nt == n_tiles - 1) && (p.N % BN) != 0;
      const bool active = !(half && g == 1);
      const int r_local = mt * BM + q * 32 + lane;
      const int64_t gr = static_cast<int64_t>(sched.rbase[e]) + r_local;
      bool row_ok = r_local < sched.rext[e];
      if (row_ok && p.layout == MOE_LAYOUT_CONTIG) row_ok = __ldg(p.m_indices + gr) >= 0;
      // single-slot combine: the row's token and weight, loaded while the tile computes
      int64_t tok = 0;
      float wtok = 0.f;
      if (p.out != nullptr && row_ok) {
        tok = __ldg(p.row_src + gr);
        wtok = __ldg(p.topk_w + tok);
      }
      int got = 1;
      if (lane == 0) got = mbar_wait_bounded(tfull, tile_no & 1, abort, p.err, p.wait_limit_ns);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      // the warp's 32 rows x 128 columns, all loads in flight, then the
      // accumulator is handed back before the stores
      uint32_t v[128];
      if (active) {
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + g * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(tbase + c * 16, r);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[c * 16 + i] = r[i];
        }
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      if (active) {
        // the warp's 32 rows x 128 columns leave in four 32-column quarters
        // through its 2 KB of staging: as one TMA store of the 32 x 32 box when
        // all 32 rows are valid D rows, else 8 lanes per row store 64-byte
        // segments (also the single-slot combine's scattered output rows)
        const bool to_out = p.out != nullptr;
        const int n0 = nt * BN + g * 128;
        uint16_t* row_base = to_out ? p.out + tok * p.ldo + n0 : p.D + gr * p.ldd + n0;
        auto rb = [](float x) { return __bfloat162float(__float2bfloat16_rn(x)); };
        const uint32_t stg = smem_u32(ostage + (warp - kEpiWarp0) * kOutStageBytes);
        const bool by_tma = p.tma_store && !to_out && __all_sync(0xffffffffu, row_ok);
        const int32_t d_row0 = static_cast<int32_t>(gr - lane);
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
          if (lane == 0 && p.tma_store) bulk_wait_read_all();   // the last TMA store has read the slot
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = qc * 4 + c;   // 16-byte chunk of the row: columns 8cc .. 8cc+7
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float a0 = __uint_as_float(v[cc * 8 + 2 * h]), a1 = __uint_as_float(v[cc * 8 + 2 * h + 1]);
              const __nv_bfloat162 bb = to_out ? __floats2bfloat162_rn(fmaf(wtok, rb(a0), 0.f), fmaf(wtok, rb(a1), 0.f))
                                               : __floats2bfloat162_rn(a0, a1);
              o[h] = *reinterpret_cast<const uint32_t*>(&bb);
            }
            st_shared_v4(stg + out_stage_slot(lane, c), make_uint4(o[0], o[1], o[2], o[3]));
          }
          if (by_tma) {
            fence_proxy_async_shared();   // this lane's staging writes, visible to the TMA
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, stg, n0 + qc * 32, d_row0);
              bulk_commit_group();
            }
            continue;
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 8 * j + (lane >> 2), c = lane & 3;   // row of the warp, chunk of the quarter
            const uint4 val = ld_shared_v4(stg + out_stage_slot(r, c));
            const bool ok_r = __shfl_sync(0xffffffffu, row_ok, r);
            uint16_t* base_r =
                reinterpret_cast<uint16_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(row_base), r));
            if (ok_r) *reinterpret_cast<uint4*>(base_r + qc * 32 + c * 8) = val;
          }
          __syncwarp();
        }
      }
    }
    // the TMA stores issued by this warp are complete before the CTA ends
    if (p.tma_store && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// =============================================================================
// Weights-as-M variant for the masked (decode) layout: 128 weight rows (one
// 128 x 128 scale block row) are the M side, the expert's tokens the N side
// (16 .. BNT per tile, sized at run time), so decode streams each expert's
// weights once per BNT tokens.  Scale factors: A = the weight block's record
// (one word for all rows, copied with core-matrix stride 0); B = the tokens'
// packed chunk -- column n of the tile reads lane n % 32, column n / 32, and the
// chunk puts token c * 32 + i at lane i, column c, so a tile that starts o rows
// into the chunk reads from column o / 32 on.  The accumulator (D^T: weight
// rows in lanes, tokens in columns) is double-buffered across tiles.
// =============================================================================
template <int BNT>
struct Ue8m0WeightsM {
  static constexpr uint32_t kW = 128 * BK;                      // weight tile
  static constexpr uint32_t kT = BNT * BK;                      // token tile (max)
  static constexpr uint32_t kOffSfW = kW + kT;                  // weight record (128 B)
  static constexpr uint32_t kOffSfT = kOffSfW + 128;            // token chunk (512 B)
  static constexpr uint32_t kStage = kW + kT + 1024;
  static constexpr int kStages = (196608 / kStage) > 8 ? 8 : (196608 / kStage);
  static constexpr int kBars = 2 * kStages + 5;                 // full, empty; tfull[2], tempty[2], drain
  static_assert(BNT == 64 || BNT == 128, "one token chunk per tile");
  static constexpr size_t smem_bytes(int E) {
    return 1024 + static_cast<size_t>(kStages) * kStage + kBars * 8 + 16 + sizeof(int32_t) * (3 * E + 1);
  }
};

template <int BNT>
__device__ void build_schedule_wm_bs(const BsArgs& p, const Sched& s, int nblk) {
  const int lane = threadIdx.x & 31;
  const int per = (p.E + 31) / 32;
  const int e0 = min(lane * per, p.E), e1 = min(e0 + per, p.E);
  int local = 0;
  bool overflow = false, bad = false;
  for (int e = e0; e < e1; ++e) {
    int c = __ldcg(p.counts + e);   // from L2: may be read before the grid dependency wait
    if (c > p.max_m) { overflow = true; c = p.max_m; }
    if (c < 0) { bad = true; c = 0; }
    s.rbase[e] = e * p.max_m;
    s.rext[e] = c;
    local += (c + BNT - 1) / BNT * nblk;
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
    run += (s.rext[e] + BNT - 1) / BNT * nblk;
  }
  if (lane == 31) s.tile0[p.E] = incl;
  if (blockIdx.x == 0) {
    if (overflow) set_err(p.err, MOE_DEV_OVERFLOW);
    if (bad) set_err(p.err, MOE_DEV_BAD_INDEX);
  }
}

template <int BNT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_ue8m0_weights_m_kernel(const __grid_constant__ TokenMaps tmT, const __grid_constant__ CUtensorMap tmW,
                                    const BsArgs p) {
  using C = Ue8m0WeightsM<BNT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int32_t* sched_mem = reinterpret_cast<int32_t*>(tmem_slot + 4);
  const Sched sched{sched_mem, sched_mem + p.E + 1, sched_mem + 2 * p.E + 1};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t tfull0 = empty0 + 8 * C::kStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const int nblk = p.N / 128;
  const int KB = p.K / BK;
  volatile int* abort = abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < 4) tma_prefetch_desc(&tmT.box[lane]);
  if (warp == 0 && lane == 4) tma_prefetch_desc(&tmW);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // the schedule reads the counts after waiting for the previous kernel, or
  // before it with MOE_GEMM_EARLY_WEIGHTS (then the producer also issues its
  // first stages' weight tiles and weight scale records before waiting)
  const bool early = (p.flags & MOE_GEMM_EARLY_WEIGHTS) != 0;
  if (!early) {
    grid_dependency_wait();
    grid_launch_dependents();
  }
  if (warp == 0) build_schedule_wm_bs<BNT>(p, sched, nblk);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool early_producer = early && warp == 0 && lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL);
  if (early && !early_producer) {
    grid_dependency_wait();
    grid_launch_dependents();
  }
  const uint32_t tmem_base = *tmem_slot;
  const int total = sched.tile0[p.E];
  if (warp < kEpiWarp0) {
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL)) {
        const uint64_t pol_w = l2_policy_evict_first();   // weights stream through once
        uint32_t it = 0;
        TileCursor cur;
        bool ok = true;
        struct Tile {
          int ncols, t_row, w_row;
          const uint32_t* sfw;   // the weight block's scale records
          const uint32_t* sft;   // the tokens' packed scale chunk
        };
        auto tile_of = [&](int t, TileCursor& c) {
          c.seek(sched, t);
          const int e = c.e;
          const int l = t - sched.tile0[e];
          const int j = l / nblk, nb = l % nblk;
          Tile tl;
          tl.ncols = (min(BNT, sched.rext[e] - j * BNT) + 15) & ~15;
          tl.t_row = sched.rbase[e] + j * BNT;
          tl.w_row = e * p.N + nb * 128;
          tl.sfw = p.sfB + (static_cast<int64_t>(e) * nblk + nb) * p.KG * 32;
          tl.sft = p.sfA + (static_cast<int64_t>(e) * p.KG * p.sf_NC + (j * BNT) / 128) * 128;
          return tl;
        };
        // a stage's weight half (the weight tile and, every fourth k-block,
        // its scale record) with the stage's whole byte count expected ...
        auto issue_w = [&](uint32_t s, int kb, const Tile& tl) {
          const bool sf = (kb & 3) == 0;
          const uint32_t st = smem_u32(smem + s * C::kStage);
          mbar_arrive_expect_tx(full0 + 8 * s, C::kW + tl.ncols * BK + (sf ? 128 + 512 : 0));
          tma_load_2d_hint(st, &tmW, full0 + 8 * s, kb * BK, tl.w_row, pol_w);
          if (sf) bulk_g2s(st + C::kOffSfW, tl.sfw + (kb >> 2) * 32, 128, full0 + 8 * s);
        };
        // ... and its token half (the token rows and their scale chunk)
        auto issue_t = [&](uint32_t s, int kb, const Tile& tl) {
          const uint32_t st = smem_u32(smem + s * C::kStage);
          for (int r = 0; r < tl.ncols;) {
            const int left = tl.ncols - r;
            const int i = left >= 128 ? 3 : left >= 64 ? 2 : left >= 32 ? 1 : 0;
            tma_load_2d(st + C::kW + r * BK, &tmT.box[i], full0 + 8 * s, kb * BK, tl.t_row + r);
            r += 16 << i;
          }
          if ((kb & 3) == 0)
            bulk_g2s(st + C::kOffSfT, tl.sft + static_cast<int64_t>(kb >> 2) * p.sf_NC * 128, 512, full0 + 8 * s);
        };
        uint32_t pre = 0;   // stages whose weight half went out before the wait
        if (early_producer) {
          TileCursor c0;
          for (int t = blockIdx.x; t < total && pre < static_cast<uint32_t>(C::kStages); t += gridDim.x) {
            const Tile tl = tile_of(t, c0);
            for (int kb = 0; kb < KB && pre < static_cast<uint32_t>(C::kStages); ++kb, ++pre) issue_w(pre, kb, tl);
          }
          grid_dependency_wait();
          grid_launch_dependents();
        }
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
          const Tile tl = tile_of(t, cur);
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1;
            if (it >= pre) {
              if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, p.err, p.wait_limit_ns)) {
                ok = false;
                break;
              }
              issue_w(s, kb, tl);
            }
            issue_t(s, kb, tl);
          }
        }
        if (!ok) {
          const uint32_t first = it > static_cast<uint32_t>(C::kStages) ? it - C::kStages : 0;
          for (uint32_t jj = first; jj < it; ++jj) {
            int dummy = 0;
            mbar_wait_bounded(full0 + 8 * (jj % C::kStages), (jj / C::kStages) & 1, &dummy, nullptr,
                              p.wait_limit_ns / 10);
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        uint32_t it = 0, acc = 0, kgroup = 0;
        bool ok = true, issued = false;
        TileCursor cur;
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++acc) {
          cur.seek(sched, t);
          const int e = cur.e;
          const int j = (t - sched.tile0[e]) / nblk;
          const int ntok = min(BNT, sched.rext[e] - j * BNT);
          const int ncols = (ntok + 15) & ~15;
          const uint32_t b = acc & 1, tph = (acc >> 1) & 1;
          if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t o32 = static_cast<uint32_t>(((j * BNT) % 128) / 32);   // tile start in its token chunk
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1;
            if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, p.err, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * C::kStage);
            if ((kb & 3) == 0 && kb > 0) ++kgroup;
            const uint32_t sfa = tmem_base + kSfCol0 + (kgroup & 1) * kSfRegion;
            if ((kb & 3) == 0) {
              tmem_cp_32x128b_x4(sfa, sdesc_cp_src(st + C::kOffSfW, 0));
              tmem_cp_32x128b_x4(sfa + 4, sdesc_cp_src(st + C::kOffSfT, 128));
            }
            const uint64_t wd = sdesc_kmajor_sw128(st);
            const uint64_t td = sdesc_kmajor_sw128(st + C::kW);
            const uint32_t idesc = idesc_e4m3_ue8m0(128, ncols, kb & 3);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              umma_e4m3_ue8m0(tmem_base + b * BNT, wd + 2 * k, td + 2 * k, idesc, sfa, sfa + 4 + o32,
                              (kb > 0 || k > 0) ? 1u : 0u);
            umma_commit(empty0 + 8 * s);
            issued = true;
          }
          if (ok) umma_commit(tfull0 + 8 * b);
          ++kgroup;
        }
        if (!ok && issued) {
          umma_commit(drain);
          int dummy = 0;
          mbar_wait_bounded(drain, 0, &dummy, nullptr, p.wait_limit_ns / 10);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lanes = weight rows q*32 .. q*32+31
    const int g = (warp - kEpiWarp0) >> 2;  // token columns: even / odd 16-column chunks
    uint32_t acc = 0;
    TileCursor cur;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++acc) {
      cur.seek(sched, t);
      const int e = cur.e;
      const int l = t - sched.tile0[e];
      const int j = l / nblk, nb = l % nblk;
      const int ntok = min(BNT, sched.rext[e] - j * BNT);
      const uint32_t b = acc & 1, tph = (acc >> 1) & 1;
      int got = 1;
      if (lane == 0) got = mbar_wait_bounded(tfull0 + 8 * b, tph, abort, p.err, p.wait_limit_ns);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      // this warp's 16-column chunks: g, g + 2, ... (up to BNT / 32 of them)
      constexpr int kMy = BNT / 32;
      uint32_t v[kMy][16];
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * BNT;
#pragma unroll
      for (int i = 0; i < kMy; ++i) {
        const int ch = g + 2 * i;
        if (ch * 16 < ntok) tmem_ld_32x32b_x16(tbase + ch * 16, v[i]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * b);
      // D[e][token][n]: per token column, the warp writes 32 consecutive n
      const int64_t n = static_cast<int64_t>(nb) * 128 + q * 32 + lane;
      uint16_t* drow = p.D + (static_cast<int64_t>(e) * p.max_m + j * BNT) * p.N + n;
#pragma unroll
      for (int i = 0; i < kMy; ++i) {
        const int ch = g + 2 * i;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int tok = ch * 16 + c;
          if (tok < ntok) {
            const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(v[i][c]));
            drow[static_cast<int64_t>(tok) * p.N] = *reinterpret_cast<const uint16_t*>(&bv);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BNT>
int launch_ue8m0_weights_m(const uint8_t* A, const uint8_t* B, BsArgs& a, cudaStream_t stream) {
  using C = Ue8m0WeightsM<BNT>;
  TokenMaps tmT;
  CUtensorMap tmW;
  const uint64_t t_rows = static_cast<uint64_t>(a.E) * a.max_m;
  for (int i = 0; i < 4; ++i) {
    const uint32_t h = (16u << i) <= t_rows ? (16u << i) : 16u;
    if (int st = make_tmap_u8_sw128(&tmT.box[i], A, t_rows, a.K, a.K, h)) return st;
  }
  if (int st = make_tmap_u8_sw128(&tmW, B, static_cast<uint64_t>(a.E) * a.N, a.K, a.K, 128)) return st;
  const size_t smem = C::smem_bytes(a.E);
  if (int st = prepare_kernel(gemm_fp8_ue8m0_weights_m_kernel<BNT>, smem, false)) return st;
  if (a.wait_limit_ns == 0) a.wait_limit_ns = kWaitLimitNs;
  if (a.flags & MOE_GEMM_DEBUG_STALL) a.wait_limit_ns = 200ull * 1000ull * 1000ull;
  const int64_t tiles_upper = static_cast<int64_t>(a.E) * ((a.max_m + BNT - 1) / BNT) * (a.N / 128);
  int64_t grid = num_sms();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) grid = 1;
  return launch_pdl(gemm_fp8_ue8m0_weights_m_kernel<BNT>, static_cast<unsigned>(grid), kThreads, smem, stream, tmT,
                    tmW, a);
}

size_t ue8m0_smem_bytes(int E) {
  return 1024 + static_cast<size_t>(kBsStages) * kBsStage + kEpiWarps * kOutStageBytes + kBsBars * 8 + 16 +
         sizeof(int32_t) * (3 * E + 1);
}

int launch_ue8m0(const uint8_t* A, int64_t a_rows, int64_t lda, const uint8_t* B, int64_t tiles_upper, BsArgs& a,
                 cudaStream_t stream) {
  CUtensorMap tmA, tmB, tmD;
  if (int st = make_tmap_u8_sw128(&tmA, A, a_rows, a.K, lda, BM)) return st;
  if (int st = make_tmap_u8_sw128(&tmB, B, static_cast<uint64_t>(a.E) * a.N, a.K, a.K, BN)) return st;
  // plain bf16 D (a_rows rows of ldd) leaves through TMA stores when it can be
  // mapped; the single-slot combine's output rows through the LSU path
  std::memset(&tmD, 0, sizeof(tmD));
  a.tma_store = 0;
  if (a.out == nullptr && a.D != nullptr &&
      make_tmap_b16_out(&tmD, a.D, static_cast<uint64_t>(a_rows), a.N, static_cast<uint64_t>(a.ldd) * 2) == MOE_OK)
    a.tma_store = 1;
  const size_t smem = ue8m0_smem_bytes(a.E);
  if (a.wait_limit_ns == 0) a.wait_limit_ns = kWaitLimitNs;
  if (a.flags & MOE_GEMM_DEBUG_STALL) a.wait_limit_ns = 200ull * 1000ull * 1000ull;
  if (int st = prepare_kernel(gemm_fp8_ue8m0_kernel, smem, false)) return st;
  int64_t grid = num_sms();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) grid = 1;
  return launch_pdl(gemm_fp8_ue8m0_kernel, static_cast<unsigned>(grid), kThreads, smem, stream, tmA, tmB, tmD, a);
}

// ---------------------------------------------------------------- packing
// The UE8M0 byte of a power-of-two fp32 scale 2^e is its exponent field e + 127
// (0xFF for an infinite scale).
__device__ __forceinline__ uint32_t ue8m0_byte(float s) { return (__float_as_uint(s) >> 23) & 0xFFu; }

// Power-of-two activation scales s[((r / G) * KB + kb) * G + r % G] (the grouped
// layout of the fp32 scales) -> packed words (see moe_fp8.h).  One thread per
// output word.
__global__ void __launch_bounds__(256) pack_ue8m0_act_kernel(const float* __restrict__ sc, int64_t groups,
                                                              int64_t G, int64_t rows, int64_t KB, int32_t KG,
                                                              int32_t NC, uint32_t* __restrict__ sf) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t words = groups * KG * NC * 128;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < words;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pos = w % 128;                      // position in the 512-byte chunk
    const int64_t c = (w / 128) % NC;                 // chunk of the group
    const int64_t gk = (w / (128 * NC)) % KG;         // k-group
    const int64_t grp = w / (128 * static_cast<int64_t>(NC) * KG);
    const int64_t i = (pos % 4) * 32 + pos / 4;       // row of the chunk stored here
    const int64_t r_in = c * 128 + i;
    const int64_t r = grp * G + r_in;
    uint32_t word = 0x7F7F7F7Fu;                      // unused bytes: scale 1
    if (r_in < G && r < rows) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t kb = gk * 4 + b;
        if (kb < KB) {
          const uint32_t byte = ue8m0_byte(sc[(grp * KB + kb) * G + r_in]);
          word = (word & ~(0xFFu << (8 * b))) | (byte << (8 * b));
        }
      }
    }
    sf[w] = word;
  }
}

// Power-of-two weight scales s[E, N/128, K/128] -> 32 copies of each block's
// packed word per k-group: sf[((e * NB + nb) * KG + g) * 32 + j].
__global__ void __launch_bounds__(256) pack_ue8m0_weight_kernel(const float* __restrict__ sc, int64_t blocks,
                                                                 int64_t KB, int32_t KG, uint32_t* __restrict__ sf) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t words = blocks * KG * 32;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < words;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t gk = (w / 32) % KG;
    const int64_t blk = w / (32 * static_cast<int64_t>(KG));
    uint32_t word = 0x7F7F7F7Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t kb = gk * 4 + b;
      if (kb < KB) word = (word & ~(0xFFu << (8 * b))) | (ue8m0_byte(sc[blk * KB + kb]) << (8 * b));
    }
    sf[w] = word;
  }
}

inline int32_t kgroups(int64_t K) { return static_cast<int32_t>((K / 128 + 3) / 4); }

}  // namespace

// GEMM2 of the UE8M0 FFN with the single-slot combine in the epilogue (k = 1,
// tokens-as-M kernel): routed row r goes to out[row_src[r]] scaled by
// topk_w[row_src[r]].  Contiguous layout when offsets != NULL, else masked.
int gemm_ue8m0_combine1(const uint8_t* A, const uint32_t* sfA, const uint8_t* B, const uint32_t* sfB,
                        const int32_t* counts, const int32_t* offsets, const int32_t* m_indices, int64_t rows,
                        int32_t E, int32_t max_m, int32_t N, int32_t K, const int32_t* row_src,
                        const float* topk_w, uint16_t* out, int64_t ldo, int32_t flags, int32_t* err,
                        cudaStream_t st) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0 && rows > 0);
  MOE_CHECK_ARG(A && sfA && B && sfB && row_src && topk_w && out && aligned16(out) && ldo >= N && ldo % 8 == 0);
  if (int rc = check_device()) return rc;
  BsArgs a{};
  a.sfA = sfA;
  a.KG = kgroups(K);
  a.sfB = sfB;
  a.E = E;
  a.N = N;
  a.K = K;
  a.err = err;
  a.flags = flags & ~MOE_GEMM_DEBUG_STALL;
  a.row_src = row_src;
  a.topk_w = topk_w;
  a.out = out;
  a.ldo = ldo;
  if (offsets != nullptr) {
    MOE_CHECK_ARG(m_indices && rows % BM == 0);
    a.sf_G = rows;
    a.sf_NC = static_cast<int32_t>(rows / BM);
    a.offsets = offsets;
    a.m_indices = m_indices;
    a.M_capacity = rows;
    a.layout = MOE_LAYOUT_CONTIG;
    return launch_ue8m0(A, rows, K, B, (rows / BM) * ((N + BN - 1) / BN), a, st);
  }
  MOE_CHECK_ARG(counts && max_m > 0 && rows == static_cast<int64_t>(E) * max_m);
  a.sf_G = max_m;
  a.sf_NC = (max_m + BM - 1) / BM;
  a.counts = counts;
  a.max_m = max_m;
  a.layout = MOE_LAYOUT_MASKED;
  return launch_ue8m0(A, rows, K, B, static_cast<int64_t>(E) * ((max_m + BM - 1) / BM) * ((N + BN - 1) / BN), a,
                      st);
}

}  // namespace moe

using namespace moe;

extern "C" int64_t moe_ue8m0_act_words(int64_t groups, int64_t G, int64_t K) {
  if (groups < 0 || G <= 0 || K <= 0 || K % 128 != 0) return -1;
  return groups * kgroups(K) * ((G + 127) / 128) * 128;
}

extern "C" int64_t moe_ue8m0_weight_words(int64_t E, int64_t N, int64_t K) {
  if (E < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return -1;
  return E * (N / 128) * kgroups(K) * 32;
}

extern "C" int moe_pack_ue8m0_act(const float* s, int64_t groups, int64_t G, int64_t rows, int64_t K,
                                  uint32_t* sf, void* stream) {
  MOE_CHECK_ARG(groups >= 0 && G > 0 && K > 0 && K % 128 == 0 && rows >= 0 && rows <= groups * G);
  if (groups == 0) return MOE_OK;
  MOE_CHECK_ARG(s && sf && (reinterpret_cast<uintptr_t>(sf) & 15u) == 0 && (reinterpret_cast<uintptr_t>(s) & 3u) == 0);
  if (int st = check_device()) return st;
  const int64_t words = moe_ue8m0_act_words(groups, G, K);
  const int64_t blocks = (words + 255) / 256;
  return launch_pdl(pack_ue8m0_act_kernel, static_cast<unsigned>(blocks < 65535 ? blocks : 65535), 256, 0,
                    as_stream(stream), s, groups, G, rows, K / 128, kgroups(K),
                    static_cast<int32_t>((G + 127) / 128), sf);
}

extern "C" int moe_pack_ue8m0_weight(const float* s, int64_t E, int64_t N, int64_t K, uint32_t* sf,
                                     void* stream) {
  MOE_CHECK_ARG(E >= 0 && N > 0 && K > 0 && N % 128 == 0 && K % 128 == 0);
  if (E == 0) return MOE_OK;
  MOE_CHECK_ARG(s && sf && (reinterpret_cast<uintptr_t>(sf) & 15u) == 0 && (reinterpret_cast<uintptr_t>(s) & 3u) == 0);
  if (int st = check_device()) return st;
  const int64_t words = moe_ue8m0_weight_words(E, N, K);
  const int64_t blocks = (words + 255) / 256;
  return launch_pdl(pack_ue8m0_weight_kernel, static_cast<unsigned>(blocks < 65535 ? blocks : 65535), 256, 0,
                    as_stream(stream), s, E * (N / 128), K / 128, kgroups(K), sf);
}

extern "C" int moe_gemm_fp8_contig_ue8m0(const uint8_t* A, int64_t lda, const uint32_t* sfA, int64_t sfA_ld,
                                         const uint8_t* B, const uint32_t* sfB, const int32_t* offsets,
                                         const int32_t* m_indices, int64_t M_capacity, int32_t E, int32_t N,
                                         int32_t K, uint16_t* D, int64_t ldd, int32_t flags, int32_t* err,
                                         void* stream) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(M_capacity >= 0 && M_capacity % BM == 0 && M_capacity < (1ll << 31));
  if (M_capacity == 0) return MOE_OK;
  MOE_CHECK_ARG(A && sfA && B && sfB && offsets && m_indices && D);
  MOE_CHECK_ARG(aligned16(A) && aligned16(B) && aligned16(D) && aligned16(sfA) && aligned16(sfB));
  MOE_CHECK_ARG(lda >= K && lda % 16 == 0 && sfA_ld >= M_capacity && sfA_ld % BM == 0 && ldd >= N && ldd % 8 == 0);
  MOE_CHECK_ARG(static_cast<int64_t>(E) * N < (1ll << 31));
  if (int st = check_device()) return st;
  BsArgs a{};
  a.sfA = sfA;
  a.sf_G = sfA_ld;
  a.sf_NC = static_cast<int32_t>(sfA_ld / BM);
  a.KG = kgroups(K);
  a.sfB = sfB;
  a.offsets = offsets;
  a.m_indices = m_indices;
  a.M_capacity = M_capacity;
  a.D = D;
  a.ldd = ldd;
  a.E = E;
  a.N = N;
  a.K = K;
  a.layout = MOE_LAYOUT_CONTIG;
  a.err = err;
  a.flags = flags;
  const int64_t tiles = (M_capacity / BM) * ((N + BN - 1) / BN);
  return launch_ue8m0(A, M_capacity, lda, B, tiles, a, as_stream(stream));
}

extern "C" int moe_gemm_fp8_masked_ue8m0(const uint8_t* A, const uint32_t* sfA, const uint8_t* B,
                                         const uint32_t* sfB, const int32_t* counts, int32_t E, int32_t max_m,
                                         int32_t N, int32_t K, int32_t expected_m, uint16_t* D, int32_t flags,
                                         int32_t* err, void* stream) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(max_m > 0 && static_cast<int64_t>(E) * max_m < (1ll << 31));
  MOE_CHECK_ARG(A && sfA && B && sfB && counts && D);
  MOE_CHECK_ARG(aligned16(A) && aligned16(B) && aligned16(D) && aligned16(sfA) && aligned16(sfB));
  MOE_CHECK_ARG(static_cast<int64_t>(E) * N < (1ll << 31));
  if (int st = check_device()) return st;
  BsArgs a{};
  a.sfA = sfA;
  a.sf_G = max_m;
  a.sf_NC = (max_m + BM - 1) / BM;
  a.KG = kgroups(K);
  a.sfB = sfB;
  a.counts = counts;
  a.D = D;
  a.ldd = N;
  a.E = E;
  a.N = N;
  a.K = K;
  a.max_m = max_m;
  a.layout = MOE_LAYOUT_MASKED;
  a.err = err;
  a.flags = flags;
  // the masked GEMM's kernel choice (moe_gemm_fp8_masked_variant): weights-as-M
  // for a few rows per expert, with token tiles of up to 128 here
  const int variant = moe_gemm_fp8_masked_variant(max_m, expected_m, flags);
  if (variant < 0) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (variant == 64) return launch_ue8m0_weights_m<64>(A, B, a, st);
  if (variant == 128 || variant == 256) return launch_ue8m0_weights_m<128>(A, B, a, st);
  const int64_t tiles = static_cast<int64_t>(E) * ((max_m + BM - 1) / BM) * ((N + BN - 1) / BN);
  return launch_ue8m0(A, static_cast<int64_t>(E) * max_m, K, B, tiles, a, st);
}
