// Grouped FP8 GEMM with 1x128 / 128x128 fp32 block scales on sm_103a tensor
// cores (tcgen05 "UMMA", accumulators in tensor memory).
//
// The pages this library follows describe a Blackwell FP8 GEMM built on UMMA
// whose API quantises and packs the input scales ("Deploying DeepSeek on GB200
// NVL72 with PD and Large Scale EP (Part I)", section "Implementation
// details", DeepGEMM bullet), with one grouped variant for prefill and one for
// decode ("Deploying DeepSeek with PD Disaggregation and Large-Scale Expert
// Parallelism on 96 H100 GPUs", section "DeepGEMM integration").  The kernel
// below is this library's own design for GB300:
//
//  * persistent: one CTA per SM walks a linear tile list built on the device
//    from the per-expert row extents (masked counts or contiguous offsets), so
//    no host synchronisation is needed and skewed experts share the SMs evenly;
//  * warp-specialised, 12 warps: warp 0 = TMA producer (4-stage ring of
//    128x128 A and 256x128 B byte tiles, 128-byte swizzle), warp 1 = a single
//    thread issuing tcgen05.mma (M=128, N=256, K=32 x4 per 128-deep block),
//    warps 4..11 = epilogue (warps 2-3 only complete warpgroup 0, which hands
//    its registers to the epilogue warpgroups with setmaxnreg);
//  * scale promotion: the fp32 scales differ per row (sA) and per 128x128
//    weight block (sB), so each 128-deep block is accumulated alone into one of
//    two TMEM buffers (2 x 256 columns), and the epilogue warps read it with
//    tcgen05.ld, multiply by sA[row, kb] * sB[nb, kb] and accumulate in fp32
//    registers while the tensor cores fill the other buffer;
//  * output: bf16 tiles go through per-warp shared-memory staging, as TMA
//    tensor stores (32 x 32 boxes) where a warp's 32 rows are all valid,
//    otherwise as 64-byte row segments from 8 lanes per row;
//  * every wait is bounded (see common.cuh): a stalled pipeline flags
//    MOE_DEV_TIMEOUT and the CTA unwinds, frees its TMEM and returns.
#include <cstring>

#include "gemm_common.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kScaleAhead = 4;                       // scale prefetch distance (k-blocks)
constexpr uint32_t kATileBytes = BM * BK;
constexpr uint32_t kBTileBytes = BN * BK;
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;

struct GemmArgs {
  const float* sA;
  int64_t sA_G;  // scale group size: masked max_m, contiguous sA_ld
  const float* sB;
  const int32_t* counts;     // masked
  const int32_t* offsets;    // contiguous
  const int32_t* m_indices;  // contiguous
  int64_t M_capacity;        // contiguous: rows of A / D / m_indices
  uint16_t* D;
  int64_t ldd;
  int32_t E, N, K, max_m, layout;
  int32_t* err;
  uint64_t wait_limit_ns;
  int32_t flags;
  // fused SwiGLU + 1x128 requantisation (tokens-as-M kernel, kSwiGLU mode)
  uint8_t* Q2;       // [rows, N/2] FP8
  float* S2;         // grouped scales, group size S2_G
  int64_t S2_G;
  // one routing slot per token (plain mode): write out[token] = bf16(w * bf16(D))
  // instead of D, the combine's arithmetic for a single slot
  const int32_t* row_src;
  const float* topk_w;
  uint16_t* out;
  int64_t ldo;
  // plain mode: bf16 D goes out through TMA stores (tmD) for warps whose 32
  // rows are all valid
  int32_t tma_store;
  int32_t ostage_slots;   // 2 KB output staging slots per epilogue warp (1 or 2)
};

// kSwiGLU: the 256-wide B tile is 128 gate rows + the matching 128 up rows
// (two 128-row TMA boxes), and the epilogue turns the tile into h = silu(g)*u
// quantised 1x128 (bytes equal GEMM1 -> bf16 -> moe_swiglu_quant), writing
// FP8 + scales instead of bf16 D.
template <bool kSwiGLU>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_tokens_m_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmD,   // bf16 D, when p.tma_store
                             const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* a_tiles = smem;
  uint8_t* b_tiles = smem + kStages * kATileBytes;
  // output staging, 1 KB aligned (the TMA store's 64-byte swizzle pattern):
  // kEpiWarps x ostage_slots x kOutStageBytes; SwiGLU mode (no bf16 output)
  // keeps its per-row amax exchange there instead, [tile parity][g][row]
  uint8_t* ostage = smem + kStages * kStageBytes;
  float* xch = reinterpret_cast<float*>(ostage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ostage + kEpiWarps * p.ostage_slots * kOutStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 8);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int32_t* sched_mem = reinterpret_cast<int32_t*>(tmem_slot + 4);
  const Sched sched{sched_mem, sched_mem + p.E + 1, sched_mem + 2 * p.E + 1};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t tfull0 = empty0 + 8 * kStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t xfull0 = tempty0 + 16;   // amax written (per tile parity)
  const uint32_t xempty0 = xfull0 + 16;   // amax read
  const int n_tiles = (p.N + BN - 1) / BN;
  const int I2 = p.N / 2;                 // SwiGLU mode: intermediate size
  const int KB = p.K / BK;
  const int NB = p.N / 128;
  volatile int* abort = abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, kEpiWarps);
      mbar_init(xfull0 + 8 * b, kEpiWarps);
      mbar_init(xempty0 + 8 * b, kEpiWarps);
    }
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
  // The local set-up above overlaps the previous kernel.  The schedule reads
  // the counts / offsets: after waiting for that kernel, or before it when the
  // caller says they were complete earlier (MOE_GEMM_EARLY_WEIGHTS), and then
  // the producer also issues its first stages' weight tiles before waiting.
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
  if (warp < kEpiWarp0) {
    regs_release_low();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL)) {
      uint32_t it = 0;
      TileCursor cur;
      bool ok = true;
      // plain: 256 consecutive weight rows; SwiGLU: gate rows then the up rows
      // of the same 128 intermediate columns
      auto load_b = [&](uint32_t s, int kb, int b_row) {
        tma_load_2d(smem_u32(b_tiles + s * kBTileBytes), &tmB, full0 + 8 * s, kb * BK, b_row);
        if (kSwiGLU)
          tma_load_2d(smem_u32(b_tiles + s * kBTileBytes + 128 * BK), &tmB, full0 + 8 * s, kb * BK, b_row + I2);
      };
      auto b_row_of = [&](int e, int l) {
        return kSwiGLU ? e * p.N + (l % n_tiles) * 128 : e * p.N + (l % n_tiles) * BN;
      };
      // early: the weight tiles of the first kStages k-blocks (stages still
      // empty), each stage expecting its A tile too, then the wait
      uint32_t pre = 0;
      if (early_producer) {
        TileCursor c0;
        for (int t = blockIdx.x; t < total && pre < static_cast<uint32_t>(kStages); t += gridDim.x) {
          c0.seek(sched, t);
          const int b_row = b_row_of(c0.e, t - sched.tile0[c0.e]);
          for (int kb = 0; kb < KB && pre < static_cast<uint32_t>(kStages); ++kb, ++pre) {
            mbar_arrive_expect_tx(full0 + 8 * pre, kStageBytes);
            load_b(pre, kb, b_row);
          }
        }
        grid_dependency_wait();
        grid_launch_dependents();
      }
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        cur.seek(sched, t);
        const int l = t - sched.tile0[cur.e];
        const int a_row = sched.rbase[cur.e] + (l / n_tiles) * BM;
        const int b_row = b_row_of(cur.e, l);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1;
          if (it < pre) {   // weights already on their way
            tma_load_2d(smem_u32(a_tiles + s * kATileBytes), &tmA, full0 + 8 * s, kb * BK, a_row);
            continue;
          }
          if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full0 + 8 * s, kStageBytes);
          tma_load_2d(smem_u32(a_tiles + s * kATileBytes), &tmA, full0 + 8 * s, kb * BK, a_row);
          load_b(s, kb, b_row);
        }
      }
      if (!ok) {
        // drain: let the copies already issued land before the CTA exits
        const uint32_t first = it > kStages ? it - kStages : 0;
        for (uint32_t j = first; j < it; ++j) {
          int dummy = 0;
          mbar_wait_bounded(full0 + 8 * (j % kStages), (j / kStages) & 1, &dummy, nullptr,
                            p.wait_limit_ns / 10);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc = 0;
      TileCursor cur;
      bool ok = true;
      const uint32_t id_full = idesc_e4m3_f32(BM, BN);
      const uint32_t id_half = idesc_e4m3_f32(BM, BN / 2);
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        cur.seek(sched, t);
        const int nt = (t - sched.tile0[cur.e]) % n_tiles;
        const bool half = (nt == n_tiles - 1) && (p.N % BN) != 0;
        const uint32_t idesc = half ? id_half : id_full;
        for (int kb = 0; kb < KB; ++kb, ++it, ++acc) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1;
          const uint32_t b = acc & 1, tph = (acc >> 1) & 1;
          if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, abort, p.err, p.wait_limit_ns) ||
              !mbar_wait_bounded(full0 + 8 * s, ph, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(a_tiles + s * kATileBytes));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(b_tiles + s * kBTileBytes));
          const uint32_t d_tmem = tmem_base + b * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // 32 bytes of K per MMA: +2 in the 16-byte address field
            umma_e4m3(d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
          umma_commit(empty0 + 8 * s);
          umma_commit(tfull0 + 8 * b);
        }
      }
      if (!ok && acc > 0) {  // wait for the MMAs in flight before TMEM is freed
        int dummy = 0;
        mbar_wait_bounded(tfull0 + 8 * ((acc - 1) & 1), ((acc - 1) >> 1) & 1, &dummy, nullptr,
                          p.wait_limit_ns / 10);
      }
    }
  }
  } else {
    regs_acquire_high();
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int g = (warp - kEpiWarp0) >> 2;  // plain: column half; SwiGLU: intermediate half
    uint32_t acc_it = 0;
    uint32_t tile_no = 0;
    TileCursor cur;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++tile_no) {
      cur.seek(sched, t);
      const int e = cur.e;
      const int l = t - sched.tile0[e];
      const int mt = l / n_tiles, nt = l % n_tiles;
      const bool half = !kSwiGLU && (nt == n_tiles - 1) && (p.N % BN) != 0;
      const bool active = !(half && g == 1);
      const int r_local = mt * BM + q * 32 + lane;
      const int64_t gr = static_cast<int64_t>(sched.rbase[e]) + r_local;
      bool row_ok = r_local < sched.rext[e];
      if (row_ok && p.layout == MOE_LAYOUT_CONTIG) row_ok = __ldg(p.m_indices + gr) >= 0;
      // single-slot combine: the row's token and weight, read now so the
      // loads are long done when the tile is stored
      int64_t tok = 0;
      float wtok = 0.f;
      if (!kSwiGLU && p.out != nullptr && row_ok) {
        tok = __ldg(p.row_src + gr);
        wtok = __ldg(p.topk_w + tok);
      }
      const int n0 = nt * BN + g * 128;
      const int64_t grp = gr / p.sA_G, pos = gr - grp * p.sA_G;
      const float* sa_ptr = p.sA + grp * KB * p.sA_G + pos;
      // plain: the weight block of this warp's 128 columns; SwiGLU: the gate
      // block (sb_ptr) and the up block (sb2_ptr) of the tile's 128 columns
      const float* sb_ptr = kSwiGLU ? p.sB + (static_cast<int64_t>(e) * NB + nt) * KB
                                    : p.sB + (static_cast<int64_t>(e) * NB + (active ? n0 / 128 : 0)) * KB;
      const float* sb2_ptr = p.sB + (static_cast<int64_t>(e) * NB + (kSwiGLU ? I2 / 128 + nt : 0)) * KB;
      // fp32 accumulators as pairs: the promotion runs as packed FMAs
      // (two round-to-nearest fp32 FMAs per instruction, same bits as fmaf).
      // SwiGLU mode: acc[0..31] gate columns, acc[32..63] up columns.
      float2 acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.f, 0.f);
      // The scales run kScaleAhead k-blocks ahead of their use in a register
      // ring: a global load has several k-blocks of work to hide behind, not
      // one.  The k-block loop is unrolled by the ring depth, so entry m is
      // loaded once and read kScaleAhead k-blocks later with no register
      // moves in between (a rotating ring's moves would each wait for the
      // load just issued, leaving one k-block of cover).
      auto load_sa = [&](int k) { return (row_ok && k < KB) ? __ldg(sa_ptr + static_cast<int64_t>(k) * p.sA_G) : 0.f; };
      auto load_sb = [&](int k) { return k < KB ? __ldg(sb_ptr + k) : 0.f; };
      auto load_sb2 = [&](int k) { return (kSwiGLU && k < KB) ? __ldg(sb2_ptr + k) : 0.f; };
      static_assert(kScaleAhead == 4, "ring below assumes 4");
      float ra[kScaleAhead], rb[kScaleAhead], ru[kScaleAhead];
#pragma unroll
      for (int m = 0; m < kScaleAhead; ++m) {
        ra[m] = load_sa(m);
        rb[m] = load_sb(m);
        ru[m] = load_sb2(m);
      }
#pragma unroll 1
      for (int kb0 = 0; ok && kb0 < KB; kb0 += kScaleAhead) {
#pragma unroll
      for (int m = 0; m < kScaleAhead; ++m) {
        const int kb = kb0 + m;
        if (kb >= KB) break;
        const uint32_t b = acc_it & 1, tph = (acc_it >> 1) & 1;
        ++acc_it;
        const float sc = ra[m] * rb[m];
        const float scu = ra[m] * ru[m];
        ra[m] = load_sa(kb + kScaleAhead);
        rb[m] = load_sb(kb + kScaleAhead);
        if (kSwiGLU) ru[m] = load_sb2(kb + kScaleAhead);
        // one lane waits, the warp follows it: tcgen05.ld is warp-collective
        int got = 1;
        if (lane == 0) got = mbar_wait_bounded(tfull0 + 8 * b, tph, abort, p.err, p.wait_limit_ns);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (active) {
          const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
          const float2 sc2 = make_float2(sc, sc);
          if (kSwiGLU) {
            const float2 scu2 = make_float2(scu, scu);
            const uint32_t tg = tmem_base + lanes + b * BN + g * 64;        // gate columns
            const uint32_t tu = tmem_base + lanes + b * BN + 128 + g * 64;  // up columns
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t r0[16], r1[16];
              tmem_ld_32x32b_x16(tg + c * 16, r0);
              tmem_ld_32x32b_x16(tu + c * 16, r1);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc[c * 8 + i] = __ffma2_rn(sc2, make_float2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1])),
                                            acc[c * 8 + i]);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc[32 + c * 8 + i] = __ffma2_rn(
                    scu2, make_float2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1])), acc[32 + c * 8 + i]);
            }
          } else {
            const uint32_t tbase = tmem_base + lanes + b * BN + g * 128;
#pragma unroll
            for (int c = 0; c < 8; c += 2) {   // two 16-column loads in flight
              uint32_t r0[16], r1[16];
              tmem_ld_32x32b_x16(tbase + c * 16, r0);
              tmem_ld_32x32b_x16(tbase + (c + 1) * 16, r1);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc[c * 8 + i] = __ffma2_rn(sc2, make_float2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1])),
                                            acc[c * 8 + i]);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc[(c + 1) * 8 + i] = __ffma2_rn(
                    sc2, make_float2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1])), acc[(c + 1) * 8 + i]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * b);
      }
      }
      if (!ok) break;
      if (!kSwiGLU) {
        // bf16 results (with the single-slot combine: bf16(fmaf(w, bf16(y), 0)),
        // the combine's arithmetic, written to the token's output row).  The
        // warp's 32 rows x 128 columns go out through its 2 KB of shared
        // staging in four 32-column quarters, so each store instruction writes
        // 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes.
        if (active) {
          const bool to_out = p.out != nullptr;
          uint16_t* row_base = to_out ? p.out + tok * p.ldo + n0 : p.D + gr * p.ldd + n0;
          const float w = wtok;
          auto rb = [](float v) { return __bfloat162float(__float2bfloat16_rn(v)); };
          const int slots = p.ostage_slots;
          const uint32_t stg0 = smem_u32(ostage + (warp - kEpiWarp0) * slots * kOutStageBytes);
          // D rows all valid for this warp: each quarter leaves as one TMA
          // store of a 32 x 32 box (the staging layout is the map's 64-byte
          // swizzle), issued by lane 0; otherwise 8 lanes per row store it
          const bool by_tma = p.tma_store && !to_out && __all_sync(0xffffffffu, row_ok);
          const int32_t d_row0 = static_cast<int32_t>(gr - lane);
#pragma unroll
          for (int qc = 0; qc < 4; ++qc) {
            // the staging slot is free once the TMA store from it has read it:
            // with two slots, all but the latest store
            const uint32_t stg = stg0 + (slots == 2 ? (qc & 1) : 0) * kOutStageBytes;
            if (lane == 0 && p.tma_store) {
              if (slots == 2)
                bulk_wait_read_le1();
              else
                bulk_wait_read_all();
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int v = qc * 4 + c;       // 16-byte chunk of the row: columns 8v .. 8v+7
              uint32_t o[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float2 a2 = acc[v * 4 + h];
                const __nv_bfloat162 bb = to_out ? __floats2bfloat162_rn(fmaf(w, rb(a2.x), 0.f), fmaf(w, rb(a2.y), 0.f))
                                                 : __floats2bfloat162_rn(a2.x, a2.y);
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
              uint16_t* base_r = reinterpret_cast<uint16_t*>(
                  __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(row_base), r));
              if (ok_r) *reinterpret_cast<uint4*>(base_r + qc * 32 + c * 8) = val;
            }
            __syncwarp();
          }
        }
      } else {
        // h = silu(g) * u from the bf16-rounded GEMM1 values (what the bf16 Y1
        // would hold), same formula as moe_swiglu_quant; h overwrites acc[0..31].
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float g0 = __bfloat162float(__float2bfloat16_rn(acc[i].x));
          const float g1 = __bfloat162float(__float2bfloat16_rn(acc[i].y));
          const float u0 = __bfloat162float(__float2bfloat16_rn(acc[32 + i].x));
          const float u1 = __bfloat162float(__float2bfloat16_rn(acc[32 + i].y));
          acc[i].x = __fdiv_rn(g0, 1.0f + expf(-g0)) * u0;
          acc[i].y = __fdiv_rn(g1, 1.0f + expf(-g1)) * u1;
          amax = fmaxf(amax, fmaxf(fabsf(acc[i].x), fabsf(acc[i].y)));
        }
        // the 1x128 block spans both warpgroups: swap the half-row amax with the
        // partner warp (same rows, other 64 columns) through shared memory,
        // ordered by a written/read mbarrier pair per tile parity (bounded waits)
        const uint32_t par = tile_no & 1, xph = (tile_no >> 1) & 1;
        int okx = 1;
        if (lane == 0) okx = mbar_wait_bounded(xempty0 + 8 * par, xph ^ 1, abort, p.err, p.wait_limit_ns);
        okx = __shfl_sync(0xffffffffu, okx, 0);
        if (!okx) {
          ok = false;
          break;
        }
        float* x = xch + par * 256;
        x[g * 128 + q * 32 + lane] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(xfull0 + 8 * par);
        if (lane == 0) okx = mbar_wait_bounded(xfull0 + 8 * par, xph, abort, p.err, p.wait_limit_ns);
        okx = __shfl_sync(0xffffffffu, okx, 0);
        if (!okx) {
          ok = false;
          break;
        }
        amax = fmaxf(amax, x[(1 - g) * 128 + q * 32 + lane]);
        __syncwarp();
        if (lane == 0) mbar_arrive(xempty0 + 8 * par);
        if (row_ok) {
          const float sc = block_scale(amax);
          uint2 qv[8];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float f[8] = {acc[4 * v].x, acc[4 * v].y, acc[4 * v + 1].x, acc[4 * v + 1].y,
                                acc[4 * v + 2].x, acc[4 * v + 2].y, acc[4 * v + 3].x, acc[4 * v + 3].y};
            qv[v] = quant8(f, sc);
          }
          uint4* dq = reinterpret_cast<uint4*>(p.Q2 + gr * I2 + nt * 128 + g * 64);
#pragma unroll
          for (int v = 0; v < 4; ++v) dq[v] = make_uint4(qv[2 * v].x, qv[2 * v].y, qv[2 * v + 1].x, qv[2 * v + 1].y);
          if (g == 0) {
            const int64_t grp2 = gr / p.S2_G, pos2 = gr - grp2 * p.S2_G;
            p.S2[(grp2 * (I2 / 128) + nt) * p.S2_G + pos2] = sc;
          }
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

size_t tokens_m_smem_bytes(int E, int slots) {
  return 1024 + static_cast<size_t>(kStages) * kStageBytes + (2 * kStages + 8) * 8 + 16 +
         sizeof(int32_t) * (3 * E + 1) + kEpiWarps * slots * kOutStageBytes;
}
// two output staging slots per warp (a quarter is written while the previous
// one's TMA store reads the other) where shared memory allows, else one
int tokens_m_slots(int E) { return tokens_m_smem_bytes(E, 2) <= kMaxSmemPerBlock ? 2 : 1; }

int launch_tokens_m(const uint8_t* A, int64_t a_rows, int64_t lda, const uint8_t* B,
                    int64_t tiles_upper, GemmArgs& args, cudaStream_t stream, bool swiglu = false) {
  CUtensorMap tmA, tmB, tmD;
  if (int st = make_tmap_u8_sw128(&tmA, A, a_rows, args.K, lda, BM)) return st;
  if (int st = make_tmap_u8_sw128(&tmB, B, static_cast<uint64_t>(args.E) * args.N, args.K, args.K,
                                  swiglu ? 128 : BN))
    return st;
  // plain bf16 D (a_rows rows of ldd) leaves through TMA stores when it can
  // be mapped; otherwise, and for the fused modes, through the LSU path
  std::memset(&tmD, 0, sizeof(tmD));
  args.tma_store = 0;
  if (!swiglu && args.out == nullptr && args.D != nullptr &&
      make_tmap_b16_out(&tmD, args.D, static_cast<uint64_t>(a_rows), args.N, static_cast<uint64_t>(args.ldd) * 2) ==
          MOE_OK)
    args.tma_store = 1;
  args.ostage_slots = tokens_m_slots(args.E);
  const size_t smem = tokens_m_smem_bytes(args.E, args.ostage_slots);
  if (args.wait_limit_ns == 0) args.wait_limit_ns = kWaitLimitNs;
  int64_t grid = num_sms();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) grid = 1;
  if (swiglu) {
    if (int st = prepare_kernel(gemm_fp8_tokens_m_kernel<true>, smem, true)) return st;
    return launch_pdl(gemm_fp8_tokens_m_kernel<true>, static_cast<unsigned>(grid), kThreads, smem, stream, tmA,
                      tmB, tmD, args);
  } else {
    if (int st = prepare_kernel(gemm_fp8_tokens_m_kernel<false>, smem, true)) return st;
    return launch_pdl(gemm_fp8_tokens_m_kernel<false>, static_cast<unsigned>(grid), kThreads, smem, stream, tmA,
                      tmB, tmD, args);
  }
}

// =============================================================================
// Tokens-as-M over a CTA pair (2-CTA cluster, UMMA M = 256).
//
// What bounds the single-CTA kernel is each SM's tile feed: 48 KB of A and B
// per 128-deep block for a 128x256 tile.  Here the two CTAs of a cluster
// compute a 256x256 tile with one M = 256 UMMA issued by the even CTA: each
// CTA stages its own 128 token rows of A and half (128 rows) of the 256 weight
// rows of B, 32 KB per block, and the tensor cores read the peer's half across
// the pair.  Each CTA's TMEM holds its 128 rows of D, drained and promoted by
// its own epilogue exactly as in the single-CTA kernel.
//
// Signalling (all waits bounded): each CTA's producer fills its own stage and
// its full barrier; in the odd CTA warp 1 relays that to the even CTA's pfull
// barrier; the even CTA's MMA thread waits full + pfull + tempty, issues, and
// its commits arrive on empty and tfull in both CTAs; every epilogue warp of
// both CTAs arrives on the even CTA's tempty.
// =============================================================================
constexpr int BM2 = 256;                              // rows per pair tile
constexpr int kPairStages = 6;
constexpr uint32_t kPairATile = 128 * BK;             // this CTA's 128 rows of A
constexpr uint32_t kPairBTile = 128 * BK;             // this CTA's half of B
constexpr uint32_t kPairStage = kPairATile + kPairBTile;
constexpr int kPairBars = 3 * kPairStages + 4;        // full, empty, pfull [S]; tfull, tempty [2]

__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_tokens_m_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                  const __grid_constant__ CUtensorMap tmB, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* a_tiles = smem;
  uint8_t* b_tiles = smem + kPairStages * kPairATile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStage);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPairBars);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int32_t* sched_mem = reinterpret_cast<int32_t*>(tmem_slot + 4);
  const Sched sched{sched_mem, sched_mem + p.E + 1, sched_mem + 2 * p.E + 1};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kPairStages;
  const uint32_t pfull0 = empty0 + 8 * kPairStages;
  const uint32_t tfull0 = pfull0 + 8 * kPairStages;
  const uint32_t tempty0 = tfull0 + 16;
  const int n_tiles = p.N / BN;
  const int KB = p.K / BK;
  const int NB = p.N / 128;
  volatile int* abort = abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
      mbar_init(pfull0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 2 * kEpiWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (warp == 0) build_schedule<BM2>(p, sched, n_tiles);
  // both CTAs' barriers are initialised before any arrival crosses the pair
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = sched.tile0[p.E];
  const int t_first = static_cast<int>(cluster_id_x());
  const int t_step = static_cast<int>(cluster_count_x());
  if (warp < kEpiWarp0) {
    regs_release_low();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL)) {
      uint32_t it = 0;
      TileCursor cur;
      bool ok = true;
      for (int t = t_first; ok && t < total; t += t_step) {
        cur.seek(sched, t);
        const int l = t - sched.tile0[cur.e];
        const int a_row = sched.rbase[cur.e] + (l / n_tiles) * BM2 + static_cast<int>(rank) * 128;
        const int b_row = cur.e * p.N + (l % n_tiles) * BN + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % kPairStages, ph = (it / kPairStages) & 1;
          if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full0 + 8 * s, kPairStage);
          tma_load_2d(smem_u32(a_tiles + s * kPairATile), &tmA, full0 + 8 * s, kb * BK, a_row);
          tma_load_2d(smem_u32(b_tiles + s * kPairBTile), &tmB, full0 + 8 * s, kb * BK, b_row);
        }
      }
      if (!ok) {
        // drain: let the copies already issued land before the CTA exits
        const uint32_t first = it > kPairStages ? it - kPairStages : 0;
        for (uint32_t j = first; j < it; ++j) {
          int dummy = 0;
          mbar_wait_bounded(full0 + 8 * (j % kPairStages), (j / kPairStages) & 1, &dummy, nullptr,
                            p.wait_limit_ns / 10);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    if (even) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      uint32_t it = 0, acc = 0;
      bool ok = true;
      const uint32_t idesc = idesc_e4m3_f32(BM2, BN);
      for (int t = t_first; ok && t < total; t += t_step) {
        for (int kb = 0; kb < KB; ++kb, ++it, ++acc) {
          const uint32_t s = it % kPairStages, ph = (it / kPairStages) & 1;
          const uint32_t b = acc & 1, tph = (acc >> 1) & 1;
          if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, abort, p.err, p.wait_limit_ns) ||
              !mbar_wait_bounded(full0 + 8 * s, ph, abort, p.err, p.wait_limit_ns) ||
              !mbar_wait_bounded(pfull0 + 8 * s, ph, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(a_tiles + s * kPairATile));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(b_tiles + s * kPairBTile));
          const uint32_t d_tmem = tmem_base + b * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // 32 bytes of K per MMA: +2 in the 16-byte address field
            umma_e4m3_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
          umma_commit_pair(empty0 + 8 * s, 0x3);
          umma_commit_pair(tfull0 + 8 * b, 0x3);
        }
      }
      if (acc > 0) {  // the last MMAs (and their commits to both CTAs) are done before teardown
        int dummy = 0;
        mbar_wait_bounded(tfull0 + 8 * ((acc - 1) & 1), ((acc - 1) >> 1) & 1, &dummy, nullptr,
                          ok ? p.wait_limit_ns : p.wait_limit_ns / 10);
      }
    } else {
      // ---------------------------------------------------------- stage relay (odd CTA)
      uint32_t it = 0;
      bool ok = true;
      const uint32_t pfull_even = cluster_map_shared(pfull0, 0);
      for (int t = t_first; ok && t < total; t += t_step) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const uint32_t s = it % kPairStages, ph = (it / kPairStages) & 1;
          if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(pfull_even + 8 * s);
        }
      }
    }
  }
  } else {
    regs_acquire_high();
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int g = (warp - kEpiWarp0) >> 2;
    const uint32_t tempty_even = cluster_map_shared(tempty0, 0);
    uint32_t acc_it = 0;
    TileCursor cur;
    bool ok = true;
    for (int t = t_first; ok && t < total; t += t_step) {
      cur.seek(sched, t);
      const int e = cur.e;
      const int l = t - sched.tile0[e];
      const int mt = l / n_tiles, nt = l % n_tiles;
      const int r_local = mt * BM2 + static_cast<int>(rank) * 128 + q * 32 + lane;
      const int64_t gr = static_cast<int64_t>(sched.rbase[e]) + r_local;
      bool row_ok = r_local < sched.rext[e];
      if (row_ok && p.layout == MOE_LAYOUT_CONTIG) row_ok = __ldg(p.m_indices + gr) >= 0;
      const int n0 = nt * BN + g * 128;
      const int64_t grp = gr / p.sA_G, pos = gr - grp * p.sA_G;
      const float* sa_ptr = p.sA + grp * KB * p.sA_G + pos;
      const float* sb_ptr = p.sB + (static_cast<int64_t>(e) * NB + n0 / 128) * KB;
      float2 acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.f, 0.f);
      // scales four k-blocks ahead; the loop is unrolled by that depth so each
      // ring register is loaded once and read four k-blocks later
      auto load_sa = [&](int k) { return (row_ok && k < KB) ? __ldg(sa_ptr + static_cast<int64_t>(k) * p.sA_G) : 0.f; };
      auto load_sb = [&](int k) { return k < KB ? __ldg(sb_ptr + k) : 0.f; };
      float ra[kScaleAhead], rb[kScaleAhead];
#pragma unroll
      for (int j = 0; j < kScaleAhead; ++j) {
        ra[j] = load_sa(j);
        rb[j] = load_sb(j);
      }
#pragma unroll 1
      for (int kb0 = 0; ok && kb0 < KB; kb0 += kScaleAhead) {
#pragma unroll
        for (int j = 0; j < kScaleAhead; ++j) {
          const int kb = kb0 + j;
          if (kb >= KB) break;
          const uint32_t b = acc_it & 1, tph = (acc_it >> 1) & 1;
          ++acc_it;
          const float sc = ra[j] * rb[j];
          ra[j] = load_sa(kb + kScaleAhead);
          rb[j] = load_sb(kb + kScaleAhead);
          int got = 1;
          if (lane == 0) got = mbar_wait_bounded(tfull0 + 8 * b, tph, abort, p.err, p.wait_limit_ns);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float2 sc2 = make_float2(sc, sc);
          const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * BN + g * 128;
#pragma unroll
          for (int c = 0; c < 8; c += 2) {   // two 16-column loads in flight
            uint32_t r0[16], r1[16];
            tmem_ld_32x32b_x16(tbase + c * 16, r0);
            tmem_ld_32x32b_x16(tbase + (c + 1) * 16, r1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              acc[c * 8 + i] = __ffma2_rn(sc2, make_float2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1])),
                                          acc[c * 8 + i]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              acc[(c + 1) * 8 + i] = __ffma2_rn(
                  sc2, make_float2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1])), acc[(c + 1) * 8 + i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_even + 8 * b);
        }
      }
      if (!ok) break;
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.D + gr * p.ldd + n0);
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          uint32_t o[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const __nv_bfloat162 bb = __floats2bfloat162_rn(acc[v * 4 + h].x, acc[v * 4 + h].y);
            o[h] = *reinterpret_cast<const uint32_t*>(&bb);
          }
          dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }

  // no CTA leaves while its peer may still read its shared memory or arrive
  // on its barriers
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

size_t pair_smem_bytes(int E) {
  return 1024 + static_cast<size_t>(kPairStages) * kPairStage + kPairBars * 8 + 16 +
         sizeof(int32_t) * (3 * E + 1);
}

// Launch the pair kernel: grid = 2 x the clusters that fit at once (at most
// one per pair tile), two CTAs per cluster.
int launch_tokens_m_pair(const uint8_t* A, int64_t a_rows, int64_t lda, const uint8_t* B,
                         int64_t pair_tiles_upper, GemmArgs& args, cudaStream_t stream) {
  CUtensorMap tmA, tmB;
  if (int st = make_tmap_u8_sw128(&tmA, A, a_rows, args.K, lda, 128)) return st;
  if (int st = make_tmap_u8_sw128(&tmB, B, static_cast<uint64_t>(args.E) * args.N, args.K, args.K, 128))
    return st;
  const size_t smem = pair_smem_bytes(args.E);
  if (args.wait_limit_ns == 0) args.wait_limit_ns = kWaitLimitNs;
  if (int st = prepare_kernel(gemm_fp8_tokens_m_pair_kernel, smem, true)) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static int max_clusters_cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (max_clusters_cached[dev] == 0) {
    int n = 0;
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    if (cudaOccupancyMaxActiveClusters(&n, gemm_fp8_tokens_m_pair_kernel, &cfg) != cudaSuccess || n < 1)
      return MOE_ERR_UNSUPPORTED;
    max_clusters_cached[dev] = n;
  }
  int64_t clusters = max_clusters_cached[dev];
  if (pair_tiles_upper < clusters) clusters = pair_tiles_upper;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  return cudaLaunchKernelEx(&cfg, gemm_fp8_tokens_m_pair_kernel, tmA, tmB, args) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// =============================================================================
// Weights-as-M variant for the masked (decode) layout.
//
// Decode sends few tokens to each expert, so a 128-row token tile would be
// mostly empty while the expert's weights stream from HBM.  Here the roles
// swap: 128 weight rows (one 128x128 scale block row) are the UMMA M side and
// the expert's tokens are the N side, sized per tile at run time in steps of
// 16 (UMMA N from 16 to BNT).  D^T sits in TMEM as [weight row (lane), token
// (column)]; the epilogue scales column c by sB[nb, kb] * sA[token c, kb].
// Stages are small (16 KB of weights + the token rows), so the ring is deep
// (4..8 stages) to keep enough bytes in flight per SM, and TMEM holds 2..8
// accumulation buffers.  A tile's token rows come in as few copies as
// possible: four tensor maps with boxes of 128, 64, 32 and 16 rows, the
// tile's rows split into 128-row boxes and at most one of each smaller box.
// =============================================================================
template <int BNT>
struct WeightsM {
  static constexpr uint32_t kWBytes = 128 * BK;                // weight tile
  static constexpr uint32_t kTBytes = BNT * BK;                // token tile (max)
  // per stage after the two tiles: the k-block's token scales (BNT floats,
  // one bulk copy) and the weight block's scale (one float, cp.async)
  static constexpr uint32_t kOffSa = kWBytes + kTBytes;
  static constexpr uint32_t kOffSb = kOffSa + BNT * 4;
  static constexpr uint32_t kStage = (kOffSb + 16 + 1023) / 1024 * 1024;   // stages stay 1 KB aligned
  // stages fill what shared memory is left after the barriers and the
  // largest schedule (kMaxExperts), at most 8
  static constexpr uint32_t kStageBudget = kMaxSmemPerBlock - 1024 - 16 * 8 * 2 - 16 - 4 * (3 * kMaxExperts + 1);
  static constexpr int kStages = (kStageBudget / kStage) > 8 ? 8 : (kStageBudget / kStage);
  static constexpr int kBufs = (512 / BNT) > 8 ? 8 : (512 / BNT);
  static constexpr int kHalf = BNT / 2;                        // columns per epilogue warpgroup
  static constexpr bool kSplitRegs = BNT > 128;                // 128 accumulators/thread need the split
  static constexpr int kPair = 2;                              // TMEM loads in flight
  static constexpr size_t smem_bytes(int E) {
    return 1024 + static_cast<size_t>(kStages) * kStage + (2 * kStages + 2 * kBufs) * 8 + 16 +
           sizeof(int32_t) * (3 * E + 1);
  }
};

// Warp 0: per expert kept rows, token tiles of BNT, tiles = token tiles x N/128.
template <int BNT>
__device__ void build_schedule_wm(const GemmArgs& p, const Sched& s, int nblk) {
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
    gemm_fp8_weights_m_kernel(const __grid_constant__ TokenMaps tmT,     // tokens  [E*max_m, K]
                              const __grid_constant__ CUtensorMap tmW,   // weights [E*N, K]
                              const GemmArgs p) {
  using C = WeightsM<BNT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 2 * C::kBufs);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int32_t* sched_mem = reinterpret_cast<int32_t*>(tmem_slot + 4);
  const Sched sched{sched_mem, sched_mem + p.E + 1, sched_mem + 2 * p.E + 1};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t tfull0 = empty0 + 8 * C::kStages;
  const uint32_t tempty0 = tfull0 + 8 * C::kBufs;
  const int nblk = p.N / 128;
  const int KB = p.K / BK;
  volatile int* abort = abort_flag;

  if (threadIdx.x == 0) {
    // a stage is full once its copies landed (the producer's expect-tx arrival
    // and its cp.async arrival) and empty once the MMAs that read it are done
    // and every epilogue warp has read its scales
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 2);
      mbar_init(empty0 + 8 * s, 1 + kEpiWarps);
    }
    for (int b = 0; b < C::kBufs; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, kEpiWarps);
    }
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
  // first stages' weight tiles before waiting)
  const bool early = (p.flags & MOE_GEMM_EARLY_WEIGHTS) != 0;
  if (!early) {
    grid_dependency_wait();
    grid_launch_dependents();
  }
  if (warp == 0) build_schedule_wm<BNT>(p, sched, nblk);
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
    if constexpr (C::kSplitRegs) regs_release_low();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !(p.flags & MOE_GEMM_DEBUG_STALL)) {
      const uint64_t pol_w = l2_policy_evict_first();   // weights stream through once
      uint32_t it = 0;
      TileCursor cur;
      bool ok = true;
      struct Tile {
        int e, j, nb, ncols, t_row, w_row;
      };
      auto tile_of = [&](int t, TileCursor& c) {
        c.seek(sched, t);
        Tile tl;
        tl.e = c.e;
        const int l = t - sched.tile0[tl.e];
        tl.j = l / nblk;
        tl.nb = l % nblk;
        tl.ncols = (min(BNT, sched.rext[tl.e] - tl.j * BNT) + 15) & ~15;
        tl.t_row = sched.rbase[tl.e] + tl.j * BNT;
        tl.w_row = tl.e * p.N + tl.nb * 128;
        return tl;
      };
      // a stage's weight half: the weight tile and the weight block's scale
      // (a 4-byte cp.async that arrives on the stage's barrier), with the
      // stage's whole byte count expected
      auto issue_w = [&](uint32_t s, int kb, const Tile& tl) {
        const uint32_t st_base = smem_u32(smem + s * C::kStage);
        mbar_arrive_expect_tx(full0 + 8 * s, C::kWBytes + tl.ncols * BK + tl.ncols * 4);
        tma_load_2d_hint(st_base, &tmW, full0 + 8 * s, kb * BK, tl.w_row, pol_w);
        cp_async_4(st_base + C::kOffSb, p.sB + (static_cast<int64_t>(tl.e) * nblk + tl.nb) * KB + kb, 4u);
        cp_async_mbar_arrive(full0 + 8 * s);
      };
      // its token half: the token scales (ncols floats, 16-byte aligned since
      // max_m and the tile start are multiples of 16) and the token rows
      // [0, ncols) in boxes of 128 while they last, then at most one each of
      // 64, 32 and 16 (ncols is a multiple of 16)
      auto issue_t = [&](uint32_t s, int kb, const Tile& tl) {
        const uint32_t st_base = smem_u32(smem + s * C::kStage);
        bulk_g2s(st_base + C::kOffSa, p.sA + (static_cast<int64_t>(tl.e) * KB + kb) * p.max_m + tl.j * BNT,
                 tl.ncols * 4, full0 + 8 * s);
        for (int r = 0; r < tl.ncols;) {
          const int left = tl.ncols - r;
          const int i = left >= 128 ? 3 : left >= 64 ? 2 : left >= 32 ? 1 : 0;
          tma_load_2d(st_base + C::kWBytes + r * BK, &tmT.box[i], full0 + 8 * s, kb * BK, tl.t_row + r);
          r += 16 << i;
        }
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
      cp_async_wait_all();   // no copy may land after the CTA has gone
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc = 0;
      TileCursor cur;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        cur.seek(sched, t);
        const int e = cur.e;
        const int j = (t - sched.tile0[e]) / nblk;
        const int ntok = min(BNT, sched.rext[e] - j * BNT);
        const int ncols = (ntok + 15) & ~15;
        const uint32_t idesc = idesc_e4m3_f32(128, ncols);
        for (int kb = 0; kb < KB; ++kb, ++it, ++acc) {
          const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1;
          const uint32_t b = acc % C::kBufs, tph = (acc / C::kBufs) & 1;
          if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, abort, p.err, p.wait_limit_ns) ||
              !mbar_wait_bounded(full0 + 8 * s, ph, abort, p.err, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st_base = smem_u32(smem + s * C::kStage);
          const uint64_t wd = sdesc_kmajor_sw128(st_base);
          const uint64_t td = sdesc_kmajor_sw128(st_base + C::kWBytes);
          const uint32_t d_tmem = tmem_base + b * BNT;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            umma_e4m3(d_tmem, wd + 2 * k, td + 2 * k, idesc, k > 0 ? 1u : 0u);
          umma_commit(empty0 + 8 * s);
          umma_commit(tfull0 + 8 * b);
        }
      }
      if (!ok && acc > 0) {
        int dummy = 0;
        const uint32_t last = acc - 1;
        mbar_wait_bounded(tfull0 + 8 * (last % C::kBufs), (last / C::kBufs) & 1, &dummy, nullptr,
                          p.wait_limit_ns / 10);
      }
    }
  }
  } else {
    if constexpr (C::kSplitRegs) regs_acquire_high();
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lanes = weight rows q*32 .. q*32+31
    const int g = (warp - kEpiWarp0) >> 2;  // token columns [g*kHalf, (g+1)*kHalf)
    uint32_t acc_it = 0;
    TileCursor cur;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
      cur.seek(sched, t);
      const int e = cur.e;
      const int l = t - sched.tile0[e];
      const int j = l / nblk, nb = l % nblk;
      const int ntok = min(BNT, sched.rext[e] - j * BNT);
      const int ncols = (ntok + 15) & ~15;
      // the two warpgroups split the tile's columns evenly (in 16-column
      // chunks), so a part-filled tile does not leave one group all the work
      const int cols_g0 = ((ncols / 16 + 1) / 2) * 16;
      const int col0 = g ? cols_g0 : 0;
      const int my_cols = g ? ncols - cols_g0 : cols_g0;
      const int nchunk = my_cols / 16;
      float2 acc[C::kHalf / 2];
#pragma unroll
      for (int i = 0; i < C::kHalf / 2; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int kb = 0; ok && kb < KB; ++kb) {
        const uint32_t b = acc_it % C::kBufs, tph = (acc_it / C::kBufs) & 1;
        const uint32_t s = acc_it % C::kStages, sph = (acc_it / C::kStages) & 1;
        ++acc_it;
        int got = 1;
        if (lane == 0) got = mbar_wait_bounded(tfull0 + 8 * b, tph, abort, p.err, p.wait_limit_ns);
        got = __shfl_sync(0xffffffffu, got, 0);
        // the stage's copies landed before its MMAs were issued; waiting on its
        // (already completed) full phase orders this warp's scale reads after them
        if (got) got = mbar_wait_bounded(full0 + 8 * s, sph, abort, p.err, p.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this k-block's scales from the stage: sB * sA per token column (the
        // product the definition forms), no global load on this path
        const uint8_t* stg = smem + s * C::kStage;
        const float sbv = *reinterpret_cast<const float*>(stg + C::kOffSb);
        const float* sa_cur = reinterpret_cast<const float*>(stg + C::kOffSa) + col0;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * BNT + col0;
#pragma unroll
        for (int ch = 0; ch < C::kHalf / 16; ch += C::kPair) {
          if (ch < nchunk) {
            uint32_t r[C::kPair][16];
            tmem_ld_32x32b_x16(tbase + ch * 16, r[0]);
            if (C::kPair == 2 && ch + 1 < nchunk) tmem_ld_32x32b_x16(tbase + (ch + 1) * 16, r[C::kPair - 1]);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < C::kPair; ++h) {
              if (ch + h < nchunk) {
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                  const int c = (ch + h) * 16 + 4 * i4;
                  const float4 a4 = *reinterpret_cast<const float4*>(sa_cur + c);   // broadcast read
                  const float2 s01 = make_float2(__fmul_rn(sbv, a4.x), __fmul_rn(sbv, a4.y));
                  const float2 s23 = make_float2(__fmul_rn(sbv, a4.z), __fmul_rn(sbv, a4.w));
                  acc[c / 2] = __ffma2_rn(
                      s01, make_float2(__uint_as_float(r[h][4 * i4]), __uint_as_float(r[h][4 * i4 + 1])), acc[c / 2]);
                  acc[c / 2 + 1] = __ffma2_rn(
                      s23, make_float2(__uint_as_float(r[h][4 * i4 + 2]), __uint_as_float(r[h][4 * i4 + 3])),
                      acc[c / 2 + 1]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(tempty0 + 8 * b);   // the accumulator buffer is free
          mbar_arrive(empty0 + 8 * s);    // this warp is done with the stage's scales
        }
      }
      if (!ok) break;
      // D[e][token][n]: a warp writes 32 consecutive n of one token per store
      const int64_t n = static_cast<int64_t>(nb) * 128 + q * 32 + lane;
      uint16_t* dcol = p.D + (static_cast<int64_t>(e) * p.max_m + j * BNT + col0) * p.N + n;
      const int valid = max(0, min(my_cols, ntok - col0));
#pragma unroll
      for (int c = 0; c < C::kHalf; ++c) {
        if (c < valid) {
          const __nv_bfloat16 v = __float2bfloat16_rn((c & 1) ? acc[c / 2].y : acc[c / 2].x);
          dcol[static_cast<int64_t>(c) * p.N] = *reinterpret_cast<const uint16_t*>(&v);
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
int launch_weights_m(const uint8_t* A, const uint8_t* B, GemmArgs& args, cudaStream_t stream) {
  using C = WeightsM<BNT>;
  TokenMaps tmT;
  CUtensorMap tmW;
  const uint64_t t_rows = static_cast<uint64_t>(args.E) * args.max_m;
  for (int i = 0; i < 4; ++i) {
    const uint32_t h = (16u << i) <= t_rows ? (16u << i) : 16u;
    if (int st = make_tmap_u8_sw128(&tmT.box[i], A, t_rows, args.K, args.K, h)) return st;
  }
  if (int st = make_tmap_u8_sw128(&tmW, B, static_cast<uint64_t>(args.E) * args.N, args.K, args.K, 128))
    return st;
  const size_t smem = C::smem_bytes(args.E);
  if (int st = prepare_kernel(gemm_fp8_weights_m_kernel<BNT>, smem, C::kSplitRegs)) return st;
  if (args.wait_limit_ns == 0) args.wait_limit_ns = kWaitLimitNs;
  const int64_t tiles_upper = static_cast<int64_t>(args.E) * ((args.max_m + BNT - 1) / BNT) * (args.N / 128);
  int64_t grid = num_sms();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) grid = 1;
  return launch_pdl(gemm_fp8_weights_m_kernel<BNT>, static_cast<unsigned>(grid), kThreads, smem, stream, tmT,
                    tmW, args);
}

}  // namespace

// GEMM1 with SwiGLU + 1x128 requantisation fused into the epilogue (used by
// moe_ffn when the tokens-as-M kernel serves the layout).  Outputs: FP8
// Q2 [rows, N/2] (row stride N/2) and fp32 scales S2 in groups of S2_G rows.
int gemm_masked_swiglu(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                       const int32_t* counts, int32_t E, int32_t max_m, int32_t N, int32_t K,
                       uint8_t* Q2, float* S2, int32_t flags, int32_t* err, cudaStream_t st) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 256 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(max_m > 0 && static_cast<int64_t>(E) * max_m < (1ll << 31));
  MOE_CHECK_ARG(A && sA && B && sB && counts && Q2 && S2 && aligned16(A) && aligned16(B) && aligned16(Q2));
  if (int rc = check_device()) return rc;
  GemmArgs a{};
  a.sA = sA;
  a.sA_G = max_m;
  a.sB = sB;
  a.counts = counts;
  a.E = E;
  a.N = N;
  a.K = K;
  a.max_m = max_m;
  a.layout = MOE_LAYOUT_MASKED;
  a.err = err;
  a.flags = flags & ~MOE_GEMM_DEBUG_STALL;
  a.Q2 = Q2;
  a.S2 = S2;
  a.S2_G = max_m;
  const int64_t tiles = static_cast<int64_t>(E) * ((max_m + BM - 1) / BM) * (N / BN);
  return launch_tokens_m(A, static_cast<int64_t>(E) * max_m, K, B, tiles, a, st, true);
}

int gemm_contig_swiglu(const uint8_t* A, int64_t lda, const float* sA, int64_t sA_ld,
                       const uint8_t* B, const float* sB, const int32_t* offsets,
                       const int32_t* m_indices, int64_t M_capacity, int32_t E, int32_t N, int32_t K,
                       uint8_t* Q2, float* S2, int64_t s2_ld, int32_t flags, int32_t* err,
                       cudaStream_t st) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 256 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(M_capacity > 0 && M_capacity % BM == 0 && M_capacity < (1ll << 31));
  MOE_CHECK_ARG(A && sA && B && sB && offsets && m_indices && Q2 && S2);
  MOE_CHECK_ARG(aligned16(A) && aligned16(B) && aligned16(Q2) && lda % 16 == 0 && sA_ld >= M_capacity &&
                s2_ld >= M_capacity);
  if (int rc = check_device()) return rc;
  GemmArgs a{};
  a.sA = sA;
  a.sA_G = sA_ld;
  a.sB = sB;
  a.offsets = offsets;
  a.m_indices = m_indices;
  a.M_capacity = M_capacity;
  a.E = E;
  a.N = N;
  a.K = K;
  a.layout = MOE_LAYOUT_CONTIG;
  a.err = err;
  a.flags = flags & ~MOE_GEMM_DEBUG_STALL;
  a.Q2 = Q2;
  a.S2 = S2;
  a.S2_G = s2_ld;
  const int64_t tiles = (M_capacity / BM) * (N / BN);
  return launch_tokens_m(A, M_capacity, lda, B, tiles, a, st, true);
}

// GEMM2 with the single-slot combine folded into the epilogue (moe_ffn, k = 1):
// each routed row r goes to out[row_src[r]] scaled by topk_w[row_src[r]].
int gemm_masked_combine1(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                         const int32_t* counts, int32_t E, int32_t max_m, int32_t N, int32_t K,
                         const int32_t* row_src, const float* topk_w, uint16_t* out, int64_t ldo,
                         int32_t flags, int32_t* err, cudaStream_t st) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(max_m > 0 && static_cast<int64_t>(E) * max_m < (1ll << 31));
  MOE_CHECK_ARG(A && sA && B && sB && counts && row_src && topk_w && out && aligned16(A) && aligned16(B) &&
                aligned16(out) && ldo >= N && ldo % 8 == 0);
  if (int rc = check_device()) return rc;
  GemmArgs a{};
  a.sA = sA;
  a.sA_G = max_m;
  a.sB = sB;
  a.counts = counts;
  a.E = E;
  a.N = N;
  a.K = K;
  a.max_m = max_m;
  a.layout = MOE_LAYOUT_MASKED;
  a.err = err;
  a.flags = flags & ~MOE_GEMM_DEBUG_STALL;
  a.row_src = row_src;
  a.topk_w = topk_w;
  a.out = out;
  a.ldo = ldo;
  const int64_t tiles = static_cast<int64_t>(E) * ((max_m + BM - 1) / BM) * ((N + BN - 1) / BN);
  return launch_tokens_m(A, static_cast<int64_t>(E) * max_m, K, B, tiles, a, st);
}

int gemm_contig_combine1(const uint8_t* A, int64_t lda, const float* sA, int64_t sA_ld, const uint8_t* B,
                         const float* sB, const int32_t* offsets, const int32_t* m_indices, int64_t M_capacity,
                         int32_t E, int32_t N, int32_t K, const int32_t* row_src, const float* topk_w,
                         uint16_t* out, int64_t ldo, int32_t flags, int32_t* err, cudaStream_t st) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(M_capacity > 0 && M_capacity % BM == 0 && M_capacity < (1ll << 31));
  MOE_CHECK_ARG(A && sA && B && sB && offsets && m_indices && row_src && topk_w && out);
  MOE_CHECK_ARG(aligned16(A) && aligned16(B) && aligned16(out) && lda % 16 == 0 && sA_ld >= M_capacity &&
                ldo >= N && ldo % 8 == 0);
  if (int rc = check_device()) return rc;
  GemmArgs a{};
  a.sA = sA;
  a.sA_G = sA_ld;
  a.sB = sB;
  a.offsets = offsets;
  a.m_indices = m_indices;
  a.M_capacity = M_capacity;
  a.E = E;
  a.N = N;
  a.K = K;
  a.layout = MOE_LAYOUT_CONTIG;
  a.err = err;
  a.flags = flags & ~MOE_GEMM_DEBUG_STALL;
  a.row_src = row_src;
  a.topk_w = topk_w;
  a.out = out;
  a.ldo = ldo;
  const int64_t tiles = (M_capacity / BM) * ((N + BN - 1) / BN);
  return launch_tokens_m(A, M_capacity, lda, B, tiles, a, st);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_gemm_fp8_contig(const uint8_t* A, int64_t lda, const float* sA, int64_t sA_ld,
                                   const uint8_t* B, const float* sB, const int32_t* offsets,
                                   const int32_t* m_indices, int64_t M_capacity, int32_t E,
                                   int32_t N, int32_t K, uint16_t* D, int64_t ldd, int32_t flags,
                                   int32_t* err, void* stream) {
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(M_capacity >= 0 && M_capacity % BM == 0 && M_capacity < (1ll << 31));
  if (M_capacity == 0) return MOE_OK;
  MOE_CHECK_ARG(A && sA && B && sB && offsets && m_indices && D);
  MOE_CHECK_ARG(aligned16(A) && aligned16(B) && aligned16(D) && aligned16(sA));
  MOE_CHECK_ARG(lda >= K && lda % 16 == 0 && sA_ld >= M_capacity && ldd >= N && ldd % 8 == 0);
  MOE_CHECK_ARG(static_cast<int64_t>(E) * N < (1ll << 31));
  if (int st = check_device()) return st;
  GemmArgs a{};
  a.sA = sA;
  a.sA_G = sA_ld;
  a.sB = sB;
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
  if ((flags & MOE_GEMM_CTA_PAIR) && N % BN == 0)
    return launch_tokens_m_pair(A, M_capacity, lda, B, (M_capacity / BM) * (N / BN), a, as_stream(stream));
  const int64_t tiles = (M_capacity / BM) * ((N + BN - 1) / BN);
  return launch_tokens_m(A, M_capacity, lda, B, tiles, a, as_stream(stream));
}

extern "C" int moe_gemm_fp8_masked_variant(int32_t max_m, int32_t expected_m, int32_t flags) {
  // Measured on GB300: weights-as-M wins only for a few tokens per expert
  // (all-experts decode, 1-8 rows each); from ~100 rows per expert the
  // tokens-as-M tile moves fewer bytes per k-block and is about 2x faster.
  const int hint = expected_m > 0 ? expected_m : max_m;
  bool weights_m = (max_m % 16 == 0) && hint <= 32;
  if (flags & MOE_GEMM_FORCE_TOKENS_M) weights_m = false;
  if (flags & MOE_GEMM_FORCE_WEIGHTS_M) {
    if (max_m % 16 != 0) return MOE_ERR_UNSUPPORTED;
    weights_m = true;
  }
  if (!weights_m) return 0;
  return hint <= 48 ? 64 : hint <= 112 ? 128 : 256;
}

extern "C" int moe_gemm_fp8_masked(const uint8_t* A, const float* sA, const uint8_t* B,
                                   const float* sB, const int32_t* counts, int32_t E,
                                   int32_t max_m, int32_t N, int32_t K, int32_t expected_m,
                                   uint16_t* D, int32_t flags, int32_t* err, void* stream) {
  (void)expected_m;
  MOE_CHECK_ARG(E >= 1 && E <= kMaxExperts && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0);
  MOE_CHECK_ARG(max_m > 0 && static_cast<int64_t>(E) * max_m < (1ll << 31));
  MOE_CHECK_ARG(A && sA && B && sB && counts && D);
  MOE_CHECK_ARG(aligned16(A) && aligned16(B) && aligned16(D) && aligned16(sA));
  MOE_CHECK_ARG(static_cast<int64_t>(E) * N < (1ll << 31));
  if (int st = check_device()) return st;
  GemmArgs a{};
  a.sA = sA;
  a.sA_G = max_m;
  a.sB = sB;
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
  if (flags & MOE_GEMM_DEBUG_STALL) a.wait_limit_ns = 200ull * 1000ull * 1000ull;
  // Kernel choice: weights-as-M streams each expert's weights once per up to 256
  // tokens and sizes the token side to the count, so it serves decode counts;
  // tokens-as-M is kept for large counts.  Host-side only: the counts stay on
  // the device.
  const int variant = moe_gemm_fp8_masked_variant(max_m, expected_m, flags);
  if (variant < 0) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (variant == 64) return launch_weights_m<64>(A, B, a, st);
  if (variant == 128) return launch_weights_m<128>(A, B, a, st);
  if (variant == 256) return launch_weights_m<256>(A, B, a, st);
  if ((flags & MOE_GEMM_CTA_PAIR) && N % BN == 0)
    return launch_tokens_m_pair(A, static_cast<int64_t>(E) * max_m, K, B,
                                static_cast<int64_t>(E) * ((max_m + BM2 - 1) / BM2) * (N / BN), a, st);
  const int64_t tiles = static_cast<int64_t>(E) * ((max_m + BM - 1) / BM) * ((N + BN - 1) / BN);
  return launch_tokens_m(A, static_cast<int64_t>(E) * max_m, K, B, tiles, a, st);
}
