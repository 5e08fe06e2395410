// Shared device/host helpers of the sm_103a MoE FP8 library: status plumbing,
// bounded mbarrier waits, TMA and tcgen05 (UMMA / TMEM) inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <utility>

#include "../../include/moe_fp8.h"

namespace moe {

// ---------------------------------------------------------------- host side
#define MOE_CHECK_ARG(cond)                 \
  do {                                      \
    if (!(cond)) return MOE_ERR_INVALID_ARG; \
  } while (0)

#define MOE_CUDA_TRY(expr)                    \
  do {                                        \
    cudaError_t e_ = (expr);                  \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Streaming-multiprocessor count of the current device (cached per device).
int num_sms();
// 0 if the current device can run the sm_103a kernels.
int check_device();
// Launch error of the last kernel -> status.
inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Every kernel is launched with programmatic dependent launch: it may start
// (and run its purely local set-up) while the previous kernel on the stream
// finishes, and waits on grid_dependency_wait() before it touches global
// memory that a neighbour reads or writes.  Every CTA of every kernel calls
// the wait before it exits, so completion stays ordered along the stream.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? MOE_OK
                                                                                      : MOE_ERR_CUDA;
}

// Permute (index pass + row gather), shared by moe_permute and moe_ffn.  With
// x != nullptr the rows are quantised from bf16 on the way (1x128 rule).
int permute_launch(const uint8_t* q, const float* s, int64_t s_ld, const uint16_t* x, int64_t ldx,
                   const int32_t* topk_ids, int64_t T, int32_t H, int32_t k,
                   int32_t expert_begin, int32_t E, int32_t layout, int32_t max_m,
                   uint8_t* q_out, float* s_out, int64_t s_out_ld, int32_t* counts,
                   int32_t* offsets, int32_t* m_indices, int32_t* row_src, int32_t* dst_row,
                   int64_t rows_capacity, int32_t* err, cudaStream_t st,
                   uint16_t* zero_out = nullptr, int64_t ldo = 0, uint8_t* sf8_out = nullptr,
                   bool fuse_index = false, int32_t* lrank = nullptr, int32_t* chunk_hist = nullptr);
// Scratch of the many-CTA index pass (used above kIdxMultiMinIds assignments
// when the caller provides it): lrank [T*k] and chunk_hist [ceil(T*k / 4096)][E]
// int32.
constexpr int64_t kIdxMultiMinIds = 8192;
inline int64_t permute_chunk_count(int64_t assignments) { return (assignments + 4095) / 4096; }

// SwiGLU + 1x128 requantisation (moe_swiglu_quant and moe_ffn): fp32 scales
// in groups of G rows, or (sf8) exponent bytes in the packed UE8M0 layout.
int swiglu_launch(const uint16_t* Y1, int64_t rows, int32_t I, const int32_t* counts, int32_t max_m,
                  const int32_t* m_indices, uint8_t* q, float* s, int64_t s_ld, bool ue8m0, uint8_t* sf8,
                  cudaStream_t st);

// GEMM1 with SwiGLU + 1x128 requantisation fused into the tokens-as-M
// epilogue (bytes equal GEMM1 -> moe_swiglu_quant); used inside moe_ffn.
int gemm_masked_swiglu(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                       const int32_t* counts, int32_t E, int32_t max_m, int32_t N, int32_t K,
                       uint8_t* Q2, float* S2, int32_t flags, int32_t* err, cudaStream_t st);
// GEMM2 with the single-slot combine in its epilogue (k = 1): routed row r is
// written to out[row_src[r]] as bf16(w * bf16(D[r])), w = topk_w[row_src[r]].
int gemm_masked_combine1(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                         const int32_t* counts, int32_t E, int32_t max_m, int32_t N, int32_t K,
                         const int32_t* row_src, const float* topk_w, uint16_t* out, int64_t ldo,
                         int32_t flags, int32_t* err, cudaStream_t st);
int gemm_contig_combine1(const uint8_t* A, int64_t lda, const float* sA, int64_t sA_ld, const uint8_t* B,
                         const float* sB, const int32_t* offsets, const int32_t* m_indices, int64_t M_capacity,
                         int32_t E, int32_t N, int32_t K, const int32_t* row_src, const float* topk_w,
                         uint16_t* out, int64_t ldo, int32_t flags, int32_t* err, cudaStream_t st);
int gemm_contig_swiglu(const uint8_t* A, int64_t lda, const float* sA, int64_t sA_ld,
                       const uint8_t* B, const float* sB, const int32_t* offsets,
                       const int32_t* m_indices, int64_t M_capacity, int32_t E, int32_t N, int32_t K,
                       uint8_t* Q2, float* S2, int64_t s2_ld, int32_t flags, int32_t* err,
                       cudaStream_t st);

// Block-scaled (UE8M0) GEMM2 with the single-slot combine in its epilogue
// (moe_ffn with MOE_FFN_UE8M0, k = 1); contiguous when offsets != NULL.
int gemm_ue8m0_combine1(const uint8_t* A, const uint32_t* sfA, const uint8_t* B, const uint32_t* sfB,
                        const int32_t* counts, const int32_t* offsets, const int32_t* m_indices, int64_t rows,
                        int32_t E, int32_t max_m, int32_t N, int32_t K, const int32_t* row_src,
                        const float* topk_w, uint16_t* out, int64_t ldo, int32_t flags, int32_t* err,
                        cudaStream_t st);

// Encode a 2-D K-major uint8 tensor map with 128-byte swizzle:
// global [rows, cols] (row stride ld bytes), box [box_rows, 128 bytes].
int make_tmap_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld_bytes, uint32_t box_rows);
// 2-D map over a row-major bf16 (16-bit) matrix for TMA stores of 32 x 32
// boxes from shared memory in the 64-byte swizzle (a 64-byte row's 16-byte
// chunk c sits at c ^ ((row >> 1) & 3)).  Same rules and codes as above.
int make_tmap_b16_out(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld_bytes);

// ---------------------------------------------------------------- device side
// Default limit of one pipeline wait.  Waits normally last microseconds; past
// the limit the kernel flags MOE_DEV_TIMEOUT, unwinds and returns.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_err(int32_t* err, int32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

// ---- programmatic dependent launch
// Wait until the grids this one depends on have completed and their memory
// is visible; then let the next grid on the stream begin launching.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity.  Returns false (and the
// caller unwinds) if another role raised *abort, or if the wait itself ran
// past limit_ns -- then it raises *abort and flags MOE_DEV_TIMEOUT.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, int32_t* err,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        set_err(err, MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// ---- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- cp.async: a 4-byte global -> shared copy that does not block the issuing
// thread; src_bytes = 0 reads nothing and writes zeros.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// One arrival on `bar` from this thread once all of its earlier cp.async
// copies have landed (counted against the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Global -> shared bulk copy (16-byte aligned, a multiple of 16 bytes) that
// completes `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Shared -> global TMA store of one box, tracked by the issuing thread's bulk
// groups.  The writes to shared memory it reads must be made visible to the
// async proxy first (fence_proxy_async_shared by each writing thread).
__device__ __forceinline__ void tma_store_2d(const void* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// all but the most recent of this thread's bulk store groups have read their source
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- tcgen05 (5th-generation tensor cores, accumulators in TMEM)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row (1024 B) swizzle atoms
// stacked along M/N (stride byte offset 1024); the leading byte offset is not
// used by swizzled K-major layouts.  Descriptor version 1 (sm_100 family).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;             // LBO (ignored), encoded 16 B
  d |= static_cast<uint64_t>(1024 >> 4) << 32;     // SBO = 1024 B
  d |= static_cast<uint64_t>(1) << 46;             // version
  d |= static_cast<uint64_t>(2) << 61;             // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f8f6f4: D fp32, A = B = E4M3, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                   // D format: F32
         | (0u << 7) | (0u << 10)                    // A, B: E4M3
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void umma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---- CTA pairs (2-CTA clusters sharing one UMMA of M = 256)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives and waits.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_wait_bounded, for barriers that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          volatile int* abort, int32_t* err,
                                                          uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++spins & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        set_err(err, MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}
// TMEM allocation for a CTA pair: warp 1 of each CTA executes these together;
// the pair gets the same columns in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// M = 256 UMMA over the pair, issued by the even CTA: A rows 0..127 from its
// shared memory, rows 128..255 from the odd CTA's at the same address; B's
// first N/2 rows from the even CTA, the rest from the odd one; each CTA's TMEM
// receives its own 128 rows of D.
__device__ __forceinline__ void umma_e4m3_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` (same address) in every CTA of `cta_mask` once the pair
// MMAs issued so far by this thread are done.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- E4M3 conversion: round to nearest even, saturating to +-448.
// Returns the byte of `a` in bits [7:0] and of `b` in bits [15:8].
__device__ __forceinline__ uint16_t e4m3x2_rn_satfinite(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}


// ---- 1x128 block quantisation helpers (one half-warp per 128-element block,
// 8 bf16 per lane): s = fp32(max(amax, 1e-4) / 448), q = e4m3(fp32(x / s)),
// both IEEE float32 divisions.  Every kernel that quantises uses these, so the
// bytes are the same whichever kernel wrote them.
constexpr float kQuantFloor = 1e-4f;
constexpr float kQuantMax = 448.0f;
// 1/448 rounded to nearest (a compile-time IEEE division), the reciprocal the
// scale division below is corrected with.
constexpr float kQuantMaxRcp = 1.0f / 448.0f;

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// x / s rounded to nearest-even for a finite, positive, normal s, given
// r = 1/s rounded to nearest: the product y = x*r is corrected once by the
// residual x - y*s, the final step of correctly rounded division by a known
// reciprocal in P. Markstein, "IA-64 and Elementary Functions" (2000).  A zero
// quotient takes x's sign, as the quotient itself would.  Every element of a
// 1x128 block divides by the same scale, so the reciprocal is taken once.
__device__ __forceinline__ float div_rn_by(float x, float s, float r) {
  const float y = x * r;
  const float e = fmaf(-y, s, x);
  return copysignf(fmaf(e, r, y), x);
}

// Two float32 lanes in one 64-bit register pair, for the packed f32x2
// arithmetic of sm_100 and later (each lane an IEEE float32 operation with
// round-to-nearest-even, subnormals kept: the same results as two scalar ops).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint2 pack_e4m3x8(const float (&q)[8]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lo |= e4m3x2_rn_satfinite(q[2 * i], q[2 * i + 1]) << (16 * i);
    hi |= e4m3x2_rn_satfinite(q[4 + 2 * i], q[4 + 2 * i + 1]) << (16 * i);
  }
  return make_uint2(lo, hi);
}

// Quantise 8 values with scale s into 8 E4M3 bytes (element 0 in the low byte):
// q = e4m3(x / s), the division correctly rounded in float32.  The steps of
// div_rn_by on pairs of lanes: y = x*r, e = y*(-s) + x (the same exact product
// as -y*s), q = e*r + y, then the sign of x.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s) {
  float q[8];
  if (isfinite(s)) {
    const float r = __frcp_rn(s);
    const uint64_t r2 = f2_pack(r, r), ns2 = f2_pack(-s, -s);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t x2 = f2_pack(f[2 * i], f[2 * i + 1]);
      const uint64_t y2 = f2_mul(x2, r2);
      const uint64_t e2 = f2_fma(y2, ns2, x2);
      f2_unpack(f2_fma(e2, r2, y2), q[2 * i], q[2 * i + 1]);
      q[2 * i] = copysignf(q[2 * i], f[2 * i]);
      q[2 * i + 1] = copysignf(q[2 * i + 1], f[2 * i + 1]);
    }
  } else {  // only from non-finite inputs
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(f[i], s);
  }
  return pack_e4m3x8(q);
}

// quant8 for a power-of-two scale s = 2^e (the UE8M0 reading, byte = e + 127,
// e in [-22, 120]): 1/s = 2^-e is exact, so x * 2^-e, one rounding, is the
// correctly rounded x / s (zero signs included) and quant8's correction step
// has nothing to correct.  An infinite s takes quant8's division path.
__device__ __forceinline__ uint2 quant8_pow2(const float (&f)[8], float s, uint8_t byte) {
  if (byte == 0xFF) return quant8(f, s);
  const float r = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);
  const uint64_t r2 = f2_pack(r, r);
  float q[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(f2_pack(f[2 * i], f[2 * i + 1]), r2), q[2 * i], q[2 * i + 1]);
  return pack_e4m3x8(q);
}

// UE8M0 (power-of-two) block scale, the other reading of the packed input
// scales: the smallest s = 2^e with max(amax, 1e-4) / s <= 448.  Writing
// a = (1 + m / 2^23) * 2^E and 448 = 1.75 * 2^8, a <= 1.75 * 2^(e + 8) first
// holds at e = E - 8 when m <= 0.75 * 2^23 and at e = E - 7 otherwise; the
// floor keeps a normal, so e stays in [-22, 120].  *byte = e + 127, so that
// s = 2^(byte - 127).  An infinite maximum gives s = inf and byte 0xFF (the
// codes then follow the non-finite division path).  x / s is then exact (a
// power-of-two divisor), so quant8 with this s gives e4m3(x / s).  Host and
// device share this code (the host copy is exported for the tests).
__host__ __device__ inline float block_scale_ue8m0(float amax, uint8_t* byte) {
  const float a = fmaxf(amax, kQuantFloor);
  uint32_t bits;
  memcpy(&bits, &a, sizeof(bits));
  const int E = static_cast<int>((bits >> 23) & 0xFFu) - 127;
  if (E == 128) {
    *byte = 0xFF;
    return a;
  }
  const int e = E - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  *byte = static_cast<uint8_t>(e + 127);
  const uint32_t sbits = static_cast<uint32_t>(e + 127) << 23;
  float s;
  memcpy(&s, &sbits, sizeof(s));
  return s;
}

// Byte offset of (row r of its scale group grp, k-block kb) in the packed
// UE8M0 activation scales (moe_fp8.h): groups of G rows, k-groups of four
// k-blocks, 128-row chunks; row i of a chunk owns word 4 * (i % 32) + i / 32,
// k-block kb its byte kb % 4.
__host__ __device__ __forceinline__ int64_t ue8m0_act_byte(int64_t grp, int64_t r, int64_t kb, int64_t KG,
                                                           int64_t NC) {
  const int64_t i = r & 127;
  return ((((grp * KG + (kb >> 2)) * NC + (r >> 7)) << 7) + 4 * (i & 31) + (i >> 5)) * 4 + (kb & 3);
}

// Where a quantising kernel puts a block scale: the fp32 value in the grouped
// layout s[((row / G) * KB + kb) * G + row % G], or -- with sf8 given -- the
// power-of-two scale's exponent byte in the packed UE8M0 layout.
struct ScaleOut {
  float* s;
  uint8_t* sf8;
  int64_t G;
  int32_t KG, NC;
  // The part of a row's scale index that does not depend on kb (one division
  // per row); put_at adds kb's part.
  __device__ __forceinline__ int64_t row_base(int64_t row, int64_t KB) const {
    const int64_t grp = ((row | G) >> 31) == 0
                            ? static_cast<int64_t>(static_cast<uint32_t>(row) / static_cast<uint32_t>(G))
                            : row / G;
    const int64_t pos = row - grp * G;
    if (sf8 != nullptr) return ue8m0_act_byte(grp, pos, 0, KG, NC);
    return grp * KB * G + pos;
  }
  __device__ __forceinline__ void put_at(int64_t base, int64_t kb, float sc, uint8_t byte) const {
    if (sf8 != nullptr)
      sf8[base + (kb >> 2) * (static_cast<int64_t>(NC) << 9) + (kb & 3)] = byte;
    else
      s[base + kb * G] = sc;
  }
  __device__ __forceinline__ void put(int64_t row, int64_t kb, int64_t KB, float sc, uint8_t byte) const {
    put_at(row_base(row, KB), kb, sc, byte);
  }
};

// s = max(amax, 1e-4) / 448 rounded to nearest: the same one-step correction
// of a product by the rounded reciprocal (of the constant 448); non-finite
// block maxima take the full division.
__device__ __forceinline__ float block_scale(float amax) {
  const float a = fmaxf(amax, kQuantFloor);
  if (!isfinite(a)) return __fdiv_rn(a, kQuantMax);
  return div_rn_by(a, kQuantMax, kQuantMaxRcp);
}


}  // namespace moe
