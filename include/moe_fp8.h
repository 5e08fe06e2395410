/*
 * moe_fp8.h -- C ABI of the GB300 (sm_103a) routed-expert FP8 MoE FFN library.
 *
 * The hot path of DeepSeek-style MoE serving on one GPU: 1x128 E4M3 activation
 * quantisation with fp32 scales, permutation into a grouped layout, a grouped
 * FP8 GEMM against 128x128 block-scaled E4M3 expert weights, SwiGLU with FP8
 * requantisation, a second grouped GEMM, and the top-k-weighted combine back to
 * token order.
 *
 * Sources.  "Deploying DeepSeek on GB200 NVL72 with PD and Large Scale EP
 * (Part I)", section "Implementation details", DeepGEMM bullet: an FP8 GEMM
 * library for Blackwell built on UMMA whose API quantises and packs the input
 * scales.  "Deploying DeepSeek with PD Disaggregation and Large-Scale Expert
 * Parallelism on 96 H100 GPUs", section "DeepGEMM integration": two grouped
 * GEMMs for MoE, one for prefill (fed by DeepEP's normal dispatch -> the
 * contiguous layout here) and one for decode (fed by the CUDA-Graph-compatible
 * low-latency dispatch -> the masked layout here).  The pages give no formulas;
 * the definitions below are this library's, each stated where it applies.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are device pointers, allocated and owned by the
 *    caller.  The library never allocates device memory and never synchronises,
 *    except moe_read_device_status.  Work is enqueued on `stream` (a
 *    cudaStream_t passed as void*; NULL = the legacy default stream), so a call
 *    sequence can be captured in a CUDA graph.  Kernels are launched with
 *    programmatic dependent launch: one may begin its local set-up while the
 *    previous kernel on the stream finishes, but it waits for that kernel's
 *    completion before touching memory, so stream order is kept.
 *  - bf16 tensors are passed as uint16_t bit patterns; FP8 tensors are uint8_t
 *    OCP E4M3FN codes (bias 7, max 448, NaN 0x7F/0xFF).
 *  - Every base pointer must be 16-byte aligned; K, H and I are multiples of 128.
 *  - Return value: MOE_OK or a negative MOE_ERR_*.  Argument errors are found on
 *    the host before anything is enqueued (nothing is launched then).  Errors
 *    only the GPU can see (a count above max_m, an expert id or row index out of
 *    range, a pipeline wait that ran past its time limit) are OR-ed as
 *    MOE_DEV_* bits into the caller's device word `err` (may be NULL to
 *    ignore); read them with moe_read_device_status.  No kernel traps.
 *  - Scale layout ("packed", MN-major): for a tensor with rows r and 128-column
 *    blocks kb, rows are split into groups of G rows; the fp32 scale of (r, kb)
 *    sits at s[((r / G) * KB + kb) * G + r % G].  The masked layout uses
 *    G = max_m (one group per expert: s[e][kb][m]); the token-order and
 *    contiguous layouts use one group, G = s_ld >= rows (s[kb][r]).
 */
#ifndef MOE_FP8_H_
#define MOE_FP8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status ------------------------------------------------------------ */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)  /* null/misaligned pointer, bad size or stride      */
#define MOE_ERR_UNSUPPORTED (-2)  /* not an sm_103/sm_100-family device, shape limits  */
#define MOE_ERR_CUDA (-3)         /* a CUDA runtime/driver call failed                 */
#define MOE_ERR_OVERFLOW (-4)     /* device: a masked count exceeded max_m (clamped)   */
#define MOE_ERR_TIMEOUT (-5)      /* device: a pipeline wait ran past its time limit   */
#define MOE_ERR_BAD_INDEX (-6)    /* device: an expert id / row index out of range     */

/* bits of the device error word */
#define MOE_DEV_OVERFLOW 0x1
#define MOE_DEV_TIMEOUT 0x2
#define MOE_DEV_BAD_INDEX 0x4

#define MOE_LAYOUT_MASKED 0
#define MOE_LAYOUT_CONTIG 1

/* GEMM flags */
#define MOE_GEMM_DEFAULT 0
#define MOE_GEMM_FORCE_TOKENS_M 0x1   /* masked: force the tokens-as-M tile kernel      */
#define MOE_GEMM_FORCE_WEIGHTS_M 0x2  /* masked: force the weights-as-M (swap AB) kernel */
#define MOE_FFN_FUSE_SWIGLU 0x4       /* moe_ffn only: where the tokens-as-M kernel serves
                                         GEMM1, run SwiGLU + 1x128 requantisation in its
                                         epilogue instead of writing bf16 Y1 and calling
                                         moe_swiglu_quant (same bytes either way)         */
#define MOE_GEMM_CTA_PAIR 0x8         /* tokens-as-M: run each 256x256 tile on a 2-CTA
                                         cluster (one M = 256 UMMA, each SM stages half
                                         of B); needs N % 256 == 0, else ignored        */
#define MOE_FFN_UE8M0 0x10            /* moe_ffn only: the power-of-two (UE8M0) reading of
                                         the packed scales end to end -- both activation
                                         quantisations take power-of-two scales, packed for
                                         the block-scaled GEMMs, which read the weights'
                                         packed scales w13_sf / w2_sf                     */
#define MOE_GEMM_EARLY_WEIGHTS 0x20   /* the routing arrays the GEMM reads (masked counts;
                                         contiguous offsets and m_indices) were complete
                                         before the kernel launched just before this call on
                                         the stream began, i.e. that kernel does not write
                                         them: the GEMM then builds its tile schedule and
                                         starts streaming weight tiles (and their scales)
                                         before it waits for that kernel (programmatic
                                         dependent launch), and loads the activations and
                                         their scales after.  moe_ffn sets it for both of
                                         its GEMMs.  Wrong results if the arrays are written
                                         by the immediately preceding kernel.             */
#define MOE_GEMM_DEBUG_STALL 0x100    /* test only: the TMA producer never issues, so the
                                         consumer's bounded wait expires and the call
                                         reports MOE_DEV_TIMEOUT (no hang, no trap)      */

/* moe_quant_fp8 flags */
#define MOE_QUANT_UE8M0 0x1           /* power-of-two block scales (the rule of
                                         moe_quant_fp8_ue8m0), written as fp32 2^e     */
/* moe_combine flags */
#define MOE_COMBINE_ACCUMULATE 0x1    /* add to the output's current values            */

/* Human-readable name of a status code. Never NULL. */
const char *moe_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int moe_version(void);

/*
 * Synchronise `stream`, read the device error word `err` (device, int32),
 * clear it to 0, and return in *status_out the most severe MOE_ERR_* it held
 * (BAD_INDEX over TIMEOUT over OVERFLOW; MOE_OK if clear).  *raw_bits_out (may
 * be NULL) receives the raw MOE_DEV_* bits.  The only call that synchronises.
 */
int moe_read_device_status(int32_t *err, void *stream, int *status_out, int32_t *raw_bits_out);

/*
 * a1 -- 1x128 activation quantisation (moe_quant_fp8).
 * Per row m and 128-column block kb of x:
 *   amax = max |x[m, kb*128 .. kb*128+127]|
 *   s    = fp32( max(amax, 1e-4) / 448 )            (IEEE float32 division)
 *   q    = e4m3_rne_satfinite( fp32( x / s ) )       (IEEE float32 division)
 * x  : device bf16 [M, K], row stride ldx (elements).
 * q  : device uint8 [M, K], row stride ldq (bytes).
 * s  : device fp32, one group: s[kb * s_ld + m], s_ld >= M.
 * flags: 0, or MOE_QUANT_UE8M0 for power-of-two scales (the rule of
 *   moe_quant_fp8_ue8m0 below; s then holds 2^e).  Unknown bits are refused.
 * Non-finite inputs: NaN elements take no part in amax (maxNum) and encode to
 * 0x7F; an infinite element makes s = inf, so the block's finite elements
 * encode to signed zeros and the infinite one to 0x7F.
 * M may be 0 (nothing is launched).
 */
int moe_quant_fp8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                  uint8_t *q, int64_t ldq, float *s, int64_t s_ld, int32_t flags,
                  int32_t *err, void *stream);

/*
 * a1 with power-of-two (UE8M0) block scales -- the alternative reading of the
 * DeepGEMM bullet's "packing of the input scales" ("Deploying DeepSeek on
 * GB200 NVL72 with PD and Large Scale EP (Part I)", Implementation details),
 * the scale format of the hardware block-scaled MMA.  Per row m and block kb:
 *   s = 2^e, e the smallest integer with max(amax, 1e-4) / 2^e <= 448
 *   q = e4m3_rne_satfinite( x / s )                  (exact: s is a power of two)
 * x, q, s, s_ld as moe_quant_fp8 (s holds the float value 2^e);
 * e8 : device uint8 (may be NULL), e8[kb * s_ld + m] = e + 127.
 */
int moe_quant_fp8_ue8m0(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t *q, int64_t ldq, float *s, uint8_t *e8, int64_t s_ld,
                        int32_t *err, void *stream);

/* The UE8M0 block-scale rule above for one block maximum, on the host:
 * returns s = 2^e and stores e + 127 in *byte_out (may be NULL).  An
 * infinite maximum gives s = inf and byte 0xFF. */
float moe_ue8m0_scale(float amax, uint8_t *byte_out);

/*
 * a3 -- 128x128 block weight quantisation (set-up, not on the timed path).
 * The a1 rule with amax taken over each 128x128 tile.
 * w : device bf16 [E, N, K] (K-major: the GEMM's B operand, out x in).
 * q : device uint8 [E, N, K];  s : device fp32 [E, N/128, K/128] (4-byte
 * alignment suffices for s, so per-expert slices may be quantised one by one).
 */
int moe_quant_weight_fp8(const uint16_t *w, int64_t E, int64_t N, int64_t K,
                         uint8_t *q, float *s, void *stream);

/*
 * a3 with power-of-two (UE8M0) tile scales: the rule of moe_quant_fp8_ue8m0
 * with amax over each 128x128 tile.  q, s as moe_quant_weight_fp8 (s holds
 * 2^e); e8 (device uint8 [E, N/128, K/128], may be NULL) holds e + 127.
 */
int moe_quant_weight_fp8_ue8m0(const uint16_t *w, int64_t E, int64_t N, int64_t K,
                               uint8_t *q, float *s, uint8_t *e8, void *stream);

/*
 * Rows a contiguous-layout buffer must be able to hold for `assignments`
 * routed rows over E experts when each segment is padded to a multiple of 128.
 */
int64_t moe_contig_rows_bound(int64_t assignments, int32_t E);

/*
 * a2 -- permute token-order FP8 rows into the grouped layout (moe_permute).
 * Assignment i = t*k + j goes to local expert e = topk_ids[t, j] - expert_begin
 * when 0 <= e < E (other ids are another rank's experts and are skipped).
 * Within an expert, rows keep ascending i (deterministic, stable).
 *
 * q, s      : device, token order, as written by moe_quant_fp8 (rows T, row
 *             stride H bytes; s[kb * s_ld + t]).
 * topk_ids  : device int32 [T, k].
 * layout = MOE_LAYOUT_MASKED: expert e owns rows [e*max_m, (e+1)*max_m) of
 *   q_out (device uint8 [E*max_m, H]) and s_out (device fp32 [E, H/128, max_m]).
 *   counts[e] (device int32 [E]) = rows kept = min(arrivals, max_m); arrivals past
 *   max_m get dst_row = -1 and set MOE_DEV_OVERFLOW.  row_src: [E*max_m].
 *   Rows >= counts[e] of q_out/s_out are left untouched.  rows_capacity is
 *   ignored; offsets and m_indices may be NULL.
 * layout = MOE_LAYOUT_CONTIG: expert segments follow each other, each padded to
 *   a multiple of 128 rows.  offsets (device int32 [E+1]): first row of each
 *   segment, offsets[E] = rows used.  m_indices (device int32 [rows_capacity]):
 *   owning expert of each real row, -1 on padding and past offsets[E].
 *   q_out: [rows_capacity, H]; s_out: s_out[kb * s_out_ld + row], s_out_ld >=
 *   rows_capacity.  counts[e] = arrivals.  rows_capacity must be at least
 *   moe_contig_rows_bound(T*k, E).  row_src: [rows_capacity].  Padding rows of
 *   q_out/s_out are left untouched.
 * row_src[row] = i of the assignment stored there, -1 elsewhere.
 * dst_row[i]   (device int32 [T*k]) = destination row, -1 if not stored.
 * Limits: E <= 1024, k <= 32.
 */
int moe_permute(const uint8_t *q, const float *s, int64_t s_ld,
                const int32_t *topk_ids, int64_t T, int32_t H, int32_t k,
                int32_t expert_begin, int32_t E, int32_t layout, int32_t max_m,
                uint8_t *q_out, float *s_out, int64_t s_out_ld,
                int32_t *counts, int32_t *offsets, int32_t *m_indices,
                int32_t *row_src, int32_t *dst_row, int64_t rows_capacity,
                int32_t *err, void *stream);

/*
 * a4 / a6 -- grouped FP8 GEMM with block-scaled operands.
 *   D[r, n] = bf16_rne( sum_kb  sA[r, kb] * sB[e, n/128, kb]
 *                              * sum_{k in kb} A[r, k] * B[e, n, k] )
 * where e is the expert owning row r.  E4M3 products are exact; the inner sum
 * runs on the tcgen05 tensor cores into TMEM, and each 128-deep block partial
 * is scaled and accumulated in fp32 by the epilogue warps.
 * B  : device uint8 [E, N, K] (K-major), sB: device fp32 [E, N/128, K/128].
 * N % 128 == 0, K % 128 == 0.
 *
 * moe_gemm_fp8_contig -- contiguous (prefill) layout, as moe_permute writes it:
 *   A [M_capacity, K] (row stride lda), sA[kb * sA_ld + r], offsets [E+1],
 *   m_indices [M_capacity]; D row stride ldd.  Rows with m_indices == -1 and
 *   rows >= offsets[E] are not written.  Segments must start at multiples of 128
 *   and lie inside [0, M_capacity): a segment that does not (offsets[e] < 0, not
 *   a multiple of 128, decreasing, or offsets[e+1] > M_capacity) is skipped --
 *   none of its rows is read or written -- and MOE_DEV_BAD_INDEX is set.
 */
int moe_gemm_fp8_contig(const uint8_t *A, int64_t lda, const float *sA, int64_t sA_ld,
                        const uint8_t *B, const float *sB,
                        const int32_t *offsets, const int32_t *m_indices, int64_t M_capacity,
                        int32_t E, int32_t N, int32_t K,
                        uint16_t *D, int64_t ldd, int32_t flags, int32_t *err, void *stream);

/*
 * moe_gemm_fp8_masked -- masked (decode) layout, as moe_permute writes it:
 *   A [E, max_m, K], sA [E, K/128, max_m], counts [E] (device; read on the
 *   GPU only, so the call is graph-capturable), D [E, max_m, N].
 *   Rows >= counts[e] of D are left untouched; counts[e] > max_m is clamped
 *   and sets MOE_DEV_OVERFLOW.  expected_m (>= 0) is a host-side hint of the
 *   typical count used to pick the tile kernel (0 = unknown).
 */
int moe_gemm_fp8_masked(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                        const int32_t *counts, int32_t E, int32_t max_m, int32_t N, int32_t K,
                        int32_t expected_m, uint16_t *D, int32_t flags, int32_t *err,
                        void *stream);

/*
 * a4 / a6 with power-of-two (UE8M0) block scales applied by the tensor cores
 * -- the reading of the DeepGEMM bullet ("Deploying DeepSeek on GB200 NVL72
 * with PD and Large Scale EP (Part I)", Implementation details: an FP8 GEMM on
 * UMMA whose API quantises and packs the input scales) in which the packed
 * scales are exponent bytes, four k-blocks per 32-bit word, that the MMA
 * consumes (tcgen05.mma kind::mxf8f6f4.block_scale).  The product is the same
 * definition as moe_gemm_fp8_*:
 *   D[r, n] = bf16_rne( sum_kb  sA[r, kb] * sB[e, n/128, kb] * sum_{k in kb} A[r, k] * B[e, n, k] )
 * with sA = 2^(a - 127), sB = 2^(b - 127) read from the packed words; the
 * accumulation is fp32 across all k-blocks in TMEM.
 *
 * Packed activation scales (sfA, uint32 words, 16-byte aligned): rows are in
 * groups of G (masked layout: G = max_m, one group per expert; contiguous:
 * one group of G = sfA_ld rows, sfA_ld a multiple of 128 >= M_capacity);
 * within a group, chunks of 128 rows.  For group grp, k-group g (k-blocks
 * 4g .. 4g+3), chunk c and row i of the chunk:
 *   word index = ((grp * KG + g) * NC + c) * 128 + 4 * (i % 32) + i / 32,
 *   KG = ceil(K / 512), NC = ceil(G / 128);
 * byte b of the word is the exponent byte (e + 127) of k-block 4g + b (0x7F
 * past the last k-block).  This order puts every row's word where the tensor
 * cores read it after one 512-byte copy into tensor memory.
 * Packed weight scales (sfB, 16-byte aligned): for expert e, 128-row block nb
 * and k-group g, 32 copies of the word whose byte b is the exponent byte of
 * block (nb, 4g + b): word index ((e * (N/128) + nb) * KG + g) * 32 + j.
 *
 * moe_ue8m0_act_words / moe_ue8m0_weight_words: sizes of the two arrays in
 * words (-1 for bad sizes).  moe_pack_ue8m0_act: power-of-two fp32 scales in
 * the grouped layout of the fp32 scales (s[((r / G) * KB + kb) * G + r % G],
 * as moe_quant_fp8 with MOE_QUANT_UE8M0 and moe_permute write them; only the
 * exponent field is read) -> sfA, for `groups` groups of G rows of which the
 * first `rows` exist (the rest pack as scale 1).  moe_pack_ue8m0_weight:
 * power-of-two fp32 weight scales [E, N/128, K/128] (moe_quant_weight_fp8_ue8m0)
 * -> sfB.
 * The GEMMs take the arguments of moe_gemm_fp8_contig / moe_gemm_fp8_masked
 * with the packed arrays in place of the fp32 scales (sfA_ld as above).
 */
int64_t moe_ue8m0_act_words(int64_t groups, int64_t G, int64_t K);
int64_t moe_ue8m0_weight_words(int64_t E, int64_t N, int64_t K);
int moe_pack_ue8m0_act(const float *s, int64_t groups, int64_t G, int64_t rows, int64_t K,
                       uint32_t *sfA, void *stream);
int moe_pack_ue8m0_weight(const float *s, int64_t E, int64_t N, int64_t K, uint32_t *sfB, void *stream);
int moe_gemm_fp8_contig_ue8m0(const uint8_t *A, int64_t lda, const uint32_t *sfA, int64_t sfA_ld,
                              const uint8_t *B, const uint32_t *sfB,
                              const int32_t *offsets, const int32_t *m_indices, int64_t M_capacity,
                              int32_t E, int32_t N, int32_t K,
                              uint16_t *D, int64_t ldd, int32_t flags, int32_t *err, void *stream);
int moe_gemm_fp8_masked_ue8m0(const uint8_t *A, const uint32_t *sfA, const uint8_t *B, const uint32_t *sfB,
                              const int32_t *counts, int32_t E, int32_t max_m, int32_t N, int32_t K,
                              int32_t expected_m, uint16_t *D, int32_t flags, int32_t *err,
                              void *stream);

/*
 * Which masked-GEMM kernel moe_gemm_fp8_masked runs for these arguments
 * (host-side, nothing launched): 0 = tokens-as-M (128 token rows x 256 weight
 * rows per tile); 64 / 128 / 256 = weights-as-M with token tiles of that many
 * columns; MOE_ERR_UNSUPPORTED if the flags ask for weights-as-M and max_m is
 * not a multiple of 16.  The choice follows expected_m (0 = use max_m):
 * weights-as-M (64-column token tiles) up to 32 expected rows per expert,
 * tokens-as-M above.  MOE_GEMM_FORCE_WEIGHTS_M with expected_m in (48, 112]
 * or above 112 selects the 128- or 256-column token tiles.
 */
int moe_gemm_fp8_masked_variant(int32_t max_m, int32_t expected_m, int32_t flags);

/*
 * a5 -- fused SwiGLU + 1x128 requantisation (moe_swiglu_quant).
 *   h[r, i] = silu(g) * u,  g = Y1[r, i], u = Y1[r, I + i]   (gate first, then up)
 * computed in fp32 (silu(g) = g / (1 + exp(-g))), never rounded to bf16, then
 * quantised by the a1 rule into q [rows, I] (row stride I) and s (groups of G rows).
 * Y1 : device bf16 [rows, 2I] (row stride 2I).
 * Row selection: masked -> counts != NULL, G = max_m, row r is processed iff
 *   r % max_m < counts[r / max_m] (at most 1024 experts = rows / max_m);
 *   contig -> counts == NULL, m_indices != NULL,
 *   G = s_ld, row r processed iff r < rows and m_indices[r] >= 0.
 * Unprocessed rows of q and s are left untouched.
 * flags: 0, or MOE_QUANT_UE8M0 for power-of-two scales (the rule of
 * moe_quant_fp8_ue8m0; s then holds 2^e).  Unknown bits are refused.
 */
int moe_swiglu_quant(const uint16_t *Y1, int64_t rows, int32_t I,
                     const int32_t *counts, int32_t max_m, const int32_t *m_indices,
                     uint8_t *q, float *s, int64_t s_ld, int32_t flags, int32_t *err, void *stream);

/*
 * a7 -- top-k-weighted combine back to token order (moe_combine).
 *   out[t, :] = bf16_rne( a[t, :] + sum_j  w[t, j] * Y2[dst_row[t*k + j], :] + shared[t, :] )
 * with a = the current out row under MOE_COMBINE_ACCUMULATE (else 0) and the
 * shared term only when shared_or_null is given (a shared expert's output,
 * weight 1).  fp32 accumulation: a, then the slots in j order, then the shared
 * row -- the same steps as routing the shared expert as one more slot of
 * weight 1, so the bits equal that formulation.  Entries with dst_row == -1 are
 * skipped (a token with none and no other term gets zeros).
 * Y2: device bf16 rows of H (row stride ldy); dst_row: device int32 [T*k];
 * topk_w: device fp32 [T, k]; shared_or_null: device bf16 [T, H] (row stride
 * lds) or NULL; out: device bf16 [T, H] (row stride ldo).  flags: 0 or
 * MOE_COMBINE_ACCUMULATE; unknown bits are refused.  dst_row values must be <
 * y_rows (else MOE_DEV_BAD_INDEX and the entry is skipped).
 */
int moe_combine(const uint16_t *Y2, int64_t ldy, int64_t y_rows,
                const int32_t *dst_row, const float *topk_w, int64_t T, int32_t k, int32_t H,
                const uint16_t *shared_or_null, int64_t lds, int32_t flags,
                uint16_t *out, int64_t ldo, int32_t *err, void *stream);

/*
 * a8 -- the whole routed-expert FFN on one stream, no host synchronisation:
 *   moe_quant_fp8 -> moe_permute -> GEMM1 (W13) -> moe_swiglu_quant -> GEMM2 (W2)
 *   -> moe_combine.
 * Weights: w13 [E, 2I, H] (gate rows [0, I), up rows [I, 2I)) with w13_s
 * [E, 2I/128, H/128]; w2 [E, H, I] with w2_s [E, H/128, I/128] (device).
 * Token I/O: x, topk_ids, topk_w and out may be device memory of the current
 * GPU or page-locked host memory that CUDA maps at the same address
 * (cudaHostAlloc / cudaMallocHost / cudaHostRegister with the mapped flag):
 * the kernels then read x, the routing and the weights of each slot and write
 * out in place across the host link, overlapped with the compute, with no
 * separate copies (the end-to-end path from host buffers).  Weights and the
 * workspace must be device memory of the current GPU.  Any other placement
 * (pageable host memory, another GPU's memory) returns MOE_ERR_INVALID_ARG
 * before anything is launched (checked with cudaPointerGetAttributes).
 * workspace: device, at least moe_ffn_workspace_size(desc) bytes, 256-byte
 * aligned; holds every intermediate.  stage_events (optional, may be NULL):
 * 7 cudaEvent_t handles recorded on `stream` before stage 1 and after each of
 * the six stages, for per-stage timing.  moe_ffn quantises each routed token
 * row straight into its expert slot (stages 1 and 2 fused, same bytes as the
 * separate calls), so events 0 and 1 are recorded back to back; with
 * MOE_FFN_FUSE_SWIGLU in gemm_flags and the tokens-as-M kernel serving GEMM1,
 * stages 3 and 4 are fused the same way (events 3 and 4 back to back).
 * With MOE_FFN_UE8M0 in gemm_flags the chain takes the power-of-two reading of
 * the scales: x and h are quantised with the rule of moe_quant_fp8_ue8m0 and
 * their scales written in the packed layout, both GEMMs run block-scaled
 * (moe_gemm_fp8_*_ue8m0) with the weights' packed scales w13_sf and w2_sf
 * (w13_s / w2_s are then not read), and MOE_FFN_FUSE_SWIGLU is ignored.
 */
typedef struct moe_ffn_desc {
  int64_t T;              /* tokens (rows of x and out); T = 0 is an
                             empty batch: the token I/O may then be null
                             and moe_ffn launches nothing               */
  int32_t H, I, k;        /* hidden, intermediate, routing slots/token  */
  int32_t expert_begin;   /* global id of local expert 0               */
  int32_t E;              /* local experts                              */
  int32_t layout;         /* MOE_LAYOUT_MASKED / MOE_LAYOUT_CONTIG      */
  int32_t max_m;          /* masked: rows per expert                    */
  int32_t expected_m;     /* masked: count hint for tile selection (0)  */
  int32_t gemm_flags;     /* MOE_GEMM_* for both GEMMs                  */
  const uint16_t *x;      /* [T, H] bf16                                */
  const int32_t *topk_ids;/* [T, k]                                     */
  const float *topk_w;    /* [T, k]                                     */
  const uint8_t *w13;
  const float *w13_s;
  const uint8_t *w2;
  const float *w2_s;
  uint16_t *out;          /* [T, H] bf16                                */
  int32_t *err;           /* device error word (may be NULL)            */
  void **stage_events;    /* optional 7 cudaEvent_t                     */
  const uint32_t *w13_sf; /* MOE_FFN_UE8M0: packed W13 scales (moe_pack_ue8m0_weight) */
  const uint32_t *w2_sf;  /* MOE_FFN_UE8M0: packed W2 scales                           */
} moe_ffn_desc;

/* Number of kernels one moe_ffn call with this descriptor launches (the same
 * choices moe_ffn makes: the routing index pass inside the quant-scatter for
 * masked batches of at most 1024 routing ids, as one kernel, or as two kernels
 * above 8192 ids; the optional SwiGLU fusion; the single-slot combine in
 * GEMM2), or a negative MOE_ERR_* for a descriptor moe_ffn would refuse.
 * Host-only, no launch. */
int moe_ffn_kernel_count(const moe_ffn_desc *desc);
size_t moe_ffn_workspace_size(const moe_ffn_desc *desc);
int moe_ffn(const moe_ffn_desc *desc, void *workspace, size_t workspace_bytes, void *stream);

/*
 * moe_ffn without a caller-supplied workspace (no counterpart in the pages:
 * this is a convenience of this library, not part of the method).
 *
 * Some callers cannot allocate device memory at the point where they run the
 * FFN: a plug-in inside an inference runtime that owns all device memory and
 * hands out only the tensors it plans, code that runs while a CUDA graph is
 * being captured (where cudaMalloc is not allowed), or a latency-critical loop
 * that must not stall on the allocator.  For them this call runs exactly the
 * moe_ffn path, but keeps every intermediate in a scratch array that is part of
 * the library's own device image, so neither the caller nor the library
 * allocates anything.  The caller still passes the inputs and the output
 * through `desc` (desc->err may be NULL, as in moe_ffn).
 *
 * Limits and rules:
 *  - The scratch holds moe_ffn_noalloc_capacity() bytes (64 MiB); every GPU
 *    that loads the library holds it until the process exits.  A descriptor
 *    whose moe_ffn_workspace_size exceeds it is rejected with
 *    MOE_ERR_UNSUPPORTED before anything is launched (the masked decode layout
 *    needs about 40 KB per row of E*max_m at hidden 7168 / intermediate 2048).
 *  - The first call on a device looks up the scratch's device address (with
 *    that device current) and caches it; make that first call before any stream
 *    capture on the device.
 *  - All calls share the one array, which keeps the last call's contents.
 *    Calls whose work overlaps on the GPU (other streams, or other host threads
 *    on the same device) race on it: serialise them.  Nothing in the scratch
 *    needs to start at zero.
 *  - Return codes as moe_ffn.
 */
size_t moe_ffn_noalloc_capacity(void);
int moe_ffn_noalloc(const moe_ffn_desc *desc, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FP8_H_ */
