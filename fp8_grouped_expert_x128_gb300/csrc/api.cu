// Host runtime of the library: status codes, device checks, TMA descriptor
// encoding, and moe_ffn -- the whole routed-expert FFN enqueued on one stream
// with no host synchronisation (graph-capturable, like the decode path the
// pages pair with DeepEP's CUDA-Graph-compatible low-latency mode: "Deploying
// DeepSeek with PD Disaggregation and Large-Scale Expert Parallelism on 96
// H100 GPUs", section "Expert parallelism based on DeepEP").
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

int check_device() {
  static int cache[64];
  static bool init = false;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (int& c : cache) c = 1;  // 1 = unknown
    init = true;
  }
  if (cache[dev] == 1) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    // The kernels are built for sm_103a only.
    cache[dev] = (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_UNSUPPORTED;
  }
  return cache[dev];
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

int make_tmap_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld_bytes, uint32_t box_rows) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return MOE_ERR_CUDA;
  if (!aligned16(base) || ld_bytes % 16 != 0 || rows == 0 || cols == 0) return MOE_ERR_INVALID_ARG;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld_bytes};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

int make_tmap_b16_out(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld_bytes) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return MOE_ERR_CUDA;
  if (!aligned16(base) || ld_bytes % 16 != 0 || rows == 0 || cols == 0) return MOE_ERR_INVALID_ARG;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld_bytes};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct FfnPlan {
  int64_t T_pad, rows, s_ld1, s_ld2;
  bool ue8m0;   // packed power-of-two activation scales (off_sa1 / off_sa2 hold words)
  size_t off_counts, off_offsets, off_mind, off_rowsrc, off_dst, off_lrank, off_hist, off_a1, off_sa1,
      off_y1, off_a2, off_sa2, off_y2, total;
};

int plan_ffn(const moe_ffn_desc* d, FfnPlan* p) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->H % 128 || d->I <= 0 || d->I % 128 || d->k < 1 || d->k > 32 ||
      d->E < 1 || d->E > 1024)
    return MOE_ERR_INVALID_ARG;
  const int64_t H = d->H, I = d->I, E = d->E;
  p->T_pad = (d->T + 3) / 4 * 4;
  if (d->layout == MOE_LAYOUT_MASKED) {
    if (d->max_m <= 0) return MOE_ERR_INVALID_ARG;
    p->rows = E * d->max_m;
    p->s_ld1 = p->s_ld2 = d->max_m;
  } else if (d->layout == MOE_LAYOUT_CONTIG) {
    p->rows = moe_contig_rows_bound(d->T * d->k, d->E);
    if (p->rows == 0) p->rows = 128;
    p->s_ld1 = p->s_ld2 = p->rows;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  p->off_counts = take(sizeof(int32_t) * E);
  p->off_offsets = take(sizeof(int32_t) * (E + 1));
  p->off_mind = take(sizeof(int32_t) * p->rows);
  p->off_rowsrc = take(sizeof(int32_t) * p->rows);
  p->off_dst = take(sizeof(int32_t) * d->T * d->k);
  // scratch of the many-CTA index pass (large batches)
  p->off_lrank = take(sizeof(int32_t) * d->T * d->k);
  p->off_hist = take(sizeof(int32_t) * static_cast<size_t>(permute_chunk_count(d->T * d->k)) * E);
  p->ue8m0 = (d->gemm_flags & MOE_FFN_UE8M0) != 0;
  // packed UE8M0 scales: masked -> one group of max_m rows per expert;
  // contiguous -> one group of `rows` rows (a multiple of 128)
  const int64_t groups = d->layout == MOE_LAYOUT_MASKED ? E : 1;
  const int64_t G = d->layout == MOE_LAYOUT_MASKED ? d->max_m : p->rows;
  auto scale_bytes = [&](int64_t K) {
    return p->ue8m0 ? sizeof(uint32_t) * static_cast<size_t>(moe_ue8m0_act_words(groups, G, K))
                    : sizeof(float) * (K / 128) * p->rows;
  };
  p->off_a1 = take(static_cast<size_t>(p->rows) * H);
  p->off_sa1 = take(scale_bytes(H));
  p->off_y1 = take(sizeof(uint16_t) * p->rows * 2 * I);
  p->off_a2 = take(static_cast<size_t>(p->rows) * I);
  p->off_sa2 = take(scale_bytes(I));
  p->off_y2 = take(sizeof(uint16_t) * p->rows * H);
  p->total = o;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_OVERFLOW: return "MOE_ERR_OVERFLOW";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX";
    default: return "MOE_ERR_UNKNOWN";
  }
}

extern "C" int moe_version(void) { return 200; }

extern "C" int moe_read_device_status(int32_t* err, void* stream, int* status_out,
                                      int32_t* raw_bits_out) {
  if (err == nullptr || status_out == nullptr) return MOE_ERR_INVALID_ARG;
  int32_t bits = 0;
  cudaStream_t st = as_stream(stream);
  MOE_CUDA_TRY(cudaMemcpyAsync(&bits, err, sizeof(bits), cudaMemcpyDeviceToHost, st));
  MOE_CUDA_TRY(cudaMemsetAsync(err, 0, sizeof(int32_t), st));
  MOE_CUDA_TRY(cudaStreamSynchronize(st));
  if (raw_bits_out) *raw_bits_out = bits;
  if (bits & MOE_DEV_BAD_INDEX)
    *status_out = MOE_ERR_BAD_INDEX;
  else if (bits & MOE_DEV_TIMEOUT)
    *status_out = MOE_ERR_TIMEOUT;
  else if (bits & MOE_DEV_OVERFLOW)
    *status_out = MOE_ERR_OVERFLOW;
  else
    *status_out = MOE_OK;
  return MOE_OK;
}

namespace {

// Where a pointer handed to moe_ffn may live.  `host_ok`: the token I/O (x,
// topk_ids, topk_w, out) may also be page-locked host memory that CUDA maps at
// the same address (cudaHostAlloc, cudaMallocHost, cudaHostRegister with the
// mapped flag); the kernels then read and write it in place across the host
// link.  Anything else (pageable host memory, another GPU's memory) would fault
// in a kernel, so it is refused before any launch.
// `on_host` (may be NULL) is set when the pointer is page-locked host memory.
int check_placement(const void* ptr, bool host_ok, bool* on_host = nullptr) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (on_host) *on_host = false;
  if (a.type == cudaMemoryTypeDevice) return a.device == dev ? MOE_OK : MOE_ERR_INVALID_ARG;
  if (a.type == cudaMemoryTypeManaged) return MOE_OK;
  if (host_ok && a.type == cudaMemoryTypeHost && a.devicePointer == ptr) {
    if (on_host) *on_host = true;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

// moe_ffn's fusion choices for a descriptor (shared with moe_ffn_kernel_count).
struct FfnFusion {
  bool swiglu;    // SwiGLU + requant in GEMM1's epilogue
  bool combine;   // single-slot combine in GEMM2's epilogue (no combine kernel)
};

// The index pass runs inside the quant-scatter kernel (no index kernel) for the
// masked layout when there are few routing ids (each CTA scans the ids before
// its token) and few slots per token.  Measured: the all-experts layer at
// T = 1 / 64 gains 4 µs per step; at ~4000 ids (c2) the scans cost 7 µs more
// than the index kernel they replace.
constexpr int64_t kFuseIndexMaxIds = 1024;
bool ffn_fuse_index(const moe_ffn_desc* d) {
  return d->layout == MOE_LAYOUT_MASKED && d->T > 0 && d->T * d->k <= kFuseIndexMaxIds && d->k <= 16;
}

FfnFusion ffn_fusion(const moe_ffn_desc* d, bool out_on_host) {
  const bool masked = d->layout == MOE_LAYOUT_MASKED;
  const int32_t gflags = d->gemm_flags & ~MOE_FFN_FUSE_SWIGLU;
  FfnFusion f;
  if (d->gemm_flags & MOE_FFN_UE8M0) {
    // the block-scaled path: no SwiGLU fusion; the single-slot combine goes
    // into GEMM2's epilogue where the tokens-as-M kernel serves it
    f.swiglu = false;
    f.combine = d->k == 1 && !out_on_host &&
                (!masked || moe_gemm_fp8_masked_variant(d->max_m, d->expected_m, gflags) == 0);
    return f;
  }
  // stages 3+4: on request (MOE_FFN_FUSE_SWIGLU) and where the tokens-as-M
  // kernel serves GEMM1, SwiGLU and the FP8 requantisation run in its
  // epilogue (no bf16 Y1 round trip); otherwise GEMM1 writes Y1 and the
  // SwiGLU kernel requantises it.
  f.swiglu = (d->gemm_flags & MOE_FFN_FUSE_SWIGLU) &&
             (!masked || moe_gemm_fp8_masked_variant(d->max_m, d->expected_m, d->gemm_flags) == 0);
  // One routing slot per token (k = 1, e.g. the prefill layout): GEMM2's
  // epilogue writes each routed row to its token's output with the combine's
  // arithmetic, and the quant-scatter pass zeroes the rows of tokens not routed
  // here, so the combine kernel and the Y2 round trip drop out.  Where the
  // weights-as-M or the CTA-pair kernel would serve GEMM2, the plain path runs,
  // and so it does when out is in host memory: GEMM2's epilogue writes each
  // row in 16-byte pieces from 32 rows at a time, which the host link serves
  // far worse than the combine kernel's whole-row stores.
  f.combine = d->k == 1 && !out_on_host && !(gflags & MOE_GEMM_CTA_PAIR) &&
              (!masked || moe_gemm_fp8_masked_variant(d->max_m, d->expected_m, gflags) == 0);
  return f;
}

}  // namespace

extern "C" int moe_ffn_kernel_count(const moe_ffn_desc* d) {
  FfnPlan p;
  if (plan_ffn(d, &p) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (d->T == 0) return 0;                                                // an empty batch launches nothing
  if (d->out == nullptr) return MOE_ERR_INVALID_ARG;
  bool out_on_host = false;
  if (int rc = check_placement(d->out, true, &out_on_host)) return rc;
  const FfnFusion f = ffn_fusion(d, out_on_host);
  // quant-scatter, with the index pass inside it, or before it as one kernel
  // or (large batches) as two
  int n = ffn_fuse_index(d) ? 1 : (d->T * d->k > kIdxMultiMinIds ? 3 : 2);
  n += f.swiglu ? 1 : 2;                                                  // GEMM1 (+ SwiGLU)
  n += 1;                                                                 // GEMM2
  n += f.combine ? 0 : 1;                                                 // combine
  return n;
}

extern "C" size_t moe_ffn_workspace_size(const moe_ffn_desc* desc) {
  FfnPlan p;
  if (plan_ffn(desc, &p) != MOE_OK) return 0;
  return p.total;
}

extern "C" int moe_ffn(const moe_ffn_desc* d, void* workspace, size_t workspace_bytes,
                       void* stream) {
  FfnPlan p;
  if (int st = plan_ffn(d, &p)) return st;
  MOE_CHECK_ARG(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255) == 0);
  MOE_CHECK_ARG(workspace_bytes >= p.total);
  const bool ue8m0 = p.ue8m0;
  MOE_CHECK_ARG(d->w13 && d->w2);
  if (ue8m0)
    MOE_CHECK_ARG(d->w13_sf && d->w2_sf && aligned16(d->w13_sf) && aligned16(d->w2_sf));
  else
    MOE_CHECK_ARG(d->w13_s && d->w2_s);
  // An empty batch (T = 0) reads and writes no token, so its token I/O may be
  // null (as an empty framework tensor's is): nothing is launched, only the
  // stage events are recorded.
  const bool empty = d->T == 0;
  if (!empty) MOE_CHECK_ARG(d->x && d->topk_ids && d->topk_w && d->out);
  if (int st = check_device()) return st;
  bool out_on_host = false;
  if (!empty) {
    const void* io[3] = {d->x, d->topk_ids, d->topk_w};
    for (const void* ptr : io)
      if (int rc = check_placement(ptr, true)) return rc;
    if (int rc = check_placement(d->out, true, &out_on_host)) return rc;
  }
  const void* on_device[5] = {d->w13, ue8m0 ? static_cast<const void*>(d->w13_sf) : d->w13_s, d->w2,
                              ue8m0 ? static_cast<const void*>(d->w2_sf) : d->w2_s, workspace};
  for (const void* ptr : on_device)
    if (int rc = check_placement(ptr, false)) return rc;
  cudaStream_t st = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return static_cast<void*>(ws + off); };
  int32_t* counts = static_cast<int32_t*>(at(p.off_counts));
  int32_t* offsets = static_cast<int32_t*>(at(p.off_offsets));
  int32_t* mind = static_cast<int32_t*>(at(p.off_mind));
  int32_t* rowsrc = static_cast<int32_t*>(at(p.off_rowsrc));
  int32_t* dst = static_cast<int32_t*>(at(p.off_dst));
  uint8_t* a1 = static_cast<uint8_t*>(at(p.off_a1));
  float* sa1 = static_cast<float*>(at(p.off_sa1));
  uint16_t* y1 = static_cast<uint16_t*>(at(p.off_y1));
  uint8_t* a2 = static_cast<uint8_t*>(at(p.off_a2));
  float* sa2 = static_cast<float*>(at(p.off_sa2));
  uint16_t* y2 = static_cast<uint16_t*>(at(p.off_y2));
  const bool masked = d->layout == MOE_LAYOUT_MASKED;
  cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(d->stage_events);
  // Under stream capture the stage events become external event-record nodes,
  // which keep their timestamps when the graph is replayed.
  unsigned ev_flags = cudaEventRecordDefault;
  if (ev) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    MOE_CUDA_TRY(cudaStreamIsCapturing(st, &cap));
    if (cap == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
  }
  auto mark = [&](int i) -> int {
    if (ev) MOE_CUDA_TRY(cudaEventRecordWithFlags(ev[i], st, ev_flags));
    return MOE_OK;
  };
  int rc;
  if (empty) {
    for (int i = 0; i < 7; ++i)
      if ((rc = mark(i))) return rc;
    return MOE_OK;
  }
  const int32_t gflags = d->gemm_flags & ~(MOE_FFN_FUSE_SWIGLU | MOE_FFN_UE8M0);
  const FfnFusion fusion = ffn_fusion(d, out_on_host);
  const bool fuse_combine = fusion.combine;
  // The routing arrays are written by the index pass: by a separate kernel two
  // launches before GEMM1 (the quant-scatter runs in between; T > 0 here), or
  // inside the quant-scatter kernel just before GEMM1 for small masked batches,
  // and in either case before GEMM2's predecessor; a GEMM whose routing arrays
  // are final may build its schedule and start streaming weights before it
  // waits for the kernel just ahead of it.
  const bool fuse_index = ffn_fuse_index(d);
  const int32_t g1flags = gflags | (fuse_index ? 0 : MOE_GEMM_EARLY_WEIGHTS);
  const int32_t g2flags = gflags | MOE_GEMM_EARLY_WEIGHTS;
  // stages 1+2: routing index pass, then each routed token row is quantised
  // straight into its expert slot (no token-order FP8 copy in between)
  if ((rc = mark(0))) return rc;
  if ((rc = mark(1))) return rc;
  if ((rc = permute_launch(nullptr, nullptr, 0, d->x, d->H, d->topk_ids, d->T, d->H, d->k,
                           d->expert_begin, d->E, d->layout, d->max_m, a1, ue8m0 ? nullptr : sa1, p.s_ld1, counts,
                           offsets, mind, rowsrc, dst, p.rows, d->err, st, fuse_combine ? d->out : nullptr,
                           d->H, ue8m0 ? reinterpret_cast<uint8_t*>(sa1) : nullptr, fuse_index,
                           static_cast<int32_t*>(at(p.off_lrank)), static_cast<int32_t*>(at(p.off_hist)))))
    return rc;
  if ((rc = mark(2))) return rc;
  if (ue8m0) {
    // the power-of-two reading end to end: block-scaled GEMMs on packed scales
    const uint32_t* sf1 = reinterpret_cast<const uint32_t*>(sa1);
    const uint32_t* sf2 = reinterpret_cast<const uint32_t*>(sa2);
    rc = masked ? moe_gemm_fp8_masked_ue8m0(a1, sf1, d->w13, d->w13_sf, counts, d->E, d->max_m, 2 * d->I, d->H,
                                            d->expected_m, y1, g1flags, d->err, stream)
                : moe_gemm_fp8_contig_ue8m0(a1, d->H, sf1, p.rows, d->w13, d->w13_sf, offsets, mind, p.rows, d->E,
                                            2 * d->I, d->H, y1, 2 * d->I, g1flags, d->err, stream);
    if (rc) return rc;
    if ((rc = mark(3))) return rc;
    if ((rc = swiglu_launch(y1, p.rows, d->I, masked ? counts : nullptr, masked ? d->max_m : 0,
                            masked ? nullptr : mind, a2, nullptr, p.s_ld2, true, reinterpret_cast<uint8_t*>(sa2),
                            st)))
      return rc;
    if ((rc = mark(4))) return rc;
    if (fuse_combine)
      rc = gemm_ue8m0_combine1(a2, sf2, d->w2, d->w2_sf, masked ? counts : nullptr, masked ? nullptr : offsets,
                               masked ? nullptr : mind, p.rows, d->E, d->max_m, d->H, d->I, rowsrc, d->topk_w,
                               d->out, d->H, g2flags, d->err, st);
    else
      rc = masked ? moe_gemm_fp8_masked_ue8m0(a2, sf2, d->w2, d->w2_sf, counts, d->E, d->max_m, d->H, d->I,
                                              d->expected_m, y2, g2flags, d->err, stream)
                  : moe_gemm_fp8_contig_ue8m0(a2, d->I, sf2, p.rows, d->w2, d->w2_sf, offsets, mind, p.rows, d->E,
                                              d->H, d->I, y2, d->H, g2flags, d->err, stream);
    if (rc) return rc;
    if ((rc = mark(5))) return rc;
    if (!fuse_combine &&
        (rc = moe_combine(y2, d->H, p.rows, dst, d->topk_w, d->T, d->k, d->H, nullptr, 0, 0, d->out, d->H, d->err,
                          stream)))
      return rc;
    return mark(6);
  }
  const bool fuse_swiglu = fusion.swiglu;
  if (fuse_swiglu) {
    if (masked)
      rc = gemm_masked_swiglu(a1, sa1, d->w13, d->w13_s, counts, d->E, d->max_m, 2 * d->I, d->H,
                              a2, sa2, g1flags, d->err, st);
    else
      rc = gemm_contig_swiglu(a1, d->H, sa1, p.s_ld1, d->w13, d->w13_s, offsets, mind, p.rows, d->E,
                              2 * d->I, d->H, a2, sa2, p.s_ld2, g1flags, d->err, st);
    if (rc) return rc;
    if ((rc = mark(3))) return rc;
    if ((rc = mark(4))) return rc;
  } else {
    if (masked)
      rc = moe_gemm_fp8_masked(a1, sa1, d->w13, d->w13_s, counts, d->E, d->max_m, 2 * d->I, d->H,
                               d->expected_m, y1, g1flags, d->err, stream);
    else
      rc = moe_gemm_fp8_contig(a1, d->H, sa1, p.s_ld1, d->w13, d->w13_s, offsets, mind, p.rows, d->E,
                               2 * d->I, d->H, y1, 2 * d->I, g1flags, d->err, stream);
    if (rc) return rc;
    if ((rc = mark(3))) return rc;
    if ((rc = moe_swiglu_quant(y1, p.rows, d->I, masked ? counts : nullptr, masked ? d->max_m : 0,
                               masked ? nullptr : mind, a2, sa2, p.s_ld2, 0, d->err, stream)))
      return rc;
    if ((rc = mark(4))) return rc;
  }
  if (fuse_combine && masked)
    rc = gemm_masked_combine1(a2, sa2, d->w2, d->w2_s, counts, d->E, d->max_m, d->H, d->I, rowsrc,
                              d->topk_w, d->out, d->H, g2flags, d->err, st);
  else if (fuse_combine)
    rc = gemm_contig_combine1(a2, d->I, sa2, p.s_ld2, d->w2, d->w2_s, offsets, mind, p.rows, d->E, d->H,
                              d->I, rowsrc, d->topk_w, d->out, d->H, g2flags, d->err, st);
  else if (masked)
    rc = moe_gemm_fp8_masked(a2, sa2, d->w2, d->w2_s, counts, d->E, d->max_m, d->H, d->I,
                             d->expected_m, y2, g2flags, d->err, stream);
  else
    rc = moe_gemm_fp8_contig(a2, d->I, sa2, p.s_ld2, d->w2, d->w2_s, offsets, mind, p.rows, d->E,
                             d->H, d->I, y2, d->H, g2flags, d->err, stream);
  if (rc) return rc;
  if ((rc = mark(5))) return rc;
  if (!fuse_combine &&
      (rc = moe_combine(y2, d->H, p.rows, dst, d->topk_w, d->T, d->k, d->H, nullptr, 0, 0, d->out, d->H, d->err,
                        stream)))
    return rc;
  return mark(6);
}
