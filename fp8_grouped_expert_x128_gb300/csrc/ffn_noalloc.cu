// moe_ffn_noalloc: the whole FFN with its intermediates in a fixed scratch
// array that lives in this library's device image, for callers that cannot
// allocate device memory themselves.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// never uses the array's name as an address (on the host it only stands in for
// the device symbol); instead, the first call on each device looks the device
// address up with cudaGetSymbolAddress while that device is current, caches it,
// and hands it to moe_ffn as its workspace.  Nothing in the workspace has to
// start at zero: every region the path reads is written earlier in the same
// call (rows past a count are read as don't-care inputs and never stored).
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_ffn_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device (set up on first use).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ffn_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_ffn_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" int moe_ffn_noalloc(const moe_ffn_desc* desc, void* stream) {
  const size_t need = moe_ffn_workspace_size(desc);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  if (int st = check_device()) return st;
  void* scratch = nullptr;
  if (int st = scratch_for_current_device(&scratch)) return st;
  return moe_ffn(desc, scratch, kNoAllocScratchBytes, stream);
}
