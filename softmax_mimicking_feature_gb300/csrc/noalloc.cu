// hh_linattn_fwd_causal_noalloc: the causal prefill for callers that cannot
// hand the library a workspace.
//
// Some callers of this code have no way to allocate device memory at the
// point where they run the prefill: a plugin interface that only passes in
// its input and output buffers, a serving loop that forbids allocation after
// start-up (allocation can stall, fragment memory or synchronise the
// device), or a plain C host program with no device allocator of its own.
// For them this entry point keeps the prefill's scratch (the per-segment
// states of long sequences) in one fixed array of device memory that is part
// of the library image.  The array exists on every GPU that loads the
// library, for as long as the process lives.
//
// Properties callers should know:
// * The first call on each device looks up the array's device address
//   (cudaGetSymbolAddress) once, with that device current.  Make that first
//   call before starting any stream capture.
// * All calls share the one array, and it keeps whatever the last call left
//   there.  Nothing in it has to start at zero: every call writes each part of
//   the scratch before it reads that part.  Calls whose kernels overlap on the
//   GPU (different streams, or concurrent host threads) race on the array and
//   must not be issued.
// * A problem whose scratch need exceeds the array's size is rejected with
//   HH_ERR_WORKSPACE before anything is launched.
// * No device or host memory is allocated by this call.

#include <mutex>

#include "hh_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];

// Device address of the scratch array for the current device (set up once).
hh_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HH_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ready[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return HH_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return HH_OK;
}

}  // namespace

extern "C" HH_API hh_status hh_linattn_fwd_causal_noalloc(
    const hh_fmap* fmap, int dtype, const void* q, const void* k, const void* v, int64_t B,
    int H, int64_t n, int chunk, void* y, float* S_out, float* z_out, int* dev_status,
    void* stream) {
  // argument checks that need no device come first, exactly as in the
  // allocating entry point (a size query of 0 also covers invalid arguments)
  const size_t need = hh_fwd_workspace_bytes(fmap, dtype, B, H, n, chunk);
  if (need > kScratchBytes) return HH_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const hh_status st = scratch_for_current_device(&scratch);
    if (st != HH_OK) return st;
  }
  return hh_linattn_fwd_causal(fmap, dtype, q, k, v, B, H, n, chunk, y, S_out, z_out, scratch,
                               need > 0 ? kScratchBytes : 0, dev_status, stream);
}
