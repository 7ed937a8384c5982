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
// * The array lives in the library's device code module.  With CUDA's lazy
//   module loading that module (and the array's 16 MiB) is loaded into a
//   context by the first call there that needs scratch, which can therefore
//   fail for lack of device memory (reported as HH_ERR_CUDA); once that call
//   has succeeded, no later call in the same context allocates anything.
// * That first call also looks up the array's device address
//   (cudaGetSymbolAddress), with the device current.  The address is kept per
//   device together with the unique id of the CUDA context it was taken in,
//   and looked up again when a call runs in another context (after a
//   cudaDeviceReset, for example).  Make the first call of a context before
//   starting any stream capture.
// * All calls share the one array, and it keeps whatever the last call left
//   there.  Nothing in it has to start at zero: every call writes each part of
//   the scratch before it reads that part.  Calls whose kernels overlap on the
//   GPU (different streams, or concurrent host threads) race on the array and
//   must not be issued.
// * Arguments are checked as in hh_linattn_fwd_causal (pointers, alignment,
//   shapes, then the device), and only then the size: a problem whose scratch
//   need exceeds the array's size is rejected with HH_ERR_WORKSPACE before
//   anything is launched.

#include <cuda.h>

#include <mutex>

#include "hh_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;   // unique id of the context ptr belongs to
  bool ready = false;
};
ScratchAddr g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  cudaGetLastError();
  return nullptr;
}

// Unique id of the calling thread's current CUDA context; false when there is
// none or the driver cannot say.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current
// context, looked up once per context.
hh_status scratch_for_current_context(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return HH_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  ScratchAddr& c = g_scratch[dev];
  if (c.ready && have_id && c.ctx_id == id) {
    *out = c.ptr;
    return HH_OK;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();   // leave no pending runtime error behind
    c.ready = false;
    return HH_ERR_CUDA;
  }
  // the lookup makes the context current if it was not yet; key on it now
  c.ready = current_context_id(&c.ctx_id);
  c.ptr = ptr;
  *out = ptr;
  return HH_OK;
}

}  // namespace

extern "C" HH_API hh_status hh_linattn_fwd_causal_noalloc(
    const hh_fmap* fmap, int dtype, const void* q, const void* k, const void* v, int64_t B,
    int H, int64_t n, int chunk, void* y, float* S_out, float* z_out, int* dev_status,
    void* stream) {
  hh::Problem p;
  hh_status st = hh::fwd_check_args(fmap, dtype, q, k, v, B, H, n, chunk, nullptr, nullptr, y,
                                    S_out, z_out, nullptr, dev_status, &p);
  if (st != HH_OK) return st;
  if (B == 0) return HH_OK;
  if (!hh::device_is_supported()) return HH_ERR_UNSUPPORTED;
  const size_t need = hh_fwd_workspace_bytes(fmap, dtype, B, H, n, chunk);
  if (need > kScratchBytes) return HH_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_for_current_context(&scratch);
    if (st != HH_OK) return st;
  }
  return hh_linattn_fwd_causal(fmap, dtype, q, k, v, B, H, n, chunk, y, S_out, z_out, scratch,
                               need > 0 ? kScratchBytes : 0, dev_status, stream);
}
