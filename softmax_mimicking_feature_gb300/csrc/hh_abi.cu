// C ABI entry points: argument validation, workspace sizing and dispatch to
// the kernels.  Every check happens on the host before anything is enqueued.

#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "hh_internal.cuh"

namespace hh {

// ---- cached device attributes ---------------------------------------------
namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int g_smem_optin[kMaxDevices];
int g_cc[kMaxDevices];
std::once_flag g_once[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

void query_device(int dev) {
  std::call_once(g_once[dev], [dev] {
    int v = 0;
    g_sm_count[dev] = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? v : 1;
    g_smem_optin[dev] =
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess ? v : 48 * 1024;
    int ma = 0, mi = 0;
    cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev);
    g_cc[dev] = ma * 10 + mi;
  });
}
}  // namespace

int device_sm_count() {
  const int dev = current_device();
  query_device(dev);
  return g_sm_count[dev];
}
int device_max_smem_optin() {
  const int dev = current_device();
  query_device(dev);
  return g_smem_optin[dev];
}
static int device_cc() {
  const int dev = current_device();
  query_device(dev);
  return g_cc[dev];
}

uint64_t wait_soft_limit_ns() {
  const char* e = getenv("HH_WAIT_SOFT_LIMIT_NS");
  if (e && *e) return strtoull(e, nullptr, 10);
  return 1000000000ull;
}

bool pdl_enabled() {
  const char* e = getenv("HH_PDL");
  return !(e && e[0] == '0');
}

// ---- validation -----------------------------------------------------------
namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Fills *p from the ABI arguments; checks shapes, kinds, overflow.
hh_status make_problem(const hh_fmap* fm, int dtype, int64_t B, int H, int64_t n, Problem* p) {
  if (!fm) return HH_ERR_INVALID_ARG;
  if (dtype != HH_F32 && dtype != HH_BF16) return HH_ERR_INVALID_ARG;
  if (fm->kind != HH_FMAP_HEDGEHOG && fm->kind != HH_FMAP_TAYLOR2 &&
      fm->kind != HH_FMAP_HEDGEHOG_SOFTMAX)
    return HH_ERR_INVALID_ARG;
  if (B < 0 || n < 0 || H < 1 || fm->d < 1) return HH_ERR_INVALID_ARG;
  const int d = fm->d;
  const bool softmax = fm->kind == HH_FMAP_HEDGEHOG_SOFTMAX;
  if (fm->kind == HH_FMAP_HEDGEHOG || softmax) {
    const bool ok = dtype == HH_F32 ? (d <= 128) : (d == 64 || d == 128);
    if (!ok) return HH_ERR_UNSUPPORTED;
    if (!fm->Wq) return HH_ERR_INVALID_ARG;
    if (softmax && (fm->bq || fm->bk)) return HH_ERR_INVALID_ARG;   // Eq. 5 has no bias
  } else {
    const bool ok = dtype == HH_F32 ? (d <= 16) : (d == 16);
    if (!ok) return HH_ERR_UNSUPPORTED;
  }
  // element counts must fit comfortably in int64 and index math
  const int64_t lim = (int64_t)1 << 40;
  if (B > lim || n > lim || (B && n && B * (int64_t)H > lim / std::max<int64_t>(n, 1)) ||
      B * (int64_t)H * n > lim / 512)
    return HH_ERR_INVALID_ARG;
  p->kind = softmax ? HH_FMAP_HEDGEHOG : fm->kind;
  p->softmax = softmax;
  p->offq = p->offk = nullptr;
  p->dtype = dtype;
  p->d = d;
  p->dp = hh_fmap_dim(p->kind, d, 0);
  p->dpp = hh_fmap_dim(p->kind, d, 1);
  p->B = B;
  p->H = H;
  p->n = n;
  const int hkv = fm->kv_heads;
  if (hkv < 0 || (hkv > 0 && (hkv > H || H % hkv != 0))) return HH_ERR_INVALID_ARG;
  p->G = hkv > 0 ? H / hkv : 1;
  if (fm->layout != HH_LAYOUT_BHND && fm->layout != HH_LAYOUT_BNHD) return HH_ERR_INVALID_ARG;
  p->seq_major = fm->layout == HH_LAYOUT_BNHD ? 1 : 0;
  if (p->kind == HH_FMAP_HEDGEHOG) {
    p->Wq = fm->Wq;
    p->bq = fm->bq;
    p->Wk = fm->Wk;
    p->bk = fm->Wk ? fm->bk : nullptr;
  } else {
    p->Wq = p->Wk = nullptr;
    p->bq = p->bk = nullptr;
  }
  return HH_OK;
}

hh_status check_ptrs_aligned(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return HH_ERR_ALIGNMENT;
  return HH_OK;
}

hh_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HH_OK : HH_ERR_CUDA; }

size_t elem_size(int dtype) { return dtype == HH_F32 ? 4 : 2; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Bytes of one softmax-map offset array ([U][off_stride(n)] float2).
size_t softmax_off_bytes(const Problem& p) {
  return align256((size_t)p.B * p.H * off_stride(p.n) * sizeof(float2));
}

bool device_ok() {
  // sm_103a code only; anything else is reported, not attempted
  return device_cc() == 103;
}

// Loss workspace: phi(Q), phi(K) in the call's dtype, then per-tile partial sums.
size_t loss_ws(const Problem& p) {
  const size_t phi = align256((size_t)p.B * p.H * p.n * p.dpp * elem_size(p.dtype));
  // per-tile partial sums (64-row tiles cover the 128-row ones), then the
  // per-head sums when the caller passes none (statistics only)
  const size_t part = align256((size_t)p.B * p.H * (ceil_div(p.n, loss_simt_tile()) + 1) *
                               sizeof(float));
  return 2 * phi + part;
}

}  // namespace
}  // namespace hh

namespace hh {

// Host-side argument checks of the prefill, in the order the entry points
// apply them (the workspace itself is not looked at).  Nothing touches a
// device.  On HH_OK, *p describes the problem.
hh_status fwd_check_args(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                         const void* v, int64_t B, int H, int64_t n, int chunk, const float* S0,
                         const float* z0, const void* y, const float* S_out, const float* z_out,
                         const void* workspace, const int* dev_status, Problem* p) {
  hh_status st = make_problem(fmap, dtype, B, H, n, p);
  if (st != HH_OK) return st;
  if (chunk != 0 && chunk != 64 && chunk != 128) return HH_ERR_UNSUPPORTED;
  if ((S_out == nullptr) != (z_out == nullptr)) return HH_ERR_INVALID_ARG;
  if (S0 != nullptr && !z0) return HH_ERR_INVALID_ARG;
  if (B == 0) return HH_OK;
  if (n > 0 && (!q || !k || !v || !y)) return HH_ERR_INVALID_ARG;
  if ((st = check_ptrs_aligned({q, k, v, y, S_out, z_out, S0, z0, p->Wq, p->bq, p->Wk, p->bk,
                                workspace})) != HH_OK)
    return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return HH_ERR_ALIGNMENT;
  return HH_OK;
}

bool device_is_supported() { return device_ok(); }

}  // namespace hh

using namespace hh;

extern "C" {

int hh_version(void) { return 100; }

const char* hh_status_str(int s) {
  switch (s) {
    case HH_OK: return "HH_OK";
    case HH_ERR_INVALID_ARG: return "HH_ERR_INVALID_ARG";
    case HH_ERR_UNSUPPORTED: return "HH_ERR_UNSUPPORTED";
    case HH_ERR_ALIGNMENT: return "HH_ERR_ALIGNMENT";
    case HH_ERR_WORKSPACE: return "HH_ERR_WORKSPACE";
    case HH_ERR_CUDA: return "HH_ERR_CUDA";
    case HH_ERR_TIMEOUT: return "HH_ERR_TIMEOUT";
    default: return "HH_ERR_UNKNOWN";
  }
}

int hh_fmap_dim(int kind, int d, int padded) {
  if (d < 1) return -1;
  if (kind == HH_FMAP_HEDGEHOG || kind == HH_FMAP_HEDGEHOG_SOFTMAX) return 2 * d;
  if (kind == HH_FMAP_TAYLOR2) {
    const int dp = 1 + d + d * d;
    return padded ? (dp + 31) / 32 * 32 : dp;
  }
  return -1;
}

hh_status hh_feature_map(const hh_fmap* fmap, int dtype, const void* x, int is_key, int64_t B,
                         int H, int64_t n, void* phi_out, void* stream) {
  Problem p;
  hh_status st = make_problem(fmap, dtype, B, H, n, &p);
  if (st != HH_OK) return st;
  if (B * H * n == 0) return HH_OK;
  if (!x || !phi_out) return HH_ERR_INVALID_ARG;
  const void* W = is_key && p.Wk ? p.Wk : p.Wq;
  const float* b = is_key && p.Wk ? p.bk : p.bq;
  if ((st = check_ptrs_aligned({x, phi_out, W, b})) != HH_OK) return st;
  if (!device_ok()) return HH_ERR_UNSUPPORTED;
  if (fmap_tc_supported(p))
    return cuda_status(
        launch_fmap_tc(p, x, is_key, phi_out, nullptr, nullptr, (cudaStream_t)stream));
  return cuda_status(launch_fmap_simt(p, x, is_key, phi_out, nullptr, (cudaStream_t)stream));
}

// Workspace of the prefill (with or without an initial state).
static size_t fwd_ws_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n,
                           bool from_state) {
  Problem p;
  if (make_problem(fmap, dtype, B, H, n, &p) != HH_OK) return 0;
  if (B * H * n == 0) return 0;
  p.has_init = from_state;
  const TcPlan pl = plan_prefill_tc(p);
  if (!pl.supported) return 0;
  // softmax map: the q and k row offsets follow the segment states
  return align256(pl.ws_bytes) + (p.softmax ? 2 * softmax_off_bytes(p) : 0);
}

size_t hh_fwd_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n,
                              int chunk) {
  (void)chunk;
  return fwd_ws_bytes(fmap, dtype, B, H, n, false);
}

size_t hh_fwd_from_state_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H,
                                         int64_t n, int chunk) {
  (void)chunk;
  return fwd_ws_bytes(fmap, dtype, B, H, n, true);
}

hh_status hh_fwd_plan(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n, int chunk,
                      int* segments, int* launches) {
  Problem p;
  hh_status st = make_problem(fmap, dtype, B, H, n, &p);
  if (st != HH_OK) return st;
  if (chunk != 0 && chunk != 64 && chunk != 128) return HH_ERR_UNSUPPORTED;
  int seg = 1, lau = (B * H * n > 0) ? 1 : 0;
  if (lau) {
    const TcPlan pl = plan_prefill_tc(p);
    if (pl.supported) {
      seg = pl.P;
      lau = pl.launches;
    }
  }
  if (segments) *segments = seg;
  if (launches) *launches = lau;
  return HH_OK;
}

// Shared body of the prefill entry points; S0 / z0 null = start from zero.
static hh_status fwd_impl(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                          const void* v, int64_t B, int H, int64_t n, int chunk, const float* S0,
                          const float* z0, void* y, float* S_out, float* z_out, void* workspace,
                          size_t ws_bytes, int* dev_status, void* stream) {
  Problem p;
  hh_status st = fwd_check_args(fmap, dtype, q, k, v, B, H, n, chunk, S0, z0, y, S_out, z_out,
                                workspace, dev_status, &p);
  if (st != HH_OK) return st;
  if (B == 0) return HH_OK;
  const bool from_state = S0 != nullptr;
  const size_t need = fwd_ws_bytes(fmap, dtype, B, H, n, from_state);
  if (need > 0 && (!workspace || ws_bytes < need)) return HH_ERR_WORKSPACE;
  if (!device_ok()) return HH_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t s_bytes = sizeof(float) * B * H * p.dpp * p.d, z_bytes = sizeof(float) * B * H * p.dpp;
  if (n == 0) {
    // no tokens: the state is the initial one (or the empty sum)
    if (S_out) {
      cudaError_t e;
      if (from_state) {
        e = S_out == S0 ? cudaSuccess
                        : cudaMemcpyAsync(S_out, S0, s_bytes, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess && z_out != z0)
          e = cudaMemcpyAsync(z_out, z0, z_bytes, cudaMemcpyDeviceToDevice, s);
      } else {
        e = cudaMemsetAsync(S_out, 0, s_bytes, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(z_out, 0, z_bytes, s);
      }
      return cuda_status(e);
    }
    return HH_OK;
  }
  p.has_init = from_state;
  p.S0 = S0;
  p.z0 = z0;
  const TcPlan pl = plan_prefill_tc(p);
  if (pl.supported) {
    // the shared-map d = 64 output pass forms the softmax-map offsets itself;
    // every other output pass, and the segment-state pass, reads them
    if (p.softmax && !(p.d == 64 && !p.Wk && pl.P == 1)) {
      // per-row offsets of the softmax map, from the feature-map kernel
      char* ob = (char*)workspace + align256(pl.ws_bytes);
      float2* offq = (float2*)ob;
      float2* offk = (float2*)(ob + softmax_off_bytes(p));
      cudaError_t e = launch_fmap_tc_qk(p, q, k, nullptr, nullptr, offq, offk, dev_status, s);
      if (e != cudaSuccess) return cuda_status(e);
      p.offq = offq;
      p.offk = offk;
    }
    return cuda_status(launch_prefill_tc(p, pl, q, k, v, y, S_out, z_out, workspace, dev_status, s));
  }
  return cuda_status(launch_prefill_simt(p, q, k, v, y, S_out, z_out, s));
}

hh_status hh_linattn_fwd_causal(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                                const void* v, int64_t B, int H, int64_t n, int chunk, void* y,
                                float* S_out, float* z_out, void* workspace, size_t ws_bytes,
                                int* dev_status, void* stream) {
  return fwd_impl(fmap, dtype, q, k, v, B, H, n, chunk, nullptr, nullptr, y, S_out, z_out,
                  workspace, ws_bytes, dev_status, stream);
}

hh_status hh_linattn_fwd_causal_from_state(const hh_fmap* fmap, int dtype, const void* q,
                                           const void* k, const void* v, int64_t B, int H,
                                           int64_t n, int chunk, const float* S0,
                                           const float* z0, void* y, float* S_out, float* z_out,
                                           void* workspace, size_t ws_bytes, int* dev_status,
                                           void* stream) {
  if (B > 0 && (!S0 || !z0)) return HH_ERR_INVALID_ARG;
  return fwd_impl(fmap, dtype, q, k, v, B, H, n, chunk, S0, z0, y, S_out, z_out, workspace,
                  ws_bytes, dev_status, stream);
}

hh_status hh_linattn_decode_step(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                                 const void* v, int64_t B, int H, float* S, float* z, void* y,
                                 void* stream) {
  Problem p;
  hh_status st = make_problem(fmap, dtype, B, H, 1, &p);
  if (st != HH_OK) return st;
  if (B == 0) return HH_OK;
  if (!q || !k || !v || !S || !z || !y) return HH_ERR_INVALID_ARG;
  if ((st = check_ptrs_aligned({q, k, v, S, z, y, p.Wq, p.bq, p.Wk, p.bk})) != HH_OK) return st;
  if (!device_ok()) return HH_ERR_UNSUPPORTED;
  return cuda_status(launch_decode(p, q, k, v, S, z, y, (cudaStream_t)stream));
}

size_t hh_loss_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n) {
  Problem p;
  if (make_problem(fmap, dtype, B, H, n, &p) != HH_OK) return 0;
  if (B * H * n == 0) return 0;
  return loss_ws(p);
}

// Shared body of hh_mimicry_loss and hh_mimicry_stats.
static hh_status mimicry_loss_impl(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                                   int64_t B, int H, int64_t n, float* loss_rows,
                                   float* loss_head_sum, float4* rows4, void* workspace,
                                   size_t ws_bytes, int* dev_status, void* stream) {
  Problem p;
  hh_status st = make_problem(fmap, dtype, B, H, n, &p);
  if (st != HH_OK) return st;
  if (B == 0) return HH_OK;
  if (!loss_head_sum && !rows4) return HH_ERR_INVALID_ARG;
  if (n > 0 && (!q || !k)) return HH_ERR_INVALID_ARG;
  if ((st = check_ptrs_aligned({q, k, loss_rows, loss_head_sum, rows4, p.Wq, p.bq, p.Wk, p.bk,
                                workspace})) != HH_OK)
    return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return HH_ERR_ALIGNMENT;
  const size_t need = hh_loss_workspace_bytes(fmap, dtype, B, H, n);
  if (need > 0 && (!workspace || ws_bytes < need)) return HH_ERR_WORKSPACE;
  if (!device_ok()) return HH_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (n == 0)
    return loss_head_sum ? cuda_status(cudaMemsetAsync(loss_head_sum, 0, sizeof(float) * B * H, s))
                         : HH_OK;
  char* ws = (char*)workspace;
  const size_t phi_bytes = align256((size_t)B * H * n * p.dpp * elem_size(dtype));
  void* phq = ws;
  void* phk = ws + phi_bytes;
  float* partial = (float*)(ws + 2 * phi_bytes);
  float* head = loss_head_sum ? loss_head_sum : partial + (size_t)B * H * ceil_div(n, 64);
  if (fmap_tc_supported(p)) {
    // the Hedgehog map: phi(k) from the feature-map kernel (each key tile is
    // read by every later query tile), phi(q) formed inside the loss kernel;
    // the softmax map: both from the feature-map kernel
    cudaError_t e = p.softmax
                        ? launch_fmap_tc_qk(p, q, k, phq, phk, nullptr, nullptr, dev_status, s)
                        : launch_fmap_tc(p, k, 1, phk, nullptr, dev_status, s);
    if (e == cudaSuccess)
      e = launch_loss_tc(p, q, k, p.softmax ? phq : nullptr, phk, loss_rows, partial, head, nullptr,
                         rows4, nullptr, dev_status, s);
    return cuda_status(e);
  }
  cudaError_t e = launch_fmap_simt(p, q, 0, phq, nullptr, s);
  if (e == cudaSuccess) e = launch_fmap_simt(p, k, 1, phk, nullptr, s);
  if (e == cudaSuccess)
    e = launch_loss_simt(p, q, k, phq, phk, loss_rows, partial, loss_simt_tile(), head, rows4, s);
  return cuda_status(e);
}

hh_status hh_mimicry_loss(const hh_fmap* fmap, int dtype, const void* q, const void* k, int64_t B,
                          int H, int64_t n, float* loss_rows, float* loss_head_sum,
                          void* workspace, size_t ws_bytes, int* dev_status, void* stream) {
  if (B > 0 && !loss_head_sum) return HH_ERR_INVALID_ARG;
  return mimicry_loss_impl(fmap, dtype, q, k, B, H, n, loss_rows, loss_head_sum, nullptr,
                           workspace, ws_bytes, dev_status, stream);
}

hh_status hh_mimicry_stats(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                           int64_t B, int H, int64_t n, float* stats_rows, void* workspace,
                           size_t ws_bytes, int* dev_status, void* stream) {
  if (B > 0 && n > 0 && !stats_rows) return HH_ERR_INVALID_ARG;
  return mimicry_loss_impl(fmap, dtype, q, k, B, H, n, nullptr, nullptr, (float4*)stats_rows,
                           workspace, ws_bytes, dev_status, stream);
}

// Workspace of hh_mimicry_loss_grad.
//   tensor-core path (bf16, d in {64, 128}): phi(q) | phi(k) | row stats
//     [U][NT*128] (c_i, 1/A_i) | phi(k) column sums per tile [U][NT][2d] |
//     per-CTA dW, db shares [2][U][NT][d*d + d] | the causal 128 x 128 tiles
//     of g in bf16 [U][NT (NT + 1) / 2][128][128]
//   CUDA-core path: phi(q) | phi(k) | row stats [U][n][3] | dL/dh(q) | dL/dh(k)
struct GradWs {
  size_t phi, stats, a, b, c, g, total;
};
static GradWs loss_grad_ws(const Problem& p) {
  GradWs w;
  const size_t U = (size_t)p.B * p.H;
  const size_t NT = (size_t)ceil_div(p.n, 128);
  w.phi = align256(U * p.n * p.dpp * elem_size(p.dtype));
  if (loss_grad_tc_shape(p)) {
    w.stats = align256(U * NT * 128 * 2 * sizeof(float));
    w.a = align256(U * NT * 2 * p.d * sizeof(float));   // column sums of phi(k) per tile
    w.b = 0;
    w.c = align256(loss_grad_tc_partial_floats(p) * sizeof(float));
    w.g = align256(loss_grad_tc_g_bytes(p));
  } else {
    w.stats = align256(U * p.n * 3 * sizeof(float));
    w.a = w.b = align256(U * p.n * p.d * sizeof(float));
    w.c = w.g = 0;
  }
  w.total = 2 * w.phi + w.stats + w.a + w.b + w.c + w.g;
  return w;
}

size_t hh_loss_grad_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n) {
  Problem p;
  if (make_problem(fmap, dtype, B, H, n, &p) != HH_OK) return 0;
  if (p.kind != HH_FMAP_HEDGEHOG || B * H * n == 0) return 0;
  return loss_grad_ws(p).total;
}

size_t hh_loss_grad_workspace_bytes_min(const hh_fmap* fmap, int dtype, int64_t B, int H,
                                        int64_t n) {
  Problem p;
  if (make_problem(fmap, dtype, B, H, n, &p) != HH_OK) return 0;
  if (p.kind != HH_FMAP_HEDGEHOG || B * H * n == 0) return 0;
  const GradWs w = loss_grad_ws(p);
  return w.total - w.g;   // the g tiles come last
}

hh_status hh_mimicry_loss_grad(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                               int64_t B, int H, int64_t n, float* dWq, float* dbq, float* dWk,
                               float* dbk, void* workspace, size_t ws_bytes, int* dev_status,
                               void* stream) {
  Problem p;
  hh_status st = make_problem(fmap, dtype, B, H, n, &p);
  if (st != HH_OK) return st;
  if (p.kind != HH_FMAP_HEDGEHOG || p.d % 8 != 0 || p.d > 128) return HH_ERR_UNSUPPORTED;
  const bool separate = fmap->Wk && fmap->Wk != fmap->Wq;
  const bool bias = !p.softmax;   // the softmax map has no bias, so no db
  if (!dWq || (bias && !dbq) || (separate && (!dWk || (bias && !dbk)))) return HH_ERR_INVALID_ARG;
  if (!separate) dWk = dbk = nullptr;
  if (!bias) dbq = dbk = nullptr;
  if (B * n > 0 && (!q || !k)) return HH_ERR_INVALID_ARG;
  if ((st = check_ptrs_aligned({q, k, dWq, dbq, dWk, dbk, p.Wq, p.bq, p.Wk, p.bk, workspace})) !=
      HH_OK)
    return st;
  if (dev_status && ((uintptr_t)dev_status & 3u)) return HH_ERR_ALIGNMENT;
  const size_t need = hh_loss_grad_workspace_bytes_min(fmap, dtype, B, H, n);
  if (need > 0 && (!workspace || ws_bytes < need)) return HH_ERR_WORKSPACE;
  if (!device_ok()) return HH_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t wbytes = sizeof(float) * H * p.d * p.d, bbytes = sizeof(float) * H * p.d;
  if (B * n == 0) {   // empty sum: zero gradient
    cudaError_t e = cudaMemsetAsync(dWq, 0, wbytes, s);
    if (e == cudaSuccess && dbq) e = cudaMemsetAsync(dbq, 0, bbytes, s);
    if (e == cudaSuccess && dWk) e = cudaMemsetAsync(dWk, 0, wbytes, s);
    if (e == cudaSuccess && dbk) e = cudaMemsetAsync(dbk, 0, bbytes, s);
    return cuda_status(e);
  }
  const bool tc = loss_grad_tc_shape(p);
  if (tc ? !loss_grad_tc_supported(p)
         : loss_grad_smem_bytes(p) > (size_t)device_max_smem_optin())
    return HH_ERR_UNSUPPORTED;
  const GradWs w = loss_grad_ws(p);
  char* ws = (char*)workspace;
  void* phq = ws;
  void* phk = ws + w.phi;
  float* stats = (float*)(ws + 2 * w.phi);
  float* wa = (float*)(ws + 2 * w.phi + w.stats);
  float* wb = (float*)(ws + 2 * w.phi + w.stats + w.a);
  float* wc = (float*)(ws + 2 * w.phi + w.stats + w.a + w.b);
  // the stored tiles of g when the workspace has room for them
  void* wg = ws_bytes >= w.total && w.g > 0 ? ws + 2 * w.phi + w.stats + w.a + w.b + w.c : nullptr;
  cudaError_t e;
  if (fmap_tc_supported(p)) {
    e = launch_fmap_tc_qk(p, q, k, phq, phk, nullptr, nullptr, dev_status, s);
  } else {
    e = launch_fmap_simt(p, q, 0, phq, nullptr, s);
    if (e == cudaSuccess) e = launch_fmap_simt(p, k, 1, phk, nullptr, s);
  }
  if (tc) {
    // wa: phi(k) column sums, wc: dW, db shares, wg: G tiles
    // the row statistics (c_i, 1/A_i) alone: no loss is returned
    if (e == cudaSuccess)
      e = launch_loss_tc(p, q, k, phq, phk, nullptr, nullptr, nullptr, stats, nullptr, wa,
                         dev_status, s);
    if (e == cudaSuccess)
      e = launch_loss_grad_tc(p, q, k, phq, phk, stats, wc, wg, dWq, dbq, dWk, dbk, dev_status,
                              s);
  } else if (e == cudaSuccess) {
    // wa, wb: dL/dh of the query and key rows
    e = launch_loss_grad(p, q, k, phq, phk, stats, wa, wb, dWq, dbq, dWk, dbk, s);
  }
  return cuda_status(e);
}

}  // extern "C"
