// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hh.h"

namespace hh {

// A validated problem description handed from the ABI layer to launchers.
struct Problem {
  int kind;        // HH_FMAP_HEDGEHOG (also for the softmax map) or HH_FMAP_TAYLOR2
  int dtype;       // hh_dtype
  int d;           // head dim
  int dp;          // unpadded feature dim
  int dpp;         // padded feature dim (row length of phi and S)
  int64_t B;
  int H;
  int G = 1;       // query heads per key/value head (grouped-query attention)
  int seq_major = 0;  // q, k, v, y are [B][n][H][d] (else [B][H][n][d])
  int64_t n;
  const void* Wq;
  const float* bq;
  const void* Wk;
  const float* bk;
  // Softmax-over-features map: phi = [exp(h - c+); exp(-h - c-)] with the
  // per-row offsets c+- = logsumexp(+-h) (bias null).  Kernels that build phi
  // from h = x W read the offsets, in log2 units (c * log2 e), from offq /
  // offk, set once they have been computed: pairs [U][off_stride(n)] (rows
  // padded to whole 128-row tiles, so a tile's offsets start 16-byte aligned).
  // The shared-map d = 64 output pass forms its own and reads neither.
  bool softmax = false;
  const float2* offq = nullptr;
  const float2* offk = nullptr;
  // Continuation: the prefill starts from this state (public layout, as the
  // S_out / z_out of a prefill or the state of decode) instead of zero.
  // has_init sizes the workspace; S0 / z0 are set for the launch.
  bool has_init = false;
  const float* S0 = nullptr;
  const float* z0 = nullptr;
};

// ---- element access in float32 for either storage type -------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 1/sqrt(2) rounded to float32: the Taylor map's pair scale.
constexpr float kInvSqrt2 = 0.70710678118654752440f;

inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
// Key/value unit (batch * Hkv + key/value head) of query unit u = b * H + h
// when G query heads share one key/value head.
__host__ __device__ __forceinline__ int64_t kv_unit(int64_t u, int H, int G) {
  return G == 1 ? u : (u / H) * (H / G) + (u % H) / G;
}

// Row of token t of head unit u (= b * H + h) in a [B][H][n][.] tensor, or in
// a [B][n][H][.] one (seq_major); multiply by the row length for the offset.
__host__ __device__ __forceinline__ int64_t row_index(int64_t u, int64_t t, int H, int64_t n,
                                                      int seq_major) {
  return seq_major ? ((u / H) * n + t) * H + u % H : u * n + t;
}

// The same for head h of batch b, without a division.
__host__ __device__ __forceinline__ int64_t row_of(int b, int h, int64_t t, int H, int64_t n,
                                                   int seq_major) {
  return seq_major ? ((int64_t)b * n + t) * H + h : ((int64_t)b * H + h) * n + t;
}

// Row stride of the softmax-map offset arrays.
inline int64_t off_stride(int64_t n) { return (n + 127) / 128 * 128; }

// Host-side argument checks shared by the prefill entry points (pointers,
// alignment, shapes; the workspace size is not checked).  No device work.
hh_status fwd_check_args(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                         const void* v, int64_t B, int H, int64_t n, int chunk, const float* S0,
                         const float* z0, const void* y, const float* S_out, const float* z_out,
                         const void* workspace, const int* dev_status, Problem* p);
// Whether the current device runs this library's kernels (sm_103).
bool device_is_supported();

// Cached device attributes (the only state the library keeps).
int device_sm_count();
int device_max_smem_optin();
// Soft wait limit for device-side bounded waits, from HH_WAIT_SOFT_LIMIT_NS.
uint64_t wait_soft_limit_ns();
// Whether kernels that support it are launched as programmatic dependents
// (HH_PDL=0 turns it off).
bool pdl_enabled();

// Launch as a programmatic dependent of the previous kernel on the stream: its
// CTAs may be scheduled, and run up to griddepcontrol.wait, while that kernel
// finishes.  Only kernels that execute griddepcontrol.wait before their first
// global-memory access (read or write) may be launched this way.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- launchers (return cudaSuccess or the launch error) ------------------
// SIMT kernels: float32 arithmetic, any supported d; T = float or bf16.
// phi (nullable): [U][n][dpp]; off (nullable, softmax map only): per-row
// offsets in log2 units, [U][off_stride(n)].
cudaError_t launch_fmap_simt(const Problem& p, const void* x, int is_key, void* phi,
                             float2* off, cudaStream_t s);
cudaError_t launch_prefill_simt(const Problem& p, const void* q, const void* k, const void* v,
                                void* y, float* S_out, float* z_out, cudaStream_t s);
// rows4 (nullable): per-row (CE, KL, H(p), H(w)).
cudaError_t launch_loss_simt(const Problem& p, const void* q, const void* k, const void* phq,
                             const void* phk, float* loss_rows, float* partial, int tile,
                             float* head_sum, float4* rows4, cudaStream_t s);
int loss_simt_tile();

// Tensor-core (tcgen05) chunked prefill for bf16.
struct TcPlan {
  bool supported = false;
  int NT = 0;        // 128-token tiles per sequence
  int P = 1;         // segments per sequence
  int L = 1;         // tiles per segment
  int M = 1;         // state-pass pieces per segment (one CTA each)
  int launches = 1;  // kernel launches per call
  size_t ws_bytes = 0;
  size_t raw_offset = 0;    // M > 1: byte offset of the piece states in the workspace
  size_t init_offset = 0;   // continuation: byte offset of the initial state in the workspace
};
TcPlan plan_prefill_tc(const Problem& p);
// Floats of one segment state in the prefill workspace: S then z.  The Taylor
// kernels keep 160 packed features (taylor_pack.cuh) instead of 288.
inline int64_t ws_segment_floats(const Problem& p) {
  return p.kind == HH_FMAP_TAYLOR2 ? (int64_t)160 * 16 + 160 : (int64_t)p.dpp * p.d + p.dpp;
}
cudaError_t launch_prefill_tc(const Problem& p, const TcPlan& pl, const void* q, const void* k,
                              const void* v, void* y, float* S_out, float* z_out, void* ws,
                              int* dev_status, cudaStream_t s);

// Segment-state pass (P > 1): per segment but the last, sum phi(k)^T v and
// sum phi(k) into the workspace.
cudaError_t launch_state_tc(const Problem& p, const TcPlan& pl, const void* k, const void* v,
                            void* ws, int* dev_status, cudaStream_t s);

// Output pass of the d = 64 Hedgehog prefill with two tiles in flight per CTA.
// init: the initial state in workspace layout (continuation) or null.
cudaError_t launch_prefill_out_d64(const Problem& p, const TcPlan& pl, const void* q,
                                   const void* k, const void* v, void* y, float* S_out,
                                   float* z_out, const void* ws, const float* init,
                                   int* dev_status, cudaStream_t s);

// Output pass of the d = 128 Hedgehog prefill (shared map): warp-specialised,
// phi(K) built with the hidden units on the TMEM lanes.
cudaError_t launch_prefill_out_d128(const Problem& p, const TcPlan& pl, const void* q,
                                    const void* k, const void* v, void* y, float* S_out,
                                    float* z_out, const void* ws, const float* init,
                                    int* dev_status, cudaStream_t s);

// Output pass of the Taylor (d = 16) prefill: scores from the closed form
// 1 + s + s^2/2 with s = q . k, state contractions on the features.
cudaError_t launch_prefill_out_taylor(const Problem& p, const TcPlan& pl, const void* q,
                                      const void* k, const void* v, void* y, float* S_out,
                                      float* z_out, const void* ws, const float* init,
                                      int* dev_status, cudaStream_t s);

// Gradient of the summed mimicry loss w.r.t. the Hedgehog map (CUDA cores,
// fp32 arithmetic): phi(q), phi(k) precomputed; stats [U][n][3]; dh [U][n][d].
size_t loss_grad_smem_bytes(const Problem& p);
cudaError_t launch_loss_grad(const Problem& p, const void* q, const void* k, const void* phq,
                             const void* phk, float* stats, float* dhq, float* dhk, float* dWq,
                             float* dbq, float* dWk, float* dbk, cudaStream_t s);

// Tensor-core (tcgen05) feature map and mimicry loss for bf16 Hedgehog d in {64, 128}.
bool fmap_tc_supported(const Problem& p);
cudaError_t launch_fmap_tc(const Problem& p, const void* x, int is_key, void* phi, float2* off,
                           int* dev_status, cudaStream_t s);
// Queries and keys in one launch (outputs nullable as above).
cudaError_t launch_fmap_tc_qk(const Problem& p, const void* q, const void* k, void* phq,
                              void* phk, float2* offq, float2* offk, int* dev_status,
                              cudaStream_t s);
// stats (nullable): [U][NT * 128] pairs (c_i, 1 / A_i) with c_i = m_i + log2 Z_i,
// so that the target weight is p_ij = 2^(s_ij log2(e) / sqrt(d) - c_i).
// rows4 (nullable): per-row (CE, KL, H(p), H(w)).  partial null (and
// loss_rows, head_sum, rows4 null): the row statistics alone, without the
// loss and its log a per pair; then colsum ([U][NT][2d] floats) receives the
// per-tile column sums of phi(k) that give A_i's off-diagonal part.
cudaError_t launch_loss_tc(const Problem& p, const void* q, const void* k, const void* phq,
                           const void* phk, float* loss_rows, float* partial, float* head_sum,
                           float* stats, float4* rows4, float* colsum, int* dev_status,
                           cudaStream_t s);
int loss_tc_tile();

// Tensor-core gradient of the summed mimicry loss for bf16 Hedgehog d in
// {64, 128}: from phi(q), phi(k) and the loss kernel's row stats, per-CTA
// dW, db shares in `part` (loss_grad_tc_partial_floats floats), then summed
// per head in a fixed order into dWq, dbq (and dWk, dbk for a separate key map).
// gbuf (loss_grad_tc_g_bytes, or null to form g on both sides): the causal
// tiles of G, written by the query side and read back by the key side.
bool loss_grad_tc_shape(const Problem& p);
bool loss_grad_tc_supported(const Problem& p);
size_t loss_grad_tc_smem_bytes(const Problem& p);
size_t loss_grad_tc_partial_floats(const Problem& p);
size_t loss_grad_tc_g_bytes(const Problem& p);
cudaError_t launch_loss_grad_tc(const Problem& p, const void* q, const void* k, const void* phq,
                                const void* phk, const float* stats, float* part, void* gbuf,
                                float* dWq, float* dbq, float* dWk, float* dbk, int* dev_status,
                                cudaStream_t s);
// dW[h] = sum x^T dh, db[h] = sum dh over the batch (CUDA cores); with one
// shared map (dWk null) both sides go into dWq, dbq.
cudaError_t launch_grad_reduce(const Problem& p, const void* q, const void* k, const float* dhq,
                               const float* dhk, float* dWq, float* dbq, float* dWk, float* dbk,
                               cudaStream_t s);

// Decode step (SIMT, HBM-streaming).
cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v,
                          float* S, float* z, void* y, cudaStream_t s);

}  // namespace hh
