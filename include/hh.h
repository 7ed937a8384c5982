/*
 * hh.h -- C ABI of the Hedgehog / Taylor causal linear-attention library
 * for NVIDIA GB300 (sm_103a).
 *
 * The operations follow "The Hedgehog & the Porcupine: Expressive Linear
 * Attentions with Softmax Mimicry" (summary of arXiv 2402.04347):
 *
 *   feature maps   phi_hh(x) = [exp(xW + b); exp(-(xW + b))]          (R^d -> R^2d)
 *                  ("The Hedgehog MLP Feature Map", Choices 1 and 3)
 *                  phi_t2(x) = [1, x, (x_i x_j / sqrt 2)_{i,j}]       (R^d -> R^{1+d+d^2})
 *                  ("The Taylor Exponential as a Bridge Result")
 *   causal output  y_i = sum_{j<=i} (phi(q_i).phi(k_j)) v_j / sum_{j<=i} phi(q_i).phi(k_j)
 *                  ("2. Context and Motivation", paper Eq. 2; running sums S, z
 *                  in "Complexity Analysis")
 *   mimicry loss   L_i = -sum_{j<=i} softmax_j(q_i.k_j / sqrt d) log(a_ij / sum_{m<=i} a_im),
 *                  a_ij = phi(q_i).phi(k_j)
 *                  ("The Attention Weight Distillation Loss", paper Eq. 4)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Ownership: the caller allocates and owns every buffer.  The library
 *   allocates no device or host memory in any call and keeps no state other
 *   than cached device attributes.
 * - Pointers: q, k, v, x, y, phi, W, b, S, z, loss buffers and the workspace
 *   are DEVICE pointers on the current CUDA device and must be 16-byte
 *   aligned (HH_ERR_ALIGNMENT otherwise).  ``stream`` is a cudaStream_t
 *   (NULL = legacy default stream).
 * - Asynchrony: every call validates its arguments on the host, enqueues its
 *   kernels on ``stream`` and returns.  HH_OK means "validated and
 *   enqueued"; a launch failure returns HH_ERR_CUDA.  Nothing is launched
 *   when validation fails.
 * - Layouts (row-major, contiguous):
 *     q, k, v, y, x    [B][H][n][d]         (decode: [B][H][d])
 *     W                [H][d][d]            W[h][k][l]: input k -> output l, h = x W + b
 *     b                [H][d]  float32      (NULL = zero bias)
 *     phi              [B][H][n][d'p]
 *     S                [B][H][d'p][d] float32,  z  [B][H][d'p] float32
 *     loss_rows        [B][H][n] float32,   loss_head_sum [B][H] float32
 *   d'p is hh_fmap_dim(kind, d, 1): 2d for Hedgehog, 1+d+d^2 rounded up
 *   to a multiple of 32 for Taylor (273 -> 288 at d = 16).  Padding
 *   features are identically zero.
 * - Types: HH_F32 means q, k, v, x, W, y, phi are float32; HH_BF16 means
 *   they are bfloat16 (round-to-nearest-even outputs).  b, S, z and loss
 *   buffers are always float32.  Arithmetic is float32 (tensor-core
 *   operands in bfloat16 for HH_BF16).
 * - Supported shapes: Hedgehog d in {64, 128}; Taylor d = 16; any
 *   HH_F32 call additionally accepts Hedgehog 1 <= d <= 128 and Taylor
 *   1 <= d <= 16.  B, n >= 0 (an empty problem launches nothing), H >= 1.
 * - Numerical domain: the exponential is not clamped; |xW + b| beyond ~80
 *   overflows float32 and produces inf/NaN (outside the supported domain).
 * - Device-detected problems: kernels that wait on asynchronous copies or
 *   tensor-core operations bound every wait in time.  When a wait passes
 *   its soft limit the kernel stores HH_ERR_TIMEOUT into ``*dev_status``
 *   (when that pointer is non-NULL) and keeps waiting up to a hard limit;
 *   past the hard limit it abandons the work, releases its tensor memory
 *   and returns.  The caller reads ``*dev_status`` after synchronising.
 *   The environment variable HH_WAIT_SOFT_LIMIT_NS overrides the soft
 *   limit (default 1e9 ns) for testing.
 * - No C++ exception crosses this interface.
 */
#ifndef HH_H_
#define HH_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HH_API __attribute__((visibility("default")))
#else
#define HH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HH_OK = 0,
  HH_ERR_INVALID_ARG = 1,  /* null pointer, negative size, overflow, unknown enum  */
  HH_ERR_UNSUPPORTED = 2,  /* valid but not implemented: head dim, chunk, device   */
  HH_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned                     */
  HH_ERR_WORKSPACE = 4,    /* workspace missing or smaller than the queried size   */
  HH_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed                    */
  HH_ERR_TIMEOUT = 6       /* device-side: a bounded wait passed its limit         */
} hh_status;

typedef enum { HH_F32 = 0, HH_BF16 = 1 } hh_dtype;

/* Layout of the [B] x [H] x [n] x [d] tensors q, k, v, y of the prefill, loss,
 * statistics and gradient calls and x of hh_feature_map (d contiguous in both):
 *   HH_LAYOUT_BHND  [B][H][n][d]
 *   HH_LAYOUT_BNHD  [B][n][H][d]  (the head-interleaved output of a fused
 *                                  projection, used without a transpose)
 * Under grouped key/value heads k, v are [B][Hkv][n][d] / [B][n][Hkv][d].
 * States, per-row outputs (loss rows, statistics) and phi from
 * hh_feature_map stay [B][H][...]. */
typedef enum { HH_LAYOUT_BHND = 0, HH_LAYOUT_BNHD = 1 } hh_layout;

/* HH_FMAP_HEDGEHOG: [exp(xW + b); exp(-(xW + b))] ("The Hedgehog MLP
 *   Feature Map", Choices 1 and 3).
 * HH_FMAP_TAYLOR2: [1, x, vec(x x^T) / sqrt 2] ("The Taylor Exponential as a
 *   Bridge Result").
 * HH_FMAP_HEDGEHOG_SOFTMAX: [softmax(xW); softmax(-xW)], each half a softmax
 *   over the d learned directions, no bias (Choice 4, Eq. 5, with the
 *   negation block of Choice 3 normalised the same way).  bq and bk must be
 *   NULL.  Every call that takes a Hedgehog map takes this one except
 *   hh_mimicry_loss_grad. */
typedef enum {
  HH_FMAP_HEDGEHOG = 0,
  HH_FMAP_TAYLOR2 = 1,
  HH_FMAP_HEDGEHOG_SOFTMAX = 2
} hh_fmap_kind;

/* A per-layer feature map.  For the Hedgehog kinds, Wq/bq map the queries and
 * Wk/bk the keys; Wk == NULL means the keys share Wq/bq (one map per head used
 * for both queries and keys, as the pages describe).  Taylor ignores W and b. */
typedef struct {
  int32_t kind;        /* hh_fmap_kind                                      */
  int32_t d;           /* head dimension                                    */
  const void* Wq;      /* [H][d][d] in the call's dtype (Hedgehog only)     */
  const float* bq;     /* [H][d] float32 or NULL                            */
  const void* Wk;      /* [H][d][d] or NULL (shared with Wq)                */
  const float* bk;     /* [H][d] or NULL; ignored when Wk is NULL           */
  int32_t kv_heads;    /* key/value heads Hkv: 0 or H for one per query head;
                        * else H is a multiple of Hkv and query head h reads
                        * key/value head h / (H / Hkv) (grouped-query
                        * attention): k, v are [B][Hkv][n][d] ([B][Hkv][d] for
                        * decode).  Maps, states and outputs stay per query
                        * head.                                              */
  int32_t layout;      /* hh_layout of q, k, v, y (0: [B][H][n][d])           */
} hh_fmap;

/* Library version, major*10000 + minor*100 + patch. */
HH_API int hh_version(void);

/* Human-readable name of a status code (static string, never NULL). */
HH_API const char* hh_status_str(int status);

/* Feature dimension d' of a map: 2d (Hedgehog kinds) or 1+d+d^2 (Taylor, the
 * count printed in "The Taylor Exponential as a Bridge Result").  With
 * padded != 0 the Taylor count is rounded up to a multiple of 32.  Returns
 * -1 for an unknown kind or d < 1. */
HH_API int hh_fmap_dim(int kind, int d, int padded);

/* phi(x) for every row of x.
 * Source: "The Hedgehog MLP Feature Map", Choices 1 and 3 (Hedgehog);
 * "The Taylor Exponential as a Bridge Result" (Taylor).
 * x: [B][H][n][d] (dtype); is_key selects Wk/bk instead of Wq/bq;
 * phi_out: [B][H][n][d'p] (dtype), fully overwritten including padding.
 * Hedgehog output order: feature l < d is exp(h_l), feature d + l is exp(-h_l);
 * the softmax kind divides each half by its sum over l. */
HH_API hh_status hh_feature_map(const hh_fmap* fmap, int dtype, const void* x, int is_key,
                         int64_t B, int H, int64_t n, void* phi_out, void* stream);

/* Bytes of device workspace hh_linattn_fwd_causal needs for this problem
 * on the current device (0 when none).  Returns 0 for invalid arguments. */
HH_API size_t hh_fwd_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n,
                              int chunk);

/* Planning query for hh_linattn_fwd_causal on the current device: the
 * number of sequence segments each (batch, head) is split into and the
 * number of kernel launches one call makes.  Either output may be NULL. */
HH_API hh_status hh_fwd_plan(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n,
                             int chunk, int* segments, int* launches);

/* Causal linear attention over whole sequences (chunked prefill).
 * Source: "The Hedgehog & the Porcupine: Expressive Linear Attentions with
 * Softmax Mimicry", section "2. Context and Motivation" (the linear-attention
 * equation for y_i, paper Eq. 2); "Complexity Analysis" for the
 * running sums S_i = sum_{j<=i} phi(k_j)^T v_j and z_i = sum_{j<=i} phi(k_j).
 * q, k, v: [B][H][n][d] (dtype); y: [B][H][n][d] (dtype), overwritten.
 * chunk: 0 (library default), 64 or 128 -- the intra-chunk block length of
 * the chunked evaluation; the result is the same causal sum for any value.
 * S_out / z_out: NULL, or [B][H][d'p][d] / [B][H][d'p] float32 receiving the
 * state after the last token (S_n, z_n), the input of
 * hh_linattn_decode_step.  Both or neither must be given.
 * workspace: device scratch of at least hh_fwd_workspace_bytes(...) bytes
 * (may be NULL when that is 0); its contents on entry are ignored.
 * dev_status: NULL or a device int the kernels may set to HH_ERR_TIMEOUT. */
HH_API hh_status hh_linattn_fwd_causal(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                                const void* v, int64_t B, int H, int64_t n, int chunk, void* y,
                                float* S_out, float* z_out, void* workspace, size_t ws_bytes,
                                int* dev_status, void* stream);

/* hh_linattn_fwd_causal without a workspace argument.  The paper has no
 * counterpart to this entry point: it exists for callers that cannot allocate
 * device memory when they run the prefill (a plugin interface that only
 * passes its input and output buffers, a serving loop that forbids allocation
 * after start-up, a C host program without a device allocator).  Arguments
 * and results are those of hh_linattn_fwd_causal, and they are checked in the
 * same order (pointers, alignment and shapes, then the device) before the
 * size check below.
 * Scratch: a fixed 16 MiB device array inside the library, present on every
 * GPU that loads the library until the process exits.  A problem needing more
 * scratch than that (hh_fwd_workspace_bytes > 16 MiB) returns
 * HH_ERR_WORKSPACE and launches nothing.
 * First call: with CUDA's lazy module loading, the first call in a context
 * that needs scratch loads the library's device module, whose 16 MiB array is
 * then committed; that call can fail for lack of device memory
 * (HH_ERR_CUDA).  It also looks up the array's address, once per device and
 * CUDA context (a call in a new context, e.g. after cudaDeviceReset, looks it
 * up again); make it before any stream capture.  After it, no call allocates.
 * All calls share the array: calls that overlap on the GPU race and must not
 * be issued. */
HH_API hh_status hh_linattn_fwd_causal_noalloc(const hh_fmap* fmap, int dtype, const void* q,
                                               const void* k, const void* v, int64_t B, int H,
                                               int64_t n, int chunk, void* y, float* S_out,
                                               float* z_out, int* dev_status, void* stream);

/* Bytes of device workspace hh_linattn_fwd_causal_from_state needs (0 when none). */
HH_API size_t hh_fwd_from_state_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H,
                                                int64_t n, int chunk);

/* Causal prefill continuing from a given state: token t of this call sees
 * S0 + sum_{j<=t} phi(k_j)^T v_j and z0 + sum_{j<=t} phi(k_j), as if the
 * tokens that produced S0, z0 had come first.  Source: "Complexity Analysis"
 * (the running sums S and z carry all earlier tokens).
 * S0: [B][H][d'p][d] and z0: [B][H][d'p] float32 in the layout of S_out /
 * z_out (what hh_linattn_fwd_causal exports and hh_linattn_decode_step
 * updates); both required.  S_out / z_out may alias S0 / z0 (updated in
 * place).  Other arguments as hh_linattn_fwd_causal; the workspace must be at
 * least hh_fwd_from_state_workspace_bytes(...) bytes.  Taylor states are
 * folded onto the symmetric feature pairs (rows (i, j) and (j, i) enter as
 * their sum), which leaves every output unchanged. */
HH_API hh_status hh_linattn_fwd_causal_from_state(const hh_fmap* fmap, int dtype, const void* q,
                                                  const void* k, const void* v, int64_t B, int H,
                                                  int64_t n, int chunk, const float* S0,
                                                  const float* z0, void* y, float* S_out,
                                                  float* z_out, void* workspace, size_t ws_bytes,
                                                  int* dev_status, void* stream);

/* One recurrent decode step for B sequences x H heads.
 * Source: "Complexity Analysis" (running sums S and z, output
 * phi(q_t) S_t / phi(q_t).z_t); the state after the step includes token t.
 * q, k, v: [B][H][d] (dtype); S: [B][H][d'p][d] float32 and z: [B][H][d'p]
 * float32 are read and updated in place; y: [B][H][d] (dtype), overwritten.
 * Element order of every floating-point sum is fixed (deterministic). */
HH_API hh_status hh_linattn_decode_step(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                                 const void* v, int64_t B, int H, float* S, float* z, void* y,
                                 void* stream);

/* Bytes of device workspace hh_mimicry_loss and hh_mimicry_stats need (0 when none). */
HH_API size_t hh_loss_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H, int64_t n);

/* Attention-weight distillation cross-entropy (paper Eq. 4) per query.
 * Source: "The Attention Weight Distillation Loss".  Target: causal
 * softmax(q k^T / sqrt d); prediction: a_ij / sum_{m<=i} a_im with
 * a_ij = phi(q_i).phi(k_j); natural logarithm.
 * q, k: [B][H][n][d] (dtype).  loss_rows: NULL or [B][H][n] float32
 * receiving L_i; loss_head_sum: [B][H] float32 receiving sum_i L_i (summed in
 * a fixed order).  workspace: at least hh_loss_workspace_bytes(...) bytes. */
HH_API hh_status hh_mimicry_loss(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                          int64_t B, int H, int64_t n, float* loss_rows, float* loss_head_sum,
                          void* workspace, size_t ws_bytes, int* dev_status, void* stream);

/* Per-query attention statistics next to the loss, one float4 per row:
 *   [0] CE_i    the cross-entropy of hh_mimicry_loss (paper Eq. 4)
 *   [1] KL_i    KL(p_i || w_i) = CE_i - H(p_i), the divergence the HH digest
 *               (section A.3, attention distillation) names beside CE
 *   [2] H(p_i)  entropy of the causal softmax target
 *   [3] H(w_i)  entropy of the linear-attention weights w_ij = a_ij / A_i
 * (entropies as in "The Two Missing Properties as Design Specifications":
 * -sum_j w log w, natural log).
 * q, k: [B][H][n][d] (dtype); stats_rows: [B][H][n][4] float32, 16-byte
 * aligned, overwritten.  workspace: at least hh_loss_workspace_bytes(...). */
HH_API hh_status hh_mimicry_stats(const hh_fmap* fmap, int dtype, const void* q, const void* k,
                                  int64_t B, int H, int64_t n, float* stats_rows,
                                  void* workspace, size_t ws_bytes, int* dev_status,
                                  void* stream);

/* Bytes of device workspace hh_mimicry_loss_grad needs (0 when none).  For
 * bf16 at d = 64 or 128 it holds, besides O(n) per-row data, the causal
 * 128 x 128 tiles of dL/da_ij in bf16 (2 bytes per causal pair, rounded up to
 * whole tiles: about B H n^2 bytes), so that each (query, key) pair is scored
 * once: the query side writes them and the key side reads them back. */
HH_API size_t hh_loss_grad_workspace_bytes(const hh_fmap* fmap, int dtype, int64_t B, int H,
                                           int64_t n);

/* The smallest workspace hh_mimicry_loss_grad accepts (0 when none): the
 * O(n) part of hh_loss_grad_workspace_bytes without the tiles of dL/da.
 * Given at least this much but less than hh_loss_grad_workspace_bytes, the
 * call forms dL/da on both sides, the query and the key side each scoring
 * every pair (one launch instead of two; slower, same result up to
 * rounding), so that long sequences do not need about B H n^2 bytes. */
HH_API size_t hh_loss_grad_workspace_bytes_min(const hh_fmap* fmap, int dtype, int64_t B, int H,
                                               int64_t n);

/* Gradient of the summed distillation loss sum_{b,h,i} L_i (paper Eq. 4) with
 * respect to the Hedgehog feature-map parameters.  Source: "The Attention
 * Weight Distillation Loss" (only the feature maps are trained; q, k and the
 * softmax target are frozen) and "The Hedgehog MLP Feature Map", Choices 1
 * and 3.  With g_ij = 1/A_i - p_ij / a_ij (j <= i):
 *   dL/dphi(q_i) = sum_j g_ij phi(k_j), dL/dphi(k_j) = sum_i g_ij phi(q_i),
 *   dL/dh = dL/dphi_+ e^h - dL/dphi_- e^-h, dW = sum_x x^T dL/dh, db = sum_x dL/dh.
 * q, k: [B][H][n][d] (dtype).  dWq [H][d][d], dbq [H][d] float32 receive the
 * gradient w.r.t. Wq, bq summed over the batch (overwritten, not accumulated).
 * With a separate key map (fmap->Wk set and != Wq) dWk [H][d][d] and dbk [H][d]
 * receive the key-side gradient and must be non-NULL; with one shared map both
 * sides are summed into dWq, dbq and dWk, dbk are ignored.
 * Softmax map (HH_FMAP_HEDGEHOG_SOFTMAX, Choice 4, Eq. 5: no bias): each half
 * goes through the softmax Jacobian instead,
 *   dL/dh = phi_+ (dL/dphi_+ - <dL/dphi_+, phi_+>) - phi_- (dL/dphi_- - <dL/dphi_-, phi_->),
 * only dWq (and dWk) are written and dbq, dbk are ignored (may be NULL).
 * Hedgehog maps only (Taylor has no parameters: HH_ERR_UNSUPPORTED); d a
 * multiple of 8, at most 128.
 * workspace: at least hh_loss_grad_workspace_bytes(...) bytes, or at least
 * hh_loss_grad_workspace_bytes_min(...) for the slower path that stores no
 * tiles of dL/da; less than that returns HH_ERR_WORKSPACE. */
HH_API hh_status hh_mimicry_loss_grad(const hh_fmap* fmap, int dtype, const void* q,
                                      const void* k, int64_t B, int H, int64_t n, float* dWq,
                                      float* dbq, float* dWk, float* dbk, void* workspace,
                                      size_t ws_bytes, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HH_H_ */
