// Chunked causal linear attention on the 5th-generation tensor cores.
//
// "The Hedgehog & the Porcupine" summary: "2. Context and Motivation" (paper Eq. 2) defines
//   y_i = phi(q_i) sum_{j<=i} phi(k_j)^T v_j / phi(q_i) sum_{j<=i} phi(k_j),
// "Complexity Analysis" the running sums S = sum phi(k)^T v and z = sum phi(k);
// the map is "The Hedgehog MLP Feature Map" (Choices 1 and 3).  This file holds
// the planning, the scan and the generic output pass (d = 64 with a separate
// key map); the shared-map d = 64 pass is tc_prefill2.cu, the d = 128 pass
// tc_prefill128.cu, the Taylor pass tc_taylor.cu, the state passes tc_state.cu.
//
// Evaluation order (per 128-token tile t of one (batch, head) sequence segment):
//   H_Q = Q_t W, H_K = K_t W                          (tcgen05)
//   phi(Q_t) -> TMEM (bf16 pairs, the A operand of the next MMAs)
//   phi(K_t) -> shared memory (bf16, 128B-swizzled panels); z += colsum phi(K_t)
//   S_bf16 <- S (TMEM fp32 state of the tokens before tile t)
//   Sc = phi(Q_t) phi(K_t)^T;  S += phi(K_t)^T V_t     (tcgen05)
//   P = bf16(tril(Sc)), rowsum(P)
//   O = P V_t + phi(Q_t) S_bf16                         (tcgen05)
//   y = O / (rowsum(P) + phi(Q_t) . z_before)
// A 128-row tile covers two 64-token chunks with the exact causal mask, so
// the result is the same causal sum for chunk 64 or 128.
//
// Long sequences are cut into segments processed by different CTAs.  A
// state pass (tc_state.cu) writes each segment's sum of phi(k)^T v and phi(k)
// into the workspace, a scan kernel turns those into inclusive prefix sums
// (in segment order), and this output pass starts segment s from prefix s-1.
//
// Roles: thread 0 issues TMA loads and MMAs; all 8 warps run the epilogues
// (warp w owns TMEM lanes 32*(w%4).. and one half of the columns).  Every
// wait on an mbarrier is bounded in time (see tc_ptx.cuh).

#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "taylor_pack.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace hh {
namespace {

using namespace tc;

constexpr int kTile = 128;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// Hedgehog, d in {64, 128}: features [exp(h_0..h_{d-1}), exp(-h_0..-h_{d-1})].
template <int D>
struct Cfg {
  static constexpr int DP = 2 * D;           // feature dim
  static constexpr int DPP = 2 * D;          // padded feature dim (rows of S)
  static constexpr int NMB = DP / 128;       // 128-feature M blocks of S
  static constexpr int PHK_PANELS = DP / 64; // 64-feature panels of phi(K)
  static constexpr int KSTEPS_F = DP / 16;   // MMA k-steps over features
  // TMEM columns
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_Y = NMB * D;       // H_Q (fp32) -> phi(Q) (bf16 pairs)
  static constexpr uint32_t TM_X = TM_Y + D;      // H_K -> Sc -> O
  static constexpr uint32_t TM_COLS = (TM_X + 128 <= 256) ? 256 : 512;
  // shared memory (byte offsets from a 1024-aligned base)
  static constexpr uint32_t W_BYTES = D * D * 2;
  static constexpr uint32_t XT_BYTES = kTile * D * 2;     // one Q or K tile
  static constexpr uint32_t OFF_W = 0;
  static constexpr uint32_t OFF_WK = OFF_W + W_BYTES;     // second map (d = 64 only)
  static constexpr uint32_t OFF_R1 = OFF_WK + (D == 64 ? W_BYTES : 0);
  static constexpr uint32_t OFF_Q = OFF_R1;
  static constexpr uint32_t OFF_K = OFF_R1 + XT_BYTES;
  static constexpr uint32_t OFF_SB = OFF_R1;              // S_bf16 [DP][D] aliases Q/K
  static constexpr uint32_t OFF_V = OFF_R1 + 2 * XT_BYTES;
  static constexpr uint32_t OFF_PHK = OFF_V + XT_BYTES;   // phi(K) panels; P aliases
  static constexpr uint32_t OFF_END = OFF_PHK + PHK_PANELS * 16384;
  static_assert(DP * D * 2 <= 2 * XT_BYTES, "S_bf16 must fit in the Q/K region");
};

template <int D>
struct Smem {
  using C = Cfg<D>;
  static constexpr int ZN = 384;
  // scalars after the operand area
  static constexpr uint32_t OFF_Z = C::OFF_END;                  // float[ZN]
  static constexpr uint32_t OFF_ZP = OFF_Z + ZN * 4;             // float[4][ZN]
  static constexpr uint32_t OFF_DQ = OFF_ZP + 4 * ZN * 4;        // float[2][128]
  static constexpr uint32_t OFF_RS = OFF_DQ + 2 * 128 * 4;       // float[2][128]
  static constexpr uint32_t OFF_BQ = OFF_RS + 2 * 128 * 4;       // float[128]
  static constexpr uint32_t OFF_BK = OFF_BQ + 128 * 4;           // float[128]
  static constexpr uint32_t OFF_BAR = OFF_BK + 128 * 4;          // 4 x u64
  static constexpr uint32_t OFF_MISC = OFF_BAR + 4 * 8;          // tmem base, abort
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t ALLOC = BYTES + 1024;                // slack for alignment
};

struct PrefillArgs {
  CUtensorMap tq, tk, tv, twq, twk, ty;   // ty: y rows, 128-row boxes
  float* ws;        // [U][P-1][DPP*D + DPP]: segment states (S then z), scanned in place
  const float* init;  // [U][DPP*D + DPP] initial state in the same layout, or null
  float* S_out;     // [U][DPP][D] or null
  float* z_out;     // [U][DPP] or null
  const float* bq;
  const float* bk;
  const float2* offq;   // softmax map: [U][NT*128] per-row offsets (log2 units), else null
  const float2* offk;
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int H;
  int P;            // segments per unit
  int L;            // tiles per segment
  int NT;           // tiles per unit
  int sep_wk;       // distinct key map loaded in the second W buffer
  int G;            // query heads per key/value head
  int seq;          // q, k, v, y are [B][n][H][D]
};

// ---------------------------------------------------------------------------
// warp-level helpers
// ---------------------------------------------------------------------------

// Sum of 32 per-lane vectors a[0..31] across the warp: afterwards lane L holds
// the sum over lanes of a[L] in a[0].  31 shuffles (recursive halving).
__device__ __forceinline__ void warp_transpose_sum(float (&a)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? a[i] : a[i + o];
      const float keep = upper ? a[i + o] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

// Write 8 consecutive bf16 (4 packed words) of row r, 16-byte chunk `chunk`
// (0..7) of a 128B-swizzled panel at byte address `panel`.
__device__ __forceinline__ void st_panel_chunk(uint32_t panel, int r, int chunk, uint32_t a,
                                               uint32_t b, uint32_t c, uint32_t d) {
  st_shared_v4(panel + sw128_chunk(r, chunk), a, b, c, d);
}

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)(32 * (warp & 3)) << 16; }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// Hedgehog d = 64 needs 256 TMEM columns and ~108 KB of shared memory, so two
// CTAs share an SM (one's MMAs overlap the other's epilogues).
template <int D>
constexpr int min_blocks() { return D == 64 ? 2 : 1; }

template <int D>
__global__ void __launch_bounds__(kThreads, min_blocks<D>())
prefill_tc_kernel(const __grid_constant__ PrefillArgs A) {
  // the next kernel may be scheduled now; global memory is touched only after
  // the kernels before this one have completed
  pdl_launch_dependents();
  pdl_wait();
  using C = Cfg<D>;
  using SM = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* z_s = reinterpret_cast<float*>(sm + SM::OFF_Z);
  float* zp_s = reinterpret_cast<float*>(sm + SM::OFF_ZP);
  float* dq_s = reinterpret_cast<float*>(sm + SM::OFF_DQ);
  float* rs_s = reinterpret_cast<float*>(sm + SM::OFF_RS);
  float* bq_s = reinterpret_cast<float*>(sm + SM::OFF_BQ);
  float* bk_s = reinterpret_cast<float*>(sm + SM::OFF_BK);
  const uint32_t bar_load = sb + SM::OFF_BAR;
  const uint32_t bar_w = bar_load + 8;
  const uint32_t bar_mma = bar_load + 16;
  const uint32_t bar_sc = bar_load + 24;   // the score MMAs of group 2 alone
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + SM::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp & 3, half = warp >> 2;
  const int row = 32 * g + lane;  // TMEM lane / tile row owned by this thread

  const int64_t unit = blockIdx.x / A.P;
  const int64_t kvu = kv_unit(unit, A.H, A.G);   // k, v of this query head
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int seg = blockIdx.x % A.P;
  const int h = (int)(unit % A.H);
  const int t_begin = seg * A.L;
  const int t_end = min(A.NT, t_begin + A.L);

  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};
  bool failed = false;

  // ---- setup ----
  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_w, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_sc, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&A.tk);
    prefetch_tmap(&A.tv);
    prefetch_tmap(&A.tq);
  }
  // ---- loads of one tile ----
  auto issue_loads = [&](int t) {
    const int r0 = t * kTile;
    uint32_t bytes = C::XT_BYTES * 3;
    mbar_expect_tx(bar_load, bytes);
    for (int i = 0; i < D / 64; ++i) {
      tma_load_rows(sb + C::OFF_Q + i * 16384, &A.tq, bar_load, 64 * i, r0, ub, uh, A.seq);
      tma_load_rows(sb + C::OFF_K + i * 16384, &A.tk, bar_load, 64 * i, r0, ub, kh, A.seq);
      tma_load_rows(sb + C::OFF_V + i * 16384, &A.tv, bar_load, 64 * i, r0, ub, kh, A.seq);
    }
  };
  __syncthreads();  // barriers initialised before the first copy is issued
  if (tid == 0) {
    const int nmaps = A.sep_wk ? 2 : 1;
    mbar_expect_tx(bar_w, C::W_BYTES * nmaps);
    for (int i = 0; i < D / 64; ++i) {
      tma_load_3d(sb + C::OFF_W + i * (D * 128), &A.twq, bar_w, 64 * i, 0, h);
      if (A.sep_wk) tma_load_3d(sb + C::OFF_WK + i * (D * 128), &A.twk, bar_w, 64 * i, 0, h);
    }
    issue_loads(t_begin);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  for (int i = tid; i < D; i += kThreads) {
    bq_s[i] = A.bq ? A.bq[(size_t)h * D + i] : 0.f;
    bk_s[i] = A.bk ? A.bk[(size_t)h * D + i] : 0.f;
  }
  const size_t seg_elems = (size_t)C::DPP * D + C::DPP;
  // the state before this segment: the scanned prefix, the initial state
  // (continuation) or none
  const float* prefix = seg > 0 ? A.ws + ((size_t)unit * (A.P - 1) + seg - 1) * seg_elems
                                : (A.init ? A.init + (size_t)unit * seg_elems : nullptr);
  // initial z: the state of the tokens before this segment
  for (int f = tid; f < SM::ZN; f += kThreads)
    z_s[f] = (prefix && f < C::DPP) ? __ldcg(prefix + (size_t)C::DPP * D + f) : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // initial S in TMEM: zeros, or the prefix state of the preceding segments
  {
    for (int mb = half; mb < C::NMB; mb += 2) {
      const int f = mb * 128 + row;
      const bool frow = prefix && f < C::DPP;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 64) {
        constexpr int CW = D < 64 ? D : 64;
        float4 v4[CW / 4];
#pragma unroll
        for (int j = 0; j < CW / 4; ++j)
          v4[j] = frow ? __ldcg(reinterpret_cast<const float4*>(prefix + ws_s_index(f, c0 + 4 * j, D)))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CW; j += 16) {
          uint32_t r[16];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            r[4 * e] = __float_as_uint(v4[j / 4 + e].x);
            r[4 * e + 1] = __float_as_uint(v4[j / 4 + e].y);
            r[4 * e + 2] = __float_as_uint(v4[j / 4 + e].z);
            r[4 * e + 3] = __float_as_uint(v4[j / 4 + e].w);
          }
          tmem_st16(tmem + lane_base(warp) + C::TM_S + mb * D + c0 + j, r);
        }
      }
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint32_t ph_load = 0, ph_w = 0, ph_mma = 0, ph_sc = 0;



  // descriptors of fixed operands
  constexpr uint32_t IDESC_H = idesc_bf16(128, D, 0, 1);       // X[K-major] * W[MN-major]
  constexpr uint32_t IDESC_SC = idesc_bf16(128, 128, 0, 0);    // phiQ[tmem] * phiK[K-major]
  constexpr uint32_t IDESC_SU = idesc_bf16(128, D, 1, 1);      // phiK^T[MN] * V[MN]
  constexpr uint32_t IDESC_PV = idesc_bf16(128, D, 0, 1);      // P[K-major] * V[MN]
  constexpr uint32_t IDESC_QS = idesc_bf16(128, D, 0, 1);      // phiQ[tmem] * S_bf16[MN]
  // V as an MN-major B operand (rows = tokens = K, columns = d = N)
  auto v_desc = [&](int ks) -> uint64_t {
    return smem_desc(sb + C::OFF_V + ks * 2048, kTile * 128, 1024, 2);
  };
  const uint32_t w_key_off = A.sep_wk ? C::OFF_WK : C::OFF_W;

  for (int t = t_begin; t < t_end && !failed; ++t) {
    const int r0 = t * kTile;
    const int nvalid = (int)min((int64_t)kTile, A.n - r0);
    // softmax map: this row's offsets for phi = [exp(h - c+); exp(-h - c-)],
    // requested here so that their latency passes under group 1
    float2 oq = make_float2(0.f, 0.f), ok_ = make_float2(0.f, 0.f);
    if (A.offq && row < nvalid) {
      const size_t r = (size_t)unit * A.NT * kTile + (size_t)r0 + row;
      oq = A.offq[r];
      ok_ = A.offk[r];
    }

    // ================= group 1: H = X W (Hedgehog) =================
    if (tid == 0) {
      // epilogue 1 below overwrites the y tile of the previous tile, staged in
      // the phi(K) panels; every thread passes the group-1 barrier first
      tma_store_wait_read_all();
      bool ok = mbar_wait(bar_load, ph_load, wp);
      if (t == t_begin) ok = ok && mbar_wait(bar_w, ph_w, wp);
      tc_fence_after();
      if (ok) {
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = (ks * 16 / 64) * 16384 + ((ks * 16) % 64) * 2;
          const uint64_t bq = smem_desc(sb + C::OFF_W + ks * 2048, D * 128, 1024, 2);
          const uint64_t bk = smem_desc(sb + w_key_off + ks * 2048, D * 128, 1024, 2);
          mma_ss(tmem + C::TM_Y, smem_desc(sb + C::OFF_Q + koff, 16, 1024, 2), bq, IDESC_H,
                 ks > 0);
          mma_ss(tmem + C::TM_X, smem_desc(sb + C::OFF_K + koff, 16, 1024, 2), bk, IDESC_H,
                 ks > 0);
        }
        mma_commit(bar_mma);
        // the next tile's Q, K, V into L2 now: their loads wait for group 3
        // (S_bf16 replaces Q / K) and then hit L2
        if (t + 1 < t_end)
          for (int i = 0; i < D / 64; ++i) {
            tma_prefetch_rows(&A.tq, 64 * i, (t + 1) * kTile, ub, uh, A.seq);
            tma_prefetch_rows(&A.tk, 64 * i, (t + 1) * kTile, ub, kh, A.seq);
            tma_prefetch_rows(&A.tv, 64 * i, (t + 1) * kTile, ub, kh, A.seq);
          }
      } else {
        failed = true;
      }
    }
    ph_load ^= 1;
    if (t == t_begin) ph_w ^= 1;
    if (!mbar_wait(bar_mma, ph_mma, wp)) failed = true;
    ph_mma ^= 1;
    tc_fence_after();
    if (__syncthreads_or(failed)) { failed = true; break; }

    // ================= epilogue 1: features, S_bf16, z =================
    // -- phi(Q) into TMEM, denominator part phi(q) . z_before
    {
      float dq = 0.f;
      constexpr int HC = D / 2;  // H columns per warp half
      uint32_t hv[HC];
#pragma unroll
      for (int c = 0; c < HC; c += 32)
        tmem_ld32(tmem + lane_base(warp) + C::TM_Y + half * HC + c,
                  *reinterpret_cast<uint32_t(*)[32]>(&hv[c]));
      tmem_ld_wait();
      tc_fence_before();
      __syncthreads();  // every warp holds its H_Q columns before any overwrite
      tc_fence_after();
      uint32_t pp[HC / 2], pn[HC / 2];
#pragma unroll
      for (int j = 0; j < HC; j += 2) {
        const int l = half * HC + j;
        const float h0 = __uint_as_float(hv[j]) + bq_s[l];
        const float h1 = __uint_as_float(hv[j + 1]) + bq_s[l + 1];
        const uint32_t p = pack_bf16(ex2_approx(fmaf(h0, kLog2e, -oq.x)),
                                     ex2_approx(fmaf(h1, kLog2e, -oq.x)));
        const uint32_t m = pack_bf16(ex2_approx(fmaf(-h0, kLog2e, -oq.y)),
                                     ex2_approx(fmaf(-h1, kLog2e, -oq.y)));
        pp[j / 2] = p;
        pn[j / 2] = m;
        dq += bf16_lo(p) * z_s[l] + bf16_hi(p) * z_s[l + 1] + bf16_lo(m) * z_s[D + l] +
              bf16_hi(m) * z_s[D + l + 1];
      }
      // feature f -> packed column f/2: positive block at half*HC/2, negative at D/2 + half*HC/2
#pragma unroll
      for (int c = 0; c < HC / 2; c += 16) {
        tmem_st16(tmem + lane_base(warp) + C::TM_Y + half * (HC / 2) + c,
                  *reinterpret_cast<const uint32_t(*)[16]>(&pp[c]));
        tmem_st16(tmem + lane_base(warp) + C::TM_Y + D / 2 + half * (HC / 2) + c,
                  *reinterpret_cast<const uint32_t(*)[16]>(&pn[c]));
      }
      dq_s[half * 128 + row] = dq;
    }

    // -- phi(K) into shared memory panels, column sums into zp
    {
      const bool valid = row < nvalid;
      constexpr int HC = D / 2;
#pragma unroll
      for (int c = 0; c < HC; c += 32) {
        uint32_t hv[32];
        tmem_ld32(tmem + lane_base(warp) + C::TM_X + half * HC + c, hv);
        tmem_ld_wait();
        float ep[32], en[32];
        uint32_t wp_[16], wn_[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int l = half * HC + c + j;
          const float h0 = __uint_as_float(hv[j]) + bk_s[l];
          const float h1 = __uint_as_float(hv[j + 1]) + bk_s[l + 1];
          uint32_t p = pack_bf16(ex2_approx(fmaf(h0, kLog2e, -ok_.x)),
                                 ex2_approx(fmaf(h1, kLog2e, -ok_.x)));
          uint32_t m = pack_bf16(ex2_approx(fmaf(-h0, kLog2e, -ok_.y)),
                                 ex2_approx(fmaf(-h1, kLog2e, -ok_.y)));
          if (!valid) p = m = 0u;
          wp_[j / 2] = p;
          wn_[j / 2] = m;
          ep[j] = bf16_lo(p); ep[j + 1] = bf16_hi(p);
          en[j] = bf16_lo(m); en[j + 1] = bf16_hi(m);
        }
        const int fpos = half * HC + c;          // first positive feature of this chunk
        const int fneg = D + half * HC + c;      // first negative feature
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          st_panel_chunk(sb + C::OFF_PHK + (fpos / 64) * 16384, row, (fpos % 64) / 8 + q4,
                         wp_[4 * q4], wp_[4 * q4 + 1], wp_[4 * q4 + 2], wp_[4 * q4 + 3]);
          st_panel_chunk(sb + C::OFF_PHK + (fneg / 64) * 16384, row, (fneg % 64) / 8 + q4,
                         wn_[4 * q4], wn_[4 * q4 + 1], wn_[4 * q4 + 2], wn_[4 * q4 + 3]);
        }
        warp_transpose_sum(ep, lane);
        warp_transpose_sum(en, lane);
        zp_s[g * SM::ZN + fpos + lane] = ep[0];
        zp_s[g * SM::ZN + fneg + lane] = en[0];
      }
    }

    // -- S_bf16 <- S (state before this tile), the B operand of phi(Q) S
    {
      // S_bf16 panel: [DP rows][D cols] as D/64 column blocks of [DP rows x 128 B]
      constexpr int CPW = (C::NMB == 2) ? D : D / 2;   // columns handled by this warp
      const int mb = (C::NMB == 2) ? half : 0;
      const int cbase = (C::NMB == 2) ? 0 : half * (D / 2);
      const int f = mb * 128 + row;
#pragma unroll
      for (int c = 0; c < CPW; c += 32) {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base(warp) + C::TM_S + mb * D + cbase + c, sv);
        tmem_ld_wait();
        const int col = cbase + c;
        const uint32_t panel = sb + C::OFF_SB + (col / 64) * (C::DP * 128);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = 8 * q4;
          st_panel_chunk(panel, f, (col % 64) / 8 + q4,
                         pack_bf16(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                         pack_bf16(__uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3])),
                         pack_bf16(__uint_as_float(sv[j + 4]), __uint_as_float(sv[j + 5])),
                         pack_bf16(__uint_as_float(sv[j + 6]), __uint_as_float(sv[j + 7])));
        }
      }
    }
    tmem_st_wait();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // z += column sums of this tile's phi(K) (after every reader of z_before)
    for (int f = tid; f < C::DPP; f += kThreads)
      z_s[f] += ((zp_s[f] + zp_s[SM::ZN + f]) + zp_s[2 * SM::ZN + f]) + zp_s[3 * SM::ZN + f];

    // ================= group 2: Sc, S update =================
    // The scores are committed on their own: epilogue 2 reads them while the
    // state update runs, and group 3's phi(Q) S half is issued as soon as they
    // are out of TMEM (O reuses their columns); only P V waits for P.
    if (tid == 0) {
      for (int ks = 0; ks < C::KSTEPS_F; ++ks) {
        const uint32_t koff = (ks * 16 / 64) * 16384 + ((ks * 16) % 64) * 2;
        mma_ts(tmem + C::TM_X, tmem + C::TM_Y + ks * 8,
               smem_desc(sb + C::OFF_PHK + koff, 16, 1024, 2), IDESC_SC, ks > 0);
      }
      mma_commit(bar_sc);
      for (int mb = 0; mb < C::NMB; ++mb)
        for (int ks = 0; ks < kTile / 16; ++ks)
          mma_ss(tmem + C::TM_S + mb * D,
                 smem_desc(sb + C::OFF_PHK + (2 * mb) * 16384 + ks * 2048, 16384, 1024, 2),
                 v_desc(ks), IDESC_SU, 1);
      mma_commit(bar_mma);
    }
    if (!mbar_wait(bar_sc, ph_sc, wp)) failed = true;
    ph_sc ^= 1;
    tc_fence_after();

    // ================= epilogue 2: P = bf16(tril(Sc)), row sums =================
    uint32_t pw[32];   // this thread's 64 keys of P as bf16 pairs
    {
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base(warp) + C::TM_X + half * 64 + c, sv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int key = half * 64 + c + j;
          const float a0 = (key <= row) ? __uint_as_float(sv[j]) : 0.f;
          const float a1 = (key + 1 <= row) ? __uint_as_float(sv[j + 1]) : 0.f;
          const uint32_t w2 = pack_bf16(a0, a1);
          pw[(c + j) / 2] = w2;
          rs += bf16_lo(w2) + bf16_hi(w2);
        }
      }
      rs_s[half * 128 + row] = rs;
    }
    tc_fence_before();
    __syncthreads();   // every read of Sc is done: its columns take O
    tc_fence_after();
    // ================= group 3a: O = phi(Q) S_bf16 =================
    if (tid == 0) {
      for (int ks = 0; ks < C::KSTEPS_F; ++ks) {
        const uint64_t bdesc = smem_desc(sb + C::OFF_SB + ks * 2048, C::DP * 128, 1024, 2);
        mma_ts(tmem + C::TM_X, tmem + C::TM_Y + ks * 8, bdesc, IDESC_QS, ks > 0);
      }
    }
    // P overwrites phi(K), which the state update reads
    if (!mbar_wait(bar_mma, ph_mma, wp)) failed = true;
    ph_mma ^= 1;
    tc_fence_after();
    // P panel: [128 rows][128 keys] K-major, key block = half (16 KB each)
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4)
      st_panel_chunk(sb + C::OFF_PHK + half * 16384, row, q4, pw[4 * q4], pw[4 * q4 + 1],
                     pw[4 * q4 + 2], pw[4 * q4 + 3]);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ================= group 3b: O += P V =================
    if (tid == 0) {
      for (int ks = 0; ks < kTile / 16; ++ks) {
        const uint32_t koff = (ks * 16 / 64) * 16384 + ((ks * 16) % 64) * 2;
        mma_ss(tmem + C::TM_X, smem_desc(sb + C::OFF_PHK + koff, 16, 1024, 2), v_desc(ks),
               IDESC_PV, 1);
      }
      mma_commit(bar_mma);   // covers group 3a too
    }
    if (!mbar_wait(bar_mma, ph_mma, wp)) failed = true;
    ph_mma ^= 1;
    tc_fence_after();
    if (tid == 0 && t + 1 < t_end && !failed) issue_loads(t + 1);

    // ================= epilogue 3: y = O / den =================
    // y is staged in the phi(K) / P panels (group 3 has read P) as 128B-swizzled
    // [128 x 64] panels and written by one TMA store per panel; the map clips
    // rows past n.
    {
      const float den = (dq_s[row] + dq_s[128 + row]) + (rs_s[row] + rs_s[128 + row]);
      const float inv = 1.f / den;
      constexpr int HC = D / 2;
#pragma unroll
      for (int c = 0; c < HC; c += 32) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base(warp) + C::TM_X + half * HC + c, ov);
        tmem_ld_wait();
        const int col = half * HC + c;   // 32 columns from col
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = 8 * q4;
          st_panel_chunk(sb + C::OFF_PHK + (col / 64) * 16384, row, (col % 64) / 8 + q4,
                         pack_bf16(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv),
                         pack_bf16(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv),
                         pack_bf16(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv),
                         pack_bf16(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv));
        }
      }
      fence_proxy_async();
    }
    tc_fence_before();
    if (__syncthreads_or(failed)) { failed = true; break; }
    tc_fence_after();
    if (tid == 0) {
#pragma unroll
      for (int x = 0; x < D / 64; ++x)
        tma_store_rows(&A.ty, sb + C::OFF_PHK + x * 16384, 64 * x, r0, ub, uh, A.seq);
      tma_store_commit();
    }
  }
  if (tid == 0) tma_store_wait_all();   // y written (and its panels read) before the export

  // ---- export the final state of the last segment (row-major S_out, z_out) ----
  __syncthreads();
  if (!failed && A.S_out && seg == A.P - 1) {
    float* Sdst = A.S_out + (size_t)unit * C::DPP * D;
    float* zdst = A.z_out + (size_t)unit * C::DPP;
    for (int mb = half; mb < C::NMB; mb += 2) {
      const int f = mb * 128 + row;
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t sv[16];
        tmem_ld16(tmem + lane_base(warp) + C::TM_S + mb * D + c0, sv);
        tmem_ld_wait();
        if (f < C::DPP) {
          float4* dst = reinterpret_cast<float4*>(Sdst + (size_t)f * D + c0);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[q4] = make_float4(__uint_as_float(sv[4 * q4]), __uint_as_float(sv[4 * q4 + 1]),
                                  __uint_as_float(sv[4 * q4 + 2]), __uint_as_float(sv[4 * q4 + 3]));
        }
      }
    }
    for (int f = tid; f < C::DPP; f += kThreads) zdst[f] = z_s[f];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, C::TM_COLS);
}

// In-place inclusive scan over the P-1 segment states of every unit, one
// float4 position per thread, summed in segment order after the initial
// state (continuation) when there is one.  The segments are read in batches
// of four, all loads of a batch issued before its stores, so a thread waits
// for one round trip per batch rather than one per segment.
__global__ void segment_scan_kernel(float4* __restrict__ ws, const float4* __restrict__ init,
                                    int64_t units, int pm1, int64_t elems4) {
  // the next kernel may be scheduled now; global memory is touched only after
  // the kernels before this one have completed
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = units * elems4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t u = i / elems4, e = i % elems4;
    float4* p = ws + (size_t)u * pm1 * elems4 + e;
    float4 acc = init ? __ldcg(init + (size_t)u * elems4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kBatch = 4;
    for (int s0 = 0; s0 < pm1; s0 += kBatch) {
      float4 x[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (s0 + j < pm1) x[j] = __ldcg(p + (size_t)(s0 + j) * elems4);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (s0 + j >= pm1) break;
        if (s0 + j == 0 && !init) {
          acc = x[0];   // the first segment's own sum stays as written
          continue;
        }
        acc.x += x[j].x;
        acc.y += x[j].y;
        acc.z += x[j].z;
        acc.w += x[j].w;
        __stcg(p + (size_t)(s0 + j) * elems4, acc);
      }
    }
  }
}

// The same scan when the state pass summed each segment in m > 1 pieces:
// the pm1 * m piece states of a unit are read from raw in order and the
// running sum after each segment's last piece is written to ws.
__global__ void piece_scan_kernel(float4* __restrict__ ws, const float4* __restrict__ raw,
                                  const float4* __restrict__ init, int64_t units, int pm1, int m,
                                  int64_t elems4) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= units * elems4) return;
  const int64_t u = i / elems4, e = i % elems4;
  const int np = pm1 * m;
  const float4* src = raw + (size_t)u * np * elems4 + e;
  float4* dst = ws + (size_t)u * pm1 * elems4 + e;
  float4 acc = init ? __ldcg(init + (size_t)u * elems4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kBatch = 4;
  for (int s0 = 0; s0 < np; s0 += kBatch) {
    float4 x[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (s0 + j < np) x[j] = __ldcg(src + (size_t)(s0 + j) * elems4);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int t = s0 + j;
      if (t >= np) break;
      acc.x += x[j].x;
      acc.y += x[j].y;
      acc.z += x[j].z;
      acc.w += x[j].w;
      if ((t + 1) % m == 0) __stcg(dst + (size_t)((t + 1) / m - 1) * elems4, acc);
    }
  }
}

// Initial state (continuation) from the public layout -- S [dp_pub][D] and
// z [dp_pub] per unit, as prefill exports it -- into the workspace layout of
// the segment states (ws_s_index, then z).  Taylor keeps the 160 packed
// features of taylor_pack.cuh: a pair (i, j), i < j, stands for public rows
// r0 = (i, j) and r1 = (j, i), and phi_packed(q) . S_packed equals
// phi_pub(q) . S_pub with S_packed = (S[r0] + S[r1]) / sqrt2; the diagonal,
// the constant and the linear features map one to one.
__global__ void init_state_kernel(const float* __restrict__ S0, const float* __restrict__ z0,
                                  float* __restrict__ init, int64_t units, int D, int dp_ws,
                                  int dp_pub, int taylor) {
  // the first kernel of a call: the next one is scheduled only once this one
  // has waited for the work before the call (later kernels of the call may
  // read its inputs before their own wait)
  pdl_wait();
  pdl_launch_dependents();
  const int64_t per = (int64_t)dp_ws * D + dp_ws;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= units * per) return;
  const int64_t u = i / per, e = i % per;
  const float* Su = S0 + (size_t)u * dp_pub * D;
  const float* zu = z0 + (size_t)u * dp_pub;
  const bool is_z = e >= (int64_t)dp_ws * D;
  const int f = is_z ? (int)(e - (int64_t)dp_ws * D) : (int)(e / D);
  const int c = is_z ? 0 : (int)(e % D);
  auto pub = [&](int r) { return is_z ? zu[r] : Su[(size_t)r * D + c]; };
  float val = 0.f;
  if (!taylor) {
    val = f < dp_pub ? pub(f) : 0.f;
  } else {
    int r0 = 0, r1 = 0;
    float scale = 1.f;
    const int cnt = tp::public_rows(f, r0, r1, scale);
    if (cnt == 1) val = pub(r0);
    else if (cnt == 2) val = (pub(r0) + pub(r1)) * scale;
  }
  float* dst = init + (size_t)u * per;
  if (is_z) dst[(size_t)dp_ws * D + f] = val;
  else dst[ws_s_index(f, c, D)] = val;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------



TcPlan plan_prefill_tc(const Problem& p) {
  TcPlan pl;
  pl.supported = (p.dtype == HH_BF16) &&
                 ((p.kind == HH_FMAP_HEDGEHOG && (p.d == 64 || (p.d == 128 && !p.Wk))) ||
                  (p.kind == HH_FMAP_TAYLOR2 && p.d == 16));
  const int64_t U = p.B * p.H;
  pl.NT = ceil_div(p.n, kTile);
  // One sequence per CTA while there are at least as many sequences as SMs;
  // below that, split each sequence so the grid covers the SMs once.
  const int64_t slots = (int64_t)device_sm_count();
  int64_t P = U > 0 ? std::max<int64_t>(1, slots / U) : 1;
  const char* e = getenv("HH_PREFILL_SEGMENTS");
  if (e && *e) P = std::max(1, atoi(e));
  P = std::min<int64_t>(P, std::max(1, pl.NT));
  pl.L = pl.NT > 0 ? ceil_div(pl.NT, P) : 1;
  pl.P = pl.NT > 0 ? ceil_div(pl.NT, pl.L) : 1;
  // The Taylor state pass runs two CTAs per SM: split each segment's state
  // into pieces so that its grid fills both slots of every SM once.
  if (pl.P > 1) {
    int64_t m = p.kind == HH_FMAP_TAYLOR2 ? 2 * slots / (U * (pl.P - 1)) : 1;
    const char* em = getenv("HH_STATE_PIECES");
    if (em && *em) m = atoi(em);
    pl.M = (int)std::max<int64_t>(1, std::min<int64_t>(m, pl.L));
  }
  pl.launches = (pl.P > 2 || pl.M > 1) ? 3 : (pl.P > 1 ? 2 : 1);
  const size_t per = (size_t)ws_segment_floats(p) * sizeof(float);
  pl.ws_bytes = pl.P > 1 ? (size_t)U * (pl.P - 1) * per : 0;
  if (pl.M > 1) {
    pl.raw_offset = pl.ws_bytes;
    pl.ws_bytes += (size_t)U * (pl.P - 1) * pl.M * per;
  }
  if (p.has_init) {
    // the initial state in workspace layout follows the segment states; the
    // scan also runs for two segments
    pl.init_offset = pl.ws_bytes;
    pl.ws_bytes += (size_t)U * (size_t)ws_segment_floats(p) * sizeof(float);
    pl.launches = 1 + (pl.P > 1 ? 3 : 1);
  }
  return pl;
}

// Initial state (continuation), segment-state pass and scan, then the output
// pass of the map: the Taylor, the shared-map d = 64 and the d = 128 passes
// have kernels of their own; d = 64 with a separate key map runs
// prefill_tc_kernel.
template <int KIND, int D>
static cudaError_t launch_kind(const Problem& p, const TcPlan& pl, const void* q, const void* k,
                               const void* v, void* y, float* S_out, float* z_out, void* ws,
                               int* dev_status, cudaStream_t s) {
  const uint64_t U = (uint64_t)p.B * p.H;
  float* init = nullptr;
  if (p.S0) {
    if (!p.has_init || !p.z0) return cudaErrorInvalidValue;
    init = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + pl.init_offset);
    const int64_t per = ws_segment_floats(p);
    const int64_t total = (int64_t)U * per;
    cudaError_t e = launch_pdl(init_state_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256),
                               0, s, p.S0, p.z0, init, (int64_t)U, D, (int)(per / (D + 1)),
                               p.dpp, KIND == HH_FMAP_TAYLOR2 ? 1 : 0);
    if (e != cudaSuccess) return e;
  }
  if (pl.P > 1) {
    cudaError_t e = launch_state_tc(p, pl, k, v, ws, dev_status, s);
    if (e != cudaSuccess) return e;
    if (pl.P > 2 || pl.M > 1 || init) {
      const int64_t elems4 = ws_segment_floats(p) / 4;
      const int64_t n4 = (int64_t)U * elems4;
      const dim3 grid((unsigned)((n4 + 255) / 256));
      if (pl.M > 1)
        e = launch_pdl(piece_scan_kernel, grid, dim3(256), 0, s, reinterpret_cast<float4*>(ws),
                       reinterpret_cast<const float4*>(reinterpret_cast<const char*>(ws) +
                                                       pl.raw_offset),
                       reinterpret_cast<const float4*>(init), (int64_t)U, pl.P - 1, pl.M, elems4);
      else
        e = launch_pdl(segment_scan_kernel, grid, dim3(256), 0, s, reinterpret_cast<float4*>(ws),
                       reinterpret_cast<const float4*>(init), (int64_t)U, pl.P - 1, elems4);
      if (e != cudaSuccess) return e;
    }
  }
  if constexpr (KIND == HH_FMAP_TAYLOR2) {
    return launch_prefill_out_taylor(p, pl, q, k, v, y, S_out, z_out, ws, init, dev_status, s);
  } else {
    if (D == 64 && !p.Wk)
      return launch_prefill_out_d64(p, pl, q, k, v, y, S_out, z_out, ws, init, dev_status, s);
    if constexpr (D == 128) {
      return launch_prefill_out_d128(p, pl, q, k, v, y, S_out, z_out, ws, init, dev_status, s);
    } else {
      PrefillArgs a;
      memset(&a, 0, sizeof(a));
      const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
      bool ok = make_rows_map(&a.tq, q, D, p.n, p.H, p.B, 64, kTile, sw, p.seq_major) &&
                make_rows_map(&a.tk, k, D, p.n, p.H / p.G, p.B, 64, kTile, sw, p.seq_major) &&
                make_rows_map(&a.tv, v, D, p.n, p.H / p.G, p.B, 64, kTile, sw, p.seq_major) &&
                make_plane_map(&a.twq, p.Wq, D, D, p.H, 64, D, sw) &&
                make_plane_map(&a.twk, p.Wk ? p.Wk : p.Wq, D, D, p.H, 64, D, sw) &&
                make_rows_map(&a.ty, y, D, p.n, p.H, p.B, 64, kTile, sw, p.seq_major);
      if (!ok) return cudaErrorInvalidValue;
      a.ws = reinterpret_cast<float*>(ws);
      a.init = init;
      a.S_out = S_out;
      a.z_out = z_out;
      a.bq = p.bq;
      a.bk = p.Wk ? p.bk : p.bq;
      a.offq = p.offq;
      a.offk = p.offk;
      if (p.softmax && (!p.offq || !p.offk)) return cudaErrorInvalidValue;
      a.dev_status = dev_status;
      a.soft_ns = wait_soft_limit_ns();
      a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
      a.n = p.n;
      a.H = p.H;
      a.P = pl.P;
      a.L = pl.L;
      a.NT = pl.NT;
      a.sep_wk = p.Wk ? 1 : 0;
      a.G = p.G;
      a.seq = p.seq_major;
      const size_t smem = Smem<D>::ALLOC;
      auto kern = prefill_tc_kernel<D>;
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return launch_pdl(kern, dim3((unsigned)(U * pl.P)), dim3(kThreads), smem, s, a);
    }
  }
}

cudaError_t launch_prefill_tc(const Problem& p, const TcPlan& pl, const void* q, const void* k,
                              const void* v, void* y, float* S_out, float* z_out, void* ws,
                              int* dev_status, cudaStream_t s) {
  if (p.kind == HH_FMAP_TAYLOR2)
    return launch_kind<HH_FMAP_TAYLOR2, 16>(p, pl, q, k, v, y, S_out, z_out, ws, dev_status, s);
  if (p.d == 64)
    return launch_kind<HH_FMAP_HEDGEHOG, 64>(p, pl, q, k, v, y, S_out, z_out, ws, dev_status, s);
  return launch_kind<HH_FMAP_HEDGEHOG, 128>(p, pl, q, k, v, y, S_out, z_out, ws, dev_status, s);
}

}  // namespace hh
