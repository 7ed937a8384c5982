// Tensor-core gradient of the summed mimicry loss w.r.t. the Hedgehog map.
//
// "The Attention Weight Distillation Loss" (Hedgehog & Porcupine summary)
// trains only the feature maps.  With a_ij = phi(q_i).phi(k_j), A_i the causal
// row sum of a, and p the causal softmax(q k^T / sqrt d), the loss
// L_i = ln A_i - sum_j p_ij ln a_ij has
//   g_ij = dL/da_ij = 1/A_i - p_ij / a_ij                        (j <= i)
//   dL/dphi(q_i) = sum_j g_ij phi(k_j),   dL/dphi(k_j) = sum_i g_ij phi(q_i)
// and through phi = [e^h; e^-h] ("The Hedgehog MLP Feature Map", Choices 1
// and 3)  dL/dh = dL/dphi_+ * e^h - dL/dphi_- * e^-h.
//
// grad_tc_kernel: one CTA per 128-row resident tile, query side (resident
// queries, streamed keys) or key side (resident keys, streamed later
// queries).  Given room for G in the workspace the query side runs first and
// stores every causal 128 x 128 tile of G (bf16, the values its own
// dPhi product uses), and the key side, a second launch, streams those tiles
// with phi(q) instead of forming S, A and g again: each pair is scored once.
// Otherwise both sides form g, in one launch.  Per 64-row streamed step:
//   S = X Y^T and A = phi(X) phi(Y)^T on tcgen05 into one of two TMEM stages;
//   eight epilogue warps turn (S, A) and the query rows' (c_i, 1/A_i) from the
//   loss kernel (p_ij = 2^(s_ij log2e / sqrt d - c_i)) into g, rounded to bf16
//   and written back over the S columns they came from;
//   dPhi (TMEM, 128 x 2d fp32) += G phi(Y), G the TMEM operand and phi(Y) the
//   MN-major smem operand.
// A loader warp streams Y (two smem stages) and phi(Y) (three stages, with
// the query stats on the key side); an issuer warp keeps S/A of step t+1 on
// the tensor core while the epilogue works on step t.  At the end the
// epilogue forms dL/dh = dPhi_+ e^h - dPhi_- e^-h of the tile's rows, stores it
// as two bf16 terms (hi + lo) and one more MMA gives the tile's share of
//   dL/dW = X^T dL/dh,  dL/db = 1^T dL/dh
// written to a per-CTA partial; grad_partials_kernel sums the partials of each
// head in a fixed order.
// Softmax map (Choice 4, Eq. 5: phi_+ = softmax(h), phi_- = softmax(-h), no
// bias): dL/dh = phi_+ (dPhi_+ - <dPhi_+, phi_+>) - phi_- (dPhi_- - <dPhi_-,
// phi_->), the softmax Jacobian of each half.  The two warps that share a row
// each hold half of its columns; they swap their partial dots through shared
// memory before forming dL/dh.  There is no db.

#include <math.h>
#include <string.h>

#include <algorithm>

#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace hh {
namespace {

using namespace tc;

constexpr int kRT = 128;           // resident rows per CTA
constexpr int kST = 64;            // streamed rows per step
constexpr int kThreads = 320;      // 8 epilogue warps, MMA issuer warp, loader warp
constexpr int kIssuerWarp = 8, kLoaderWarp = 9;


struct GradArgs {
  // [0]: query side (X = q, Y = k), [1]: key side (X = k, Y = q)
  CUtensorMap tx[2], tpx[2], ty[2], tpy[2];
  CUtensorMap tg;        // G tiles as [tile][128 query rows][128 keys], 64 x 64 boxes
  const float2* stats;   // [U][npad] (c_i, 1/A_i) of the query rows
  float* part;           // [2][U][NT][D * D + D] per-CTA dW, db shares
  __nv_bfloat16* gbuf;   // [U][NT (NT + 1) / 2][128][128]: G tile (i, j <= i) at i (i + 1) / 2 + j
  int sides;             // 0: both sides form g; 1: query side, storing G; 2: key side, reading G
  int64_t ntt;           // G tiles per unit, NT (NT + 1) / 2
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n, U;
  int H, G;              // heads; query heads per key/value head
  int HG;                // (batch, head) units per scheduling group
  int seq;               // q, k are [B][n][H][D]
  int NT;                // 128-row tiles per sequence
  int npad;              // NT * 128
  float s_scale;         // log2(e) / sqrt(d)
  int softmax;           // phi(X), phi(Y) are the softmax map
};

template <int D>
struct GradCfg {
  static constexpr int DP = 2 * D;
  static constexpr uint32_t X_BYTES = kRT * D * 2;
  static constexpr uint32_t PX_BYTES = kRT * DP * 2;
  static constexpr uint32_t Y_BYTES = kST * D * 2;
  static constexpr uint32_t PY_BYTES = kST * DP * 2;
  static constexpr uint32_t ST_BYTES = kST * 8;
  // a stored G chunk, 64 query rows x 128 keys: two 8 KB panels of 64 keys
  static constexpr uint32_t G_BYTES = kST * kRT * 2;
  static constexpr uint32_t OFF_X = 0;                       // D/64 panels of 16 KB
  static constexpr uint32_t OFF_PX = OFF_X + X_BYTES;        // DP/64 panels of 16 KB
  static constexpr uint32_t OFF_Y = OFF_PX + PX_BYTES;       // 2 stages, D/64 panels of 8 KB
  static constexpr uint32_t OFF_PY = OFF_Y + 2 * Y_BYTES;    // 3 stages, DP/64 panels of 8 KB
  static constexpr uint32_t OFF_ST = OFF_PY + 3 * PY_BYTES;  // 3 stages of 64 (c, 1/A)
  // key side reading G: RG_NS stages of [G chunk | phi(Y) chunk] from offset
  // 0, over everything else; X and phi(X) are loaded once the last stage
  // has been read, for the end phase only.  D = 64 grows its allocation for
  // them; at D = 128 four stages fit below the stats.
  static constexpr uint32_t RG_STAGE = G_BYTES + PY_BYTES;
  static constexpr int RG_NS = 4;
  static constexpr uint32_t OFF_BAR = OFF_ST + 3 * ST_BYTES > RG_NS * RG_STAGE
                                          ? OFF_ST + 3 * ST_BYTES
                                          : RG_NS * RG_STAGE;   // 18 barriers
  static constexpr uint32_t OFF_MISC = OFF_BAR + 18 * 8;
  static constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;
  // end phase: dL/dh as bf16 hi and lo tiles [128 rows][D] (MN-major, 16 KB
  // panels of 64 columns) over the phi(Y) stages; the ones operand of the db
  // product over the Y stages
  static constexpr uint32_t OFF_DH = OFF_PY;
  static constexpr uint32_t DH_BYTES = kRT * D * 2;
  static constexpr uint32_t OFF_ONES = OFF_Y;
  static_assert(2 * DH_BYTES <= 3 * PY_BYTES, "dh tiles exceed the phi(Y) stages");
  // softmax map: per-row partial dots [2 halves][128 rows] float2, after the dh tiles
  static constexpr uint32_t OFF_DOT = OFF_PY + 2 * DH_BYTES;
  static_assert(2 * DH_BYTES + 2 * kRT * 8 <= 3 * PY_BYTES, "row dots exceed the phi(Y) stages");
  static_assert(2 * Y_BYTES >= (D == 64 ? 16384u : 32768u), "ones operand exceeds the Y stages");
  // TMEM columns: S(s) = 128 s, A(s) = 128 s + 64, dPhi = 256 .. 256 + DP.
  // G(s): D = 64 has room for two stages of its own at 384 + 32 s, so S/A of
  // step t+2 waits only for the epilogue to have read step t; for D = 128
  // G(s) goes over the first 16 columns of each 32-column half of S(s) (read
  // already), and S/A of step t+2 waits for G phi(Y) of step t.
  // End phase: X^T dh at 0 (D columns), for D = 128 also 1^T dh at 128.
  static constexpr bool SEP_G = D == 64;
  static constexpr uint32_t TM_ACC = 256;
  static constexpr uint32_t TM_G = 384;
  static constexpr uint32_t TM_DW = 0, TM_DB = 128;
};

__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

__device__ __forceinline__ int clamp32(int64_t v) { return v < 0 ? 0 : (v > 32 ? 32 : (int)v); }

// g of one 32-column chunk.  Query side: columns are keys, (c, 1/A) of the
// row.  Key side: columns are queries, (c, 1/A) per column from stc.
// Columns outside [lo, hi) are zero.
template <bool KEYS>
__device__ __forceinline__ void make_g(const uint32_t (&sv)[32], const uint32_t (&av)[32],
                                       float c_row, float ia_row, const float2* stc, int lo,
                                       int hi, float s_scale, uint32_t (&gw)[16]) {
  const bool full = lo == 0 && hi == 32;
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float g[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float c = KEYS ? stc[e + u].x : c_row;
      const float ia = KEYS ? stc[e + u].y : ia_row;
      const float p = ex2_approx(fmaf(__uint_as_float(sv[e + u]), s_scale, -c));
      const float gv = ia - __fdividef(p, __uint_as_float(av[e + u]));
      g[u] = (full || (e + u >= lo && e + u < hi)) ? gv : 0.f;
    }
    gw[e / 2] = pack_bf16(g[0], g[1]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) grad_tc_kernel(const __grid_constant__ GradArgs A) {
  using C = GradCfg<D>;
  constexpr int DP = C::DP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t bar_x = sb + C::OFF_BAR;   // resident X, phi(X) landed
  const uint32_t bar_y = bar_x + 8;         // (2) Y stage landed
  const uint32_t bar_py = bar_x + 24;       // (3) phi(Y) stage (+ stats) landed
  const uint32_t bar_pyfree = bar_x + 48;   // (3) phi(Y) stage read by its G phi(Y) MMAs
  const uint32_t bar_sa = bar_x + 72;       // (2) S, A MMAs of TMEM stage s done (Y stage free)
  const uint32_t bar_g = bar_x + 88;        // (2) G of TMEM stage s written
  const uint32_t bar_gphi = bar_x + 104;    // (2) G phi(Y) of TMEM stage s done
  const uint32_t bar_acc = bar_x + 120;     // all accumulation done (one barrier)
  const uint32_t bar_free = bar_x + 128;    // (2) epilogue has read S, A of stage s (SEP_G)
  // key side reading G: (RG_NS) stage landed / read by its MMAs, over the
  // Y, phi(Y) and S/A barriers that side does not use (all of count 1)
  const uint32_t rg_full = bar_x + 8, rg_empty = bar_x + 48;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 4);
  // bar_acc is reused for the final dW / db product (phase 1)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Units in groups of HG; within a group heavy tiles first, the two sides
  // interleaved (when one launch holds both).  The CTAs in flight then
  // stream the rows of a few heads only, which stay in L2 across that
  // group's tiles.
  const int nsides = A.sides == 0 ? 2 : 1;
  const int64_t GT = nsides * (int64_t)A.HG * A.NT;
  // The query side storing g takes the groups in reverse order, so that it
  // starts on the heads whose rows the statistics kernel read last and the
  // key side (natural order) starts on the g tiles it wrote last, while they
  // may still be in L2.
  const int64_t ngrp = (A.U + A.HG - 1) / A.HG;
  const int64_t grp = A.sides == 1 ? ngrp - 1 - (int64_t)blockIdx.x / GT : (int64_t)blockIdx.x / GT;
  const int64_t within = blockIdx.x % GT;
  const int64_t gsz = min((int64_t)A.HG, A.U - grp * A.HG);
  const int side = A.sides == 0 ? (int)(within & 1) : A.sides - 1;
  const int64_t wu = A.sides == 0 ? within >> 1 : within;
  const int rank = (int)(wu / gsz);
  const int64_t unit = grp * A.HG + wu % gsz;
  const bool store_g = A.sides == 1, read_g = A.sides == 2;
  const int64_t kvu = kv_unit(unit, A.H, A.G);   // raw k of this query head
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int rt = side ? rank : A.NT - 1 - rank;   // resident tile
  const int64_t r0 = (int64_t)rt * kRT;
  // streamed rows: keys 0 .. min(r0 + 128, n) (query side) or queries r0 .. n (key side)
  const int64_t y_begin = side ? r0 : 0;
  const int64_t y_end = side ? A.n : min(r0 + kRT, A.n);
  const int T = (int)((y_end - y_begin + kST - 1) / kST);
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    mbar_init(bar_x, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_y + 8 * s, 1);
      mbar_init(bar_sa + 8 * s, 1);
      mbar_init(bar_g + 8 * s, 8);
      mbar_init(bar_gphi + 8 * s, 1);
      mbar_init(bar_free + 8 * s, 8);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(bar_py + 8 * s, 1);
      mbar_init(bar_pyfree + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the next kernel may be scheduled now; global memory is touched only after
  // the kernels before this one have completed
  pdl_launch_dependents();
  pdl_wait();
  __syncthreads();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoaderWarp) {
    // ---------------- loader: TMA ----------------
    if (lane == 0) {
      bool ok = true;
      auto load_x = [&]() {
        mbar_expect_tx(bar_x, C::X_BYTES + C::PX_BYTES);
        for (int i = 0; i < D / 64; ++i)
          tma_load_rows(sb + C::OFF_X + i * 16384, &A.tx[side], bar_x, 64 * i, (int)r0,
                        ub, side ? kh : uh, A.seq);
        for (int i = 0; i < DP / 64; ++i)
          tma_load_3d(sb + C::OFF_PX + i * 16384, &A.tpx[side], bar_x, 64 * i, (int)r0,
                      (int)unit);
      };
      if (read_g) {
        // rows y0 .. y0 + 63 of G tile (query tile y0 / 128, key tile rt)
        // and of phi(Y), into stage t % RG_NS once its last reader is done
        for (int t = 0; t < T && ok; ++t) {
          const int s = t % C::RG_NS;
          const int64_t y0 = y_begin + (int64_t)t * kST;
          if (t >= C::RG_NS) ok = mbar_wait_poll(rg_empty + 8 * s, (t / C::RG_NS - 1) & 1, wp);
          if (!ok) break;
          const uint32_t st = sb + s * C::RG_STAGE;
          const int qi = (int)(y0 / kRT);
          const int tile = (int)(unit * A.ntt + (int64_t)qi * (qi + 1) / 2 + rt);
          mbar_expect_tx(rg_full + 8 * s, C::G_BYTES + C::PY_BYTES);
          for (int i = 0; i < 2; ++i)
            tma_load_3d(st + i * 8192, &A.tg, rg_full + 8 * s, 64 * i, (int)(y0 % kRT), tile);
          for (int i = 0; i < DP / 64; ++i)
            tma_load_3d(st + C::G_BYTES + i * 8192, &A.tpy[side], rg_full + 8 * s, 64 * i,
                        (int)y0, (int)unit);
        }
        // X, phi(X) over the stages once every MMA has read them
        ok = ok && mbar_wait_poll(bar_acc, 0, wp);
        if (ok) load_x();
      } else {
        load_x();
      }
      // Y(t) after S/A(t-2) read its stage; phi(Y)(t) after G phi(Y)(t-3)
      for (int t = 0; t < (read_g ? 0 : T) && ok; ++t) {
        const int s = t & 1, p = t % 3;
        const int64_t y0 = y_begin + (int64_t)t * kST;
        if (t >= 2) ok = mbar_wait_poll(bar_sa + 8 * s, ((t >> 1) - 1) & 1, wp);
        if (!ok) break;
        mbar_expect_tx(bar_y + 8 * s, C::Y_BYTES);
        for (int i = 0; i < D / 64; ++i)
          tma_load_rows(sb + C::OFF_Y + s * C::Y_BYTES + i * 8192, &A.ty[side], bar_y + 8 * s,
                        64 * i, (int)y0, ub, side ? uh : kh, A.seq);
        if (t >= 3) ok = mbar_wait_poll(bar_pyfree + 8 * p, (t / 3 - 1) & 1, wp);
        if (!ok) break;
        mbar_expect_tx(bar_py + 8 * p, C::PY_BYTES + (side ? C::ST_BYTES : 0));
        for (int i = 0; i < DP / 64; ++i)
          tma_load_3d(sb + C::OFF_PY + p * C::PY_BYTES + i * 8192, &A.tpy[side], bar_py + 8 * p,
                      64 * i, (int)y0, (int)unit);
        if (side)
          bulk_load(sb + C::OFF_ST + p * C::ST_BYTES, A.stats + unit * A.npad + y0, C::ST_BYTES,
                    bar_py + 8 * p);
      }
    }
  } else if (warp == kIssuerWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t ID_SA = idesc_bf16(128, kST, 0, 0);
      constexpr uint32_t ID_G = idesc_bf16(128, DP, 0, 1);
      // K-major 128B-swizzled panels: resident panels 16 KB (1024 units),
      // streamed panels 8 KB (512 units); a 16-element k-step moves 32 bytes
      const uint64_t dX = smem_desc(sb + C::OFF_X, 16, 1024, 2);
      const uint64_t dPX = smem_desc(sb + C::OFF_PX, 16, 1024, 2);
      auto kx = [](int ks) { return (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2); };
      auto ky = [](int ks) { return (uint64_t)((ks >> 2) * 512 + (ks & 3) * 2); };
      auto issue_g = [&](int u) -> bool {
        const int s = u & 1, p = u % 3;
        if (!mbar_wait_poll(bar_g + 8 * s, (u >> 1) & 1, wp)) return false;
        tc_fence_after();
        // phi(Y) as the MN-major B operand: 64-feature blocks 8 KB apart
        // (LBO), 8-row groups 1 KB apart (SBO); 16 rows per k-step = 2 KB
        const uint64_t dPYmn = smem_desc(sb + C::OFF_PY + p * C::PY_BYTES, 8192, 1024, 2);
        // G: 16 rows of k per step = 8 TMEM columns; the two 32-row halves
        // of the step sit 32 columns apart
#pragma unroll
        for (int ks = 0; ks < kST / 16; ++ks) {
          const uint32_t ga = C::SEP_G ? tmem + C::TM_G + 32 * s + 8 * ks
                                       : tmem + 128 * s + 32 * (ks >> 1) + 8 * (ks & 1);
          mma_ts(tmem + C::TM_ACC, ga, dPYmn + 128 * ks, ID_G, (u > 0 || ks > 0) ? 1 : 0);
        }
        mma_commit(bar_gphi + 8 * s);
        mma_commit(bar_pyfree + 8 * p);
        return true;
      };
      // (the key side reading G loads X only for the end phase)
      bool ok = read_g || mbar_wait_poll(bar_x, 0, wp);
      if (read_g) {
        // dPhi += G^T phi(Y): A = the stored G chunk as an MN-major operand
        // (keys contiguous: 64-key panels 8 KB apart, 8-row groups 1 KB
        // apart), B = phi(Y) MN-major as above; 16 query rows per k-step
        constexpr uint32_t ID_GS = idesc_bf16(128, DP, 1, 1);
        for (int t = 0; t < T && ok; ++t) {
          const int s = t % C::RG_NS;
          ok = mbar_wait_poll(rg_full + 8 * s, (t / C::RG_NS) & 1, wp);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = sb + s * C::RG_STAGE;
          const uint64_t dG = smem_desc(st, 8192, 1024, 2);
          const uint64_t dPYmn = smem_desc(st + C::G_BYTES, 8192, 1024, 2);
#pragma unroll
          for (int ks = 0; ks < kST / 16; ++ks)
            mma_ss(tmem + C::TM_ACC, dG + 128 * ks, dPYmn + 128 * ks, ID_GS,
                   (t > 0 || ks > 0) ? 1 : 0);
          mma_commit(rg_empty + 8 * s);
        }
        if (ok) mma_commit(bar_acc);
      }
      for (int t = 0; t < (read_g ? 0 : T) && ok; ++t) {
        const int s = t & 1, p = t % 3;
        ok = mbar_wait_poll(bar_y + 8 * s, (t >> 1) & 1, wp);
        ok = ok && mbar_wait_poll(bar_py + 8 * p, (t / 3) & 1, wp);
        // TMEM stage s is free once the epilogue has read S/A(t-2) (SEP_G) or
        // once G(t-2) written over it has been consumed
        if (ok && t >= 2)
          ok = mbar_wait_poll((C::SEP_G ? bar_free : bar_gphi) + 8 * s, ((t >> 1) - 1) & 1, wp);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dY = smem_desc(sb + C::OFF_Y + s * C::Y_BYTES, 16, 1024, 2);
        const uint64_t dPY = smem_desc(sb + C::OFF_PY + p * C::PY_BYTES, 16, 1024, 2);
        const uint32_t ts = tmem + 128 * s;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) mma_ss(ts, dX + kx(ks), dY + ky(ks), ID_SA, ks > 0);
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ss(ts + 64, dPX + kx(ks), dPY + ky(ks), ID_SA, ks > 0);
        mma_commit(bar_sa + 8 * s);
        if (t >= 1) ok = issue_g(t - 1);
      }
      if (!read_g && ok) {
        ok = issue_g(T - 1);
        if (ok) mma_commit(bar_acc);
      }
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int half = warp >> 2, row = 32 * (warp & 3) + lane;
    const uint32_t lb = lane_base(warp);
    const int64_t ri = r0 + row;                 // this thread's resident row
    const bool row_ok = ri < A.n;
    float c_row = 0.f, ia_row = 0.f;
    if (!side && row_ok) {
      const float2 st = A.stats[unit * A.npad + ri];
      c_row = st.x;
      ia_row = st.y;
    }
    bool ok = true;
    // this thread's row of the stored G tiles (query side): tile (rt, j) at
    // rt (rt + 1) / 2 + j, row `row`, 128 keys
    __nv_bfloat16* grow = store_g ? A.gbuf + ((size_t)unit * A.ntt + (size_t)rt * (rt + 1) / 2) *
                                                 (size_t)(kRT * kRT) + (size_t)row * kRT
                                  : nullptr;
    for (int t = 0; t < (read_g ? 0 : T); ++t) {
      const int s = t & 1, p = t % 3;
      if (!mbar_wait(bar_sa + 8 * s, (t >> 1) & 1, wp)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = tmem + lb + 128 * s + 32 * half;
      uint32_t sv[32], av[32];
      tmem_ld32x2(ts, sv, ts + 64, av);
      if (C::SEP_G) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_free + 8 * s);
      }
      // admitted columns of this 32-column chunk
      // the key side reads this step's query stats (landed with phi(Y))
      if (side && !mbar_wait(bar_py + 8 * p, (t / 3) & 1, wp)) { ok = false; break; }
      const int64_t cbase = y_begin + (int64_t)t * kST + 32 * half;
      int lo = 0, hi = 0;
      if (row_ok) {
        if (!side) {   // keys j <= i
          hi = clamp32(ri - cbase + 1);
        } else {       // queries i >= j, i < n
          lo = clamp32(ri - cbase);
          hi = clamp32(A.n - cbase);
        }
      }
      const float2* stc =
          reinterpret_cast<const float2*>(sm + C::OFF_ST + p * C::ST_BYTES) + 32 * half;
      uint32_t gw[16];
      if (side)
        make_g<true>(sv, av, c_row, ia_row, stc, lo, hi, A.s_scale, gw);
      else
        make_g<false>(sv, av, c_row, ia_row, stc, lo, hi, A.s_scale, gw);
      if (store_g) {   // keys cbase .. cbase + 31: key tile cbase / 128
        uint4* d4 = reinterpret_cast<uint4*>(grow + (size_t)(cbase / kRT) * (kRT * kRT) +
                                             (int)(cbase % kRT));
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4)
          d4[w4] = make_uint4(gw[4 * w4], gw[4 * w4 + 1], gw[4 * w4 + 2], gw[4 * w4 + 3]);
      }
      if (C::SEP_G) {
        // G stage s: free once G phi(Y) of step t-2 is done
        if (t >= 2 && !mbar_wait(bar_gphi + 8 * s, ((t >> 1) - 1) & 1, wp)) { ok = false; break; }
        tmem_st16(tmem + lb + C::TM_G + 32 * s + 16 * half, gw);
      } else {
        // over the first 16 of this half's 32 S columns (already read)
        tmem_st16(ts, gw);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_g + 8 * s);
    }
    // a last query tile of at most 64 rows streams only the first 64 keys of
    // its diagonal tile: the other 64 (all past the sequence) are stored as
    // zeros, so that the key side reads written values only
    if (store_g && (int64_t)T * kST < r0 + kRT) {
      uint4* d4 = reinterpret_cast<uint4*>(grow + (size_t)rt * (kRT * kRT) +
                                           (int)((int64_t)T * kST - r0) + 32 * half);
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) d4[w4] = make_uint4(0u, 0u, 0u, 0u);
    }
    ok = ok && mbar_wait(bar_acc, 0, wp);
    // the key side reading G loads X, phi(X) only now
    if (read_g) ok = ok && mbar_wait(bar_x, 0, wp);
    if (ok) tc_fence_after();
    // softmax map: the row dots <dPhi_+, phi_+>, <dPhi_-, phi_->, from this
    // thread's half of the columns and the partner warp's (warp ^ 4)
    float cp = 0.f, cn = 0.f;
    if (A.softmax) {
      float sp = 0.f, sn = 0.f;
      if (ok) {
#pragma unroll
        for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
          uint32_t vp[32], vn[32];
          tmem_ld32x2(tmem + lb + C::TM_ACC + c0, vp, tmem + lb + C::TM_ACC + D + c0, vn);
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            const int fp = c0 + 8 * q8, fn = D + c0 + 8 * q8;
            const uint4 pp = *reinterpret_cast<const uint4*>(
                sm + C::OFF_PX + (fp >> 6) * 16384 + sw128_chunk(row, (fp & 63) >> 3));
            const uint4 pn = *reinterpret_cast<const uint4*>(
                sm + C::OFF_PX + (fn >> 6) * 16384 + sw128_chunk(row, (fn & 63) >> 3));
            const uint32_t wpp[4] = {pp.x, pp.y, pp.z, pp.w}, wpn[4] = {pn.x, pn.y, pn.z, pn.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const int e = 8 * q8 + 2 * w;
              sp = fmaf(__uint_as_float(vp[e]), bf16_lo(wpp[w]), sp);
              sp = fmaf(__uint_as_float(vp[e + 1]), bf16_hi(wpp[w]), sp);
              sn = fmaf(__uint_as_float(vn[e]), bf16_lo(wpn[w]), sn);
              sn = fmaf(__uint_as_float(vn[e + 1]), bf16_hi(wpn[w]), sn);
            }
          }
        }
      }
      float2* dots = reinterpret_cast<float2*>(sm + C::OFF_DOT);
      dots[half * kRT + row] = make_float2(sp, sn);
      named_bar_sync(2, 256);
      const float2 o = dots[(half ^ 1) * kRT + row];
      cp = sp + o.x;   // the same sum on both warps: addition commutes
      cn = sn + o.y;
    }
    if (ok) {
      // dL/dh of this row's half of the columns -> bf16 hi + lo tiles
#pragma unroll
      for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
        uint32_t vp[32], vn[32];
        tmem_ld32x2(tmem + lb + C::TM_ACC + c0, vp, tmem + lb + C::TM_ACC + D + c0, vn);
        uint32_t hw[16], lw[16];
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          const int fp = c0 + 8 * q8, fn = D + c0 + 8 * q8;
          const uint4 pp = *reinterpret_cast<const uint4*>(
              sm + C::OFF_PX + (fp >> 6) * 16384 + sw128_chunk(row, (fp & 63) >> 3));
          const uint4 pn = *reinterpret_cast<const uint4*>(
              sm + C::OFF_PX + (fn >> 6) * 16384 + sw128_chunk(row, (fn & 63) >> 3));
          const uint32_t wpp[4] = {pp.x, pp.y, pp.z, pp.w}, wpn[4] = {pn.x, pn.y, pn.z, pn.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int e = 8 * q8 + 2 * w;
            const float d0 = (__uint_as_float(vp[e]) - cp) * bf16_lo(wpp[w]) -
                             (__uint_as_float(vn[e]) - cn) * bf16_lo(wpn[w]);
            const float d1 = (__uint_as_float(vp[e + 1]) - cp) * bf16_hi(wpp[w]) -
                             (__uint_as_float(vn[e + 1]) - cn) * bf16_hi(wpn[w]);
            const uint32_t h = pack_bf16(d0, d1);
            hw[e / 2] = h;
            lw[e / 2] = pack_bf16(d0 - bf16_lo(h), d1 - bf16_hi(h));
          }
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int f = c0 + 8 * cc;
          const uint32_t off = (f >> 6) * 16384 + sw128_chunk(row, (f & 63) >> 3);
          st_shared_v4(sb + C::OFF_DH + off, hw[4 * cc], hw[4 * cc + 1], hw[4 * cc + 2],
                       hw[4 * cc + 3]);
          st_shared_v4(sb + C::OFF_DH + C::DH_BYTES + off, lw[4 * cc], lw[4 * cc + 1],
                       lw[4 * cc + 2], lw[4 * cc + 3]);
        }
      }
      // ones operand of the db product, [128 rows][64] per panel:
      // D = 64: column 0 is one (row 64 of the product is db); D = 128: all ones
      {
        const uint32_t one2 = 0x3F803F80u;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int chunk = 4 * half + cc;
          if (D == 64) {
            const uint32_t w0 = chunk == 0 ? 0x3F80u : 0u;
            st_shared_v4(sb + C::OFF_ONES + sw128_chunk(row, chunk), w0, 0u, 0u, 0u);
          } else {
            st_shared_v4(sb + C::OFF_ONES + sw128_chunk(row, chunk), one2, one2, one2, one2);
            st_shared_v4(sb + C::OFF_ONES + 16384 + sw128_chunk(row, chunk), one2, one2, one2,
                         one2);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
    }
    // all eight epilogue warps have written their rows (or given up)
    named_bar_sync(1, 256);
    ok = ok && !*(volatile int*)abort_flag;
    if (ok && tid == 0) {
      tc_fence_after();
      // X^T [dh_hi + dh_lo]: A = X^T (MN-major: 64-feature blocks at LBO),
      // B = dh (MN-major: 64-column blocks 16 KB apart); 16 rows per k-step
      constexpr uint32_t ID_W = idesc_bf16(128, D, 1, 1);
      const uint64_t dA = smem_desc(sb + C::OFF_X, D == 64 ? (C::OFF_ONES - C::OFF_X) : 16384,
                                    1024, 2);
      const uint64_t dHi = smem_desc(sb + C::OFF_DH, 16384, 1024, 2);
      const uint64_t dLo = smem_desc(sb + C::OFF_DH + C::DH_BYTES, 16384, 1024, 2);
#pragma unroll
      for (int ks = 0; ks < kRT / 16; ++ks) {
        mma_ss(tmem + C::TM_DW, dA + 128 * ks, dHi + 128 * ks, ID_W, ks > 0);
        mma_ss(tmem + C::TM_DW, dA + 128 * ks, dLo + 128 * ks, ID_W, 1);
      }
      if (D == 128) {
        const uint64_t dOnes = smem_desc(sb + C::OFF_ONES, 16384, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < kRT / 16; ++ks) {
          mma_ss(tmem + C::TM_DB, dOnes + 128 * ks, dHi + 128 * ks, ID_W, ks > 0);
          mma_ss(tmem + C::TM_DB, dOnes + 128 * ks, dLo + 128 * ks, ID_W, 1);
        }
      }
      mma_commit(bar_acc);
    }
    if (ok && mbar_wait(bar_acc, 1, wp)) {
      tc_fence_after();
      // row a of the product (TMEM lane) -> partial [a][l]; db from row 64
      // (D = 64) or row 0 of the ones product (D = 128)
      const int a = row;
      float* part = A.part + (((size_t)side * A.U + unit) * A.NT + rt) * (size_t)(D * D + D);
#pragma unroll
      for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lb + C::TM_DW + c0, v);
        float* dst = nullptr;
        if (a < D) dst = part + (size_t)a * D + c0;
        else if (D == 64 && a == 64) dst = part + D * D + c0;
        if (dst) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                            __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        }
        if (D == 128) {
          tmem_ld32(tmem + lb + C::TM_DB + c0, v);
          if (a == 0) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(part + D * D + c0 + e) =
                  make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                              __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// dW[h] (and db[h], stored after it in `part` order) summed over the batch,
// the tiles and the selected sides, in a fixed order.  grid: (ceil((D*D+D)/256), H, outs)
__global__ void grad_partials_kernel(const float* __restrict__ part, float* __restrict__ dW0,
                                     float* __restrict__ db0, float* __restrict__ dW1,
                                     float* __restrict__ db1, int64_t B, int H, int NT, int D,
                                     int separate) {
  // the next kernel may be scheduled now; global memory is touched only after
  // the kernels before this one have completed
  pdl_launch_dependents();
  pdl_wait();
  const int per = D * D + D;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= per) return;
  const int h = blockIdx.y, out = blockIdx.z;
  const int64_t U = B * H;
  float acc = 0.f;
  for (int side = 0; side < 2; ++side) {
    if (separate && side != out) continue;
    for (int64_t b = 0; b < B; ++b) {
      const float* src = part + ((size_t)side * U + b * H + h) * NT * (size_t)per + e;
      for (int t = 0; t < NT; ++t) acc += src[(size_t)t * per];
    }
  }
  float* dW = out ? dW1 : dW0;
  float* db = out ? db1 : db0;
  if (e < D * D) dW[(size_t)h * D * D + e] = acc;
  else if (db) db[(size_t)h * D + (e - D * D)] = acc;   // null: the softmax map has no bias
}

template <int D>
cudaError_t grad_tc_t(const Problem& p, const void* q, const void* k, const void* phq,
                      const void* phk, const float* stats, float* part, void* gbuf,
                      int* dev_status, cudaStream_t s) {
  GradArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  const void* x[2] = {q, k};
  const void* px[2] = {phq, phk};
  bool ok = true;
  for (int side = 0; side < 2; ++side) {
    // raw k (x[1]) has U / G planes under grouped key/value heads
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    ok = ok && make_rows_map(&a.tx[side], x[side], D, p.n, side ? p.H / p.G : p.H, p.B, 64, kRT, sw,
                             p.seq_major) &&
         make_plane_map(&a.tpx[side], px[side], 2 * D, p.n, U, 64, kRT, sw) &&
         make_rows_map(&a.ty[side], x[1 - side], D, p.n, side ? p.H : p.H / p.G, p.B, 64, kST, sw,
                       p.seq_major) &&
         make_plane_map(&a.tpy[side], px[1 - side], 2 * D, p.n, U, 64, kST, sw);
  }
  a.NT = ceil_div(p.n, kRT);
  a.ntt = (int64_t)a.NT * (a.NT + 1) / 2;
  if (gbuf)
    ok = ok && make_plane_map(&a.tg, gbuf, kRT, kRT, U * (uint64_t)a.ntt, 64, kST,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  a.stats = reinterpret_cast<const float2*>(stats);
  a.part = part;
  a.gbuf = reinterpret_cast<__nv_bfloat16*>(gbuf);
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.U = (int64_t)U;
  a.H = p.H;
  a.G = p.G;
  // scheduling groups: q, k and their features (bf16, 3D values per token
  // each) of a group's heads within about a third of the L2
  {
    const double per_unit = (double)p.n * 6.0 * D * 2.0;
    const int64_t hg = std::max<int64_t>(1, (int64_t)(40e6 / std::max(per_unit, 1.0)));
    // equal groups (the largest divisor of U within the budget), so that no
    // short group runs its heavy tiles last
    int64_t g = std::min<int64_t>((int64_t)U, hg);
    while ((int64_t)U % g) --g;
    a.HG = (int)g;
  }
  a.seq = p.seq_major;
  a.npad = a.NT * kRT;
  a.s_scale = 1.4426950408889634f / sqrtf((float)D);
  a.softmax = p.softmax ? 1 : 0;
  const size_t smem = GradCfg<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(grad_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (!gbuf) {
    a.sides = 0;
    return launch_pdl(grad_tc_kernel<D>, dim3((unsigned)(2 * U * a.NT)), dim3(kThreads), smem, s, a);
  }
  // the query side stores G; the key side, launched after it, reads it
  a.sides = 1;
  e = launch_pdl(grad_tc_kernel<D>, dim3((unsigned)(U * a.NT)), dim3(kThreads), smem, s, a);
  if (e != cudaSuccess) return e;
  a.sides = 2;
  return launch_pdl(grad_tc_kernel<D>, dim3((unsigned)(U * a.NT)), dim3(kThreads), smem, s, a);
}

}  // namespace

bool loss_grad_tc_shape(const Problem& p) {
  return p.dtype == HH_BF16 && p.kind == HH_FMAP_HEDGEHOG && (p.d == 64 || p.d == 128);
}

bool loss_grad_tc_supported(const Problem& p) {
  return loss_grad_tc_shape(p) && loss_grad_tc_smem_bytes(p) <= (size_t)device_max_smem_optin();
}

size_t loss_grad_tc_smem_bytes(const Problem& p) {
  return p.d == 64 ? GradCfg<64>::ALLOC : GradCfg<128>::ALLOC;
}

size_t loss_grad_tc_partial_floats(const Problem& p) {
  return (size_t)2 * p.B * p.H * ceil_div(p.n, kRT) * ((size_t)p.d * p.d + p.d);
}

size_t loss_grad_tc_g_bytes(const Problem& p) {
  const size_t nt = (size_t)ceil_div(p.n, kRT);
  return (size_t)p.B * p.H * (nt * (nt + 1) / 2) * kRT * kRT * 2;
}

cudaError_t launch_loss_grad_tc(const Problem& p, const void* q, const void* k, const void* phq,
                                const void* phk, const float* stats, float* part, void* gbuf,
                                float* dWq, float* dbq, float* dWk, float* dbk, int* dev_status,
                                cudaStream_t s) {
  if (p.B * p.H * p.n == 0) return cudaSuccess;
  cudaError_t e = p.d == 64 ? grad_tc_t<64>(p, q, k, phq, phk, stats, part, gbuf, dev_status, s)
                            : grad_tc_t<128>(p, q, k, phq, phk, stats, part, gbuf, dev_status, s);
  if (e != cudaSuccess) return e;
  const int per = p.d * p.d + p.d;
  const int separate = dWk != nullptr;
  dim3 grid((unsigned)ceil_div(per, 256), (unsigned)p.H, separate ? 2u : 1u);
  return launch_pdl(grad_partials_kernel, grid, dim3(256), 0, s, (const float*)part, dWq, dbq, dWk,
                    dbk, (int64_t)p.B, (int)p.H, (int)ceil_div(p.n, kRT), (int)p.d, separate);
}

}  // namespace hh
