// Tensor-core Hedgehog feature map and attention-weight distillation loss.
//
// "The Hedgehog & the Porcupine" summary: "The Hedgehog MLP Feature Map"
// (Choices 1 and 3) for phi(x) = [exp(xW + b); exp(-(xW + b))], and "The
// Attention Weight Distillation Loss" (paper Eq. 4) for
//   L_i = -sum_{j<=i} softmax_j(q_i.k_j / sqrt d) log(a_ij / sum_{m<=i} a_im),
//   a_ij = phi(q_i).phi(k_j).
//
// fmap_tc_kernel: one CTA per 128-row tile of one (batch, head) sequence.
//   H = X W on tcgen05 (fp32 in TMEM); the epilogue adds b, exponentiates
//   both signs and stores phi rows as bf16.  For the softmax-over-features map
//   (Choice 4, Eq. 5; no bias) it first forms the row offsets
//   c+- = logsumexp(+-h) over the d directions (max, then sum of exponentials,
//   each combined across the two warp halves that share a row) and stores
//   exp(+-h - c+-), and/or the offsets themselves for kernels that build phi
//   from h on their own.
//
// loss_tc_kernel: one CTA per (batch*head, 128-query tile); key tiles of 128
//   run j = 0 .. i.  A producer warp TMA-loads K_j and phi(K_j) and issues
//   S = Q K_j^T and A = phi(Q) phi(K_j)^T into one of two TMEM stages; eight
//   epilogue warps keep, per query row, an online-softmax state
//     m (running max of s log2 e), Z = sum 2^{s' - m}, T = sum 2^{s' - m} log2 a,
//     Asum = sum a
//   so that L = ln Asum - ln 2 * T / Z, which equals Eq. 4 because the target
//   weights sum to one.  The statistics variant also keeps
//     U = sum 2^{s' - m} s'  and  V = sum a log2 a
//   for the entropies H(p) = ln Z + ln 2 (m - U / Z) and
//   H(w) = ln Asum - ln 2 V / Asum of "The Two Missing Properties as Design
//   Specifications", and KL = L - H(p).  The smem operands of tile j+1 are loaded as soon as
//   the MMAs of tile j have read them, and those MMAs run while the epilogue
//   works on tile j.

#include <math.h>
#include <string.h>

#include <algorithm>

#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace hh {
namespace {

using namespace tc;

constexpr int kTile = 128;


__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

// ===========================================================================
// feature map
// ===========================================================================
// One launch maps one or two inputs ("sides", e.g. q and k); the grid is
// sides x U x NT tiles.
struct FmapArgs {
  CUtensorMap tx[2], tw[2], tphi[2];
  __nv_bfloat16* phi[2];   // [U][n][2D] or null (written through tphi)
  float2* off[2];          // [U][NT*128] softmax-map offsets (log2 units) or null
  const float* bias[2];    // [H][D] or null
  int kv[2];               // input indexed by key/value head (keys under grouping)
  int G;                   // query heads per key/value head
  int seq;                 // inputs are [B][n][H][D]
  int sides;
  int softmax;
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int H;
  int NT;
};

template <int D>
__global__ void __launch_bounds__(256) fmap_tc_kernel(const __grid_constant__ FmapArgs A) {
  constexpr uint32_t W_BYTES = D * D * 2, X_BYTES = kTile * D * 2;
  // the phi tile ([128 rows][2D], 64-feature panels of 16 KB, 128B swizzle) is
  // staged over W and X once the MMA has read them, then stored by TMA
  constexpr uint32_t PHI_BYTES = kTile * 2 * D * 2;
  constexpr uint32_t AREA = (W_BYTES + X_BYTES) > PHI_BYTES ? (W_BYTES + X_BYTES) : PHI_BYTES;
  constexpr uint32_t TM_COLS = D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t OFF_W = 0, OFF_X = W_BYTES;
  float* bias_s = reinterpret_cast<float*>(sm + AREA);
  float2* red = reinterpret_cast<float2*>(bias_s + 136);   // [2 halves][128 rows]
  const uint32_t bar_load = smem_u32(bias_s + 128);
  const uint32_t bar_mma = bar_load + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bias_s + 128 + 4);
  int* abort_flag = reinterpret_cast<int*>(bias_s + 128 + 5);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = warp >> 2, row = 32 * (warp & 3) + lane;
  const unsigned per_side = gridDim.x / A.sides;
  const int side = (int)(blockIdx.x / per_side);
  const int64_t unit = (blockIdx.x % per_side) / A.NT;
  const int t = (blockIdx.x % per_side) % A.NT;
  const int h = (int)(unit % A.H);
  const int64_t r0 = (int64_t)t * kTile;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // global memory is touched only after the kernels before this one have
  // completed; only then may the next kernel be scheduled (this kernel can be
  // the first of a call, whose later kernels may read the call's inputs early)
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(bar_load, W_BYTES + X_BYTES);
    for (int i = 0; i < D / 64; ++i) {
      tma_load_3d(sb + OFF_W + i * (D * 128), &A.tw[side], bar_load, 64 * i, 0, h);
      tma_load_rows(sb + OFF_X + i * 16384, &A.tx[side], bar_load, 64 * i, (int)r0,
                    (int)(unit / A.H), A.kv[side] ? h / A.G : h, A.seq);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  const float* bias = A.bias[side];
  for (int i = tid; i < D; i += 256) bias_s[i] = bias ? bias[(size_t)h * D + i] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (tid == 0) {
    ok = mbar_wait(bar_load, 0, wp);
    tc_fence_after();
    if (ok) {
      constexpr uint32_t IDESC = idesc_bf16(128, D, 0, 1);
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t koff = (ks * 16 / 64) * 16384 + ((ks * 16) % 64) * 2;
        mma_ss(tmem, smem_desc(sb + OFF_X + koff, 16, 1024, 2),
               smem_desc(sb + OFF_W + ks * 2048, D * 128, 1024, 2), IDESC, ks > 0);
      }
      mma_commit(bar_mma);
    }
  }
  if (__syncthreads_or(!ok)) {
    ok = false;
  } else {
    ok = mbar_wait(bar_mma, 0, wp);
    tc_fence_after();
  }
  if (__syncthreads_and(ok)) {
    constexpr int HC = D / 2;
    const bool valid = r0 + row < A.n;
    const uint32_t trow = tmem + lane_base(warp) + half * HC;
    // softmax map: row offsets op = c+ log2 e, on = c- log2 e (zero otherwise)
    float op = 0.f, on = 0.f;
    if (A.softmax) {
      float mx = -INFINITY, mn = INFINITY;
#pragma unroll
      for (int c = 0; c < HC; c += 32) {
        uint32_t hv[32];
        tmem_ld32(trow + c, hv);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          mx = fmaxf(mx, __uint_as_float(hv[j]));
          mn = fminf(mn, __uint_as_float(hv[j]));
        }
      }
      red[half * 128 + row] = make_float2(mx, mn);
      __syncthreads();
      float2 o = red[(1 - half) * 128 + row];
      const float mp = fmaxf(mx, o.x) * kLog2e, mq = -fminf(mn, o.y) * kLog2e;
      float sp = 0.f, sn = 0.f;
#pragma unroll
      for (int c = 0; c < HC; c += 32) {
        uint32_t hv[32];
        tmem_ld32(trow + c, hv);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          sp += ex2_approx(fmaf(__uint_as_float(hv[j]), kLog2e, -mp));
          sn += ex2_approx(fmaf(-__uint_as_float(hv[j]), kLog2e, -mq));
        }
      }
      __syncthreads();   // the partner has read red before it is overwritten
      red[half * 128 + row] = make_float2(sp, sn);
      __syncthreads();
      o = red[(1 - half) * 128 + row];
      op = mp + __log2f(sp + o.x);
      on = mq + __log2f(sn + o.y);
      if (A.off[side] && half == 0 && valid)
        A.off[side][(size_t)unit * A.NT * kTile + r0 + row] = make_float2(op, on);
    }
    const bool write_phi = A.phi[side] != nullptr;
#pragma unroll
    for (int c = 0; c < HC; c += 32) {
      if (!write_phi) break;
      uint32_t hv[32];
      tmem_ld32(trow + c, hv);
      uint32_t pp[16], pn[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int l = half * HC + c + j;
        const float h0 = __uint_as_float(hv[j]) + bias_s[l];
        const float h1 = __uint_as_float(hv[j + 1]) + bias_s[l + 1];
        pp[j / 2] = pack_bf16(ex2_approx(fmaf(h0, kLog2e, -op)), ex2_approx(fmaf(h1, kLog2e, -op)));
        pn[j / 2] = pack_bf16(ex2_approx(fmaf(-h0, kLog2e, -on)), ex2_approx(fmaf(-h1, kLog2e, -on)));
      }
      // features f = half*HC + c .. +32 (positive) and D + f (negative):
      // four 16-byte chunks each in the swizzled panel of their feature block
      const int fp = half * HC + c, fn = D + half * HC + c;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        st_shared_v4(sb + (fp / 64) * 16384 + sw128_chunk(row, (fp % 64) / 8 + q4), pp[4 * q4],
                     pp[4 * q4 + 1], pp[4 * q4 + 2], pp[4 * q4 + 3]);
        st_shared_v4(sb + (fn / 64) * 16384 + sw128_chunk(row, (fn % 64) / 8 + q4), pn[4 * q4],
                     pn[4 * q4 + 1], pn[4 * q4 + 2], pn[4 * q4 + 3]);
      }
    }
    if (write_phi) {
      // whole 128-byte rows per panel; rows past n are clipped by the store
      fence_proxy_async();
      __syncthreads();
      if (tid == 0) {
        for (int i = 0; i < 2 * D / 64; ++i)
          tma_store_3d(&A.tphi[side], sb + i * 16384, 64 * i, (int)r0, (int)unit);
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ===========================================================================
// mimicry loss
// ===========================================================================
struct LossArgs {
  CUtensorMap tq, tk, tpq, tpk;
  CUtensorMap tw;      // fuse_q: W [H][D][D] of the query map
  const float* bias;   // fuse_q: b [H][D] of the query map, or null
  int fuse_q;          // phi(Q) formed here from Q W + b (Hedgehog map) instead of read
  float* loss_rows;    // [U][n] or null
  float* partial;      // [U][NT]
  float2* stats;       // [U][NT * 128] (c_i, 1 / A_i) or null; c_i = m_i + log2 Z_i
  float4* rows4;       // [U][n] (CE, KL, H(p), H(w)); used by the STATS variant
  const float* colsum; // [U][NT][DP] per-tile column sums of phi(k); row statistics mode
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int64_t U;
  int NT;
  int H, G;            // heads; query heads per key/value head
  int HG;              // (batch, head) units per scheduling group
  int seq;             // q, k are [B][n][H][D]
  float s_scale;       // log2(e) / sqrt(d)
};

template <int D>
struct LossCfg {
  static constexpr int DP = 2 * D;
  static constexpr uint32_t Q_BYTES = kTile * D * 2;
  static constexpr uint32_t PQ_BYTES = kTile * DP * 2;
  // Q resident; K and phi(K) in two stages each.  phi(Q) is staged once in
  // the second phi(K) stage and copied into TMEM, where it stays.
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;          // 2 stages
  static constexpr uint32_t OFF_PK = OFF_K + 2 * Q_BYTES;     // 2 stages
  static constexpr uint32_t OFF_END = OFF_PK + 2 * PQ_BYTES;
  // row scalars for merging the two column halves, over the first K stage
  // once every MMA has completed
  static constexpr uint32_t OFF_ST = OFF_K;                   // float[6][128]: m, Z, T, Asum, U, V
  static constexpr uint32_t OFF_RL = OFF_ST + 6 * 128 * 4;    // float[128] row losses
  static_assert(OFF_RL + 128 * 4 <= OFF_K + Q_BYTES, "row scalars fit one K stage");
  // barriers: per stage K, phi(K) landed; K, phi(K) read; S ready; S drained
  // (6 x 2); Q + phi(Q) (or W) landed; phi(Q) in TMEM; A ready; A read; H = Q W ready
  enum { B_K = 0, B_PK = 2, B_KR = 4, B_PKR = 6, B_S = 8, B_SF = 10, B_Q = 12, B_QT = 13,
         B_A = 14, B_AF = 15, B_H = 16, B_COUNT = 17 };
  static constexpr uint32_t OFF_BAR = OFF_END;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;
  // row statistics mode: sum of phi(k) over the key tiles before this query tile
  static constexpr uint32_t OFF_ZP = OFF_MISC + 16;           // float[DP]
  static constexpr uint32_t ALLOC = OFF_ZP + DP * 4 + 1024;
  static_assert(ALLOC <= 232448, "shared memory");
  // TMEM: S stages at 0 and 128, A at 256, phi(Q) (bf16 pairs) at 384
  static constexpr uint32_t TM_A = 256, TM_PQ = 384;
};

constexpr int kLossThreads = 320;  // 8 epilogue warps, MMA issuer warp 8, loader warp 9

// MODE 0: the loss; 1: the loss and the per-row statistics (rows4); 2: only
// the row statistics (c_i, 1/A_i) the gradient takes (no log a, no loss);
// 3: as 2, with the weights a_ij formed for the diagonal key tile only: the
// earlier key tiles add phi(q_i) . sum_j phi(k_j) to A_i (the linear form of
// the causal row sum), from the per-tile column sums of phi(k).
template <int D, int MODE>
__global__ void __launch_bounds__(kLossThreads, 1) loss_tc_kernel(const __grid_constant__ LossArgs A) {
  using C = LossCfg<D>;
  constexpr bool STATS = MODE == 1, ROWSTATS = MODE >= 2, LINA = MODE == 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* st_s = reinterpret_cast<float*>(sm + C::OFF_ST);
  float* rl_s = reinterpret_cast<float*>(sm + C::OFF_RL);
  const uint32_t bars = sb + C::OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Units are taken in groups of HG, each group's query tiles heavy first:
  // the CTAs in flight at any time then read the keys of a few heads only,
  // whose K and phi(K) stay in L2 while every query tile of those heads
  // streams them (all heads at once would not fit).
  const int64_t GT = (int64_t)A.HG * A.NT;
  const int64_t grp = blockIdx.x / GT, within = blockIdx.x % GT;
  const int64_t gsz = min((int64_t)A.HG, A.U - grp * A.HG);
  const int qt = A.NT - 1 - (int)(within / gsz);
  const int64_t unit = grp * A.HG + within % gsz;
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int64_t q0 = (int64_t)qt * kTile;
  const int nkt = qt + 1;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    for (int b = 0; b < C::B_COUNT; ++b)
      mbar_init(bar(b), (b == C::B_SF || b == C::B_SF + 1 || b == C::B_QT || b == C::B_AF) ? 8 : 1);
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
  bool failed = false;

  auto load_k = [&](int j) {
    const int s = j & 1;
    mbar_expect_tx(bar(C::B_K + s), C::Q_BYTES);
    for (int i = 0; i < D / 64; ++i)
      tma_load_rows(sb + C::OFF_K + s * C::Q_BYTES + i * 16384, &A.tk, bar(C::B_K + s), 64 * i,
                    j * kTile, ub, kh, A.seq);
  };
  auto load_pk = [&](int j) {
    const int s = j & 1;
    mbar_expect_tx(bar(C::B_PK + s), C::PQ_BYTES);
    for (int i = 0; i < C::DP / 64; ++i)
      tma_load_3d(sb + C::OFF_PK + s * C::PQ_BYTES + i * 16384, &A.tpk, bar(C::B_PK + s), 64 * i,
                  j * kTile, (int)unit);
  };

  if (warp == 9) {
    // ---------------- loader ----------------
    //   Q and phi(Q), or W (into the second phi(K) stage) first, K(0),
    //   phi(K)(0), K(1); phi(K)(1) once phi(Q) has gone to TMEM; then K(j),
    //   phi(K)(j) into stage j & 1 as soon as the MMAs of tile j - 2 have read
    //   that stage
    if (lane == 0) {
      mbar_expect_tx(bar(C::B_Q), C::Q_BYTES + (A.fuse_q ? D * D * 2 : C::PQ_BYTES));
      for (int i = 0; i < D / 64; ++i)
        tma_load_rows(sb + C::OFF_Q + i * 16384, &A.tq, bar(C::B_Q), 64 * i, (int)q0, ub, uh, A.seq);
      if (A.fuse_q) {
        for (int i = 0; i < D / 64; ++i)
          tma_load_3d(sb + C::OFF_PK + C::PQ_BYTES + i * (D * 128), &A.tw, bar(C::B_Q), 64 * i, 0,
                      uh);
      } else {
        for (int i = 0; i < C::DP / 64; ++i)
          tma_load_3d(sb + C::OFF_PK + C::PQ_BYTES + i * 16384, &A.tpq, bar(C::B_Q), 64 * i,
                      (int)q0, (int)unit);
      }
      load_k(0);
      if (LINA) {
        // the diagonal key tile's phi(K) only, into the first stage
        mbar_expect_tx(bar(C::B_PK), C::PQ_BYTES);
        for (int i = 0; i < C::DP / 64; ++i)
          tma_load_3d(sb + C::OFF_PK + i * 16384, &A.tpk, bar(C::B_PK), 64 * i, (nkt - 1) * kTile,
                      (int)unit);
      } else {
        load_pk(0);
      }
      if (nkt > 1) load_k(1);
      int nk = nkt < 2 ? nkt : 2, npk = LINA ? nkt : 1;
      IdleClock clk;
      bool ok = true;
      while ((nk < nkt || npk < nkt) && ok) {
        bool progress = false;
        if (nk < nkt && mbar_probe(bar(C::B_KR + (nk & 1)), ((nk - 2) >> 1) & 1)) {
          load_k(nk++);
          progress = true;
        }
        if (npk < nkt &&
            (npk == 1 ? mbar_probe(bar(C::B_QT), 0)
                      : mbar_probe(bar(C::B_PKR + (npk & 1)), ((npk - 2) >> 1) & 1))) {
          load_pk(npk++);
          progress = true;
        }
        if (progress) clk.progress();
        else ok = clk.idle(wp);
      }
      if (!ok) failed = true;
    }
  } else if (warp == 8) {
    // ---------------- MMA issuer ----------------
    //   S(j) = Q K_j^T into S stage j & 1 once K_j landed and the epilogue has
    //   drained that stage (tile j - 2);  A(j) = phi(Q) phi(K_j)^T (phi(Q)
    //   from TMEM) once phi(K_j) landed and the epilogue has copied A(j - 1)
    //   out of the accumulator
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(128, 128, 0, 0);
      auto kmaj = [](int ks) { return (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2); };
      const uint64_t dq = smem_desc(sb + C::OFF_Q, 16, 1024, 2);
      bool ok = true;
      if (A.fuse_q) {
        // H_Q = Q W into the A accumulator (free until A(0)), W as the MN-major B
        constexpr uint32_t ID_H = idesc_bf16(128, D, 0, 1);
        ok = mbar_wait_poll(bar(C::B_Q), 0, wp);
        if (ok) {
          tc_fence_after();
          const uint64_t dw = smem_desc(sb + C::OFF_PK + C::PQ_BYTES, D * 128, 1024, 2);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_ss(tmem + C::TM_A, dq + kmaj(ks), dw + ks * 128, ID_H, ks > 0);
          mma_commit(bar(C::B_H));
        }
      }
      ok = ok && mbar_wait_poll(bar(C::B_QT), 0, wp);
      for (int j = 0; j < nkt && ok; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        ok = mbar_wait_poll(bar(C::B_K + s), ph, wp) &&
             (j < 2 || mbar_wait_poll(bar(C::B_SF + s), ph ^ 1, wp));
        if (!ok) break;
        tc_fence_after();
        const uint64_t dk = smem_desc(sb + C::OFF_K + s * C::Q_BYTES, 16, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + s * 128, dq + kmaj(ks), dk + kmaj(ks), IDESC, ks > 0);
        mma_commit(bar(C::B_S + s));
        mma_commit(bar(C::B_KR + s));
        if (LINA && j < nkt - 1) continue;   // weights of the diagonal tile only
        const int ps = LINA ? 0 : s;
        ok = mbar_wait_poll(bar(C::B_PK + ps), LINA ? 0u : ph, wp) &&
             (LINA || j < 1 || mbar_wait_poll(bar(C::B_AF), (j - 1) & 1, wp));
        if (!ok) break;
        tc_fence_after();
        const uint64_t dpk = smem_desc(sb + C::OFF_PK + ps * C::PQ_BYTES, 16, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < C::DP / 16; ++ks)
          mma_ts(tmem + C::TM_A, tmem + C::TM_PQ + ks * 8, dpk + kmaj(ks), IDESC, ks > 0);
        mma_commit(bar(C::B_A));
        mma_commit(bar(C::B_PKR + ps));
      }
      if (!ok) failed = true;
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int half = warp >> 2, row = 32 * (warp & 3) + lane;
    const uint32_t lb = lane_base(warp);
    const int64_t qi = q0 + row;
    // row statistics mode: the sum of phi(k) over key tiles 0 .. qt-1 (in tile
    // order) into shared memory, and phi(q_i) . that sum over this thread's
    // features, formed below from the same bf16 phi(q) the MMAs read
    float zdot = 0.f;
    const float* zp_s = reinterpret_cast<const float*>(sm + C::OFF_ZP);
    if constexpr (LINA) {
      float* zw = reinterpret_cast<float*>(sm + C::OFF_ZP);
      for (int f = tid; f < C::DP; f += 256) {
        const float* cs = A.colsum + (size_t)unit * A.NT * C::DP + f;
        float acc = 0.f;
        for (int t = 0; t < qt; ++t) acc += __ldg(cs + (size_t)t * C::DP);
        zw[f] = acc;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
    // phi(Q) into TMEM once, as bf16 pairs in the public feature order
    // (exp(+h) in packed columns [0, D/2), exp(-h) in [D/2, D)).  Read:
    // row `row`, features [DP/2 * half, +DP/2) from the staged tile (DP/64
    // panels of [128 rows x 64], 128-byte swizzle) into columns
    // [D/2 * half, +D/2).  Formed: hidden units [D/2 * half, +D/2) of
    // H_Q = Q W, a = (h + b) log2(e), exp2(+-a).
    if (!mbar_wait(bar(A.fuse_q ? C::B_H : C::B_Q), 0, wp)) {
      failed = true;
    } else if (A.fuse_q) {
      tc_fence_after();
      const float* bq = A.bias ? A.bias + (size_t)uh * D : nullptr;
#pragma unroll 1
      for (int u0 = (D / 2) * half; u0 < (D / 2) * half + D / 2; u0 += 32) {
        uint32_t hv[32];
        tmem_ld32(tmem + lb + C::TM_A + u0, hv);
        uint32_t pp[16], pn[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float b0 = bq ? __ldg(bq + u0 + j) * kLog2e : 0.f;
          const float b1 = bq ? __ldg(bq + u0 + j + 1) * kLog2e : 0.f;
          const float a0 = fmaf(__uint_as_float(hv[j]), kLog2e, b0);
          const float a1 = fmaf(__uint_as_float(hv[j + 1]), kLog2e, b1);
          pp[j / 2] = pack_bf16(ex2_approx(a0), ex2_approx(a1));
          pn[j / 2] = pack_bf16(ex2_approx(-a0), ex2_approx(-a1));
        }
        if constexpr (LINA) {
#pragma unroll
          for (int j2 = 0; j2 < 16; ++j2) {
            const int f = u0 + 2 * j2;
            zdot = fmaf(bf16_lo(pp[j2]), zp_s[f], zdot);
            zdot = fmaf(bf16_hi(pp[j2]), zp_s[f + 1], zdot);
            zdot = fmaf(bf16_lo(pn[j2]), zp_s[D + f], zdot);
            zdot = fmaf(bf16_hi(pn[j2]), zp_s[D + f + 1], zdot);
          }
        }
        tmem_st16(tmem + lb + C::TM_PQ + u0 / 2, pp);
        tmem_st16(tmem + lb + C::TM_PQ + D / 2 + u0 / 2, pn);
      }
      tmem_st_wait();
    } else {
      const uint32_t pq = sb + C::OFF_PK + C::PQ_BYTES;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {   // 32 packed columns = 64 features
        const int f0 = (C::DP / 2) * half + 2 * c0;
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(
              sm + (pq - sb) + (f0 / 64) * 16384 + sw128_chunk(row, q));
          w[4 * q] = v4.x;
          w[4 * q + 1] = v4.y;
          w[4 * q + 2] = v4.z;
          w[4 * q + 3] = v4.w;
        }
        if constexpr (LINA) {
#pragma unroll
          for (int k2 = 0; k2 < 32; ++k2) {
            zdot = fmaf(bf16_lo(w[k2]), zp_s[f0 + 2 * k2], zdot);
            zdot = fmaf(bf16_hi(w[k2]), zp_s[f0 + 2 * k2 + 1], zdot);
          }
        }
        tmem_st32(tmem + lb + C::TM_PQ + (D / 2) * half + c0, w);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C::B_QT));   // phi(Q) is in TMEM; its staging stage is free

    // online state; Z, T and the weight sum are kept as two interleaved partial
    // sums so consecutive keys do not form one long dependency chain
    float m = -INFINITY, Z0 = 0.f, Z1 = 0.f, T0 = 0.f, T1 = 0.f, A0 = 0.f, A1 = 0.f;
    float U0 = 0.f, U1 = 0.f, V0 = 0.f, V1 = 0.f;   // STATS only
    const int64_t kmax = min(qi, A.n - 1);   // last key admitted for this row
    for (int j = 0; j < nkt && !failed; ++j) {
      const int s = j & 1;
      // weights of this key tile (mode 3: the diagonal tile only)
      const bool wj = !LINA || j == nkt - 1;
      if ((wj && !mbar_wait(bar(C::B_A), LINA ? 0u : (uint32_t)(j & 1), wp)) ||
          !mbar_wait(bar(C::B_S + s), (j >> 1) & 1, wp)) {
        failed = true;
        break;
      }
      tc_fence_after();
      // A(j) out of the accumulator first, so A(j+1) can start under this tile
      uint32_t av[64];
      if (wj) {
        tmem_ld32x2(tmem + lb + C::TM_A + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&av[0]),
                    tmem + lb + C::TM_A + half * 64 + 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&av[32]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_AF));
      }
      const int64_t k0 = (int64_t)j * kTile + half * 64;
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t sv[32];
        tmem_ld32(tmem + lb + s * 128 + half * 64 + c, sv);
        const int nval = (int)max((int64_t)0, min((int64_t)32, kmax - (k0 + c) + 1));
        if (nval == 32) {
          // every key of the chunk is admitted: no masking
          float c0 = __uint_as_float(sv[0]), c1 = __uint_as_float(sv[1]);
          float c2 = __uint_as_float(sv[2]), c3 = __uint_as_float(sv[3]);
#pragma unroll
          for (int e = 4; e < 32; e += 4) {
            c0 = fmaxf(c0, __uint_as_float(sv[e]));
            c1 = fmaxf(c1, __uint_as_float(sv[e + 1]));
            c2 = fmaxf(c2, __uint_as_float(sv[e + 2]));
            c3 = fmaxf(c3, __uint_as_float(sv[e + 3]));
          }
          const float mn = fmaxf(m, fmaxf(fmaxf(c0, c1), fmaxf(c2, c3)) * A.s_scale);
          const float f = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
          Z0 *= f; Z1 *= f; T0 *= f; T1 *= f;
          if constexpr (STATS) { U0 *= f; U1 *= f; }
          m = mn;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            if constexpr (ROWSTATS) {
              Z0 += ex2_approx(fmaf(__uint_as_float(sv[e]), A.s_scale, -m));
              Z1 += ex2_approx(fmaf(__uint_as_float(sv[e + 1]), A.s_scale, -m));
              if (wj) {
                A0 += __uint_as_float(av[c + e]);
                A1 += __uint_as_float(av[c + e + 1]);
              }
              continue;
            }
            const float a0 = __uint_as_float(av[c + e]), a1 = __uint_as_float(av[c + e + 1]);
            const float l0 = __log2f(a0), l1 = __log2f(a1);
            if constexpr (STATS) {
              const float s0 = __uint_as_float(sv[e]) * A.s_scale;
              const float s1 = __uint_as_float(sv[e + 1]) * A.s_scale;
              const float p0 = ex2_approx(s0 - m), p1 = ex2_approx(s1 - m);
              Z0 += p0;
              Z1 += p1;
              T0 = fmaf(p0, l0, T0);
              T1 = fmaf(p1, l1, T1);
              U0 = fmaf(p0, s0, U0);
              U1 = fmaf(p1, s1, U1);
              V0 = fmaf(a0, l0, V0);
              V1 = fmaf(a1, l1, V1);
            } else {
              const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), A.s_scale, -m));
              const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), A.s_scale, -m));
              Z0 += p0;
              Z1 += p1;
              T0 = fmaf(p0, l0, T0);
              T1 = fmaf(p1, l1, T1);
            }
            A0 += a0;
            A1 += a1;
          }
        } else if (nval > 0) {
          float cm = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < nval) cm = fmaxf(cm, __uint_as_float(sv[e]));
          const float mn = fmaxf(m, cm * A.s_scale);
          const float f = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
          Z0 *= f; Z1 *= f; T0 *= f; T1 *= f;
          if constexpr (STATS) { U0 *= f; U1 *= f; }
          m = mn;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e < nval) {
              if constexpr (ROWSTATS) {
                Z0 += ex2_approx(fmaf(__uint_as_float(sv[e]), A.s_scale, -m));
                if (wj) A0 += __uint_as_float(av[c + e]);
                continue;
              }
              const float a = __uint_as_float(av[c + e]);
              const float la = __log2f(a);
              const float sl = __uint_as_float(sv[e]) * A.s_scale;
              const float p = ex2_approx(sl - m);
              Z0 += p;
              T0 = fmaf(p, la, T0);
              A0 += a;
              if constexpr (STATS) {
                U0 = fmaf(p, sl, U0);
                V0 = fmaf(a, la, V0);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_SF + s));
    }
    float Z = Z0 + Z1, T = T0 + T1, As = A0 + A1 + zdot, Us = U0 + U1, Vs = V0 + V1;
    // the row scalars go over the first K stage: wait until every MMA has read
    // it (the last A, which follows the last S in issue order)
    if (!failed && nkt > 0)
      failed = !mbar_wait(bar(C::B_A), LINA ? 0u : (uint32_t)((nkt - 1) & 1), wp);
    asm volatile("bar.sync 1, 256;" ::: "memory");
    // merge the two column halves of each row
    if (half == 1) {
      st_s[row] = m;
      st_s[128 + row] = Z;
      st_s[256 + row] = T;
      st_s[384 + row] = As;
      if constexpr (STATS) {
        st_s[512 + row] = Us;
        st_s[640 + row] = Vs;
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (half == 0) {
      const float m2 = st_s[row], Z2 = st_s[128 + row], T2 = st_s[256 + row], A2 = st_s[384 + row];
      const float mn = fmaxf(m, m2);
      const float f1 = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
      const float f2 = (m2 == -INFINITY) ? 0.f : ex2_approx(m2 - mn);
      const float Zt = Z * f1 + Z2 * f2, Tt = T * f1 + T2 * f2, At = As + A2;
      const bool valid = qi < A.n;
      const float L = valid && !ROWSTATS ? (logf(At) - 0.69314718055994531f * (Tt / Zt)) : 0.f;
      rl_s[row] = L;
      if (valid && A.loss_rows) A.loss_rows[(size_t)unit * A.n + qi] = L;
      // row statistics for the gradient: p_ij = 2^(s_ij log2e / sqrt d - c_i)
      if (A.stats)
        A.stats[(size_t)unit * A.NT * kTile + qi] =
            valid ? make_float2(mn + __log2f(Zt), 1.f / At) : make_float2(0.f, 0.f);
      if constexpr (STATS) {
        const float Ut = Us * f1 + st_s[512 + row] * f2, Vt = Vs + st_s[640 + row];
        constexpr float kLn2 = 0.69314718055994531f;
        const float Hp = logf(Zt) + kLn2 * (mn - Ut / Zt);
        const float Hw = logf(At) - kLn2 * (Vt / At);
        if (valid) A.rows4[(size_t)unit * A.n + qi] = make_float4(L, L - Hp, Hp, Hw);
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (!ROWSTATS && tid == 0) {
      float acc = 0.f;
      for (int r = 0; r < kTile; ++r) acc += rl_s[r];
      A.partial[(size_t)unit * A.NT + qt] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
  (void)failed;
}

// Column sums of phi(k) over each 128-row tile (rows < n), for the row
// statistics mode: one CTA per (unit, tile), 256 threads; thread t sums the
// 8 features 8 (t % (DP/8)) .. +7 over rows t / (DP/8) + r (256 / (DP/8)),
// then the row groups are added in a fixed order.
template <int DP>
__global__ void __launch_bounds__(256) phi_colsum_kernel(const __nv_bfloat16* __restrict__ phk,
                                                         float* __restrict__ colsum, int64_t n,
                                                         int NT, int dpp) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int FG = DP / 8, RG = 256 / FG;   // feature groups, row groups
  __shared__ float part[RG][DP];
  const int64_t unit = blockIdx.x / NT;
  const int tile = blockIdx.x % NT;
  const int fg = threadIdx.x % FG, rg = threadIdx.x / FG;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int64_t r0 = (int64_t)tile * 128;
  const __nv_bfloat16* base = phk + ((size_t)unit * n) * dpp + 8 * fg;
  for (int r = rg; r < 128; r += RG) {
    if (r0 + r >= n) break;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + (size_t)(r0 + r) * dpp));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] += bf16_lo(w[k]);
      acc[2 * k + 1] += bf16_hi(w[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part[rg][8 * fg + k] = acc[k];
  __syncthreads();
  for (int f = threadIdx.x; f < DP; f += 256) {
    float t = 0.f;
    for (int g = 0; g < RG; ++g) t += part[g][f];
    colsum[((size_t)unit * NT + tile) * DP + f] = t;
  }
}

__global__ void sum_partials_tc_kernel(const float* __restrict__ partial, float* __restrict__ out,
                                       int64_t heads, int ntiles) {
  // the next kernel may be scheduled now; global memory is touched only after
  // the kernels before this one have completed
  pdl_launch_dependents();
  pdl_wait();
  const int64_t bh = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (bh >= heads) return;
  float acc = 0.f;
  for (int t = 0; t < ntiles; ++t) acc += partial[(size_t)bh * ntiles + t];
  out[bh] = acc;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

bool fmap_tc_supported(const Problem& p) {
  return p.dtype == HH_BF16 && p.kind == HH_FMAP_HEDGEHOG && (p.d == 64 || p.d == 128);
}

// sides: inputs x[i] (is_key[i] picks the key map), outputs phi[i] / off[i]
template <int D>
static cudaError_t fmap_tc_t(const Problem& p, int sides, const void* const* x,
                             const int* is_key, void* const* phi, float2* const* off,
                             int* dev_status, cudaStream_t s) {
  FmapArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  for (int i = 0; i < sides; ++i) {
    const void* W = is_key[i] && p.Wk ? p.Wk : p.Wq;
    a.kv[i] = is_key[i] && p.G > 1;
    if (!make_rows_map(&a.tx[i], x[i], D, p.n, a.kv[i] ? p.H / p.G : p.H, p.B, 64, kTile,
                       CU_TENSOR_MAP_SWIZZLE_128B, p.seq_major) ||
        !make_plane_map(&a.tw[i], W, D, D, p.H, 64, D, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    a.phi[i] = reinterpret_cast<__nv_bfloat16*>(phi[i]);
    if (phi[i] && !make_plane_map(&a.tphi[i], phi[i], 2 * D, p.n, U, 64, kTile,
                                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    a.off[i] = p.softmax ? off[i] : nullptr;
    a.bias[i] = is_key[i] && p.Wk ? p.bk : p.bq;
  }
  a.sides = sides;
  a.G = p.G;
  a.seq = p.seq_major;
  a.softmax = p.softmax ? 1 : 0;
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.H = p.H;
  a.NT = ceil_div(p.n, kTile);
  const size_t area = std::max<size_t>((size_t)D * D * 2 + kTile * D * 2, (size_t)kTile * 2 * D * 2);
  const size_t smem = area + 136 * 4 + 256 * 8 + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(fmap_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(fmap_tc_kernel<D>, dim3((unsigned)(sides * U * a.NT)), dim3(256), smem, s, a);
}

cudaError_t launch_fmap_tc(const Problem& p, const void* x, int is_key, void* phi, float2* off,
                           int* dev_status, cudaStream_t s) {
  if (p.B * p.H * p.n == 0) return cudaSuccess;
  return p.d == 64 ? fmap_tc_t<64>(p, 1, &x, &is_key, &phi, &off, dev_status, s)
                   : fmap_tc_t<128>(p, 1, &x, &is_key, &phi, &off, dev_status, s);
}

cudaError_t launch_fmap_tc_qk(const Problem& p, const void* q, const void* k, void* phq,
                              void* phk, float2* offq, float2* offk, int* dev_status,
                              cudaStream_t s) {
  if (p.B * p.H * p.n == 0) return cudaSuccess;
  const void* x[2] = {q, k};
  const int key[2] = {0, 1};
  void* phi[2] = {phq, phk};
  float2* off[2] = {offq, offk};
  return p.d == 64 ? fmap_tc_t<64>(p, 2, x, key, phi, off, dev_status, s)
                   : fmap_tc_t<128>(p, 2, x, key, phi, off, dev_status, s);
}

template <int D>
static cudaError_t loss_tc_t(const Problem& p, const void* q, const void* k, const void* phq,
                             const void* phk, float* loss_rows, float* partial, float* head_sum,
                             float* stats, float4* rows4, float* colsum, int* dev_status,
                             cudaStream_t s) {
  LossArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  // no phi(q) given: the kernel forms phi(Q) from Q W + b (the Hedgehog map;
  // the softmax map needs its row offsets first and comes with phi(q))
  const bool fuse = phq == nullptr;
  if (fuse && p.softmax) return cudaErrorInvalidValue;
  bool ok = make_rows_map(&a.tq, q, D, p.n, p.H, p.B, 64, kTile, sw, p.seq_major) &&
            make_rows_map(&a.tk, k, D, p.n, p.H / p.G, p.B, 64, kTile, sw, p.seq_major) &&
            (fuse ? make_plane_map(&a.tw, p.Wq, D, D, p.H, 64, D, sw)
                  : make_plane_map(&a.tpq, phq, 2 * D, p.n, U, 64, kTile, sw)) &&
            make_plane_map(&a.tpk, phk, 2 * D, p.n, U, 64, kTile, sw);
  if (!ok) return cudaErrorInvalidValue;
  a.fuse_q = fuse ? 1 : 0;
  a.bias = fuse ? p.bq : nullptr;
  a.loss_rows = loss_rows;
  a.partial = partial;
  a.stats = reinterpret_cast<float2*>(stats);
  a.rows4 = rows4;
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.U = (int64_t)U;
  a.NT = ceil_div(p.n, kTile);
  a.H = p.H;
  a.G = p.G;
  // scheduling groups: the K and phi(K) of a group's heads (bf16, 3D values
  // per token) within about a sixth of the L2 (a third measured 0.3-3% slower
  // on the Llama-2 and GPT-2 shapes, loss and gradient alike)
  {
    const double per_unit = (double)p.n * 3.0 * D * 2.0;
    const int64_t hg = std::max<int64_t>(1, (int64_t)(20e6 / std::max(per_unit, 1.0)));
    // equal groups (the largest divisor of U within the budget), so that no
    // short group runs its heavy tiles last
    int64_t g = std::min<int64_t>((int64_t)U, hg);
    while ((int64_t)U % g) --g;
    a.HG = (int)g;
  }
  a.seq = p.seq_major;
  a.s_scale = 1.4426950408889634f / sqrtf((float)D);
  const size_t smem = LossCfg<D>::ALLOC;
  // no loss asked for (no partial sums): the row statistics alone; at d = 128
  // with the off-diagonal row sums in linear form, from column sums of phi(k)
  // per key tile (at d = 64 the weight MMAs cost less than that extra launch:
  // 226 vs 219 us per GPT-2-shaped gradient call)
  const bool rowstats = !partial;
  const bool lina = rowstats && D == 128;
  if (rowstats && (!stats || loss_rows || head_sum || rows4)) return cudaErrorInvalidValue;
  if (lina && (!colsum || !phk)) return cudaErrorInvalidValue;
  a.colsum = colsum;
  if (lina) {
    cudaError_t e = launch_pdl(phi_colsum_kernel<2 * D>, dim3((unsigned)(U * a.NT)), dim3(256), 0, s,
                               reinterpret_cast<const __nv_bfloat16*>(phk), colsum, (int64_t)p.n,
                               a.NT, 2 * D);
    if (e != cudaSuccess) return e;
  }
  auto kern = rows4 ? loss_tc_kernel<D, 1>
                    : (lina ? loss_tc_kernel<D, 3>
                            : (rowstats ? loss_tc_kernel<D, 2> : loss_tc_kernel<D, 0>));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3((unsigned)(U * a.NT)), dim3(kLossThreads), smem, s, a);
  if (e != cudaSuccess || rowstats) return e;
  e = launch_pdl(sum_partials_tc_kernel, dim3((unsigned)ceil_div(U, 128)), dim3(128), 0, s,
                 (const float*)partial, head_sum, (int64_t)U, a.NT);
  return e;
}

cudaError_t launch_loss_tc(const Problem& p, const void* q, const void* k, const void* phq,
                           const void* phk, float* loss_rows, float* partial, float* head_sum,
                           float* stats, float4* rows4, float* colsum, int* dev_status,
                           cudaStream_t s) {
  return p.d == 64 ? loss_tc_t<64>(p, q, k, phq, phk, loss_rows, partial, head_sum, stats, rows4,
                                   colsum, dev_status, s)
                   : loss_tc_t<128>(p, q, k, phq, phk, loss_rows, partial, head_sum, stats, rows4,
                                    colsum, dev_status, s);
}

int loss_tc_tile() { return kTile; }


}  // namespace hh
