// Chunked causal prefill for Hedgehog d = 64 with two tiles in flight.
//
// Same mathematics as prefill_tc_kernel ("2. Context and Motivation", paper Eq. 2, and
// "Complexity Analysis" of "The Hedgehog & the Porcupine" summary; the map of
// "The Hedgehog MLP Feature Map", Choices 1 and 3), reorganised so that the
// serial chain of one 128-token tile overlaps the next tile's:
//
//   warp 8 (MMA issuer): every tcgen05.mma, each group issued as soon as its
//   inputs are ready (it polls the barriers without blocking); issuing a group
//   can stall while the tensor pipe is busy, so
//   warp 9 (loader) issues the TMA loads of the next tiles on its own
//     G1(t): H_Q = Q_t W, H_K = K_t W
//     G2(t): Sc = phi(Q_t) phi(K_t)^T (committed on its own);  [S z] += phi(K_t)^T [V_t 1]
//     G3(t): [O den] = P_t [V_t e0] + phi(Q_t) [S_bf16(t) z2(t)]
//   The normaliser rides along as extra columns of the same MMAs (N = 80):
//   column 64 of the state is z; for the output, e0 = (1, 0, ...) gives the
//   row sums of P and z2 = (z_hi, z_lo, 0, ...) = z split into two bf16, so
//   columns 64 and 65 of O sum to the denominator rowsum(P) + phi(q) . z.
//   warps 0-7 (epilogue) run the phases below for both slots, interleaved as
//   E2(t-1), E1(t), E3(t-1):
//     E1 : phi(Q_t) -> TMEM (bf16 pairs), phi(K_t) -> smem          (after G1(t))
//          S_bf16(t) <- S, z2(t) <- z as a bf16 hi/lo pair (state of the
//          tokens before t)                                         (after G2(t-1))
//          -- only then may G2(t) update S --
//     E2 : P_t = bf16(tril(Sc)); blocks above the diagonal are zero
//          without reading Sc, blocks below it need no mask; built
//          after the Sc MMAs, stored over phi(K) after all of G2(t)
//     E3 : y = O / den, staged in the P panel (free once G3(t) has read it)
//          and stored by TMA, one 32-row slab per warp pair       (after G3(t))
// Each tile owns one slot of TMEM (H_Q/phi(Q), H_K/Sc/O) and smem (V, phi(K) ->
// P -> y, S_bf16, z2); Q and K sit in a separate two-stage ring that is
// refilled as soon as G1 has read it, so the loads of tile t+2 do not wait for
// G3(t).  The running state [S z] (fp32) stays in TMEM and passes between the
// groups in tile order.  All mbarrier waits are bounded (tc_ptx.cuh).

#include <math.h>
#include <string.h>

#include <algorithm>

#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace hh {
namespace {

using namespace tc;

constexpr int D = 64, DP = 128, TILE = 128;
constexpr int kThreads = 320;   // 8 epilogue warps, warp 8 issues MMAs, warp 9 issues loads

// TMEM columns
constexpr uint32_t TM_S = 0;     // [S z 0]: features (lanes) x 80, column 64 = z
__host__ __device__ constexpr uint32_t TM_Y(int s) { return 128 + 192 * s; }        // 64 cols
__host__ __device__ constexpr uint32_t TM_X(int s) { return 128 + 192 * s + 64; }   // 128 cols

// shared memory
constexpr uint32_t OFF_W = 0;
constexpr uint32_t OFF_QK = 8192;                         // 2 stages of Q, K (16 KB each)
__host__ __device__ constexpr uint32_t qk_off(int st) { return OFF_QK + st * 32768; }
constexpr uint32_t SLOT_BASE = OFF_QK + 2 * 32768, SLOT_BYTES = 65536;
// per slot: V, phi(K) -> P -> y (two panels), S_bf16 (read by G3)
constexpr uint32_t S_V = 0, S_PHK = 16384, S_SB = 49152;
__host__ __device__ constexpr uint32_t slot_off(int s) { return SLOT_BASE + s * SLOT_BYTES; }
// [128 x 64] SW128 panel holding three 16-column N blocks: logical columns
// 0..15 are e0 (row r = (1, 0, ...), the extra N block of V), 16 + 16s.. are
// z2 of slot s (row f = (z_hi, z_lo, 0, ...), the extra N block of S_bf16).
// A descriptor reaches block j by a start address 32j bytes into the row; it
// sits after the slots because the leading-byte offset field is unsigned.
constexpr uint32_t OFF_E0 = SLOT_BASE + 2 * SLOT_BYTES;
constexpr uint32_t OFF_BQ = OFF_E0 + 16384;               // float[64]: b * log2(e)
constexpr uint32_t OFF_BAR = OFF_BQ + 256;                // 19 x u64 (20 reserved)
constexpr uint32_t OFF_TM = OFF_BAR + 160;
// softmax map: per-row partial maxima, then sums, swapped between the two warps
// that hold a row's column halves ([2 slots][2 halves][128 rows] float4)
constexpr uint32_t OFF_XCH = OFF_TM + 16;
constexpr uint32_t SMEM_BYTES = OFF_XCH + 2 * 4096 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// leading-byte offsets from the V and S_bf16 blocks to their e0 / z2 blocks:
// positive and within the descriptor's 14-bit field (16-byte units)
static_assert(OFF_E0 > slot_off(1) + S_SB && OFF_E0 + 64 - slot_off(0) - S_V < (16384u << 4),
              "descriptor offsets");

enum Bar {
  B_W = 0, B_LDQK = 1, B_LDV = 3, B_G1 = 5, B_G2 = 7, B_G3 = 9, B_E1A = 11, B_E12 = 13, B_E3 = 15,
  B_G2A = 17   // the score MMAs of G2 (Sc) alone
};

struct Args2 {
  CUtensorMap tq, tk, tv, tw, ty;   // ty: y rows, 32-row boxes
  const float* ws;   // [U][P-1][DP*D + DP] inclusive prefixes of segment states
  const float* init; // [U][DP*D + DP] initial state (continuation), same layout, or null
  float* S_out;
  float* z_out;
  const float* bias;
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int H, P, L, NT;
  int G;               // query heads per key/value head
  int seq;             // q, k, v, y are [B][n][H][D]
};

__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

// The bound of 384 threads caps registers at 168 per thread: warps 0, 4, 8
// (and 1, 5, 9) share one SM sub-partition's 16K registers.
// SM: softmax-over-features map, phi = [exp(h - c+); exp(-h - c-)] (no bias),
// the per-row offsets c+- = logsumexp(+-h) formed in the exponential phase.
template <bool SM>
__global__ void __launch_bounds__(384, 1) prefill_tc2_kernel(const __grid_constant__ Args2 A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* bq_s = reinterpret_cast<float*>(sm + OFF_BQ);
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TM);
  int* abort_flag = reinterpret_cast<int*>(sm + OFF_TM + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x / A.P;
  const int64_t kvu = kv_unit(unit, A.H, A.G);   // k, v of this query head
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int seg = blockIdx.x % A.P;
  const int h = (int)(unit % A.H);
  const int t_begin = seg * A.L;
  const int nt = min(A.NT, t_begin + A.L) - t_begin;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    mbar_init(bar(B_W), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_LDQK + s), 1);
      mbar_init(bar(B_LDV + s), 1);
      mbar_init(bar(B_G1 + s), 1);
      mbar_init(bar(B_G2 + s), 1);
      mbar_init(bar(B_G3 + s), 1);
      mbar_init(bar(B_E1A + s), 8);
      mbar_init(bar(B_E12 + s), 8);
      mbar_init(bar(B_E3 + s), 8);
      mbar_init(bar(B_G2A + s), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&A.tq);
    prefetch_tmap(&A.tk);
    prefetch_tmap(&A.tv);
    prefetch_tmap(&A.ty);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  for (int i = tid; i < 1024; i += kThreads) {
    // e0 block: logical column 0 of every row = 1; z2 blocks: zero until E1
    // writes columns (z_hi, z_lo) of their first chunk
    const int r = i >> 3, ch = i & 7;
    st_shared_v4(sb + OFF_E0 + sw128_chunk(r, ch), ch == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
  // W and the first two tiles into L2 while the kernels before this one
  // finish: a prefetch only warms the cache, so it may run before the wait
  // below (any later write to these rows still reaches L2 before the loads)
  if (warp == 8 && lane == 0) {
    tma_prefetch_3d(&A.tw, 0, 0, h);
    for (int i = 0; i < 2 && i < nt; ++i) {
      const int r0 = (t_begin + i) * TILE;
      tma_prefetch_rows(&A.tq, 0, r0, ub, uh, A.seq);
      tma_prefetch_rows(&A.tk, 0, r0, ub, kh, A.seq);
      tma_prefetch_rows(&A.tv, 0, r0, ub, kh, A.seq);
    }
  }
  // everything above touches only this CTA's shared memory and TMEM; the next
  // kernel may be scheduled now, and this one reads and writes global memory
  // only once the kernels before it have completed
  pdl_launch_dependents();
  pdl_wait();
  __syncthreads();

  auto load_qk = [&](int i) {
    const int s = i & 1;
    const int r0 = (t_begin + i) * TILE;
    const uint32_t base = sb + qk_off(s);
    mbar_expect_tx(bar(B_LDQK + s), 2 * 16384);
    tma_load_rows(base, &A.tq, bar(B_LDQK + s), 0, r0, ub, uh, A.seq);
    tma_load_rows(base + 16384, &A.tk, bar(B_LDQK + s), 0, r0, ub, kh, A.seq);
  };
  auto load_v = [&](int i) {
    const int s = i & 1;
    mbar_expect_tx(bar(B_LDV + s), 16384);
    tma_load_rows(sb + slot_off(s) + S_V, &A.tv, bar(B_LDV + s), 0, (t_begin + i) * TILE, ub,
                  kh, A.seq);
  };
  if (warp == 8 && lane == 0) {
    mbar_expect_tx(bar(B_W), 8192u);
    tma_load_3d(sb + OFF_W, &A.tw, bar(B_W), 0, 0, h);
    for (int i = 0; i < 2 && i < nt; ++i) {
      load_qk(i);
      load_v(i);
    }
  }
  for (int i = tid; i < D; i += kThreads)
    bq_s[i] = A.bias ? A.bias[(size_t)h * D + i] * kLog2e : 0.f;
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // initial state: the prefix of the preceding segments, the given initial
  // state (continuation, first segment) or zeros
  if (warp < 4) {
    const int f = 32 * warp + lane;  // feature = TMEM lane
    const float* prefix =
        seg > 0 ? A.ws + ((size_t)unit * (A.P - 1) + seg - 1) * (size_t)(DP * D + DP)
                : (A.init ? A.init + (size_t)unit * (DP * D + DP) : nullptr);
    uint32_t r[32];
    for (int c0 = 0; c0 < D; c0 += 32) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 v4 = prefix ? __ldcg(reinterpret_cast<const float4*>(prefix + ws_s_index(f, c0 + j, D)))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        r[j] = __float_as_uint(v4.x);
        r[j + 1] = __float_as_uint(v4.y);
        r[j + 2] = __float_as_uint(v4.z);
        r[j + 3] = __float_as_uint(v4.w);
      }
      tmem_st32(tmem + lane_base(warp) + TM_S + c0, r);
    }
    const float z0 = prefix ? __ldcg(prefix + (size_t)DP * D + f) : 0.f;
    uint32_t zr[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) zr[j] = 0u;
    zr[0] = __float_as_uint(z0);
    tmem_st16(tmem + lane_base(warp) + TM_S + 64, zr);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 8) {
    // ======================= producer =======================
    if (lane == 0) {
      constexpr uint32_t ID_H = idesc_bf16(128, D, 0, 1);
      constexpr uint32_t ID_SC = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t ID_SU = idesc_bf16(128, D + 16, 1, 1);   // [S z] += phiK^T [V 1]
      constexpr uint32_t ID_PV = idesc_bf16(128, D + 16, 0, 1);   // [O den]
      bool ok = mbar_wait(bar(B_W), 0, wp);
      // Descriptor bases: a k-step only moves the 14-bit start-address field
      // (address >> 4), so each MMA below is one 64-bit add plus the instruction.
      // MN-major B operands with N = 80 span two 64-column blocks: the second
      // block (e0 for V, z2 for S_bf16) sits one leading-byte offset further.
      struct SlotDesc { uint64_t q, k, pk, pm, v, sbf; };
      auto slot_desc = [&](int s2) {
        const uint32_t base = sb + slot_off(s2);
        SlotDesc d;
        d.q = smem_desc(sb + qk_off(s2), 16, 1024, 2);           // K-major, 32 B per k-step
        d.k = smem_desc(sb + qk_off(s2) + 16384, 16, 1024, 2);
        d.pk = smem_desc(base + S_PHK, 16, 1024, 2);      // phi(K) / P as K-major operand
        d.pm = smem_desc(base + S_PHK, 16384, 1024, 2);   // phi(K)^T as MN-major operand
        // MN-major, 2048 B per k-step; the second N block is e0 / z2 of this slot
        d.v = smem_desc(base + S_V, OFF_E0 - (slot_off(s2) + S_V), 1024, 2);
        d.sbf = smem_desc(base + S_SB, OFF_E0 + 32 * (1 + s2) - (slot_off(s2) + S_SB), 1024, 2);
        return d;
      };
      const SlotDesc sd0 = slot_desc(0), sd1 = slot_desc(1);
      const uint64_t dW = smem_desc(sb + OFF_W, D * 128, 1024, 2);
      // k-step offsets in 16-byte units: K-major inside 64-element panels, MN-major rows
      auto kmaj = [](int ks) { return (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2); };
      // descriptors of a slot picked field by field (a reference to one of the
      // two structs would put them in local memory)
      auto G1 = [&](int i) {
        const int s = i & 1;
        const uint64_t dq = s ? sd1.q : sd0.q, dk = s ? sd1.k : sd0.k;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          mma_ss(tmem + TM_Y(s), dq + 2 * ks, dW + 128 * ks, ID_H, ks > 0);
          mma_ss(tmem + TM_X(s), dk + 2 * ks, dW + 128 * ks, ID_H, ks > 0);
        }
        mma_commit(bar(B_G1 + s));
      };
      auto G2 = [&](int i) {
        const int s = i & 1;
        const uint64_t pk = s ? sd1.pk : sd0.pk, pm = s ? sd1.pm : sd0.pm;
        const uint64_t dv = s ? sd1.v : sd0.v;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tmem + TM_X(s), tmem + TM_Y(s) + ks * 8, pk + kmaj(ks), ID_SC, ks > 0);
        mma_commit(bar(B_G2A + s));   // E2 may read Sc while the state update runs
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ss(tmem + TM_S, pm + 128 * ks, dv + 128 * ks, ID_SU, 1);
        mma_commit(bar(B_G2 + s));
      };
      auto G3 = [&](int i) {
        const int s = i & 1;
        const uint64_t pk = s ? sd1.pk : sd0.pk, dv = s ? sd1.v : sd0.v;
        const uint64_t sbf = s ? sd1.sbf : sd0.sbf;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ss(tmem + TM_X(s), pk + kmaj(ks), dv + 128 * ks, ID_PV, ks > 0);
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tmem + TM_X(s), tmem + TM_Y(s) + ks * 8, sbf + 128 * ks, ID_PV, 1);
        mma_commit(bar(B_G3 + s));
      };
      // The groups run in the order the epilogue consumes them.  Its step i is
      // E2(i-1), E1(i), E3(i-1), so the producer's step i is
      //   G3(i-1)  once E2(i-1) is done
      //   G2(i)    once E1(i) is done and V(i) has landed
      //   G1(i+1)  once Q(i+1), K(i+1) have landed and E3(i-1) has freed the TMEM slot
      // Each wait is on the one barrier the next group needs (polled, bounded).
      if (ok && nt > 0) ok = mbar_wait_poll(bar(B_LDQK), 0, wp);
      if (ok && nt > 0) G1(0);
      for (int i = 0; i <= nt && ok; ++i) {
        if (i >= 1) {
          ok = mbar_wait_poll(bar(B_E12 + ((i - 1) & 1)), ((i - 1) >> 1) & 1, wp);
          if (!ok) break;
          G3(i - 1);
        }
        if (i < nt) {
          ok = mbar_wait_poll(bar(B_E1A + (i & 1)), (i >> 1) & 1, wp) &&
               mbar_wait_poll(bar(B_LDV + (i & 1)), (i >> 1) & 1, wp);
          if (!ok) break;
          G2(i);
        }
        if (i + 1 < nt) {
          const int j = i + 1;
          ok = mbar_wait_poll(bar(B_LDQK + (j & 1)), (j >> 1) & 1, wp) &&
               (j < 2 || mbar_wait_poll(bar(B_E3 + (j & 1)), ((j - 2) >> 1) & 1, wp));
          if (!ok) break;
          G1(j);
        }
      }
    }
  } else if (warp == 9) {
    // ======================= loader =======================
    //   LQK(i)  Q, K into stage i&1  once G1(i-2) has completed (H = X W read them)
    //   LV(i)   V into slot i&1      once G3(i-2) has completed (S += phi(K)^T V, P V done)
    if (lane == 0) {
      int nqk = nt < 2 ? nt : 2, nv = nqk;
      IdleClock clk;
      bool ok = true;
      while ((nqk < nt || nv < nt) && ok) {
        bool progress = false;
        if (nqk < nt && mbar_probe(bar(B_G1 + (nqk & 1)), ((nqk - 2) >> 1) & 1)) {
          load_qk(nqk++);
          progress = true;
        }
        if (nv < nt && mbar_probe(bar(B_G3 + (nv & 1)), ((nv - 2) >> 1) & 1)) {
          load_v(nv++);
          progress = true;
        }
        if (progress) {
          clk.progress();
        } else {
          ok = clk.idle(wp);
          __nanosleep(32);
        }
      }
    }
  } else {
    // ======================= epilogue warps =======================
    // All eight warps work on one phase at a time; phases of the two slots are
    // software-pipelined as E2(i-1), E1(i), E3(i-1) so that G3(i-1) runs under
    // E1(i), G2(i) under E3(i-1) and G1(i+1) under the next E2.  Warp w owns
    // TMEM lanes 32*(w%4).. (rows / features) and column half c = w / 4.
    const int c = warp >> 2;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lb = lane_base(warp);
    const int g = warp & 3;
    bool good = true;

    auto E1 = [&](int i) {
      const int s = i & 1;
      const uint32_t par = (i >> 1) & 1;
      const uint32_t base = sb + slot_off(s);
      const bool valid = (int64_t)(t_begin + i) * TILE + row < A.n;
      float2 oq = make_float2(0.f, 0.f), ok_ = make_float2(0.f, 0.f);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G1 + s), par, wp))) { good = false; return; }
      tc_fence_after();
      // H_Q and H_K columns [32c, 32c+32) of this warp's rows, one wait for both
      uint32_t hv[32], hk[32];
      tmem_ld32x2(tmem + lb + TM_Y(s) + 32 * c, hv, tmem + lb + TM_X(s) + 32 * c, hk);
      // in place: (h + b) log2(e), one FFMA each (the bias is stored pre-scaled and
      // re-read from shared memory every tile rather than held in registers)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 b4 = ld_shared_f4_volatile(sb + OFF_BQ + 4 * (32 * c + 4 * q));
        const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hv[4 * q + e] = __float_as_uint(fmaf(__uint_as_float(hv[4 * q + e]), kLog2e, bb[e]));
          hk[4 * q + e] = __float_as_uint(fmaf(__uint_as_float(hk[4 * q + e]), kLog2e, bb[e]));
        }
      }
      // softmax map: the row offsets c+- = log2 sum_l 2^(+-a_l), a = h log2 e, of
      // this row of Q and of K, each as max + log2 sum 2^(. - max).  The row's
      // 64 columns sit in two warps (c = 0, 1); each posts its partial maxima,
      // then its partial sums, in this slot's exchange area (slot i & 1: the
      // pair's barriers of E1(i + 1) order the reuse) and adds the partner's.
      float4 mx4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float4* xch = reinterpret_cast<float4*>(sm + OFF_XCH + s * 4096);
      if constexpr (SM) {
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = __uint_as_float(hv[j]), y = __uint_as_float(hk[j]);
          m0 = fmaxf(m0, x);
          m1 = fmaxf(m1, -x);
          m2 = fmaxf(m2, y);
          m3 = fmaxf(m3, -y);
        }
        mx4 = make_float4(m0, m1, m2, m3);
        xch[c * TILE + row] = mx4;
      }
      // phi(Q) overwrites H_Q in place, and phi(K) below the y slab E3(i-2)
      // staged in these rows of panel 0: wait for both warps of these lanes to
      // hold their H_Q columns and for the slab's store to have read it
      if (c == 0 && lane == 0 && i >= 2) tma_store_wait_read_all();
      __syncwarp();
      tc_fence_before();
      named_bar_sync(2 + g, 64);
      tc_fence_after();
      if constexpr (SM) {
        const float4 o = xch[(c ^ 1) * TILE + row];
        mx4 = make_float4(fmaxf(mx4.x, o.x), fmaxf(mx4.y, o.y), fmaxf(mx4.z, o.z),
                          fmaxf(mx4.w, o.w));
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = __uint_as_float(hv[j]), y = __uint_as_float(hk[j]);
          s0 += ex2_approx(x - mx4.x);
          s1 += ex2_approx(-x - mx4.y);
          s2 += ex2_approx(y - mx4.z);
          s3 += ex2_approx(-y - mx4.w);
        }
        named_bar_sync(2 + g, 64);   // the partner has read the maxima
        xch[c * TILE + row] = make_float4(s0, s1, s2, s3);
        named_bar_sync(2 + g, 64);
        const float4 o2 = xch[(c ^ 1) * TILE + row];
        // own + partner on both warps: the same sums (addition commutes)
        oq = make_float2(mx4.x + __log2f(s0 + o2.x), mx4.y + __log2f(s1 + o2.y));
        ok_ = make_float2(mx4.z + __log2f(s2 + o2.z), mx4.w + __log2f(s3 + o2.w));
      }
      // phi(Q): H_Q columns [32c, 32c+32) -> packed columns [16c, +16) (exp(+h))
      // and [32 + 16c, +16) (exp(-h)), one half at a time
#pragma unroll
      for (int sgn = 0; sgn < 2; ++sgn) {
        const float sg = sgn ? -1.f : 1.f;
        float oo = 0.f;
        if constexpr (SM) oo = sgn ? oq.y : oq.x;
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float a0 = __uint_as_float(hv[j]), a1 = __uint_as_float(hv[j + 1]);
          if constexpr (SM) pk[j / 2] = pack_bf16(ex2_approx(sg * a0 - oo), ex2_approx(sg * a1 - oo));
          else pk[j / 2] = pack_bf16(ex2_approx(sg * a0), ex2_approx(sg * a1));
        }
        tmem_st16(tmem + lb + TM_Y(s) + 32 * sgn + 16 * c, pk);
      }
      // phi(K): features [32c, +32) -> panel 0 chunks [4c, +4); [64 + 32c, +32) -> panel 1
      {
        const uint32_t (&hv)[32] = hk;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t wpos[4], wneg[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * q4 + 2 * e;
            const float a0 = __uint_as_float(hv[j]), a1 = __uint_as_float(hv[j + 1]);
            if constexpr (SM) {
              wpos[e] = valid ? pack_bf16(ex2_approx(a0 - ok_.x), ex2_approx(a1 - ok_.x)) : 0u;
              wneg[e] = valid ? pack_bf16(ex2_approx(-a0 - ok_.y), ex2_approx(-a1 - ok_.y)) : 0u;
            } else {
              wpos[e] = valid ? pack_bf16(ex2_approx(a0), ex2_approx(a1)) : 0u;
              wneg[e] = valid ? pack_bf16(ex2_approx(-a0), ex2_approx(-a1)) : 0u;
            }
          }
          st_shared_v4(base + S_PHK + sw128_chunk(row, 4 * c + q4), wpos[0], wpos[1], wpos[2],
                       wpos[3]);
          st_shared_v4(base + S_PHK + 16384 + sw128_chunk(row, 4 * c + q4), wneg[0], wneg[1],
                       wneg[2], wneg[3]);
        }
      }
      // S_bf16 and z of the tokens before this tile; G2(i) may run only after this
      if (i > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G2 + ((i - 1) & 1)), ((i - 1) >> 1) & 1, wp))) {
          good = false;
          return;
        }
        tc_fence_after();
      }
      {
        uint32_t sv[32], z0 = 0u, z1;
        // feature `row`, columns [32c, +32); warps of column half 0 also take z
        if (c == 0) tmem_ld32_ld2(tmem + lb + TM_S, sv, tmem + lb + TM_S + 64, z0, z1);
        else tmem_ld32(tmem + lb + TM_S + 32, sv);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = 8 * q4;
          st_shared_v4(base + S_SB + sw128_chunk(row, 4 * c + q4),
                       pack_bf16(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                       pack_bf16(__uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3])),
                       pack_bf16(__uint_as_float(sv[j + 4]), __uint_as_float(sv[j + 5])),
                       pack_bf16(__uint_as_float(sv[j + 6]), __uint_as_float(sv[j + 7])));
        }
        if (c == 0) {
          // z of feature `row` as z_hi + z_lo (both bf16) in columns 0, 1 of its z2 row
          // (G3(i-2), the last reader of this slot's z2 block, completed before E3(i-2))
          const float z = __uint_as_float(z0);
          const float zl = z - __bfloat162float(__float2bfloat16_rn(z));
          st_shared_v4(sb + OFF_E0 + sw128_chunk(row, 2 + 2 * s), pack_bf16(z, zl), 0u, 0u, 0u);
        }
      }
      tmem_st_wait();
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E1A + s));
    };

    auto E2 = [&](int i) {
      const int s = i & 1;
      const uint32_t par = (i >> 1) & 1;
      const uint32_t base = sb + slot_off(s);
      // Sc is complete once the score MMAs of G2 are; the state update of G2
      // still reads phi(K) from the panels P goes to, so P is built in registers
      // first and stored once all of G2 has completed
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G2A + s), par, wp))) { good = false; return; }
      tc_fence_after();
      uint32_t w[32];
      const bool zero = c == 1 && g < 2;   // keys 64..127 of rows 0..63: above the diagonal
      if (!zero) {
        const bool diag = (c == 0) == (g < 2);   // the 64 x 64 blocks on the diagonal
        uint32_t sc[64];
        tmem_ld64(tmem + lb + TM_X(s) + 64 * c, sc);   // keys [64c, +64)
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          const int key = 64 * c + j;
          float a0 = __uint_as_float(sc[j]);
          float a1 = __uint_as_float(sc[j + 1]);
          if (diag) {
            a0 = key <= row ? a0 : 0.f;
            a1 = key + 1 <= row ? a1 : 0.f;
          }
          w[j / 2] = pack_bf16(a0, a1);
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G2 + s), par, wp))) { good = false; return; }
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 8; ++q)   // keys [64c + 8q, +8) -> chunk q of panel c
        st_shared_v4(base + S_PHK + c * 16384 + sw128_chunk(row, q), zero ? 0u : w[4 * q],
                     zero ? 0u : w[4 * q + 1], zero ? 0u : w[4 * q + 2], zero ? 0u : w[4 * q + 3]);
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E12 + s));
    };

    auto E3 = [&](int i) {
      const int s = i & 1;
      const uint32_t par = (i >> 1) & 1;
      const int64_t r0 = (int64_t)(t_begin + i) * TILE;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G3 + s), par, wp))) { good = false; return; }
      tc_fence_after();
      uint32_t ov[32], d0, d1;
      // columns [32c, +32) of O; 64, 65: rowsum(P) + phi(q) . z_hi, phi(q) . z_lo
      tmem_ld32_ld2(tmem + lb + TM_X(s) + 32 * c, ov, tmem + lb + TM_X(s) + 64, d0, d1);
      const float inv = __frcp_rn(__uint_as_float(d0) + __uint_as_float(d1));
      // y row `row`, columns [32c, +32) -> panel 0 of the P buffer (SW128 rows)
      const uint32_t ys = sb + slot_off(s) + S_PHK;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int j = 8 * q4;
        st_shared_v4(ys + sw128_chunk(row, 4 * c + q4),
                     pack_bf16(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv),
                     pack_bf16(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv),
                     pack_bf16(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv),
                     pack_bf16(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv));
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar_sync(2 + g, 64);   // rows 32g.. of both column halves are staged
      // one store per 32-row slab; the map clips rows past n, and a slab that
      // starts past n is not stored at all
      if (c == 0 && lane == 0 && r0 + 32 * g < A.n) {
        tma_store_rows(&A.ty, ys + 32 * g * 128, 0, (int)r0 + 32 * g, ub, uh, A.seq);
        tma_store_commit();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E3 + s));
    };

    for (int step = 0; step <= nt && good; ++step) {
      if (step >= 1) E2(step - 1);
      if (step < nt && good) E1(step);
      if (step >= 1 && good) E3(step - 1);
    }
    if (c == 0 && lane == 0) tma_store_wait_all();   // y written before the CTA retires
  }

  // ---- export the final state of the last segment ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (A.S_out && seg == A.P - 1 && warp < 4 && !*(volatile int*)abort_flag) {
    const int f = 32 * warp + lane;
    uint32_t sv[64];
    tmem_ld64(tmem + lane_base(warp) + TM_S, sv);
    float4* dst = reinterpret_cast<float4*>(A.S_out + ((size_t)unit * DP + f) * D);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      dst[j] = make_float4(__uint_as_float(sv[4 * j]), __uint_as_float(sv[4 * j + 1]),
                           __uint_as_float(sv[4 * j + 2]), __uint_as_float(sv[4 * j + 3]));
    uint32_t z0, z1;
    tmem_ld2(tmem + lane_base(warp) + TM_S + 64, z0, z1);
    A.z_out[(size_t)unit * DP + f] = __uint_as_float(z0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}


}  // namespace

// Output pass of the d = 64 Hedgehog prefill (two tiles in flight per CTA) for a
// feature map shared by queries and keys.
cudaError_t launch_prefill_out_d64(const Problem& p, const TcPlan& pl, const void* q,
                                   const void* k, const void* v, void* y, float* S_out,
                                   float* z_out, const void* ws, const float* init,
                                   int* dev_status, cudaStream_t s) {
  Args2 a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  if (p.Wk) return cudaErrorInvalidValue;  // one map shared by queries and keys
  const int Hkv = p.H / p.G;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  bool ok = make_rows_map(&a.tq, q, D, p.n, p.H, p.B, 64, TILE, sw, p.seq_major) &&
            make_rows_map(&a.tk, k, D, p.n, Hkv, p.B, 64, TILE, sw, p.seq_major) &&
            make_rows_map(&a.tv, v, D, p.n, Hkv, p.B, 64, TILE, sw, p.seq_major) &&
            make_plane_map(&a.tw, p.Wq, D, D, p.H, 64, D, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_rows_map(&a.ty, y, D, p.n, p.H, p.B, 64, 32, sw, p.seq_major);
  if (!ok) return cudaErrorInvalidValue;
  a.ws = reinterpret_cast<const float*>(ws);
  a.init = init;
  a.S_out = S_out;
  a.z_out = z_out;
  a.bias = p.bq;
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.H = p.H;
  a.P = pl.P;
  a.L = pl.L;
  a.NT = pl.NT;
  a.G = p.G;
  a.seq = p.seq_major;
  auto kern = p.softmax ? prefill_tc2_kernel<true> : prefill_tc2_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)(U * pl.P)), dim3(kThreads), SMEM_BYTES, s, a);
}

}  // namespace hh
