// Segment-state pass of the chunked prefill on the 5th-generation tensor cores.
//
// For each segment of a (batch, head) sequence it writes
//   S_seg = sum_j phi(k_j)^T v_j   and   z_seg = sum_j phi(k_j)
// over the segment's tokens: the running sums of "Complexity Analysis" in
// "The Hedgehog & the Porcupine" summary ("2. Context and Motivation", paper Eq. 2), for the
// Hedgehog map ("The Hedgehog MLP Feature Map", Choices 1 and 3) or the
// degree-2 Taylor map ("The Taylor Exponential as a Bridge Result").  The
// output pass starts segment s from the inclusive scan of segments < s.
//
// Three kernels, one CTA per segment each: state_tc_kernel (Hedgehog,
// d = 64), state_t128_kernel (Hedgehog, d = 128, phi(K) kept in TMEM) and
// state_taylor_kernel (Taylor, d = 16).
//
// state_tc_kernel: warp 8 (one lane) issues TMA loads and MMAs; warps 0-7
// build phi(K) (warp w owns TMEM lanes 32*(w%4).. and column half w/4).
// Per 128-token tile t:
//   G1(t): H_K = K_t W into TMEM
//   E1(t): H_K -> registers ("H read"), exponentials, then phi(K_t) ->
//          128B-swizzled shared panels once G2(t-1) has consumed the old ones
//   G2(t): S += phi(K_t)^T V_t,  z += phi(K_t)^T 1         (tcgen05)
// G1(t+1) is issued as soon as E1(t) has read H_K, so it and G2(t) run
// under the exponentials of the next tile.  K and V are double-buffered.
// Every mbarrier wait is bounded in time (tc_ptx.cuh).

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

constexpr int TILE = 128;
constexpr int kThreads = 288;  // 8 feature warps + 1 issue warp

// Hedgehog, d in {64, 128}: 2d features, S rows as 128-feature M blocks.
template <int D>
struct SCfg {
  static constexpr int DPP = 2 * D;
  static constexpr int NMB = 2 * D / 128;
  static constexpr int NV = D == 128 ? 1 : 2;                  // V stages
  static constexpr uint32_t TM_S = 0;                          // NMB x [128 x D]
  static constexpr uint32_t TM_Z = NMB * D;                    // NMB x [128 x 16]
  static constexpr uint32_t TM_H = D == 64 ? 192 : 384;        // [128 x D]
  static constexpr uint32_t TM_COLS = D == 64 ? 256 : 512;
  static_assert(TM_Z + 16 * NMB <= TM_H && TM_H + D <= TM_COLS, "TMEM layout");
  static constexpr uint32_t XT = TILE * D * 2;                 // one K or V tile
  static constexpr uint32_t OFF_W = 0;
  static constexpr uint32_t OFF_ONES = D * D * 2;              // [128 x 16] bf16 ones, SW32
  static constexpr uint32_t OFF_K = OFF_ONES + 4096;
  static constexpr uint32_t OFF_V = OFF_K + 2 * XT;
  static constexpr uint32_t OFF_PHK = OFF_V + NV * XT;         // [2D/64] panels of 16 KB
  static constexpr uint32_t OFF_END = OFF_PHK + (2 * D / 64) * 16384;
};

enum {
  SB_W = 0, SB_LDK = 1 /* 2 */, SB_LDV = 3 /* 2 */, SB_G1 = 5, SB_HREAD = 6, SB_E1 = 7,
  SB_G2 = 8, SB_COUNT = 9
};

template <int D>
struct SSmem {
  using C = SCfg<D>;
  static constexpr uint32_t OFF_B = C::OFF_END;                // bias float[128]
  static constexpr uint32_t OFF_BAR = OFF_B + 512;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8 * SB_COUNT; // tmem base, abort flag
  static constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;      // + alignment slack
  static_assert(ALLOC <= 227 * 1024, "shared memory");
};

struct StateArgs {
  CUtensorMap tk, tv, tw;
  const __nv_bfloat16* kraw;   // k itself (the Taylor pass reads its rows directly)
  float* ws;          // [U][(P-1)*M][DPP*D + DPP]: S (ws_s_index layout) then z
  const float* bias;  // [H][D] of the key map (Hedgehog) or null
  const float2* off;  // [U][NT*128] softmax-map offsets of the keys (log2 units) or null
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int H, P, L, NT;
  int M;              // pieces per segment: each CTA sums one piece of a segment
  int G;              // query heads per key/value head
  int seq;            // k, v are [B][n][Hkv][D]
};

// The piece of a segment this CTA sums: piece j of segment s covers tiles
// [s L + j Lp, s L + (j + 1) Lp) with Lp = ceil(L / M), cut at the segment's
// end (a piece past it is empty and exports zeros).  `index` orders the
// pieces of a unit by position, which is the order the scan adds them in.
struct StatePiece {
  int64_t unit;
  int index, t_begin, nt;
};
__device__ __forceinline__ StatePiece state_piece(const StateArgs& A) {
  StatePiece r;
  if (A.M == 1) {   // one piece per segment
    r.unit = blockIdx.x / (A.P - 1);
    r.index = blockIdx.x % (A.P - 1);
    r.t_begin = r.index * A.L;
    r.nt = min(A.NT, r.t_begin + A.L) - r.t_begin;
    return r;
  }
  const int npc = (A.P - 1) * A.M;
  r.unit = blockIdx.x / npc;
  r.index = blockIdx.x % npc;
  const int seg = r.index / A.M, j = r.index % A.M;
  const int lp = (A.L + A.M - 1) / A.M;
  const int b = seg * A.L + min(j * lp, A.L);
  const int e = min(seg * A.L + min((j + 1) * lp, A.L), A.NT);
  r.t_begin = b;
  r.nt = max(0, e - b);
  return r;
}

__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) state_tc_kernel(const __grid_constant__ StateArgs A) {
  using C = SCfg<D>;
  using SM = SSmem<D>;
  constexpr int NV = C::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* b_s = reinterpret_cast<float*>(sm + SM::OFF_B);
  const uint32_t bars = sb + SM::OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + SM::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const StatePiece pc = state_piece(A);
  const int64_t unit = pc.unit;
  const int64_t kvu = kv_unit(unit, A.H, A.G);   // k, v of this query head
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int h = (int)(unit % A.H);
  const int t_begin = pc.t_begin;
  const int nt = pc.nt;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    for (int b = 0; b < SB_COUNT; ++b)
      mbar_init(bar(b), (b == SB_HREAD || b == SB_E1) ? 8 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // W and the first two tiles into L2 while the kernels before this one
  // finish (a prefetch only warms the cache, so it may precede the wait)
  if (warp == 8 && lane == 0 && nt > 0)
    for (int x = 0; x < (D + 63) / 64; ++x) {
      tma_prefetch_3d(&A.tw, 64 * x, 0, h);
      for (int i = 0; i < 2 && i < nt; ++i) {
        tma_prefetch_rows(&A.tk, 64 * x, (t_begin + i) * TILE, ub, kh, A.seq);
        tma_prefetch_rows(&A.tv, 64 * x, (t_begin + i) * TILE, ub, kh, A.seq);
      }
    }
  // global memory is touched only after the kernels before this one have
  // completed; only then may the next kernel be scheduled, so the kernels
  // after this one in a call may read the call's inputs before their own wait
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();

  auto load_k = [&](int i) {
    const uint32_t dst = sb + C::OFF_K + (i & 1) * C::XT;
    const uint32_t b = bar(SB_LDK + (i & 1));
    mbar_expect_tx(b, C::XT);
    for (int x = 0; x < (D + 63) / 64; ++x)
      tma_load_rows(dst + x * 16384, &A.tk, b, 64 * x, (t_begin + i) * TILE, ub,
                    kh, A.seq);
  };
  auto load_v = [&](int i) {
    const uint32_t dst = sb + C::OFF_V + (i % NV) * C::XT;
    const uint32_t b = bar(SB_LDV + (i % NV));
    mbar_expect_tx(b, C::XT);
    for (int x = 0; x < (D + 63) / 64; ++x)
      tma_load_rows(dst + x * 16384, &A.tv, b, 64 * x, (t_begin + i) * TILE, ub,
                    kh, A.seq);
  };
  if (warp == 8 && lane == 0 && nt > 0) {
    mbar_expect_tx(bar(SB_W), D * D * 2);
    for (int x = 0; x < D / 64; ++x)
      tma_load_3d(sb + C::OFF_W + x * (D * 128), &A.tw, bar(SB_W), 64 * x, 0, h);
    load_k(0);
    load_v(0);
    if (nt > 1) {
      load_k(1);
      if (NV == 2) load_v(1);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  for (int i = tid; i < D; i += kThreads) b_s[i] = A.bias ? A.bias[(size_t)h * D + i] : 0.f;
  // ones operand of the z MMA ([128 tokens x 16] bf16)
  for (int i = tid; i < 4096 / 16; i += kThreads)
    st_shared_v4(sb + C::OFF_ONES + 16 * i, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // S = 0, z = 0 (lanes = features)
  if (warp < 4) {
    uint32_t zr[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) zr[j] = 0u;
    for (int mb = 0; mb < C::NMB; ++mb) {
      for (int c0 = 0; c0 < D; c0 += 16)
        tmem_st16(tmem + lane_base(warp) + C::TM_S + mb * D + c0, zr);
      tmem_st16(tmem + lane_base(warp) + C::TM_Z + 16 * mb, zr);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 8) {
    // ======================= issue warp =======================
    if (lane == 0 && nt > 0) {
      constexpr uint32_t ID_H = idesc_bf16(128, D, 0, 1);   // K[K-major] W[MN-major]
      constexpr uint32_t ID_SU = idesc_bf16(128, D, 1, 1);  // phiK^T[MN] V[MN]
      constexpr uint32_t ID_Z = idesc_bf16(128, 16, 1, 1);  // phiK^T[MN] ones[MN]
      auto g1 = [&](int i) {
        const uint32_t kb = sb + C::OFF_K + (i & 1) * C::XT;
        // descriptor bases; a k-step only moves the start-address field (16-byte units)
        const uint64_t dk = smem_desc(kb, 16, 1024, 2);
        const uint64_t dw = smem_desc(sb + C::OFF_W, D * 128, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + C::TM_H, dk + (ks / 4) * 1024 + (ks % 4) * 2, dw + ks * 128, ID_H, ks > 0);
        mma_commit(bar(SB_G1));
      };
      bool ok = mbar_wait_poll(bar(SB_W), 0, wp) && mbar_wait_poll(bar(SB_LDK), 0, wp);
      tc_fence_after();
      if (ok) g1(0);
      for (int i = 0; i < nt && ok; ++i) {
        if (i + 1 < nt) {
          // H_K is free once every feature warp has read H_K(i)
          ok = mbar_wait_poll(bar(SB_LDK + ((i + 1) & 1)), ((i + 1) >> 1) & 1, wp) &&
               mbar_wait_poll(bar(SB_HREAD), i & 1, wp);
          if (!ok) break;
          tc_fence_after();
          g1(i + 1);
        }
        ok = mbar_wait_poll(bar(SB_E1), i & 1, wp) &&
             mbar_wait_poll(bar(SB_LDV + (i % NV)), (i / NV) & 1, wp);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vb = sb + C::OFF_V + (i % NV) * C::XT;
        const uint64_t dphk = smem_desc(sb + C::OFF_PHK, 16384, 1024, 2);
        const uint64_t dv = smem_desc(vb, TILE * 128, 1024, 2);
        const uint64_t dones = smem_desc(sb + C::OFF_ONES, 16, 256, 6);
#pragma unroll
        for (int mb = 0; mb < C::NMB; ++mb)
#pragma unroll
          for (int ks = 0; ks < TILE / 16; ++ks) {
            const uint64_t a = dphk + (2 * mb) * 1024 + ks * 128;
            mma_ss(tmem + C::TM_S + mb * D, a, dv + ks * 128, ID_SU, 1);
            mma_ss(tmem + C::TM_Z + 16 * mb, a, dones + ks * 32, ID_Z, 1);
          }
        mma_commit(bar(SB_G2));
        // K stage i&1: G1(i) is done with it
        if (i + 2 < nt) load_k(i + 2);
        if (NV == 2) {
          // V stage (i+1)&1 held V(i-1), consumed by G2(i-1) (E1(i) waited for it)
          if (i + 1 < nt && i + 1 >= 2) load_v(i + 1);
        } else if (i + 1 < nt) {
          ok = mbar_wait(bar(SB_G2), i & 1, wp);
          if (ok) load_v(i + 1);
        }
      }
      if (!ok) *(volatile int*)abort_flag = 1;
    }
  } else {
    // ======================= feature warps =======================
    const int c = warp >> 2;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t phk = sb + C::OFF_PHK;
    for (int i = 0; i < nt; ++i) {
      const bool valid = (int64_t)(t_begin + i) * TILE + row < A.n;
      constexpr int HC = D / 2;  // H columns of this warp's half
      // softmax map: phi = [exp(h - c+); exp(-h - c-)], offsets in log2 units
      float2 o = make_float2(0.f, 0.f);
      if (A.off && valid)
        o = A.off[(size_t)unit * A.NT * TILE + (size_t)(t_begin + i) * TILE + row];
      if (!__all_sync(0xffffffffu, mbar_wait(bar(SB_G1), i & 1, wp))) break;
      tc_fence_after();
      uint32_t hv[HC];
      if constexpr (HC == 64) tmem_ld64(tmem + lane_base(warp) + C::TM_H + HC * c, hv);
      else tmem_ld32(tmem + lane_base(warp) + C::TM_H + HC * c, hv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SB_HREAD));
      uint32_t wpos[HC / 2], wneg[HC / 2];
#pragma unroll
      for (int j = 0; j < HC; j += 2) {
        const float h0 = __uint_as_float(hv[j]) + b_s[HC * c + j];
        const float h1 = __uint_as_float(hv[j + 1]) + b_s[HC * c + j + 1];
        wpos[j / 2] = valid ? pack_bf16(ex2_approx(fmaf(h0, kLog2e, -o.x)),
                                        ex2_approx(fmaf(h1, kLog2e, -o.x)))
                            : 0u;
        wneg[j / 2] = valid ? pack_bf16(ex2_approx(fmaf(-h0, kLog2e, -o.y)),
                                        ex2_approx(fmaf(-h1, kLog2e, -o.y)))
                            : 0u;
      }
      // the panels are free once G2(i-1) has read them
      if (i > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(SB_G2), (i - 1) & 1, wp))) break;
#pragma unroll
      for (int q = 0; q < HC / 8; ++q) {
        const int fp = HC * c + 8 * q;      // positive feature of this 16-byte chunk
        const int fn = D + HC * c + 8 * q;  // its negative twin
        st_shared_v4(phk + (fp / 64) * 16384 + sw128_chunk(row, (fp % 64) / 8), wpos[4 * q],
                     wpos[4 * q + 1], wpos[4 * q + 2], wpos[4 * q + 3]);
        st_shared_v4(phk + (fn / 64) * 16384 + sw128_chunk(row, (fn % 64) / 8), wneg[4 * q],
                     wneg[4 * q + 1], wneg[4 * q + 2], wneg[4 * q + 3]);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SB_E1));
    }
  }

  // ---- export this segment's S and z ----
  tc_fence_before();
  __syncthreads();
  if (nt > 0 && !*(volatile int*)abort_flag) mbar_wait(bar(SB_G2), (nt - 1) & 1, wp);
  tc_fence_after();
  __syncthreads();
  if (warp < 8 && !*(volatile int*)abort_flag) {
    const int c = warp >> 2;
    float* dst = A.ws + ((size_t)unit * (A.P - 1) * A.M + pc.index) * ((size_t)C::DPP * D + C::DPP);
    for (int mb = c; mb < C::NMB; mb += 2) {
      const int f = mb * 128 + 32 * (warp & 3) + lane;
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t sv[16];
        tmem_ld16(tmem + lane_base(warp) + C::TM_S + mb * D + c0, sv);
        if (f < C::DPP) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(dst + ws_s_index(f, c0 + 4 * q, D)) =
                make_float4(__uint_as_float(sv[4 * q]), __uint_as_float(sv[4 * q + 1]),
                            __uint_as_float(sv[4 * q + 2]), __uint_as_float(sv[4 * q + 3]));
        }
      }
      uint32_t zv[16];
      tmem_ld16(tmem + lane_base(warp) + C::TM_Z + 16 * mb, zv);
      if (f < C::DPP) dst[(size_t)C::DPP * D + f] = __uint_as_float(zv[0]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------------------
// Hedgehog d = 128: transposed form.  H_K^T = W^T K_t^T lands in TMEM with the
// 128 hidden units on the lanes and the tile's tokens on the columns; the
// feature warps overwrite it in place with phi(K_t)^T as bf16 pairs, which is
// directly the A operand of
//   S[+/-] += phi(K_t)^T[+/-] V_t     (A from TMEM, M = 128 features)
// so phi(K) never goes through shared memory, and z is a per-thread running
// sum over the thread's tokens.  Two H buffers let G1(t+1) run while the
// feature warps work on tile t.  Warps 0-15 build the features (warp w: TMEM
// lane quarter w % 4, token quarter w / 4 of the tile: the exponential phase
// is latency-bound, so more warps with fewer tokens each finish it sooner);
// warp 16 issues the MMAs, warp 17 the loads.
// Packed layout of one H buffer after the feature phase: the 32 tokens of
// quarter q occupy columns [32 q, +32) before and after, exp(+h) pairs in
// [32 q, +16) and exp(-h) pairs in [32 q + 16, +16), so each warp rewrites
// only the columns it has read.
// ---------------------------------------------------------------------------
namespace t128 {
constexpr int D = 128;
constexpr uint32_t XT = TILE * D * 2;                  // 32 KB
constexpr uint32_t OFF_W = 0;                          // W: 2 panels [128 i x 64 j]
constexpr uint32_t OFF_K = 32768;                      // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * XT;             // 2 stages
constexpr uint32_t OFF_ZX = OFF_V + 2 * XT;            // float[4][256] z exchange
constexpr uint32_t OFF_OX = OFF_ZX + 4096;             // float2[2][128] softmax-map offsets
constexpr uint32_t OFF_BAR = OFF_OX + 2048;
enum { B_W = 0, B_LDK = 1, B_LDV = 3, B_G1 = 5, B_E1 = 7, B_G2 = 9, B_COUNT = 11 };
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;
static_assert(ALLOC <= 227 * 1024, "shared memory");
constexpr uint32_t TM_S = 0;                           // S+ [0,128), S- [128,256)
__host__ __device__ constexpr uint32_t TM_H(int b) { return 256 + 128 * b; }
constexpr int kFeat = 16;                              // feature warps 0-15
constexpr int kMmaWarp = kFeat, kLoadWarp = kFeat + 1;
constexpr int kThreads = 32 * (kFeat + 2);
}  // namespace t128

// The bound of 640 threads caps registers at 96 per thread: five warps (0, 4,
// 8, 12, 16 and 1, 5, 9, 13, 17) share one SM sub-partition's registers.
__global__ void __launch_bounds__(640, 1) state_t128_kernel(const __grid_constant__ StateArgs A) {
  using namespace t128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + OFF_MISC + 4);
  float* zx = reinterpret_cast<float*>(sm + OFF_ZX);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const StatePiece pc = state_piece(A);
  const int64_t unit = pc.unit;
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int h = (int)(unit % A.H);
  const int t_begin = pc.t_begin;
  const int nt = pc.nt;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b)
      mbar_init(bar(b), (b == B_E1 || b == B_E1 + 1) ? kFeat : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // W and the first two tiles into L2 while the kernels before this one
  // finish (a prefetch only warms the cache, so it may precede the wait)
  if (warp == kLoadWarp && lane == 0 && nt > 0) {
    for (int x = 0; x < 2; ++x) {
      tma_prefetch_3d(&A.tw, 64 * x, 0, h);
      for (int i = 0; i < 2 && i < nt; ++i) {
        tma_prefetch_rows(&A.tk, 64 * x, (t_begin + i) * TILE, ub, kh, A.seq);
        tma_prefetch_rows(&A.tv, 64 * x, (t_begin + i) * TILE, ub, kh, A.seq);
      }
    }
  }
  // global memory is touched only after the kernels before this one have
  // completed; only then may the next kernel be scheduled, so the kernels
  // after this one in a call may read the call's inputs before their own wait
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  auto load_k = [&](int i) {
    const uint32_t dst = sb + OFF_K + (i & 1) * XT, b = bar(B_LDK + (i & 1));
    mbar_expect_tx(b, XT);
    for (int x = 0; x < 2; ++x)
      tma_load_rows(dst + x * 16384, &A.tk, b, 64 * x, (t_begin + i) * TILE, ub,
                    kh, A.seq);
  };
  // V(i) (and, for the softmax map, the tile's per-token offsets, whose smem
  // buffer is free for the same reason as V's: E1(i-2) and G2(i-2) are done)
  auto load_v = [&](int i) {
    const uint32_t dst = sb + OFF_V + (i & 1) * XT, b = bar(B_LDV + (i & 1));
    mbar_expect_tx(b, XT + (A.off ? TILE * 8 : 0));
    for (int x = 0; x < 2; ++x)
      tma_load_rows(dst + x * 16384, &A.tv, b, 64 * x, (t_begin + i) * TILE, ub,
                    kh, A.seq);
    if (A.off)
      bulk_load(sb + OFF_OX + (i & 1) * TILE * 8,
                A.off + (size_t)unit * A.NT * TILE + (size_t)(t_begin + i) * TILE, TILE * 8, b);
  };
  if (warp == kLoadWarp && lane == 0 && nt > 0) {
    mbar_expect_tx(bar(B_W), D * D * 2);
    for (int x = 0; x < 2; ++x) tma_load_3d(sb + OFF_W + x * 16384, &A.tw, bar(B_W), 64 * x, 0, h);
    for (int i = 0; i < 2 && i < nt; ++i) {
      load_k(i);
      load_v(i);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < kFeat) {   // S = 0: warp w clears lane quarter w % 4, columns [64 (w / 4), +64)
    uint32_t zr[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) zr[j] = 0u;
    const uint32_t t0 = tmem + lane_base(warp) + TM_S + 64 * (warp >> 2);
    tmem_st32(t0, zr);
    tmem_st32(t0 + 32, zr);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  float zp = 0.f, zn = 0.f;   // this thread's share of z (hidden unit j, tokens of its quarter)
  if (warp == kMmaWarp) {
    // ======================= MMA issuer =======================
    if (lane == 0 && nt > 0) {
      constexpr uint32_t ID_H = idesc_bf16(128, 128, 1, 0);   // W^T[MN-major] K^T[K-major]
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 1);   // phiK^T[TMEM] V[MN-major]
      auto g1 = [&](int i) {
        const uint32_t kb = sb + OFF_K + (i & 1) * XT;
        // descriptor bases; a k-step only moves the start-address field (16-byte units)
        const uint64_t dw = smem_desc(sb + OFF_W, 16384, 1024, 2);
        const uint64_t dk = smem_desc(kb, 16, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + TM_H(i & 1), dw + ks * 128, dk + (ks >> 2) * 1024 + (ks & 3) * 2, ID_H,
                 ks > 0);
        mma_commit(bar(B_G1 + (i & 1)));
      };
      bool ok = mbar_wait_poll(bar(B_W), 0, wp) && mbar_wait_poll(bar(B_LDK), 0, wp);
      tc_fence_after();
      if (ok) g1(0);
      for (int i = 0; i < nt && ok; ++i) {
        if (i + 1 < nt) {
          // H buffer (i+1)&1 held phi(i-1), the A operand of G2(i-1)
          ok = mbar_wait_poll(bar(B_LDK + ((i + 1) & 1)), ((i + 1) >> 1) & 1, wp) &&
               (i == 0 || mbar_wait_poll(bar(B_G2 + ((i - 1) & 1)), ((i - 1) >> 1) & 1, wp));
          if (!ok) break;
          tc_fence_after();
          g1(i + 1);
        }
        ok = mbar_wait_poll(bar(B_E1 + (i & 1)), (i >> 1) & 1, wp) &&
             mbar_wait_poll(bar(B_LDV + (i & 1)), (i >> 1) & 1, wp);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vb = sb + OFF_V + (i & 1) * XT;
        const uint64_t dv = smem_desc(vb, 16384, 1024, 2);
        const uint32_t th = tmem + TM_H(i & 1);
        // k-step ks covers tokens [16 ks, +16): quarter ks / 2, half ks % 2 of it
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int ks = 0; ks < TILE / 16; ++ks)
            mma_ts(tmem + TM_S + 128 * mb, th + 32 * (ks >> 1) + 8 * (ks & 1) + 16 * mb,
                   dv + ks * 128, ID_S, 1);
        mma_commit(bar(B_G2 + (i & 1)));
      }
      if (!ok) *(volatile int*)abort_flag = 1;
    }
  } else if (warp == kLoadWarp) {
    // ======================= loader =======================
    //   K(i) into stage i&1 once G1(i-2) has read K(i-2); V(i) once G2(i-2) has read V(i-2)
    if (lane == 0) {
      int nk = nt < 2 ? nt : 2, nv = nk;
      IdleClock clk;
      bool alive = true;
      while ((nk < nt || nv < nt) && alive) {
        bool progress = false;
        if (nk < nt && mbar_probe(bar(B_G1 + (nk & 1)), ((nk - 2) >> 1) & 1)) {
          load_k(nk++);
          progress = true;
        }
        if (nv < nt && mbar_probe(bar(B_G2 + (nv & 1)), ((nv - 2) >> 1) & 1)) {
          load_v(nv++);
          progress = true;
        }
        if (progress) clk.progress();
        else alive = clk.idle(wp);
      }
    }
  } else {
    // ======================= feature warps =======================
    // warp w: hidden unit j = 32 (w % 4) + lane (TMEM lane), tokens [32 q, +32) of the tile
    const int q = warp >> 2;
    const int j = 32 * (warp & 3) + lane;
    const uint32_t lb = lane_base(warp);
    const float bj = A.bias ? A.bias[(size_t)h * D + j] * kLog2e : 0.f;
    const float2* ox = reinterpret_cast<const float2*>(sm + OFF_OX);
    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G1 + b), (i >> 1) & 1, wp))) break;
      // softmax map: the offsets of tile i landed with V(i)
      if (A.off && !__all_sync(0xffffffffu, mbar_wait(bar(B_LDV + b), (i >> 1) & 1, wp))) break;
      tc_fence_after();
      const uint32_t tq = tmem + lb + TM_H(b) + 32 * q;
      uint32_t hv[32];
      tmem_ld32(tq, hv);
      // tokens of this quarter inside the sequence (32 except in the last tile)
      const int64_t left = A.n - ((int64_t)(t_begin + i) * TILE + 32 * q);
      const int nv = left <= 0 ? 0 : (left >= 32 ? 32 : (int)left);
      uint32_t pp[16], pn[16];
      const float2* oxt = ox + b * TILE + 32 * q;
#pragma unroll
      for (int t = 0; t < 32; t += 2) {
        const float a0 = fmaf(__uint_as_float(hv[t]), kLog2e, bj);
        const float a1 = fmaf(__uint_as_float(hv[t + 1]), kLog2e, bj);
        float e0, e1, f0, f1;
        if (A.off) {
          const float4 o2 = *reinterpret_cast<const float4*>(oxt + t);   // tokens t, t+1
          e0 = ex2_approx(a0 - o2.x); e1 = ex2_approx(a1 - o2.z);
          f0 = ex2_approx(-a0 - o2.y); f1 = ex2_approx(-a1 - o2.w);
        } else {
          e0 = ex2_approx(a0); e1 = ex2_approx(a1);
          f0 = ex2_approx(-a0); f1 = ex2_approx(-a1);
        }
        // tokens past the end of the sequence contribute nothing
        if (nv < 32) {
          if (t >= nv) e0 = f0 = 0.f;
          if (t + 1 >= nv) e1 = f1 = 0.f;
        }
        // z sums the fp32 features; the MMA operand is their bf16 rounding
        zp += e0 + e1;
        zn += f0 + f1;
        pp[t / 2] = pack_bf16(e0, e1);
        pn[t / 2] = pack_bf16(f0, f1);
      }
      tmem_st16(tq, pp);
      tmem_st16(tq + 16, pn);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E1 + b));
    }
  }

  // ---- export: S (features x 128) and z of this segment ----
  tc_fence_before();
  __syncthreads();
  if (nt > 0 && !*(volatile int*)abort_flag)
    mbar_wait(bar(B_G2 + ((nt - 1) & 1)), ((nt - 1) >> 1) & 1, wp);
  tc_fence_after();
  if (warp < kFeat) {
    const int q = warp >> 2, j = 32 * (warp & 3) + lane;
    zx[256 * q + j] = zp;
    zx[256 * q + 128 + j] = zn;
  }
  __syncthreads();
  if (warp < kFeat && !*(volatile int*)abort_flag) {
    // warp w: feature block c = (w / 4) % 2 (exp(+h) for c = 0, exp(-h) for
    // c = 1), hidden unit j, state columns [64 (w / 8), +64)
    const int c = (warp >> 2) & 1;
    const int j = 32 * (warp & 3) + lane;
    float* dst = A.ws + ((size_t)unit * (A.P - 1) * A.M + pc.index) * ((size_t)2 * D * D + 2 * D);
    const int f = 128 * c + j;
#pragma unroll 1
    for (int c0 = 64 * (warp >> 3); c0 < 64 * (warp >> 3) + 64; c0 += 32) {
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base(warp) + TM_S + 128 * c + c0, sv);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(dst + ws_s_index(f, c0 + 4 * q, D)) =
            make_float4(__uint_as_float(sv[4 * q]), __uint_as_float(sv[4 * q + 1]),
                        __uint_as_float(sv[4 * q + 2]), __uint_as_float(sv[4 * q + 3]));
    }
    // z: the four token quarters' sums in a fixed order
    if (warp >> 3 == 0)
      dst[(size_t)2 * D * D + f] = (zx[f] + zx[256 + f]) + (zx[512 + f] + zx[768 + f]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Taylor, d = 16.  The state is kept over the 160 packed features of
// taylor_pack.cuh (the same dot products as the 288 public ones).  phi(K_t)
// is built row-wise (thread = token, its 32-byte row of K loaded from global
// memory a tile ahead) into one of two shared-memory buffers, so tile t+1's
// features are written while G2(t) still reads tile t's.  With ~109 KB of
// shared memory and 256 TMEM columns two CTAs share an SM, so the pass runs
// one piece of a segment per CTA over both slots of every SM.  The state is
// kept transposed, so one MMA per 16 tokens spans every feature:
//   [S z]^T += [V_t e0]^T phi(K_t)   (M = 64, N = 160, e0 = (1, 0, ..., 0))
// [V e0]^T is the MN-major [V e0] tile read as A: rows 0-15 are V's columns,
// row 16 the ones of e0 (z), rows 17-31 zero and rows 32-63 whatever lies
// one and two blocks further (never read back).  An M = 64 accumulator holds
// row m in TMEM lane 32 (m / 16) + m % 16, so S^T sits in lanes 0-15 and
// z in lane 32.  Warp 8 issues MMAs, warp 9 issues loads.
// ---------------------------------------------------------------------------
namespace tay {
constexpr int DP = tp::F;                              // packed features (153 used)
constexpr uint32_t XT = TILE * 16 * 2;                 // 4 KB
constexpr uint32_t OFF_V = 0;                          // 2 stages, 32B-swizzled
constexpr uint32_t OFF_E0 = 8192;                      // [128 x 16], column 0 = 1
constexpr int NB = 2;                                  // phi(K) buffers
constexpr uint32_t OFF_PHK = 12288;                    // NB buffers x 3 panels of 16 KB
constexpr uint32_t PHK_BYTES = 3 * 16384;              // features 160..191 stay zero
constexpr uint32_t OFF_BAR = OFF_PHK + NB * PHK_BYTES;
enum { B_LDV = 0, B_E1 = 2, B_G2 = 4, B_COUNT = 6 };
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;
static_assert(ALLOC <= 113 * 1024, "shared memory: two CTAs per SM");
constexpr uint32_t TM_S = 0;                           // [S z]^T: 160 feature columns
constexpr uint32_t TM_COLS = 256;                      // two CTAs per SM
constexpr int kThreads = 320;
}  // namespace tay

__global__ void __launch_bounds__(tay::kThreads, 2) state_taylor_kernel(const __grid_constant__ StateArgs A) {
  using namespace tay;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const StatePiece pc = state_piece(A);
  const int64_t unit = pc.unit;
  const int64_t kvu = kv_unit(unit, A.H, A.G);   // k, v of this query head
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int t_begin = pc.t_begin;
  const int nt = pc.nt;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(bar(b), (b == B_E1 || b == B_E1 + 1) ? 8 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the first two tiles into L2 while the kernels before this one finish (a
  // prefetch only warms the cache, so it may precede the wait)
  if (warp == 8 && lane == 0)
    for (int i = 0; i < 2 && i < nt; ++i) {
      tma_prefetch_rows(&A.tk, 0, (t_begin + i) * TILE, ub, kh, A.seq);
      tma_prefetch_rows(&A.tv, 0, (t_begin + i) * TILE, ub, kh, A.seq);
    }
  // global memory is touched only after the kernels before this one have
  // completed; only then may the next kernel be scheduled, so the kernels
  // after this one in a call may read the call's inputs before their own wait
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  auto load_v = [&](int i) {
    const uint32_t b = bar(B_LDV + (i & 1));
    mbar_expect_tx(b, XT);
    tma_load_rows(sb + OFF_V + (i & 1) * XT, &A.tv, b, 0, (t_begin + i) * TILE, ub,
                    kh, A.seq);
  };
  if (warp == 8 && lane == 0)
    for (int i = 0; i < 2 && i < nt; ++i) load_v(i);
  // the rest of the piece's K rows into L2 for the feature warps' loads
  if (warp == 9 && lane == 0)
    for (int i = 2; i < nt; ++i) tma_prefetch_rows(&A.tk, 0, (t_begin + i) * TILE, ub, kh, A.seq);
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  // e0 rows (1, 0, ..., 0) with the 32-byte swizzle; phi(K) buffers zero (features 160.. stay 0)
  for (int r = tid; r < 128; r += tay::kThreads) {
    const uint32_t c0 = ((r >> 2) & 1) << 4;
    st_shared_v4(sb + OFF_E0 + r * 32 + c0, 0x3F80u, 0u, 0u, 0u);
    st_shared_v4(sb + OFF_E0 + r * 32 + (16 - c0), 0u, 0u, 0u, 0u);
  }
  for (uint32_t i = tid * 16; i < NB * PHK_BYTES; i += tay::kThreads * 16)
    st_shared_v4(sb + OFF_PHK + i, 0u, 0u, 0u, 0u);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4) {   // [S z]^T = 0 (every lane, so whichever rows the MMA uses start at zero)
    uint32_t zr[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) zr[j] = 0u;
    for (int c0 = 0; c0 < DP; c0 += 32) tmem_st32(tmem + lane_base(warp) + TM_S + c0, zr);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 8) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(64, DP, 1, 1);   // [V e0]^T[MN] phiK[MN]
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        ok = mbar_wait_poll(bar(B_E1 + (i & 1)), (i >> 1) & 1, wp) &&
             mbar_wait_poll(bar(B_LDV + (i & 1)), (i >> 1) & 1, wp);
        if (!ok) break;
        tc_fence_after();
        const uint32_t pb = sb + OFF_PHK + (i % NB) * PHK_BYTES;
        const uint32_t vb = sb + OFF_V + (i & 1) * XT;
        // A = [V e0]^T: 16-row blocks one leading-byte offset apart (V, e0,
        // then two blocks never read back); B = phi(K), 64-feature panels
        const uint64_t dv = smem_desc(vb, OFF_E0 - (OFF_V + (i & 1) * XT), 256, 6);
        const uint64_t dk = smem_desc(pb, 16384, 1024, 2);
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ss(tmem + TM_S, dv + ks * 32, dk + ks * 128, ID_S, 1);
        mma_commit(bar(B_G2 + (i & 1)));
      }
      if (!ok) *(volatile int*)abort_flag = 1;
    }
  } else if (warp == 9) {
    // ======================= loader =======================
    //   V(i) once G2(i-2) has read V(i-2)
    if (lane == 0) {
      int nv = nt < 2 ? nt : 2;
      IdleClock clk;
      bool alive = true;
      while (nv < nt && alive) {
        if (mbar_probe(bar(B_G2 + (nv & 1)), ((nv - 2) >> 1) & 1)) {
          load_v(nv++);
          clk.progress();
        } else {
          alive = clk.idle(wp);
        }
      }
    }
  } else {
    // ======================= feature warps =======================
    const int c = warp >> 2;
    const int row = 32 * (warp & 3) + lane;
    // this thread's token rows of K: [B][Hkv][n][16], or [B][n][Hkv][16]
    const int hkv = A.H / A.G;
    const size_t rs = A.seq ? (size_t)hkv * 16 : 16;
    const __nv_bfloat16* kb = A.kraw + (A.seq ? ((size_t)ub * A.n * hkv + kh) * 16
                                              : ((size_t)ub * hkv + kh) * (size_t)A.n * 16);
    auto load_row = [&](int i, uint4& lo, uint4& hi) {
      const int64_t t = (int64_t)(t_begin + i) * TILE + row;
      if (t < A.n) {
        const uint4* src = reinterpret_cast<const uint4*>(kb + (size_t)t * rs);
        lo = __ldg(src);
        hi = __ldg(src + 1);
      } else {
        lo = hi = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    uint4 nlo, nhi;
    if (nt > 0) load_row(0, nlo, nhi);
    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;
      const bool valid = (int64_t)(t_begin + i) * TILE + row < A.n;
      const uint4 klo = nlo, khi = nhi;
      if (i + 1 < nt) load_row(i + 1, nlo, nhi);   // in flight while this tile's features form
      const uint32_t kw[8] = {klo.x, klo.y, klo.z, klo.w, khi.x, khi.y, khi.z, khi.w};
      float x[16];
#pragma unroll
      for (int k2 = 0; k2 < 8; ++k2) {
        x[2 * k2] = __uint_as_float(kw[k2] << 16);
        x[2 * k2 + 1] = __uint_as_float(kw[k2] & 0xFFFF0000u);
      }
      // packed features: half 0 [0, 80), half 1 [80, 160); 16-byte chunks of 8
      uint32_t w[10][4];
      if (c == 0) {
        tp::chunk8<0>(x, valid, w[0]);   tp::chunk8<8>(x, valid, w[1]);
        tp::chunk8<16>(x, valid, w[2]);  tp::chunk8<24>(x, valid, w[3]);
        tp::chunk8<32>(x, valid, w[4]);  tp::chunk8<40>(x, valid, w[5]);
        tp::chunk8<48>(x, valid, w[6]);  tp::chunk8<56>(x, valid, w[7]);
        tp::chunk8<64>(x, valid, w[8]);  tp::chunk8<72>(x, valid, w[9]);
      } else {
        tp::chunk8<80>(x, valid, w[0]);  tp::chunk8<88>(x, valid, w[1]);
        tp::chunk8<96>(x, valid, w[2]);  tp::chunk8<104>(x, valid, w[3]);
        tp::chunk8<112>(x, valid, w[4]); tp::chunk8<120>(x, valid, w[5]);
        tp::chunk8<128>(x, valid, w[6]); tp::chunk8<136>(x, valid, w[7]);
        tp::chunk8<144>(x, valid, w[8]); tp::chunk8<152>(x, valid, w[9]);
      }
      // the buffer held phi(K(i-NB)), read by G2(i-NB)
      if (i >= NB && !__all_sync(0xffffffffu,
                                 mbar_wait(bar(B_G2 + ((i - NB) & 1)), ((i - NB) >> 1) & 1, wp)))
        break;
      const uint32_t phk = sb + OFF_PHK + (i % NB) * PHK_BYTES;
#pragma unroll
      for (int q = 0; q < 10; ++q) {
        const int f = 80 * c + 8 * q;
        st_shared_v4(phk + (f / 64) * 16384 + sw128_chunk(row, (f % 64) / 8), w[q][0], w[q][1],
                     w[q][2], w[q][3]);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E1 + b));
    }
  }

  // ---- export this segment's S and z ----
  tc_fence_before();
  __syncthreads();
  if (nt > 0 && !*(volatile int*)abort_flag)
    mbar_wait(bar(B_G2 + ((nt - 1) & 1)), ((nt - 1) >> 1) & 1, wp);
  tc_fence_after();
  __syncthreads();
  // S^T row v (TMEM lane v < 16, warp 0) holds column v of S over the 160
  // features; row 16 (lane 32, warp 1) holds z
  if (warp < 2 && !*(volatile int*)abort_flag) {
    float* dst = A.ws + ((size_t)unit * (A.P - 1) * A.M + pc.index) * ((size_t)DP * 16 + DP);
#pragma unroll 1
    for (int c0 = 0; c0 < DP; c0 += 32) {
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base(warp) + TM_S + c0, sv);
      if (warp == 0 && lane < 16) {
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[ws_s_index(c0 + j, lane, 16)] = __uint_as_float(sv[j]);
      } else if (warp == 1 && lane == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(size_t)DP * 16 + c0 + j] = __uint_as_float(sv[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}


template <int KIND, int D>
cudaError_t state_t(const Problem& p, const TcPlan& pl, const void* k, const void* v, void* ws,
                    int* dev_status, cudaStream_t s) {
  StateArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  bool ok;
  if (KIND == HH_FMAP_HEDGEHOG) {
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    ok = make_rows_map(&a.tk, k, D, p.n, p.H / p.G, p.B, 64, TILE, sw, p.seq_major) &&
         make_rows_map(&a.tv, v, D, p.n, p.H / p.G, p.B, 64, TILE, sw, p.seq_major) &&
         make_plane_map(&a.tw, p.Wk ? p.Wk : p.Wq, D, D, p.H, 64, D, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    ok = make_rows_map(&a.tk, k, 16, p.n, p.H / p.G, p.B, 16, TILE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       p.seq_major) &&
         make_rows_map(&a.tv, v, 16, p.n, p.H / p.G, p.B, 16, TILE, CU_TENSOR_MAP_SWIZZLE_32B,
                       p.seq_major);
  }
  if (!ok) return cudaErrorInvalidValue;
  // one segment per CTA: the states go straight to the scanned area; pieces
  // of segments: to the area after it, which the scan sums per segment
  a.ws = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + (pl.M > 1 ? pl.raw_offset : 0));
  a.kraw = reinterpret_cast<const __nv_bfloat16*>(k);
  a.bias = p.Wk ? p.bk : p.bq;
  a.off = p.offk;
  if (p.softmax && !p.offk) return cudaErrorInvalidValue;
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.H = p.H;
  a.P = pl.P;
  a.L = pl.L;
  a.NT = pl.NT;
  a.M = pl.M;
  a.G = p.G;
  a.seq = p.seq_major;
  const dim3 grid((unsigned)(U * (pl.P - 1) * pl.M));
  if (KIND == HH_FMAP_TAYLOR2) {
    cudaError_t e = cudaFuncSetAttribute(state_taylor_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tay::ALLOC);
    // two CTAs per SM need the largest shared-memory carveout
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(state_taylor_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               100);
    if (e != cudaSuccess) return e;
    return launch_pdl(state_taylor_kernel, grid, dim3(tay::kThreads),
                      (size_t)tay::ALLOC, s, a);
  }
  if (KIND == HH_FMAP_HEDGEHOG && D == 128) {
    cudaError_t e = cudaFuncSetAttribute(state_t128_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)t128::ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(state_t128_kernel, grid, dim3(t128::kThreads),
                      (size_t)t128::ALLOC, s, a);
  }
  if constexpr (KIND == HH_FMAP_HEDGEHOG && D == 64) {
    const size_t smem = SSmem<D>::ALLOC;
    cudaError_t e = cudaFuncSetAttribute(state_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(state_tc_kernel<D>, grid, dim3(kThreads), smem, s, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// State pass for P > 1 segments: U * (P - 1) CTAs, one per segment but the last.
cudaError_t launch_state_tc(const Problem& p, const TcPlan& pl, const void* k, const void* v,
                            void* ws, int* dev_status, cudaStream_t s) {
  if (pl.P < 2) return cudaSuccess;
  if (p.kind == HH_FMAP_TAYLOR2) return state_t<HH_FMAP_TAYLOR2, 16>(p, pl, k, v, ws, dev_status, s);
  if (p.d == 64) return state_t<HH_FMAP_HEDGEHOG, 64>(p, pl, k, v, ws, dev_status, s);
  return state_t<HH_FMAP_HEDGEHOG, 128>(p, pl, k, v, ws, dev_status, s);
}

}  // namespace hh
