// Chunked causal prefill, output pass, for the degree-2 Taylor map (d = 16).
//
// "The Taylor Exponential as a Bridge Result" (Hedgehog & Porcupine summary)
// gives phi(x) = [1, x, vec(x x^T) / sqrt2], so phi(q) . phi(k) = 1 + s + s^2/2
// with s = q . k.  The intra-tile scores therefore need one K = 16 MMA of
// Q K^T and two FMAs per element instead of a 288-deep feature contraction;
// the running state ("2. Context and Motivation", paper Eq. 2; "Complexity Analysis") still
// needs features, kept as the 160 packed features of taylor_pack.cuh (the 136
// unordered pairs carry the same dot products as the 256 ordered ones):
//   Sc(t) = Q_t K_t^T                         -> P = bf16(tril(1 + Sc + Sc^2/2))
//   [S z] += phi(K_t)^T [V_t e0]             (N = 32, z rides in column 16)
//   [O den] = P [V_t e0] + phi(Q_t) [S_bf16 z2]   (z2 = z as a bf16 hi/lo pair)
//   y = O / (den_hi + den_lo)
// Roles: warp 8 issues every tcgen05.mma as soon as its inputs are ready,
// warp 9 issues TMA loads, warps 0-7 run the epilogue phases
//   E1(t): phi(Q_t) -> TMEM, phi(K_t) -> smem, S_bf16/z2 snapshot
//   E2(t): P from Sc(t);   E3(t): y from [O den]
// in the order E1(t), E2(t), E3(t-1) per step.  phi(Q), S_bf16/z2, the score /
// output TMEM columns and P have two buffers (tile parity), so Sc(t+1) and
// E2(t+1) need not wait for E3(t).  Every mbarrier wait is bounded in time
// (tc_ptx.cuh).

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

constexpr int D = 16, DP = tp::F, TILE = 128;   // DP: packed features (153 used)
constexpr int kThreads = 320;
constexpr uint32_t XT = TILE * D * 2;                   // one Q, K or V tile: 4 KB
// shared memory (1024-aligned base); Q, K, V tiles are 32B-swizzled rows
constexpr uint32_t OFF_Q = 0, OFF_K = 8192, OFF_V = 16384;   // 2 stages each
constexpr uint32_t OFF_E0 = 24576;                      // [128 x 16], column 0 = 1
constexpr uint32_t SB_BYTES = DP * 32;                  // [160 x 16] bf16, 32B-swizzled
constexpr uint32_t OFF_SB = 28672;                      // 2 x (S_bf16 | z2)
constexpr uint32_t OFF_PHK = 49152;                     // phi(K): 4 panels [128 tok x 64 feat]
constexpr uint32_t OFF_P = OFF_PHK + 4 * 16384;         // P: 2 buffers x 2 panels [128 x 64 keys]
constexpr uint32_t OFF_BAR = OFF_P + 4 * 16384;
enum { B_LD = 0, B_SC = 2, B_SU = 4, B_G3 = 6, B_E1 = 8, B_E2 = 10, B_E3 = 12, B_COUNT = 14 };
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_SB + 4 * SB_BYTES <= OFF_PHK, "S_bf16 buffers");
// TMEM columns
constexpr uint32_t TM_S = 0;                            // 2 blocks x [S (16) | z, 0.. (16)]
__host__ __device__ constexpr uint32_t TM_Y(int b) { return 64 + 80 * b; }    // phi(Q) pairs
__host__ __device__ constexpr uint32_t TM_X(int b) { return 256 + 128 * b; }  // Sc -> [O den]

struct ArgsT {
  CUtensorMap tq, tk, tv;
  __nv_bfloat16* y;
  const float* ws;   // [U][P-1][DP*D + DP] inclusive prefixes (ws_s_index layout, then z)
  const float* init; // [U][DP*D + DP] initial state (continuation), same layout, or null
  float* S_out;      // [U][288][D] (public feature order) or null
  float* z_out;      // [U][288]
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int P, L, NT;
  int H, G;          // heads; query heads per key/value head
  int seq;           // q, k, v, y are [B][n][H][16]
};

__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

// Row r (16 bf16) of a 32B-swizzled [128 x 16] tile as floats.
__device__ __forceinline__ void load_row16(const uint8_t* tile, int r, float (&x)[16]) {
  const int sw = ((r >> 2) & 1) << 4;
  const uint4 a = *reinterpret_cast<const uint4*>(tile + r * 32 + sw);
  const uint4 b = *reinterpret_cast<const uint4*>(tile + r * 32 + (16 - sw));
  x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
  x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
  x[8] = bf16_lo(b.x); x[9] = bf16_hi(b.x); x[10] = bf16_lo(b.y); x[11] = bf16_hi(b.y);
  x[12] = bf16_lo(b.z); x[13] = bf16_hi(b.z); x[14] = bf16_lo(b.w); x[15] = bf16_hi(b.w);
}

// phi(q): 32 packed features from F0 -> 16 TMEM columns (bf16 pairs)
template <int F0>
__device__ __forceinline__ void phiq32(const float (&x)[16], uint32_t ty) {
  uint32_t w[16];
  tp::chunk8<F0>(x, true, *reinterpret_cast<uint32_t(*)[4]>(&w[0]));
  tp::chunk8<F0 + 8>(x, true, *reinterpret_cast<uint32_t(*)[4]>(&w[4]));
  tp::chunk8<F0 + 16>(x, true, *reinterpret_cast<uint32_t(*)[4]>(&w[8]));
  tp::chunk8<F0 + 24>(x, true, *reinterpret_cast<uint32_t(*)[4]>(&w[12]));
  tmem_st16(ty + F0 / 2, w);
}
template <int F0>
__device__ __forceinline__ void phiq16(const float (&x)[16], uint32_t ty) {
  uint32_t w[8];
  tp::chunk8<F0>(x, true, *reinterpret_cast<uint32_t(*)[4]>(&w[0]));
  tp::chunk8<F0 + 8>(x, true, *reinterpret_cast<uint32_t(*)[4]>(&w[4]));
  tmem_st8(ty + F0 / 2, w);
}
// phi(k): 8 packed features from F0 -> one 16-byte chunk of the swizzled panels
template <int F0>
__device__ __forceinline__ void phik8(const float (&x)[16], bool valid, uint32_t phk, int row) {
  uint32_t w[4];
  tp::chunk8<F0>(x, valid, w);
  st_shared_v4(phk + (F0 / 64) * 16384 + sw128_chunk(row, (F0 % 64) / 8), w[0], w[1], w[2], w[3]);
}

// The bound of 384 threads caps registers at 168 per thread (warps 0, 4, 8 and
// 1, 5, 9 share one SM sub-partition's registers).
__global__ void __launch_bounds__(384, 1) taylor_out_kernel(const __grid_constant__ ArgsT A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x / A.P;
  const int64_t kvu = kv_unit(unit, A.H, A.G);   // k, v of this query head
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int seg = blockIdx.x % A.P;
  const int t_begin = seg * A.L;
  const int nt = min(A.NT, t_begin + A.L) - t_begin;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(bar(b), b >= B_E1 ? 8 : 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&A.tq);
    prefetch_tmap(&A.tk);
    prefetch_tmap(&A.tv);
  }
  // the first two tiles into L2 while the kernels before this one finish (a
  // prefetch only warms the cache, so it may precede the wait)
  if (warp == 8 && lane == 0)
    for (int i = 0; i < 2 && i < nt; ++i) {
      const int r0 = (t_begin + i) * TILE;
      tma_prefetch_rows(&A.tq, 0, r0, ub, uh, A.seq);
      tma_prefetch_rows(&A.tk, 0, r0, ub, kh, A.seq);
      tma_prefetch_rows(&A.tv, 0, r0, ub, kh, A.seq);
    }
  // the next kernel may be scheduled now; global memory is touched only after
  // the kernels before this one have completed
  pdl_launch_dependents();
  pdl_wait();
  __syncthreads();
  auto load = [&](int i) {
    const int s = i & 1;
    const int r0 = (t_begin + i) * TILE;
    mbar_expect_tx(bar(B_LD + s), 3 * XT);
    tma_load_rows(sb + OFF_Q + s * XT, &A.tq, bar(B_LD + s), 0, r0, ub, uh, A.seq);
    tma_load_rows(sb + OFF_K + s * XT, &A.tk, bar(B_LD + s), 0, r0, ub, kh, A.seq);
    tma_load_rows(sb + OFF_V + s * XT, &A.tv, bar(B_LD + s), 0, r0, ub, kh, A.seq);
  };
  if (warp == 8 && lane == 0)
    for (int i = 0; i < 2 && i < nt; ++i) load(i);
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  // e0 rows (1, 0, ..., 0); z2 buffers zero (only column pair 0-1 is rewritten);
  // phi(K) panels zero (features 160..255 stay zero)
  for (int r = tid; r < 128; r += kThreads) {
    const uint32_t c0 = ((r >> 2) & 1) << 4;
    st_shared_v4(sb + OFF_E0 + r * 32 + c0, 0x3F80u, 0u, 0u, 0u);
    st_shared_v4(sb + OFF_E0 + r * 32 + (16 - c0), 0u, 0u, 0u, 0u);
  }
  for (uint32_t i = tid * 16; i < 2 * SB_BYTES; i += kThreads * 16) {
    const uint32_t b = i / SB_BYTES, o = i % SB_BYTES;
    st_shared_v4(sb + OFF_SB + b * 2 * SB_BYTES + SB_BYTES + o, 0u, 0u, 0u, 0u);
  }
  for (uint32_t i = tid * 16; i < 4 * 16384u; i += kThreads * 16)
    st_shared_v4(sb + OFF_PHK + i, 0u, 0u, 0u, 0u);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // initial [S z]: zeros, or the prefix of the preceding segments
  if (warp < 8) {
    const int c = warp >> 2;
    const float* prefix =
        seg > 0 ? A.ws + ((size_t)unit * (A.P - 1) + seg - 1) * (size_t)(DP * D + DP)
                : (A.init ? A.init + (size_t)unit * (DP * D + DP) : nullptr);
    for (int mb = c; mb < 2; mb += 2) {
      const int f = 128 * mb + 32 * (warp & 3) + lane;
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
      if (prefix && f < DP) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v4 = __ldcg(reinterpret_cast<const float4*>(prefix + ws_s_index(f, 4 * q, D)));
          r[4 * q] = __float_as_uint(v4.x);
          r[4 * q + 1] = __float_as_uint(v4.y);
          r[4 * q + 2] = __float_as_uint(v4.z);
          r[4 * q + 3] = __float_as_uint(v4.w);
        }
        r[16] = __float_as_uint(__ldcg(prefix + (size_t)DP * D + f));
      }
      tmem_st32(tmem + lane_base(warp) + TM_S + 32 * mb, r);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 8) {
    // ======================= MMA issuer =======================
    // Lane 0 issues every tcgen05 instruction, in the order the epilogue
    // consumes the groups, waiting on one barrier at a time.
    if (nt > 0 && lane == 0) {
      constexpr uint32_t ID_SC = idesc_bf16(128, 128, 0, 0);   // Q[K-major] K[K-major]
      constexpr uint32_t ID_SU = idesc_bf16(128, 32, 1, 1);    // phiK^T[MN] [V e0][MN]
      constexpr uint32_t ID_O = idesc_bf16(128, 32, 0, 1);     // P or phiQ x [V e0] or [S z2]
      // descriptor bases; a k-step only moves the start-address field (16-byte units)
      const uint64_t dphk = smem_desc(sb + OFF_PHK, 16384, 1024, 2);
      const uint64_t dp0 = smem_desc(sb + OFF_P, 16, 1024, 2);
      auto dv = [&](int s) {   // [V e0]: the e0 block one leading-byte offset after V
        return smem_desc(sb + OFF_V + s * XT, OFF_E0 - (OFF_V + s * XT), 256, 6);
      };
      auto Sc = [&](int i) {
        const int s = i & 1;
        const uint64_t da = smem_desc(sb + OFF_Q + s * XT, 16, 256, 6);
        const uint64_t db = smem_desc(sb + OFF_K + s * XT, 16, 256, 6);
        tc_fence_after();
        mma_ss(tmem + TM_X(s), da, db, ID_SC, 0);
        mma_commit(bar(B_SC + s));
      };
      auto SU = [&](int i) {
        const int s = i & 1;
        const uint64_t v = dv(s);
        tc_fence_after();
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int ks = 0; ks < TILE / 16; ++ks)
            mma_ss(tmem + TM_S + 32 * mb, dphk + (2 * mb) * 1024 + ks * 128, v + ks * 32, ID_SU, 1);
        mma_commit(bar(B_SU + s));
      };
      auto G3 = [&](int i) {
        const int s = i & 1;
        const uint64_t v = dv(s);
        const uint64_t dsb = smem_desc(sb + OFF_SB + s * 2 * SB_BYTES, SB_BYTES, 256, 6);
        const uint32_t ty = tmem + TM_Y(s);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ss(tmem + TM_X(s), dp0 + s * 2048 + (ks >> 2) * 1024 + (ks & 3) * 2, v + ks * 32,
                 ID_O, ks > 0);
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tmem + TM_X(s), ty + ks * 8, dsb + ks * 32, ID_O, 1);
        mma_commit(bar(B_G3 + s));
      };
      // The epilogue runs E1(i), E2(i), E3(i-1) per step, so the groups are
      // consumed in the order Sc(0), Sc(1), then per tile i
      //   Sc(i)   (i >= 2) once Q, K of tile i have landed and E3(i-2) has freed
      //           its score / output columns
      //   SU(i)   once E1(i) has written phi(K_i) and the snapshot
      //   G3(i)   once E2(i) has written P_i
      bool ok = true;
      for (int i = 0; i < 2 && i < nt && ok; ++i) {
        ok = mbar_wait_poll(bar(B_LD + i), 0, wp);
        if (ok) Sc(i);
      }
      for (int i = 0; i < nt && ok; ++i) {
        if (i >= 2) {
          ok = mbar_wait_poll(bar(B_LD + (i & 1)), (i >> 1) & 1, wp) &&
               mbar_wait_poll(bar(B_E3 + (i & 1)), ((i - 2) >> 1) & 1, wp);
          if (!ok) break;
          Sc(i);
        }
        ok = mbar_wait_poll(bar(B_E1 + (i & 1)), (i >> 1) & 1, wp);
        if (!ok) break;
        SU(i);
        ok = mbar_wait_poll(bar(B_E2 + (i & 1)), (i >> 1) & 1, wp);
        if (!ok) break;
        G3(i);
      }
    }
  } else if (warp == 9) {
    // ======================= loader =======================
    // Q, K, V of tile i into stage i&1 once G3(i-2) has completed: every MMA
    // and epilogue read of tile i-2 precedes it.
    if (lane == 0) {
      for (int i = 2; i < nt; ++i) {
        if (!mbar_wait_poll(bar(B_G3 + (i & 1)), ((i - 2) >> 1) & 1, wp)) break;
        load(i);
      }
    }
  } else {
    // ======================= epilogue warps =======================
    // warp w: TMEM lanes / tile rows 32 (w % 4).., half c = w / 4 of the columns
    const int c = warp >> 2;
    const int g = warp & 3;
    const int row = 32 * g + lane;
    const uint32_t lb = lane_base(warp);
    bool good = true;

    auto E1 = [&](int i) {
      const int s = i & 1;
      const bool valid = (int64_t)(t_begin + i) * TILE + row < A.n;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_LD + s), (i >> 1) & 1, wp))) { good = false; return; }
      // phi(Q): half 0 packed features [0, 80), half 1 [80, 160) -> TMEM column pairs
      {
        float x[16];
        load_row16(sm + OFF_Q + s * XT, row, x);
        const uint32_t ty = tmem + lb + TM_Y(s);
        if (c == 0) {
          phiq32<0>(x, ty);
          phiq32<32>(x, ty);
          phiq16<64>(x, ty);
        } else {
          phiq32<80>(x, ty);
          phiq32<112>(x, ty);
          phiq16<144>(x, ty);
        }
      }
      // phi(K) and the state snapshot need SU(i-1) done (it read phi(K(i-1)), updated S)
      if (i > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SU + ((i - 1) & 1)), ((i - 1) >> 1) & 1, wp))) {
          good = false;
          return;
        }
        tc_fence_after();
      }
      {
        float x[16];
        load_row16(sm + OFF_K + s * XT, row, x);
        const uint32_t phk = sb + OFF_PHK;
        if (c == 0) {
          phik8<0>(x, valid, phk, row);   phik8<8>(x, valid, phk, row);
          phik8<16>(x, valid, phk, row);  phik8<24>(x, valid, phk, row);
          phik8<32>(x, valid, phk, row);  phik8<40>(x, valid, phk, row);
          phik8<48>(x, valid, phk, row);  phik8<56>(x, valid, phk, row);
          phik8<64>(x, valid, phk, row);  phik8<72>(x, valid, phk, row);
        } else {
          phik8<80>(x, valid, phk, row);  phik8<88>(x, valid, phk, row);
          phik8<96>(x, valid, phk, row);  phik8<104>(x, valid, phk, row);
          phik8<112>(x, valid, phk, row); phik8<120>(x, valid, phk, row);
          phik8<128>(x, valid, phk, row); phik8<136>(x, valid, phk, row);
          phik8<144>(x, valid, phk, row); phik8<152>(x, valid, phk, row);
        }
      }
      // S_bf16 and z2 (z as z_hi + z_lo) of the tokens before this tile
      const uint32_t sbb = sb + OFF_SB + s * 2 * SB_BYTES;
      for (int mb = c; mb < 2; mb += 2) {
        const int f = 128 * mb + row;
        uint32_t sv[32];
        tmem_ld32(tmem + lb + TM_S + 32 * mb, sv);
        if (f < DP) {
          const uint32_t sw = ((f >> 2) & 1) << 4;
          st_shared_v4(sbb + f * 32 + sw,
                       pack_bf16(__uint_as_float(sv[0]), __uint_as_float(sv[1])),
                       pack_bf16(__uint_as_float(sv[2]), __uint_as_float(sv[3])),
                       pack_bf16(__uint_as_float(sv[4]), __uint_as_float(sv[5])),
                       pack_bf16(__uint_as_float(sv[6]), __uint_as_float(sv[7])));
          st_shared_v4(sbb + f * 32 + (16 - sw),
                       pack_bf16(__uint_as_float(sv[8]), __uint_as_float(sv[9])),
                       pack_bf16(__uint_as_float(sv[10]), __uint_as_float(sv[11])),
                       pack_bf16(__uint_as_float(sv[12]), __uint_as_float(sv[13])),
                       pack_bf16(__uint_as_float(sv[14]), __uint_as_float(sv[15])));
          const float z = __uint_as_float(sv[16]);
          const float zl = z - __bfloat162float(__float2bfloat16_rn(z));
          st_shared_v4(sbb + SB_BYTES + f * 32 + sw, pack_bf16(z, zl), 0u, 0u, 0u);
        }
      }
      tmem_st_wait();
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E1 + s));
    };

    auto E2 = [&](int i) {
      const int s = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SC + s), (i >> 1) & 1, wp))) { good = false; return; }
      tc_fence_after();
      // keys [64c + 32 h2, +32) = block kc of 32 keys: above the diagonal (kc > g)
      // zero, below it no mask; p = 1 + s + s^2/2 = phi(q) . phi(k)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int kc = 2 * c + h2;
        const uint32_t panel = sb + OFF_P + s * 32768 + c * 16384;
        if (kc > g) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(panel + sw128_chunk(row, 4 * h2 + q4), 0u, 0u, 0u, 0u);
        } else {
          uint32_t sv[32];
          tmem_ld32(tmem + lb + TM_X(s) + 32 * kc, sv);
          const bool diag = kc == g;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = 8 * q4 + 2 * e;   // within this 32-key block
              const float s0 = __uint_as_float(sv[key]), s1 = __uint_as_float(sv[key + 1]);
              float p0 = fmaf(s0, fmaf(s0, 0.5f, 1.f), 1.f);
              float p1 = fmaf(s1, fmaf(s1, 0.5f, 1.f), 1.f);
              if (diag) {
                p0 = key <= lane ? p0 : 0.f;
                p1 = key + 1 <= lane ? p1 : 0.f;
              }
              w4[e] = pack_bf16(p0, p1);
            }
            st_shared_v4(panel + sw128_chunk(row, 4 * h2 + q4), w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E2 + s));
    };

    auto E3 = [&](int i) {
      const int s = i & 1;
      const int64_t r0 = (int64_t)(t_begin + i) * TILE;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G3 + s), (i >> 1) & 1, wp))) { good = false; return; }
      tc_fence_after();
      uint32_t ov[16], d0, d1;
      tmem_ld16(tmem + lb + TM_X(s), ov);
      tmem_ld2(tmem + lb + TM_X(s) + 16, d0, d1);   // rowsum(P) + phi(q).z_hi, phi(q).z_lo
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E3 + s));   // the X columns are free for Sc(i+1)
      const float inv = __frcp_rn(__uint_as_float(d0) + __uint_as_float(d1));
      if (r0 + row < A.n) {
        const int j = 8 * c;
        *reinterpret_cast<uint4*>(A.y + (size_t)row_of(ub, uh, r0 + row, A.H, A.n, A.seq) * D + j) = make_uint4(
            pack_bf16(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv),
            pack_bf16(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv),
            pack_bf16(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv),
            pack_bf16(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv));
      }
    };

    for (int i = 0; i <= nt && good; ++i) {
      if (i < nt) {
        E1(i);
        if (good) E2(i);
      }
      if (good && i >= 1) E3(i - 1);
    }
  }

  // ---- export the final state of the last segment ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (A.S_out && seg == A.P - 1 && warp < 8 && !*(volatile int*)abort_flag) {
    // the last SU completed before the last G3 (issue order), which E3 waited for;
    // packed feature f goes to its public row(s) [1, x, x_i x_j / sqrt2 (i-major)]
    const int c = warp >> 2;
    float* Sd = A.S_out + (size_t)unit * tp::DPUB * D;
    float* zd = A.z_out + (size_t)unit * tp::DPUB;
    for (int mb = c; mb < 2; mb += 2) {
      const int f = 128 * mb + 32 * (warp & 3) + lane;
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base(warp) + TM_S + 32 * mb, sv);
      int r[2];
      float scale;
      const int nr = f < DP ? tp::public_rows(f, r[0], r[1], scale) : 0;
      for (int t = 0; t < nr; ++t) {
        float4* dst = reinterpret_cast<float4*>(Sd + (size_t)r[t] * D);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_float4(__uint_as_float(sv[4 * q]) * scale,
                               __uint_as_float(sv[4 * q + 1]) * scale,
                               __uint_as_float(sv[4 * q + 2]) * scale,
                               __uint_as_float(sv[4 * q + 3]) * scale);
        zd[r[t]] = __uint_as_float(sv[16]) * scale;
      }
    }
    if (warp == 0 && lane < tp::DPUB - 273) {   // zero pad rows 273..287
      float4* dst = reinterpret_cast<float4*>(Sd + (size_t)(273 + lane) * D);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      zd[273 + lane] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

// Output pass of the Taylor (d = 16) prefill: U * P CTAs, one per segment.
cudaError_t launch_prefill_out_taylor(const Problem& p, const TcPlan& pl, const void* q,
                                      const void* k, const void* v, void* y, float* S_out,
                                      float* z_out, const void* ws, const float* init,
                                      int* dev_status, cudaStream_t s) {
  ArgsT a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  if (p.kind != HH_FMAP_TAYLOR2 || p.d != 16) return cudaErrorInvalidValue;
  // 16-column rows (32 bytes), 32-byte swizzle: the layout the MMA descriptors expect
  const auto sw = CU_TENSOR_MAP_SWIZZLE_32B;
  bool ok = make_rows_map(&a.tq, q, D, p.n, p.H, p.B, 16, TILE, sw, p.seq_major) &&
            make_rows_map(&a.tk, k, D, p.n, p.H / p.G, p.B, 16, TILE, sw, p.seq_major) &&
            make_rows_map(&a.tv, v, D, p.n, p.H / p.G, p.B, 16, TILE, sw, p.seq_major);
  if (!ok) return cudaErrorInvalidValue;
  a.y = reinterpret_cast<__nv_bfloat16*>(y);
  a.ws = reinterpret_cast<const float*>(ws);
  a.init = init;
  a.S_out = S_out;
  a.z_out = z_out;
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.P = pl.P;
  a.L = pl.L;
  a.NT = pl.NT;
  a.H = p.H;
  a.G = p.G;
  a.seq = p.seq_major;
  cudaError_t e = cudaFuncSetAttribute(taylor_out_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(taylor_out_kernel, dim3((unsigned)(U * pl.P)), dim3(kThreads),
                    (size_t)SMEM_BYTES, s, a);
}

}  // namespace hh
