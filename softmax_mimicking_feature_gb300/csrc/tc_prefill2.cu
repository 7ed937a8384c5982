// Chunked causal prefill for Hedgehog d = 64 with two tiles in flight.
//
// Same mathematics as prefill_tc_kernel (section 2 / paper Eq. 2 and
// "Complexity Analysis" of "The Hedgehog & the Porcupine" summary; the map of
// "The Hedgehog MLP Feature Map", Choices 1 and 3), reorganised so that the
// serial chain of one 128-token tile overlaps the next tile's:
//
//   warp 8 (producer): TMA loads and every tcgen05.mma, each issued as soon as
//   its inputs are ready (the producer polls the barriers without blocking)
//     G1(t): H_Q = Q_t W, H_K = K_t W
//     G2(t): Sc = phi(Q_t) phi(K_t)^T;  S += phi(K_t)^T V_t;  Z += phi(K_t)^T 1
//     G3(t): O = P_t V_t + phi(Q_t) S_bf16(t)
//   warps 0-3 / 4-7 (two epilogue groups) take alternate tiles:
//     E1 : phi(Q_t) -> TMEM (bf16 pairs), phi(K_t) -> smem          (after G1(t))
//          S_bf16(t) <- S, z(t) <- Z  (state of the tokens before t)  (after G2(t-1))
//          -- only then may G2(t) update S --
//          den(t) = phi(Q_t) . z(t)
//     E2 : P_t = bf16(tril(Sc)), den += rowsum                      (after G2(t))
//     E3 : y = O / den                                              (after G3(t))
// Each group owns one slot of TMEM (H_Q/phi(Q), H_K/Sc/O) and smem (Q/K ->
// S_bf16, V, phi(K) -> P); the running state S (fp32) and its normaliser Z
// (fp32, as an MMA with an all-ones operand) stay in TMEM and pass between
// the groups in tile order.  All mbarrier waits are bounded (tc_ptx.cuh).

#include <math.h>
#include <string.h>

#include <algorithm>

#include "tc_ptx.cuh"

namespace hh {
namespace {

using namespace tc;

constexpr int D = 64, DP = 128, TILE = 128;
constexpr int kThreads = 288;

// TMEM columns
constexpr uint32_t TM_S = 0;     // S: features (lanes) x 64
constexpr uint32_t TM_Z = 64;    // z: 16 identical columns
__host__ __device__ constexpr uint32_t TM_Y(int s) { return 128 + 192 * s; }        // 64 cols
__host__ __device__ constexpr uint32_t TM_X(int s) { return 128 + 192 * s + 64; }   // 128 cols

// shared memory
constexpr uint32_t OFF_W = 0, OFF_WK = 8192, OFF_ONES = 16384;
constexpr uint32_t SLOT_BASE = 20480, SLOT_BYTES = 81920;
constexpr uint32_t S_Q = 0, S_K = 16384, S_V = 32768, S_PHK = 49152;  // S_bf16 aliases S_Q
__host__ __device__ constexpr uint32_t slot_off(int s) { return SLOT_BASE + s * SLOT_BYTES; }
constexpr uint32_t OFF_ZS = SLOT_BASE + 2 * SLOT_BYTES;   // float[2][128]
constexpr uint32_t OFF_BQ = OFF_ZS + 1024;                // float[64]
constexpr uint32_t OFF_BK = OFF_BQ + 256;                 // float[64]
constexpr uint32_t OFF_BAR = OFF_BK + 256;                // 16 x u64
constexpr uint32_t OFF_TM = OFF_BAR + 128;
constexpr uint32_t SMEM_BYTES = OFF_TM + 16 + 1024;

enum Bar { B_W = 0, B_LD = 1, B_G1 = 3, B_G2 = 5, B_G3 = 7, B_E1A = 9, B_E12 = 11, B_E3 = 13 };

struct Args2 {
  CUtensorMap tq, tk, tv, twq, twk;
  __nv_bfloat16* y;
  const float* ws;   // [U][P-1][DP*D + DP] inclusive prefixes of segment states
  float* S_out;
  float* z_out;
  const float* bq;
  const float* bk;
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int H, P, L, NT, sep_wk;
};

__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc2_kernel(const __grid_constant__ Args2 A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* zs = reinterpret_cast<float*>(sm + OFF_ZS);
  float* bq_s = reinterpret_cast<float*>(sm + OFF_BQ);
  float* bk_s = reinterpret_cast<float*>(sm + OFF_BK);
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TM);
  int* abort_flag = reinterpret_cast<int*>(sm + OFF_TM + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x / A.P;
  const int seg = blockIdx.x % A.P;
  const int h = (int)(unit % A.H);
  const int t_begin = seg * A.L;
  const int nt = min(A.NT, t_begin + A.L) - t_begin;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    mbar_init(bar(B_W), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_LD + s), 1);
      mbar_init(bar(B_G1 + s), 1);
      mbar_init(bar(B_G2 + s), 1);
      mbar_init(bar(B_G3 + s), 1);
      mbar_init(bar(B_E1A + s), 4);
      mbar_init(bar(B_E12 + s), 4);
      mbar_init(bar(B_E3 + s), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&A.tq);
    prefetch_tmap(&A.tk);
    prefetch_tmap(&A.tv);
  }
  __syncthreads();

  auto issue_loads = [&](int i) {
    const int s = i & 1;
    const int r0 = (t_begin + i) * TILE;
    const uint32_t base = sb + slot_off(s);
    mbar_expect_tx(bar(B_LD + s), 3 * 16384);
    tma_load_3d(base + S_Q, &A.tq, bar(B_LD + s), 0, r0, (int)unit);
    tma_load_3d(base + S_K, &A.tk, bar(B_LD + s), 0, r0, (int)unit);
    tma_load_3d(base + S_V, &A.tv, bar(B_LD + s), 0, r0, (int)unit);
  };
  if (warp == 8 && lane == 0) {
    mbar_expect_tx(bar(B_W), 8192u * (A.sep_wk ? 2 : 1));
    tma_load_3d(sb + OFF_W, &A.twq, bar(B_W), 0, 0, h);
    if (A.sep_wk) tma_load_3d(sb + OFF_WK, &A.twk, bar(B_W), 0, 0, h);
    issue_loads(0);
    if (nt > 1) issue_loads(1);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  for (int i = tid; i < D; i += kThreads) {
    bq_s[i] = A.bq ? A.bq[(size_t)h * D + i] : 0.f;
    bk_s[i] = A.bk ? A.bk[(size_t)h * D + i] : 0.f;
  }
  for (int i = tid; i < 4096 / 16; i += kThreads)   // bf16 ones: the B operand of Z += phi(K)^T 1
    st_shared_v4(sb + OFF_ONES + 16 * i, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // initial state: zeros, or the prefix of the preceding segments
  if (warp < 4) {
    const int f = 32 * warp + lane;  // feature = TMEM lane
    const float* prefix =
        seg > 0 ? A.ws + ((size_t)unit * (A.P - 1) + seg - 1) * (size_t)(DP * D + DP) : nullptr;
    uint32_t r[32];
    for (int c0 = 0; c0 < D; c0 += 32) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 v4 = prefix ? __ldcg(reinterpret_cast<const float4*>(prefix + (size_t)f * D + c0 + j))
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
    for (int j = 0; j < 16; ++j) zr[j] = __float_as_uint(z0);
    tmem_st16(tmem + lane_base(warp) + TM_Z, zr);
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
      constexpr uint32_t ID_SU = idesc_bf16(128, D, 1, 1);
      constexpr uint32_t ID_Z = idesc_bf16(128, 16, 1, 1);
      constexpr uint32_t ID_PV = idesc_bf16(128, D, 0, 1);
      const uint32_t wk_off = A.sep_wk ? OFF_WK : OFF_W;
      bool ok = mbar_wait(bar(B_W), 0, wp);
      auto G1 = [&](int i) {
        const int s = i & 1;
        tc_fence_after();
        const uint32_t base = sb + slot_off(s);
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t bw = smem_desc(sb + OFF_W + ks * 2048, D * 128, 1024, 2);
          const uint64_t bwk = smem_desc(sb + wk_off + ks * 2048, D * 128, 1024, 2);
          mma_ss(tmem + TM_Y(s), smem_desc(base + S_Q + ks * 32, 16, 1024, 2), bw, ID_H, ks > 0);
          mma_ss(tmem + TM_X(s), smem_desc(base + S_K + ks * 32, 16, 1024, 2), bwk, ID_H, ks > 0);
        }
        mma_commit(bar(B_G1 + s));
      };
      auto G2 = [&](int i) {
        const int s = i & 1;
        tc_fence_after();
        const uint32_t base = sb + slot_off(s);
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tmem + TM_X(s), tmem + TM_Y(s) + ks * 8,
                 smem_desc(base + S_PHK + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024, 2), ID_SC,
                 ks > 0);
        for (int ks = 0; ks < TILE / 16; ++ks) {
          const uint64_t a = smem_desc(base + S_PHK + ks * 2048, 16384, 1024, 2);
          mma_ss(tmem + TM_S, a, smem_desc(base + S_V + ks * 2048, 16384, 1024, 2), ID_SU, 1);
          mma_ss(tmem + TM_Z, a, smem_desc(sb + OFF_ONES + ks * 512, 16, 256, 6), ID_Z, 1);
        }
        mma_commit(bar(B_G2 + s));
      };
      auto G3 = [&](int i) {
        const int s = i & 1;
        tc_fence_after();
        const uint32_t base = sb + slot_off(s);
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ss(tmem + TM_X(s),
                 smem_desc(base + S_PHK + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024, 2),
                 smem_desc(base + S_V + ks * 2048, 16384, 1024, 2), ID_PV, ks > 0);
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tmem + TM_X(s), tmem + TM_Y(s) + ks * 8,
                 smem_desc(base + S_Q + ks * 2048, DP * 128, 1024, 2), ID_PV, 1);
        mma_commit(bar(B_G3 + s));
      };
      // Each action runs once its inputs are ready; per kind they run in tile order.
      //   L(i)  loads into slot i&1   needs G3(i-2) complete (S_bf16, V, P no longer read)
      //   G1(i)                       needs L(i) landed and E3(i-2) done (TMEM slot free)
      //   G2(i)                       needs E1(i) done
      //   G3(i)                       needs E2(i) done
      int nL = nt < 2 ? nt : 2, n1 = 0, n2 = 0, n3 = 0;
      uint64_t t_last = globaltimer();
      bool reported = false;
      while (ok && n3 < nt) {
        bool progress = false;
        if (n2 < n1 && mbar_probe(bar(B_E1A + (n2 & 1)), (n2 >> 1) & 1)) {
          G2(n2++);
          progress = true;
        } else if (n3 < n2 && mbar_probe(bar(B_E12 + (n3 & 1)), (n3 >> 1) & 1)) {
          G3(n3++);
          progress = true;
        } else if (nL < nt && n3 > nL - 2 &&
                   mbar_probe(bar(B_G3 + (nL & 1)), ((nL - 2) >> 1) & 1)) {
          issue_loads(nL++);
          progress = true;
        } else if (n1 < nL && mbar_probe(bar(B_LD + (n1 & 1)), (n1 >> 1) & 1) &&
                   (n1 < 2 || mbar_probe(bar(B_E3 + (n1 & 1)), ((n1 - 2) >> 1) & 1))) {
          G1(n1++);
          progress = true;
        }
        if (progress) {
          t_last = globaltimer();
        } else {
          const uint64_t dt = globaltimer() - t_last;
          if (!reported && dt >= A.soft_ns) {
            reported = true;
            report_timeout(wp);
          }
          if (dt >= A.hard_ns) {
            *(volatile int*)abort_flag = 1;
            ok = false;
          }
          if (*(volatile int*)abort_flag) ok = false;
        }
      }
    }
  } else {
    // ======================= epilogue groups =======================
    const int eg = warp >> 2;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lb = lane_base(warp);
    const uint32_t base = sb + slot_off(eg);
    float* zsn = zs + eg * 128;
    for (int i = eg; i < nt; i += 2) {
      const uint32_t par = (i >> 1) & 1;
      const int64_t r0 = (int64_t)(t_begin + i) * TILE;
      const bool valid = r0 + row < A.n;

      // ---- E1: phi(Q) into TMEM, phi(K) into smem panels ----
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G1 + eg), par, wp))) break;
      tc_fence_after();
      {
        uint32_t hv[64];
        tmem_ld64(tmem + lb + TM_Y(eg), hv);
        uint32_t pp[32], pn[32];
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          const float h0 = __uint_as_float(hv[j]) + bq_s[j];
          const float h1 = __uint_as_float(hv[j + 1]) + bq_s[j + 1];
          pp[j / 2] = pack_bf16(ex2_approx(h0 * kLog2e), ex2_approx(h1 * kLog2e));
          pn[j / 2] = pack_bf16(ex2_approx(-h0 * kLog2e), ex2_approx(-h1 * kLog2e));
        }
        tmem_st32(tmem + lb + TM_Y(eg), pp);
        tmem_st32(tmem + lb + TM_Y(eg) + 32, pn);
      }
      {
        uint32_t hv[64];
        tmem_ld64(tmem + lb + TM_X(eg), hv);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t wpos[4], wneg[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * c + 2 * e;
            const float h0 = __uint_as_float(hv[j]) + bk_s[j];
            const float h1 = __uint_as_float(hv[j + 1]) + bk_s[j + 1];
            wpos[e] = valid ? pack_bf16(ex2_approx(h0 * kLog2e), ex2_approx(h1 * kLog2e)) : 0u;
            wneg[e] = valid ? pack_bf16(ex2_approx(-h0 * kLog2e), ex2_approx(-h1 * kLog2e)) : 0u;
          }
          st_shared_v4(base + S_PHK + sw128_chunk(row, c), wpos[0], wpos[1], wpos[2], wpos[3]);
          st_shared_v4(base + S_PHK + 16384 + sw128_chunk(row, c), wneg[0], wneg[1], wneg[2],
                       wneg[3]);
        }
      }
      // S_bf16 and z of the tokens before this tile; G2(t) may run only after this
      if (i > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G2 + ((i - 1) & 1)), ((i - 1) >> 1) & 1, wp))) break;
        tc_fence_after();
      }
      {
        uint32_t sv[64];
        tmem_ld64(tmem + lb + TM_S, sv);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int j = 8 * c;
          st_shared_v4(base + S_Q + sw128_chunk(row, c),
                       pack_bf16(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                       pack_bf16(__uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3])),
                       pack_bf16(__uint_as_float(sv[j + 4]), __uint_as_float(sv[j + 5])),
                       pack_bf16(__uint_as_float(sv[j + 6]), __uint_as_float(sv[j + 7])));
        }
        uint32_t zv[16];
        tmem_ld16(tmem + lb + TM_Z, zv);
        zsn[row] = __uint_as_float(zv[0]);
      }

      tmem_st_wait();
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E1A + eg));
      named_bar_sync(1 + eg, 128);   // z snapshot of every feature written
      float den = 0.f;
      {
        uint32_t qp[64];
        tmem_ld64(tmem + lb + TM_Y(eg), qp);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          den += bf16_lo(qp[c]) * zsn[2 * c] + bf16_hi(qp[c]) * zsn[2 * c + 1];
      }

      // ---- E2: P = bf16(tril(Sc)) and its row sums ----
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G2 + eg), par, wp))) break;
      tc_fence_after();
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t sv[64];
        tmem_ld64(tmem + lb + TM_X(eg) + 64 * hb, sv);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = 64 * hb + 8 * c + 2 * e;
            const float a0 = key <= row ? __uint_as_float(sv[8 * c + 2 * e]) : 0.f;
            const float a1 = key + 1 <= row ? __uint_as_float(sv[8 * c + 2 * e + 1]) : 0.f;
            w4[e] = pack_bf16(a0, a1);
            den += bf16_lo(w4[e]) + bf16_hi(w4[e]);
          }
          st_shared_v4(base + S_PHK + hb * 16384 + sw128_chunk(row, c), w4[0], w4[1], w4[2], w4[3]);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E12 + eg));

      // ---- E3: y = O / den ----
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_G3 + eg), par, wp))) break;
      tc_fence_after();
      {
        uint32_t ov[64];
        tmem_ld64(tmem + lb + TM_X(eg), ov);
        const float inv = 1.f / den;
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(A.y + ((size_t)unit * A.n + r0 + row) * D);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int j = 8 * c;
            dst[c] = make_uint4(
                pack_bf16(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv),
                pack_bf16(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv),
                pack_bf16(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv),
                pack_bf16(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_E3 + eg));
    }
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
    uint32_t zv[16];
    tmem_ld16(tmem + lane_base(warp) + TM_Z, zv);
    A.z_out[(size_t)unit * DP + f] = __uint_as_float(zv[0]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t planes,
              uint32_t box_rows) {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Output pass of the d = 64 Hedgehog prefill (two tiles in flight per CTA).
cudaError_t launch_prefill_out_d64(const Problem& p, const TcPlan& pl, const void* q,
                                   const void* k, const void* v, void* y, float* S_out,
                                   float* z_out, const void* ws, int* dev_status, cudaStream_t s) {
  Args2 a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  bool ok = make_map(&a.tq, q, D, p.n, U, TILE) && make_map(&a.tk, k, D, p.n, U, TILE) &&
            make_map(&a.tv, v, D, p.n, U, TILE) && make_map(&a.twq, p.Wq, D, D, p.H, D) &&
            make_map(&a.twk, p.Wk ? p.Wk : p.Wq, D, D, p.H, D);
  if (!ok) return cudaErrorInvalidValue;
  a.y = reinterpret_cast<__nv_bfloat16*>(y);
  a.ws = reinterpret_cast<const float*>(ws);
  a.S_out = S_out;
  a.z_out = z_out;
  a.bq = p.bq;
  a.bk = p.Wk ? p.bk : p.bq;
  a.dev_status = dev_status;
  a.soft_ns = wait_soft_limit_ns();
  a.hard_ns = std::max<uint64_t>(a.soft_ns, 4000000000ull);
  a.n = p.n;
  a.H = p.H;
  a.P = pl.P;
  a.L = pl.L;
  a.NT = pl.NT;
  a.sep_wk = p.Wk ? 1 : 0;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc2_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  prefill_tc2_kernel<<<(unsigned)(U * pl.P), kThreads, SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace hh
