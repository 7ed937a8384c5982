// Chunked causal prefill, output pass, for Hedgehog d = 128 (feature dim 256)
// with one map shared by queries and keys.
//
// Mathematics: "The Hedgehog & the Porcupine" summary, "2. Context and
// Motivation" (paper Eq. 2) for y, "Complexity Analysis" for the running sums
// S = sum phi(k)^T v and z = sum phi(k); the map is "The Hedgehog MLP Feature
// Map", Choices 1 and 3 (Choice 4, Eq. 5, with the softmax-map offsets).
//
// At d = 128 the fp32 state S [256 x 128] alone takes half of the tensor
// memory, so one 128-token tile is in flight.  The pass is organised to keep
// that tile's chain short:
//   warp 16 (MMA issuer) issues every group as soon as its inputs are ready,
//   warp 17 (loads and stores) moves tiles by TMA,
//   warps 0-15 (epilogue) run the CUDA-core phases, four warps per TMEM lane
//   quarter, each on a quarter of the columns (the phases are latency-bound,
//   so more warps with less work each finish them sooner).
// Per tile t (groups G on the tensor pipe, phases E on the epilogue), in the
// order of the chain:
//   G1K  H_K^T = W^T K_t^T        hidden units on the TMEM lanes, tokens on columns
//        (issued once G3a(t-1) is done: it overwrites the columns of phi(Q)(t-1))
//   G1Q  H_Q   = Q_t W            tokens on the lanes
//   E1K  phi(K_t) -> shared memory as [feature][token] rows: thread j owns hidden
//        unit j, so z (the column sums of phi(K)) is a per-thread sum
//   E1Q  phi(Q_t) -> TMEM in place of H_Q (bf16 pairs, A operand of G2S / G3a),
//        and phi(q) . z_before per row
//   G2S  Sc = phi(Q_t) phi(K_t)^T
//   E1S  S_bf16 <- S, the state of the tokens before t (B operand of G3a)
//   G2U  S += phi(K_t)^T V_t
//   E2   P = bf16(tril(Sc)) and its row sums (Sc released as soon as it is
//        loaded); P over phi(K) once G2U has read it
//   G3a  O = phi(Q_t) S_bf16
//   G3b  O += P V_t
//   E3   y = O / (rowsum(P) + phi(q) . z_before), staged over V_t for a TMA store
// The epilogue phases loop over 32-column chunks rather than unrolling whole
// rows: the first tile of every CTA runs its code cold, and a compact body
// costs less there than it loses to one more TMEM-load wait per chunk.
// A 128-row tile covers two 64-token chunks with the exact causal mask.
//
// Feature order inside the pass: the 256 features are grouped by pairs of
// hidden units, f = 4 p + 2 s + e for hidden unit u = 2 p + e (e = 0, 1) and
// sign s (0: exp(+h), 1: exp(-h)).  As bf16 pairs, the two columns H_Q[:, u]
// and H_Q[:, u + 1] (u even) then become packed columns u (exp(+h) of both)
// and u + 1 (exp(-h) of both): each epilogue thread converts its own columns
// in place, in registers, with no exchange between threads.  Workspace
// states, the initial state and the exported S, z use the public order
// (exp(+h) block, then exp(-h) block) and are mapped on the way in and out.
//
// Long sequences are cut into segments exactly as for the other output passes:
// segment s starts from the scanned state of segments 0..s-1 (tc_prefill.cu,
// tc_state.cu).  Every mbarrier wait is bounded (tc_ptx.cuh).

#include <math.h>
#include <string.h>

#include <algorithm>

#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace hh {
namespace {

using namespace tc;

namespace p128 {
constexpr int D = 128, DP = 256, TILE = 128;
constexpr int kEpi = 16;                 // epilogue warps 0-15
constexpr int kMmaWarp = kEpi, kLoadWarp = kEpi + 1;
constexpr int kThreads = 32 * (kEpi + 2);

// TMEM columns
constexpr uint32_t TM_S = 0;     // S: block c (internal features 128c..) x 128 columns at 128 c
// Two 128-column regions swap roles every tile: tile t uses region t % 2 for
// H_K^T -> Sc -> O and the other for H_Q -> phi(Q) (bf16 pairs).  H_K^T of
// tile t+1 can then be computed as soon as G3a(t) has read phi(Q)(t), while
// E3(t) still reads O(t) from the other region.
__host__ __device__ constexpr uint32_t TM_A(int t) { return 256 + 128 * (t & 1); }
__host__ __device__ constexpr uint32_t TM_B(int t) { return 384 - 128 * (t & 1); }

// shared memory (byte offsets from a 1024-aligned base).  K has a buffer of
// its own, so K(t+1) loads while tile t is still in flight; Q shares its
// buffer with the first panel of S_bf16.  Small per-tile arrays live in
// regions that are dead while they are used.
constexpr uint32_t OFF_W = 0;                   // W [128 d][128 hidden]: 2 panels [128 x 64]
constexpr uint32_t OFF_K = 32768;               // K tile: 2 panels [128 tokens x 64]
constexpr uint32_t OFF_Q = OFF_K + 32768;       // Q tile: 2 panels [128 tokens x 64]
constexpr uint32_t OFF_SB = OFF_Q;              // S_bf16 [256 features][128]: 2 panels [256 x 64]
constexpr uint32_t OFF_SB1 = OFF_SB + 32768;    //   its second panel
constexpr uint32_t OFF_ZT = OFF_SB1;           // float[4][256] column sums of phi(K) per token
                                                //   quarter, read before the snapshot overwrites them
constexpr uint32_t OFF_OK = OFF_SB1 + 4096;     // float2[16 warps][32] key offsets of each warp's
                                                //   token quarter (softmax map), likewise
constexpr uint32_t OFF_V = OFF_SB + 65536;      // V tile: 2 panels [128 tokens x 64]; then y
constexpr uint32_t OFF_PHK = OFF_V + 32768;     // phi(K) [256 features][128 tokens]: 2 panels
                                                // [256 x 64]; then P (2 panels [128 x 64])
constexpr uint32_t OFF_DQ = OFF_PHK + 32768;    // float[4][128] phi(q) . z partials  } upper half of
constexpr uint32_t OFF_RS = OFF_DQ + 2048;      // float[4][128] row sums of P        } phi(K), P's time
constexpr uint32_t OFF_Z = OFF_PHK + 65536;     // float[256] z before the tile (internal order)
constexpr uint32_t OFF_BS = OFF_Z + 1024;       // float[128] b * log2(e)
constexpr uint32_t OFF_BAR = OFF_BS + 512;
enum Bar {
  B_W, B_LDK, B_LDQ, B_LDV, B_G1K, B_G1Q, B_E1K, B_E1Q, B_E1S, B_G2S, B_G2U, B_E2A, B_E2B,
  B_G3A, B_G3, B_E3, B_COUNT
};
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;   // tmem base, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
}  // namespace p128

struct Args128 {
  CUtensorMap tq, tk, tv, tw, ty;
  const float* ws;     // [U][P-1][DP*D + DP] inclusive prefixes of segment states (public order)
  const float* init;   // [U][DP*D + DP] initial state (continuation), same layout, or null
  float* S_out;        // [U][DP][D] or null
  float* z_out;        // [U][DP] or null
  const float* bias;   // [H][D] or null
  const float2* offq;  // softmax map: [U][NT*128] per-row offsets (log2 units), else null
  const float2* offk;
  int* dev_status;
  uint64_t soft_ns, hard_ns;
  int64_t n;
  int H, P, L, NT;
  int G;      // query heads per key/value head
  int seq;    // q, k, v, y are [B][n][H][D]
  int early;  // an earlier kernel of this call has waited for the work before
              // the call: q, k, v and W may be read before this kernel's wait
};

__device__ __forceinline__ uint32_t lane_base(int warp) {
  return (uint32_t)(32 * (warp & 3)) << 16;
}

// Public feature (exp(+h) block 0..127, exp(-h) block 128..255) of internal
// feature f = 4 p + 2 s + e (hidden unit 2 p + e, sign s).
__device__ __forceinline__ int public_feature(int f) {
  return ((f >> 1) & 1) * 128 + 2 * (f >> 2) + (f & 1);
}
// Internal feature of hidden unit u with sign s.
__device__ __forceinline__ int internal_feature(int u, int s) {
  return 4 * (u >> 1) + 2 * s + (u & 1);
}

// The bound of 640 threads caps registers at 96 per thread: five warps (0, 4,
// 8, 12, 16 and 1, 5, 9, 13, 17) share one SM sub-partition's registers.
// SM: softmax-over-features map (offsets from the feature-map kernel).
template <bool SM>
__global__ void __launch_bounds__(640, 1) prefill_t128_kernel(const __grid_constant__ Args128 A) {
  using namespace p128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int b) { return bars + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + OFF_MISC + 4);
  float* z_s = reinterpret_cast<float*>(sm + OFF_Z);
  float* zt_s = reinterpret_cast<float*>(sm + OFF_ZT);
  float* dq_s = reinterpret_cast<float*>(sm + OFF_DQ);
  float* rs_s = reinterpret_cast<float*>(sm + OFF_RS);
  float* bs_s = reinterpret_cast<float*>(sm + OFF_BS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x / A.P;
  // batch, query head and key/value head of this unit (split once)
  const int ub = (int)(unit / A.H), uh = (int)(unit % A.H), kh = uh / A.G;
  const int seg = blockIdx.x % A.P;
  const int t_begin = seg * A.L;
  const int nt = min(A.NT, t_begin + A.L) - t_begin;
  WaitPolicy wp{A.soft_ns, A.hard_ns, A.dev_status, abort_flag};

  if (tid == 0) {
    for (int b = 0; b < B_COUNT; ++b) {
      const bool by_warps =
          b == B_E1K || b == B_E1Q || b == B_E1S || b == B_E2A || b == B_E2B || b == B_E3;
      mbar_init(bar(b), by_warps ? kEpi : 1);
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
  auto load_k = [&](int i) {
    const int r0 = (t_begin + i) * TILE;
    mbar_expect_tx(bar(B_LDK), 32768);
    for (int x = 0; x < 2; ++x)
      tma_load_rows(sb + OFF_K + x * 16384, &A.tk, bar(B_LDK), 64 * x, r0, ub, kh, A.seq);
  };
  auto load_q = [&](int i) {
    const int r0 = (t_begin + i) * TILE;
    mbar_expect_tx(bar(B_LDQ), 32768);
    for (int x = 0; x < 2; ++x)
      tma_load_rows(sb + OFF_Q + x * 16384, &A.tq, bar(B_LDQ), 64 * x, r0, ub, uh, A.seq);
  };
  auto load_v = [&](int i) {
    const int r0 = (t_begin + i) * TILE;
    mbar_expect_tx(bar(B_LDV), 32768);
    for (int x = 0; x < 2; ++x)
      tma_load_rows(sb + OFF_V + x * 16384, &A.tv, bar(B_LDV), 64 * x, r0, ub, kh, A.seq);
  };
  auto prefetch_tile = [&](int i) {
    const int r0 = (t_begin + i) * TILE;
    for (int x = 0; x < 2; ++x) {
      tma_prefetch_rows(&A.tq, 64 * x, r0, ub, uh, A.seq);
      tma_prefetch_rows(&A.tk, 64 * x, r0, ub, kh, A.seq);
      tma_prefetch_rows(&A.tv, 64 * x, r0, ub, kh, A.seq);
    }
  };
  auto first_loads = [&]() {
    mbar_expect_tx(bar(B_W), D * D * 2);
    for (int x = 0; x < 2; ++x) tma_load_3d(sb + OFF_W + x * 16384, &A.tw, bar(B_W), 64 * x, 0, uh);
    load_k(0);
    load_q(0);
    load_v(0);
    if (nt > 1) prefetch_tile(1);
  };
  const bool loader = warp == kLoadWarp && lane == 0 && nt > 0;
  if (A.early) {
    // The inputs of this call (q, k, v, W) are final: the first kernel of the
    // call let the next one be scheduled only after its own wait for the
    // work before the call, and every later kernel of it after that.  So W
    // and the first tile may land while the kernels before this one finish;
    // the workspace (segment prefixes) is read only after the wait below.
    __syncthreads();   // the barriers are initialised
    if (loader) first_loads();
  } else if (loader) {
    // this kernel may be the call's first: W and the first tile into L2
    // only (a prefetch just warms the cache, so it may precede the wait)
    const int r0 = t_begin * TILE;
    for (int x = 0; x < 2; ++x) {
      tma_prefetch_3d(&A.tw, 64 * x, 0, uh);
      tma_prefetch_rows(&A.tk, 64 * x, r0, ub, kh, A.seq);
      tma_prefetch_rows(&A.tq, 64 * x, r0, ub, uh, A.seq);
      tma_prefetch_rows(&A.tv, 64 * x, r0, ub, kh, A.seq);
    }
  }
  // the next kernel may be scheduled now; this one reads the workspace and
  // writes global memory only once the kernels before it have completed
  pdl_launch_dependents();
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  if (!A.early && loader) first_loads();
  for (int i = tid; i < D; i += kThreads) bs_s[i] = A.bias ? A.bias[(size_t)uh * D + i] * kLog2e : 0.f;
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // initial state: the prefix of the preceding segments, the given initial
  // state (continuation, first segment) or zeros; public -> internal order
  // warp w: lane quarter w % 4, column quarter w / 4: feature row 128 c + r
  // (c = w / 8) and state columns [64 ((w / 4) % 2), +64)
  if (warp < kEpi) {
    const int q = warp >> 2, c = q >> 1, r = 32 * (warp & 3) + lane;
    const int fp = public_feature(128 * c + r);
    const size_t per = (size_t)DP * D + DP;
    const float* prefix = seg > 0 ? A.ws + ((size_t)unit * (A.P - 1) + seg - 1) * per
                                  : (A.init ? A.init + (size_t)unit * per : nullptr);
    // all 64 values of this thread requested at once (one L2 round trip)
    const int cb = 64 * (q & 1);
    uint32_t v[64];
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      const float4 v4 = prefix ? __ldcg(reinterpret_cast<const float4*>(prefix + ws_s_index(fp, cb + j, D)))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      v[j] = __float_as_uint(v4.x);
      v[j + 1] = __float_as_uint(v4.y);
      v[j + 2] = __float_as_uint(v4.z);
      v[j + 3] = __float_as_uint(v4.w);
    }
    const float zv = ((q & 1) == 0 && prefix) ? __ldcg(prefix + (size_t)DP * D + fp) : 0.f;
    tmem_st32(tmem + lane_base(warp) + TM_S + 128 * c + cb, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
    tmem_st32(tmem + lane_base(warp) + TM_S + 128 * c + cb + 32,
              *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
    if ((q & 1) == 0) z_s[128 * c + r] = zv;
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kMmaWarp) {
    // ======================= MMA issuer =======================
    if (lane == 0 && nt > 0) {
      constexpr uint32_t ID_HKT = idesc_bf16(128, 128, 1, 0);  // W^T[MN-major] K^T[K-major]
      constexpr uint32_t ID_MN = idesc_bf16(128, 128, 0, 1);   // A K-major / TMEM, B MN-major
      // descriptor bases; a k-step only moves the 14-bit start-address field (16-byte units)
      const uint64_t dWa = smem_desc(sb + OFF_W, 16384, 1024, 2);     // W^T as MN-major A
      const uint64_t dWb = smem_desc(sb + OFF_W, 16384, 1024, 2);     // W as MN-major B
      const uint64_t dQ = smem_desc(sb + OFF_Q, 16, 1024, 2);         // K-major
      const uint64_t dK = smem_desc(sb + OFF_K, 16, 1024, 2);
      const uint64_t dV = smem_desc(sb + OFF_V, 16384, 1024, 2);      // MN-major, N = d
      const uint64_t dPk = smem_desc(sb + OFF_PHK, 16, 1024, 2);      // phi(K)^T as K-major A
      const uint64_t dPn = smem_desc(sb + OFF_PHK, 32768, 1024, 2);   // phi(K)^T as MN-major B
      const uint64_t dSb = smem_desc(sb + OFF_SB, 32768, 1024, 2);    // S_bf16, MN-major B
      const uint64_t dP = smem_desc(sb + OFF_PHK, 16, 1024, 2);       // P, K-major A
      auto kmaj = [](int ks) { return (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2); };
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const uint32_t par = i & 1;
        const uint32_t tA = tmem + TM_A(i), tB = tmem + TM_B(i);
        // G1K: K of tile i landed; region A(i) held phi(Q)(i-1), the A operand of
        // G3a(i-1) (issued by this thread before, waited for here)
        ok = (i > 0 || mbar_wait_poll(bar(B_W), 0, wp)) &&
             mbar_wait_poll(bar(B_LDK), par, wp) &&
             (i == 0 || mbar_wait_poll(bar(B_G3A), par ^ 1, wp));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tA, dWa + 128 * ks, dK + kmaj(ks), ID_HKT, ks > 0);
        mma_commit(bar(B_G1K));
        // G1Q: Q(i) landed (it is requested later than K(i); E1K runs
        // meanwhile) and E3(i-1) has read O(i-1) out of region B(i)
        ok = mbar_wait_poll(bar(B_LDQ), par, wp) &&
             (i == 0 || mbar_wait_poll(bar(B_E3), par ^ 1, wp));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tB, dQ + kmaj(ks), dWb + 128 * ks, ID_MN, ks > 0);
        mma_commit(bar(B_G1Q));
        // G2S: phi(K) in shared memory, phi(Q) in TMEM (H_K^T has been read out of A)
        ok = mbar_wait_poll(bar(B_E1K), par, wp) && mbar_wait_poll(bar(B_E1Q), par, wp);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tA, tB + 8 * ks, dPn + 128 * ks, ID_MN, ks > 0);
        mma_commit(bar(B_G2S));
        // G2U: S_bf16 holds the state before the tile, V(i) landed
        ok = mbar_wait_poll(bar(B_E1S), par, wp) && mbar_wait_poll(bar(B_LDV), par, wp);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int ks = 0; ks < TILE / 16; ++ks)
            mma_ss(tmem + TM_S + 128 * mb, dPk + (ks >> 2) * 2048 + mb * 1024 + (ks & 3) * 2,
                   dV + 128 * ks, ID_MN, 1);
        mma_commit(bar(B_G2U));
        // G3a: Sc has been read out of A
        ok = mbar_wait_poll(bar(B_E2A), par, wp);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks)
          mma_ts(tA, tB + 8 * ks, dSb + 128 * ks, ID_MN, ks > 0);
        mma_commit(bar(B_G3A));
        // G3b: P is in shared memory
        ok = mbar_wait_poll(bar(B_E2B), par, wp);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ss(tA, dP + kmaj(ks), dV + 128 * ks, ID_MN, 1);
        mma_commit(bar(B_G3));
      }
      if (!ok) *(volatile int*)abort_flag = 1;
    }
  } else if (warp == kLoadWarp) {
    // ======================= loads and stores =======================
    //   K (i+1) once G1K(i) has read K(i);
    //   Q (i+1) once G3a(i) has read S_bf16, whose first panel overwrites Q;
    //   y(i), staged over V(i), once E3(i) has written it; then V(i+1).
    if (lane == 0 && nt > 0) {
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const uint32_t par = i & 1;
        if (i + 1 < nt) {
          ok = mbar_wait_poll(bar(B_G1K), par, wp);
          if (!ok) break;
          load_k(i + 1);
          ok = mbar_wait_poll(bar(B_G3A), par, wp);
          if (!ok) break;
          load_q(i + 1);
        }
        ok = mbar_wait_poll(bar(B_E3), par, wp);
        if (!ok) break;
        const int r0 = (t_begin + i) * TILE;
        tma_store_rows(&A.ty, sb + OFF_V, 0, r0, ub, uh, A.seq);
        tma_store_rows(&A.ty, sb + OFF_V + 16384, 64, r0, ub, uh, A.seq);
        tma_store_commit();
        if (i + 1 < nt) {
          tma_store_wait_read_all();
          load_v(i + 1);
          if (i + 2 < nt) prefetch_tile(i + 2);
        }
      }
      if (!ok) *(volatile int*)abort_flag = 1;
      tma_store_wait_all();   // y written before the CTA retires
    }
  } else {
    // ======================= epilogue warps =======================
    // Warp w owns TMEM lanes 32 (w % 4).. and column quarter q = w / 4: in E1K
    // hidden unit j = lane and tokens [32q, +32); elsewhere tile row r = lane
    // and columns [32q, +32).
    const int q = warp >> 2;
    const int g = warp & 3;
    const int r = 32 * g + lane;
    const uint32_t lb = lane_base(warp);
    // A wait that gives up (hard time limit) clears `good`: the warp then
    // skips all further work but still passes every named barrier, so the
    // other epilogue warps never wait for it there.  `good` is warp-uniform.
    bool good = true;
    auto wait_all = [&](int b, uint32_t par) {
      good = good && __all_sync(0xffffffffu, mbar_wait(bar(b), par, wp));
      return good;
    };
    auto epi_sync = [&]() { named_bar_sync(1, 32 * kEpi); };
    // softmax map: lane l holds the key offsets of token 32 q + l of the next
    // tile, loaded a tile ahead
    const float2* offk_u = A.offk + (size_t)unit * A.NT * TILE + (size_t)t_begin * TILE + 32 * q + lane;
    float2 ok_next = make_float2(0.f, 0.f);
    if (SM && nt > 0) ok_next = __ldg(offk_u);
    for (int i = 0; i < nt; ++i) {
      const uint32_t par = i & 1;
      const int64_t r0 = (int64_t)(t_begin + i) * TILE;
      // softmax map: this row's query offsets, requested before they are needed
      float2 oq = make_float2(0.f, 0.f);
      if (SM) oq = A.offq[(size_t)unit * A.NT * TILE + (size_t)r0 + r];

      // ---------------- E1K: phi(K) rows of hidden unit j = r ----------------
      // phi(K) overwrites the dq / rs partials of the previous tile: every
      // warp must be past its E3 (G1K no longer waits for E3)
      if (i > 0) epi_sync();
      wait_all(B_G1K, par);
      tc_fence_after();
      // softmax map: this warp's copy of its quarter's key offsets, over the
      // snapshot panel (G3a of the previous tile, its last reader, completed
      // before G1K was issued); the next tile's are requested at once
      float2* okw = reinterpret_cast<float2*>(sm + OFF_OK) + 32 * warp;
      if (SM) {
        okw[lane] = ok_next;
        __syncwarp();
        if (i + 1 < nt) ok_next = __ldg(offk_u + (size_t)(i + 1) * TILE);
      }
      const int fpos = internal_feature(r, 0), fneg = internal_feature(r, 1);
      if (good) {
        const float bj = bs_s[r];
        float zp = 0.f, zn = 0.f;
        // two rows per thread; lanes with bit 2 set store their negative row
        // first, so each store's 32 rows cover all eight 16-byte bank groups
        // of the swizzle four times (no extra wavefronts)
        const bool neg_first = (r & 4) != 0;
        const int f0 = neg_first ? fneg : fpos, f1 = neg_first ? fpos : fneg;
        const uint32_t panel = sb + OFF_PHK + (q >> 1) * 32768;   // tokens [64 (q/2), +64)
        uint32_t hk[32];
        tmem_ld32(tmem + lb + TM_A(i) + 32 * q, hk);
        // tokens of this quarter inside the sequence (32 except in the last tile)
        const int64_t left = A.n - (r0 + 32 * q);
        const int nv = left <= 0 ? 0 : (left >= 32 ? 32 : (int)left);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t wpos[4], wneg[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tt = 8 * qq + 2 * e;
            const float a0 = fmaf(__uint_as_float(hk[tt]), kLog2e, bj);
            const float a1 = fmaf(__uint_as_float(hk[tt + 1]), kLog2e, bj);
            float e0, e1, f0, f1;
            if (SM) {
              const float4 o2 = *reinterpret_cast<const float4*>(okw + tt);
              e0 = ex2_approx(a0 - o2.x); e1 = ex2_approx(a1 - o2.z);
              f0 = ex2_approx(-a0 - o2.y); f1 = ex2_approx(-a1 - o2.w);
            } else {
              e0 = ex2_approx(a0); e1 = ex2_approx(a1);
              f0 = ex2_approx(-a0); f1 = ex2_approx(-a1);
            }
            // tokens past the end of the sequence contribute nothing
            if (nv < 32) {
              if (tt >= nv) e0 = f0 = 0.f;
              if (tt + 1 >= nv) e1 = f1 = 0.f;
            }
            // z sums the fp32 features; the MMA operand is their bf16 rounding
            // (a relative mismatch of at most 2^-9 per term, inside the output's
            // own bf16 rounding)
            zp += e0 + e1;
            zn += f0 + f1;
            wpos[e] = pack_bf16(e0, e1);
            wneg[e] = pack_bf16(f0, f1);
          }
          const int ch = 4 * (q & 1) + qq;   // 16-byte chunk of the 128-byte row
          st_shared_v4(panel + sw128_chunk(f0, ch), neg_first ? wneg[0] : wpos[0],
                       neg_first ? wneg[1] : wpos[1], neg_first ? wneg[2] : wpos[2],
                       neg_first ? wneg[3] : wpos[3]);
          st_shared_v4(panel + sw128_chunk(f1, ch), neg_first ? wpos[0] : wneg[0],
                       neg_first ? wpos[1] : wneg[1], neg_first ? wpos[2] : wneg[2],
                       neg_first ? wpos[3] : wneg[3]);
        }
        // this thread's share of z: the column sums of phi(K) for its hidden
        // unit over its token quarter (added to z once every reader of
        // z_before is done)
        zt_s[256 * q + fpos] = zp;
        zt_s[256 * q + fneg] = zn;
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (good && lane == 0) mbar_arrive(bar(B_E1K));

      // ---------------- E1Q: phi(Q) in place, phi(q) . z_before ----------------
      float dq = 0.f;   // this thread's quarter of phi(q) . z_before (shared after G2U)
      wait_all(B_G1Q, par);
      tc_fence_after();
      if (good) {
        // columns 32q + u, u + 1 (u even) of H_Q become packed columns 32q + u
        // (exp(+h) of both) and 32q + u + 1 (exp(-h) of both): internal
        // features 4 (16q + u/2) .. + 3.  Bias and z are re-read from shared
        // memory at their point of use (volatile loads: hoisted, they would
        // cost registers).
        uint32_t hq[32];
        tmem_ld32(tmem + lb + TM_B(i) + 32 * q, hq);
        const uint32_t zaddr = sb + OFF_Z + 4 * 64 * q;
        const uint32_t baddr = sb + OFF_BS + 4 * 32 * q;
#pragma unroll
        for (int u = 0; u < 32; u += 4) {
          const float4 b4 = ld_shared_f4_volatile(baddr + 4 * u);
          const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float a0 = fmaf(__uint_as_float(hq[u + e]), kLog2e, bb[e]);
            const float a1 = fmaf(__uint_as_float(hq[u + e + 1]), kLog2e, bb[e + 1]);
            const uint32_t p = pack_bf16(ex2_approx(a0 - oq.x), ex2_approx(a1 - oq.x));
            const uint32_t m = pack_bf16(ex2_approx(-a0 - oq.y), ex2_approx(-a1 - oq.y));
            hq[u + e] = p;
            hq[u + e + 1] = m;
            const float4 zz = ld_shared_f4_volatile(zaddr + 8 * (u + e));
            dq += bf16_lo(p) * zz.x + bf16_hi(p) * zz.y + bf16_lo(m) * zz.z + bf16_hi(m) * zz.w;
          }
        }
        tmem_st32(tmem + lb + TM_B(i) + 32 * q, hq);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (good && lane == 0) mbar_arrive(bar(B_E1Q));

      // Every warp is past its reads of z_before (E1Q) and has written its
      // column sums: z takes the four token quarters' sums in order; then the
      // snapshot may overwrite them and the key offsets (same panel).
      epi_sync();
      if (good && q < 2) {
        const int f = 128 * q + r;   // one internal feature per thread of the first half
        z_s[f] = z_s[f] + ((zt_s[f] + zt_s[256 + f]) + (zt_s[512 + f] + zt_s[768 + f]));
      }
      epi_sync();

      // ---------------- E1S: S_bf16 <- S (the state before this tile) ----------------
      // feature row 128 (q / 2) + r, columns [64 (q % 2), +64); over Q, which
      // G1Q (complete) has read; G2U of the previous tile completed before G1K
      // of this one
      if (good) {
        const int c = q >> 1;
        const int f = 128 * c + r;
        const uint32_t panel = sb + OFF_SB + (q & 1) * 32768;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t sv[32];
          tmem_ld32(tmem + lb + TM_S + 128 * c + 64 * (q & 1) + c0, sv);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int j = 8 * q4;
            st_shared_v4(panel + sw128_chunk(f, c0 / 8 + q4),
                         pack_bf16(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])),
                         pack_bf16(__uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3])),
                         pack_bf16(__uint_as_float(sv[j + 4]), __uint_as_float(sv[j + 5])),
                         pack_bf16(__uint_as_float(sv[j + 6]), __uint_as_float(sv[j + 7])));
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (good && lane == 0) mbar_arrive(bar(B_E1S));

      // ---------------- E2: P = bf16(tril(Sc)), row sums ----------------
      wait_all(B_G2S, par);
      tc_fence_after();
      if (good) {
        uint32_t pw[16];   // keys [32q, +32) of row r as bf16 pairs
        float rs = 0.f;
        if (g < q) {
          // every row of this warp lies above the keys of quarter q: P = 0
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_E2A));
#pragma unroll
          for (int j = 0; j < 16; ++j) pw[j] = 0u;
        } else {
          uint32_t sv[32];
          tmem_ld32(tmem + lb + TM_A(i) + 32 * q, sv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_E2A));   // Sc is out of A: G3a may overwrite it
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int key = 32 * q + j;
            const float a0 = key <= r ? __uint_as_float(sv[j]) : 0.f;
            const float a1 = key + 1 <= r ? __uint_as_float(sv[j + 1]) : 0.f;
            const uint32_t w2 = pack_bf16(a0, a1);
            pw[j / 2] = w2;
            rs += bf16_lo(w2) + bf16_hi(w2);
          }
        }
        // P, and the row's dq and rs partials, over phi(K) once G2U, the last
        // reader of phi(K), has completed
        if (wait_all(B_G2U, par)) {
          const uint32_t panel = sb + OFF_PHK + (q >> 1) * 16384;   // keys [64 (q/2), +64)
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            st_shared_v4(panel + sw128_chunk(r, 4 * (q & 1) + qq), pw[4 * qq], pw[4 * qq + 1],
                         pw[4 * qq + 2], pw[4 * qq + 3]);
          dq_s[128 * q + r] = dq;
          rs_s[128 * q + r] = rs;
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_E2B));
        }
      }
      epi_sync();   // every row's dq and rs partials are in shared memory

      // ---------------- E3: y = O / den ----------------
      wait_all(B_G3, par);
      tc_fence_after();
      if (good) {
        const float den = ((dq_s[r] + dq_s[128 + r]) + (dq_s[256 + r] + dq_s[384 + r])) +
                          ((rs_s[r] + rs_s[128 + r]) + (rs_s[256 + r] + rs_s[384 + r]));
        const float inv = 1.f / den;
        const uint32_t panel = sb + OFF_V + (q >> 1) * 16384;   // y columns [64 (q/2), +64), over V
        uint32_t ov[32];
        tmem_ld32(tmem + lb + TM_A(i) + 32 * q, ov);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int j = 8 * qq;
          st_shared_v4(panel + sw128_chunk(r, 4 * (q & 1) + qq),
                       pack_bf16(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv),
                       pack_bf16(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv),
                       pack_bf16(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv),
                       pack_bf16(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv));
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (good && lane == 0) mbar_arrive(bar(B_E3));
    }
  }

  // ---- export the final state of the last segment (public order) ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (A.S_out && seg == A.P - 1 && warp < kEpi && nt > 0 && !*(volatile int*)abort_flag) {
    // the last G2U is complete: E2 of the last tile waited for it
    const int q = warp >> 2, c = q >> 1, r = 32 * (warp & 3) + lane;
    const int fp = public_feature(128 * c + r);
    float4* dst = reinterpret_cast<float4*>(A.S_out + ((size_t)unit * DP + fp) * D);
#pragma unroll 1
    for (int c0 = 64 * (q & 1); c0 < 64 * (q & 1) + 64; c0 += 32) {
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base(warp) + TM_S + 128 * c + c0, sv);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[c0 / 4 + j] = make_float4(__uint_as_float(sv[4 * j]), __uint_as_float(sv[4 * j + 1]),
                                      __uint_as_float(sv[4 * j + 2]), __uint_as_float(sv[4 * j + 3]));
    }
    if ((q & 1) == 0) A.z_out[(size_t)unit * DP + fp] = z_s[128 * c + r];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

// Output pass of the d = 128 Hedgehog prefill for a map shared by queries and keys.
cudaError_t launch_prefill_out_d128(const Problem& p, const TcPlan& pl, const void* q,
                                    const void* k, const void* v, void* y, float* S_out,
                                    float* z_out, const void* ws, const float* init,
                                    int* dev_status, cudaStream_t s) {
  using namespace p128;
  Args128 a;
  memset(&a, 0, sizeof(a));
  const uint64_t U = (uint64_t)p.B * p.H;
  if (p.Wk || p.d != D) return cudaErrorInvalidValue;
  if (p.softmax && (!p.offq || !p.offk)) return cudaErrorInvalidValue;
  const int Hkv = p.H / p.G;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  bool ok = make_rows_map(&a.tq, q, D, p.n, p.H, p.B, 64, TILE, sw, p.seq_major) &&
            make_rows_map(&a.tk, k, D, p.n, Hkv, p.B, 64, TILE, sw, p.seq_major) &&
            make_rows_map(&a.tv, v, D, p.n, Hkv, p.B, 64, TILE, sw, p.seq_major) &&
            make_plane_map(&a.tw, p.Wq, D, D, p.H, 64, D, sw) &&
            make_rows_map(&a.ty, y, D, p.n, p.H, p.B, 64, TILE, sw, p.seq_major);
  if (!ok) return cudaErrorInvalidValue;
  a.ws = reinterpret_cast<const float*>(ws);
  a.init = init;
  a.S_out = S_out;
  a.z_out = z_out;
  a.bias = p.bq;
  a.offq = p.offq;
  a.offk = p.offk;
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
  // a state pass, an initial-state kernel or the softmax-map offsets ran
  // first in this call (each of them waits before it lets the next start)
  a.early = (pl.P > 1 || init || p.softmax) ? 1 : 0;
  auto kern = p.softmax ? prefill_t128_kernel<true> : prefill_t128_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)(U * pl.P)), dim3(kThreads), SMEM_BYTES, s, a);
}

}  // namespace hh
