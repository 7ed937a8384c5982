// Float32 CUDA-core kernels: feature map, chunked causal prefill and the
// mimicry loss.  These carry the float32 workloads (1e-5 parity), where the
// tensor cores' bf16/tf32 operands would not be precise enough, and accept
// any head dimension up to 128 (Taylor: up to 16).
//
// Math follows "The Hedgehog & the Porcupine" summary: Choices 1/3 of "The
// Hedgehog MLP Feature Map", "The Taylor Exponential as a Bridge Result",
// "2. Context and Motivation" (paper Eq. 2) and "Complexity Analysis" for the causal output,
// and "The Attention Weight Distillation Loss" (paper Eq. 4).

#include <math.h>

#include "hh_internal.cuh"

namespace hh {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// phi of one row held in shared memory (xs[0..d)), written to out[0..dpp) by
// one whole warp.
// Hedgehog: out[l] = exp(h_l), out[d+l] = exp(-h_l), h = x W + b.
// Softmax map (Choice 4, Eq. 5; no bias): out[l] = exp(h_l - c+),
//   out[d+l] = exp(-h_l - c-), c+- = logsumexp over l of +-h; *off (if given)
//   receives (c+, c-) log2 e.
// Taylor: [1, x, x_i x_j / sqrt2 (i-major)], zero padding.
template <typename T>
__device__ __forceinline__ void phi_row(int kind, bool softmax, int d, int dpp, const float* xs,
                                        const T* W, const float* b, float* out, float2* off,
                                        int lane) {
  if (kind == HH_FMAP_HEDGEHOG) {
    float mx = -INFINITY, mn = INFINITY;
    for (int l = lane; l < d; l += 32) {
      float h = b ? b[l] : 0.f;
      for (int k = 0; k < d; ++k) h = fmaf(xs[k], to_f(W[(size_t)k * d + l]), h);
      if (softmax) {
        out[l] = h;
        mx = fmaxf(mx, h);
        mn = fminf(mn, h);
      } else {
        out[l] = expf(h);
        out[d + l] = expf(-h);
      }
    }
    if (softmax) {
      mx = warp_max(mx);
      mn = -warp_max(-mn);
      float sp = 0.f, sn = 0.f;
      for (int l = lane; l < d; l += 32) {
        sp += expf(out[l] - mx);
        sn += expf(mn - out[l]);
      }
      sp = warp_sum(sp);
      sn = warp_sum(sn);
      const float cp = mx + logf(sp), cn = logf(sn) - mn;
      for (int l = lane; l < d; l += 32) {
        const float h = out[l];
        out[l] = expf(h - cp);
        out[d + l] = expf(-h - cn);
      }
      if (off && lane == 0) *off = make_float2(cp * 1.4426950408889634f, cn * 1.4426950408889634f);
    }
  } else {
    for (int f = lane; f < dpp; f += 32) {
      float val;
      if (f == 0) {
        val = 1.f;
      } else if (f <= d) {
        val = xs[f - 1];
      } else if (f <= d + d * d) {
        int p = f - 1 - d;
        val = xs[p / d] * xs[p % d] * kInvSqrt2;
      } else {
        val = 0.f;
      }
      out[f] = val;
    }
  }
}

// ---------------------------------------------------------------------------
// Feature map: one block per group of rows; one warp per row.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
fmap_simt_kernel(const T* __restrict__ x, const T* __restrict__ W, const float* __restrict__ bias,
                 T* __restrict__ phi, float2* __restrict__ off, int kind, int softmax, int d,
                 int dpp, int H, int G, int seq, int64_t n, int64_t rows) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = kThreads / 32;
  float* xs = sm + warp * (128 + 320);
  float* out = xs + 128;
  for (int64_t r = (int64_t)blockIdx.x * nwarps + warp; r < rows; r += (int64_t)gridDim.x * nwarps) {
    const int h = (int)((r / n) % H);
    // x row: of this query head, or of its key/value head (G > 1: keys)
    const int64_t xr = row_index(kv_unit(r / n, H, G), r % n, H / G, n, seq);
    for (int k = lane; k < d; k += 32) xs[k] = to_f(x[xr * d + k]);
    __syncwarp();
    const T* Wh = W ? W + (size_t)h * d * d : nullptr;
    const float* bh = bias ? bias + (size_t)h * d : nullptr;
    float2* orow = off ? off + (r / n) * ((n + 127) / 128 * 128) + r % n : nullptr;
    phi_row<T>(kind, softmax != 0, d, dpp, xs, Wh, bh, out, orow, lane);
    __syncwarp();
    if (phi)
      for (int f = lane; f < dpp; f += 32) phi[r * dpp + f] = from_f<T>(out[f]);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Chunked causal prefill: one block per (batch, head); chunks of C tokens.
//   A = tril(phi(Q_c) phi(K_c)^T);  y = (A V_c + phi(Q_c) S) / (rowsum A + phi(Q_c) z)
//   S += phi(K_c)^T V_c;  z += phi(K_c)^T 1
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    T* __restrict__ y, float* __restrict__ S_out, float* __restrict__ z_out,
                    const float* __restrict__ S0, const float* __restrict__ z0,
                    const T* __restrict__ Wq, const float* __restrict__ bq,
                    const T* __restrict__ Wk, const float* __restrict__ bk, int kind,
                    int softmax, int d, int dpp, int H, int G, int seq, int64_t n, int C) {
  extern __shared__ float sm[];
  // phi rows are padded to an odd stride so that a warp reading one feature of
  // 32 consecutive rows hits 32 different banks
  const int ps = dpp + 1;
  float* S = sm;                       // [dpp][d]
  float* z = S + (size_t)dpp * d;      // [dpp]
  float* phq = z + dpp;                // [C][ps]
  float* phk = phq + (size_t)C * ps;   // [C][ps]
  float* vv = phk + (size_t)C * ps;    // [C][d]
  float* A = vv + (size_t)C * d;       // [C][C]
  float* xs = A + (size_t)C * C;       // [C][d]  raw rows
  float* xk = xs + (size_t)C * d;      // [C][d]
  float* den = xk + (size_t)C * d;     // [C]

  const int64_t bh = blockIdx.x;
  const int h = (int)(bh % H);
  // batch, query head and key/value head of this unit; element offset of
  // token t of this head in q / y, and in k / v
  const int ub = (int)(bh / H), uh = (int)(bh % H), kh = uh / G;
  auto qrow = [&](int64_t t) { return (size_t)row_of(ub, uh, t, H, n, seq) * d; };
  auto kvrow = [&](int64_t t) { return (size_t)row_of(ub, kh, t, H / G, n, seq) * d; };
  const T* Wqh = Wq ? Wq + (size_t)h * d * d : nullptr;
  const T* Wkh = Wk ? Wk + (size_t)h * d * d : nullptr;
  const float* bqh = bq ? bq + (size_t)h * d : nullptr;
  const float* bkh = bk ? bk + (size_t)h * d : nullptr;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // the state before the first token: zero, or the given one (continuation)
  for (int i = tid; i < dpp * d; i += kThreads) S[i] = S0 ? S0[(size_t)bh * dpp * d + i] : 0.f;
  for (int i = tid; i < dpp; i += kThreads) z[i] = z0 ? z0[(size_t)bh * dpp + i] : 0.f;
  __syncthreads();

  for (int64_t c0 = 0; c0 < n; c0 += C) {
    const int nc = (int)min((int64_t)C, n - c0);
    for (int i = tid; i < C * d; i += kThreads) {
      const int r = i / d;
      const bool ok = r < nc;
      xs[i] = ok ? to_f(q[qrow(c0 + r) + (i % d)]) : 0.f;
      xk[i] = ok ? to_f(k[kvrow(c0 + r) + (i % d)]) : 0.f;
      vv[i] = ok ? to_f(v[kvrow(c0 + r) + (i % d)]) : 0.f;
    }
    __syncthreads();
    for (int r = warp; r < C; r += kThreads / 32) {
      phi_row<T>(kind, softmax != 0, d, dpp, xs + (size_t)r * d, Wqh, bqh, phq + (size_t)r * ps,
                 nullptr, lane);
      phi_row<T>(kind, softmax != 0, d, dpp, xk + (size_t)r * d, Wkh, bkh, phk + (size_t)r * ps,
                 nullptr, lane);
      if (r >= nc)  // ragged tail: padded keys contribute nothing
        for (int f = lane; f < dpp; f += 32) phk[(size_t)r * ps + f] = 0.f;
    }
    __syncthreads();
    // The three contractions below run on 4 x 4 register blocks (8 shared
    // loads per 16 FMAs instead of 32); every output still sums its terms in
    // the same order as a plain loop, so results do not depend on the blocking.
    // A = tril(phi(Q) phi(K)^T): blocks wholly above the diagonal are zero.
    for (int blk = tid; blk < (C / 4) * (C / 4); blk += kThreads) {
      const int r0 = 4 * (blk / (C / 4)), j0 = 4 * (blk % (C / 4));
      float a[4][4] = {};
      if (j0 <= r0) {
        for (int f = 0; f < dpp; ++f) {
          float qv[4], kv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qv[e] = phq[(size_t)(r0 + e) * ps + f];
            kv[e] = phk[(size_t)(j0 + e) * ps + f];
          }
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) a[r][c] = fmaf(qv[r], kv[c], a[r][c]);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) A[(r0 + r) * C + j0 + c] = (j0 + c <= r0 + r) ? a[r][c] : 0.f;
    }
    __syncthreads();
    for (int r = tid; r < C; r += kThreads) {
      float dn = 0.f;
      for (int j = 0; j <= r; ++j) dn += A[r * C + j];
      float di = 0.f;
      for (int f = 0; f < dpp; ++f) di = fmaf(phq[(size_t)r * ps + f], z[f], di);
      den[r] = dn + di;
    }
    __syncthreads();
    // y = (A V + phi(Q) S) / den on 4 rows x 4 columns per thread (A is zero
    // above the diagonal, so running j to the block's last row adds exact zeros)
    const int dq4 = (d + 3) / 4;
    for (int blk = tid; blk < (C / 4) * dq4; blk += kThreads) {
      const int r0 = 4 * (blk / dq4), c0v = 4 * (blk % dq4);
      if (r0 >= nc) continue;
      float num[4][4] = {}, ni[4][4] = {};
      const int jmax = min(r0 + 3, nc - 1);
      for (int j = 0; j <= jmax; ++j) {
        float av[4], vc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          av[e] = A[(r0 + e) * C + j];
          vc[e] = c0v + e < d ? vv[j * d + c0v + e] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) num[r][c] = fmaf(av[r], vc[c], num[r][c]);
      }
      for (int f = 0; f < dpp; ++f) {
        float qv[4], sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qv[e] = phq[(size_t)(r0 + e) * ps + f];
          sc[e] = c0v + e < d ? S[(size_t)f * d + c0v + e] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) ni[r][c] = fmaf(qv[r], sc[c], ni[r][c]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (r0 + r < nc && c0v + c < d)
            y[qrow(c0 + r0 + r) + c0v + c] = from_f<T>((num[r][c] + ni[r][c]) / den[r0 + r]);
    }
    __syncthreads();
    // S += phi(K)^T V on 4 features x 4 columns per thread
    for (int blk = tid; blk < ((dpp + 3) / 4) * dq4; blk += kThreads) {
      const int f0 = 4 * (blk / dq4), c0v = 4 * (blk % dq4);
      float acc[4][4] = {};
      for (int j = 0; j < nc; ++j) {
        float kv[4], vc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kv[e] = f0 + e < dpp ? phk[(size_t)j * ps + f0 + e] : 0.f;
          vc[e] = c0v + e < d ? vv[j * d + c0v + e] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(kv[r], vc[c], acc[r][c]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (f0 + r < dpp && c0v + c < d) S[(size_t)(f0 + r) * d + c0v + c] += acc[r][c];
    }
    for (int f = tid; f < dpp; f += kThreads) {
      float acc = 0.f;
      for (int j = 0; j < nc; ++j) acc += phk[(size_t)j * ps + f];
      z[f] += acc;
    }
    __syncthreads();
  }
  if (S_out) {
    for (int i = tid; i < dpp * d; i += kThreads) S_out[(size_t)bh * dpp * d + i] = S[i];
    for (int i = tid; i < dpp; i += kThreads) z_out[(size_t)bh * dpp + i] = z[i];
  }
}

// ---------------------------------------------------------------------------
// Mimicry loss: one block per (batch*head, tile of 64 queries).  Four threads
// share a query row; each keeps an online-softmax state over its keys:
//   M = running max of s, Z = sum e^{s-M}, T = sum e^{s-M} log a, A = sum a,
//   U = sum e^{s-M} s, V = sum a log a
// and the row's loss is log A - T / Z (= -sum_j p_j log(a_j / A)); the
// entropies are H(p) = log Z + M - U / Z and H(w) = log A - V / A.
// ---------------------------------------------------------------------------
constexpr int kLossRows = 64;
constexpr int kLossKeys = 32;

struct OnlineCE {
  float M, Z, T, A, U, V;
};

__device__ __forceinline__ OnlineCE ce_merge(OnlineCE x, OnlineCE y) {
  OnlineCE r;
  r.M = fmaxf(x.M, y.M);
  const float fx = (x.M == -INFINITY) ? 0.f : expf(x.M - r.M);
  const float fy = (y.M == -INFINITY) ? 0.f : expf(y.M - r.M);
  r.Z = x.Z * fx + y.Z * fy;
  r.T = x.T * fx + y.T * fy;
  r.A = x.A + y.A;
  r.U = x.U * fx + y.U * fy;
  r.V = x.V + y.V;
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
loss_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ phq,
                 const T* __restrict__ phk, float* __restrict__ loss_rows,
                 float* __restrict__ partial, float4* __restrict__ rows4, int d, int dpp,
                 int64_t n, int ntiles, int H, int G, int seq) {
  extern __shared__ float sm[];
  // rows padded to odd strides: the lanes of a warp read one element of 8
  // query rows and 4 key rows, which then sit in different banks
  const int ds = d + 1, ps = dpp + 1;
  float* qs = sm;                                  // [64][ds]
  float* pq = qs + kLossRows * ds;                 // [64][ps]
  float* ks = pq + (size_t)kLossRows * ps;         // [32][ds]
  float* pk = ks + kLossKeys * ds;                 // [32][ps]
  float* rowL = pk + (size_t)kLossKeys * ps;       // [64]

  const int64_t bh = blockIdx.x / ntiles;
  const int tile = (int)(blockIdx.x % ntiles);
  const int64_t r0 = (int64_t)tile * kLossRows;
  const int tid = threadIdx.x;
  const int row = tid >> 2, part = tid & 3;
  const int64_t i = r0 + row;
  const float scale = rsqrtf((float)d);
  const int ub = (int)(bh / H), uh = (int)(bh % H), kh = uh / G;   // batch, q head, kv head

  for (int e = tid; e < kLossRows * d; e += kThreads) {
    const int64_t rr = r0 + e / d;
    qs[(e / d) * ds + e % d] = rr < n ? to_f(q[(size_t)row_of(ub, uh, rr, H, n, seq) * d + e % d]) : 0.f;
  }
  for (int e = tid; e < kLossRows * dpp; e += kThreads) {
    const int64_t rr = r0 + e / dpp;
    pq[(e / dpp) * ps + e % dpp] = rr < n ? to_f(phq[((size_t)bh * n + rr) * dpp + e % dpp]) : 0.f;
  }
  OnlineCE st = {-INFINITY, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int64_t last = min(n, r0 + kLossRows) - 1;
  for (int64_t k0 = 0; k0 <= last; k0 += kLossKeys) {
    __syncthreads();
    for (int e = tid; e < kLossKeys * d; e += kThreads) {
      const int64_t j = k0 + e / d;
      ks[(e / d) * ds + e % d] = j < n ? to_f(k[(size_t)row_of(ub, kh, j, H / G, n, seq) * d + e % d]) : 0.f;
    }
    for (int e = tid; e < kLossKeys * dpp; e += kThreads) {
      const int64_t j = k0 + e / dpp;
      pk[(e / dpp) * ps + e % dpp] = j < n ? to_f(phk[((size_t)bh * n + j) * dpp + e % dpp]) : 0.f;
    }
    __syncthreads();
    if (i < n) {
      for (int jj = 0; jj < kLossKeys / 4; ++jj) {
        const int jl = part * (kLossKeys / 4) + jj;
        const int64_t j = k0 + jl;
        if (j > i) break;
        float s = 0.f, a = 0.f;
        for (int t = 0; t < d; ++t) s = fmaf(qs[row * ds + t], ks[jl * ds + t], s);
        for (int f = 0; f < dpp; ++f) a = fmaf(pq[(size_t)row * ps + f], pk[(size_t)jl * ps + f], a);
        s *= scale;
        if (s > st.M) {
          const float c = (st.M == -INFINITY) ? 0.f : expf(st.M - s);
          st.Z *= c;
          st.T *= c;
          st.U *= c;
          st.M = s;
        }
        const float e = expf(s - st.M);
        const float la = logf(a);
        st.Z += e;
        st.T = fmaf(e, la, st.T);
        st.A += a;
        st.U = fmaf(e, s, st.U);
        st.V = fmaf(a, la, st.V);
      }
    }
  }
  // merge the four partial states of a row (adjacent lanes)
  for (int off = 1; off < 4; off <<= 1) {
    OnlineCE o;
    o.M = __shfl_xor_sync(0xffffffffu, st.M, off);
    o.Z = __shfl_xor_sync(0xffffffffu, st.Z, off);
    o.T = __shfl_xor_sync(0xffffffffu, st.T, off);
    o.A = __shfl_xor_sync(0xffffffffu, st.A, off);
    o.U = __shfl_xor_sync(0xffffffffu, st.U, off);
    o.V = __shfl_xor_sync(0xffffffffu, st.V, off);
    st = ce_merge(st, o);
  }
  if (part == 0) {
    const float L = (i < n) ? (logf(st.A) - st.T / st.Z) : 0.f;
    rowL[row] = L;
    if (loss_rows && i < n) loss_rows[(size_t)bh * n + i] = L;
    if (rows4 && i < n) {
      const float Hp = logf(st.Z) + st.M - st.U / st.Z;
      const float Hw = logf(st.A) - st.V / st.A;
      rows4[(size_t)bh * n + i] = make_float4(L, L - Hp, Hp, Hw);
    }
  }
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f;
    for (int r = 0; r < kLossRows; ++r) acc += rowL[r];
    partial[(size_t)bh * ntiles + tile] = acc;
  }
}

// Per-head sum of the per-tile partial sums, in tile order.
__global__ void sum_partials_kernel(const float* __restrict__ partial, float* __restrict__ out,
                                    int64_t heads, int ntiles) {
  const int64_t bh = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (bh >= heads) return;
  float acc = 0.f;
  for (int t = 0; t < ntiles; ++t) acc += partial[(size_t)bh * ntiles + t];
  out[bh] = acc;
}

size_t prefill_smem_bytes(int d, int dpp, int C) {
  return sizeof(float) * ((size_t)dpp * d + dpp + 2 * (size_t)C * (dpp + 1) + (size_t)C * d +
                          (size_t)C * C + 2 * (size_t)C * d + C);
}

}  // namespace

int loss_simt_tile() { return kLossRows; }

template <typename T>
static cudaError_t fmap_simt_t(const Problem& p, const void* x, int is_key, void* phi,
                               float2* off, cudaStream_t s) {
  const int64_t rows = p.B * p.H * p.n;
  if (rows == 0) return cudaSuccess;
  const T* W = (const T*)(is_key && p.Wk ? p.Wk : p.Wq);
  const float* b = is_key && p.Wk ? p.bk : p.bq;
  const int warps = kThreads / 32;
  const int64_t blocks64 = (rows + warps - 1) / warps;
  const int blocks = (int)std::min<int64_t>(blocks64, (int64_t)device_sm_count() * 16);
  const size_t smem = sizeof(float) * warps * (128 + 320);
  fmap_simt_kernel<T><<<blocks, kThreads, smem, s>>>((const T*)x, W, b, (T*)phi,
                                                     p.softmax ? off : nullptr, p.kind,
                                                     p.softmax ? 1 : 0, p.d, p.dpp, p.H,
                                                     is_key ? p.G : 1, p.seq_major, p.n, rows);
  return cudaGetLastError();
}

cudaError_t launch_fmap_simt(const Problem& p, const void* x, int is_key, void* phi,
                             float2* off, cudaStream_t s) {
  return p.dtype == HH_F32 ? fmap_simt_t<float>(p, x, is_key, phi, off, s)
                           : fmap_simt_t<__nv_bfloat16>(p, x, is_key, phi, off, s);
}

template <typename T>
static cudaError_t prefill_simt_t(const Problem& p, const void* q, const void* k, const void* v,
                                  void* y, float* S_out, float* z_out, cudaStream_t s) {
  const int64_t units = p.B * p.H;
  if (units == 0) return cudaSuccess;
  const size_t cap = (size_t)std::min(device_max_smem_optin(), 200 * 1024);
  int C = 64;
  while (C > 8 && prefill_smem_bytes(p.d, p.dpp, C) > cap) C >>= 1;
  const size_t smem = prefill_smem_bytes(p.d, p.dpp, C);
  if (smem > cap) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(prefill_simt_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const T* Wk = (const T*)(p.Wk ? p.Wk : p.Wq);
  const float* bk = p.Wk ? p.bk : p.bq;
  prefill_simt_kernel<T><<<(unsigned)units, kThreads, smem, s>>>(
      (const T*)q, (const T*)k, (const T*)v, (T*)y, S_out, z_out, p.S0, p.z0, (const T*)p.Wq,
      p.bq, Wk, bk,
      p.kind, p.softmax ? 1 : 0, p.d, p.dpp, p.H, p.G, p.seq_major, p.n, C);
  return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const Problem& p, const void* q, const void* k, const void* v,
                                void* y, float* S_out, float* z_out, cudaStream_t s) {
  return p.dtype == HH_F32 ? prefill_simt_t<float>(p, q, k, v, y, S_out, z_out, s)
                           : prefill_simt_t<__nv_bfloat16>(p, q, k, v, y, S_out, z_out, s);
}

template <typename T>
static cudaError_t loss_simt_t(const Problem& p, const void* q, const void* k, const void* phq,
                               const void* phk, float* loss_rows, float* partial, int tile,
                               float* head_sum, float4* rows4, cudaStream_t s) {
  const int64_t units = p.B * p.H;
  if (units == 0) return cudaSuccess;
  const int ntiles = ceil_div(p.n, kLossRows);
  const size_t smem = sizeof(float) * ((size_t)kLossRows * (p.d + 1) +
                                       (size_t)kLossRows * (p.dpp + 1) +
                                       (size_t)kLossKeys * (p.d + 1) +
                                       (size_t)kLossKeys * (p.dpp + 1) + kLossRows);
  cudaError_t e = cudaFuncSetAttribute(loss_simt_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (ntiles > 0) {
    const int64_t blocks = units * ntiles;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    loss_simt_kernel<T><<<(unsigned)blocks, kThreads, smem, s>>>((const T*)q, (const T*)k, (const T*)phq,
                                                     (const T*)phk, loss_rows, partial, rows4,
                                                     p.d, p.dpp, p.n, ntiles, p.H, p.G,
                                                     p.seq_major);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  sum_partials_kernel<<<ceil_div(units, 128), 128, 0, s>>>(partial, head_sum, units, ntiles);
  (void)tile;
  return cudaGetLastError();
}

cudaError_t launch_loss_simt(const Problem& p, const void* q, const void* k, const void* phq,
                             const void* phk, float* loss_rows, float* partial, int tile,
                             float* head_sum, float4* rows4, cudaStream_t s) {
  return p.dtype == HH_F32
             ? loss_simt_t<float>(p, q, k, phq, phk, loss_rows, partial, tile, head_sum, rows4, s)
             : loss_simt_t<__nv_bfloat16>(p, q, k, phq, phk, loss_rows, partial, tile, head_sum,
                                          rows4, s);
}

}  // namespace hh
