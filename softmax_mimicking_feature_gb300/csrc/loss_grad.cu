// Gradient of the summed mimicry loss w.r.t. the Hedgehog feature map.
//
// "The Attention Weight Distillation Loss" (Hedgehog & Porcupine summary):
// only the feature maps are trained; q, k and the softmax target are frozen.
// With a_ij = phi(q_i).phi(k_j), A_i = sum_{j<=i} a_ij, p the causal
// softmax(q k^T / sqrt d) and L_i = ln A_i - sum_j p_ij ln a_ij:
//   g_ij = dL/da_ij = 1/A_i - p_ij / a_ij                     (j <= i)
//   dL/dphi(q_i) = sum_j g_ij phi(k_j),   dL/dphi(k_j) = sum_i g_ij phi(q_i)
//   dL/dh = dL/dphi_+ * e^h - dL/dphi_- * e^-h   (phi = [e^h; e^-h], "The Hedgehog
//   MLP Feature Map", Choices 1 and 3)
//   dL/dW = sum_x x^T dL/dh(x),  dL/db = sum_x dL/dh(x)
// For the softmax map (Choice 4, Eq. 5, no bias) the step to dL/dh is the
// softmax Jacobian of each half instead, and there is no db (write_dh).
// Three CUDA-core kernels, fp32 arithmetic on phi(q), phi(k) precomputed by
// the feature-map kernel:
//   grad_query_kernel: per 32-query tile, a first sweep over the keys gives the
//     row statistics (softmax max and sum, A_i; kept for the key side), a
//     second forms g and dL/dh(q)
//   grad_key_kernel:   per 32-key tile, sweeps the later query tiles for dL/dh(k)
//   grad_reduce_kernel: dW, db per head (summed over the batch); also used
//     after the tensor-core kernels for bf16

#include <math.h>

#include <algorithm>

#include "hh_internal.cuh"

namespace hh {
namespace {

constexpr int kT = 32;         // query / key tile
constexpr int kThreads = 256;  // thread t: tile row t / 8, lane-group slot t % 8

struct GradSmem {
  float* xs;    // [kT][d]    resident rows (q for the query side, k for the key side)
  float* pxs;   // [kT][dpp]  their features
  float* ys;    // [kT][d]    streamed rows
  float* pys;   // [kT][dpp]
  float* G;     // [kT][kT+1] g of the tile pair
  float* st;    // [kT][3]    M, Z, A of query rows (streamed tiles on the key side)
};

__host__ __device__ inline size_t grad_smem_bytes(int d, int dpp) {
  return sizeof(float) * ((size_t)2 * kT * d + (size_t)2 * kT * dpp + kT * (kT + 1) + kT * 3);
}

__device__ inline GradSmem carve(float* sm, int d, int dpp) {
  GradSmem g;
  g.xs = sm;
  g.pxs = g.xs + kT * d;
  g.ys = g.pxs + kT * dpp;
  g.pys = g.ys + kT * d;
  g.G = g.pys + kT * dpp;
  g.st = g.G + kT * (kT + 1);
  return g;
}

// Rows [row0, row0 + kT) of head h of batch b of a tensor with Hx heads in the
// [B][Hx][n][width] layout, or [B][n][Hx][width] (seq); zero past n.
template <typename T>
__device__ inline void load_tile(float* dst, const T* src, int b, int h, int Hx, int seq,
                                 int64_t row0, int64_t n, int width) {
  for (int i = threadIdx.x; i < kT * width; i += kThreads) {
    const int r = i / width;
    dst[i] = row0 + r < n ? to_f(src[row_of(b, h, row0 + r, Hx, n, seq) * width + i % width])
                          : 0.f;
  }
}

// s (scaled q.k) and a (phi(q).phi(k)) of query row rq (in qs/pqs) and key row rk (in ks/pks)
__device__ inline void pair(const float* qs, const float* pqs, const float* ks, const float* pks,
                            int rq, int rk, int d, int dpp, float scale, float& s, float& a) {
  float s0 = 0.f, s1 = 0.f, a0 = 0.f, a1 = 0.f;
  const float* q = qs + rq * d;
  const float* k = ks + rk * d;
  for (int c = 0; c < d; c += 2) {
    s0 = fmaf(q[c], k[c], s0);
    s1 = fmaf(q[c + 1], k[c + 1], s1);
  }
  const float* pq = pqs + rq * dpp;
  const float* pk = pks + rk * dpp;
  for (int f = 0; f < dpp; f += 2) {
    a0 = fmaf(pq[f], pk[f], a0);
    a1 = fmaf(pq[f + 1], pk[f + 1], a1);
  }
  s = (s0 + s1) * scale;
  a = a0 + a1;
}

// dL/dh of the tile's rows: each thread parks its dL/dphi slots (features
// slot + 8 i) in scratch [kT][dpp] (the streamed-feature buffer, free once
// the sweep is done), then combines dL/dphi_+ e^h - dL/dphi_- e^-h.
// Softmax map (Choice 4, Eq. 5; px holds phi_+ = softmax(h), phi_- =
// softmax(-h)): each half goes through the softmax Jacobian,
//   dL/dh = phi_+ (dL/dphi_+ - <dL/dphi_+, phi_+>) - phi_- (dL/dphi_- - <dL/dphi_-, phi_->),
// with the 2 kT row dots in `dots` (the g tile, also free by then).
__device__ inline void write_dh(const float (&acc)[32], float* scratch, const float* px,
                                float* dots, int r, int slot, int d, int dpp, int64_t rows_left,
                                bool softmax, float* dh) {
  const int nf = dpp / 8;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < nf) scratch[r * dpp + slot + 8 * i] = acc[i];
  __syncthreads();
  if (softmax) {
    if (threadIdx.x < 2 * kT) {
      const int rr = threadIdx.x >> 1, f0 = (threadIdx.x & 1) * d;
      float s = 0.f;
      for (int f = f0; f < f0 + d; ++f) s = fmaf(scratch[rr * dpp + f], px[rr * dpp + f], s);
      dots[threadIdx.x] = s;
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < kT * d; e += kThreads) {
    const int rr = e / d, f = e % d;
    if (rr >= rows_left) continue;
    const float cp = softmax ? dots[2 * rr] : 0.f, cn = softmax ? dots[2 * rr + 1] : 0.f;
    dh[(int64_t)rr * d + f] = (scratch[rr * dpp + f] - cp) * px[rr * dpp + f] -
                              (scratch[rr * dpp + f + d] - cn) * px[rr * dpp + f + d];
  }
}

// grid: (U * ceil(n / kT)); block: query tile qt of unit u
template <typename T>
__global__ void __launch_bounds__(kThreads) grad_query_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ phq,
    const T* __restrict__ phk, float* __restrict__ stats, float* __restrict__ dhq, int d, int dpp,
    int64_t n, int ntiles, int H, int G, int seq, int softmax) {
  extern __shared__ float sm[];
  const GradSmem S = carve(sm, d, dpp);
  const int64_t u = blockIdx.x / ntiles;
  const int ub = (int)(u / H), uh = (int)(u % H), kh = uh / G;   // batch, q head, kv head
  const int qt = blockIdx.x % ntiles;
  const int64_t q0 = (int64_t)qt * kT;
  const int t = threadIdx.x, r = t / 8, slot = t % 8;
  const int64_t qi = q0 + r;
  const float scale = rsqrtf((float)d);
  load_tile(S.xs, q, ub, uh, H, seq, q0, n, d);
  load_tile(S.pxs, phq, (int)u, 0, 1, 0, q0, n, dpp);

  // sweep 1: M_i = max s, Z_i = sum e^{s - M}, A_i = sum a over j <= i
  float m = -INFINITY, z = 0.f, asum = 0.f;
  for (int kt = 0; kt <= qt; ++kt) {
    __syncthreads();
    load_tile(S.ys, k, ub, kh, H / G, seq, (int64_t)kt * kT, n, d);
    load_tile(S.pys, phk, (int)u, 0, 1, 0, (int64_t)kt * kT, n, dpp);
    __syncthreads();
    for (int c = slot; c < kT; c += 8) {
      const int64_t kj = (int64_t)kt * kT + c;
      if (kj > qi || qi >= n) continue;
      float s, a;
      pair(S.xs, S.pxs, S.ys, S.pys, r, c, d, dpp, scale, s, a);
      if (s > m) {
        z = z * expf(m - s) + 1.f;
        m = s;
      } else {
        z += expf(s - m);
      }
      asum += a;
    }
  }
  // merge the 8 threads of a row (lanes 8r'..8r'+7 of the warp)
  for (int o = 1; o < 8; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    const float a2 = __shfl_xor_sync(0xffffffffu, asum, o);
    const float mn = fmaxf(m, m2);
    z = (m == -INFINITY ? 0.f : z * expf(m - mn)) + (m2 == -INFINITY ? 0.f : z2 * expf(m2 - mn));
    m = mn;
    asum += a2;
  }
  if (slot == 0 && qi < n) {
    float* st = stats + (u * n + qi) * 3;
    st[0] = m;
    st[1] = z;
    st[2] = asum;
  }

  // sweep 2: g and dL/dphi(q) = sum_j g_ij phi(k_j)
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  const float invA = qi < n ? 1.f / asum : 0.f, invZ = qi < n ? 1.f / z : 0.f;
  const int nf = dpp / 8;
  for (int kt = 0; kt <= qt; ++kt) {
    __syncthreads();
    load_tile(S.ys, k, ub, kh, H / G, seq, (int64_t)kt * kT, n, d);
    load_tile(S.pys, phk, (int)u, 0, 1, 0, (int64_t)kt * kT, n, dpp);
    __syncthreads();
    for (int c = slot; c < kT; c += 8) {
      const int64_t kj = (int64_t)kt * kT + c;
      float g = 0.f;
      if (kj <= qi && qi < n) {
        float s, a;
        pair(S.xs, S.pxs, S.ys, S.pys, r, c, d, dpp, scale, s, a);
        g = invA - expf(s - m) * invZ / a;
      }
      S.G[r * (kT + 1) + c] = g;
    }
    __syncthreads();
    for (int c = 0; c < kT; ++c) {
      const float gv = S.G[r * (kT + 1) + c];
      const float* pk = S.pys + c * dpp;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nf) acc[i] = fmaf(gv, pk[slot + 8 * i], acc[i]);
    }
  }
  write_dh(acc, S.pys, S.pxs, S.G, r, slot, d, dpp, n - q0, softmax != 0, dhq + (u * n + q0) * d);
}

// grid: (U * ceil(n / kT)); block: key tile kt of unit u
template <typename T>
__global__ void __launch_bounds__(kThreads) grad_key_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ phq,
    const T* __restrict__ phk, const float* __restrict__ stats, float* __restrict__ dhk, int d,
    int dpp, int64_t n, int ntiles, int H, int G, int seq, int softmax) {
  extern __shared__ float sm[];
  const GradSmem S = carve(sm, d, dpp);
  const int64_t u = blockIdx.x / ntiles;
  const int ub = (int)(u / H), uh = (int)(u % H), kh = uh / G;   // batch, q head, kv head
  const int kt = blockIdx.x % ntiles;
  const int64_t k0 = (int64_t)kt * kT;
  const int t = threadIdx.x, r = t / 8, slot = t % 8;   // r: key row of the tile
  const float scale = rsqrtf((float)d);
  load_tile(S.xs, k, ub, kh, H / G, seq, k0, n, d);
  load_tile(S.pxs, phk, (int)u, 0, 1, 0, k0, n, dpp);
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  const int nf = dpp / 8;
  for (int qt = kt; qt < ntiles; ++qt) {
    __syncthreads();
    load_tile(S.ys, q, ub, uh, H, seq, (int64_t)qt * kT, n, d);
    load_tile(S.pys, phq, (int)u, 0, 1, 0, (int64_t)qt * kT, n, dpp);
    for (int i = threadIdx.x; i < kT * 3; i += kThreads) {
      const int64_t row = (int64_t)qt * kT + i / 3;
      S.st[i] = row < n ? stats[(u * n + row) * 3 + i % 3] : 1.f;
    }
    __syncthreads();
    // G[query c][key r] for the pair (query tile qt, this key tile)
    for (int c = slot; c < kT; c += 8) {
      const int64_t qi = (int64_t)qt * kT + c, kj = k0 + r;
      float g = 0.f;
      if (kj <= qi && qi < n) {
        float s, a;
        pair(S.ys, S.pys, S.xs, S.pxs, c, r, d, dpp, scale, s, a);
        const float* st = S.st + c * 3;
        g = 1.f / st[2] - expf(s - st[0]) / st[1] / a;
      }
      S.G[c * (kT + 1) + r] = g;
    }
    __syncthreads();
    for (int c = 0; c < kT; ++c) {
      const float gv = S.G[c * (kT + 1) + r];
      const float* pq = S.pys + c * dpp;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nf) acc[i] = fmaf(gv, pq[slot + 8 * i], acc[i]);
    }
  }
  write_dh(acc, S.pys, S.pxs, S.G, r, slot, d, dpp, n - k0, softmax != 0, dhk + (u * n + k0) * d);
}

// dW[h][a][l] = sum_{b, t} x[b,h,t,a] dh[b,h,t,l] (+ the key side when shared);
// a side whose x is raw k reads key/value head h / G (kvx1, kvx2),
// db[h][l] = sum dh (skipped when db is null: the softmax map has no bias).  grid: (H * ceil(d / 32) * ceil(d / 32)), 256 threads:
// thread -> (a, l) pairs of one 32 x 32 block; tokens in smem chunks of 32.
template <typename T>
__global__ void __launch_bounds__(kThreads) grad_reduce_kernel(
    const T* __restrict__ x1, const float* __restrict__ dh1, const T* __restrict__ x2,
    const float* __restrict__ dh2, float* __restrict__ dW, float* __restrict__ db, int64_t B,
    int H, int64_t n, int d, int G1, int G2, int seq) {
  __shared__ float xs[32][33];
  __shared__ float hs[32][33];
  const int nb = (d + 31) / 32;
  const int h = blockIdx.x / (nb * nb);
  const int a0 = (blockIdx.x / nb) % nb * 32, l0 = blockIdx.x % nb * 32;
  const int t = threadIdx.x, ta = t / 8, tl = (t % 8) * 4;   // 4 (a, l) pairs per thread
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, dbacc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int side = 0; side < (x2 ? 2 : 1); ++side) {
    const T* x = side ? x2 : x1;
    const float* dh = side ? dh2 : dh1;
    for (int64_t b = 0; b < B; ++b) {
      const size_t base = ((size_t)b * H + h) * n;
      const int Gs = side ? G2 : G1;
      const int hx = h / Gs;   // head of x (the key/value head when x is k under grouping)
      for (int64_t t0 = 0; t0 < n; t0 += 32) {
        __syncthreads();
        for (int i = t; i < 32 * 32; i += kThreads) {
          const int rr = i / 32, cc = i % 32;
          const bool ok = t0 + rr < n;
          xs[rr][cc] = ok && a0 + cc < d
                           ? to_f(x[row_of((int)b, hx, t0 + rr, H / Gs, n, seq) * d + a0 + cc])
                           : 0.f;
          hs[rr][cc] = ok && l0 + cc < d ? dh[(base + t0 + rr) * d + l0 + cc] : 0.f;
        }
        __syncthreads();
        for (int rr = 0; rr < 32; ++rr) {
          const float xv = xs[rr][ta];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[j] = fmaf(xv, hs[rr][tl + j], acc[j]);
            if (a0 == 0 && ta == 0) dbacc[j] += hs[rr][tl + j];
          }
        }
      }
    }
  }
  if (a0 + ta < d)
    for (int j = 0; j < 4; ++j)
      if (l0 + tl + j < d) dW[((size_t)h * d + a0 + ta) * d + l0 + tl + j] = acc[j];
  if (db && a0 == 0 && ta == 0)
    for (int j = 0; j < 4; ++j)
      if (l0 + tl + j < d) db[(size_t)h * d + l0 + tl + j] = dbacc[j];
}

template <typename T>
cudaError_t grad_t(const Problem& p, const void* q, const void* k, const void* phq,
                   const void* phk, float* stats, float* dhq, float* dhk, float* dWq, float* dbq,
                   float* dWk, float* dbk, cudaStream_t s) {
  const int64_t U = p.B * p.H;
  const int ntiles = ceil_div(p.n, kT);
  const size_t smem = grad_smem_bytes(p.d, p.dpp);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(grad_query_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(grad_key_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  grad_query_kernel<T><<<(unsigned)(U * ntiles), kThreads, smem, s>>>(
      (const T*)q, (const T*)k, (const T*)phq, (const T*)phk, stats, dhq, p.d, p.dpp, p.n, ntiles,
      p.H, p.G, p.seq_major, p.softmax ? 1 : 0);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  grad_key_kernel<T><<<(unsigned)(U * ntiles), kThreads, smem, s>>>(
      (const T*)q, (const T*)k, (const T*)phq, (const T*)phk, stats, dhk, p.d, p.dpp, p.n, ntiles,
      p.H, p.G, p.seq_major, p.softmax ? 1 : 0);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_grad_reduce(p, q, k, dhq, dhk, dWq, dbq, dWk, dbk, s);
}

template <typename T>
cudaError_t reduce_t(const Problem& p, const void* q, const void* k, const float* dhq,
                     const float* dhk, float* dWq, float* dbq, float* dWk, float* dbk,
                     cudaStream_t s) {
  const int nb = (p.d + 31) / 32;
  const unsigned grid = (unsigned)(p.H * nb * nb);
  if (dWk) {   // separate key map: each side to its own parameters
    grad_reduce_kernel<T><<<grid, kThreads, 0, s>>>((const T*)q, dhq, (const T*)nullptr, nullptr,
                                                    dWq, dbq, p.B, p.H, p.n, p.d, 1, 1, p.seq_major);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    grad_reduce_kernel<T><<<grid, kThreads, 0, s>>>((const T*)k, dhk, (const T*)nullptr, nullptr,
                                                    dWk, dbk, p.B, p.H, p.n, p.d, p.G, 1, p.seq_major);
  } else {
    grad_reduce_kernel<T><<<grid, kThreads, 0, s>>>((const T*)q, dhq, (const T*)k, dhk, dWq, dbq,
                                                    p.B, p.H, p.n, p.d, 1, p.G, p.seq_major);
  }
  return cudaGetLastError();
}

}  // namespace

size_t loss_grad_smem_bytes(const Problem& p) { return grad_smem_bytes(p.d, p.dpp); }

cudaError_t launch_grad_reduce(const Problem& p, const void* q, const void* k, const float* dhq,
                               const float* dhk, float* dWq, float* dbq, float* dWk, float* dbk,
                               cudaStream_t s) {
  if (p.dtype == HH_F32) return reduce_t<float>(p, q, k, dhq, dhk, dWq, dbq, dWk, dbk, s);
  return reduce_t<__nv_bfloat16>(p, q, k, dhq, dhk, dWq, dbq, dWk, dbk, s);
}

cudaError_t launch_loss_grad(const Problem& p, const void* q, const void* k, const void* phq,
                             const void* phk, float* stats, float* dhq, float* dhk, float* dWq,
                             float* dbq, float* dWk, float* dbk, cudaStream_t s) {
  if (p.dtype == HH_F32)
    return grad_t<float>(p, q, k, phq, phk, stats, dhq, dhk, dWq, dbq, dWk, dbk, s);
  return grad_t<__nv_bfloat16>(p, q, k, phq, phk, stats, dhq, dhk, dWq, dbq, dWk, dbk, s);
}

}  // namespace hh
