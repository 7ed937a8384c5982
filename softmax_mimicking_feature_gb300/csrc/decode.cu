// Recurrent decode step: one block per (sequence, head).
//
// "The Hedgehog & the Porcupine" summary, "Complexity Analysis": the state
// S = sum_j phi(k_j)^T v_j ([d'][d]) and z = sum_j phi(k_j) ([d']) absorb the
// new token, then y_t = phi(q_t) S_t / (phi(q_t) . z_t).
//
// The step is bound by HBM: every (sequence, head) reads and writes its fp32
// state once (2 * 4 * (d'd + d') bytes), while phi(q_t), phi(k_t) cost two
// d x d GEMVs against an L2-resident W.  S rows are streamed with 16-byte
// loads/stores marked evict-first (the state is touched once per step), with
// eight loads in flight per thread before the first use.

#include <math.h>

#include "hh_internal.cuh"

namespace hh {
namespace {

constexpr int kDecThreads = 256;
constexpr int kUnroll = 8;

template <typename T>
__device__ __forceinline__ void load_vec(const T* src, float* dst, int d, int tid) {
  for (int i = tid; i < d; i += kDecThreads) dst[i] = to_f(src[i]);
}

template <int VW> struct Vec;
template <> struct Vec<4> { using type = float4; };
template <> struct Vec<1> { using type = float; };

template <typename T, int VW>
__global__ void __launch_bounds__(kDecThreads)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              float* __restrict__ S, float* __restrict__ z, T* __restrict__ y,
              const T* __restrict__ Wq, const float* __restrict__ bq,
              const T* __restrict__ Wk, const float* __restrict__ bk, int kind, int softmax,
              int d, int dpp, int H, int G) {
  __shared__ float qs[128], ks[128], vs[128];
  __shared__ float phq[320], phk[320];
  __shared__ __align__(16) float ypart[kDecThreads * 4];
  __shared__ float dpart[kDecThreads / 32];
  __shared__ float lse[2][2];   // softmax map: (c+, c-) of the query and of the key

  const int64_t u = blockIdx.x;  // (sequence, head) unit
  const int h = (int)(u % H);
  const int tid = threadIdx.x;
  load_vec(q + (size_t)u * d, qs, d, tid);
  const int64_t ukv = kv_unit(u, H, G);   // k, v of this query head
  load_vec(k + (size_t)ukv * d, ks, d, tid);
  load_vec(v + (size_t)ukv * d, vs, d, tid);
  __syncthreads();

  // phi(q_t), phi(k_t)
  if (kind == HH_FMAP_HEDGEHOG) {
    const T* Wqh = Wq + (size_t)h * d * d;
    const T* Wkh = Wk + (size_t)h * d * d;
    // threads [0, d) do queries, [128, 128 + d) do keys
    const int l = tid & 127;
    const bool key = tid >= 128;
    if (l < d) {
      const T* Wh = key ? Wkh : Wqh;
      const float* xs = key ? ks : qs;
      const float* bb = key ? bk : bq;
      float hv = bb ? bb[(size_t)h * d + l] : 0.f;
      for (int kk = 0; kk < d; ++kk) hv = fmaf(xs[kk], to_f(Wh[(size_t)kk * d + l]), hv);
      float* out = key ? phk : phq;
      if (softmax) {
        out[l] = hv;
      } else {
        out[l] = expf(hv);
        out[d + l] = expf(-hv);
      }
    }
    if (softmax) {
      // "The Hedgehog MLP Feature Map", Choice 4 (Eq. 5): each half divided by
      // its sum over the d directions; warp 0 reduces the query, warp 4 the key
      __syncthreads();
      const int warp = tid >> 5, lane = tid & 31;
      if (warp == 0 || warp == 4) {
        const float* hs = warp ? phk : phq;
        float mx = -INFINITY, mn = INFINITY;
        for (int i = lane; i < d; i += 32) {
          mx = fmaxf(mx, hs[i]);
          mn = fminf(mn, hs[i]);
        }
        for (int o = 16; o > 0; o >>= 1) {
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        float sp = 0.f, sn = 0.f;
        for (int i = lane; i < d; i += 32) {
          sp += expf(hs[i] - mx);
          sn += expf(mn - hs[i]);
        }
        for (int o = 16; o > 0; o >>= 1) {
          sp += __shfl_xor_sync(0xffffffffu, sp, o);
          sn += __shfl_xor_sync(0xffffffffu, sn, o);
        }
        if (lane == 0) {
          lse[warp ? 1 : 0][0] = mx + logf(sp);
          lse[warp ? 1 : 0][1] = logf(sn) - mn;
        }
      }
      __syncthreads();
      if (l < d) {
        float* out = key ? phk : phq;
        const float hv = out[l];
        out[l] = expf(hv - lse[key][0]);
        out[d + l] = expf(-hv - lse[key][1]);
      }
    }
  } else {
    for (int f = tid; f < dpp; f += kDecThreads) {
      float a, b;
      if (f == 0) {
        a = b = 1.f;
      } else if (f <= d) {
        a = qs[f - 1];
        b = ks[f - 1];
      } else if (f <= d + d * d) {
        const int p = f - 1 - d;
        a = qs[p / d] * qs[p % d] * kInvSqrt2;
        b = ks[p / d] * ks[p % d] * kInvSqrt2;
      } else {
        a = b = 0.f;
      }
      phq[f] = a;
      phk[f] = b;
    }
  }
  __syncthreads();

  // z update and denominator phi(q) . z_new (fixed-order block reduction)
  float dacc = 0.f;
  float* zu = z + (size_t)u * dpp;
  for (int f = tid; f < dpp; f += kDecThreads) {
    const float zn = zu[f] + phk[f];
    zu[f] = zn;
    dacc = fmaf(phq[f], zn, dacc);
  }
  for (int off = 16; off > 0; off >>= 1) dacc += __shfl_xor_sync(0xffffffffu, dacc, off);
  if ((tid & 31) == 0) dpart[tid >> 5] = dacc;

  // S streaming: thread owns vector column cv of rows f = rg, rg + R, ...
  const int colsv = d / VW;
  const int R = kDecThreads / colsv;  // row groups
  const int rg = tid / colsv, cv = tid % colsv;
  using V = typename Vec<VW>::type;
  float acc[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e) acc[e] = 0.f;
  if (rg < R) {
    float vv[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) vv[e] = vs[VW * cv + e];
    V* Su = reinterpret_cast<V*>(S + (size_t)u * dpp * d);
    for (int f0 = rg; f0 < dpp; f0 += R * kUnroll) {
      V s[kUnroll];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int f = f0 + t * R;
        if (f < dpp) s[t] = __ldcs(Su + (size_t)f * colsv + cv);
      }
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const int f = f0 + t * R;
        if (f < dpp) {
          const float pk = phk[f], pq = phq[f];
          float* sf = reinterpret_cast<float*>(&s[t]);
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            sf[e] = fmaf(pk, vv[e], sf[e]);
            acc[e] = fmaf(pq, sf[e], acc[e]);
          }
          __stcs(Su + (size_t)f * colsv + cv, s[t]);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < VW; ++e) ypart[tid * VW + e] = acc[e];
  __syncthreads();
  if (tid < d) {
    const int c = tid;
    float num = 0.f;
    for (int g = 0; g < R; ++g) num += ypart[(g * colsv + c / VW) * VW + c % VW];
    float den = 0.f;
    for (int w = 0; w < kDecThreads / 32; ++w) den += dpart[w];
    y[(size_t)u * d + c] = from_f<T>(num / den);
  }
}

}  // namespace

template <typename T>
static cudaError_t decode_t(const Problem& p, const void* q, const void* k, const void* v,
                            float* S, float* z, void* y, cudaStream_t s) {
  const int64_t units = p.B * p.H;
  if (units == 0) return cudaSuccess;
  const T* Wk = (const T*)(p.Wk ? p.Wk : p.Wq);
  const float* bk = p.Wk ? p.bk : p.bq;
  if (p.d % 4 == 0)
    decode_kernel<T, 4><<<(unsigned)units, kDecThreads, 0, s>>>(
        (const T*)q, (const T*)k, (const T*)v, S, z, (T*)y, (const T*)p.Wq, p.bq, Wk, bk,
        p.kind, p.softmax ? 1 : 0, p.d, p.dpp, p.H, p.G);
  else
    decode_kernel<T, 1><<<(unsigned)units, kDecThreads, 0, s>>>(
        (const T*)q, (const T*)k, (const T*)v, S, z, (T*)y, (const T*)p.Wq, p.bq, Wk, bk,
        p.kind, p.softmax ? 1 : 0, p.d, p.dpp, p.H, p.G);
  return cudaGetLastError();
}

cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v,
                          float* S, float* z, void* y, cudaStream_t s) {
  return p.dtype == HH_F32 ? decode_t<float>(p, q, k, v, S, z, y, s)
                           : decode_t<__nv_bfloat16>(p, q, k, v, S, z, y, s);
}

}  // namespace hh
