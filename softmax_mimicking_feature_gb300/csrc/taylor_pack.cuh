// Packed degree-2 Taylor features used inside the tensor-core kernels.
//
// "The Taylor Exponential as a Bridge Result" (Hedgehog & Porcupine summary)
// defines phi(x) = [1, x, vec(x x^T) / sqrt2] with all d^2 ordered pairs, so
// that phi(q) . phi(k) = 1 + q.k + (q.k)^2 / 2.  The ordered pairs (i, j) and
// (j, i) carry the same value, so the same dot product comes from the 136
// unordered pairs with weights
//   x_i x_i / sqrt2   (diagonal)      x_i x_j   (i < j)
// since sum_{i,j} q_i q_j k_i k_j / 2 = sum_i q_i^2 k_i^2 / 2 + sum_{i<j} q_i q_j k_i k_j.
// Packed order (160 stored features, multiple of 32):
//   [0, 136)   pairs (i, j), i <= j, i-major
//   136        1
//   [137, 153) x_0 .. x_15
//   [153, 160) 0
// A state built from packed features maps back to the public layout
// [1, x, x_i x_j / sqrt2 (i-major, 288 rows with the zero pad)] row by row:
//   public 17 + 16 i + j and 17 + 16 j + i  <-  packed (i, j) * (i == j ? 1 : 1/sqrt2)
//   public 0 <- packed 136,   public 1 + i <- packed 137 + i.

#pragma once

#include "tc_ptx.cuh"

namespace hh {
namespace tp {

constexpr int F = 160;      // stored packed features
constexpr int NPAIR = 136;  // unordered pairs of 16 coordinates
constexpr int DPUB = 288;   // public stored features (273 used)

// first packed index of row i of the pair triangle
__host__ __device__ constexpr int row_off(int i) { return 16 * i - i * (i - 1) / 2; }
__host__ __device__ constexpr int pair_i(int f) {
  int i = 0;
  while (i < 15 && row_off(i + 1) <= f) ++i;
  return i;
}
__host__ __device__ constexpr int pair_j(int f) { return pair_i(f) + (f - row_off(pair_i(f))); }

// packed feature FI of x (FI a compile-time constant)
template <int FI>
__device__ __forceinline__ float feat(const float (&x)[16]) {
  if constexpr (FI < NPAIR) {
    constexpr int i = pair_i(FI), j = pair_j(FI);
    if constexpr (i == j) return x[i] * x[i] * kInvSqrt2;
    else return x[i] * x[j];
  } else if constexpr (FI == NPAIR) {
    return 1.f;
  } else if constexpr (FI < NPAIR + 17) {
    return x[FI - NPAIR - 1];
  } else {
    return 0.f;
  }
}

// 8 packed features from F0 as 4 bf16 pairs (zero when !valid)
template <int F0>
__device__ __forceinline__ void chunk8(const float (&x)[16], bool valid, uint32_t (&w)[4]) {
  w[0] = valid ? tc::pack_bf16(feat<F0>(x), feat<F0 + 1>(x)) : 0u;
  w[1] = valid ? tc::pack_bf16(feat<F0 + 2>(x), feat<F0 + 3>(x)) : 0u;
  w[2] = valid ? tc::pack_bf16(feat<F0 + 4>(x), feat<F0 + 5>(x)) : 0u;
  w[3] = valid ? tc::pack_bf16(feat<F0 + 6>(x), feat<F0 + 7>(x)) : 0u;
}

// Public rows of packed feature f (runtime): up to two rows and the factor.
__device__ __forceinline__ int public_rows(int f, int& r0, int& r1, float& scale) {
  if (f < NPAIR) {
    int i = 0;
    while (i < 15 && row_off(i + 1) <= f) ++i;
    const int j = i + (f - row_off(i));
    r0 = 17 + 16 * i + j;
    r1 = 17 + 16 * j + i;
    scale = (i == j) ? 1.f : kInvSqrt2;
    return i == j ? 1 : 2;
  }
  scale = 1.f;
  if (f == NPAIR) { r0 = 0; return 1; }
  if (f < NPAIR + 17) { r0 = f - NPAIR; return 1; }
  return 0;
}

}  // namespace tp
}  // namespace hh
