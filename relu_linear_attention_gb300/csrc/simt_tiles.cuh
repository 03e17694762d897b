// Small fp32 GEMM micro-tiles in shared memory for the CUDA-core kernels (sm_103a).
//
// Each thread accumulates a 4 x 4 tile acc[y][x]. The tile's rows m are rows (or columns) m0 .. m0+3
// of the A operand, always contiguous; its columns are n0 + NS * x (x = 0..3): NS = 1 gives four
// contiguous columns (float4 loads of B), a larger NS spreads them so that neighbouring lanes,
// which take neighbouring n0, touch neighbouring rows or columns of B (with a row stride of 4 times
// an odd number of floats, eight consecutive rows start in eight different 4-bank groups). K is a
// multiple of 4 for the forms that step k by 4. Pointers are already offset to row m0 / column n0.
#pragma once

#include <cuda_runtime.h>

namespace rapt {
namespace simt {

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// acc[y][x] += sum_k A[y*lda + k] * B[(NS*x)*ldb + k]       (B contiguous along k)
template <int NS>
__device__ __forceinline__ void mt_dot(float (&acc)[4][4], const float* A, int lda, const float* B,
                                       int ldb, int K) {
  for (int k = 0; k < K; k += 4) {
    float4 a[4], b[4];
#pragma unroll
    for (int y = 0; y < 4; ++y) a[y] = ld4(A + y * lda + k);
#pragma unroll
    for (int x = 0; x < 4; ++x) b[x] = ld4(B + NS * x * ldb + k);
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        acc[y][x] = fmaf(a[y].x, b[x].x, acc[y][x]);
        acc[y][x] = fmaf(a[y].y, b[x].y, acc[y][x]);
        acc[y][x] = fmaf(a[y].z, b[x].z, acc[y][x]);
        acc[y][x] = fmaf(a[y].w, b[x].w, acc[y][x]);
      }
  }
}
// B element (k, x) of the column forms below.
template <int NS>
__device__ __forceinline__ void ld_brow(const float* B, float (&b)[4]) {
  if constexpr (NS == 1) {
    const float4 t = ld4(B);
    b[0] = t.x; b[1] = t.y; b[2] = t.z; b[3] = t.w;
  } else {
#pragma unroll
    for (int x = 0; x < 4; ++x) b[x] = B[NS * x];
  }
}
// acc[y][x] += sum_k A[y*lda + k] * B[k*ldb + NS*x]         (A along k, B along n)
template <int NS>
__device__ __forceinline__ void mt_outer(float (&acc)[4][4], const float* A, int lda,
                                         const float* B, int ldb, int K) {
  for (int k = 0; k < K; k += 4) {
    float4 a[4];
    float b[4][4];
#pragma unroll
    for (int y = 0; y < 4; ++y) a[y] = ld4(A + y * lda + k);
#pragma unroll
    for (int u = 0; u < 4; ++u) ld_brow<NS>(B + (k + u) * ldb, b[u]);
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const float av[4] = {a[y].x, a[y].y, a[y].z, a[y].w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(av[u], b[u][x], acc[y][x]);
    }
  }
}
// acc[y][x] += sum_k A[k*lda + y] * B[k*ldb + NS*x]         (A along m, B along n)
template <int NS>
__device__ __forceinline__ void mt_tn(float (&acc)[4][4], const float* A, int lda, const float* B,
                                      int ldb, int K) {
  for (int k = 0; k < K; ++k) {
    const float4 a = ld4(A + k * lda);
    float b[4];
    ld_brow<NS>(B + k * ldb, b);
    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(av[y], b[x], acc[y][x]);
  }
}

}  // namespace simt
}  // namespace rapt
