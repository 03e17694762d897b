// Backward of the RLA-2 feature map f = ReLU(RoPE(RMSNorm(x))) for one token row, shared by the
// CUDA-core and tensor-core backward kernels (sm_103a). The lane mapping is feature_row's
// (common.cuh): TPR lanes per row, lane r owns elements [r*EPT, (r+1)*EPT).
#pragma once

#include "common.cuh"

namespace rapt {

template <typename T>
__device__ __forceinline__ void store2(T* p, float a, float b);
template <>
__device__ __forceinline__ void store2<float>(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// Backward of f = ReLU(RoPE(RMSNorm(x))) for one token row, the lane mapping of feature_row
// (TPR lanes per row, lane r owns elements [r*EPT, (r+1)*EPT)), on the row's input values already
// loaded into f (zeros for an invalid row). df: the row's gradient of f in shared memory. Writes
// dx (valid rows only) and adds this row's gain gradient dy_hat * x * rinv into dg. Every lane of
// the warp must call it together (shuffles over the full warp).
template <int D, typename T>
__device__ __forceinline__ void feature_vals_bwd(const float (&f)[FeatureLayout<D>::EPT],
                                                 bool valid, const float* gamma, int pos,
                                                 const FeatureArgs& fa, int r, const float* df,
                                                 T* dx, float (&dg)[FeatureLayout<D>::EPT]) {
  using FL = FeatureLayout<D>;
  constexpr int EPT = FL::EPT;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < EPT; ++i) ss = fmaf(f[i], f[i], ss);
#pragma unroll
  for (int off = FL::TPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rinv = rsqrtf(ss * (1.0f / D) + fa.eps_norm);
  float u[EPT];  // gamma * dy_hat
  float dot = 0.f;
#pragma unroll
  for (int m = 0; m < EPT / 2; ++m) {
    const int e = r * EPT + 2 * m;
    const float g0 = gamma[e], g1 = gamma[e + 1];
    const float y0 = f[2 * m] * rinv * g0;
    const float y1 = f[2 * m + 1] * rinv * g1;
    float s, c;
    rope_sincos(pos, fa.rope_hi[e >> 1], fa.rope_lo[e >> 1], s, c);
    const float a = fmaf(y0, c, -y1 * s);  // the forward's pre-activation, same arithmetic
    const float b = fmaf(y0, s, y1 * c);
    const float da = (valid && a > 0.f) ? df[e] : 0.f;
    const float db = (valid && b > 0.f) ? df[e + 1] : 0.f;
    const float h0 = fmaf(da, c, db * s);   // inverse rotation
    const float h1 = fmaf(-da, s, db * c);
    dg[2 * m] = fmaf(h0, f[2 * m] * rinv, dg[2 * m]);
    dg[2 * m + 1] = fmaf(h1, f[2 * m + 1] * rinv, dg[2 * m + 1]);
    u[2 * m] = g0 * h0;
    u[2 * m + 1] = g1 * h1;
    dot = fmaf(u[2 * m], f[2 * m], dot);
    dot = fmaf(u[2 * m + 1], f[2 * m + 1], dot);
  }
#pragma unroll
  for (int off = FL::TPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  const float c3 = rinv * rinv * rinv * dot * (1.0f / D);
  if (valid) {
#pragma unroll
    for (int m = 0; m < EPT / 2; ++m)
      store2<T>(dx + r * EPT + 2 * m, fmaf(rinv, u[2 * m], -f[2 * m] * c3),
                fmaf(rinv, u[2 * m + 1], -f[2 * m + 1] * c3));
  }
}

// feature_vals_bwd with the row's load.
template <int D, typename T>
__device__ __forceinline__ void feature_row_bwd(const T* x, bool valid, const float* gamma,
                                                int pos, const FeatureArgs& fa, int r,
                                                const float* df, T* dx,
                                                float (&dg)[FeatureLayout<D>::EPT]) {
  constexpr int EPT = FeatureLayout<D>::EPT;
  float f[EPT];
  if (valid) {
    RowLoad<T, EPT>::run(x + r * EPT, f);
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i) f[i] = 0.f;
  }
  feature_vals_bwd<D, T>(f, valid, gamma, pos, fa, r, df, dx, dg);
}

}  // namespace rapt
