// Device helpers shared by the RLA-2 / RAPT kernels (sm_103a).
//
// Feature map of RLA-2 (neuralnet.cpp page "线性注意力家族：RLA / RAPT / RLA-2 与 GPU 落地",
// 08-rapt-algorithm.md §1, §3, §4.2): q' = ReLU(RoPE(RMSNorm(q))), same for k; v is untouched.
// RMSNorm statistics and gains are fp32 (ruDNN README §7); RoPE rotates adjacent pairs
// (2j, 2j+1) (candle "05-nn/layers", rotary_emb, interleaved variant) by p * base^(-2j/d).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rapt {

constexpr int kMaxD = 128;

// Per-call feature settings, passed by value as a kernel parameter.
// rope_hi[j] + rope_lo[j] = base^(-2j/d) / (2 pi): the pair's frequency in TURNS per position,
// split into two floats on the host (computed in double). Keeping the angle in turns lets the
// kernel take the fractional part exactly (see rope_sincos) before any rounding of 2 pi.
struct FeatureArgs {
  float eps_norm;
  int gamma_stride;  // 0: one gain vector for all heads; d: gains are [H, d]
  float rope_hi[kMaxD / 2];
  float rope_lo[kMaxD / 2];
};

// sin / cos of the RoPE angle p * theta_j.
// The angle in turns, p * (hi + lo), is formed as h + e + p*lo with h = fl(p*hi) and e the exact
// rounding error of that product (an FMA gives it exactly; a two-product split). h - rint(h) is
// exact for |h| < 2^23, so the reduced angle t in [-1/2, 1/2] turn carries ~1e-8 turn absolute
// error at any position, instead of the ~p * 2^-24 rad of a plain fp32 product. The hardware
// sine/cosine is then evaluated on |2 pi t| <= pi, its accurate range.
__device__ __forceinline__ void rope_sincos(int p, float fhi, float flo, float& s, float& c) {
  const float pf = static_cast<float>(p);
  const float h = pf * fhi;
  const float e = fmaf(pf, fhi, -h);
  const float t = (h - rintf(h)) + fmaf(pf, flo, e);
  __sincosf(t * 6.283185307179586f, &s, &c);
}

// ---------------------------------------------------------------------------------------------
// Loads of N consecutive elements as floats (N even; 16-byte aligned rows make every access
// naturally aligned).
template <typename T, int N>
struct RowLoad;

template <int N>
struct RowLoad<float, N> {
  static __device__ __forceinline__ void run(const float* p, float (&f)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 4) {
        const float4 x = *reinterpret_cast<const float4*>(p + i);
        f[i] = x.x; f[i + 1] = x.y; f[i + 2] = x.z; f[i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < N; i += 2) {
        const float2 x = *reinterpret_cast<const float2*>(p + i);
        f[i] = x.x; f[i + 1] = x.y;
      }
    }
  }
};

template <int N>
struct RowLoad<__nv_bfloat16, N> {
  static __device__ __forceinline__ void run(const __nv_bfloat16* p, float (&f)[N]) {
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(p + i);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[m]));
          f[i + 2 * m] = g.x; f[i + 2 * m + 1] = g.y;
        }
      }
    } else if constexpr (N % 4 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 4) {
        const uint2 x = *reinterpret_cast<const uint2*>(p + i);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
        f[i] = a.x; f[i + 1] = a.y; f[i + 2] = b.x; f[i + 3] = b.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < N; i += 2) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p + i));
        f[i] = a.x; f[i + 1] = a.y;
      }
    }
  }
};

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Stores 4 consecutive values (16-byte aligned for fp32, 8-byte for bf16).
__device__ __forceinline__ void store4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
  __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&lo);
  w.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = w;
}

// ---------------------------------------------------------------------------------------------
// Feature row: a group of TPR consecutive lanes (TPR a power of two <= 32, group aligned inside
// the warp) turns one token's d-vector x into f = ReLU(RoPE(RMSNorm(x))). Lane r of the group owns
// elements [r*EPT, (r+1)*EPT), EPT = D / TPR (even, so RoPE pairs never straddle lanes).
// All lanes of the warp must call this together (the reduction shuffles across the full warp).
template <int D>
struct FeatureLayout {
  static constexpr int TPR = (D / 2) < 32 ? (D / 2) : 32;
  static constexpr int EPT = D / TPR;
  static constexpr int ROWS_PER_WARP = 32 / TPR;
};

// The arithmetic of feature_row on values already loaded into f (the lane's EPT elements; zeros
// for an invalid row), so that a caller can issue the loads of several rows before using them.
template <int D>
__device__ __forceinline__ void feature_vals(float (&f)[FeatureLayout<D>::EPT], bool valid,
                                             const float* gamma, int pos, const FeatureArgs& fa,
                                             int r) {
  using FL = FeatureLayout<D>;
  constexpr int EPT = FL::EPT;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < EPT; ++i) ss = fmaf(f[i], f[i], ss);
#pragma unroll
  for (int off = FL::TPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rinv = rsqrtf(ss * (1.0f / D) + fa.eps_norm);
#pragma unroll
  for (int m = 0; m < EPT / 2; ++m) {
    const int e = r * EPT + 2 * m;  // even element index: pair j = e / 2
    const float y0 = f[2 * m] * rinv * gamma[e];
    const float y1 = f[2 * m + 1] * rinv * gamma[e + 1];
    float s, c;
    rope_sincos(pos, fa.rope_hi[e >> 1], fa.rope_lo[e >> 1], s, c);
    const float a = fmaf(y0, c, -y1 * s);
    const float b = fmaf(y0, s, y1 * c);
    f[2 * m] = valid ? fmaxf(a, 0.f) : 0.f;
    f[2 * m + 1] = valid ? fmaxf(b, 0.f) : 0.f;
  }
}

template <int D, typename T>
__device__ __forceinline__ void feature_row(const T* x, bool valid, const float* gamma, int pos,
                                            const FeatureArgs& fa, int r,
                                            float (&f)[FeatureLayout<D>::EPT]) {
  using FL = FeatureLayout<D>;
  constexpr int EPT = FL::EPT;
  if (valid) {
    RowLoad<T, EPT>::run(x + r * EPT, f);
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i) f[i] = 0.f;
  }
  feature_vals<D>(f, valid, gamma, pos, fa, r);
}

}  // namespace rapt
