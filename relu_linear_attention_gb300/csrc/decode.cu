// One RLA-2 decode step for N sequences (08-rapt-algorithm.md §4.2 forward_step), sm_103a.
//
// Per (sequence, head): features of the new token at its position; then, in ONE pass over the
// fp32 state S (d x d, key-major) and z:
//   S[i][:] += k'_i v,   z += k',   out = q' S / (q' . z + eps)     (update first, then read)
// The pass is a pure HBM stream: every element of S is read once and written once with 128-bit
// coalesced accesses (a warp covers 512 contiguous bytes of one row), all rows of a thread are
// loaded before any is used so that a CTA keeps d*d*4 bytes in flight, and the column sums of
// q'_i S[i][j] are reduced through shared memory. No host round trip (the reference engine took
// one for q'.z).
#include "kernels.h"

namespace rapt {
namespace {

constexpr int kThreads = 256;

template <int D>
struct DecodeCfg {
  static constexpr int CG = D / 4;                          // float4 column groups per row
  static constexpr int RG_ALL = kThreads / CG;              // thread rows available
  static constexpr int RG = RG_ALL < D ? RG_ALL : D;        // thread rows used
  static constexpr int ROWS = D / RG;                       // state rows per thread
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a) {
  using FL = FeatureLayout<D>;
  using Cfg = DecodeCfg<D>;
  constexpr int CG = Cfg::CG, RG = Cfg::RG, ROWS = Cfg::ROWS;
  __shared__ __align__(16) float qf[D];
  __shared__ __align__(16) float kf[D];
  __shared__ __align__(16) float vs[D];
  __shared__ __align__(16) float red[RG][D];
  __shared__ float den_s;

  const int nh = blockIdx.x;
  const int n = nh / a.H, h = nh % a.H;
  const long base = static_cast<long>(nh) * D;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pos = a.positions[n];

  if (warp < 2) {
    const int grp = lane / FL::TPR, r = lane % FL::TPR;
    const T* src = static_cast<const T*>(warp == 0 ? a.q : a.k) + base;
    const float* g = (warp == 0 ? a.gamma_q : a.gamma_k) + h * a.fa.gamma_stride;
    float f[FL::EPT];
    feature_row<D, T>(src, grp == 0, g, pos, a.fa, r, f);
    if (grp == 0) {
      float* dst = warp == 0 ? qf : kf;
#pragma unroll
      for (int e = 0; e < FL::EPT; ++e) dst[r * FL::EPT + e] = f[e];
    }
  } else if (warp == 2) {
    const T* src = static_cast<const T*>(a.v) + base;
    for (int j = lane; j < D; j += 32) vs[j] = to_f<T>(src[j]);
  }
  __syncthreads();

  if (warp == 0) {  // z += k', den = q' . z_new + eps
    float s = 0.f;
    for (int i = lane; i < D; i += 32) {
      const float zn = a.z[base + i] + kf[i];
      a.z[base + i] = zn;
      s = fmaf(qf[i], zn, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) den_s = s + a.eps_den;
  }

  const int cg = tid % CG, rg = tid / CG;
  if (rg < RG) {
    float* S = a.S + static_cast<long>(nh) * D * D;
    float4 sv[ROWS];
#pragma unroll
    for (int m = 0; m < ROWS; ++m)
      sv[m] = __ldcs(reinterpret_cast<const float4*>(S + (rg + m * RG) * D + 4 * cg));
    const float4 vv = *reinterpret_cast<const float4*>(vs + 4 * cg);
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
    for (int m = 0; m < ROWS; ++m) {
      const int i = rg + m * RG;
      const float ki = kf[i], qi = qf[i];
      float4 s4 = sv[m];
      s4.x = fmaf(ki, vv.x, s4.x);
      s4.y = fmaf(ki, vv.y, s4.y);
      s4.z = fmaf(ki, vv.z, s4.z);
      s4.w = fmaf(ki, vv.w, s4.w);
      __stcs(reinterpret_cast<float4*>(S + i * D + 4 * cg), s4);
      acc0 = fmaf(qi, s4.x, acc0);
      acc1 = fmaf(qi, s4.y, acc1);
      acc2 = fmaf(qi, s4.z, acc2);
      acc3 = fmaf(qi, s4.w, acc3);
    }
    *reinterpret_cast<float4*>(&red[rg][4 * cg]) = make_float4(acc0, acc1, acc2, acc3);
  }
  __syncthreads();
  if (tid < D) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < RG; ++g) s += red[g][tid];
    static_cast<T*>(a.out)[base + tid] = from_float<T>(s / den_s);
  }
}

template <typename T, int D>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t stream) {
  const long grid = static_cast<long>(a.N) * a.H;
  if (grid == 0) return cudaSuccess;
  decode_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_d(int d, const DecodeArgs& a, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_t<T, 16>(a, stream);
    case 32: return launch_t<T, 32>(a, stream);
    case 64: return launch_t<T, 64>(a, stream);
    case 128: return launch_t<T, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(DType dt, int d, const DecodeArgs& a, cudaStream_t stream) {
  return dt == DType::F32 ? launch_d<float>(d, a, stream) : launch_d<__nv_bfloat16>(d, a, stream);
}

}  // namespace rapt
