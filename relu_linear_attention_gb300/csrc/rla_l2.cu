// Original RLA, non-causal, L2 denominator (08-rapt-algorithm.md §2.1, §2.2), sm_103a.
//
//   q' = ReLU(q), k' = ReLU(k);  M_V = K'^T V,  M_K = K'^T K'  (d x d each, over all L tokens)
//   out_t = q'_t M_V / (sqrt(q'_t^T M_K q'_t) + eps)
// By associativity sum_i s_ti v_i = q'_t (K'^T V) and sum_i s_ti^2 = q'_t^T (K'^T K') q'_t, so
// the L x L score matrix is never formed (§2.2: K'^T V first, then Q'(K'^T V)).
//
// Three launches on the caller's stream:
//   1. moments:  per (batch row, head, token split) the partial [M_V | M_K] (d x 2d, fp32) of
//                its split, written to the workspace (no atomics: the result is deterministic);
//   2. reduce:   sum of the partials in split order -> one [M_V | M_K] per (batch row, head);
//   3. readout:  per tile of tokens, q' [M_V | M_K] and the denominator, then out.
#include "kernels.h"

namespace rapt {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;      // tokens per shared-memory tile in the moment kernel
constexpr int kOutTile = 64;  // tokens per CTA in the readout kernel

int l2_nsplit(int B, int L, int H) {
  const long bh = static_cast<long>(B) * H;
  long want = (2L * 152 + bh - 1) / bh;          // about two CTAs per SM
  long cap = (L + 255) / 256;                    // at least 256 tokens per split
  long s = want < cap ? want : cap;
  return static_cast<int>(s < 1 ? 1 : s);
}

int l2_split_len(int L, int nsplit) {
  int s = (L + nsplit - 1) / nsplit;
  return ((s + kTok - 1) / kTok) * kTok;
}

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&f)[4]) { RowLoad<T, 4>::run(p, f); }

// Column mapping of the d x 2d moment tile: thread column tj owns W-wide groups
// j = g * (16 W) + tj * W + w, so 16 threads read 16 consecutive W-vectors (no bank conflicts).
template <int D>
struct MomCfg {
  static constexpr int TI = D / 16;          // rows per thread
  static constexpr int TJ = (2 * D) / 16;    // columns per thread
  static constexpr int W = TJ < 4 ? TJ : 4;  // contiguous columns per group
  static constexpr int G = TJ / W;           // groups
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) l2_moments_kernel(const L2Args a, int nsplit, int split_len) {
  using Cfg = MomCfg<D>;
  constexpr int TI = Cfg::TI, W = Cfg::W, G = Cfg::G;
  __shared__ __align__(16) float Ks[kTok][D];
  __shared__ __align__(16) float Xs[kTok][2 * D];  // [v | k']

  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int s0 = split * split_len;
  const int s1 = min(a.L, s0 + split_len);
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);

  float acc[TI][G * W];
#pragma unroll
  for (int i = 0; i < TI; ++i)
#pragma unroll
    for (int j = 0; j < G * W; ++j) acc[i][j] = 0.f;

  for (int t0 = s0; t0 < s1; t0 += kTok) {
    for (int idx = threadIdx.x; idx < kTok * (D / 4); idx += kThreads) {
      const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
      const int t = t0 + r;
      float kk[4] = {0.f, 0.f, 0.f, 0.f}, vv[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < s1) {
        const long off = ((static_cast<long>(b) * a.L + t) * a.H + h) * D + c4;
        load4(k + off, kk);
        load4(v + off, vv);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) kk[m] = fmaxf(kk[m], 0.f);
      *reinterpret_cast<float4*>(&Ks[r][c4]) = make_float4(kk[0], kk[1], kk[2], kk[3]);
      *reinterpret_cast<float4*>(&Xs[r][D + c4]) = make_float4(kk[0], kk[1], kk[2], kk[3]);
      *reinterpret_cast<float4*>(&Xs[r][c4]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
    }
    __syncthreads();
#pragma unroll 4
    for (int r = 0; r < kTok; ++r) {
      float av[TI], bv[G * W];
#pragma unroll
      for (int i = 0; i < TI; ++i) av[i] = Ks[r][ti * TI + i];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int w = 0; w < W; ++w) bv[g * W + w] = Xs[r][g * 16 * W + tj * W + w];
#pragma unroll
      for (int i = 0; i < TI; ++i)
#pragma unroll
        for (int j = 0; j < G * W; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }

  float* part = a.ws + (static_cast<long>(bh) * nsplit + split) * D * (2 * D);
#pragma unroll
  for (int i = 0; i < TI; ++i)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int w = 0; w < W; ++w)
        part[(ti * TI + i) * (2 * D) + g * 16 * W + tj * W + w] = acc[i][g * W + w];
}

// M[bh] = sum over splits (in order) of the partials.
__global__ void __launch_bounds__(kThreads) l2_reduce_kernel(const float* ws, long n_bh, int nsplit,
                                                             int mat4, float* M) {
  const long total = n_bh * mat4;
  for (long idx = blockIdx.x * static_cast<long>(kThreads) + threadIdx.x; idx < total;
       idx += static_cast<long>(gridDim.x) * kThreads) {
    const long bh = idx / mat4, e = idx % mat4;
    const float4* p = reinterpret_cast<const float4*>(ws) + bh * nsplit * mat4 + e;
    float4 s = p[0];
    for (int sp = 1; sp < nsplit; ++sp) {
      const float4 x = p[static_cast<long>(sp) * mat4];
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    reinterpret_cast<float4*>(M)[idx] = s;
  }
}

template <int D>
struct OutSmem {
  static constexpr int Ms = 0;                        // [D][2D]
  static constexpr int QsT = Ms + D * 2 * D;          // [D][kOutTile]
  static constexpr int Os = QsT + D * kOutTile;       // [kOutTile][D + 4]
  static constexpr int total = Os + kOutTile * (D + 4);
  static constexpr size_t bytes = static_cast<size_t>(total) * sizeof(float);
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) l2_out_kernel(const L2Args a, long m_offset) {
  using SM = OutSmem<D>;
  constexpr int NJ = D / 4;  // columns per thread (4 threads per token)
  extern __shared__ __align__(16) float sm[];
  float* Ms = sm + SM::Ms;
  float* QsT = sm + SM::QsT;
  float* Os = sm + SM::Os;

  const int tile = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int t0 = tile * kOutTile;
  const T* q = static_cast<const T*>(a.q);
  T* out = static_cast<T*>(a.out);

  const float4* Mg = reinterpret_cast<const float4*>(a.ws + m_offset + static_cast<long>(bh) * D * 2 * D);
  for (int idx = threadIdx.x; idx < D * 2 * D / 4; idx += kThreads)
    reinterpret_cast<float4*>(Ms)[idx] = Mg[idx];
  for (int idx = threadIdx.x; idx < kOutTile * (D / 4); idx += kThreads) {
    const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
    const int t = t0 + r;
    float f[4] = {0.f, 0.f, 0.f, 0.f};
    if (t < a.L) load4(q + ((static_cast<long>(b) * a.L + t) * a.H + h) * D + c4, f);
#pragma unroll
    for (int m = 0; m < 4; ++m) QsT[(c4 + m) * kOutTile + r] = fmaxf(f[m], 0.f);
  }
  __syncthreads();

  const int tt = threadIdx.x / 4, cg = threadIdx.x % 4;
  float an[NJ], aw[NJ];
#pragma unroll
  for (int m = 0; m < NJ; ++m) an[m] = aw[m] = 0.f;
  for (int i = 0; i < D; ++i) {
    const float qv = QsT[i * kOutTile + tt];
    const float* row = Ms + i * 2 * D;
#pragma unroll
    for (int m = 0; m < NJ; ++m) {
      an[m] = fmaf(qv, row[cg + 4 * m], an[m]);
      aw[m] = fmaf(qv, row[D + cg + 4 * m], aw[m]);
    }
  }
  float d2 = 0.f;
#pragma unroll
  for (int m = 0; m < NJ; ++m) d2 = fmaf(aw[m], QsT[(cg + 4 * m) * kOutTile + tt], d2);
  d2 += __shfl_xor_sync(0xffffffffu, d2, 1);
  d2 += __shfl_xor_sync(0xffffffffu, d2, 2);
  const float den = sqrtf(d2) + a.eps;
#pragma unroll
  for (int m = 0; m < NJ; ++m) Os[tt * (D + 4) + cg + 4 * m] = an[m] / den;
  __syncthreads();
  for (int idx = threadIdx.x; idx < kOutTile * (D / 4); idx += kThreads) {
    const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
    const int t = t0 + r;
    if (t < a.L) {
      const float* o = Os + r * (D + 4) + c4;
      store4(out + ((static_cast<long>(b) * a.L + t) * a.H + h) * D + c4, o[0], o[1], o[2], o[3]);
    }
  }
}

template <typename T, int D>
cudaError_t launch_t(const L2Args& a, cudaStream_t stream) {
  const int nsplit = l2_nsplit(a.B, a.L, a.H);
  const int split_len = l2_split_len(a.L, nsplit);
  const long n_bh = static_cast<long>(a.B) * a.H;
  const int mat4 = D * 2 * D / 4;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  l2_moments_kernel<T, D><<<dim3(nsplit, static_cast<unsigned>(n_bh)), kThreads, 0, stream>>>(a, nsplit, split_len);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long red_total = n_bh * mat4;
  long red_grid = (red_total + kThreads - 1) / kThreads;
  if (red_grid > 152L * 16) red_grid = 152L * 16;
  l2_reduce_kernel<<<static_cast<unsigned>(red_grid), kThreads, 0, stream>>>(
      a.ws, n_bh, nsplit, mat4, a.ws + n_bh * nsplit * static_cast<long>(mat4) * 4);
  note_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  constexpr size_t smem = OutSmem<D>::bytes;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(l2_out_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long m_offset = n_bh * nsplit * static_cast<long>(D) * 2 * D;
  const unsigned tiles = static_cast<unsigned>((a.L + kOutTile - 1) / kOutTile);
  l2_out_kernel<T, D><<<dim3(tiles, static_cast<unsigned>(n_bh)), kThreads, smem, stream>>>(a, m_offset);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_d(int d, const L2Args& a, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_t<T, 16>(a, stream);
    case 32: return launch_t<T, 32>(a, stream);
    case 64: return launch_t<T, 64>(a, stream);
    case 128: return launch_t<T, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The same three launches with a caller-chosen number of token splits; the workspace at a.ws
// holds (nsplit + 1) * B * H * d * 2d floats.
template <typename T, int D>
cudaError_t launch_t_splits(const L2Args& a, int nsplit, cudaStream_t stream) {
  const int split_len = l2_split_len(a.L, nsplit);
  const long n_bh = static_cast<long>(a.B) * a.H;
  const int mat4 = D * 2 * D / 4;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  l2_moments_kernel<T, D><<<dim3(nsplit, static_cast<unsigned>(n_bh)), kThreads, 0, stream>>>(a, nsplit, split_len);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long red_total = n_bh * mat4;
  long red_grid = (red_total + kThreads - 1) / kThreads;
  if (red_grid > 152L * 16) red_grid = 152L * 16;
  l2_reduce_kernel<<<static_cast<unsigned>(red_grid), kThreads, 0, stream>>>(
      a.ws, n_bh, nsplit, mat4, a.ws + n_bh * nsplit * static_cast<long>(mat4) * 4);
  note_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr size_t smem = OutSmem<D>::bytes;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(l2_out_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long m_offset = n_bh * nsplit * static_cast<long>(D) * 2 * D;
  const unsigned tiles = static_cast<unsigned>((a.L + kOutTile - 1) / kOutTile);
  l2_out_kernel<T, D><<<dim3(tiles, static_cast<unsigned>(n_bh)), kThreads, smem, stream>>>(a, m_offset);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_d_splits(int d, const L2Args& a, int nsplit, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_t_splits<T, 16>(a, nsplit, stream);
    case 32: return launch_t_splits<T, 32>(a, nsplit, stream);
    case 64: return launch_t_splits<T, 64>(a, nsplit, stream);
    case 128: return launch_t_splits<T, 128>(a, nsplit, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The moments only: partials into a.ws, then their sum into M (plain [bh][D][2D] fp32).
template <typename T, int D>
cudaError_t launch_moments_plain_t(const L2Args& a, float* M, cudaStream_t stream) {
  const int nsplit = l2_nsplit(a.B, a.L, a.H);
  const int split_len = l2_split_len(a.L, nsplit);
  const long n_bh = static_cast<long>(a.B) * a.H;
  const int mat4 = D * 2 * D / 4;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  l2_moments_kernel<T, D><<<dim3(nsplit, static_cast<unsigned>(n_bh)), kThreads, 0, stream>>>(a, nsplit, split_len);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long red_total = n_bh * mat4;
  long red_grid = (red_total + kThreads - 1) / kThreads;
  if (red_grid > 152L * 16) red_grid = 152L * 16;
  l2_reduce_kernel<<<static_cast<unsigned>(red_grid), kThreads, 0, stream>>>(a.ws, n_bh, nsplit, mat4, M);
  note_launches(1);
  return cudaGetLastError();
}

// The readout only, from the plain moments M (the same layout).
template <typename T, int D>
cudaError_t launch_readout_plain_t(const L2Args& a, const float* M, cudaStream_t stream) {
  const long n_bh = static_cast<long>(a.B) * a.H;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  constexpr size_t smem = OutSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(l2_out_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  L2Args b = a;
  b.ws = const_cast<float*>(M);  // read only
  const unsigned tiles = static_cast<unsigned>((a.L + kOutTile - 1) / kOutTile);
  l2_out_kernel<T, D><<<dim3(tiles, static_cast<unsigned>(n_bh)), kThreads, smem, stream>>>(b, 0L);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_plain_d(int d, const L2Args& a, float* Mout, const float* Min, cudaStream_t s) {
  const bool mom = Mout != nullptr;
  switch (d) {
    case 16: return mom ? launch_moments_plain_t<T, 16>(a, Mout, s) : launch_readout_plain_t<T, 16>(a, Min, s);
    case 32: return mom ? launch_moments_plain_t<T, 32>(a, Mout, s) : launch_readout_plain_t<T, 32>(a, Min, s);
    case 64: return mom ? launch_moments_plain_t<T, 64>(a, Mout, s) : launch_readout_plain_t<T, 64>(a, Min, s);
    case 128: return mom ? launch_moments_plain_t<T, 128>(a, Mout, s) : launch_readout_plain_t<T, 128>(a, Min, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t l2_moments_ws_bytes(int B, int L, int H, int d) {
  return static_cast<size_t>(B) * H * l2_nsplit(B, L, H) * d * 2 * d * sizeof(float);
}
cudaError_t launch_l2_moments_plain(DType dt, int d, const L2Args& a, float* M, cudaStream_t stream) {
  return dt == DType::F32 ? launch_plain_d<float>(d, a, M, nullptr, stream)
                          : launch_plain_d<__nv_bfloat16>(d, a, M, nullptr, stream);
}
cudaError_t launch_l2_readout_plain(DType dt, int d, const L2Args& a, const float* M, cudaStream_t stream) {
  return dt == DType::F32 ? launch_plain_d<float>(d, a, nullptr, M, stream)
                          : launch_plain_d<__nv_bfloat16>(d, a, nullptr, M, stream);
}

int l2_default_splits(int B, int L, int H) { return l2_nsplit(B, L, H); }

size_t l2_workspace_bytes_for_splits(int B, int H, int d, int nsplit) {
  return static_cast<size_t>(B) * H * (nsplit + 1) * d * 2 * d * sizeof(float);
}

cudaError_t launch_rla_l2_with_splits(DType dt, int d, const L2Args& a, int nsplit,
                                      cudaStream_t stream) {
  return dt == DType::F32 ? launch_d_splits<float>(d, a, nsplit, stream)
                          : launch_d_splits<__nv_bfloat16>(d, a, nsplit, stream);
}

size_t l2_workspace_bytes(int B, int L, int H, int d) {
  const long n_bh = static_cast<long>(B) * H;
  const int nsplit = l2_nsplit(B, L, H);
  return static_cast<size_t>(n_bh) * (nsplit + 1) * d * 2 * d * sizeof(float);
}

cudaError_t launch_rla_l2(DType dt, int d, const L2Args& a, cudaStream_t stream) {
  return dt == DType::F32 ? launch_d<float>(d, a, stream) : launch_d<__nv_bfloat16>(d, a, stream);
}

}  // namespace rapt
