// One sequence split across GPUs: the state of a shard, and the state a shard starts from.
//
// The RLA-2 state is a plain sum over tokens, S_t = sum_{i<=t} k'_i v_i^T and z_t = sum k'_i
// (08-rapt-algorithm.md §3), so it can be accumulated chunk by chunk in parallel and the partial
// sums added afterwards (the chunk-parallel accumulation of §1 and §3). A sequence cut into W
// consecutive shards of L tokens, one per GPU, is therefore computed in three steps:
//   1. every shard's increment (dS, dz) = sum over its own tokens (shard_state_*, here);
//   2. the W increments are gathered on every GPU (one all-gather, by the caller);
//   3. shard r starts from S0 + dS_0 + ... + dS_{r-1} (state_prefix_kernel, here) and runs the
//      ordinary causal prefill from that initial state, with RoPE positions continuing from the
//      shard's first token.
// Step 1 reuses the tensor-core state kernel of the prefill (bf16, d in {64, 128}) or, for the
// other cases, the CUDA-core kernel below; both write per-block records that state_sum_kernel adds
// up in block order. Every sum has a fixed order, so the results are bitwise repeatable.
#include "common.cuh"
#include "kernels.h"
#include "simt_tiles.cuh"
#include "tc_features.cuh"

namespace rapt {
namespace {

using feat::Rec;

constexpr int kThreads = 256;
constexpr int kTok = 32;  // tokens per shared-memory tile of the CUDA-core state kernel

template <int D>
struct StateSmem {
  static constexpr int LD = D + 4;  // padded row stride: float4 aligned, rows in distinct bank groups
  static constexpr int KF = 0;                 // [kTok][LD] k'
  static constexpr int VS = KF + kTok * LD;    // [kTok][LD] v
  static constexpr int total = VS + kTok * LD;
};

// CUDA-core state increment of one block of blk_len tokens of one (batch row, head): K'^T V and
// the column sums of k', written as one record in the tensor-core kernels' layout (the float4 of
// row i and columns 4c..4c+3 at float4 index c * D + i, then the D sums). fp32 arithmetic.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) shard_state_simt(const PrefillArgs a, float* rec,
                                                             int blk_len, int nblk) {
  using SM = StateSmem<D>;
  using FL = FeatureLayout<D>;
  constexpr int LD = SM::LD, NQ = D / 4;
  constexpr int NT = NQ * NQ;                              // 4 x 4 tiles of K'^T V
  constexpr int TPT = (NT + kThreads - 1) / kThreads;      // tiles per thread
  __shared__ __align__(16) float sm[SM::total];
  float* Kf = sm + SM::KF;
  float* Vs = sm + SM::VS;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x % nblk, bh = blockIdx.x / nblk;
  const int h = bh % a.H, b = bh / a.H;
  const long row0 = static_cast<long>(b) * a.doc_len;
  const int n = a.doc_len;
  const int s0 = blk * blk_len, s1 = min(n, s0 + blk_len);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const float* gk = a.gamma_k + h * a.fa.gamma_stride;

  float acc[TPT][4][4];
#pragma unroll
  for (int u = 0; u < TPT; ++u)
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[u][y][x] = 0.f;
  float zsum = 0.f;

  const int grp = lane / FL::TPR, r = lane % FL::TPR;
  constexpr int kRowsPerPass = (kThreads / 32) * FL::ROWS_PER_WARP;
  for (int t0 = s0; t0 < s1; t0 += kTok) {
    __syncthreads();  // the previous tile's reads are done
    for (int rr = warp * FL::ROWS_PER_WARP + grp; rr < kTok; rr += kRowsPerPass) {
      const int t = t0 + rr;
      const bool valid = t < s1;
      float f[FL::EPT];
      feature_row<D, T>(k + ((row0 + (valid ? t : 0)) * a.H + h) * D, valid, gk, a.pos_offset + t,
                        a.fa, r, f);
#pragma unroll
      for (int e = 0; e < FL::EPT; ++e) Kf[rr * LD + r * FL::EPT + e] = f[e];
    }
    for (int idx = tid; idx < kTok * NQ; idx += kThreads) {
      const int rr = idx / NQ, j4 = 4 * (idx % NQ);
      float f4[4] = {0.f, 0.f, 0.f, 0.f};
      if (t0 + rr < s1) RowLoad<T, 4>::run(v + ((row0 + t0 + rr) * a.H + h) * D + j4, f4);
      *reinterpret_cast<float4*>(Vs + rr * LD + j4) = make_float4(f4[0], f4[1], f4[2], f4[3]);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < TPT; ++u) {
      const int task = tid + u * kThreads;
      if (task < NT) {
        const int i0 = 4 * (task / NQ), j0 = 4 * (task % NQ);
        simt::mt_tn<1>(acc[u], Kf + i0, LD, Vs + j0, LD, kTok);
      }
    }
    if (tid < D)
      for (int t = 0; t < kTok; ++t) zsum += Kf[t * LD + tid];
  }
  float4* dst = reinterpret_cast<float4*>(rec + (static_cast<long>(bh) * nblk + blk) * Rec<D>::FLOATS);
#pragma unroll
  for (int u = 0; u < TPT; ++u) {
    const int task = tid + u * kThreads;
    if (task < NT) {
      const int i0 = 4 * (task / NQ), c = task % NQ;
#pragma unroll
      for (int y = 0; y < 4; ++y)
        dst[c * D + i0 + y] = make_float4(acc[u][y][0], acc[u][y][1], acc[u][y][2], acc[u][y][3]);
    }
  }
  if (tid < D) rec[(static_cast<long>(bh) * nblk + blk) * Rec<D>::FLOATS + Rec<D>::Z + tid] = zsum;
}

// S[bh] (row-major d x d) and z[bh] from the nblk records of (batch row, head) bh, added in block
// order. One thread per float4 of S (and per element of z).
template <int D>
__global__ void __launch_bounds__(kThreads) state_sum_kernel(const float* rec, int nblk, long n_bh,
                                                             float* S, float* z) {
  constexpr int Q = D * D / 4;
  const long idx = blockIdx.x * static_cast<long>(kThreads) + threadIdx.x;
  const long bh = idx / (Q + D);
  if (bh >= n_bh) return;
  const int e = static_cast<int>(idx % (Q + D));
  const float* base = rec + bh * nblk * Rec<D>::FLOATS;
  if (e < Q) {
    const int i = e % D, c = e / D;  // record layout: float4 (i, 4c .. 4c+3) at c * D + i
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < nblk; ++g) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(base + g * Rec<D>::FLOATS) + e);
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    *reinterpret_cast<float4*>(S + (bh * D + i) * D + 4 * c) = s;
  } else {
    const int j = e - Q;
    float s = 0.f;
    for (int g = 0; g < nblk; ++g) s += __ldcg(base + g * Rec<D>::FLOATS + Rec<D>::Z + j);
    z[bh * D + j] = s;
  }
}

// out = init (or 0) + parts[0] + ... + parts[r-1], element-wise over n4 float4 (rank order).
__global__ void __launch_bounds__(kThreads) state_prefix_kernel(const float4* parts, long n4,
                                                                int r, const float4* init,
                                                                float4* out) {
  for (long i = blockIdx.x * static_cast<long>(kThreads) + threadIdx.x; i < n4;
       i += static_cast<long>(gridDim.x) * kThreads) {
    float4 s = init != nullptr ? init[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < r; ++w) {
      const float4 x = parts[static_cast<long>(w) * n4 + i];
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    out[i] = s;
  }
}

template <typename T, int D>
cudaError_t launch_simt_t(const PrefillArgs& a, float* rec, int blk_len, int nblk, cudaStream_t s) {
  const long grid = static_cast<long>(a.n_docs) * a.H * nblk;
  shard_state_simt<T, D><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a, rec, blk_len, nblk);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt_d(int d, const PrefillArgs& a, float* rec, int blk_len, int nblk,
                          cudaStream_t s) {
  switch (d) {
    case 16: return launch_simt_t<T, 16>(a, rec, blk_len, nblk, s);
    case 32: return launch_simt_t<T, 32>(a, rec, blk_len, nblk, s);
    case 64: return launch_simt_t<T, 64>(a, rec, blk_len, nblk, s);
    case 128: return launch_simt_t<T, 128>(a, rec, blk_len, nblk, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_sum_d(const float* rec, int nblk, long n_bh, float* S, float* z, cudaStream_t s) {
  const long total = n_bh * (D * D / 4 + D);
  state_sum_kernel<D><<<static_cast<unsigned>((total + kThreads - 1) / kThreads), kThreads, 0, s>>>(
      rec, nblk, n_bh, S, z);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

ShardPlan shard_state_plan(DType dt, int B, int L, int H, int d) {
  // Blocks of whole 128-token chunks (tensor cores) or 32-token tiles (CUDA cores), as many as
  // fill about one wave of CTAs (one CTA per SM on the tensor-core path, several otherwise).
  ShardPlan p{};
  p.tc = tc_supported(dt, d);
  const int unit = p.tc ? 128 : kTok;
  const long bh = static_cast<long>(B) * H;
  const int units_max = L > 0 ? (L + unit - 1) / unit : 1;
  const long want = p.tc ? 152 : 4 * 152;
  long nblk = (want + bh - 1) / bh;
  if (nblk > units_max) nblk = units_max;
  if (nblk < 1) nblk = 1;
  const int per = static_cast<int>((units_max + nblk - 1) / nblk);
  p.blk_len = per * unit;
  p.nblk = L > 0 ? (L + p.blk_len - 1) / p.blk_len : 1;
  p.ws_bytes = static_cast<size_t>(bh) * p.nblk * d * (d + 1) * sizeof(float);
  return p;
}

cudaError_t launch_shard_state(DType dt, int d, const PrefillArgs& a, const ShardPlan& p, float* ws,
                               float* S, float* z, cudaStream_t stream) {
  const long n_bh = static_cast<long>(a.n_docs) * a.H;
  if (n_bh == 0) return cudaSuccess;
  cudaError_t e;
  if (p.tc) {
    TcArgs ta{};
    ta.p = a;
    ta.ws = ws;
    ta.seg_len = p.blk_len;
    ta.nseg_max = 1;
    ta.blk_len = p.blk_len;
    ta.blk_per_seg = 1;
    ta.nblk_max = p.nblk;
    ta.whole_doc = 1;
    e = launch_state_tc(d, ta, stream);
  } else {
    e = dt == DType::F32 ? launch_simt_d<float>(d, a, ws, p.blk_len, p.nblk, stream)
                         : launch_simt_d<__nv_bfloat16>(d, a, ws, p.blk_len, p.nblk, stream);
  }
  if (e != cudaSuccess) return e;
  switch (d) {
    case 16: return launch_sum_d<16>(ws, p.nblk, n_bh, S, z, stream);
    case 32: return launch_sum_d<32>(ws, p.nblk, n_bh, S, z, stream);
    case 64: return launch_sum_d<64>(ws, p.nblk, n_bh, S, z, stream);
    case 128: return launch_sum_d<128>(ws, p.nblk, n_bh, S, z, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_state_prefix(const float* parts, long n, int r, const float* init, float* out,
                                cudaStream_t stream) {
  const long n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  long grid = (n4 + kThreads - 1) / kThreads;
  if (grid > 152L * 8) grid = 152L * 8;
  state_prefix_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(parts), n4, r, reinterpret_cast<const float4*>(init),
      reinterpret_cast<float4*>(out));
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rapt
