// Causal original RLA (L2 denominator) on CUDA cores (fp32 arithmetic, fp32 or bf16 tensors).
//
// 08-rapt-algorithm.md §2.1 (closed form, eps 1e-6 outside the root, features ReLU(q), ReLU(k)
// with no norm and no RoPE), §2.2 (the causal state restarts at document boundaries) and §4.1
// (the prefix scan's two states):
//   S_t = sum_{i<=t} k'_i v_i^T,  A_t = sum_{i<=t} k'_i k'_i^T,
//   out_t = q'_t S_t / (sqrt(q'_t^T A_t q'_t) + eps).
// In chunked form (C = 32 tokens) with P = (Q'_c K'_c^T) masked to tau <= t:
//   num = P V_c + Q'_c S,   den^2 = rowsum(P (.) P) + rowsum((Q'_c A) (.) Q'_c),
// then S += K'_c^T V_c and A += K'_c^T K'_c. Documents are cut into segments: launch 1 writes the
// increments (K'^T V, K'^T K') of every segment but a document's last, launch 2 runs one CTA per
// (document, head, segment) from the sum of the earlier segments' increments (in segment order,
// so results are bitwise repeatable).
#include "kernels.h"
#include "simt_tiles.cuh"
#include "tc_features.cuh"

namespace rapt {
namespace {

using feat::doc_bounds;
using namespace simt;

constexpr int kC = 32;
constexpr int kThreads = 256;
constexpr int kSMs = 152;

template <int D>
struct L2cSmem {
  static constexpr int LD = D + 4;  // row stride: LD / 4 odd
  static constexpr int LC = kC + 4;
  static constexpr int ST = 0;             // [D][LD] S
  static constexpr int AT = ST + D * LD;   // [D][LD] A
  static constexpr int QF = AT + D * LD;   // [C][LD] q'
  static constexpr int KF = QF + kC * LD;  // [C][LD] k'
  static constexpr int VS = KF + kC * LD;  // [C][LD] v
  static constexpr int PS = VS + kC * LD;  // [C][LC] masked scores
  static constexpr int SQ = PS + kC * LC;  // [C] q'^T A q' of the chunk's rows
  static constexpr int DEN = SQ + kC;      // [C]
  static constexpr int total = DEN + kC;
  static constexpr size_t bytes = static_cast<size_t>(total) * sizeof(float);
  static_assert(bytes <= 232448, "shared memory budget");
};

// ReLU(x) of C rows starting at token t0 into a [C][LD] tile (tail rows zero).
template <int D, typename T>
__device__ __forceinline__ void relu_tile(const T* x, long row0, int n, int t0, int H, int h,
                                          float* tile, bool relu) {
  constexpr int LD = L2cSmem<D>::LD;
  for (int idx = threadIdx.x; idx < kC * (D / 4); idx += kThreads) {
    const int rr = idx / (D / 4), j4 = 4 * (idx % (D / 4));
    float f[4] = {0.f, 0.f, 0.f, 0.f};
    if (t0 + rr < n) RowLoad<T, 4>::run(x + ((row0 + t0 + rr) * H + h) * D + j4, f);
    if (relu)
#pragma unroll
      for (int e = 0; e < 4; ++e) f[e] = fmaxf(f[e], 0.f);
    *reinterpret_cast<float4*>(tile + rr * LD + j4) = make_float4(f[0], f[1], f[2], f[3]);
  }
}

// S += K'^T V and A += K'^T K' for the chunk in Kf / Vs (D x D tiles of 4 x 4 per task).
template <int D>
__device__ __forceinline__ void add_chunk(float* St, float* At, const float* Kf, const float* Vs) {
  constexpr int LD = L2cSmem<D>::LD, NQ = D / 4;
  for (int task = threadIdx.x; task < 2 * NQ * NQ; task += kThreads) {
    const bool a = task >= NQ * NQ;
    const int tt = a ? task - NQ * NQ : task;
    const int i0 = 4 * (tt / NQ), j0 = 4 * (tt % NQ);
    float acc[4][4] = {};
    mt_tn<1>(acc, Kf + i0, LD, (a ? Kf : Vs) + j0, LD, kC);
    float* M = a ? At : St;
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) M[(i0 + y) * LD + j0 + x] += acc[y][x];
  }
}

// Launch 1: the increments of every segment that another segment of its document follows.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) l2c_state_kernel(const L2cArgs b) {
  using SM = L2cSmem<D>;
  constexpr int LD = SM::LD;
  extern __shared__ __align__(16) float sm[];
  float* St = sm + SM::ST;
  float* At = sm + SM::AT;
  float* Kf = sm + SM::KF;
  float* Vs = sm + SM::VS;
  const PrefillArgs& a = b.p;
  const int seg = blockIdx.x % b.nseg, unit = blockIdx.x / b.nseg;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  if (s1 >= n) return;  // a document's last (or an empty) segment: nobody reads its increment
  for (int idx = threadIdx.x; idx < D * D; idx += kThreads) {
    St[(idx / D) * LD + idx % D] = 0.f;
    At[(idx / D) * LD + idx % D] = 0.f;
  }
  for (int t0 = s0; t0 < s1; t0 += kC) {
    __syncthreads();
    relu_tile<D, T>(static_cast<const T*>(a.k), row0, n, t0, a.H, h, Kf, true);
    relu_tile<D, T>(static_cast<const T*>(a.v), row0, n, t0, a.H, h, Vs, false);
    __syncthreads();
    add_chunk<D>(St, At, Kf, Vs);
  }
  __syncthreads();
  float* rec = b.rec + (static_cast<long>(unit) * b.nseg + seg) * (2L * D * D);
  for (int idx = threadIdx.x; idx < D * D; idx += kThreads) {
    rec[idx] = St[(idx / D) * LD + idx % D];
    rec[D * D + idx] = At[(idx / D) * LD + idx % D];
  }
}

// Launch 2: the output, chunks in order.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) l2c_kernel(const L2cArgs b) {
  using SM = L2cSmem<D>;
  constexpr int LD = SM::LD, LC = SM::LC, NQ = D / 4;
  extern __shared__ __align__(16) float sm[];
  float* St = sm + SM::ST;
  float* At = sm + SM::AT;
  float* Qf = sm + SM::QF;
  float* Kf = sm + SM::KF;
  float* Vs = sm + SM::VS;
  float* Ps = sm + SM::PS;
  float* Sq = sm + SM::SQ;
  float* Den = sm + SM::DEN;
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x;
  const int seg = blockIdx.x % b.nseg, unit = blockIdx.x / b.nseg;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  if (!doc_bounds(a, doc, row0, n) && seg == 0 && h == 0 && tid == 0 && a.dev_status != nullptr)
    atomicOr(a.dev_status, 1u);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  if (s0 >= s1) return;
  const long rec = 2L * D * D;
  const float* rf = b.rec + static_cast<long>(unit) * b.nseg * rec;
  for (int idx = tid; idx < D * D; idx += kThreads) {
    float s = 0.f, m = 0.f;
    for (int sp = 0; sp < seg; ++sp) {
      s += rf[sp * rec + idx];
      m += rf[sp * rec + D * D + idx];
    }
    St[(idx / D) * LD + idx % D] = s;
    At[(idx / D) * LD + idx % D] = m;
  }
  T* out = static_cast<T*>(a.out);
  for (int t0 = s0; t0 < s1; t0 += kC) {
    __syncthreads();
    relu_tile<D, T>(static_cast<const T*>(a.q), row0, n, t0, a.H, h, Qf, true);
    relu_tile<D, T>(static_cast<const T*>(a.k), row0, n, t0, a.H, h, Kf, true);
    relu_tile<D, T>(static_cast<const T*>(a.v), row0, n, t0, a.H, h, Vs, false);
    __syncthreads();
    if (tid < 64) {  // P[t][tau] = q'_t . k'_tau, tau <= t
      const int m0 = 4 * (tid / 8), nb = tid % 8;
      float acc[4][4] = {};
      mt_dot<8>(acc, Qf + m0 * LD, LD, Kf + nb * LD, LD, D);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int t = m0 + y, tau = nb + 8 * x;
          Ps[t * LC + tau] = tau <= t ? acc[y][x] : 0.f;
        }
    }
    __syncthreads();
    // num = P V + Q' S (kept in registers); q'^T A q' = rowsum((Q' A) (.) Q')
    const bool has = tid < 8 * NQ;
    const int m0 = 4 * (tid / NQ), n0 = 4 * (tid % NQ);
    float num[4][4] = {};
    if (has) {
      mt_outer<1>(num, Ps + m0 * LC, LC, Vs + n0, LD, kC);
      mt_outer<1>(num, Qf + m0 * LD, LD, St + n0, LD, D);
      float qa[4][4] = {};
      mt_outer<1>(qa, Qf + m0 * LD, LD, At + n0, LD, D);
      float part[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const float4 qq = ld4(Qf + (m0 + y) * LD + n0);
        part[y] = qa[y][0] * qq.x + qa[y][1] * qq.y + qa[y][2] * qq.z + qa[y][3] * qq.w;
      }
#pragma unroll
      for (int off = NQ / 2; off > 0; off >>= 1)
#pragma unroll
        for (int y = 0; y < 4; ++y) part[y] += __shfl_xor_sync(0xffffffffu, part[y], off);
      if (tid % NQ == 0)
#pragma unroll
        for (int y = 0; y < 4; ++y) Sq[m0 + y] = part[y];
    }
    __syncthreads();
    if (tid < kC) {
      float ss = Sq[tid];
      for (int tau = 0; tau < kC; ++tau) ss = fmaf(Ps[tid * LC + tau], Ps[tid * LC + tau], ss);
      Den[tid] = sqrtf(fmaxf(ss, 0.f)) + b.eps;
    }
    __syncthreads();
    if (has) {
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int t = m0 + y;
        if (t0 + t < n) {
          const float den = Den[t];
          store4(out + ((row0 + t0 + t) * a.H + h) * D + n0, num[y][0] / den, num[y][1] / den,
                 num[y][2] / den, num[y][3] / den);
        }
      }
    }
    add_chunk<D>(St, At, Kf, Vs);  // reads Kf / Vs only; S and A reads of this chunk are done
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

template <typename T, int D>
cudaError_t launch_t(const L2cArgs& b, cudaStream_t stream) {
  constexpr size_t smem = L2cSmem<D>::bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    if ((e = set_smem(l2c_state_kernel<T, D>, smem)) != cudaSuccess) return e;
    if ((e = set_smem(l2c_kernel<T, D>, smem)) != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long grid = static_cast<long>(b.p.n_docs) * b.p.H * b.nseg;
  if (grid == 0) return cudaSuccess;
  if (b.nseg > 1) {
    l2c_state_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(b);
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  l2c_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(b);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_d(int d, const L2cArgs& b, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_t<T, 16>(b, stream);
    case 32: return launch_t<T, 32>(b, stream);
    case 64: return launch_t<T, 64>(b, stream);
    case 128: return launch_t<T, 128>(b, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

L2cPlan l2c_plan(int n_docs, int H, int max_seqlen, int d) {
  // One CTA per SM; a plan costs its waves of kSMs CTAs times the chunks of a segment (plus one
  // of set-up); a longer plan must be clearly (5 %) cheaper to win.
  L2cPlan p{1, 0, 0};
  const int chunks_max = max_seqlen > 0 ? (max_seqlen + kC - 1) / kC : 1;
  const long units = static_cast<long>(n_docs) * H;
  double best = 1e300;
  for (int nseg = 1; nseg <= 64 && nseg <= chunks_max; ++nseg) {
    const int seg_chunks = (chunks_max + nseg - 1) / nseg;
    const double waves = static_cast<double>((units * nseg + kSMs - 1) / kSMs);
    const double cost = waves * (seg_chunks + 1.0);
    if (cost < 0.95 * best) {
      best = cost;
      p.nseg = nseg;
      p.seg_len = seg_chunks * kC;
    }
  }
  if (p.seg_len == 0) p.seg_len = chunks_max * kC;
  p.ws_bytes = p.nseg > 1 ? static_cast<size_t>(units) * p.nseg * 2 * d * d * sizeof(float) : 0;
  return p;
}

cudaError_t launch_l2_causal_simt(DType dt, int d, const L2cArgs& b, cudaStream_t stream) {
  return dt == DType::F32 ? launch_d<float>(d, b, stream) : launch_d<__nv_bfloat16>(d, b, stream);
}

}  // namespace rapt
