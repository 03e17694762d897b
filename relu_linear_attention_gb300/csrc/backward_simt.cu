// Backward of causal RLA-2 on CUDA cores (fp32 arithmetic, fp32 or bf16 tensors), sm_103a.
//
// Gradients of a loss with upstream gradient g_t = dL/dout_t (08-rapt-algorithm.md §4.2
// "backward": one prefix scan, two suffix scans, then the feature chain). Per document and head,
// with s_{t,tau} = q'_t . k'_tau for tau <= t:
//   den_t   = sum_{tau<=t} s_{t,tau} + eps,   num_t = sum_{tau<=t} s_{t,tau} v_tau
//   gnum_t  = g_t / den_t,                     scale_t = -(g_t . num_t) / den_t^2
//   dq'_t   = S_t gnum_t + scale_t z_t                       (prefix state S_t, z_t)
//   dk'_tau = R_tau v_tau + w_tau,   dv_tau = R_tau^T k'_tau  (suffix state
//             R_tau = sum_{t>=tau} q'_t gnum_t^T,  w_tau = sum_{t>=tau} scale_t q'_t)
// then through ReLU (the gradient passes where the pre-activation is > 0), the inverse RoPE
// rotation and RMSNorm (input and gain). In chunked form (C = 32 tokens), each chunk splits every
// sum into the state carried in from earlier (later) chunks and a masked C x C block.
//
// The in-chunk block A[t][tau] = gnum_t . v_tau + scale_t (tau <= t) is a difference of two terms
// that nearly cancel where a query sees few keys (for the first token of a document it is
// (g . v) eps / den^2 while each term is ~ (g . v) / den). It is formed as
//   A[t][tau] = ( sum_{sigma<=t in chunk} s_{t,sigma} (c_{t,tau} - c_{t,sigma})
//                 + c_{t,tau} sst_t - nst_t + eps c_{t,tau} ) / den_t^2,   c_{t,tau} = g_t . v_tau,
// with sst_t = q'_t . z and nst_t = g_t . (q'_t S) of the state before the chunk: the same value,
// but the cancelling part is the difference of equal products inside a document's first chunk,
// which is exact, so the gradient keeps its fp32 accuracy relative to its own size.
//
// Four launches on the caller's stream:
//   1. bwd_state_kernel: K'^T V and sum k' of every segment but a document's last (the prefix
//      states the segments of launch 2 start from);
//   2. bwd_forward_kernel, one CTA per (document, head, segment), chunks in order: den, scale and
//      gnum of every token (den and scale saved for launch 3), dq' and dq, the gain partials of q,
//      and the segment's increment of the suffix state (Q'^T Gnum, sum scale q');
//   3. bwd_reverse_kernel, one CTA per (document, head, segment), chunks in reverse: the suffix
//      state from the later segments' increments, dk', dv, dk and the gain partials of k;
//   4. bwd_gain_kernel (+ bwd_gain_final where the partials are many): the gain partials summed in a
//      fixed order.
// No float atomics anywhere: every sum has a fixed order, so results are bitwise repeatable.
#include "feature_bwd.cuh"
#include "kernels.h"
#include "simt_tiles.cuh"
#include "tc_features.cuh"

namespace rapt {
namespace {

using feat::doc_bounds;
using namespace simt;

constexpr int kC = 32;  // chunk length (tokens)
constexpr int kThreads = 256;
constexpr int kSMs = 152;

// Shared-memory layout in floats. Row strides are padded by 4 floats: float4 alignment is kept and
// rows r, r+1, ..., r+7 start in eight different 4-bank groups (LD / 4 = D / 4 + 1 is odd).
template <int D>
struct BwdSmem {
  static constexpr int LD = D + 4;
  static constexpr int LC = kC + 4;
  static constexpr int ST = 0;                  // [D][LD] carried state: S (launch 2) or R (launch 3)
  static constexpr int RT = ST + D * LD;        // [D][LD] launch 2: the segment's increment of R
  static constexpr int QF = RT + D * LD;        // [C][LD] q' (launch 2: later dq')
  static constexpr int KF = QF + kC * LD;       // [C][LD] k' (launch 3: later dk')
  static constexpr int VS = KF + kC * LD;       // [C][LD] v
  static constexpr int GS = VS + kC * LD;       // [C][LD] g, then gnum = g / den
  static constexpr int PS = GS + kC * LD;       // [C][LC] masked scores P[t][tau]
  static constexpr int AS = PS + kC * LC;       // [C][LC] g_t . v_tau, then A[t][tau] (masked)
  static constexpr int ZS = AS + kC * LC;       // [D] z (launch 2) or w (launch 3)
  static constexpr int WS = ZS + D;             // [D] launch 2: the segment's increment of w
  static constexpr int DEN = WS + D;            // [C] den_t
  static constexpr int SCL = DEN + kC;          // [C] scale_t
  static constexpr int SST = SCL + kC;          // [C] q'_t . z of the state before the chunk
  static constexpr int NST = SST + kC;          // [C] g_t . (q'_t S) of the state before the chunk
  static constexpr int total = NST + kC;
  static constexpr size_t bytes = static_cast<size_t>(total) * sizeof(float);
  static_assert(bytes <= 232448, "shared memory budget");
  static_assert(PS + (kThreads / FeatureLayout<D>::TPR) * D <= ZS, "gain partials fit in PS + AS");
};

// Features of C rows starting at token t0 of the document into a [C][LD] tile (tail rows zero).
template <int D, typename T>
__device__ __forceinline__ void feature_tile(const T* x, long row0, int n, int t0, int H, int h,
                                             const float* gamma, int pos0, const FeatureArgs& fa,
                                             float* tile) {
  using FL = FeatureLayout<D>;
  constexpr int LD = BwdSmem<D>::LD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / FL::TPR, r = lane % FL::TPR;
  constexpr int kRowsPerPass = (kThreads / 32) * FL::ROWS_PER_WARP;
  for (int rr = warp * FL::ROWS_PER_WARP + grp; rr < kC; rr += kRowsPerPass) {
    const int t = t0 + rr;
    const bool valid = t < n;
    float f[FL::EPT];
    feature_row<D, T>(x + ((row0 + (valid ? t : 0)) * H + h) * D, valid, gamma, pos0 + t, fa, r, f);
#pragma unroll
    for (int e = 0; e < FL::EPT; ++e) tile[rr * LD + r * FL::EPT + e] = f[e];
  }
}

// Raw rows (v or g) of C tokens into a [C][LD] tile as fp32 (tail rows zero).
template <int D, typename T>
__device__ __forceinline__ void raw_tile(const T* x, long row0, int n, int t0, int H, int h,
                                         float* tile) {
  constexpr int LD = BwdSmem<D>::LD;
  for (int idx = threadIdx.x; idx < kC * (D / 4); idx += kThreads) {
    const int rr = idx / (D / 4), j4 = 4 * (idx % (D / 4));
    float f4[4] = {0.f, 0.f, 0.f, 0.f};
    if (t0 + rr < n) RowLoad<T, 4>::run(x + ((row0 + t0 + rr) * H + h) * D + j4, f4);
    *reinterpret_cast<float4*>(tile + rr * LD + j4) = make_float4(f4[0], f4[1], f4[2], f4[3]);
  }
}

// Gain partials of one CTA: each thread's dg (its EPT elements) summed over the feature groups in
// a fixed order into out[D]. scratch: kThreads / TPR * D floats of shared memory.
template <int D>
__device__ __forceinline__ void store_gain_partial(const float (&dg)[FeatureLayout<D>::EPT],
                                                   float* scratch, float* out) {
  using FL = FeatureLayout<D>;
  constexpr int G = kThreads / FL::TPR;
  const int grp = threadIdx.x / FL::TPR, r = threadIdx.x % FL::TPR;
#pragma unroll
  for (int e = 0; e < FL::EPT; ++e) scratch[grp * D + r * FL::EPT + e] = dg[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += scratch[g * D + threadIdx.x];
    out[threadIdx.x] = s;
  }
}

// P[t][tau] = q'_t . k'_tau (masked to tau <= t) into Ps, and c[t][tau] = g_t . v_tau into As (Gs
// still holds the raw g). Warps 0-1 take P, warps 2-3 take c. Ends with a barrier.
template <int D>
__device__ __forceinline__ void score_tiles(const float* Qf, const float* Kf, const float* Vs,
                                            const float* Gs, float* Ps, float* As) {
  constexpr int LD = BwdSmem<D>::LD, LC = BwdSmem<D>::LC;
  const int tid = threadIdx.x;
  if (tid < 128) {
    const bool p = tid < 64;
    const int task = tid & 63, m0 = 4 * (task / 8), nb = task % 8;
    float acc[4][4] = {};
    mt_dot<8>(acc, (p ? Qf : Gs) + m0 * LD, LD, (p ? Kf : Vs) + nb * LD, LD, D);
    float* out = p ? Ps : As;
#pragma unroll
    for (int y = 0; y < 4; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int t = m0 + y, tau = nb + 8 * x;
        out[t * LC + tau] = (!p || tau <= t) ? acc[y][x] : 0.f;
      }
  }
  __syncthreads();
}

// A[t][tau] = gnum_t . v_tau + scale_t for tau <= t (0 above the diagonal), in the form whose
// cancelling part is exact (see the file comment), written over c in As; and gnum = g / den over
// Gs. Needs Ps, As = c, Den, Sst, Nst. Ends with a barrier.
template <int D>
__device__ __forceinline__ void build_a(const float* Ps, float* As, float* Gs, const float* Den,
                                        const float* Sst, const float* Nst, float eps) {
  constexpr int LD = BwdSmem<D>::LD, LC = BwdSmem<D>::LC;
  static_assert(kThreads * 4 == kC * kC, "four elements of A per thread");
  const int tid = threadIdx.x;
  const int t = tid / 8, tau0 = 4 * (tid % 8);
  const float den = Den[t];
  const float inv2 = 1.0f / (den * den);
  const float sst = Sst[t], nst = Nst[t];
  float av[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int tau = tau0 + u;
    float r = 0.f;
    if (tau <= t) {
      const float c = As[t * LC + tau];
      float acc = 0.f;
      for (int sg = 0; sg <= t; ++sg) acc = fmaf(Ps[t * LC + sg], c - As[t * LC + sg], acc);
      r = (acc + fmaf(c, sst, -nst) + eps * c) * inv2;
    }
    av[u] = r;
  }
  for (int idx = tid; idx < kC * D; idx += kThreads) {
    const int tt = idx / D;
    Gs[tt * LD + idx % D] = Gs[tt * LD + idx % D] / Den[tt];
  }
  __syncthreads();
  *reinterpret_cast<float4*>(As + t * LC + tau0) = make_float4(av[0], av[1], av[2], av[3]);
  __syncthreads();
}

// ------------------------------------------------------------------------------------------------
// Launch 1: K'^T V and sum k' of every segment that another segment of its document follows.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_state_kernel(const BwdArgs b) {
  using SM = BwdSmem<D>;
  constexpr int LD = SM::LD, NQ = D / 4;
  extern __shared__ __align__(16) float sm[];
  float* St = sm + SM::ST;
  float* Kf = sm + SM::KF;
  float* Vs = sm + SM::VS;
  float* Zs = sm + SM::ZS;
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x;
  const int seg = blockIdx.x % b.nseg, unit = blockIdx.x / b.nseg;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  if (s1 >= n) return;  // the document's last (or an empty) segment: nobody reads its increment
  for (int idx = tid; idx < D * D; idx += kThreads) St[(idx / D) * LD + idx % D] = 0.f;
  if (tid < D) Zs[tid] = 0.f;
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const float* gk = a.gamma_k + h * a.fa.gamma_stride;
  for (int t0 = s0; t0 < s1; t0 += kC) {
    __syncthreads();  // the previous chunk's reads of Kf / Vs are done
    feature_tile<D, T>(k, row0, n, t0, a.H, h, gk, a.pos_offset, a.fa, Kf);
    raw_tile<D, T>(v, row0, n, t0, a.H, h, Vs);
    __syncthreads();
    for (int task = tid; task < NQ * NQ; task += kThreads) {
      const int i0 = 4 * (task / NQ), j0 = 4 * (task % NQ);
      float acc[4][4] = {};
      mt_tn<1>(acc, Kf + i0, LD, Vs + j0, LD, kC);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) St[(i0 + y) * LD + j0 + x] += acc[y][x];
    }
    if (tid < D) {
      float s = 0.f;
      for (int t = 0; t < kC; ++t) s += Kf[t * LD + tid];
      Zs[tid] += s;
    }
  }
  __syncthreads();
  float* rec = b.rec_fwd + (static_cast<long>(unit) * b.nseg + seg) * (D * D + D);
  for (int idx = tid; idx < D * D; idx += kThreads) rec[idx] = St[(idx / D) * LD + idx % D];
  if (tid < D) rec[D * D + tid] = Zs[tid];
}

// ------------------------------------------------------------------------------------------------
// Launch 2: chunks in order. den, scale, gnum; dq' = A K' + S gnum + scale z, then dq; the
// segment's increment of the suffix state.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_forward_kernel(const BwdArgs b) {
  using SM = BwdSmem<D>;
  using FL = FeatureLayout<D>;
  constexpr int LD = SM::LD, LC = SM::LC, NQ = D / 4;
  extern __shared__ __align__(16) float sm[];
  float* St = sm + SM::ST;
  float* Rt = sm + SM::RT;
  float* Qf = sm + SM::QF;
  float* Kf = sm + SM::KF;
  float* Vs = sm + SM::VS;
  float* Gs = sm + SM::GS;
  float* Ps = sm + SM::PS;
  float* As = sm + SM::AS;
  float* Zs = sm + SM::ZS;
  float* Ws = sm + SM::WS;
  float* Den = sm + SM::DEN;
  float* Scl = sm + SM::SCL;
  float* Sst = sm + SM::SST;
  float* Nst = sm + SM::NST;
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % b.nseg, unit = blockIdx.x / b.nseg;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  if (!doc_bounds(a, doc, row0, n) && seg == 0 && h == 0 && tid == 0 && a.dev_status != nullptr)
    atomicOr(a.dev_status, 1u);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  const long rec = static_cast<long>(D) * D + D;
  const float* rf = b.rec_fwd + static_cast<long>(unit) * b.nseg * rec;
  // the prefix state at the segment's start: the earlier segments' increments, in order
  for (int idx = tid; idx < D * D; idx += kThreads) {
    float s = 0.f;
    for (int sp = 0; sp < seg && s0 < n; ++sp) s += rf[sp * rec + idx];
    St[(idx / D) * LD + idx % D] = s;
    Rt[(idx / D) * LD + idx % D] = 0.f;
  }
  if (tid < D) {
    float s = 0.f;
    for (int sp = 0; sp < seg && s0 < n; ++sp) s += rf[sp * rec + D * D + tid];
    Zs[tid] = s;
    Ws[tid] = 0.f;
  }
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* g = static_cast<const T*>(b.dout);
  T* dq = static_cast<T*>(b.dq);
  const float* gq = a.gamma_q + h * a.fa.gamma_stride;
  const float* gk = a.gamma_k + h * a.fa.gamma_stride;
  float dg[FL::EPT] = {};
  const int grp = lane / FL::TPR, r = lane % FL::TPR;
  constexpr int kRowsPerPass = (kThreads / 32) * FL::ROWS_PER_WARP;

  for (int t0 = s0; t0 < s1; t0 += kC) {
    __syncthreads();  // the previous chunk is done with every tile (and the initial state is set)
    feature_tile<D, T>(q, row0, n, t0, a.H, h, gq, a.pos_offset, a.fa, Qf);
    feature_tile<D, T>(k, row0, n, t0, a.H, h, gk, a.pos_offset, a.fa, Kf);
    raw_tile<D, T>(v, row0, n, t0, a.H, h, Vs);
    raw_tile<D, T>(g, row0, n, t0, a.H, h, Gs);
    __syncthreads();
    score_tiles<D>(Qf, Kf, Vs, Gs, Ps, As);
    // nst_t = g_t . (q'_t S): the state's part of g . num (the numerator itself is never stored)
    if (tid < 8 * NQ) {
      const int m0 = 4 * (tid / NQ), n0 = 4 * (tid % NQ);
      float acc[4][4] = {};
      mt_outer<1>(acc, Qf + m0 * LD, LD, St + n0, LD, D);
      float part[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const float4 gg = ld4(Gs + (m0 + y) * LD + n0);
        part[y] = acc[y][0] * gg.x + acc[y][1] * gg.y + acc[y][2] * gg.z + acc[y][3] * gg.w;
      }
#pragma unroll
      for (int off = NQ / 2; off > 0; off >>= 1)
#pragma unroll
        for (int y = 0; y < 4; ++y) part[y] += __shfl_xor_sync(0xffffffffu, part[y], off);
      if (tid % NQ == 0)
#pragma unroll
        for (int y = 0; y < 4; ++y) Nst[m0 + y] = part[y];
    }
    __syncthreads();
    // den_t = q'_t . z + sum_tau P[t][tau] + eps;  scale_t = -(g_t . num_t) / den_t^2
    if (tid < kC) {
      const int t = tid;
      const bool valid = t0 + t < n;
      float sst = 0.f;
      for (int i = 0; i < D; ++i) sst = fmaf(Qf[t * LD + i], Zs[i], sst);
      float ps = 0.f, pc = 0.f;
      for (int tau = 0; tau < kC; ++tau) {
        ps += Ps[t * LC + tau];
        pc = fmaf(Ps[t * LC + tau], As[t * LC + tau], pc);
      }
      const float den = valid ? sst + ps + a.eps_den : 1.f;
      const float scale = valid ? -(Nst[t] + pc) / (den * den) : 0.f;
      Den[t] = den;
      Scl[t] = scale;
      Sst[t] = sst;
      if (valid) {
        const long o = (row0 + t0 + t) * a.H + h;
        b.den[o] = den;
        b.scl[o] = scale;
        b.sst[o] = sst;
        b.nst[o] = Nst[t];
      }
    }
    __syncthreads();
    build_a<D>(Ps, As, Gs, Den, Sst, Nst, a.eps_den);
    // dq'[t][i] = sum_tau A[t][tau] k'_tau[i] + sum_j gnum_t[j] S[i][j] + scale_t z[i]  (columns
    // i = nb + NQ x), kept in registers; the segment's increments R += Q'^T Gnum, w += sum scale q'
    const bool has_dq = tid < 8 * NQ;
    const int m0q = 4 * (tid / NQ), nbq = tid % NQ;
    float dqa[4][4] = {};
    if (has_dq) {
      mt_outer<NQ>(dqa, As + m0q * LC, LC, Kf + nbq, LD, kC);
      mt_dot<NQ>(dqa, Gs + m0q * LD, LD, St + nbq * LD, LD, D);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) dqa[y][x] = fmaf(Scl[m0q + y], Zs[nbq + NQ * x], dqa[y][x]);
    }
    for (int task = tid; task < NQ * NQ; task += kThreads) {
      const int i0 = 4 * (task / NQ), j0 = 4 * (task % NQ);
      float acc[4][4] = {};
      mt_tn<1>(acc, Qf + i0, LD, Gs + j0, LD, kC);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) Rt[(i0 + y) * LD + j0 + x] += acc[y][x];
    }
    if (tid < D) {
      float w = 0.f;
      for (int t = 0; t < kC; ++t) w = fmaf(Scl[t], Qf[t * LD + tid], w);
      Ws[tid] += w;
    }
    __syncthreads();
    // dq' over q' (no longer needed); then the prefix state takes this chunk
    if (has_dq)
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) Qf[(m0q + y) * LD + nbq + NQ * x] = dqa[y][x];
    for (int task = tid; task < NQ * NQ; task += kThreads) {
      const int i0 = 4 * (task / NQ), j0 = 4 * (task % NQ);
      float acc[4][4] = {};
      mt_tn<1>(acc, Kf + i0, LD, Vs + j0, LD, kC);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) St[(i0 + y) * LD + j0 + x] += acc[y][x];
    }
    if (tid < D) {
      float s = 0.f;
      for (int t = 0; t < kC; ++t) s += Kf[t * LD + tid];
      Zs[tid] += s;
    }
    __syncthreads();
    // back through the features of q
    for (int rr = warp * FL::ROWS_PER_WARP + grp; rr < kC; rr += kRowsPerPass) {
      const int t = t0 + rr;
      const bool valid = t < n;
      const long off = ((row0 + (valid ? t : 0)) * a.H + h) * D;
      feature_row_bwd<D, T>(q + off, valid, gq, a.pos_offset + t, a.fa, r, Qf + rr * LD, dq + off, dg);
    }
  }
  __syncthreads();
  if (seg > 0 && s0 < n) {  // the suffix-state increment this segment hands to earlier ones
    float* rr = b.rec_rev + (static_cast<long>(unit) * b.nseg + seg) * rec;
    for (int idx = tid; idx < D * D; idx += kThreads) rr[idx] = Rt[(idx / D) * LD + idx % D];
    if (tid < D) rr[D * D + tid] = Ws[tid];
  }
  store_gain_partial<D>(dg, Ps, b.dgp_q + (static_cast<long>(unit) * b.nseg + seg) * D);
}

// ------------------------------------------------------------------------------------------------
// Launch 3: chunks in reverse. dv = P^T Gnum + K' R, dk' = A^T Q' + V R^T + w, then dk.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_reverse_kernel(const BwdArgs b) {
  using SM = BwdSmem<D>;
  using FL = FeatureLayout<D>;
  constexpr int LD = SM::LD, LC = SM::LC, NQ = D / 4;
  extern __shared__ __align__(16) float sm[];
  float* St = sm + SM::ST;  // R
  float* Qf = sm + SM::QF;
  float* Kf = sm + SM::KF;
  float* Vs = sm + SM::VS;
  float* Gs = sm + SM::GS;
  float* Ps = sm + SM::PS;
  float* As = sm + SM::AS;
  float* Zs = sm + SM::ZS;  // w
  float* Den = sm + SM::DEN;
  float* Scl = sm + SM::SCL;
  float* Sst = sm + SM::SST;
  float* Nst = sm + SM::NST;
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % b.nseg, unit = blockIdx.x / b.nseg;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  const long rec = static_cast<long>(D) * D + D;
  const float* rr = b.rec_rev + static_cast<long>(unit) * b.nseg * rec;
  // the suffix state at the segment's end: the later segments' increments, in segment order
  for (int idx = tid; idx < D * D; idx += kThreads) {
    float s = 0.f;
    for (int sp = seg + 1; sp < b.nseg && sp * b.seg_len < n; ++sp) s += rr[sp * rec + idx];
    St[(idx / D) * LD + idx % D] = s;
  }
  if (tid < D) {
    float s = 0.f;
    for (int sp = seg + 1; sp < b.nseg && sp * b.seg_len < n; ++sp) s += rr[sp * rec + D * D + tid];
    Zs[tid] = s;
  }
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* g = static_cast<const T*>(b.dout);
  T* dk = static_cast<T*>(b.dk);
  T* dv = static_cast<T*>(b.dv);
  const float* gq = a.gamma_q + h * a.fa.gamma_stride;
  const float* gk = a.gamma_k + h * a.fa.gamma_stride;
  float dg[FL::EPT] = {};
  const int grp = lane / FL::TPR, r = lane % FL::TPR;
  constexpr int kRowsPerPass = (kThreads / 32) * FL::ROWS_PER_WARP;
  const int nch = s1 > s0 ? (s1 - s0 + kC - 1) / kC : 0;

  for (int c = nch - 1; c >= 0; --c) {
    const int t0 = s0 + c * kC;
    __syncthreads();
    feature_tile<D, T>(q, row0, n, t0, a.H, h, gq, a.pos_offset, a.fa, Qf);
    feature_tile<D, T>(k, row0, n, t0, a.H, h, gk, a.pos_offset, a.fa, Kf);
    raw_tile<D, T>(v, row0, n, t0, a.H, h, Vs);
    raw_tile<D, T>(g, row0, n, t0, a.H, h, Gs);
    if (tid < kC) {
      const bool valid = t0 + tid < n;
      const long o = (row0 + t0 + tid) * a.H + h;
      Den[tid] = valid ? b.den[o] : 1.f;
      Scl[tid] = valid ? b.scl[o] : 0.f;
      Sst[tid] = valid ? b.sst[o] : 0.f;
      Nst[tid] = valid ? b.nst[o] : 0.f;
    }
    __syncthreads();
    score_tiles<D>(Qf, Kf, Vs, Gs, Ps, As);
    build_a<D>(Ps, As, Gs, Den, Sst, Nst, a.eps_den);
    // rows tau = m0 .. m0+3 of dv (columns n0 .. n0+3) and of dk' (columns nb + NQ x)
    const bool has = tid < 8 * NQ;
    const int m0 = 4 * (tid / NQ), nb = tid % NQ;
    float dka[4][4] = {};
    if (has) {
      float acc[4][4] = {};
      mt_tn<1>(acc, Ps + m0, LC, Gs + 4 * nb, LD, kC);
      mt_outer<1>(acc, Kf + m0 * LD, LD, St + 4 * nb, LD, D);
#pragma unroll
      for (int y = 0; y < 4; ++y)
        if (t0 + m0 + y < n)
          store4(dv + ((row0 + t0 + m0 + y) * a.H + h) * D + 4 * nb, acc[y][0], acc[y][1],
                 acc[y][2], acc[y][3]);
      mt_tn<NQ>(dka, As + m0, LC, Qf + nb, LD, kC);
      mt_dot<NQ>(dka, Vs + m0 * LD, LD, St + nb * LD, LD, D);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) dka[y][x] += Zs[nb + NQ * x];
    }
    __syncthreads();
    // dk' over k'; then the suffix state takes this chunk
    if (has)
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) Kf[(m0 + y) * LD + nb + NQ * x] = dka[y][x];
    for (int task = tid; task < NQ * NQ; task += kThreads) {
      const int i0 = 4 * (task / NQ), j0 = 4 * (task % NQ);
      float acc[4][4] = {};
      mt_tn<1>(acc, Qf + i0, LD, Gs + j0, LD, kC);
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) St[(i0 + y) * LD + j0 + x] += acc[y][x];
    }
    if (tid < D) {
      float w = 0.f;
      for (int t = 0; t < kC; ++t) w = fmaf(Scl[t], Qf[t * LD + tid], w);
      Zs[tid] += w;
    }
    __syncthreads();
    for (int rw = warp * FL::ROWS_PER_WARP + grp; rw < kC; rw += kRowsPerPass) {
      const int t = t0 + rw;
      const bool valid = t < n;
      const long off = ((row0 + (valid ? t : 0)) * a.H + h) * D;
      feature_row_bwd<D, T>(k + off, valid, gk, a.pos_offset + t, a.fa, r, Kf + rw * LD, dk + off, dg);
    }
  }
  __syncthreads();
  store_gain_partial<D>(dg, Ps, b.dgp_k + (static_cast<long>(unit) * b.nseg + seg) * D);
}

// ------------------------------------------------------------------------------------------------
// Launch 4: gains. dgamma[h][c] (or dgamma[c] when shared) = the partials of every (document,
// segment) (and head, when shared). One CTA of 8 warps per 32 outputs (lane = output): warp w
// sums the items w, w + 8, ... of the (document, [head,] segment) list in order, then the eight
// warp sums are added in warp order, so the result is bitwise repeatable. blockIdx.y: 0 = q, 1 = k.
// Sums the gain partials (item = (document * nh + head offset) * nseg + segment, D values each) of
// items [it0, it1), it0 = blockIdx.z * per_split, for 32 output elements per CTA (blockIdx.y: 0 = q,
// 1 = k), warp w taking items it0 + w, it0 + w + 8, ... and the warps added in order. With a
// scratch buffer the CTA's sum is the first of two stages and goes to
// scratch[(y * gridDim.z + z) * n_out + e]; without one it is the gain's gradient.
__global__ void __launch_bounds__(256)
    bwd_gain_kernel(const BwdArgs b, int D, int per_split, float* scratch) {
  const PrefillArgs& a = b.p;
  const bool per_head = a.fa.gamma_stride != 0;
  const int n_out = per_head ? a.H * D : D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  const float* part = blockIdx.y == 0 ? b.dgp_q : b.dgp_k;
  float* out = blockIdx.y == 0 ? b.dgamma_q : b.dgamma_k;
  if (out == nullptr) return;  // uniform
  __shared__ float ws[8][32];
  float s = 0.f;
  if (e < n_out) {
    const int c = e % D;
    const int nh = per_head ? 1 : a.H;        // heads per output
    const int h0 = per_head ? e / D : 0;
    const int items = a.n_docs * nh * b.nseg;
    const int it0 = blockIdx.z * per_split, it1 = min(items, it0 + per_split);
    // walked with counters (one division at the start, none in the loop)
    int seg = (it0 + warp) % b.nseg, dh = (it0 + warp) / b.nseg;
    const int dseg = 8 % b.nseg, ddh = 8 / b.nseg;
#pragma unroll 4
    for (int it = it0 + warp; it < it1; it += 8) {  // (unrolled: the loads are issued ahead of the adds)
      const int doc = dh / nh, h = h0 + dh % nh;
      s += __ldg(part + ((static_cast<long>(doc) * a.H + h) * b.nseg + seg) * D + c);
      seg += dseg;
      dh += ddh;
      if (seg >= b.nseg) {
        seg -= b.nseg;
        ++dh;
      }
    }
  }
  ws[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < n_out) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += ws[w][lane];
    if (scratch != nullptr) scratch[(static_cast<long>(blockIdx.y) * gridDim.z + blockIdx.z) * n_out + e] = t;
    else out[e] = t;
  }
}

// Second stage: the splits' sums of every output element added in split order.
__global__ void __launch_bounds__(256) bwd_gain_final(const BwdArgs b, int n_out, int splits,
                                                      const float* scratch) {
  const int e = blockIdx.x * 256 + threadIdx.x;
  float* out = blockIdx.y == 0 ? b.dgamma_q : b.dgamma_k;
  if (out == nullptr || e >= n_out) return;
  const float* p = scratch + static_cast<long>(blockIdx.y) * splits * n_out + e;
  float t = 0.f;
  for (int g = 0; g < splits; ++g) t += p[static_cast<long>(g) * n_out];
  out[e] = t;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

template <typename T, int D>
cudaError_t launch_t(const BwdArgs& b, cudaStream_t stream) {
  constexpr size_t smem = BwdSmem<D>::bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    if ((e = set_smem(bwd_state_kernel<T, D>, smem)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_forward_kernel<T, D>, smem)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_reverse_kernel<T, D>, smem)) != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long grid = static_cast<long>(b.p.n_docs) * b.p.H * b.nseg;
  if (grid == 0) return cudaSuccess;
  if (b.nseg > 1) {
    bwd_state_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(b);
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  bwd_forward_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(b);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_reverse_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(b);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_bwd_gain(b, D, stream);
}

template <typename T>
cudaError_t launch_d(int d, const BwdArgs& b, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_t<T, 16>(b, stream);
    case 32: return launch_t<T, 32>(b, stream);
    case 64: return launch_t<T, 64>(b, stream);
    case 128: return launch_t<T, 128>(b, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

BwdPlan bwd_plan(int n_docs, int H, int max_seqlen, long total_rows, int d, bool tc) {
  // One CTA per SM (the kernels take most of the shared memory). A document is cut into nseg
  // segments of seg_len tokens (a multiple of the chunk: 32 tokens on the CUDA cores, 128 on the
  // tensor cores); the cost of a plan is its waves of kSMs CTAs times the chunks of a segment
  // (plus one chunk of set-up per wave).
  BwdPlan p{};
  const int ck = tc ? 128 : kC;
  const int chunks_max = max_seqlen > 0 ? (max_seqlen + ck - 1) / ck : 1;
  const long units = static_cast<long>(n_docs) * H;
  double best = 1e300;
  for (int nseg = 1; nseg <= 64 && nseg <= chunks_max; ++nseg) {
    const int seg_chunks = (chunks_max + nseg - 1) / nseg;
    const long ctas = units * nseg;
    const double waves = static_cast<double>((ctas + kSMs - 1) / kSMs);
    const double cost = waves * (seg_chunks + 1.0);
    if (cost < 0.95 * best) {
      best = cost;
      p.nseg = nseg;
      p.seg_len = seg_chunks * ck;
    }
  }
  if (p.nseg == 0) {
    p.nseg = 1;
    p.seg_len = chunks_max * ck;
  }
  p.blk_per_seg = 1;
  if (tc && p.nseg > 1) {  // prefix-state blocks: the earlier segments' blocks should fill one wave
    const int sc = p.seg_len / ck;
    for (int f = 8; f > 1; f /= 2)
      if (sc % f == 0 && units * (p.nseg - 1) * f <= kSMs) {
        p.blk_per_seg = f;
        break;
      }
  }
  // suffix-state blocks: the later segments' blocks should fill one wave of CTAs
  p.rblk_per_seg = 1;
  if (tc && p.nseg > 1) {
    const int sc = p.seg_len / ck;
    for (int f = 8; f > 1; f /= 2)
      if (sc % f == 0 && units * (p.nseg - 1) * f <= kSMs) {
        p.rblk_per_seg = f;
        break;
      }
  }
  p.nblk_max = (p.nseg - 1) * p.blk_per_seg;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const int dr = tc ? 128 : d;  // the tensor-core records keep the 128 x 128 layout at d = 64
  const size_t rec = static_cast<size_t>(dr) * (dr + 1) * sizeof(float);
  const size_t recs_f = up(static_cast<size_t>(units) * (tc ? p.nblk_max : p.nseg) * rec);
  const size_t recs_r = up(static_cast<size_t>(units) * p.nseg * p.rblk_per_seg * rec);
  const size_t rows = up(static_cast<size_t>(total_rows) * H * sizeof(float));
  const size_t feats = tc ? up(static_cast<size_t>(total_rows) * H * d * 2) : 0;
  p.chunks_max = tc ? chunks_max : 0;
  const size_t gp = up(static_cast<size_t>(units) * (tc ? chunks_max : p.nseg) * d * sizeof(float));
  p.off_rev = recs_f;
  p.off_den = p.off_rev + recs_r;
  p.off_scl = p.off_den + rows;
  p.off_sst = p.off_scl + rows;
  p.off_nst = p.off_sst + rows;
  p.off_qf = p.off_nst + rows;
  p.off_kf = p.off_qf + feats;
  p.off_dqf = p.off_kf + feats;
  p.off_dkf = p.off_dqf + feats;
  p.off_dgq = p.off_dkf + feats;
  p.off_dgk = p.off_dgq + gp;
  p.off_order = p.off_dgk + gp;
  p.ws_bytes = p.off_order + (tc ? up(static_cast<size_t>(n_docs) * sizeof(int)) : 0);
  return p;
}

cudaError_t launch_bwd_gain(const BwdArgs& b, int d, cudaStream_t stream) {
  if (b.dgamma_q == nullptr && b.dgamma_k == nullptr) return cudaSuccess;
  const bool per_head = b.p.fa.gamma_stride != 0;
  const int n_out = per_head ? b.p.H * d : d;
  const long items = static_cast<long>(b.p.n_docs) * (per_head ? 1 : b.p.H) * b.nseg;
  const unsigned gx = static_cast<unsigned>((n_out + 31) / 32);
  // Many items per output element (gains shared by the heads of many documents and chunks): the
  // items are cut into splits summed by separate CTAs, then the splits are added in order. The
  // splits' sums go to the per-row den region of the workspace, which the passes no longer need.
  const long room = static_cast<long>(b.p.total_rows) * b.p.H / (2L * n_out);
  long splits = items > 512 ? (items + 255) / 256 : 1;
  splits = splits > 128 ? 128 : splits;
  splits = splits > room ? room : splits;
  if (splits <= 1) {
    bwd_gain_kernel<<<dim3(gx, 2, 1), 256, 0, stream>>>(b, d, static_cast<int>(items), nullptr);
    note_launches(1);
    return cudaGetLastError();
  }
  const int per_split = static_cast<int>((items + splits - 1) / splits);
  bwd_gain_kernel<<<dim3(gx, 2, static_cast<unsigned>(splits)), 256, 0, stream>>>(b, d, per_split, b.den);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_gain_final<<<dim3(static_cast<unsigned>((n_out + 255) / 256), 2), 256, 0, stream>>>(
      b, n_out, static_cast<int>(splits), b.den);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_backward_simt(DType dt, int d, const BwdArgs& b, cudaStream_t stream) {
  return dt == DType::F32 ? launch_d<float>(d, b, stream) : launch_d<__nv_bfloat16>(d, b, stream);
}

}  // namespace rapt
