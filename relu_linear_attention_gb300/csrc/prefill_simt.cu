// Chunked causal RLA-2 forward on CUDA cores (fp32 FFMA), sm_103a.
//
// This is the fp32-input path (its tolerance, 1e-4 relative, is below what bf16/tf32 tensor-core
// operands can deliver) and the reference GPU path for every dtype. It computes, per document
// and head (08-rapt-algorithm.md §3, chunk-parallel accumulation of the state):
//   for each chunk of C tokens:   P = (Q'_c K'_c^T) masked to tau <= t
//                                 num = P V_c + Q'_c S,   den = rowsum(P) + Q'_c z + eps
//                                 out = num / den
//                                 S += K'_c^T V_c,  z += colsum(K'_c)        (after the read)
// which equals the per-token recurrence S_t = S_{t-1} + k'_t v_t^T, out_t = q'_t S_t / (q'_t z_t
// + eps) exactly up to summation order. One CTA owns one (document, head, block of DVB value
// columns) and walks the document's chunks in order with S (d x DVB) and z resident in shared
// memory. Dense prefill is the same kernel with B documents of L tokens. The bidirectional form
// (08-rapt-algorithm.md §4.1, causal=false: every token sees its whole document) walks the chunks
// twice: first only the state update over the whole document, then num = Q'_c S, den = Q'_c z +
// eps for every chunk.
#include "kernels.h"

namespace rapt {
namespace {

constexpr int kC = 64;  // chunk length (tokens)
constexpr int kThreads = 256;

template <int D>
struct SimtCfg {
  static constexpr int DVB = D > 64 ? 64 : D;  // value columns per CTA
  static constexpr int NCB = D / DVB;          // column blocks per head
  static constexpr int CG = DVB / 4;           // float4 column groups
};

// Shared-memory layout, in floats (every offset is a multiple of 4 floats).
template <int D>
struct SimtSmem {
  static constexpr int DVB = SimtCfg<D>::DVB;
  static constexpr int QsT = 0;               // [D][C]   q' transposed
  static constexpr int KsT = QsT + D * kC;    // [D][C]   k' transposed (score GEMM)
  static constexpr int Ks = KsT + D * kC;     // [C][D]   k' (state update)
  static constexpr int Vs = Ks + kC * D;      // [C][DVB] value columns of this CTA
  static constexpr int Ss = Vs + kC * DVB;    // [D][DVB] state S (key-major)
  static constexpr int PsT = Ss + D * DVB;    // [C][C]   masked scores, PsT[tau][t]
  static constexpr int Zs = PsT + kC * kC;    // [D]      normaliser z
  static constexpr int Dens = Zs + D;         // [C]      denominators of the chunk
  static constexpr int total = Dens + kC;
  static constexpr size_t bytes = static_cast<size_t>(total) * sizeof(float);
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const PrefillArgs a) {
  using Cfg = SimtCfg<D>;
  using SM = SimtSmem<D>;
  using FL = FeatureLayout<D>;
  constexpr int DVB = Cfg::DVB;
  constexpr int NCB = Cfg::NCB;
  constexpr int CG = Cfg::CG;
  constexpr int EPT = FL::EPT;

  extern __shared__ __align__(16) float sm[];
  float* QsT = sm + SM::QsT;
  float* KsT = sm + SM::KsT;
  float* Ks = sm + SM::Ks;
  float* Vs = sm + SM::Vs;
  float* Ss = sm + SM::Ss;
  float* PsT = sm + SM::PsT;
  float* Zs = sm + SM::Zs;
  float* Dens = sm + SM::Dens;

  const int tid = threadIdx.x;
  const int cb = blockIdx.x % NCB;
  const int h = (blockIdx.x / NCB) % a.H;
  const int doc = blockIdx.x / (NCB * a.H);

  // Document bounds. Varlen bounds are validated on the device: a malformed document is
  // skipped (treated as empty) and reported, never read out of bounds.
  long row0 = 0;
  int n = 0;
  if (a.cu_seqlens != nullptr) {
    const int s = a.cu_seqlens[doc];
    const int e = a.cu_seqlens[doc + 1];
    const int prev = doc > 0 ? a.cu_seqlens[doc - 1] : 0;  // a decrease flags both neighbours
    const bool bad = s < 0 || e < s || prev > s || e > a.total_rows || (doc == 0 && s != 0) ||
                     (doc == a.n_docs - 1 && e != a.total_rows) || (e - s) > a.max_seqlen;
    if (bad) {
      if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 1u);
    } else {
      row0 = s;
      n = e - s;
    }
  } else {
    row0 = static_cast<long>(doc) * a.doc_len;
    n = a.doc_len;
  }

  const long bh = static_cast<long>(doc) * a.H + h;
  const float* gq = a.gamma_q + h * a.fa.gamma_stride;
  const float* gk = a.gamma_k + h * a.fa.gamma_stride;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  T* out = static_cast<T*>(a.out);

  for (int idx = tid; idx < D * DVB; idx += kThreads) {
    const int i = idx / DVB, j = idx % DVB;
    Ss[idx] = a.S0 != nullptr ? a.S0[(bh * D + i) * D + cb * DVB + j] : 0.f;
  }
  for (int i = tid; i < D; i += kThreads) Zs[i] = a.z0 != nullptr ? a.z0[bh * D + i] : 0.f;
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  const int grp = lane / FL::TPR, r = lane % FL::TPR;
  constexpr int kRowsPerPass = (kThreads / 32) * FL::ROWS_PER_WARP;
  static_assert(kC % kRowsPerPass == 0, "every lane must run the same number of feature rows");

  // Causal: one pass reads every chunk out and then adds it to the state. Bidirectional
  // (08-rapt-algorithm.md §4.1, causal=false): a first pass sums the whole document's state, a
  // second reads every chunk out against it (no intra-chunk scores). All flags are CTA-uniform.
  const bool causal = !a.bidir;
  for (int pass = 0; pass < (causal ? 1 : 2); ++pass) {
  const bool upd = causal || pass == 0;  // this pass adds the chunks to the state
  const bool rd = causal || pass == 1;   // this pass writes the output
  for (int t0 = 0; t0 < n; t0 += kC) {
    // ---- features of the chunk (tail rows become zeros: they add nothing anywhere)
    for (int rr = warp * FL::ROWS_PER_WARP + grp; rr < kC; rr += kRowsPerPass) {
      const int t = t0 + rr;
      const bool valid = t < n;
      const long off = ((row0 + (valid ? t : 0)) * a.H + h) * D;
      float f[EPT];
      if (rd) {
        feature_row<D, T>(q + off, valid, gq, a.pos_offset + t, a.fa, r, f);
#pragma unroll
        for (int e = 0; e < EPT; ++e) QsT[(r * EPT + e) * kC + rr] = f[e];
      }
      if (upd) {
        feature_row<D, T>(k + off, valid, gk, a.pos_offset + t, a.fa, r, f);
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          KsT[(r * EPT + e) * kC + rr] = f[e];
          Ks[rr * D + r * EPT + e] = f[e];
        }
      }
    }
    for (int idx = upd ? tid : kC * CG; idx < kC * CG; idx += kThreads) {
      const int rr = idx / CG, j4 = (idx % CG) * 4;
      const int t = t0 + rr;
      float f4[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < n) RowLoad<T, 4>::run(v + ((row0 + t) * a.H + h) * D + cb * DVB + j4, f4);
      *reinterpret_cast<float4*>(Vs + rr * DVB + j4) = make_float4(f4[0], f4[1], f4[2], f4[3]);
    }
    __syncthreads();

    // ---- masked scores P[t][tau] = q'_t . k'_tau for tau <= t (stored transposed)
    if (causal) {
      const int ty = tid / 16, tx = tid % 16;
      float acc[4][4] = {};
      for (int i = 0; i < D; ++i) {
        const float4 qa = ld4(QsT + i * kC + 4 * ty);
        const float4 kb = ld4(KsT + i * kC + 4 * tx);
        const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
        const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
          for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(qv[y], kv[x], acc[y][x]);
      }
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int t = 4 * ty + y, tau = 4 * tx + x;
          PsT[tau * kC + t] = tau <= t ? acc[y][x] : 0.f;
        }
    }
    __syncthreads();

    // ---- denominators and numerators (intra-chunk part + carried state)
    if (rd && tid < kC) {
      float s = 0.f;
      if (causal)
        for (int tau = 0; tau < kC; ++tau) s += PsT[tau * kC + tid];
      for (int i = 0; i < D; ++i) s = fmaf(QsT[i * kC + tid], Zs[i], s);
      Dens[tid] = s + a.eps_den;
    }
    const bool has_num = rd && tid < 16 * CG;
    const int ny = tid / CG, nx = tid % CG;
    float acc[4][4] = {};
    if (has_num) {
      for (int tau = 0; tau < (causal ? kC : 0); ++tau) {
        const float4 p = ld4(PsT + tau * kC + 4 * ny);
        const float4 w = ld4(Vs + tau * DVB + 4 * nx);
        const float pv[4] = {p.x, p.y, p.z, p.w};
        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
          for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(pv[y], wv[x], acc[y][x]);
      }
      for (int i = 0; i < D; ++i) {
        const float4 p = ld4(QsT + i * kC + 4 * ny);
        const float4 w = ld4(Ss + i * DVB + 4 * nx);
        const float pv[4] = {p.x, p.y, p.z, p.w};
        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
          for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(pv[y], wv[x], acc[y][x]);
      }
    }
    __syncthreads();  // Dens ready; every read of S and z for this chunk is done
    if (has_num) {
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int t = 4 * ny + y;
        if (t0 + t < n) {
          const float den = Dens[t];
          store4(out + ((row0 + t0 + t) * a.H + h) * D + cb * DVB + 4 * nx, acc[y][0] / den,
                 acc[y][1] / den, acc[y][2] / den, acc[y][3] / den);
        }
      }
    }

    // ---- state update S += K'^T V, z += colsum K'
    for (int blk = upd ? tid : (D / 4) * CG; blk < (D / 4) * CG; blk += kThreads) {
      const int bi = blk / CG, bj = blk % CG;
      float u[4][4] = {};
      for (int tau = 0; tau < kC; ++tau) {
        const float4 kk = ld4(Ks + tau * D + 4 * bi);
        const float4 w = ld4(Vs + tau * DVB + 4 * bj);
        const float kv[4] = {kk.x, kk.y, kk.z, kk.w};
        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
          for (int x = 0; x < 4; ++x) u[y][x] = fmaf(kv[y], wv[x], u[y][x]);
      }
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 4; ++x) Ss[(4 * bi + y) * DVB + 4 * bj + x] += u[y][x];
    }
    if (upd && tid < D) {
      float s = 0.f;
      for (int tau = 0; tau < kC; ++tau) s += Ks[tau * D + tid];
      Zs[tid] += s;
    }
    __syncthreads();
  }
  }

  if (a.S_final != nullptr && causal) {
    for (int idx = tid; idx < D * DVB; idx += kThreads) {
      const int i = idx / DVB, j = idx % DVB;
      a.S_final[(bh * D + i) * D + cb * DVB + j] = Ss[idx];
    }
  }
  if (a.z_final != nullptr && causal && cb == 0) {
    for (int i = tid; i < D; i += kThreads) a.z_final[bh * D + i] = Zs[i];
  }
}

template <typename T, int D>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t stream) {
  constexpr size_t smem = SimtSmem<D>::bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(prefill_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long grid = static_cast<long>(a.n_docs) * a.H * SimtCfg<D>::NCB;
  if (grid == 0) return cudaSuccess;
  prefill_simt_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_d(int d, const PrefillArgs& a, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_t<T, 16>(a, stream);
    case 32: return launch_t<T, 32>(a, stream);
    case 64: return launch_t<T, 64>(a, stream);
    case 128: return launch_t<T, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill_simt(DType dt, int d, const PrefillArgs& a, cudaStream_t stream) {
  return dt == DType::F32 ? launch_d<float>(d, a, stream) : launch_d<__nv_bfloat16>(d, a, stream);
}

}  // namespace rapt
