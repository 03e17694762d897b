// Causal original RLA (L2 denominator) on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a;
// bf16, d in {64, 128}, dense batch rows or packed documents, fp32 accumulation and fp32 states.
//
// 08-rapt-algorithm.md §2.1 (closed form, eps outside the root; q' = ReLU(q), k' = ReLU(k)), §2.2
// (a query reads the accumulated causal state, which restarts at every document), §4.1 (the
// scan's two prefix states):
//   S_t = sum_{i<=t} k'_i v_i^T,  A_t = sum_{i<=t} k'_i k'_i^T,
//   out_t = q'_t S_t / (sqrt(q'_t^T A_t q'_t) + eps).
// Chunked (C = 128 tokens), with P = Q'K'^T masked to tau <= t and S~, A~ bf16 copies of the fp32
// states before the chunk:
//   phase 2:  P = Q'K'^T,  X = Q' A~ (committed), then S += K'^T V,  A += K'^T K' (run during phase 3)
//   phase 3:  den_t = sqrt(sum_tau P^2 + q'_t . X_t) + eps (fp32; P from exact bf16 features),
//             P~ = P masked, in bf16
//   phase 4:  X = Q' S~ + P~ V
//   phase 5:  out = X / den; S, A -> S~, A~ for the next chunk.
// Dense batch rows may be cut into segments of seg_len tokens; segment s starts from the moments
// [K'^T V | K'^T K'] of the splits before it, computed by the non-causal L2 path's moments kernel
// with the same split length (summed in split order: deterministic), and is launched as a
// programmatic dependent of it (segment 0 needs no moments and starts at once). Packed documents
// run one CTA per (document, head), the longest documents first. d = 64 pads K'^T to M = 128 with a
// zero block (TMEM rows 64..127 of S and A stay zero). One CTA per (document, head, segment), 512
// threads in lockstep phases, one thread issuing the MMAs and the TMA copies: the next chunk's q, k,
// v tiles are requested as soon as the current chunk's last MMA has read its tiles, so they arrive
// while the chunk's output and state copies are written. Every wait is bounded (~1 s); a CTA whose
// wait gives up writes NaN over its rows.
#include <cuda.h>

#include "kernels.h"
#include "tc_features.cuh"
#include "tc_tiles.cuh"
#include "tc_utils.cuh"
#include "tensor_map.h"

namespace rapt {
namespace {

using feat::lds16;
using feat::sts16;
using namespace tct;

constexpr int kC = 128;
constexpr int kThreads = 512;

template <int D>
struct LayC {
  static constexpr uint32_t TILE = (D / 64) * 16384;  // 128 rows x D columns, bf16
  static constexpr uint32_t STILE = D * D * 2;        // a D x D state copy, bf16
  static constexpr uint32_t QF = 0, KF = TILE;        // k' (d = 64: + a zero block)
  static constexpr uint32_t VS = KF + 32768;
  static constexpr uint32_t SS = VS + TILE, AS = SS + STILE;
  static constexpr uint32_t PS = AS + STILE;          // P~, 128 x 128
  static constexpr uint32_t RED = PS + 32768;         // partial den^2 [4][128]
  static constexpr uint32_t BAR = RED + 4 * kC * 4;   // three mbarriers
  static constexpr uint32_t MISC = BAR + 24;          // TMEM base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(QF % 1024 == 0 && KF % 1024 == 0 && VS % 1024 == 0 && SS % 1024 == 0 &&
                AS % 1024 == 0 && PS % 1024 == 0, "tile alignment");
  // TMEM columns: P, X, S, A
  static constexpr uint32_t TP = 0, TX = 128, TS = 128 + D, TA = 128 + 2 * D;
  static_assert(TA + D <= 512, "TMEM budget");
};

// The chunk's raw q, k, v rows (rows t.. of the row-major [rows, H, D] tensors) into their tiles by
// TMA, D / 64 boxes each, completing on one mbarrier; one thread calls it. Rows past the tensor
// read as zero.
template <int D>
__device__ __forceinline__ void tma_qkv(const CUtensorMap* tq, const CUtensorMap* tk,
                                        const CUtensorMap* tv, uint32_t base, int h, int t,
                                        uint32_t bar) {
  using L = LayC<D>;
  tc::mbar_arrive_expect_tx(bar, 3 * L::TILE);
#pragma unroll
  for (int jb = 0; jb < D / 64; ++jb) {
    tc::tma_load_3d(base + L::QF + jb * 16384, tq, 64 * jb, h, t, bar);
    tc::tma_load_3d(base + L::KF + jb * 16384, tk, 64 * jb, h, t, bar);
    tc::tma_load_3d(base + L::VS + jb * 16384, tv, 64 * jb, h, t, bar);
  }
}

// In place: q and k tiles rectified (bf16 max(0, x) on the bit patterns: a set sign bit, negative
// or -0, becomes +0).
template <int D>
__device__ __forceinline__ void rectify_qk(uint32_t base) {
  using L = LayC<D>;
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  for (int idx = threadIdx.x; idx < 2 * kC * CPR; idx += kThreads) {
    const int r = (idx / CPR) & (kC - 1), m = idx % CPR;
    const uint32_t addr = base + (idx < kC * CPR ? L::QF : L::KF) + tile_off(r, m);
    uint4 v = lds16(addr);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t lo = (w[e] & 0x8000u) ? 0u : (w[e] & 0xFFFFu);
      const uint32_t hi = (w[e] & 0x80000000u) ? 0u : (w[e] & 0xFFFF0000u);
      w[e] = lo | hi;
    }
    sts16(addr, make_uint4(w[0], w[1], w[2], w[3]));
  }
}

// Bounds of document `doc` (dense: batch row doc); false if cu_seqlens is malformed there (the
// document is then skipped and reported).
__device__ __forceinline__ bool l2c_doc(const L2cTcArgs& a, int doc, long& row0, int& n) {
  if (a.cu_seqlens == nullptr) {
    row0 = static_cast<long>(doc) * a.doc_len;
    n = a.doc_len;
    return true;
  }
  const int s = a.cu_seqlens[doc], e = a.cu_seqlens[doc + 1];
  const int prev = doc > 0 ? a.cu_seqlens[doc - 1] : 0;
  const bool bad = s < 0 || e < s || prev > s || e > a.total_rows || (doc == 0 && s != 0) ||
                   (doc == a.n_docs - 1 && e != a.total_rows) || (e - s) > a.max_seqlen;
  row0 = bad ? 0 : s;
  n = bad ? 0 : e - s;
  return !bad;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    l2c_tc_kernel(const L2cTcArgs a, const __grid_constant__ CUtensorMap tq,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using L = LayC<D>;
  constexpr int NG = D / 32;  // 32-column groups of the D-wide products
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % a.nseg, unit = blockIdx.x / a.nseg;
  const int h = unit % a.H, slot = unit / a.H;
  const int doc = a.order != nullptr ? a.order[slot] : slot;
  long row0;
  int n;
  const bool good = l2c_doc(a, doc, row0, n);
  if (!good && seg == 0 && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 1u);
  const int s0 = seg * a.seg_len, s1 = min(n, s0 + a.seg_len);
  if (s0 >= s1) return;  // uniform, before any allocation
  const int nch = (s1 - s0 + kC - 1) / kC;
  const long bh = static_cast<long>(doc) * a.H + h;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  float* red = reinterpret_cast<float*>(smem + L::RED);
  const uint32_t bar1 = base + L::BAR, bar2 = bar1 + 8, bar_ld = bar1 + 16;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;
  if (warp == 0 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar1, 1);
    tc::mbar_init(bar2, 1);
    tc::mbar_init(bar_ld, 1);
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  if (D == 64 && !misaligned) {  // zero block that pads k'^T to M = 128 rows
    for (int i = tid; i < 16384 / 16; i += kThreads) sts16(base + L::KF + 16384 + i * 16, make_uint4(0, 0, 0, 0));
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int q4 = warp & 3, gw = warp >> 2;
  const int t = 32 * q4 + lane;  // tile row = TMEM lane
  const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
  bool bad = *s_abort != 0;

  // the first chunk's tiles do not depend on the moments launch
  int tma_issued = 0;  // chunks whose tiles have been requested (thread 0)
  if (tid == 0 && !bad) {
    tma_qkv<D>(&tq, &tk, &tv, base, h, static_cast<int>(row0 + s0), bar_ld);
    tma_issued = 1;
  }
  // the states at the segment's start: the moments of the earlier splits, in split order; rows and
  // columns past D (d = 64) are the zero padding of TMEM
  if (!bad && gw < NG) {
    float sv[32], av[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) sv[e] = av[e] = 0.f;
    if (seg > 0 && t < D) {
      tc::grid_dep_wait();
      const float4* part = reinterpret_cast<const float4*>(a.ws) +
                           bh * (a.nseg - 1) * (D * 2 * D / 4);
      for (int sp = 0; sp < seg; ++sp) {
        const float4* ps = part + static_cast<long>(sp) * (D * 2 * D / 4);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float4 x = __ldcg(ps + (8 * gw + jj) * D + t);
          const float4 y = __ldcg(ps + (D / 4 + 8 * gw + jj) * D + t);
          sv[4 * jj] += x.x; sv[4 * jj + 1] += x.y; sv[4 * jj + 2] += x.z; sv[4 * jj + 3] += x.w;
          av[4 * jj] += y.x; av[4 * jj + 1] += y.y; av[4 * jj + 2] += y.z; av[4 * jj + 3] += y.w;
        }
      }
    }
    if (t < D) {
      state_put(tmem + tl + L::TS + 32 * gw, base + L::SS, t, gw, sv);
      state_put(tmem + tl + L::TA + 32 * gw, base + L::AS, t, gw, av);
    } else {  // d = 64: zero TMEM rows 64..127 of S and A
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      tc::tmem_st16(tmem + tl + L::TS + 32 * gw, z);
      tc::tmem_st16(tmem + tl + L::TS + 32 * gw + 16, z);
      tc::tmem_st16(tmem + tl + L::TA + 32 * gw, z);
      tc::tmem_st16(tmem + tl + L::TA + 32 * gw + 16, z);
      tc::tmem_wait_st();
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  for (int c = 0; c < nch && !bad; ++c) {
    const int t0 = s0 + c * kC;
    // ---- phase 1: the chunk's q, k, v (TMA, requested one chunk ahead); q' = ReLU(q), k' = ReLU(k)
    if (!tc::mbar_wait(bar_ld, c & 1, kWait)) atomicExch(s_abort, 1);
    rectify_qk<D>(base);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- phase 2: P = Q'K'^T, X = Q'A~, S += K'^T V, A += K'^T K'
    if (tid == 0) {
      constexpr uint32_t ID_P = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_KM = tc::idesc_bf16(128, D, false, true);
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, D, true, true);
#pragma unroll 1
      for (int kk = 0; kk < D / 16; ++kk) {
        tc::mma_bf16(tmem + L::TP, kmaj(base + L::QF, kk), kmaj(base + L::KF, kk), ID_P, kk > 0);
        tc::mma_bf16(tmem + L::TX, kmaj(base + L::QF, kk), mnmaj(base + L::AS, kk, D * 128), ID_KM,
                     kk > 0);
      }
      tc::mma_commit(bar1);  // P and X: the row sums can start while the states are updated
      // (the state updates complete before phase 4's products, whose commit covers them)
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk) {
        tc::mma_bf16(tmem + L::TS, mnmaj(base + L::KF, kk, 16384), mnmaj(base + L::VS, kk, 16384),
                     ID_MM, 1u);
        tc::mma_bf16(tmem + L::TA, mnmaj(base + L::KF, kk, 16384), mnmaj(base + L::KF, kk, 16384),
                     ID_MM, 1u);
      }
    }
    if (!wait_mma(bar1, c & 1)) atomicExch(s_abort, 1);
    // ---- phase 3: den^2 = sum P^2 + q' . X;  P~ (masked, bf16)
    float den;
    {
      float pv[32];
      tmem_ld32(tmem + tl + L::TP + 32 * gw, pv);
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        pv[j] = 32 * gw + j <= t ? pv[j] : 0.f;
        part = fmaf(pv[j], pv[j], part);
      }
      if (gw < NG) {
        float xv[32];
        tmem_ld32(tmem + tl + L::TX + 32 * gw, xv);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float f[8];
          unpack8(lds16(base + L::QF + tile_off(t, 4 * gw + m)), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) part = fmaf(f[e], xv[8 * m + e], part);
        }
      }
      red[gw * kC + t] = part;
      store_row32<false>(base + L::PS, t, gw, pv);
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      const float ss = red[t] + red[kC + t] + red[2 * kC + t] + red[3 * kC + t];
      den = sqrtf(fmaxf(ss, 0.f)) + a.eps;
    }
    if (*reinterpret_cast<volatile int*>(s_abort)) { bad = true; break; }
    // ---- phase 4: X = Q'S~ + P~V
    if (tid == 0) {
      constexpr uint32_t ID_KM = tc::idesc_bf16(128, D, false, true);
#pragma unroll 1
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_bf16(tmem + L::TX, kmaj(base + L::QF, kk), mnmaj(base + L::SS, kk, D * 128), ID_KM,
                     kk > 0);
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk)
        tc::mma_bf16(tmem + L::TX, kmaj(base + L::PS, kk), mnmaj(base + L::VS, kk, 16384), ID_KM, 1u);
      tc::mma_commit(bar2);
    }
    if (!wait_mma(bar2, c & 1)) atomicExch(s_abort, 1);
    // every MMA has read q', k', v: the next chunk's tiles may arrive while this one finishes
    if (tid == 0 && c + 1 < nch && !*reinterpret_cast<volatile int*>(s_abort)) {
      tma_qkv<D>(&tq, &tk, &tv, base, h, static_cast<int>(row0 + t0 + kC), bar_ld);
      ++tma_issued;
    }
    // ---- phase 5: out = X / den; S, A -> S~, A~
    if (gw < NG) {
      float xv[32];
      tmem_ld32(tmem + tl + L::TX + 32 * gw, xv);
      const float inv = 1.0f / den;
#pragma unroll
      for (int j = 0; j < 32; ++j) xv[j] *= inv;
      if (t0 + t < s1) {
        __nv_bfloat16* dst = out + ((row0 + t0 + t) * a.H + h) * D + 32 * gw;
#pragma unroll
        for (int m = 0; m < 4; ++m) *reinterpret_cast<uint4*>(dst + 8 * m) = feat::pack8(xv + 8 * m);
      }
      if (t < D) {
        float sv[32];
        tmem_ld32(tmem + tl + L::TS + 32 * gw, sv);
        store_row32<true>(base + L::SS, t, gw, sv);
        tmem_ld32(tmem + tl + L::TA + 32 * gw, sv);
        store_row32<true>(base + L::AS, t, gw, sv);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(s_abort)) { bad = true; break; }
  }
  bad = bad || *reinterpret_cast<volatile int*>(s_abort) != 0;
  if (tid == 0 && tma_issued > 0) tc::mbar_wait(bar_ld, (tma_issued - 1) & 1, kWait);
  __syncthreads();
  if (bad) {  // a wait gave up: NaN over this segment's rows, so the failure cannot pass for a result
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out);
    for (long r = s0 + tid / (D / 8); r < s1; r += kThreads / (D / 8))
      *reinterpret_cast<uint4*>(o + ((row0 + r) * a.H + h) * D + 8 * (tid % (D / 8))) =
          make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0 && !misaligned) tc::tmem_dealloc(tmem, 512);
}

template <int D>
cudaError_t launch_d(const L2cTcArgs& a, const L2Args& mom, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(l2c_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(LayC<D>::BYTES));
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long grid = static_cast<long>(a.n_docs) * a.H * a.nseg;
  if (grid == 0 || a.total_rows == 0) return cudaSuccess;
  // dense segments after the first start from the moments of the splits before them
  const bool with_moments = a.nseg > 1;
  if (with_moments && (e = launch_l2_moments_tc(D, mom, a.nseg - 1, a.seg_len, stream)) != cudaSuccess)
    return e;
  CUtensorMap tq, tk, tv;
  if ((e = make_rows_map(&tq, a.q, a.total_rows, a.H, D)) != cudaSuccess) return e;
  if ((e = make_rows_map(&tk, a.k, a.total_rows, a.H, D)) != cudaSuccess) return e;
  if ((e = make_rows_map(&tv, a.v, a.total_rows, a.H, D)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LayC<D>::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = with_moments ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, l2c_tc_kernel<D>, a, tq, tk, tv);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool l2c_tc_supported(DType dt, int d) { return dt == DType::BF16 && (d == 64 || d == 128); }

L2cPlan l2c_tc_plan(int B, int L, int H, int d) {
  // One CTA per SM: a plan costs its waves of 152 CTAs times the chunks of a segment (plus one of
  // set-up); a longer plan must be clearly (5 %) cheaper to win. The workspace holds the moments of
  // every split but a batch row's last.
  L2cPlan p{1, 0, 0};
  const int chunks = L > 0 ? (L + kC - 1) / kC : 1;
  const long units = static_cast<long>(B) * H;
  double best = 1e300;
  for (int nseg = 1; nseg <= 64 && nseg <= chunks; ++nseg) {
    const int seg_chunks = (chunks + nseg - 1) / nseg;
    const double waves = static_cast<double>((units * nseg + 151) / 152);
    const double cost = waves * (seg_chunks + 1.0);
    if (cost < 0.95 * best) {
      best = cost;
      p.nseg = nseg;
      p.seg_len = seg_chunks * kC;
    }
  }
  if (p.seg_len == 0) p.seg_len = chunks * kC;
  p.ws_bytes = p.nseg > 1 ? static_cast<size_t>(units) * (p.nseg - 1) * d * 2 * d * sizeof(float) : 0;
  return p;
}

size_t l2c_tc_varlen_ws_bytes(int n_docs) {
  return n_docs <= 1024 ? static_cast<size_t>(n_docs) * sizeof(int) : 0;
}

cudaError_t launch_l2_causal_tc(int d, L2cTcArgs a, void* ws, cudaStream_t stream) {
  L2Args mom{};
  mom.k = a.k;
  mom.v = a.v;
  mom.ws = static_cast<float*>(ws);
  mom.B = a.n_docs;
  mom.L = a.doc_len;
  mom.H = a.H;
  mom.eps = a.eps;
  a.ws = static_cast<const float*>(ws);
  a.order = nullptr;
  if (a.cu_seqlens != nullptr && l2c_tc_varlen_ws_bytes(a.n_docs) > 0) {
    // packed documents: one CTA per (document, head), the longest documents dispatched first
    int* order = static_cast<int*>(ws);
    const cudaError_t e = launch_doc_order(a.cu_seqlens, a.n_docs, a.total_rows, order, stream);
    if (e != cudaSuccess) return e;
    a.order = order;
  }
  return d == 128 ? launch_d<128>(a, mom, stream) : launch_d<64>(a, mom, stream);
}

}  // namespace rapt
