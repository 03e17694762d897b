// Causal original RLA (L2 denominator) on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a;
// dense bf16, d = 128, fp32 accumulation and fp32 states.
//
// 08-rapt-algorithm.md §2.1 (closed form, eps outside the root; q' = ReLU(q), k' = ReLU(k)), §2.2
// (a query reads the accumulated causal state), §4.1 (the scan's two prefix states):
//   S_t = sum_{i<=t} k'_i v_i^T,  A_t = sum_{i<=t} k'_i k'_i^T,
//   out_t = q'_t S_t / (sqrt(q'_t^T A_t q'_t) + eps).
// Chunked (C = 128 tokens), with P = Q'K'^T masked to tau <= t and S~, A~ bf16 copies of the fp32
// states before the chunk:
//   phase 2:  P = Q'K'^T,  X = Q' A~ (committed), then S += K'^T V,  A += K'^T K' (run during phase 3)
//   phase 3:  den_t = sqrt(sum_tau P^2 + q'_t . X_t) + eps (fp32; P from exact bf16 features),
//             P~ = P masked, in bf16
//   phase 4:  X = Q' S~ + P~ V
//   phase 5:  out = X / den; S, A -> S~, A~ for the next chunk.
// Documents (batch rows) are cut into segments of seg_len tokens; segment s starts from the
// moments [K'^T V | K'^T K'] of the splits before it, computed by the non-causal L2 path's moments
// kernel with the same split length (summed in split order: deterministic). One CTA per (batch row,
// head, segment), 512 threads in lockstep phases, one thread issuing the MMAs and the TMA copies:
// the next chunk's q, k, v tiles are requested as soon as the current chunk's last MMA has read
// its tiles, so they arrive while the chunk's output and state copies are written. Every wait is
// bounded (~1 s); a CTA whose wait gives up writes NaN over its rows.
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
constexpr uint32_t kTile = 32768;

struct LayC {
  static constexpr uint32_t QF = 0, KF = kTile, VS = 2 * kTile, SS = 3 * kTile, AS = 4 * kTile;
  static constexpr uint32_t PS = 5 * kTile;
  static constexpr uint32_t RED = 6 * kTile;         // partial den^2 [4][128]
  static constexpr uint32_t BAR = RED + 4 * kC * 4;  // three mbarriers
  static constexpr uint32_t MISC = BAR + 24;         // TMEM base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};
constexpr uint32_t kTP = 0, kTX = 128, kTS = 256, kTA = 384;  // TMEM columns: P, X, S, A

// The chunk's raw q, k, v rows into their tiles by TMA (two 64-column boxes each), completing on
// one mbarrier; one thread calls it. Rows past the tensor read as zero.
__device__ __forceinline__ void tma_qkv(const CUtensorMap* tq, const CUtensorMap* tk,
                                        const CUtensorMap* tv, uint32_t base, int h, int t, int bb,
                                        uint32_t bar) {
  tc::mbar_arrive_expect_tx(bar, 3 * kTile);
#pragma unroll
  for (int jb = 0; jb < 2; ++jb) {
    tc::tma_load_4d(base + LayC::QF + jb * 16384, tq, 64 * jb, h, t, bb, bar);
    tc::tma_load_4d(base + LayC::KF + jb * 16384, tk, 64 * jb, h, t, bb, bar);
    tc::tma_load_4d(base + LayC::VS + jb * 16384, tv, 64 * jb, h, t, bb, bar);
  }
}

// In place: q and k tiles rectified (bf16 max(0, x) on the bit patterns: a set sign bit, negative
// or -0, becomes +0). The 4-D maps read rows past the batch row's end as zero already.
__device__ __forceinline__ void rectify_qk(uint32_t base) {
  for (int idx = threadIdx.x; idx < 2 * kC * 16; idx += kThreads) {
    const uint32_t addr =
        base + (idx < kC * 16 ? LayC::QF : LayC::KF) + tile_off((idx >> 4) & (kC - 1), idx & 15);
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

__global__ void __launch_bounds__(kThreads, 1)
    l2c_tc_kernel(const L2Args a, int nseg, int seg_len, const __grid_constant__ CUtensorMap tq,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % nseg, bh = blockIdx.x / nseg;
  const int bb = bh / a.H, h = bh % a.H;
  const int n = a.L;
  const long row0 = static_cast<long>(bb) * a.L;
  const int s0 = seg * seg_len, s1 = min(n, s0 + seg_len);
  if (s0 >= s1) return;  // uniform, before any allocation
  const int nch = (s1 - s0 + kC - 1) / kC;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  float* red = reinterpret_cast<float*>(smem + LayC::RED);
  const uint32_t bar1 = base + LayC::BAR, bar2 = bar1 + 8, bar_ld = bar1 + 16;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + LayC::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + LayC::MISC + 4);
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
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int q4 = warp & 3, gw = warp >> 2;
  const int t = 32 * q4 + lane;  // tile row = TMEM lane
  const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
  bool bad = *s_abort != 0;

  // the states at the segment's start: the moments of the earlier splits, in split order
  if (!bad) {
    const float4* part = reinterpret_cast<const float4*>(a.ws) +
                         static_cast<long>(bh) * nseg * (kD * 2 * kD / 4);
    float sv[32], av[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) sv[e] = av[e] = 0.f;
    for (int sp = 0; sp < seg; ++sp) {
      const float4* ps = part + static_cast<long>(sp) * (kD * 2 * kD / 4);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float4 x = __ldcg(ps + (8 * gw + jj) * kD + t);
        const float4 y = __ldcg(ps + (kD / 4 + 8 * gw + jj) * kD + t);
        sv[4 * jj] += x.x; sv[4 * jj + 1] += x.y; sv[4 * jj + 2] += x.z; sv[4 * jj + 3] += x.w;
        av[4 * jj] += y.x; av[4 * jj + 1] += y.y; av[4 * jj + 2] += y.z; av[4 * jj + 3] += y.w;
      }
    }
    state_put(tmem + tl + kTS + 32 * gw, base + LayC::SS, t, gw, sv);
    state_put(tmem + tl + kTA + 32 * gw, base + LayC::AS, t, gw, av);
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  int tma_issued = 0;  // chunks whose tiles have been requested (thread 0)
  if (tid == 0 && !bad) {
    tma_qkv(&tq, &tk, &tv, base, h, s0, bb, bar_ld);
    tma_issued = 1;
  }
  for (int c = 0; c < nch && !bad; ++c) {
    const int t0 = s0 + c * kC;
    // ---- phase 1: the chunk's q, k, v (TMA, requested one chunk ahead); q' = ReLU(q), k' = ReLU(k)
    if (!tc::mbar_wait(bar_ld, c & 1, kWait)) atomicExch(s_abort, 1);
    rectify_qk(base);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- phase 2: P = Q'K'^T, X = Q'A~, S += K'^T V, A += K'^T K'
    if (tid == 0) {
      constexpr uint32_t ID_KK = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_KM = tc::idesc_bf16(128, 128, false, true);
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, 128, true, true);
#pragma unroll 1
      for (int kk = 0; kk < kD / 16; ++kk) {
        tc::mma_bf16(tmem + kTP, kmaj(base + LayC::QF, kk), kmaj(base + LayC::KF, kk), ID_KK, kk > 0);
        tc::mma_bf16(tmem + kTX, kmaj(base + LayC::QF, kk), mnmaj(base + LayC::AS, kk, kD * 128),
                     ID_KM, kk > 0);
      }
      tc::mma_commit(bar1);  // P and X: the row sums can start while the states are updated
      // (the state updates complete before phase 4's products, whose commit covers them)
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk) {
        tc::mma_bf16(tmem + kTS, mnmaj(base + LayC::KF, kk, 16384), mnmaj(base + LayC::VS, kk, 16384),
                     ID_MM, 1u);
        tc::mma_bf16(tmem + kTA, mnmaj(base + LayC::KF, kk, 16384), mnmaj(base + LayC::KF, kk, 16384),
                     ID_MM, 1u);
      }
    }
    if (!wait_mma(bar1, c & 1)) atomicExch(s_abort, 1);
    // ---- phase 3: den^2 = sum P^2 + q' . X;  P~ (masked, bf16)
    float den;
    {
      float pv[32], xv[32];
      tmem_ld32(tmem + tl + kTP + 32 * gw, pv);
      tmem_ld32(tmem + tl + kTX + 32 * gw, xv);
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        pv[j] = 32 * gw + j <= t ? pv[j] : 0.f;
        part = fmaf(pv[j], pv[j], part);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float f[8];
        unpack8(lds16(base + LayC::QF + tile_off(t, 4 * gw + m)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(f[e], xv[8 * m + e], part);
      }
      red[gw * kC + t] = part;
      store_row32<false>(base + LayC::PS, t, gw, pv);
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
      constexpr uint32_t ID_KM = tc::idesc_bf16(128, 128, false, true);
#pragma unroll 1
      for (int kk = 0; kk < kD / 16; ++kk)
        tc::mma_bf16(tmem + kTX, kmaj(base + LayC::QF, kk), mnmaj(base + LayC::SS, kk, kD * 128),
                     ID_KM, kk > 0);
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk)
        tc::mma_bf16(tmem + kTX, kmaj(base + LayC::PS, kk), mnmaj(base + LayC::VS, kk, 16384), ID_KM,
                     1u);
      tc::mma_commit(bar2);
    }
    if (!wait_mma(bar2, c & 1)) atomicExch(s_abort, 1);
    // every MMA has read q', k', v: the next chunk's tiles may arrive while this one finishes
    if (tid == 0 && c + 1 < nch && !*reinterpret_cast<volatile int*>(s_abort)) {
      tma_qkv(&tq, &tk, &tv, base, h, t0 + kC, bb, bar_ld);
      ++tma_issued;
    }
    // ---- phase 5: out = X / den; S, A -> S~, A~
    {
      float xv[32];
      tmem_ld32(tmem + tl + kTX + 32 * gw, xv);
      const float inv = 1.0f / den;
#pragma unroll
      for (int j = 0; j < 32; ++j) xv[j] *= inv;
      if (t0 + t < n) {
        __nv_bfloat16* dst = out + ((row0 + t0 + t) * a.H + h) * kD + 32 * gw;
#pragma unroll
        for (int m = 0; m < 4; ++m) *reinterpret_cast<uint4*>(dst + 8 * m) = feat::pack8(xv + 8 * m);
      }
      float sv[32];
      tmem_ld32(tmem + tl + kTS + 32 * gw, sv);
      store_row32<true>(base + LayC::SS, t, gw, sv);
      tmem_ld32(tmem + tl + kTA + 32 * gw, sv);
      store_row32<true>(base + LayC::AS, t, gw, sv);
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
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out);
    for (long r = s0 + tid / 16; r < s1; r += kThreads / 16)
      *reinterpret_cast<uint4*>(o + ((row0 + r) * a.H + h) * kD + 8 * (tid % 16)) =
          make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0 && !misaligned) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

bool l2c_tc_supported(DType dt, int d, bool varlen) { return dt == DType::BF16 && d == kD && !varlen; }

L2cPlan l2c_tc_plan(int B, int L, int H) {
  // One CTA per SM: a plan costs its waves of 152 CTAs times the chunks of a segment (plus one of
  // set-up); a longer plan must be clearly (5 %) cheaper to win.
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
  p.ws_bytes = p.nseg > 1 ? static_cast<size_t>(units) * p.nseg * kD * 2 * kD * sizeof(float) : 0;
  return p;
}

cudaError_t launch_l2_causal_tc(const L2Args& a, int nseg, int seg_len, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(l2c_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(LayC::BYTES));
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long grid = static_cast<long>(a.B) * a.H * nseg;
  if (grid == 0 || a.L == 0) return cudaSuccess;
  if (nseg > 1 && (e = launch_l2_moments_tc(a, nseg, seg_len, stream)) != cudaSuccess) return e;
  CUtensorMap tq, tk, tv;
  if ((e = make_bshd_map(&tq, a.q, a.B, a.L, a.H, kD)) != cudaSuccess) return e;
  if ((e = make_bshd_map(&tk, a.k, a.B, a.L, a.H, kD)) != cudaSuccess) return e;
  if ((e = make_bshd_map(&tv, a.v, a.B, a.L, a.H, kD)) != cudaSuccess) return e;
  l2c_tc_kernel<<<static_cast<unsigned>(grid), kThreads, LayC::BYTES, stream>>>(a, nseg, seg_len, tq,
                                                                              tk, tv);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rapt
