// Original RLA with the L2 denominator (08-rapt-algorithm.md §2.1, §2.2) on the 5th-generation
// tensor cores (tcgen05 + TMEM), sm_103a; bf16 inputs, d in {64, 128}, fp32 accumulation:
//
//   q' = ReLU(q), k' = ReLU(k);  M_V = K'^T V,  M_K = K'^T K'  (d x d each, over all L tokens)
//   out_t = q'_t M_V / (sqrt(q'_t^T M_K q'_t) + eps)
//
// By associativity the L x L score matrix is never formed (§2.2: K'^T V first, then Q'(K'^T V));
// both moments come out of one GEMM, [M_V | M_K] = K'^T [V | K'], and both readouts out of one
// more, q' [M_V | M_K]: N = 2d columns each, the tensor core's widest single-CTA shape at d = 128.
//
// Three launches on the caller's stream:
//   1. moments (one CTA per batch row, head and token split): raw k and v tiles arrive by TMA in a
//      ring of stages, four warps apply the ReLU to k in place, one thread issues the GEMM into
//      TMEM; the fp32 partial [M_V | M_K] of the split is written out (no atomics: deterministic);
//   2. reduce: the partials summed in split order, written as the bf16 [M_V | M_K] operand of
//      launch 3 in the exact shared-memory layout the tensor core reads (one bulk copy there);
//   3. readout (one CTA per batch row, head and token split): q tiles by TMA, ReLU in place, one
//      GEMM per 128-token tile into one of two TMEM accumulators; eight epilogue warps (two per
//      row, half of the columns each) form den = sqrt(sum_j q'_j (q'M_K)_j) + eps from the same
//      bf16 q' the GEMM read and write out = num / den over the q tile; one thread stores it by TMA.
// Launches 2 and 3 are programmatic dependents of the launch before them (set-up and the first
// q tiles overlap the predecessor's tail).
// Tensor maps are 4-D ([B, L, H, d]), so tiles past the end of a batch row read as zero and are
// not written back. Every wait is bounded; a CTA whose wait gives up writes NaN results (the
// moments of its split, or its output rows), so a failure cannot pass for a result.
#include <cuda.h>

#include <cstring>

#include "kernels.h"
#include "tc_utils.cuh"
#include "tensor_map.h"

namespace rapt {
namespace {

constexpr int kC = 128;                        // tokens per tile = MMA M (readout) or K (moments)
constexpr long long kWait = 2000000000LL;      // ~1 s
constexpr int kP1Threads = 192;                // warps 0-3: ReLU + epilogue; 4: TMA; 5: MMA
constexpr int kP2Threads = 448;                // warps 0-7: epilogue; 8-11: ReLU; 12: TMA; 13: MMA
constexpr int kStages = 3;

// In-place ReLU of 8 bf16 values.
__device__ __forceinline__ uint4 relu8(uint4 x) {
  const __nv_bfloat162 z = __float2bfloat162_rn(0.f);
  uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w[i]);
    v = __hmax2(v, z);
    w[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return x;
}
// bar.sync over a group, returning the OR of every member's flag (so all members agree).
__device__ __forceinline__ int group_sync_or(uint32_t id, uint32_t n, int flag) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %3, 0;\n bar.red.or.pred q, %1, %2, p;\n"
      " selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(id), "r"(n), "r"(flag)
      : "memory");
  return r;
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts16(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ------------------------------------------------------------------------------------------------
// Launch 1: moments. Shared memory: kStages stages of [v blocks | k' blocks | zero block at d = 64]
// (each block 128 tokens x 64 columns, 16 KB, 128-byte swizzle).
template <int D>
struct P1 {
  static constexpr int DB = D / 64;
  static constexpr int N = 2 * D;
  static constexpr uint32_t TILE = DB * 16384;
  static constexpr uint32_t STAGE = 2 * TILE + (D == 64 ? 16384 : 0);
  static constexpr uint32_t BAR = kStages * STAGE;  // full[S] relu[S] empty[S] done
  static constexpr uint32_t MISC = BAR + (3 * kStages + 1) * 8;
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kP1Threads, 1)
    l2_tc_moments(const L2Args a, int nsplit, int split_len, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
  using L = P1<D>;
  constexpr int S = kStages, N = L::N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tc::grid_launch_dependents();  // the reduce launch may be scheduled; it waits for this grid
  const int sp = blockIdx.x % nsplit, bh = blockIdx.x / nsplit;
  const int b = bh / a.H, h = bh % a.H;
  const int t0 = sp * split_len;
  const int t1 = min(a.L, t0 + split_len);
  const int nchunks = t1 > t0 ? (t1 - t0 + kC - 1) / kC : 0;
  float4* part = reinterpret_cast<float4*>(a.ws + (static_cast<long>(bh) * nsplit + sp) * D * N);

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  const uint32_t bar_full = base + L::BAR, bar_relu = bar_full + 8 * S;
  const uint32_t bar_empty = bar_relu + 8 * S, bar_done = bar_empty + 8 * S;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;  // uniform; the swizzled layouts need 1 KB

  if (warp == 0 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), N);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(bar_full + 8 * s, 1);
      tc::mbar_init(bar_relu + 8 * s, 128);
      tc::mbar_init(bar_empty + 8 * s, 1);
    }
    tc::mbar_init(bar_done, 1);
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  if (D == 64) {  // zero block that pads k'^T to M = 128 rows, one per stage
    for (int i = tid; i < S * 1024; i += kP1Threads)
      sts16(base + (i / 1024) * L::STAGE + 2 * L::TILE + (i % 1024) * 16, make_uint4(0, 0, 0, 0));
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const bool run = !*s_abort;

  if (warp == 4) {
    if (lane == 0 && run) {  // TMA: v then k of each tile into a free stage
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % S;
        if (c >= S && !tc::mbar_wait(bar_empty + 8 * s, ((c / S) - 1) & 1, kWait)) {
          atomicExch(s_abort, 1);
          break;
        }
        const uint32_t st = base + s * L::STAGE;
        tc::mbar_arrive_expect_tx(bar_full + 8 * s, 2 * L::TILE);
#pragma unroll
        for (int jb = 0; jb < L::DB; ++jb) {
          tc::tma_load_4d(st + jb * 16384, &tv, 64 * jb, h, t0 + c * kC, b, bar_full + 8 * s);
          tc::tma_load_4d(st + L::TILE + jb * 16384, &tk, 64 * jb, h, t0 + c * kC, b, bar_full + 8 * s);
        }
      }
    }
  } else if (warp == 5) {
    if (lane == 0 && run) {  // MMA: [M_V | M_K] += K'^T [V | K'], M = 128 (d rows, zero-padded at d = 64)
      constexpr uint32_t ID = tc::idesc_bf16(128, N, true, true);
      int ok = 1;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % S;
        ok = tc::mbar_wait(bar_relu + 8 * s, (c / S) & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t st = base + s * L::STAGE;
        const uint64_t da = tc::desc_sw128(st + L::TILE, 16384, 1024);
        const uint64_t db = tc::desc_sw128(st, 16384, 1024);
#pragma unroll 1
        for (int k = 0; k < kC / 16; ++k)
          tc::mma_bf16(tmem, da + static_cast<uint64_t>(k) * 128, db + static_cast<uint64_t>(k) * 128, ID,
                       (c > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(bar_empty + 8 * s);
      }
      if (!ok) atomicExch(s_abort, 1);
      tc::mma_commit(bar_done);
    }
  } else {
    // ReLU of the k blocks, in place
    if (run) {
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % S;
        if (!tc::mbar_wait(bar_full + 8 * s, (c / S) & 1, kWait)) {
          atomicExch(s_abort, 1);
          break;
        }
        const uint32_t kb = base + s * L::STAGE + L::TILE;
#pragma unroll 4
        for (int i = tid; i < static_cast<int>(L::TILE / 16); i += 128) sts16(kb + i * 16, relu8(lds16(kb + i * 16)));
        tc::fence_async_smem();
        tc::mbar_arrive(bar_relu + 8 * s);
      }
    }
    // epilogue: TMEM lane i = row i of [M_V | M_K] -> partial, float4 (i, 4j..4j+3) at j * D + i
    const int ok = run && tc::mbar_wait(bar_done, 0, kWait);
    const int good = __all_sync(0xffffffffu, ok && !*reinterpret_cast<volatile int*>(s_abort));
    tc::fence_after_sync();
    const int er = 32 * warp + lane;
    if (32 * warp < D) {
      const uint32_t tl = static_cast<uint32_t>(32 * warp) << 16;
      for (int j0 = 0; j0 < N; j0 += 16) {
        uint32_t u[16];
        if (good && nchunks > 0) {
          tc::tmem_ld16(tmem + tl + j0, u);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = good ? 0u : 0x7fc00000u;  // zeros, or NaN on failure
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
          __stcg(part + (j0 / 4 + e) * D + er,
                 make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                             __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3])));
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && !misaligned) tc::tmem_dealloc(tmem, N);
}

// ------------------------------------------------------------------------------------------------
// Launch 2: the split partials of one (batch row, head), summed in split order, as the bf16 B
// operand of the readout GEMM: [M_V | M_K] with rows = K (q' feature i) and 64-column blocks of
// N (output column j), each block D rows x 128 bytes, 16-byte chunk c of row i at c ^ (i & 7).
template <int D>
__global__ void __launch_bounds__(256) l2_tc_reduce(const float* ws, int nsplit, long img_offset) {
  constexpr int N = 2 * D;
  constexpr int Q = D * N / 4;  // float4 per partial
  const int bh = blockIdx.y;
  tc::grid_launch_dependents();  // the readout may set up and load its first q tiles
  tc::grid_dep_wait();           // the partials of the moments launch
  const float4* p = reinterpret_cast<const float4*>(ws) + static_cast<long>(bh) * nsplit * Q;
  uint8_t* img = reinterpret_cast<uint8_t*>(const_cast<float*>(ws) + img_offset) + static_cast<long>(bh) * D * N * 2;
  for (int e = blockIdx.x * 256 + threadIdx.x; e < Q; e += gridDim.x * 256) {
    float4 m = __ldcg(p + e);
    for (int s = 1; s < nsplit; ++s) {
      const float4 x = __ldcg(p + static_cast<long>(s) * Q + e);
      m.x += x.x; m.y += x.y; m.z += x.z; m.w += x.w;
    }
    const int i = e % D, j = 4 * (e / D);
    const int jb = j / 64, cc = (j % 64) / 8, half = (j % 8) / 4;
    const uint2 w = make_uint2(tc::pack_bf16x2(m.x, m.y), tc::pack_bf16x2(m.z, m.w));
    *reinterpret_cast<uint2*>(img + jb * (D * 128) + i * 128 + ((cc ^ (i & 7)) << 4) + half * 8) = w;
  }
}

// The split partials of one (batch row, head), summed in split order, as the plain fp32
// [M_V | M_K] (row i, column j at i * 2D + j) of the moments-only entry point.
template <int D>
__global__ void __launch_bounds__(256) l2_tc_plain(const float* ws, int nsplit, float* M) {
  constexpr int N = 2 * D;
  constexpr int Q = D * N / 4;
  const int bh = blockIdx.y;
  const float4* p = reinterpret_cast<const float4*>(ws) + static_cast<long>(bh) * nsplit * Q;
  for (int e = blockIdx.x * 256 + threadIdx.x; e < Q; e += gridDim.x * 256) {
    float4 m = __ldcg(p + e);
    for (int s = 1; s < nsplit; ++s) {
      const float4 x = __ldcg(p + static_cast<long>(s) * Q + e);
      m.x += x.x; m.y += x.y; m.z += x.z; m.w += x.w;
    }
    const int i = e % D, j = 4 * (e / D);
    *reinterpret_cast<float4*>(M + (static_cast<long>(bh) * D + i) * N + j) = m;
  }
}

// The plain fp32 [M_V | M_K] of the readout-only entry point as the bf16 B operand image of the
// readout GEMM (the layout l2_tc_reduce writes).
template <int D>
__global__ void __launch_bounds__(256) l2_tc_image(const float* M, uint8_t* img_all) {
  constexpr int N = 2 * D;
  constexpr int Q = D * N / 4;
  const int bh = blockIdx.y;
  tc::grid_launch_dependents();  // the readout may set up and load its first q tiles
  uint8_t* img = img_all + static_cast<long>(bh) * D * N * 2;
  for (int e = blockIdx.x * 256 + threadIdx.x; e < Q; e += gridDim.x * 256) {
    const int i = e / (N / 4), j = 4 * (e % (N / 4));
    const float4 m = __ldg(reinterpret_cast<const float4*>(M + (static_cast<long>(bh) * D + i) * N + j));
    const int jb = j / 64, cc = (j % 64) / 8, half = (j % 8) / 4;
    const uint2 w = make_uint2(tc::pack_bf16x2(m.x, m.y), tc::pack_bf16x2(m.z, m.w));
    *reinterpret_cast<uint2*>(img + jb * (D * 128) + i * 128 + ((cc ^ (i & 7)) << 4) + half * 8) = w;
  }
}

// ------------------------------------------------------------------------------------------------
// Launch 3: readout. Shared memory: the [M_V | M_K] image, kStages q tiles (each 128 tokens x d,
// K-major blocks of 64 columns; out is written over the tile q' was read from), and the partial
// den^2 of the two column halves of every row. Warps 0-7 are the epilogue, two per TMEM lane
// quarter (warp % 4), each taking half of a row's columns; warps 8-11 apply the ReLU.
template <int D>
struct P2 {
  static constexpr int S = 4;  // q tile stages (four tiles of loads and stores in flight)
  static constexpr int DB = D / 64;
  static constexpr int N = 2 * D;
  static constexpr int HALF = D / 2;
  static constexpr uint32_t MB = (N / 64) * D * 128;
  static constexpr uint32_t QT = DB * 16384;
  static constexpr uint32_t QS = MB;
  static constexpr uint32_t DP = QS + S * QT;               // partial den^2 [2 halves][128 rows]
  // mfull, qfull[S], relu[S], staged[S], accf[2], accfree[2]
  static constexpr uint32_t BAR = DP + 2 * kC * 4;
  static constexpr uint32_t MISC = BAR + (1 + 3 * S + 4) * 8;
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(MB % 1024 == 0 && QT % 1024 == 0, "tile alignment");
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(2 * N <= 512, "TMEM budget");
};
constexpr uint32_t kBarEpi = 1;  // named barrier of the 256 epilogue threads

template <int D>
__global__ void __launch_bounds__(kP2Threads, 1)
    l2_tc_readout(const L2Args a, int nsplit, int split_chunks, long img_offset,
                  const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap to) {
  using L = P2<D>;
  constexpr int S = L::S, N = L::N, HALF = L::HALF;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.x % nsplit, bh = blockIdx.x / nsplit;
  const int b = bh / a.H, h = bh % a.H;
  const int total = (a.L + kC - 1) / kC;
  const int c0 = sp * split_chunks;
  const int n = min(total, c0 + split_chunks) - c0;
  if (n <= 0) return;  // uniform, before any allocation
  const uint8_t* img = reinterpret_cast<const uint8_t*>(a.ws + img_offset) + static_cast<long>(bh) * L::MB;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  const uint32_t bar_m = base + L::BAR, bar_qfull = bar_m + 8, bar_relu = bar_qfull + 8 * S;
  const uint32_t bar_staged = bar_relu + 8 * S, bar_accf = bar_staged + 8 * S, bar_accfree = bar_accf + 16;
  float* dpart = reinterpret_cast<float*>(smem + L::DP);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;

  if (warp == 0 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 2 * N);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_m, 1);
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(bar_qfull + 8 * s, 1);
      tc::mbar_init(bar_relu + 8 * s, 128);
      tc::mbar_init(bar_staged + 8 * s, 256);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(bar_accf + 8 * x, 1);
      tc::mbar_init(bar_accfree + 8 * x, 256);
    }
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const bool run = !*s_abort;
  auto tile = [&](int s) { return base + L::QS + s * L::QT; };

  if (warp == 12) {
    if (lane == 0 && run) {  // TMA: q tiles in, out tiles back, and the moments once
      int ok = 1;
      for (int i = 0; i < n + S && ok; ++i) {
        if (i >= S) {  // the tile S back is staged: store it, then its buffer is free
          const int j = i - S, s = j % S;
          ok = tc::mbar_wait(bar_staged + 8 * s, (j / S) & 1, kWait);
          if (!ok) break;
#pragma unroll
          for (int jb = 0; jb < L::DB; ++jb)
            tc::tma_store_4d(&to, tile(s) + jb * 16384, 64 * jb, h, (c0 + j) * kC, b);
          tc::bulk_commit();
          tc::bulk_wait_read0();
        }
        if (i < n) {
          const int s = i % S;
          tc::mbar_arrive_expect_tx(bar_qfull + 8 * s, L::QT);
#pragma unroll
          for (int jb = 0; jb < L::DB; ++jb)
            tc::tma_load_4d(tile(s) + jb * 16384, &tq, 64 * jb, h, (c0 + i) * kC, b, bar_qfull + 8 * s);
        }
        if (i == 0) {
          // the moments come from the reduce launch, which may still be running
          tc::grid_dep_wait();
          tc::mbar_arrive_expect_tx(bar_m, L::MB);
          tc::bulk_g2s(base, img, L::MB, bar_m);
        }
      }
      if (!ok) atomicExch(s_abort, 1);
      tc::bulk_wait0();
    }
  } else if (warp == 13) {
    if (lane == 0 && run) {  // MMA: [num | q'M_K] = Q' [M_V | M_K], M = 128 tokens, N = 2d, K = d
      constexpr uint32_t ID = tc::idesc_bf16(128, N, false, true);
      const uint64_t dm = tc::desc_sw128(base, D * 128, 1024);
      int ok = tc::mbar_wait(bar_m, 0, kWait);
      for (int i = 0; i < n && ok; ++i) {
        const int s = i % S, x = i & 1;
        ok = tc::mbar_wait(bar_relu + 8 * s, (i / S) & 1, kWait) &&
             (i < 2 || tc::mbar_wait(bar_accfree + 8 * x, ((i >> 1) - 1) & 1, kWait));
        if (!ok) break;
        tc::fence_after_sync();
        const uint64_t dq = tc::desc_sw128(tile(s), 16, 1024);
#pragma unroll 1
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t kofs = static_cast<uint64_t>((k / 4) * 1024 + (k % 4) * 2);
          tc::mma_bf16(tmem + x * N, dq + kofs, dm + static_cast<uint64_t>(k) * 128, ID, k > 0);
        }
        tc::mma_commit(bar_accf + 8 * x);
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else if (warp >= 8) {
    if (run) {  // ReLU of the q tiles, in place
      const int rt = tid - 256;
      for (int i = 0; i < n; ++i) {
        const int s = i % S;
        if (!tc::mbar_wait(bar_qfull + 8 * s, (i / S) & 1, kWait)) {
          atomicExch(s_abort, 1);
          break;
        }
        const uint32_t qb = tile(s);
#pragma unroll 4
        for (int u = rt; u < static_cast<int>(L::QT / 16); u += 128) sts16(qb + u * 16, relu8(lds16(qb + u * 16)));
        tc::fence_async_smem();
        tc::mbar_arrive(bar_relu + 8 * s);
      }
    }
  } else if (run) {
    // epilogue: TMEM lane = token row er of the tile; this thread owns columns [c0h, c0h + HALF)
    const int q4 = warp & 3, g = warp >> 2;
    const int er = 32 * q4 + lane;
    const int c0h = g * HALF;
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    for (int i = 0; i < n; ++i) {
      const int s = i % S, x = i & 1;
      const int ok = tc::mbar_wait(bar_accf + 8 * x, (i >> 1) & 1, kWait);
      // uniform over the 256 epilogue threads (the named barriers below need all of them)
      if (group_sync_or(kBarEpi, 256, !ok)) {
        atomicExch(s_abort, 1);
        break;
      }
      tc::fence_after_sync();
      const uint32_t acc = tmem + tl + x * N;
      const uint32_t qb = tile(s);
      // partial den^2 over this half: sum_j q'_j (q'M_K)_j with the bf16 q' of the GEMM, 32
      // columns per TMEM round trip
      float2 d2 = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int j0 = c0h; j0 < c0h + HALF; j0 += 32) {
        uint32_t y[2][16];
        tc::tmem_ld16(acc + D + j0, y[0]);
        tc::tmem_ld16(acc + D + j0 + 16, y[1]);
        const uint32_t blk = qb + static_cast<uint32_t>(j0 / 64) * 16384;
        uint4 qv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) qv[m] = lds16(blk + tc::sw128(er, (j0 % 64) / 8 + m));
        tc::tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t qw[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d2 = __ffma2_rn(make_float2(__uint_as_float(qw[e] << 16), __uint_as_float(qw[e] & 0xffff0000u)),
                            make_float2(__uint_as_float(y[m >> 1][8 * (m & 1) + 2 * e]),
                                        __uint_as_float(y[m >> 1][8 * (m & 1) + 2 * e + 1])),
                            d2);
        }
      }
      dpart[g * kC + er] = d2.x + d2.y;
      // the numerator's half row is requested from TMEM before the barrier: its latency overlaps
      // the wait for the other half's den partial
      uint32_t u[HALF / 16][16];
#pragma unroll
      for (int m = 0; m < HALF / 16; ++m) tc::tmem_ld16(acc + c0h + 16 * m, u[m]);
      tc::named_sync(kBarEpi, 256);
      const float inv = 1.0f / (sqrtf(dpart[er] + dpart[kC + er]) + a.eps);  // fixed order
      tc::tmem_wait_ld();
      // out = num / den over this half of the row (the bytes this thread read q' from)
#pragma unroll
      for (int m = 0; m < HALF / 16; ++m) {
        const int j0 = c0h + 16 * m;
        float f[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(u[m][e]) * inv;
        const uint32_t blk = qb + static_cast<uint32_t>(j0 / 64) * 16384;
        sts16(blk + tc::sw128(er, (j0 % 64) / 8),
              make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]),
                         tc::pack_bf16x2(f[4], f[5]), tc::pack_bf16x2(f[6], f[7])));
        sts16(blk + tc::sw128(er, (j0 % 64) / 8 + 1),
              make_uint4(tc::pack_bf16x2(f[8], f[9]), tc::pack_bf16x2(f[10], f[11]),
                         tc::pack_bf16x2(f[12], f[13]), tc::pack_bf16x2(f[14], f[15])));
      }
      tc::fence_before_sync();
      tc::mbar_arrive(bar_accfree + 8 * x);
      tc::fence_async_smem();
      tc::mbar_arrive(bar_staged + 8 * s);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*s_abort) {  // a wait gave up: this CTA's rows read as NaN rather than as a result
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const __nv_bfloat16 nan = __float2bfloat16(__int_as_float(0x7fc00000));
    for (long r = tid; r < static_cast<long>(n) * kC * D; r += kP2Threads) {
      const long t = static_cast<long>(c0) * kC + r / D;
      if (t < a.L) out[((static_cast<long>(b) * a.L + t) * a.H + h) * D + r % D] = nan;
    }
  }
  if (warp == 0 && !misaligned) tc::tmem_dealloc(tmem, 2 * N);
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes, unsigned long long& configured) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && ((configured >> dev) & 1ull)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && dev < 64) configured |= 1ull << dev;
  return e;
}

// Token splits per (batch row, head): as many CTAs as fit one wave of 152 SMs, at least one tile each.
int l2_tc_splits(int B, int L, int H) {
  const long bh = static_cast<long>(B) * H;
  const long tiles = (L + kC - 1) / kC;
  long s = bh >= 152 ? 1 : 152 / bh;
  if (s > tiles) s = tiles;
  return static_cast<int>(s < 1 ? 1 : s);
}

template <int D>
cudaError_t launch_l2_tc_d(const L2Args& a, cudaStream_t stream) {
  static unsigned long long cfg1 = 0, cfg2 = 0;
  cudaError_t e = set_smem(l2_tc_moments<D>, P1<D>::BYTES, cfg1);
  if (e == cudaSuccess) e = set_smem(l2_tc_readout<D>, P2<D>::BYTES, cfg2);
  if (e != cudaSuccess) return e;
  const long n_bh = static_cast<long>(a.B) * a.H;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  CUtensorMap tq, tk, tv, to;
  e = make_bshd_map(&tq, a.q, a.B, a.L, a.H, D);
  if (e == cudaSuccess) e = make_bshd_map(&tk, a.k, a.B, a.L, a.H, D);
  if (e == cudaSuccess) e = make_bshd_map(&tv, a.v, a.B, a.L, a.H, D);
  if (e == cudaSuccess) e = make_bshd_map(&to, a.out, a.B, a.L, a.H, D);
  if (e != cudaSuccess) return e;
  const int tiles = (a.L + kC - 1) / kC;
  const int nsplit = l2_tc_splits(a.B, a.L, a.H);
  const int split_chunks = (tiles + nsplit - 1) / nsplit;
  const long img_offset = n_bh * nsplit * static_cast<long>(D) * 2 * D;
  l2_tc_moments<D><<<static_cast<unsigned>(n_bh * nsplit), kP1Threads, P1<D>::BYTES, stream>>>(
      a, nsplit, split_chunks * kC, tk, tv);
  note_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the reduce and the readout are programmatic dependents of the launch before them: each starts
  // while its predecessor finishes and waits for it (griddepcontrol.wait) before reading its output
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  const int q4 = D * 2 * D / 4;
  cfg.gridDim = dim3(static_cast<unsigned>((q4 + 255) / 256), static_cast<unsigned>(n_bh));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, l2_tc_reduce<D>, static_cast<const float*>(a.ws), nsplit, img_offset);
  note_launches(1);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(n_bh * nsplit));
  cfg.blockDim = dim3(kP2Threads);
  cfg.dynamicSmemBytes = P2<D>::BYTES;
  e = cudaLaunchKernelEx(&cfg, l2_tc_readout<D>, a, nsplit, split_chunks, img_offset, tq, to);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool l2_tc_supported(DType dt, int d) { return dt == DType::BF16 && (d == 64 || d == 128); }

size_t l2_tc_workspace_bytes(int B, int L, int H, int d) {
  const long n_bh = static_cast<long>(B) * H;
  const long mat = static_cast<long>(d) * 2 * d;
  return static_cast<size_t>(n_bh * l2_tc_splits(B, L, H) * mat * 4 + n_bh * mat * 2);
}

namespace {
template <int D>
cudaError_t launch_moments_split_d(const L2Args& a, int nsplit, int split_len, cudaStream_t stream) {
  static unsigned long long cfg1 = 0;
  cudaError_t e = set_smem(l2_tc_moments<D>, P1<D>::BYTES, cfg1);
  if (e != cudaSuccess) return e;
  const long n_bh = static_cast<long>(a.B) * a.H;
  if (n_bh == 0 || a.L == 0 || nsplit == 0) return cudaSuccess;
  CUtensorMap tk, tv;
  e = make_bshd_map(&tk, a.k, a.B, a.L, a.H, D);
  if (e == cudaSuccess) e = make_bshd_map(&tv, a.v, a.B, a.L, a.H, D);
  if (e != cudaSuccess) return e;
  l2_tc_moments<D><<<static_cast<unsigned>(n_bh * nsplit), kP1Threads, P1<D>::BYTES, stream>>>(
      a, nsplit, split_len, tk, tv);
  note_launches(1);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_l2_moments_tc(int d, const L2Args& a, int nsplit, int split_len, cudaStream_t stream) {
  return d == 128 ? launch_moments_split_d<128>(a, nsplit, split_len, stream)
                  : launch_moments_split_d<64>(a, nsplit, split_len, stream);
}

cudaError_t launch_rla_l2_tc(int d, const L2Args& a, cudaStream_t stream) {
  return d == 128 ? launch_l2_tc_d<128>(a, stream) : launch_l2_tc_d<64>(a, stream);
}

namespace {
template <int D>
cudaError_t launch_moments_plain_d(const L2Args& a, float* M, cudaStream_t stream) {
  static unsigned long long cfg1 = 0;
  cudaError_t e = set_smem(l2_tc_moments<D>, P1<D>::BYTES, cfg1);
  if (e != cudaSuccess) return e;
  const long n_bh = static_cast<long>(a.B) * a.H;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  CUtensorMap tk, tv;
  e = make_bshd_map(&tk, a.k, a.B, a.L, a.H, D);
  if (e == cudaSuccess) e = make_bshd_map(&tv, a.v, a.B, a.L, a.H, D);
  if (e != cudaSuccess) return e;
  const int tiles = (a.L + kC - 1) / kC;
  const int nsplit = l2_tc_splits(a.B, a.L, a.H);
  const int split_chunks = (tiles + nsplit - 1) / nsplit;
  l2_tc_moments<D><<<static_cast<unsigned>(n_bh * nsplit), kP1Threads, P1<D>::BYTES, stream>>>(
      a, nsplit, split_chunks * kC, tk, tv);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int q4 = D * 2 * D / 4;
  l2_tc_plain<D><<<dim3(static_cast<unsigned>((q4 + 255) / 256), static_cast<unsigned>(n_bh)), 256, 0,
                   stream>>>(a.ws, nsplit, M);
  note_launches(1);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_readout_plain_d(const L2Args& a, const float* M, cudaStream_t stream) {
  static unsigned long long cfg2 = 0;
  cudaError_t e = set_smem(l2_tc_readout<D>, P2<D>::BYTES, cfg2);
  if (e != cudaSuccess) return e;
  const long n_bh = static_cast<long>(a.B) * a.H;
  if (n_bh == 0 || a.L == 0) return cudaSuccess;
  CUtensorMap tq, to;
  e = make_bshd_map(&tq, a.q, a.B, a.L, a.H, D);
  if (e == cudaSuccess) e = make_bshd_map(&to, a.out, a.B, a.L, a.H, D);
  if (e != cudaSuccess) return e;
  const int tiles = (a.L + kC - 1) / kC;
  const int nsplit = l2_tc_splits(a.B, a.L, a.H);
  const int split_chunks = (tiles + nsplit - 1) / nsplit;
  const int q4 = D * 2 * D / 4;
  l2_tc_image<D><<<dim3(static_cast<unsigned>((q4 + 255) / 256), static_cast<unsigned>(n_bh)), 256, 0,
                   stream>>>(M, reinterpret_cast<uint8_t*>(a.ws));
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the readout is a programmatic dependent of the image launch (set-up and q tiles overlap it)
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(n_bh * nsplit));
  cfg.blockDim = dim3(kP2Threads);
  cfg.dynamicSmemBytes = P2<D>::BYTES;
  e = cudaLaunchKernelEx(&cfg, l2_tc_readout<D>, a, nsplit, split_chunks, 0L, tq, to);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

size_t l2_tc_moments_ws_bytes(int B, int L, int H, int d) {
  return static_cast<size_t>(B) * H * l2_tc_splits(B, L, H) * d * 2 * d * sizeof(float);
}
size_t l2_tc_readout_ws_bytes(int B, int H, int d) {
  return static_cast<size_t>(B) * H * d * 2 * d * 2;
}
cudaError_t launch_l2_tc_moments_plain(int d, const L2Args& a, float* M, cudaStream_t stream) {
  return d == 128 ? launch_moments_plain_d<128>(a, M, stream) : launch_moments_plain_d<64>(a, M, stream);
}
cudaError_t launch_l2_tc_readout_plain(int d, const L2Args& a, const float* M, cudaStream_t stream) {
  return d == 128 ? launch_readout_plain_d<128>(a, M, stream) : launch_readout_plain_d<64>(a, M, stream);
}

}  // namespace rapt
