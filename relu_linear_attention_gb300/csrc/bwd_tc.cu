// Backward of causal RLA-2 on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a; bf16
// tensors, d = 64 or 128, fp32 accumulation and fp32 states. The passes keep 128-column tiles in
// shared memory; at d = 64 only the first 64-column block of a streamed tile is loaded (the second
// is cleared once), the products whose output has d columns run with N = d and those that contract
// over the features with K = d, and the state records keep the 128 x 128 layout.
//
// The gradients of sum dout . out (08-rapt-algorithm.md §4.2 "backward": the main and z scans,
// gnum = g / den and scale = -(g . num) / den^2, two suffix scans, then ReLU, RoPE and RMSNorm
// backwards) in chunked form, C = 128 tokens per chunk (the MMA's M), in seven launches. First,
// fully parallel over (document, head, chunk): q' and k' (bf16) of every row into the workspace
// (bwd_tc_featmap). Documents are cut into segments; the prefix state at each segment's start is the
// sum of per-block increments S = sum k'v^T, z = sum k' of the blocks before it (bwd_tc_blockstate
// <true>). Per document, head and segment:
//
// Pass A (chunks in order; prefix state S = sum k'v^T in TMEM, its bf16 copy S~ in shared memory):
//   P  = Q'K'^T,  Cv = G V^T,  U = G S~^T,  S += K'^T V                     (one MMA group)
//   per row t: den = q'.z + sum_{tau<=t} P + eps,  nst = q'_t . U_t = g_t . (q'_t S~),
//              pc = sum_{tau<=t} P Cv,  scale = -(nst + pc) / den^2
//   A'[t][tau] = (c ps - pc + c sst - nst + eps c) / den  (c = Cv[t][tau], ps = sum P, sst = q'.z)
//              = den (gnum_t . v_tau + scale_t), in the form whose cancelling part is exact for a
//              query that sees a single key (see backward_simt.cu)
//   U += A'~ K'                                                                (second MMA group)
//   dq'_t = U_t / den_t + scale_t z (bf16, to the workspace); den, scale, sst, nst of every row go
//   to the workspace for pass B.
// Between the passes, the suffix state at each segment's end is the sum of per-block increments
// R = sum q' gnum^T, w = sum scale q' of the later blocks (bwd_tc_blockstate<false>).
// Pass B (chunks in reverse; suffix state R = sum q' gnum^T in TMEM, bf16 copy R~, w = sum scale q'):
//   P = Q'K'^T,  Cv = G V^T (raw bf16 g and v: c exact)                    (first group)
//   then, while gnum = g / den, P~ and A are formed:  dv = K' R~
//   P~ = P masked to tau <= t;  A[t][tau] = A'/den
//   dv += P~^T Gnum,  R += Q'^T Gnum,  dk' = V R~^T                          (second group)
//   dk' += A^T Q' (+ w)                                                      (third group)
//   dk' (bf16) to the workspace, dv out.
// The passes stage a whole chunk's dq' (pass A) and dk', dv (pass B) in shared memory that the
// chunk's MMAs no longer read and write them with TMA tile stores; a document's ragged last chunk
// is written row by row.
// Then, fully parallel over (document, head, chunk), dq and dk through the feature map (ReLU mask,
// inverse RoPE rotation, RMSNorm backward) from dq', dk' and the raw q, k, with gain partials
// (bwd_tc_features, one launch per tensor: dq's runs beside pass B on the caller's stream while the
// rest runs on a stream of higher priority), and the gains summed in a fixed order. With packed
// documents the passes take the documents longest first.
// The passes run one CTA per (document, head, segment) with 512 worker threads in lockstep phases:
// they read TMEM rows (thread = TMEM lane = tile row, four warps per lane quarter splitting the
// columns) and do the per-row arithmetic. In pass B one of them issues the MMAs and the TMA copies
// of the next chunk's tiles and commits them to mbarriers; pass A has a 17th warp for that, which
// waits on mbarriers the workers arrive at (rows cleared, A' written, S~ written), so the first
// products overlap the workers' row sums. Every wait is bounded (~1 s); a CTA whose wait gives up
// sets RAPT_DEV_INTERNAL in the status word and writes NaN results, so a failure cannot pass for one.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "feature_bwd.cuh"
#include "kernels.h"
#include "tc_features.cuh"
#include "tc_tiles.cuh"
#include "tc_utils.cuh"
#include "tensor_map.h"

namespace rapt {
namespace {

using feat::doc_bounds;
using feat::lds16;
using feat::ldg16;
using feat::sts16;
using namespace tct;

constexpr int kC = 128;
constexpr int kThreads = 512;               // the lockstep worker threads (16 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kThreadsA = kThreads + 32;     // pass A: + one warp that issues the MMAs and loads
constexpr uint32_t kBarWork = 1;             // named barrier of pass A's worker warps
constexpr uint32_t kTile = 32768;          // 128 rows x 128 bf16 columns (two 64-column blocks)

// Shared memory (bytes from a 1024-byte aligned base). Both passes use the same map: six bf16
// tiles (the fifth, XS, holds S~ in pass A and R~ in pass B; the last, AS, holds A' in pass A and
// P~ then A in pass B), then fp32 vectors.
struct Lay {
  static constexpr uint32_t QF = 0, KF = kTile, VS = 2 * kTile, GS = 3 * kTile, XS = 4 * kTile;
  static constexpr uint32_t AS = 5 * kTile;
  static constexpr uint32_t ZS = 6 * kTile;                   // z (pass A) / w (pass B) [D]
  static constexpr uint32_t ZP = ZS + kD * 4;                 // per-warp k' column sums [16][D]
  static constexpr uint32_t ROW = ZP + kWarps * kD * 4;       // den, scale, sst, nst [4][128]
  static constexpr uint32_t RED = ROW + 4 * kC * 4;           // partial row sums [3][4][128]
  static constexpr uint32_t BAR = RED + 3 * 4 * kC * 4;       // eight mbarriers
  static constexpr uint32_t MISC = BAR + 8 * 8;               // TMEM base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

// TMEM columns.
constexpr uint32_t kTP = 0, kTG = 128, kTU = 256, kTS = 384;  // pass A: P, Cv, U, S
constexpr uint32_t kTDV = 384, kTDK = 0, kTR = 256;           // pass B: dv, dk' (over P), R

// Features of the chunk's 128 rows of x (q or k) into a bf16 tile: warp w takes rows w, w + 16, ...
// (FeatureLayout: lane r owns elements 4r .. 4r+3); the loads of all its rows are issued before
// any is used. With z given, also q'_t . z of every row into sst[]; the lane's column sums of the
// features are added to zc; with out given, the bf16 features of the valid rows are stored there
// ([T, H, D], for pass B).
constexpr int kRPW = kC / kWarps;  // rows per warp

constexpr int kRB = kRPW / 2;  // rows of a warp loaded together (two batches per tile)


// One chunk's 128 rows of nt [rows, H, D] tensors into their tiles by TMA (two 64-column boxes
// each, in the swizzled operand layout), completing on one mbarrier; one thread calls it. Rows
// past the tensor read as zero; rows past the document but inside the tensor are other tokens,
// which the caller clears after the wait.
template <int NT, int D>
__device__ __forceinline__ void tma_chunk(const CUtensorMap* const (&maps)[NT],
                                          const uint32_t (&tiles)[NT], int h, int row, uint32_t bar) {
  tc::mbar_arrive_expect_tx(bar, NT * kC * D * 2);
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int jb = 0; jb < D / 64; ++jb) tc::tma_load_3d(tiles[i] + jb * 16384, maps[i], 64 * jb, h, row, bar);
}

// The same rows fetched into L2 only (no shared memory, no completion), a chunk before their load:
// the load, which must wait until the chunk before has read its tiles, then finds them there.
template <int NT, int D>
__device__ __forceinline__ void prefetch_chunk(const CUtensorMap* const (&maps)[NT], int h, int row) {
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int jb = 0; jb < D / 64; ++jb) tc::tma_prefetch_3d(maps[i], 64 * jb, h, row);
}

// At d = 64 the second 64-column block of the streamed tiles (QF, KF, VS, GS: the first four) is
// never loaded: it is cleared once, so that the products whose M runs over the 128 feature rows
// (K'^T V, Q'^T Gnum) see zeros there. The worker threads call it.
template <int D>
__device__ __forceinline__ void clear_upper_blocks(uint32_t base) {
  if (D == 64) {
    for (int idx = threadIdx.x; idx < 4 * 1024; idx += kThreads)
      feat::sts16(base + (idx >> 10) * kTile + 16384 + 16 * (idx & 1023), make_uint4(0, 0, 0, 0));
  }
}

// The per-row phases on the d feature columns give each of the four column groups W = d / 4 of
// them: W consecutive fp32 TMEM columns of this thread's lane (two such reads in flight together
// in the x2 form), and W values as bf16 into row r, columns W g .. W g + W - 1 of a tile.
template <int W>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float (&v)[W]) {
  if constexpr (W == 32) {
    tmem_ld32(taddr, v);
  } else {
    uint32_t u[16];
    tc::tmem_ld16(taddr, u);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(u[e]);
  }
}
template <int W>
__device__ __forceinline__ void tmem_ldnx2(uint32_t ta, float (&va)[W], uint32_t tb, float (&vb)[W]) {
  if constexpr (W == 32) {
    tmem_ld32x2(ta, va, tb, vb);
  } else {
    uint32_t u[2][16];
    tc::tmem_ld16(ta, u[0]);
    tc::tmem_ld16(tb, u[1]);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      va[e] = __uint_as_float(u[0][e]);
      vb[e] = __uint_as_float(u[1][e]);
    }
  }
}
template <bool DROWS, int W>
__device__ __forceinline__ void store_rown(uint32_t tile, int r, int g, const float (&v)[W]) {
#pragma unroll
  for (int m = 0; m < W / 8; ++m) {
    const int ch = (W / 8) * g + m;
    feat::sts16(tile + (DROWS ? dtile_off(r, ch) : tile_off(r, ch)), feat::pack8(v + 8 * m));
  }
}

// Rows nvalid .. 127 of a tile set to zero (all threads).
__device__ __forceinline__ void clear_rows(uint32_t tile, int nvalid) {
  for (int idx = threadIdx.x + nvalid * 16; idx < kC * 16; idx += kThreads)
    sts16(tile + tile_off(idx >> 4, idx & 15), make_uint4(0, 0, 0, 0));
}

// Sums over the features of a chunk (bf16 in the tile, by TMA from the workspace; warp w takes rows
// w, w + 16, ...): with z given, q'.z of every row into sst[] (zero past
// the document); the column sums of the rows inside the document are added to zc.
template <int D>
__device__ __forceinline__ void feature_sums(uint32_t tile, int n, int t0, const float* z, float* sst,
                                             float (&zc)[4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // d = 128: a row per warp load, lane r on elements 4r .. 4r+3; d = 64: two rows per load, one
  // per half warp
  constexpr int RPL = D == 64 ? 2 : 1;
  const int sub = D == 64 ? lane >> 4 : 0, cl = D == 64 ? lane & 15 : lane;
  float zl[4] = {0.f, 0.f, 0.f, 0.f};
  if (z != nullptr) {
    const float4 zz = *reinterpret_cast<const float4*>(z + 4 * cl);
    zl[0] = zz.x; zl[1] = zz.y; zl[2] = zz.z; zl[3] = zz.w;
  }
  constexpr int NL = kRPW / RPL;  // loads per warp
#pragma unroll 1
  for (int i0 = 0; i0 < NL; i0 += kRB) {
    uint32_t lo[kRB], hi[kRB];
#pragma unroll
    for (int i = 0; i < kRB; ++i) {
      const int rr = warp + kWarps * (RPL * (i0 + i) + sub);
      const uint32_t addr = tile + tile_off(rr, cl >> 1) + (cl & 1) * 8;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(lo[i]), "=r"(hi[i]) : "r"(addr) : "memory");
    }
#pragma unroll
    for (int i = 0; i < kRB; ++i) {
      const int rr = warp + kWarps * (RPL * (i0 + i) + sub);
      const bool valid = t0 + rr < n;
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&lo[i]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi[i]));
      const float f[4] = {valid ? a.x : 0.f, valid ? a.y : 0.f, valid ? b.x : 0.f, valid ? b.y : 0.f};
      if (z != nullptr) {
        float sdot = f[0] * zl[0] + f[1] * zl[1] + f[2] * zl[2] + f[3] * zl[3];
#pragma unroll
        for (int off = D == 64 ? 8 : 16; off > 0; off >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, off);
        if (cl == 0) sst[rr] = sdot;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) zc[e] += f[e];
    }
  }
  if (D == 64) {  // both halves' rows of the same columns
#pragma unroll
    for (int e = 0; e < 4; ++e) zc[e] += __shfl_xor_sync(0xffffffffu, zc[e], 16);
  }
}

// ------------------------------------------------------------------------------------------------
// Pass A: chunks in order.
template <int D>
__global__ void __launch_bounds__(kThreadsA, 1)
    bwd_tc_forward(const BwdArgs b, const __grid_constant__ CUtensorMap tmqf,
                   const __grid_constant__ CUtensorMap tmkf, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmdq) {
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % b.nseg, slot = blockIdx.x / b.nseg;  // packed: longest first
  const int h = slot % a.H, doc = b.order != nullptr ? b.order[slot / a.H] : slot / a.H;
  const int unit = doc * a.H + h;
  long row0;
  int n;
  if (!doc_bounds(a, doc, row0, n) && h == 0 && seg == 0 && tid == 0 && a.dev_status != nullptr)
    atomicOr(a.dev_status, 1u);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  const int nch = s1 > s0 ? (s1 - s0 + kC - 1) / kC : 0;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  float* zs = reinterpret_cast<float*>(smem + Lay::ZS);
  float* zp = reinterpret_cast<float*>(smem + Lay::ZP);
  float* den_s = reinterpret_cast<float*>(smem + Lay::ROW);
  float* scl_s = den_s + kC;
  float* sst_s = scl_s + kC;
  float* red = reinterpret_cast<float*>(smem + Lay::RED);
  const uint32_t bar1 = base + Lay::BAR, bar2 = bar1 + 8, bar1b = bar1 + 16, bar_ld = bar1 + 24;
  // worker warps -> issuer: the chunk's tiles cleared (ready), A' written (a_ready), S~ written and
  // S read (s_ready; completion 0 is the segment's initial state)
  const uint32_t bar_ready = bar1 + 32, bar_aready = bar1 + 40, bar_sready = bar1 + 48;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Lay::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + Lay::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;

  if (warp == 0 && !misaligned && nch > 0) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar1, 1);
    tc::mbar_init(bar2, 1);
    tc::mbar_init(bar1b, 1);
    tc::mbar_init(bar_ld, 1);
    tc::mbar_init(bar_ready, kWarps);
    tc::mbar_init(bar_aready, kWarps);
    tc::mbar_init(bar_sready, kWarps);
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int q4 = warp & 3, gw = warp >> 2;  // TMEM lane quarter, column group (32 columns)
  const int t = 32 * q4 + lane;             // this thread's tile row (= TMEM lane)
  const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
  // the first chunk's tiles are requested before the state is summed (they do not overlap it)
  const CUtensorMap* const maps[4] = {&tmqf, &tmkf, &tmv, &tmg};
  const uint32_t ld_tiles[4] = {base + Lay::QF, base + Lay::KF, base + Lay::VS, base + Lay::GS};
  if (tid == 0 && nch > 0 && !*s_abort) tma_chunk<4, D>(maps, ld_tiles, h, static_cast<int>(row0 + s0), bar_ld);
  // the prefix state at the segment's start: the increments of the blocks before it, in order
  // (the worker warps: lane quarter q4, column group gw < 4; the issuing warp takes no part)
  constexpr int GD = D / 32;  // column groups of 32 that hold one of the d feature columns
  constexpr int W = D / 4;    // d columns per column group in the per-row phases
  if (nch > 0 && warp < kWarps) {
    clear_upper_blocks<D>(base);
    const int nb = seg * b.blk_per_seg;
    constexpr long R4 = static_cast<long>(kD) * (kD + 1) / 4;
    const float4* rec = reinterpret_cast<const float4*>(b.rec_fwd) + static_cast<long>(unit) * b.nblk_max * R4;
    float sv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) sv[e] = 0.f;
#pragma unroll 2  // two records' loads in flight together
    for (int blk = 0; blk < (D == 128 || gw < GD ? nb : 0); ++blk) {
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float4 x = __ldcg(rec + blk * R4 + (8 * gw + jj) * kD + t);
        sv[4 * jj] += x.x; sv[4 * jj + 1] += x.y; sv[4 * jj + 2] += x.z; sv[4 * jj + 3] += x.w;
      }
    }
    state_put(tmem + tl + kTS + 32 * gw, base + Lay::XS, t, gw, sv);
    if (tid < kD) {
      float z = 0.f;
      for (int blk = 0; blk < nb; ++blk) z += __ldcg(b.rec_fwd + (static_cast<long>(unit) * b.nblk_max + blk) * (R4 * 4) + kD * kD + tid);
      zs[tid] = z;
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  __nv_bfloat16* dqf_out = static_cast<__nv_bfloat16*>(b.dqf);
  bool bad = *s_abort != 0;

  if (warp == kWarps) {
    // ============================================ MMA issue and tile loads (one thread)
    if (lane == 0) {
      // the products with d output columns have N = d
      constexpr uint32_t ID_KK = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_U = tc::idesc_bf16(128, D, false, false);
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, D, true, true);
      constexpr uint32_t ID = tc::idesc_bf16(128, D, false, true);
      bool ok = !bad;  // false only once a wait has given up
      int loads = 0;
      for (int c = 0; c < nch && ok; ++c) {
        const int t0 = s0 + c * kC;
        // P = Q'K'^T, Cv = G V^T once the workers have cleared the rows past the document
        ok = tc::mbar_wait(bar_ready, c & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          tc::mma_bf16(tmem + kTP, kmaj(base + Lay::QF, kk), kmaj(base + Lay::KF, kk), ID_KK, kk > 0);
          tc::mma_bf16(tmem + kTG, kmaj(base + Lay::GS, kk), kmaj(base + Lay::VS, kk), ID_KK, kk > 0);
        }
        tc::mma_commit(bar1);  // P and Cv: the row sums can start
        // U = G S~^T and S += K'^T V once the previous chunk has read U and S and written S~
        ok = tc::mbar_wait(bar_sready, c & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_bf16(tmem + kTU, kmaj(base + Lay::GS, kk), kmaj_d(base + Lay::XS, kk), ID_U, kk > 0);
        tc::mma_commit(bar1b);
#pragma unroll 1
        for (int kk = 0; kk < kC / 16; ++kk)
          tc::mma_bf16(tmem + kTS, mnmaj(base + Lay::KF, kk, 16384), mnmaj(base + Lay::VS, kk, 16384),
                       ID_MM, 1u);
        // U += A'~ K' once A' is written
        ok = tc::mbar_wait(bar_aready, c & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int kk = 0; kk < kC / 16; ++kk)
          tc::mma_bf16(tmem + kTU, kmaj(base + Lay::AS, kk), mnmaj(base + Lay::KF, kk, 16384), ID, 1u);
        tc::mma_commit(bar2);
        // every MMA and every worker (A' was their last read of q') is done with the tiles: the
        // next chunk's may arrive while this one finishes
        if (c + 1 < nch) {
          ok = tc::mbar_wait(bar2, c & 1, kWait);
          if (!ok || *reinterpret_cast<volatile int*>(s_abort)) break;
          tma_chunk<4, D>(maps, ld_tiles, h, static_cast<int>(row0 + t0 + kC), bar_ld);
          ++loads;
        }
      }
      if (!ok) atomicExch(s_abort, 1);
      // a copy requested but not waited for (an early exit) must land before the CTA leaves: this
      // thread's load k (from 1; chunk 0's was the worker's) completes bar_ld's phase k
      if (loads > 0) tc::mbar_wait(bar_ld, loads & 1, kWait);
    }
  } else {
  if (!bad && nch > 0) {  // the initial S~ is written (completion 0 of s_ready)
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar_sready);
  }
  for (int c = 0; c < nch && !bad; ++c) {
    const int t0 = s0 + c * kC;
    // ---- phase 1: the chunk's tiles (TMA; q' and k' from the feature kernel); q'.z of every
    // row and the column sums of k'; rows past the document cleared
    if (!tc::mbar_wait(bar_ld, c & 1, kWait)) atomicExch(s_abort, 1);
    if (tid == 0 && c + 1 < nch) prefetch_chunk<4, D>(maps, h, static_cast<int>(row0 + t0 + kC));
    if (t0 + kC > n) {  // uniform over the CTA
      clear_rows(base + Lay::QF, n - t0);
      clear_rows(base + Lay::KF, n - t0);
      clear_rows(base + Lay::VS, n - t0);
      clear_rows(base + Lay::GS, n - t0);
      tc::fence_async_smem();
      tc::named_sync(kBarWork, kThreads);
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar_ready);  // the first products may start
    float zc[4] = {0.f, 0.f, 0.f, 0.f}, dummy[4] = {0.f, 0.f, 0.f, 0.f};
    feature_sums<D>(base + Lay::QF, n, t0, zs, sst_s, dummy);
    feature_sums<D>(base + Lay::KF, n, t0, nullptr, nullptr, zc);
    if (4 * lane < D) {
#pragma unroll
      for (int e = 0; e < 4; ++e) zp[warp * kD + 4 * lane + e] = zc[e];
    }
    if (tid == 0) tc::bulk_wait_read0();  // the previous chunk's dq' store has read AS
    tc::fence_async_smem();
    tc::fence_before_sync();
    tc::named_sync(kBarWork, kThreads);
    tc::fence_after_sync();
    // ---- phase 2 (the issuing warp): P = Q'K'^T, Cv = G V^T, U = G S~^T, S += K'^T V
    if (!wait_mma(bar1, c & 1)) atomicExch(s_abort, 1);
    // ---- phase 3: row sums, den, scale, A'
    const bool valid = t0 + t < n;
    float pv[32], cv[32];
    tmem_ld32x2(tmem + tl + kTP + 32 * gw, pv, tmem + tl + kTG + 32 * gw, cv);
    float ps = 0.f, pc = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool vis = 32 * gw + j <= t;
      ps += vis ? pv[j] : 0.f;
      pc += vis ? pv[j] * cv[j] : 0.f;
    }
    float nst = 0.f;
    if (!wait_mma(bar1b, c & 1)) atomicExch(s_abort, 1);
    {  // U has d columns
      float u[W];
      tmem_ldn<W>(tmem + tl + kTU + W * gw, u);
#pragma unroll
      for (int m = 0; m < W / 8; ++m) {
        float f[8];
        unpack8(lds16(base + Lay::QF + tile_off(t, (W / 8) * gw + m)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) nst += f[e] * u[8 * m + e];
      }
    }
    red[(0 * 4 + gw) * kC + t] = ps;
    red[(1 * 4 + gw) * kC + t] = pc;
    red[(2 * 4 + gw) * kC + t] = nst;
    tc::fence_before_sync();
    tc::named_sync(kBarWork, kThreads);
    ps = red[t] + red[kC + t] + red[2 * kC + t] + red[3 * kC + t];
    pc = red[4 * kC + t] + red[5 * kC + t] + red[6 * kC + t] + red[7 * kC + t];
    nst = red[8 * kC + t] + red[9 * kC + t] + red[10 * kC + t] + red[11 * kC + t];
    const float sst = sst_s[t];
    const float den = valid ? sst + ps + a.eps_den : 1.f;
    const float scale = valid ? -(nst + pc) / (den * den) : 0.f;
    if (gw == 0) {
      den_s[t] = den;
      scl_s[t] = scale;
      if (valid) {
        const long o = (row0 + t0 + t) * a.H + h;
        b.den[o] = den;
        b.scl[o] = scale;
        b.sst[o] = sst;
        b.nst[o] = nst;
      }
    }
    {
      const float inv = 1.0f / den;
      float av[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float cc = cv[j];
        const float num = (cc * ps - pc) + (fmaf(cc, sst, -nst) + a.eps_den * cc);
        av[j] = (32 * gw + j <= t) ? num * inv : 0.f;
      }
      store_row32<false>(base + Lay::AS, t, gw, av);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar_aready);  // every read of q' is done, A' is written
    // ---- phase 4 (the issuing warp): U += A'~ K'; then the next chunk's tiles
    if (!wait_mma(bar2, c & 1)) atomicExch(s_abort, 1);
    // ---- phase 5: dq' = U / den + scale z (bf16, to the workspace); S -> S~ (d columns)
    {
      float u[W], sv[W];
      tmem_ldnx2<W>(tmem + tl + kTU + W * gw, u, tmem + tl + kTS + W * gw, sv);
      const float inv = 1.0f / den;
#pragma unroll
      for (int j = 0; j < W; ++j) u[j] = fmaf(u[j], inv, scale * zs[W * gw + j]);
      if (t0 + kC <= n) {  // a whole chunk: staged in AS (its last reader, phase 4, is done)
        store_rown<false, W>(base + Lay::AS, t, gw, u);
      } else if (valid && (D == 64 || gw < b.d / 32)) {  // the ragged last chunk row by row
        __nv_bfloat16* dst = dqf_out + ((row0 + t0 + t) * a.H + h) * b.d + W * gw;
#pragma unroll
        for (int m = 0; m < W / 8; ++m) *reinterpret_cast<uint4*>(dst + 8 * m) = feat::pack8(u + 8 * m);
      }
      if (D == 128 || t < D) store_rown<true, W>(base + Lay::XS, t, gw, sv);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar_sready);  // U and S read, S~ written: the next products
    tc::named_sync(kBarWork, kThreads);
    if (tid == 0 && t0 + kC <= n) {
#pragma unroll
      for (int jb = 0; jb < D / 64; ++jb)
        tc::tma_store_3d(&tmdq, base + Lay::AS + jb * 16384, 64 * jb, h, static_cast<int>(row0 + t0));
      tc::bulk_commit();
    }
    // ---- phase 6: z += column sums of k'
    if (tid < D) {
      float zz = zs[tid];
      for (int w = 0; w < kWarps; ++w) zz += zp[w * kD + tid];
      zs[tid] = zz;
    }
    // zs is read before the next chunk uses it; the workers leave together
    if (feat::group_sync_or(kBarWork, kThreads, *reinterpret_cast<volatile int*>(s_abort))) {
      bad = true;
      break;
    }
  }
  if (tid == 0) tc::bulk_wait0();  // the dq' tile stores are complete before the NaN fill or exit
  }
  __syncthreads();
  bad = *reinterpret_cast<volatile int*>(s_abort) != 0;
  if (bad) {  // a wait gave up: NaN dq' over the segment, so the failure cannot pass for a result
    const int cpr = b.d / 8;  // 16-byte chunks per row
    for (long r = s0 + tid / cpr; r < s1; r += kThreads / cpr)
      *reinterpret_cast<uint4*>(dqf_out + ((row0 + r) * a.H + h) * b.d + 8 * (tid % cpr)) =
          make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0 && !misaligned && nch > 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// Pass B: chunks in reverse.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_reverse(const BwdArgs b, const __grid_constant__ CUtensorMap tmqf,
                   const __grid_constant__ CUtensorMap tmkf, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmdv,
                   const __grid_constant__ CUtensorMap tmdk) {
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % b.nseg, slot = blockIdx.x / b.nseg;  // packed: longest first
  const int h = slot % a.H, doc = b.order != nullptr ? b.order[slot / a.H] : slot / a.H;
  const int unit = doc * a.H + h;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int s0 = seg * b.seg_len, s1 = min(n, s0 + b.seg_len);
  const int nch = s1 > s0 ? (s1 - s0 + kC - 1) / kC : 0;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  float* ws = reinterpret_cast<float*>(smem + Lay::ZS);  // w
  float* den_s = reinterpret_cast<float*>(smem + Lay::ROW);
  float* scl_s = den_s + kC;
  float* sst_s = scl_s + kC;
  float* nst_s = sst_s + kC;
  float* red = reinterpret_cast<float*>(smem + Lay::RED);
  const uint32_t bar1 = base + Lay::BAR, bar2 = bar1 + 8, bar3 = bar2 + 8, bar4 = bar3 + 8;
  const uint32_t bar_ld = bar4 + 8;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Lay::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + Lay::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;

  if (warp == 0 && !misaligned && nch > 0) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar1, 1);
    tc::mbar_init(bar2, 1);
    tc::mbar_init(bar3, 1);
    tc::mbar_init(bar4, 1);
    tc::mbar_init(bar_ld, 1);
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int q4 = warp & 3, gw = warp >> 2;
  const int t = 32 * q4 + lane;
  const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
  // the tiles arrive in two groups, each as soon as the previous chunk's MMAs are done with them:
  // k', v, gnum after the dv group (bar_ld), q' after the last group (bar4); the first chunk's
  // are requested before the suffix state is summed (they do not overlap it)
  const CUtensorMap* const maps3[3] = {&tmkf, &tmv, &tmg};
  const uint32_t ld_tiles3[3] = {base + Lay::KF, base + Lay::VS, base + Lay::GS};
  const CUtensorMap* const maps1[1] = {&tmqf};
  const uint32_t ld_tiles1[1] = {base + Lay::QF};
  const uint32_t bar_ldq = bar4;
  int tma_issued = 0, tmaq_issued = 0;  // chunks whose tiles have been requested (thread 0)
  if (tid == 0 && nch > 0 && !*s_abort) {
    tma_chunk<3, D>(maps3, ld_tiles3, h, static_cast<int>(row0 + s0 + (nch - 1) * kC), bar_ld);
    tma_chunk<1, D>(maps1, ld_tiles1, h, static_cast<int>(row0 + s0 + (nch - 1) * kC), bar_ldq);
    tma_issued = tmaq_issued = 1;
  }
  constexpr int GD = D / 32;  // column groups of 32 that hold one of the d feature columns
  constexpr int W = D / 4;    // d columns per column group in the per-row phases
  clear_upper_blocks<D>(base);
  // the suffix state at the segment's end: the later segments' increments, in segment order
  if (nch > 0) {
    constexpr long REC = static_cast<long>(kD) * kD + kD;
    // the records of the blocks that start inside the document, in block order
    const int rlen = b.seg_len / b.rblk_per_seg;
    const float* rr = b.rec_rev + static_cast<long>(unit) * b.nseg * b.rblk_per_seg * REC;
    const int k0 = (seg + 1) * b.rblk_per_seg, k1 = min(b.nseg * b.rblk_per_seg, (n + rlen - 1) / rlen);
    float rv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) rv[e] = 0.f;
#pragma unroll 2  // two records' loads in flight together
    for (int kb = k0; kb < (D == 128 || gw < GD ? k1 : k0); ++kb) {
      const float4* src = reinterpret_cast<const float4*>(rr + kb * REC + t * kD + 32 * gw);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float4 x = __ldcg(src + jj);
        rv[4 * jj] += x.x; rv[4 * jj + 1] += x.y; rv[4 * jj + 2] += x.z; rv[4 * jj + 3] += x.w;
      }
    }
    state_put(tmem + tl + kTR + 32 * gw, base + Lay::XS, t, gw, rv);
    if (tid < kD) {
      float w = 0.f;
      for (int kb = k0; kb < k1; ++kb) w += __ldcg(rr + kb * REC + kD * kD + tid);
      ws[tid] = w;
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(b.dv);
  __nv_bfloat16* dkf_out = static_cast<__nv_bfloat16*>(b.dkf);
  bool bad = *s_abort != 0;
  int it = 0;  // chunks done (the mbarrier phases)

  // the row scalars of pass A (den, scale, sst, nst) of a chunk, loaded one chunk ahead
  auto row_scalars = [&](int tc0, float (&v)[4]) {
    const bool vr = tid < kC && tc0 + tid < n;
    const long o = (row0 + tc0 + tid) * a.H + h;
    v[0] = vr ? __ldg(b.den + o) : 1.f;
    v[1] = vr ? __ldg(b.scl + o) : 0.f;
    v[2] = vr ? __ldg(b.sst + o) : 0.f;
    v[3] = vr ? __ldg(b.nst + o) : 0.f;
  };
  float rs_next[4];
  row_scalars(s0 + (nch - 1) * kC, rs_next);
  for (int c = nch - 1; c >= 0 && !bad; --c, ++it) {
    const int t0 = s0 + c * kC;
    // ---- phase 1: q', k' (stored by pass A), v and g by TMA; the row scalars of pass A; rows
    // past the document cleared
    if (tid < kC) {
      den_s[tid] = rs_next[0];
      scl_s[tid] = rs_next[1];
      sst_s[tid] = rs_next[2];
      nst_s[tid] = rs_next[3];
    }
    if (c > 0) row_scalars(t0 - kC, rs_next);  // the earlier chunk's, one chunk ahead
    if (!tc::mbar_wait(bar_ld, it & 1, kWait) || !tc::mbar_wait(bar_ldq, it & 1, kWait))
      atomicExch(s_abort, 1);
    if (tid == 0 && c > 0) {  // the earlier chunk's tiles into L2 while this one runs
      prefetch_chunk<3, D>(maps3, h, static_cast<int>(row0 + t0 - kC));
      prefetch_chunk<1, D>(maps1, h, static_cast<int>(row0 + t0 - kC));
    }
    if (tid == 0) tc::bulk_wait_read0();  // the previous chunk's dk' store has read AS
    __syncthreads();  // den_s
    for (int idx = tid + (n - t0) * 16; idx < kC * 16; idx += kThreads) {  // (n > t0)
      const int r = idx >> 4, m = idx & 15;
      sts16(base + Lay::GS + tile_off(r, m), make_uint4(0, 0, 0, 0));
      sts16(base + Lay::QF + tile_off(r, m), make_uint4(0, 0, 0, 0));
      sts16(base + Lay::KF + tile_off(r, m), make_uint4(0, 0, 0, 0));
      sts16(base + Lay::VS + tile_off(r, m), make_uint4(0, 0, 0, 0));
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(s_abort)) { bad = true; break; }
    // ---- phase 2: P = Q'K'^T, Cv = G V^T (from the raw bf16 g and v, so that c = g . v is exact
    // to fp32 accumulation: A below is a difference of nearly equal terms for keys that few
    // queries see, the last ones of a document); then, while phase 3 runs on the CUDA cores, the
    // product that needs no P~, A or gnum: dv = K' R~
    if (tid == 0) {
      constexpr uint32_t ID = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_KM = tc::idesc_bf16(128, D, false, true);
#pragma unroll 1
      for (int kk = 0; kk < D / 16; ++kk) {
        tc::mma_bf16(tmem + kTP, kmaj(base + Lay::QF, kk), kmaj(base + Lay::KF, kk), ID, kk > 0);
        tc::mma_bf16(tmem + kTG, kmaj(base + Lay::GS, kk), kmaj(base + Lay::VS, kk), ID, kk > 0);
      }
      tc::mma_commit(bar1);
#pragma unroll 1
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_bf16(tmem + kTDV, kmaj(base + Lay::KF, kk), mnmaj(base + Lay::XS, kk, kD * 128),
                     ID_KM, kk > 0);
    }
    {  // meanwhile the partial increment of w = sum_t scale_t q'_t: column i, rows RP (tid / D) ..
       // + RP - 1, into the third section of RED (added to w once this chunk's dk' has used it)
      constexpr int RP = kC * D / kThreads;
      const int i = tid & (D - 1), r0 = RP * (tid / D);
      const int m = i >> 3, e = i & 7;
      float dw = 0.f;
#pragma unroll 4
      for (int r = r0; r < r0 + RP; ++r) {
        uint32_t word;
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(word)
                     : "r"(base + Lay::QF + tile_off(r, m) + 4 * (e >> 1))
                     : "memory");
        const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&word));
        dw = fmaf(scl_s[r], (e & 1) ? p.y : p.x, dw);
      }
      red[8 * kC + tid] = dw;  // partial tid / D of column i
    }
    if (!wait_mma(bar1, it & 1)) atomicExch(s_abort, 1);
    // ---- phase 3: gnum = g / den in place (the products that read g are done); P~ (masked) into
    // AS; A kept in registers
    for (int idx = tid; idx < kC * D / 8; idx += kThreads) {
      const int r = idx / (D / 8), m = idx % (D / 8);
      if (t0 + r < n) {
        const uint32_t ga = base + Lay::GS + tile_off(r, m);
        float f[8];
        unpack8(lds16(ga), f);
        const float inv = 1.0f / den_s[r];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= inv;
        sts16(ga, feat::pack8(f));
      }
    }
    const float den = den_s[t], sst = sst_s[t], nst = nst_s[t];
    float pv[32], av[32];
    tmem_ld32x2(tmem + tl + kTP + 32 * gw, pv, tmem + tl + kTG + 32 * gw, av);  // av: c = g . v
    float ps = 0.f, pc = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool vis = 32 * gw + j <= t;
      pv[j] = vis ? pv[j] : 0.f;
      ps += pv[j];
      pc += pv[j] * av[j];
    }
    red[(0 * 4 + gw) * kC + t] = ps;
    red[(1 * 4 + gw) * kC + t] = pc;
    store_row32<false>(base + Lay::AS, t, gw, pv);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(s_abort)) { bad = true; break; }
    ps = red[t] + red[kC + t] + red[2 * kC + t] + red[3 * kC + t];
    pc = red[4 * kC + t] + red[5 * kC + t] + red[6 * kC + t] + red[7 * kC + t];
    {
      const float inv2 = 1.0f / (den * den);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float cc = av[j];
        const float num = (cc * ps - pc) + (fmaf(cc, sst, -nst) + a.eps_den * cc);
        av[j] = (32 * gw + j <= t) ? num * inv2 : 0.f;
      }
    }
    // ---- phase 4: dv += P~^T Gnum; R += Q'^T Gnum (R~ in XS is not touched); dk' = V R~^T (over
    // P, which phase 3 has read)
    if (tid == 0) {
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, D, true, true);
      constexpr uint32_t ID_KK = tc::idesc_bf16(128, D, false, false);
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk)
        tc::mma_bf16(tmem + kTDV, mnmaj(base + Lay::AS, kk, 16384), mnmaj(base + Lay::GS, kk, 16384),
                     ID_MM, 1u);
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk)
        tc::mma_bf16(tmem + kTR, mnmaj(base + Lay::QF, kk, 16384), mnmaj(base + Lay::GS, kk, 16384),
                     ID_MM, 1u);
#pragma unroll 1
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_bf16(tmem + kTDK, kmaj(base + Lay::VS, kk), kmaj_d(base + Lay::XS, kk), ID_KK, kk > 0);
      tc::mma_commit(bar2);
    }
    if (!wait_mma(bar2, it & 1)) atomicExch(s_abort, 1);
    // k', v and gnum are read by every MMA that needs them: the earlier chunk's may arrive
    if (tid == 0 && c > 0 && !*reinterpret_cast<volatile int*>(s_abort)) {
      tma_chunk<3, D>(maps3, ld_tiles3, h, static_cast<int>(row0 + t0 - kC), bar_ld);
      ++tma_issued;
    }
    // ---- phase 5: A over P~ (the dv MMAs have read it)
    store_row32<false>(base + Lay::AS, t, gw, av);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (*reinterpret_cast<volatile int*>(s_abort)) { bad = true; break; }
    // ---- phase 6: dk' += A^T Q'; dv (complete) out meanwhile
    if (tid == 0) {
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, D, true, true);
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk)
        tc::mma_bf16(tmem + kTDK, mnmaj(base + Lay::AS, kk, 16384), mnmaj(base + Lay::QF, kk, 16384),
                     ID_MM, 1u);
      tc::mma_commit(bar3);  // dk' done, and with it every MMA of the chunk (R included)
    }
    // a whole chunk's dv and dk' are staged in shared memory and written by TMA (full lines); the
    // ragged last chunk of a document is written row by row (a tile store would reach past it)
    const bool whole = t0 + kC <= n;
    {
      float o[W];
      tmem_ldn<W>(tmem + tl + kTDV + W * gw, o);
      if (whole) {  // into XS: R~'s last readers (the first two groups) are done
        store_rown<false, W>(base + Lay::XS, t, gw, o);
      } else if (t0 + t < n) {
        __nv_bfloat16* dst = dv + ((row0 + t0 + t) * a.H + h) * D + W * gw;
#pragma unroll
        for (int m = 0; m < W / 8; ++m)
          *reinterpret_cast<uint4*>(dst + 8 * m) = feat::pack8(o + 8 * m);
      }
    }
    if (whole) {
      tc::fence_async_smem();
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb)
          tc::tma_store_3d(&tmdv, base + Lay::XS + jb * 16384, 64 * jb, h, static_cast<int>(row0 + t0));
        tc::bulk_commit();
      }
    }
    if (!wait_mma(bar3, it & 1)) atomicExch(s_abort, 1);
    // every MMA of the chunk has completed and no CUDA-core read of q' is left: the earlier
    // chunk's q' may arrive while this one finishes
    if (tid == 0 && c > 0 && !*reinterpret_cast<volatile int*>(s_abort)) {
      tma_chunk<1, D>(maps1, ld_tiles1, h, static_cast<int>(row0 + t0 - kC), bar_ldq);
      ++tmaq_issued;
    }
    // ---- phase 7: dk' + w into the staging, w += sum_t scale_t q'_t, R -> R~
    {
      {
        float o[W];
        tmem_ldn<W>(tmem + tl + kTDK + W * gw, o);
#pragma unroll
        for (int j = 0; j < W; ++j) o[j] += ws[W * gw + j];
        if (whole) {  // into AS: A's last reader (the third group) is done
          store_rown<false, W>(base + Lay::AS, t, gw, o);
        } else if (t0 + t < n) {  // dk' (bf16) to the workspace
          __nv_bfloat16* dst = dkf_out + ((row0 + t0 + t) * a.H + h) * D + W * gw;
#pragma unroll
          for (int m = 0; m < W / 8; ++m) *reinterpret_cast<uint4*>(dst + 8 * m) = feat::pack8(o + 8 * m);
        }
      }
      tc::fence_async_smem();
      if (tid == 0) tc::bulk_wait_read0();  // the dv store has read XS (R~ is rewritten below)
      tc::fence_before_sync();
      __syncthreads();  // w is read
      if (whole && tid == 0) {
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb)
          tc::tma_store_3d(&tmdk, base + Lay::AS + jb * 16384, 64 * jb, h, static_cast<int>(row0 + t0));
        tc::bulk_commit();
      }
      if (tid < D) {
        float dw = 0.f;
#pragma unroll
        for (int p = 0; p < kThreads / D; ++p) dw += red[8 * kC + p * D + tid];
        ws[tid] += dw;
      }
      if (D == 128 || t < D) {
        float rv[W];
        tmem_ldn<W>(tmem + tl + kTR + W * gw, rv);
        store_rown<true, W>(base + Lay::XS, t, gw, rv);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(s_abort)) { bad = true; break; }
  }
  bad = bad || *reinterpret_cast<volatile int*>(s_abort) != 0;
  if (tid == 0 && tma_issued > 0) tc::mbar_wait(bar_ld, (tma_issued - 1) & 1, kWait);
  if (tid == 0 && tmaq_issued > 0) tc::mbar_wait(bar_ldq, (tmaq_issued - 1) & 1, kWait);
  if (tid == 0) tc::bulk_wait0();  // the tile stores are complete before the NaN fill or exit
  __syncthreads();
  if (bad) {  // a wait gave up: NaN dk' and dv over the segment
    const int cpr = b.d / 8;  // 16-byte chunks per row
    for (long r = s0 + tid / cpr; r < s1; r += kThreads / cpr) {
      const long o = ((row0 + r) * a.H + h) * b.d + 8 * (tid % cpr);
      const uint4 nan = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
      *reinterpret_cast<uint4*>(dkf_out + o) = nan;
      *reinterpret_cast<uint4*>(dv + o) = nan;
    }
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0 && !misaligned && nch > 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// The state increments of blocks of a document, both of the form X_blk = sum_{t in blk} a_t b_t^T
// and x_blk = sum_t s_t a_t, accumulated chunk by chunk on the tensor core:
//   kFwd (before pass A): the prefix-state increments of the blocks before a document's last
//     segment (blk_per_seg per segment), S = sum k' v^T and z = sum k' (k' from the feature
//     kernel), in the prefill state kernel's record format (float4 j * D + i holds S[i][4j..4j+3],
//     then z);
//   otherwise (between the passes): the suffix-state increments of the blocks of the segments
//     after a document's first (rblk_per_seg per segment), R = sum q' gnum^T and w = sum scale q'
//     (gnum = g / den), as records [R row-major | w].
template <bool kFwd, int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_blockstate(const BwdArgs b, const __grid_constant__ CUtensorMap tma_a,
                      const __grid_constant__ CUtensorMap tma_b) {
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_seg = kFwd ? b.blk_per_seg : b.rblk_per_seg;
  const int nblk = kFwd ? b.nblk_max : b.nseg * b.rblk_per_seg;  // records per (document, head)
  const int kb = blockIdx.x % nblk, unit = blockIdx.x / nblk;
  const int seg = kb / per_seg;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int blen = b.seg_len / per_seg;
  const int s0 = kb * blen, s1 = min(n, s0 + blen);
  if (s0 >= s1) return;
  if (kFwd) {  // only the blocks before the document's last segment are read
    if (seg >= (n + b.seg_len - 1) / b.seg_len - 1) return;
  } else {
    if (seg == 0) return;  // nobody reads the first segment's increments
  }
  const int nch = (s1 - s0 + kC - 1) / kC;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  float* ws = reinterpret_cast<float*>(smem + Lay::ZS);
  float* scl_s = reinterpret_cast<float*>(smem + Lay::ROW);  // [2][128]: scale, 1 / den
  float* red = reinterpret_cast<float*>(smem + Lay::RED);
  const uint32_t bar1 = base + Lay::BAR, bar_ld0 = bar1 + 8;  // MMA done; tiles of set 0 / 1
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Lay::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + Lay::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;
  if (warp == 0 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 128);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar1, 1);
    tc::mbar_init(bar_ld0, 1);
    tc::mbar_init(bar_ld0 + 8, 1);
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  if (tid < kD) ws[tid] = 0.f;
  clear_upper_blocks<D>(base);
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  // a_t and b_t of even chunks in tiles QF / GS, of odd chunks in KF / VS, by TMA two chunks ahead
  const CUtensorMap* const maps[2] = {&tma_a, &tma_b};
  auto tiles = [&](int set, uint32_t (&t)[2]) {
    t[0] = base + (set ? Lay::KF : Lay::QF);
    t[1] = base + (set ? Lay::VS : Lay::GS);
  };
  int issued0 = 0, issued1 = 0;  // chunks requested per set (thread 0)
  if (tid == 0 && !*s_abort) {
    for (int c = 0; c < 2 && c < nch; ++c) {
      uint32_t t[2];
      tiles(c, t);
      tma_chunk<2, D>(maps, t, h, static_cast<int>(row0 + s0 + c * kC), bar_ld0 + 8 * c);
    }
    issued0 = 1;
    issued1 = nch > 1 ? 1 : 0;
  }
  // the row scalars (scale and 1 / den) of a chunk, loaded one chunk ahead into registers
  auto row_scalars = [&](int t0, float& sc, float& id) {
    const bool vr = tid < kC && t0 + tid < n;
    const long o = (row0 + t0 + tid) * a.H + h;
    sc = vr ? (kFwd ? 1.f : __ldg(b.scl + o)) : 0.f;
    id = (vr && !kFwd) ? __ldg(b.den + o) : 1.f;
  };
  float sc_next, den_next;
  row_scalars(s0, sc_next, den_next);
  bool bad = *s_abort != 0;
  for (int c = 0; c < nch && !bad; ++c) {
    const int t0 = s0 + c * kC, set = c & 1;
    uint32_t t[2];
    tiles(set, t);
    if (tid < kC) {
      scl_s[tid] = sc_next;
      scl_s[kC + tid] = 1.0f / den_next;
    }
    if (c + 1 < nch) row_scalars(t0 + kC, sc_next, den_next);
    if (!tc::mbar_wait(bar_ld0 + 8 * set, (c >> 1) & 1, kWait)) atomicExch(s_abort, 1);
    __syncthreads();  // scl_s
    // rows past the document cleared; reverse: b = g / den in place
    if (!kFwd || t0 + kC > n) {
      for (int idx = tid; idx < kC * D / 8; idx += kThreads) {
        const int r = idx / (D / 8), m = idx % (D / 8);
        const uint32_t ga = t[1] + tile_off(r, m);
        if (t0 + r >= n) {
          sts16(ga, make_uint4(0, 0, 0, 0));
          sts16(t[0] + tile_off(r, m), make_uint4(0, 0, 0, 0));
        } else if (!kFwd) {
          float f[8];
          unpack8(lds16(ga), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] *= scl_s[kC + r];
          sts16(ga, feat::pack8(f));
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, D, true, true);
#pragma unroll 1
      for (int kk = 0; kk < kC / 16; ++kk)
        tc::mma_bf16(tmem, mnmaj(t[0], kk, 16384), mnmaj(t[1], kk, 16384), ID_MM,
                     (c > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(bar1);
    }
    {  // partial increment of x: column i of a, rows RP (tid / D) .. + RP - 1
      constexpr int RP = kC * D / kThreads;
      const int i = tid & (D - 1), r0 = RP * (tid / D);
      const int m = i >> 3, e = i & 7;
      float dw = 0.f;
#pragma unroll 4
      for (int r = r0; r < r0 + RP; ++r) {
        uint32_t word;
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(word)
                     : "r"(t[0] + tile_off(r, m) + 4 * (e >> 1))
                     : "memory");
        const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&word));
        dw = fmaf(scl_s[r], (e & 1) ? p.y : p.x, dw);
      }
      red[tid] = dw;  // partial tid / D of column i
    }
    if (!wait_mma(bar1, c & 1)) atomicExch(s_abort, 1);
    __syncthreads();  // the MMA and every thread are done with this set's tiles
    if (tid == 0 && c + 2 < nch && !*reinterpret_cast<volatile int*>(s_abort)) {
      tma_chunk<2, D>(maps, t, h, static_cast<int>(row0 + t0 + 2 * kC), bar_ld0 + 8 * set);
      if (set) ++issued1;
      else ++issued0;
    }
    if (tid < D) {
      float dw = 0.f;
#pragma unroll
      for (int p = 0; p < kThreads / D; ++p) dw += red[p * D + tid];
      ws[tid] += dw;
    }
    bad = *reinterpret_cast<volatile int*>(s_abort) != 0;
    __syncthreads();
  }
  if (tid == 0) {  // copies still in flight land before the CTA leaves
    if (issued0 > 0) tc::mbar_wait(bar_ld0, (issued0 - 1) & 1, kWait);
    if (issued1 > 0) tc::mbar_wait(bar_ld0 + 8, (issued1 - 1) & 1, kWait);
  }
  // the record (TMEM lane i = row i of X), then x; NaN if a wait gave up
  constexpr long REC = static_cast<long>(kD) * kD + kD;
  float* rec = (kFwd ? b.rec_fwd : b.rec_rev) + (static_cast<long>(unit) * nblk + kb) * REC;
  const int q4 = warp & 3, gw = warp >> 2;
  const int tr = 32 * q4 + lane;
  float rv[32];
  if (D == 64 && gw >= D / 32) {  // columns past d: the product has N = d
#pragma unroll
    for (int e = 0; e < 32; ++e) rv[e] = 0.f;
  } else if (!bad) {
    tmem_ld32(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 32 * gw, rv);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) rv[e] = __int_as_float(0x7fc00000);
  }
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    const float4 x4 = make_float4(rv[4 * jj], rv[4 * jj + 1], rv[4 * jj + 2], rv[4 * jj + 3]);
    if (kFwd) reinterpret_cast<float4*>(rec)[(8 * gw + jj) * kD + tr] = x4;
    else *reinterpret_cast<float4*>(rec + tr * kD + 32 * gw + 4 * jj) = x4;
  }
  if (tid < kD) rec[kD * kD + tid] = bad ? __int_as_float(0x7fc00000) : ws[tid];
  if (bad && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0 && !misaligned) tc::tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------------------------------------
// Before the passes, fully parallel: q' = ReLU(RoPE(RMSNorm(q))) and k' likewise (bf16) of every
// row into the workspace, where the forward and reverse passes take their q', k' tiles from. One
// CTA per (document, head, chunk, q or k), 256 threads (128 at d = 64, so that twice the CTAs,
// each with half the bytes, keep as many loads in flight per SM): the chunk's raw rows arrive in
// shared memory by TMA; a thread owns 8 consecutive elements of a row (d / 8 threads per row) and
// works on packed fp32 pairs, with the gains and the RoPE frequencies and per-pass rotation in
// shared memory.
template <int D>
struct MapCfg {
  static constexpr int THREADS = D == 64 ? 128 : 256;
  static constexpr uint32_t SMEM = kC * D * 2 + 1024;  // one tile (+ alignment slack)
};

template <int D>
__global__ void __launch_bounds__(MapCfg<D>::THREADS)
    bwd_tc_featmap(const BwdArgs b, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k) {
  constexpr int NT = MapCfg<D>::THREADS;
  constexpr int TPR = D / 8, RPP = NT / TPR, NPASS = kC / RPP;
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x;
  const int which = blockIdx.x & 1;  // 0: q, 1: k
  const int chunk = (blockIdx.x >> 1) % b.chunks_max, unit = (blockIdx.x >> 1) / b.chunks_max;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int t0 = chunk * kC;
  if (t0 >= n) return;  // uniform
  __shared__ __align__(16) float tabmem[4 * D];
  __shared__ __align__(8) uint64_t bar_storage;
  extern __shared__ __align__(1024) uint8_t fsmem[];
  const uint32_t tile = (tc::smem_u32(fsmem) + 1023u) & ~1023u;  // the chunk's raw rows (TMA)
  const uint32_t bar = tc::smem_u32(&bar_storage);
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    const CUtensorMap* const maps[1] = {which ? &tm_k : &tm_q};
    const uint32_t tl[1] = {tile};
    tma_chunk<1, D>(maps, tl, h, static_cast<int>(row0 + t0), bar);
  }
  const feat::FeatTab tab = feat::feat_tab<D>(reinterpret_cast<uint8_t*>(tabmem));
  feat::fill_tab<D>(tab, a, h, RPP, tid, NT);
  __syncthreads();
  const int prow = tid / TPR, part = tid % TPR, e0 = 8 * part;
  const long rstride = static_cast<long>(a.H) * D;
  const long off0 = (row0 + t0 + prow) * rstride + static_cast<long>(h) * D + e0;
  __nv_bfloat16* xf = static_cast<__nv_bfloat16*>(which ? b.kf : b.qf) + off0;
  float2 g0[2], g1[2];
  feat::split_load<D>(which ? tab.gk : tab.gq, part, g0, g1);
  feat::Rot step, rot;
  feat::tab_step(tab, e0 / 2, step);
  feat::tab_rot_at(tab, a.pos_offset + t0 + prow, e0 / 2, rot);
  if (!tc::mbar_wait(bar, 0, kWait)) {  // NaN features, so the failure cannot pass for a result
    for (int p = 0; p < NPASS; ++p)
      if (t0 + p * RPP + prow < n)
        *reinterpret_cast<uint4*>(xf + p * RPP * rstride) =
            make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
    return;
  }
#pragma unroll
  for (int p = 0; p < NPASS; ++p) {
    if (p > 0) feat::rot_step(rot, step);
    const int r = p * RPP + prow;
    feat::Pairs f = feat::unpack_pairs(feat::lds16(tile + tile_off(r, part)));
    const float ss = feat::row_sum<TPR>(feat::sumsq(f));
    float2 ga[2] = {g0[0], g0[1]}, gb[2] = {g1[0], g1[1]};
    feat::scale_gains(ga, gb, rsqrtf(ss * (1.0f / D) + a.fa.eps_norm));
    feat::rope_relu(f, ga, gb, rot);
    if (t0 + r < n) *reinterpret_cast<uint4*>(xf + p * RPP * rstride) = feat::pack_pairs(f);
  }
}

// After the passes: dq and dk through the feature map from dq', dk' (bf16, in the workspace) and the
// raw q, k, with the gain partials of every (document, head, 128-token chunk). Same layout as the
// feature kernel (256 threads, 16 per row, packed fp32 pairs). Per row, with r = 1/rms(x) and the
// forward's pre-activations (a, b) = R(y) of y = x r gamma (R: the pair's rotation):
//   (da, db) = the feature gradient where the pre-activation is positive, else 0 (ReLU),
//   h = R^T (da, db) (the inverse rotation), u = gamma h,
//   dx = r u - x r^3 (u . x) / d,   dgamma += h x r.
// The chunk's rows of x and of its feature gradient are staged in shared memory by TMA (two 32 KB
// tiles per CTA, three CTAs per SM; at d = 64 two 16 KB tiles, 128 threads and six CTAs per SM),
// so that each SM has ~200 KB of loads in flight. One launch
// takes one of q (which = 0) and k (which = 1): dq needs only pass A's dq', so it runs while the
// reverse pass does.
template <int D>
struct FeatCfg {
  static constexpr int THREADS = D == 64 ? 128 : 256, MIN_CTAS = D == 64 ? 6 : 3;
  static constexpr uint32_t TILE = kC * D * 2;            // one chunk's rows (D / 64 blocks)
  static constexpr uint32_t SMEM = 2 * TILE + 1024;       // two tiles (+ alignment slack)
};

template <int D>
__global__ void __launch_bounds__(FeatCfg<D>::THREADS, FeatCfg<D>::MIN_CTAS)
    bwd_tc_features(const BwdArgs b, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_dq,
                    const __grid_constant__ CUtensorMap tm_dk, const int which) {
  constexpr int NT = FeatCfg<D>::THREADS;
  constexpr int TPR = D / 8, RPP = NT / TPR, NPASS = kC / RPP;
  constexpr int WARPS = NT / 32;
  const PrefillArgs& a = b.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x % b.chunks_max, unit = blockIdx.x / b.chunks_max;
  const int h = unit % a.H, doc = unit / a.H;
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);
  const int t0 = chunk * kC;
  __shared__ __align__(16) float tabmem[4 * D];
  __shared__ __align__(16) float scratch[WARPS * D];
  __shared__ __align__(8) uint64_t bar_storage;
  extern __shared__ __align__(1024) uint8_t fsmem[];
  const uint32_t tiles_base = (tc::smem_u32(fsmem) + 1023u) & ~1023u;  // 1024-byte aligned
  const uint32_t bar = tc::smem_u32(&bar_storage);
  const int prow = tid / TPR, part = tid % TPR, e0 = 8 * part;
  float2 dga[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // gain gradient, Pairs layout
  float2 dgb[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  bool failed = false;
  if (t0 < n) {  // uniform; a chunk past the document's end contributes zero partials
    if (tid == 0) {
      tc::mbar_init(bar, 1);
      tc::mbar_fence_init();
    }
    __syncthreads();
    if (tid == 0) {
      const CUtensorMap* const maps[2] = {which ? &tm_k : &tm_q, which ? &tm_dk : &tm_dq};
      const uint32_t tl[2] = {tiles_base, tiles_base + FeatCfg<D>::TILE};
      tma_chunk<2, D>(maps, tl, h, static_cast<int>(row0 + t0), bar);
    }
    const feat::FeatTab tab = feat::feat_tab<D>(reinterpret_cast<uint8_t*>(tabmem));
    feat::fill_tab<D>(tab, a, h, RPP, tid, NT);
    __syncthreads();
    const long rstride = static_cast<long>(a.H) * D;
    const long off0 = (row0 + t0 + prow) * rstride + static_cast<long>(h) * D + e0;
    __nv_bfloat16* dx = static_cast<__nv_bfloat16*>(which ? b.dk : b.dq) + off0;
    float2 g0[2], g1[2];
    feat::split_load<D>(which ? tab.gk : tab.gq, part, g0, g1);
    feat::Rot step, rot;
    feat::tab_step(tab, e0 / 2, step);
    feat::tab_rot_at(tab, a.pos_offset + t0 + prow, e0 / 2, rot);
    failed = !tc::mbar_wait(bar, 0, kWait);
#pragma unroll 1
    for (int p0 = 0; p0 < NPASS && !failed; p0 += 2) {
      uint4 rx[2], rd[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // rows past the document (other tokens or zero fill) are masked
        const int r = (p0 + i) * RPP + prow;
        const bool valid = t0 + r < n;
        rx[i] = valid ? feat::lds16(tiles_base + tile_off(r, part)) : make_uint4(0, 0, 0, 0);
        rd[i] = valid ? feat::lds16(tiles_base + FeatCfg<D>::TILE + tile_off(r, part)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int p = p0 + i;
        if (p > 0) feat::rot_step(rot, step);
        const bool valid = t0 + p * RPP + prow < n;
        const feat::Pairs f = feat::unpack_pairs(rx[i]), d = feat::unpack_pairs(rd[i]);
        const float r = rsqrtf(feat::row_sum<TPR>(feat::sumsq(f)) * (1.0f / D) + a.fa.eps_norm);
        const float2 r2 = make_float2(r, r);
        float2 dotv = make_float2(0.f, 0.f);
        float2 u0[2], u1[2];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const float2 xr0 = __fmul2_rn(f.x0[g], r2), xr1 = __fmul2_rn(f.x1[g], r2);
          const float2 y0 = __fmul2_rn(xr0, g0[g]), y1 = __fmul2_rn(xr1, g1[g]);
          const float2 ns = make_float2(-rot.s[g].x, -rot.s[g].y);
          const float2 pa = __ffma2_rn(y0, rot.c[g], __fmul2_rn(y1, ns));   // pre-activations
          const float2 pb = __ffma2_rn(y0, rot.s[g], __fmul2_rn(y1, rot.c[g]));
          const float2 da = make_float2(pa.x > 0.f ? d.x0[g].x : 0.f, pa.y > 0.f ? d.x0[g].y : 0.f);
          const float2 db = make_float2(pb.x > 0.f ? d.x1[g].x : 0.f, pb.y > 0.f ? d.x1[g].y : 0.f);
          const float2 h0 = __ffma2_rn(da, rot.c[g], __fmul2_rn(db, rot.s[g]));  // R^T (da, db)
          const float2 h1 = __ffma2_rn(db, rot.c[g], __fmul2_rn(da, ns));
          dga[g] = __ffma2_rn(h0, xr0, dga[g]);
          dgb[g] = __ffma2_rn(h1, xr1, dgb[g]);
          u0[g] = __fmul2_rn(g0[g], h0);
          u1[g] = __fmul2_rn(g1[g], h1);
          dotv = __ffma2_rn(u0[g], f.x0[g], dotv);
          dotv = __ffma2_rn(u1[g], f.x1[g], dotv);
        }
        const float dot = feat::row_sum<TPR>(dotv.x + dotv.y);
        const float c3 = r * r * r * dot * (1.0f / D);
        const float2 c32 = make_float2(-c3, -c3);
        feat::Pairs o;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          o.x0[g] = __ffma2_rn(f.x0[g], c32, __fmul2_rn(r2, u0[g]));
          o.x1[g] = __ffma2_rn(f.x1[g], c32, __fmul2_rn(r2, u1[g]));
        }
        if (valid) *reinterpret_cast<uint4*>(dx + p * RPP * rstride) = feat::pack_pairs(o);
      }
    }
  }
  // the CTA's gain partial: each thread's rows, then the warp's two rows, then the warps in order
  float dg[8];
  feat::pairs_to8(feat::Pairs{{dga[0], dga[1]}, {dgb[0], dgb[1]}}, dg);
  feat::warp_colsum<TPR>(dg);
  if (lane < TPR) {
#pragma unroll
    for (int e = 0; e < 8; ++e) scratch[warp * D + e0 + e] = dg[e];
  }
  __syncthreads();
  if (tid < D) {
    float sum = 0.f;
    for (int w = 0; w < WARPS; ++w) sum += scratch[w * D + tid];
    (which ? b.dgp_k : b.dgp_q)[(static_cast<long>(unit) * b.chunks_max + chunk) * D + tid] =
        failed ? __int_as_float(0x7fc00000) : sum;  // a wait that gave up cannot pass for a result
  }
  if (failed && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
}

}  // namespace

bool bwd_tc_supported(DType dt, int d) { return dt == DType::BF16 && (d == 64 || d == 128); }

namespace {
// Per thread and device: a stream of the greatest priority that carries the backward's critical
// path (feature map, block states, both passes, dk), forked from the caller's stream and joined back
// to it, and the three events of the fork, the hand-over after pass A and the join. The feature
// backward of q runs on the caller's stream meanwhile; with the priorities the passes' CTAs are
// dispatched first and it fills the SMs they leave idle.
struct Side {
  unsigned long long ctx = 0;  // the context the handles belong to (its unique id)
  cudaStream_t hi = nullptr;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
};
// The unique id of the calling thread's current context (0 if it cannot be read): handles made in
// a context that has since been destroyed (a device reset) are never reused.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || f1 == nullptr || f2 == nullptr)
      return 0;
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}
cudaError_t side_stream(int dev, Side*& out) {
  thread_local Side side[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Side& sd = side[dev];
  const unsigned long long ctx = current_context_id();
  if (ctx == 0) return cudaErrorDeviceUninitialized;
  if (sd.hi == nullptr || sd.ctx != ctx) {  // the handles of a destroyed context are left alone
    int least = 0, greatest = 0;
    Side n;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&n.hi, cudaStreamNonBlocking, greatest);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&n.ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      for (cudaEvent_t ev : n.ev)
        if (ev != nullptr) cudaEventDestroy(ev);
      if (n.hi != nullptr) cudaStreamDestroy(n.hi);
      return e;
    }
    n.ctx = ctx;
    sd = n;
  }
  out = &sd;
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_backward_tc(const BwdArgs& b, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    for (const void* f : {reinterpret_cast<const void*>(bwd_tc_forward<64>),
                          reinterpret_cast<const void*>(bwd_tc_forward<128>),
                          reinterpret_cast<const void*>(bwd_tc_reverse<64>),
                          reinterpret_cast<const void*>(bwd_tc_reverse<128>),
                          reinterpret_cast<const void*>(bwd_tc_blockstate<true, 64>),
                          reinterpret_cast<const void*>(bwd_tc_blockstate<true, 128>),
                          reinterpret_cast<const void*>(bwd_tc_blockstate<false, 64>),
                          reinterpret_cast<const void*>(bwd_tc_blockstate<false, 128>)}) {
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(Lay::BYTES));
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(bwd_tc_features<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(FeatCfg<64>::SMEM));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_tc_features<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(FeatCfg<128>::SMEM));
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  const long grid = static_cast<long>(b.p.n_docs) * b.p.H * b.nseg;
  if (grid == 0) return cudaSuccess;
  const long fgrid = static_cast<long>(b.p.n_docs) * b.p.H * b.chunks_max;  // per tensor
  const int d = b.d;  // the tensors' head size
  Side* side = nullptr;
  if ((e = side_stream(dev, side)) != cudaSuccess) return e;
  const cudaStream_t user = stream;
  if ((e = cudaEventRecord(side->ev[0], user)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(side->hi, side->ev[0], 0)) != cudaSuccess) return e;
  stream = side->hi;
  // from here on every exit joins the side stream back to the caller's stream first
  const auto join = [&](cudaError_t err) {
    cudaError_t j = cudaEventRecord(side->ev[2], side->hi);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(user, side->ev[2], 0);
    return err != cudaSuccess ? err : j;
  };
  CUtensorMap tmq, tmk;
  if ((e = make_rows_map(&tmq, b.p.q, b.p.total_rows, b.p.H, d)) != cudaSuccess) return join(e);
  if ((e = make_rows_map(&tmk, b.p.k, b.p.total_rows, b.p.H, d)) != cudaSuccess) return join(e);
  if (d == 128)
    bwd_tc_featmap<128><<<static_cast<unsigned>(2 * fgrid), MapCfg<128>::THREADS, MapCfg<128>::SMEM, stream>>>(b, tmq, tmk);
  else
    bwd_tc_featmap<64><<<static_cast<unsigned>(2 * fgrid), MapCfg<64>::THREADS, MapCfg<64>::SMEM, stream>>>(b, tmq, tmk);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return join(e);
  if (b.order != nullptr) {  // packed documents: the passes take the longest first
    if ((e = launch_doc_order(b.p.cu_seqlens, b.p.n_docs, b.p.total_rows, b.order, stream)) != cudaSuccess)
      return join(e);
  }
  // TMA maps of the row-major [rows, H, D] tensors the kernels stream
  CUtensorMap tmv, tmg, tmqf, tmkf;
  const long rows = b.p.total_rows;
  if ((e = make_rows_map(&tmv, b.p.v, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if ((e = make_rows_map(&tmg, b.dout, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if ((e = make_rows_map(&tmqf, b.qf, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if ((e = make_rows_map(&tmkf, b.kf, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if (b.nseg > 1) {  // the prefix-state increments of the blocks before each document's last segment
    const unsigned g = static_cast<unsigned>(static_cast<long>(b.p.n_docs) * b.p.H * b.nblk_max);
    if (d == 128) bwd_tc_blockstate<true, 128><<<g, kThreads, Lay::BYTES, stream>>>(b, tmkf, tmv);
    else bwd_tc_blockstate<true, 64><<<g, kThreads, Lay::BYTES, stream>>>(b, tmkf, tmv);
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return join(e);
  }
  // dq', dk' (written by the passes, read by the feature kernel) and dv
  CUtensorMap tmdq, tmdk, tmdv;
  if ((e = make_rows_map(&tmdq, b.dqf, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if ((e = make_rows_map(&tmdk, b.dkf, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if ((e = make_rows_map(&tmdv, b.dv, rows, b.p.H, d)) != cudaSuccess) return join(e);
  if (d == 128)
    bwd_tc_forward<128><<<static_cast<unsigned>(grid), kThreadsA, Lay::BYTES, stream>>>(b, tmqf, tmkf, tmv, tmg, tmdq);
  else
    bwd_tc_forward<64><<<static_cast<unsigned>(grid), kThreadsA, Lay::BYTES, stream>>>(b, tmqf, tmkf, tmv, tmg, tmdq);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return join(e);
  // dq through the feature map needs only pass A: on the caller's stream, beside the reverse pass
  if ((e = cudaEventRecord(side->ev[1], stream)) != cudaSuccess) return join(e);
  if ((e = cudaStreamWaitEvent(user, side->ev[1], 0)) != cudaSuccess) return join(e);
  if (d == 128)
    bwd_tc_features<128><<<static_cast<unsigned>(fgrid), FeatCfg<128>::THREADS, FeatCfg<128>::SMEM, user>>>(
        b, tmq, tmk, tmdq, tmdk, 0);
  else
    bwd_tc_features<64><<<static_cast<unsigned>(fgrid), FeatCfg<64>::THREADS, FeatCfg<64>::SMEM, user>>>(
        b, tmq, tmk, tmdq, tmdk, 0);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return join(e);
  if (b.nseg > 1) {
    const unsigned g = static_cast<unsigned>(grid * b.rblk_per_seg);
    if (d == 128) bwd_tc_blockstate<false, 128><<<g, kThreads, Lay::BYTES, stream>>>(b, tmqf, tmg);
    else bwd_tc_blockstate<false, 64><<<g, kThreads, Lay::BYTES, stream>>>(b, tmqf, tmg);
    note_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return join(e);
  }
  if (d == 128)
    bwd_tc_reverse<128><<<static_cast<unsigned>(grid), kThreads, Lay::BYTES, stream>>>(b, tmqf, tmkf, tmv, tmg, tmdv, tmdk);
  else
    bwd_tc_reverse<64><<<static_cast<unsigned>(grid), kThreads, Lay::BYTES, stream>>>(b, tmqf, tmkf, tmv, tmg, tmdv, tmdk);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return join(e);
  if (d == 128)
    bwd_tc_features<128><<<static_cast<unsigned>(fgrid), FeatCfg<128>::THREADS, FeatCfg<128>::SMEM, stream>>>(
        b, tmq, tmk, tmdq, tmdk, 1);
  else
    bwd_tc_features<64><<<static_cast<unsigned>(fgrid), FeatCfg<64>::THREADS, FeatCfg<64>::SMEM, stream>>>(
        b, tmq, tmk, tmdq, tmdk, 1);
  note_launches(1);
  if ((e = join(cudaGetLastError())) != cudaSuccess) return e;
  BwdArgs g = b;  // the gain partials are per (document, head, chunk)
  g.nseg = b.chunks_max;
  return launch_bwd_gain(g, d, user);
}

}  // namespace rapt
