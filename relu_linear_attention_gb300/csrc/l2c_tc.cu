// Causal original RLA (L2 denominator) on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a;
// bf16, d in {64, 128}, dense batch rows or packed documents, fp32 accumulation and fp32 states.
//
// 08-rapt-algorithm.md §2.1 (closed form, eps outside the root; q' = ReLU(q), k' = ReLU(k)), §2.2
// (a query reads the accumulated causal state, which restarts at every document), §4.1 (the
// scan's two prefix states):
//   S_t = sum_{i<=t} k'_i v_i^T,  A_t = sum_{i<=t} k'_i k'_i^T,
//   out_t = q'_t S_t / (sqrt(q'_t^T A_t q'_t) + eps).
// Chunked (C = 128 tokens), with P = Q'K'^T masked to tau <= t and S~, A~ bf16 copies of the fp32
// states before the chunk, three groups of products per chunk on the tensor core:
//   g1:  P = Q'K'^T,  X = Q'A~
//   g2:  S += K'^T V,  A += K'^T K'
//   g3:  X = Q'S~ + P~V           (P~ = P masked, in bf16, read from TMEM)
//   den_t = sqrt(sum_tau P^2 + q'_t . X_t) + eps after g1 (fp32; P from exact bf16 features),
//   out = X / den after g3; A -> A~ after g2 and S -> S~ after g3, for the next chunk.
// Dense batch rows may be cut into segments of seg_len tokens; segment s starts from the moments
// [K'^T V | K'^T K'] of the splits before it, computed by the non-causal L2 path's moments kernel
// with the same split length (summed in split order: deterministic), and is launched as a
// programmatic dependent of it (segment 0 needs no moments and starts at once). Packed documents
// run one CTA per (document, head), the longest documents first. d = 64 pads K'^T to M = 128 with a
// zero block (TMEM rows 64..127 of S and A stay zero).
// One CTA per (document, head, segment), warp-specialised (768 threads):
//   warps 0-15  converters, four per TMEM lane quarter (32 columns each): the row sums of den^2
//               and P~ after g1, A~ after g2, the output and S~ after g3;
//   warps 16-21 rectifiers: q' = ReLU(q), k' = ReLU(k) in place in the two q and k slots;
//   warp 22     issues the MMAs (one thread): P of chunk c runs while the converters finish chunk
//               c - 1, g2 while they form den and P~, g3 once P~ is written;
//   warp 23     TMA (one thread): q and k two chunks ahead (two slots each), v one chunk ahead.
// Hand-offs are mbarriers (qk_full, qk_ready per slot; v_full; g1, g2, g3 commits; conv1, x_free,
// a_conv, s_conv from the converters); every wait is bounded (~1 s); a CTA whose wait gives up
// writes NaN over its rows.
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
constexpr int kConvWarps = 16;                 // four per TMEM lane quarter, 32 columns each
constexpr int kRectWarps = 6;
constexpr int kWarpIssue = kConvWarps + kRectWarps;
constexpr int kWarpTma = kWarpIssue + 1;
constexpr int kThreads = 32 * (kWarpTma + 1);  // 768: six warpgroups
constexpr uint32_t kBarQuarter = 1;            // 1..4: the four converter warps of a lane quarter
// Register split (setmaxnreg draws on the launch allocation: threads x launch registers): the
// converters' warpgroups hold a row's 32 scores and 32 products at once; the others need few.
constexpr int kLaunchRegs = 80, kRegsConv = 96, kRegsOther = 48;
static_assert(32 * kConvWarps * kRegsConv + (kThreads - 32 * kConvWarps) * kRegsOther <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(kConvWarps % 4 == 0 && kThreads % 128 == 0, "warpgroup-aligned roles");

// Shared memory (bytes from a 1024-byte aligned base): two q slots and two k slots (a chunk's raw
// rows by TMA, rectified in place; a k slot is 32 KB so that d = 64 has the zero block that pads
// k'^T to M = 128), one v tile, the bf16 state copies S~ and A~ (D rows), the converters' partial
// den^2 sums, mbarriers.
template <int D>
struct LayC {
  static constexpr uint32_t TILE = (D / 64) * 16384;  // 128 rows x D columns, bf16
  static constexpr uint32_t STILE = D * D * 2;        // a D x D state copy, bf16
  static constexpr uint32_t Q0 = 0, Q1 = TILE;
  static constexpr uint32_t K0 = 2 * TILE, K1 = K0 + 32768;
  static constexpr uint32_t VS = K1 + 32768;
  static constexpr uint32_t SS = VS + TILE, AS = SS + STILE;
  static constexpr uint32_t RED = AS + STILE;         // partial den^2 [4 column groups][128 rows]
  // qk_full[2] qk_ready[2] v_full g1 g2 g3 conv1 x_free a_conv s_conv
  static constexpr uint32_t BAR = RED + 4 * kC * 4;
  static constexpr int NBAR = 12;
  static constexpr uint32_t MISC = BAR + NBAR * 8;    // TMEM base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(Q1 % 1024 == 0 && K0 % 1024 == 0 && VS % 1024 == 0 && SS % 1024 == 0 &&
                AS % 1024 == 0, "tile alignment");
  // TMEM columns: P (its bf16 P~ written over the upper half of each 32-column group), X (q'A~,
  // then the numerator q'S~ + P~V), S, A
  static constexpr uint32_t TP = 0, TX = 128, TS = 128 + D, TA = 128 + 2 * D;
  static_assert(TA + D <= 512, "TMEM budget");
};

// Rows [row, row + 128) of head h of a row-major [rows, H, D] tensor into a tile by TMA (D / 64
// boxes; rows past the tensor read as zero); one thread calls it.
template <int D>
__device__ __forceinline__ void tma_tile(const CUtensorMap* m, uint32_t tile, int h, int row, uint32_t bar) {
#pragma unroll
  for (int jb = 0; jb < D / 64; ++jb) tc::tma_load_3d(tile + jb * 16384, m, 64 * jb, h, row, bar);
}

// bf16 max(x, 0) of eight packed values, one packed max per pair (a NaN becomes 0, -0 may stay
// -0: either is a zero operand of the products).
__device__ __forceinline__ uint4 relu8(uint4 v) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) asm("max.bf16x2 %0, %0, %1;" : "+r"(w[e]) : "r"(0u));
  return make_uint4(w[0], w[1], w[2], w[3]);
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
  const uint32_t bar_qkfull = base + L::BAR, bar_qkready = bar_qkfull + 16, bar_vfull = bar_qkfull + 32;
  const uint32_t bar_g1 = bar_qkfull + 40, bar_g2 = bar_qkfull + 48, bar_g3 = bar_qkfull + 56;
  const uint32_t bar_conv1 = bar_qkfull + 64, bar_xfree = bar_qkfull + 72;
  const uint32_t bar_aconv = bar_qkfull + 80, bar_sconv = bar_qkfull + 88;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;
  if (warp == 0 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar_qkfull + 8 * i, 1);
      tc::mbar_init(bar_qkready + 8 * i, 32 * kRectWarps);
    }
    tc::mbar_init(bar_vfull, 1);
    tc::mbar_init(bar_g1, 1);
    tc::mbar_init(bar_g2, 1);
    tc::mbar_init(bar_g3, 1);
    tc::mbar_init(bar_conv1, kConvWarps);
    tc::mbar_init(bar_xfree, kConvWarps);
    tc::mbar_init(bar_aconv, kConvWarps);
    tc::mbar_init(bar_sconv, kConvWarps);
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  if (D == 64 && !misaligned) {  // zero blocks that pad k'^T to M = 128 rows (both k slots)
    for (int i = tid; i < 2 * 16384 / 16; i += kThreads)
      sts16(base + L::K0 + (i >> 10) * 32768 + 16384 + (i & 1023) * 16, make_uint4(0, 0, 0, 0));
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const bool bad0 = *s_abort != 0;

  if (warp < kConvWarps) {
    // ================================================================ converters (warps 0-15)
    tc::regs_inc<kRegsConv>();
    const int q4 = warp & 3, gw = warp >> 2;
    const int t = 32 * q4 + lane;  // tile row = TMEM lane
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    int bad = bad0;
    // the states at the segment's start: the moments of the earlier splits, in split order; rows
    // and columns past D (d = 64) are the zero padding of TMEM (completion 0 of a_conv and s_conv)
    if (!bad && gw < NG) {
      float sv[32], av[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) sv[e] = av[e] = 0.f;
      if (seg > 0 && t < D) {
        tc::grid_dep_wait();
        const float4* part = reinterpret_cast<const float4*>(a.ws) + bh * (a.nseg - 1) * (D * 2 * D / 4);
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
    __syncwarp();
    if (lane == 0) {
      tc::mbar_arrive(bar_aconv);
      tc::mbar_arrive(bar_sconv);
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    for (int c = 0; c < nch && !bad0; ++c) {
      const int s = c & 1, t0 = s0 + c * kC;
      // ---- den^2 = sum_{tau <= t} P^2 + q' . (q' A~) of the rows, and P~ (masked, bf16, over the
      // upper half of this warp's 32 P columns: keys 32 gw .. 32 gw + 31)
      int ok = tc::mbar_wait(bar_g1, c & 1, kWait);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;
      tc::fence_after_sync();
      float part = 0.f;
      if (!bad) {
        // this warp's scores and products (both TMEM reads in flight together), then its q' columns
        const bool live = 32 * gw <= 32 * q4;  // warp-uniform: keys not all after the quarter's rows
        const bool prod = gw < NG;             // warp-uniform: the warp has product columns
        uint32_t up[2][16], ux[2][16];
        if (live) {
          tc::tmem_ld16(tmem + tl + L::TP + 32 * gw, up[0]);
          tc::tmem_ld16(tmem + tl + L::TP + 32 * gw + 16, up[1]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) up[0][e] = up[1][e] = 0u;
        }
        if (prod) {
          tc::tmem_ld16(tmem + tl + L::TX + 32 * gw, ux[0]);
          tc::tmem_ld16(tmem + tl + L::TX + 32 * gw + 16, ux[1]);
        }
        tc::tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = __uint_as_float(up[j >> 4][j & 15]), p1 = __uint_as_float(up[j >> 4][(j & 15) + 1]);
          const float x0 = 32 * gw + j <= t ? p0 : 0.f;
          const float x1 = 32 * gw + j + 1 <= t ? p1 : 0.f;
          part = fmaf(x0, x0, part);
          part = fmaf(x1, x1, part);
          w[j / 2] = tc::pack_bf16x2(x0, x1);
        }
        tc::tmem_st16(tmem + tl + L::TP + 32 * gw + 16, w);
        if (prod) {
          const uint32_t qb = base + (s ? L::Q1 : L::Q0);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float f[8];
            unpack8(lds16(qb + tile_off(t, 4 * gw + m)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) part = fmaf(f[e], __uint_as_float(ux[m >> 1][8 * (m & 1) + e]), part);
          }
        }
        tc::tmem_wait_st();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_conv1);  // P~ written, q'A~ read: the numerator may start
      // the four column groups' partial sums (the first barrier: the previous chunk's are read)
      tc::named_sync(kBarQuarter + q4, 128);
      red[gw * kC + t] = part;
      tc::named_sync(kBarQuarter + q4, 128);
      const float den = sqrtf(fmaxf(red[t] + red[kC + t] + red[2 * kC + t] + red[3 * kC + t], 0.f)) + a.eps;
      // ---- A (after this chunk) -> A~ for the next chunk's q'A~ (this chunk's has read A~)
      ok = tc::mbar_wait(bar_g2, c & 1, kWait);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;
      tc::fence_after_sync();
      if (!bad && gw < NG && t < D) {
        float v[32];
        tmem_ld32(tmem + tl + L::TA + 32 * gw, v);
        store_row32<true>(base + L::AS, t, gw, v);
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_aconv);
      // ---- out = (q'S~ + P~V) / den; then S -> S~ (the numerator has read the previous S~)
      ok = tc::mbar_wait(bar_g3, c & 1, kWait);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;
      tc::fence_after_sync();
      // out rows of 32 columns: four 16-byte chunks per row and thread, transposed across each
      // group of four lanes (rows 4i .. 4i+3) so that a store writes 64 contiguous bytes of a row
      // from four lanes: every store instruction of the warp covers 8 rows instead of 32
      if (!bad && gw < NG) {
        float xv[32];
        tmem_ld32(tmem + tl + L::TX + 32 * gw, xv);
        const float inv = 1.0f / den;
#pragma unroll
        for (int j = 0; j < 32; ++j) xv[j] *= inv;
        uint4 ch[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) ch[m] = feat::pack8(xv + 8 * m);
        const bool b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // exchange 2 x 2 blocks of chunks with lane ^ 2
          const uint4 snd = b1 ? ch[m] : ch[m + 2];
          uint4 rcv;
          rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, 2);
          rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, 2);
          rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, 2);
          rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, 2);
          if (b1) ch[m] = rcv; else ch[m + 2] = rcv;
        }
#pragma unroll
        for (int k2 = 0; k2 < 4; k2 += 2) {  // then single chunks with lane ^ 1
          const uint4 snd = b0 ? ch[k2] : ch[k2 + 1];
          uint4 rcv;
          rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, 1);
          rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, 1);
          rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, 1);
          rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, 1);
          if (b0) ch[k2] = rcv; else ch[k2 + 1] = rcv;
        }
        // lane 4i + j now holds chunk j of rows 4i .. 4i + 3 (of this warp's 32)
        const int g4 = lane & ~3, jc = lane & 3;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int r = t0 + 32 * q4 + g4 + m;
          if (r < s1)
            *reinterpret_cast<uint4*>(out + ((row0 + r) * a.H + h) * D + 32 * gw + 8 * jc) = ch[m];
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_xfree);
      if (!bad && gw < NG && t < D) {
        float v[32];
        tmem_ld32(tmem + tl + L::TS + 32 * gw, v);
        store_row32<true>(base + L::SS, t, gw, v);
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_sconv);
      if (bad) atomicExch(s_abort, 1);
      // the quarter's four warps leave together (they meet at its named barrier every chunk)
      if (feat::group_sync_or(kBarQuarter + q4, 128, *reinterpret_cast<volatile int*>(s_abort))) break;
    }
    if (bad) atomicExch(s_abort, 1);
  } else {
  tc::regs_dec<kRegsOther>();  // one call site for the last two warpgroups
  if (warp < kWarpIssue) {
    // ================================================================ rectifiers (warps 16-21)
    // q' = ReLU(q), k' = ReLU(k) in place, as soon as a slot's raw rows have landed
    const int rt = tid - 32 * kConvWarps;
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    for (int c = 0; c < nch && !bad0; ++c) {
      const int s = c & 1;
      const bool ok = tc::mbar_wait(bar_qkfull + 8 * s, (c >> 1) & 1, kWait);
      if (!ok) atomicExch(s_abort, 1);
      if (*reinterpret_cast<volatile int*>(s_abort)) break;
      const uint32_t qb = base + (s ? L::Q1 : L::Q0), kb = base + (s ? L::K1 : L::K0);
#pragma unroll 4
      for (int idx = rt; idx < 2 * kC * CPR; idx += 32 * kRectWarps) {
        const int r = (idx / CPR) & (kC - 1), m = idx % CPR;
        const uint32_t addr = (idx < kC * CPR ? qb : kb) + tile_off(r, m);
        sts16(addr, relu8(lds16(addr)));
      }
      tc::fence_async_smem();
      tc::mbar_arrive(bar_qkready + 8 * s);
    }
  } else if (warp == kWarpIssue) {
    // ================================================================ MMA issue (one thread)
    if (lane == 0 && !bad0) {
      constexpr uint32_t ID_P = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_KM = tc::idesc_bf16(128, D, false, true);
      constexpr uint32_t ID_MM = tc::idesc_bf16(128, D, true, true);
      int ok = 1;
      for (int c = 0; c < nch && ok; ++c) {
        const int s = c & 1;
        const uint32_t qf = base + (s ? L::Q1 : L::Q0), kf = base + (s ? L::K1 : L::K0);
        ok = tc::mbar_wait(bar_qkready + 8 * s, (c >> 1) & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
        // P = Q'K'^T (P~ of the previous chunk has been read by its P~V, issued before)
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_bf16(tmem + L::TP, kmaj(qf, kk), kmaj(kf, kk), ID_P, kk > 0);
        // X = Q'A~, once the previous numerator has been read and A~ holds the state before the chunk
        ok = (c == 0 || tc::mbar_wait(bar_xfree, (c - 1) & 1, kWait)) && tc::mbar_wait(bar_aconv, c & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_bf16(tmem + L::TX, kmaj(qf, kk), mnmaj(base + L::AS, kk, D * 128), ID_KM, kk > 0);
        tc::mma_commit(bar_g1);
        // S += K'^T V, A += K'^T K', once S~ and A~ have been taken from them and v has landed
        ok = tc::mbar_wait(bar_sconv, c & 1, kWait) && tc::mbar_wait(bar_vfull, c & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int kk = 0; kk < kC / 16; ++kk) {
          tc::mma_bf16(tmem + L::TS, mnmaj(kf, kk, 16384), mnmaj(base + L::VS, kk, 16384), ID_MM, 1u);
          tc::mma_bf16(tmem + L::TA, mnmaj(kf, kk, 16384), mnmaj(kf, kk, 16384), ID_MM, 1u);
        }
        tc::mma_commit(bar_g2);
        // X = Q'S~ + P~V, once the converters have written P~ and read q'A~ (S~ still holds the
        // state before the chunk: its update waits for this group)
        ok = tc::mbar_wait(bar_conv1, c & 1, kWait);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_bf16(tmem + L::TX, kmaj(qf, kk), mnmaj(base + L::SS, kk, D * 128), ID_KM, kk > 0);
#pragma unroll 1
        for (int kk = 0; kk < kC / 16; ++kk)  // keys 16 kk .. + 15: columns 32 (kk / 2) + 16 + 8 (kk % 2)
          tc::mma_bf16_ta(tmem + L::TX, tmem + L::TP + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                          mnmaj(base + L::VS, kk, 16384), ID_KM, 1u);
        tc::mma_commit(bar_g3);
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else {
    // ================================================================ TMA loads (one thread)
    if (lane == 0 && !bad0) {
      int ok = 1;
      for (int c = 0; c < 2 && c < nch; ++c) {
        tc::mbar_arrive_expect_tx(bar_qkfull + 8 * c, 2 * L::TILE);
        tma_tile<D>(&tq, base + (c ? L::Q1 : L::Q0), h, static_cast<int>(row0 + s0 + c * kC), bar_qkfull + 8 * c);
        tma_tile<D>(&tk, base + (c ? L::K1 : L::K0), h, static_cast<int>(row0 + s0 + c * kC), bar_qkfull + 8 * c);
      }
      tc::mbar_arrive_expect_tx(bar_vfull, L::TILE);
      tma_tile<D>(&tv, base + L::VS, h, static_cast<int>(row0 + s0), bar_vfull);
      // v has one buffer, so each v load waits for the previous chunk's products: its rows are
      // fetched into L2 a chunk earlier, and the load itself then finds them there
      auto prefetch_v = [&](int cc) {
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb) tc::tma_prefetch_3d(&tv, 64 * jb, h, static_cast<int>(row0 + s0 + cc * kC));
      };
      if (nch > 1) prefetch_v(1);
      for (int c = 0; c < nch; ++c) {
        // chunk c's MMAs are done with its q, k and v: the next v, and the q and k two chunks on
        ok = tc::mbar_wait(bar_g3, c & 1, kWait);
        if (!ok || *reinterpret_cast<volatile int*>(s_abort)) break;
        const int s = c & 1, t0 = s0 + c * kC;
        if (c + 1 < nch) {
          tc::mbar_arrive_expect_tx(bar_vfull, L::TILE);
          tma_tile<D>(&tv, base + L::VS, h, static_cast<int>(row0 + t0 + kC), bar_vfull);
        }
        if (c + 2 < nch) {
          prefetch_v(c + 2);
          tc::mbar_arrive_expect_tx(bar_qkfull + 8 * s, 2 * L::TILE);
          tma_tile<D>(&tq, base + (s ? L::Q1 : L::Q0), h, static_cast<int>(row0 + t0 + 2 * kC), bar_qkfull + 8 * s);
          tma_tile<D>(&tk, base + (s ? L::K1 : L::K0), h, static_cast<int>(row0 + t0 + 2 * kC), bar_qkfull + 8 * s);
        }
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  }
  }

  tc::fence_before_sync();
  __syncthreads();
  const bool bad = *reinterpret_cast<volatile int*>(s_abort) != 0;
  if (bad && tid == 0 && !misaligned) {
    // bounded chances for the copies and MMAs still in flight to land before the memory is released
    for (int i = 0; i < 2; ++i) tc::mbar_wait(bar_qkfull + 8 * i, 0, kWait / 4);
    tc::mbar_wait(bar_vfull, 0, kWait / 4);
    tc::mbar_wait(bar_g3, 0, kWait / 4);
  }
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
