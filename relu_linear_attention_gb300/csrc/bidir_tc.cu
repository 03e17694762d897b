// Bidirectional (non-causal) RLA-2 on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a;
// bf16 inputs, d in {64, 128}, fp32 accumulation.
//
// The method (08-rapt-algorithm.md §4.1, the prefix scan's causal=false mode, and §4.2, the
// bidirectional branch of the Sum-denominator layer; formula and eps of §3):
//   q' = ReLU(RoPE(RMSNorm(q))), k' likewise;  over the whole document
//   S = K'^T V (d x d),  z = sum_tau k'_tau,  out_t = q'_t S / (q'_t . z + eps)
// so the L x L score matrix is never formed. Two launches on the caller's stream:
//   1. state blocks: the causal prefill's state kernel in whole-document mode, i.e. K'^T V and the
//      column sums of k' of every block of blk_len tokens (features on 16 producer warps, one GEMM
//      per 128-token chunk into TMEM), fp32 records in the workspace;
//   2. readout, one CTA per (document, head, run of 128-token tiles), a programmatic dependent of
//      launch 1: q tiles arrive by TMA from the start; once launch 1 is complete, the twenty
//      epilogue and feature warps sum the document's block records in block order (deterministic)
//      straight into the bf16 B operand of S in shared memory (the layout the tensor core reads)
//      and z in fp32; sixteen feature warps turn each q tile into q' in place, several rows at a
//      time, and form the fp32 q'.z of every row; one thread issues O = Q' S into one of two TMEM
//      accumulators; four epilogue warps scale O by 1 / (q'.z + eps) and stage whole tiles for a
//      TMA store (the ragged last tile of a document is written row by row, so no store reaches
//      past it).
// Every wait is bounded; a readout CTA whose wait gives up writes NaN over its rows and sets
// RAPT_DEV_INTERNAL.
#include <cuda.h>

#include <cstring>

#include "kernels.h"
#include "tc_features.cuh"
#include "tc_utils.cuh"
#include "tensor_map.h"

namespace rapt {
namespace {

using namespace feat;

constexpr int kC = 128;                    // tokens per tile = MMA M
constexpr long long kWait = 2000000000LL;  // ~1 s
constexpr int kStages = 5;                 // q tiles in flight
constexpr int kEpi = 128;                  // warps 0-3: epilogue (one TMEM lane quarter each)
constexpr int kFeat = 512;                 // the next warps: features (16)
constexpr int kWarpTma = (kEpi + kFeat) / 32;  // then one TMA warp and one MMA warp
constexpr int kWarpMma = kWarpTma + 1;
constexpr int kThreads = kEpi + kFeat + 64;
constexpr uint32_t kDevBadDoc = 1u, kDevInternal = 2u;

// The document's state in the readout CTA: S as the bf16 B operand (rows = K = feature i,
// 64-column blocks of N = value column j, each block D rows x 128 bytes, 16-byte chunk c of row i
// at c ^ (i & 7)), then z (D floats).
template <int D>
struct Img {
  static constexpr uint32_t S_BYTES = D * D * 2;
  static constexpr uint32_t BYTES = S_BYTES + D * 4;
};
constexpr int kBuild = kEpi + kFeat;  // threads that build the state operand

// Feature mapping of the readout: a thread owns 8 consecutive elements (one 16-byte chunk, four
// RoPE pairs) of one row; TPR threads per row, RPP rows per pass.
template <int D>
struct FeatMap {
  static constexpr int TPR = D / 8;
  static constexpr int RPP = kFeat / TPR;
  static constexpr int NPASS = kC / RPP;
};

template <int D>
struct Lay {
  static constexpr int DB = D / 64;
  static constexpr uint32_t QT = DB * 16384;                          // one q tile
  static constexpr uint32_t QS = (Img<D>::BYTES + 1023) / 1024 * 1024;  // q tiles (after S and z)
  static constexpr uint32_t INV = QS + kStages * QT;                  // 1 / den [stage][128]
  static constexpr uint32_t TAB = INV + kStages * kC * 4;             // FeatTab (8 D floats)
  // sready, qfull[S], feat[S], staged[S], accf[2], accfree[2]
  static constexpr uint32_t BAR = TAB + 8 * D * 4;
  static constexpr uint32_t MISC = BAR + (1 + 3 * kStages + 4) * 8;   // TMEM base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(QT % 1024 == 0, "tile alignment");
  static_assert(BYTES <= 232448, "shared memory budget");
};

// ------------------------------------------------------------------------------------------------
// Launch 2: readout.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bidir_readout(const PrefillArgs a, int nsplit, int split_chunks, const float* recs, int blk_len,
                  int nblk_max, const __grid_constant__ CUtensorMap tq,
                  const __grid_constant__ CUtensorMap to) {
  using L = Lay<D>;
  using FM = FeatMap<D>;
  constexpr int S = kStages, TPR = FM::TPR, RPP = FM::RPP, NPASS = FM::NPASS;
  constexpr int NB = NPASS < 4 ? NPASS : 4;  // feature rows a thread works on at once
  static_assert(NPASS % NB == 0, "feature batches");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.x % nsplit, unit = blockIdx.x / nsplit;
  const int doc = unit / a.H, h = unit % a.H;
  long row0;
  int n;
  if (!doc_bounds(a, doc, row0, n)) {
    if (sp == 0 && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevBadDoc);
    return;
  }
  const int c0 = sp * split_chunks;
  const int ntile = min((n + kC - 1) / kC, c0 + split_chunks) - c0;
  if (ntile <= 0) return;  // uniform, before any allocation

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  const uint32_t bar_m = base + L::BAR, bar_qfull = bar_m + 8, bar_feat = bar_qfull + 8 * S;
  const uint32_t bar_staged = bar_feat + 8 * S, bar_accf = bar_staged + 8 * S, bar_accfree = bar_accf + 16;
  float* inv_den = reinterpret_cast<float*>(smem + L::INV);
  const float* zs = reinterpret_cast<const float*>(smem + Img<D>::S_BYTES);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);
  const bool misaligned = (base & 1023u) != 0;  // uniform; the swizzled layouts need 1 KB

  if (warp == 0 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 2 * D);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_m, kBuild);
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(bar_qfull + 8 * s, 1);
      tc::mbar_init(bar_feat + 8 * s, kFeat);
      tc::mbar_init(bar_staged + 8 * s, kEpi);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(bar_accf + 8 * x, 1);
      tc::mbar_init(bar_accfree + 8 * x, kEpi);
    }
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  const FeatTab tab = feat_tab<D>(smem + L::TAB);
  fill_tab<D>(tab, a, h, RPP, tid, kThreads);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const bool run = !*s_abort;
  auto tile = [&](int s) { return base + L::QS + s * L::QT; };
  auto whole = [&](int i) { return (c0 + i) * kC + kC <= n; };

  if (warp < kWarpTma) {
    // S and z of the document: launch 1's block records, summed in block order
    tc::grid_dep_wait();
    if (run) {
      const float* rec = recs + static_cast<long>(unit) * nblk_max * Rec<D>::FLOATS;
      const int nblk = (n + blk_len - 1) / blk_len;
      for (int e = tid; e < D * D / 4; e += kBuild) {
        float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b = 0; b < nblk; ++b) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(rec + b * Rec<D>::FLOATS) + e);
          m.x += x.x; m.y += x.y; m.z += x.z; m.w += x.w;
        }
        // record float4 e holds row i = e % D, columns 4 (e / D) .. + 3
        const int i = e % D, j = 4 * (e / D);
        const int jb = j / 64, cc = (j % 64) / 8, half = (j % 8) / 4;
        *reinterpret_cast<uint2*>(smem + jb * (D * 128) + i * 128 + ((cc ^ (i & 7)) << 4) + half * 8) =
            make_uint2(tc::pack_bf16x2(m.x, m.y), tc::pack_bf16x2(m.z, m.w));
      }
      if (tid < D) {
        float z = 0.f;
        for (int b = 0; b < nblk; ++b) z += __ldcg(rec + b * Rec<D>::FLOATS + Rec<D>::Z + tid);
        reinterpret_cast<float*>(smem + Img<D>::S_BYTES)[tid] = z;
      }
      tc::fence_async_smem();
      tc::mbar_arrive(bar_m);
    }
  }
  if (warp == kWarpTma) {
    if (lane == 0 && run) {  // TMA: q tiles in, whole output tiles back
      int ok = 1;
      for (int i = 0; i < ntile + S && ok; ++i) {
        if (i >= S) {  // the tile S back is staged: store it (if whole), then its buffer is free
          const int j = i - S, s = j % S;
          ok = tc::mbar_wait(bar_staged + 8 * s, (j / S) & 1, kWait);
          if (!ok) break;
          if (whole(j)) {
#pragma unroll
            for (int jb = 0; jb < L::DB; ++jb)
              tc::tma_store_3d(&to, tile(s) + jb * 16384, 64 * jb, h, static_cast<int>(row0 + (c0 + j) * kC));
            tc::bulk_commit();
            tc::bulk_wait_read0();
          }
        }
        if (i < ntile) {
          const int s = i % S;
          tc::mbar_arrive_expect_tx(bar_qfull + 8 * s, L::QT);
#pragma unroll
          for (int jb = 0; jb < L::DB; ++jb)
            tc::tma_load_3d(tile(s) + jb * 16384, &tq, 64 * jb, h, static_cast<int>(row0 + (c0 + i) * kC),
                            bar_qfull + 8 * s);
        }
      }
      if (!ok) atomicExch(s_abort, 1);
      tc::bulk_wait0();
    }
  } else if (warp == kWarpMma) {
    if (lane == 0 && run) {  // MMA: O = Q' S, M = 128 tokens, N = K = d
      constexpr uint32_t ID = tc::idesc_bf16(128, D, false, true);
      const uint64_t dm = tc::desc_sw128(base, D * 128, 1024);
      int ok = tc::mbar_wait(bar_m, 0, kWait);
      for (int i = 0; i < ntile && ok; ++i) {
        const int s = i % S, x = i & 1;
        ok = tc::mbar_wait(bar_feat + 8 * s, (i / S) & 1, kWait) &&
             (i < 2 || tc::mbar_wait(bar_accfree + 8 * x, ((i >> 1) - 1) & 1, kWait));
        if (!ok) break;
        tc::fence_after_sync();
        const uint64_t dq = tc::desc_sw128(tile(s), 16, 1024);
#pragma unroll 1
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t kofs = static_cast<uint64_t>((k / 4) * 1024 + (k % 4) * 2);
          tc::mma_bf16(tmem + x * D, dq + kofs, dm + static_cast<uint64_t>(k) * 128, ID, k > 0);
        }
        tc::mma_commit(bar_accf + 8 * x);
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else if (warp >= kEpi / 32) {
    if (run) {  // features of the q tiles, in place, and 1 / (q'.z + eps) of every row
      const int ft = tid - kEpi;
      const int prow = ft / TPR, part = ft % TPR, e0 = 8 * part;
      const uint32_t cblk = static_cast<uint32_t>(e0 / 64) * 16384;
      const int cidx = (e0 % 64) / 8;
      float2 gq0[2], gq1[2];
      split_load<D>(tab.gq, part, gq0, gq1);
      Rot step;
      tab_step(tab, e0 / 2, step);
      // waits are made warp-uniform: the passes shuffle across the whole warp
      int ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_m, 0, kWait));
      // z of this thread's elements in pair groups (first / second elements of pairs 2g, 2g+1)
      const float4 za = *reinterpret_cast<const float4*>(zs + e0);
      const float4 zb = *reinterpret_cast<const float4*>(zs + e0 + 4);
      const float2 zx0[2] = {make_float2(za.x, za.z), make_float2(zb.x, zb.z)};
      const float2 zx1[2] = {make_float2(za.y, za.w), make_float2(zb.y, zb.w)};
      for (int i = 0; i < ntile && ok; ++i) {
        const int s = i % S;
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_qfull + 8 * s, (i / S) & 1, kWait));
        if (!ok) break;
        Rot rot;  // angles of this thread's first row of the tile, exact
        tab_rot_at(tab, a.pos_offset + (c0 + i) * kC + prow, e0 / 2, rot);
        float* inv = inv_den + s * kC;
        const uint32_t tb = tile(s) - base + cblk;  // byte offset of this thread's column block
        // NB rows at a time: their loads, row reductions and shuffles are independent, so their
        // latencies overlap (one row per pass would leave every step of the chain exposed)
#pragma unroll 1
        for (int p0 = 0; p0 < NPASS; p0 += NB) {
          Pairs f[NB];
          float red[NB];
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            f[b] = unpack_pairs(*reinterpret_cast<const uint4*>(smem + tb + tc::sw128((p0 + b) * RPP + prow, cidx)));
            red[b] = sumsq(f[b]);
          }
#pragma unroll
          for (int b = 0; b < NB; ++b) red[b] = row_sum<TPR>(red[b]);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (p0 + b > 0) rot_step(rot, step);
            float2 g0[2] = {gq0[0], gq0[1]}, g1[2] = {gq1[0], gq1[1]};
            scale_gains(g0, g1, rsqrtf(red[b] * (1.0f / D) + a.fa.eps_norm));
            rope_relu(f[b], g0, g1, rot);
            float2 d2 = __fmul2_rn(f[b].x0[0], zx0[0]);
            d2 = __ffma2_rn(f[b].x1[0], zx1[0], d2);
            d2 = __ffma2_rn(f[b].x0[1], zx0[1], d2);
            d2 = __ffma2_rn(f[b].x1[1], zx1[1], d2);
            red[b] = d2.x + d2.y;
          }
#pragma unroll
          for (int b = 0; b < NB; ++b) red[b] = row_sum<TPR>(red[b]);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const int r = (p0 + b) * RPP + prow;
            if (part == 0) inv[r] = 1.0f / (red[b] + a.eps_den);
            sts16(base + tb + tc::sw128(r, cidx), pack_pairs(f[b]));
          }
        }
        tc::fence_async_smem();
        tc::mbar_arrive(bar_feat + 8 * s);
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else if (run) {
    // epilogue: TMEM lane = tile row er (warps 0-3, one lane quarter each)
    static_assert(kEpi == 128, "one epilogue warp per TMEM lane quarter");
    const int er = 32 * warp + lane;
    const uint32_t tl = static_cast<uint32_t>(32 * warp) << 16;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out);
    for (int i = 0; i < ntile; ++i) {
      const int s = i % S, x = i & 1;
      // feat[s] completed before the MMA began; waiting on it makes the 1 / den values visible
      const int ok = tc::mbar_wait(bar_accf + 8 * x, (i >> 1) & 1, kWait) &&
                     tc::mbar_wait(bar_feat + 8 * s, (i / S) & 1, kWait);
      if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform, so TMEM loads stay converged
        atomicExch(s_abort, 1);
        break;
      }
      tc::fence_after_sync();
      const float inv = inv_den[s * kC + er];
      const bool full = whole(i);
      const int lt = (c0 + i) * kC + er;
      __nv_bfloat16* orow = og + ((row0 + lt) * a.H + h) * D;
      const uint32_t acc = tmem + tl + x * D;
#pragma unroll 1
      for (int j0 = 0; j0 < D; j0 += 32) {
        uint32_t u[2][16];
        tc::tmem_ld16(acc + j0, u[0]);
        tc::tmem_ld16(acc + j0 + 16, u[1]);
        tc::tmem_wait_ld();
        const uint32_t blk = tile(s) + static_cast<uint32_t>(j0 / 64) * 16384;
        const int cc = (j0 % 64) / 8;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float f[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(u[m][e]) * inv;
          if (full) {  // over q' of the same row: the finished GEMM has read it
            sts16(blk + tc::sw128(er, cc + 2 * m), pack8(f));
            sts16(blk + tc::sw128(er, cc + 2 * m + 1), pack8(f + 8));
          } else if (lt < n) {
            uint4* dst = reinterpret_cast<uint4*>(orow + j0 + 16 * m);
            dst[0] = pack8(f);
            dst[1] = pack8(f + 8);
          }
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(bar_accfree + 8 * x);
      if (full) tc::fence_async_smem();
      tc::mbar_arrive(bar_staged + 8 * s);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*s_abort) {  // a wait gave up: this CTA's rows read as NaN rather than as a result
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevInternal);
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out);
    const __nv_bfloat16 nan = __float2bfloat16(__int_as_float(0x7fc00000));
    for (long r = tid; r < static_cast<long>(ntile) * kC * D; r += kThreads) {
      const long t = static_cast<long>(c0) * kC + r / D;
      if (t < n) og[((row0 + t) * a.H + h) * D + r % D] = nan;
    }
  }
  if (warp == 0 && !misaligned) tc::tmem_dealloc(tmem, 2 * D);
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

template <int D>
cudaError_t launch_d(const PrefillArgs& a, const BidirPlan& plan, void* ws, cudaStream_t stream) {
  static unsigned long long cfg = 0;
  cudaError_t e = set_smem(bidir_readout<D>, Lay<D>::BYTES, cfg);
  if (e != cudaSuccess) return e;
  const long units = static_cast<long>(a.n_docs) * a.H;
  if (units == 0 || a.total_rows == 0) return cudaSuccess;
  TcArgs ta{};
  ta.p = a;
  ta.ws = static_cast<float*>(ws);
  ta.seg_len = plan.blk_len;
  ta.nseg_max = 1;
  ta.blk_len = plan.blk_len;
  ta.blk_per_seg = 1;
  ta.nblk_max = plan.nblk_max;
  ta.whole_doc = 1;
  CUtensorMap tq, to;
  e = make_rows_map(&tq, a.q, a.total_rows, a.H, D);
  if (e == cudaSuccess) e = make_rows_map(&to, a.out, a.total_rows, a.H, D);
  if (e != cudaSuccess) return e;
  e = launch_state_tc(D, ta, stream);
  if (e != cudaSuccess) return e;
  // the readout is a programmatic dependent of the state launch: its CTAs start as that launch's
  // finish and wait for it (griddepcontrol.wait) before reading the records
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.stream = stream;
  c.attrs = pdl;
  c.numAttrs = 1;
  c.gridDim = dim3(static_cast<unsigned>(units * plan.nsplit));
  c.blockDim = dim3(kThreads);
  c.dynamicSmemBytes = Lay<D>::BYTES;
  e = cudaLaunchKernelEx(&c, bidir_readout<D>, a, plan.nsplit, plan.split_chunks,
                         static_cast<const float*>(ws), plan.blk_len, plan.nblk_max, tq, to);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

BidirPlan bidir_plan(int n_docs, int H, int max_seqlen, int d) {
  // Launch 1 runs one CTA per SM: pick the block length (in 128-token chunks) that minimises
  // waves x (chunks per block + about one chunk of set-up and write-out). Launch 3 likewise: the
  // split of each document's tiles that minimises waves x tiles per CTA. Ties go to fewer CTAs.
  BidirPlan p{};
  const long units = static_cast<long>(n_docs) * H;
  const int chunks = max_seqlen > 0 ? (max_seqlen + kC - 1) / kC : 1;
  double best = 1e300;
  for (int cpb = chunks; cpb >= 1; --cpb) {
    const long nblk = (chunks + cpb - 1) / cpb;
    const double cost = static_cast<double>((units * nblk + 151) / 152) * (cpb + 1.0);
    if (cost < best) {
      best = cost;
      p.blk_len = cpb * kC;
      p.nblk_max = static_cast<int>(nblk);
    }
  }
  best = 1e300;
  for (int ns = 1; ns <= chunks; ++ns) {
    const int per = (chunks + ns - 1) / ns;
    if (ns > 1 && (ns - 1) * per >= chunks) continue;  // a split with no tile
    const double cost = static_cast<double>((units * ns + 151) / 152) * (per + 1.0);
    if (cost < best) {
      best = cost;
      p.nsplit = ns;
      p.split_chunks = per;
    }
  }
  const size_t rec = static_cast<size_t>(d) * (d + 1) * sizeof(float);
  p.ws_bytes = static_cast<size_t>(units) * p.nblk_max * rec;
  return p;
}

cudaError_t launch_bidir_tc(int d, const PrefillArgs& a, const BidirPlan& plan, void* ws,
                            cudaStream_t stream) {
  return d == 128 ? launch_d<128>(a, plan, ws, stream) : launch_d<64>(a, plan, ws, stream);
}

}  // namespace rapt
