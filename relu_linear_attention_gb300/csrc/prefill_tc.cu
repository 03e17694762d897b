// Chunked causal RLA-2 forward on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
// bf16 inputs, d in {64, 128}; fp32 accumulation and fp32 state.
//
// The method (08-rapt-algorithm.md §3): q' = ReLU(RoPE(RMSNorm(q))), k' likewise,
// S_t = S_{t-1} + k'_t v_t^T, z_t = z_{t-1} + k'_t, out_t = q'_t S_t / (q'_t . z_t + 1e-4), with
// the state restarting at every document (§2.2, §4.1). It is evaluated chunk by chunk (C = 128
// tokens, the chunk-parallel form of §1 and §3) as four bf16 x bf16 -> fp32 tile GEMMs per chunk:
//
//   O  = Q'_c S~_{c-1}        (128 x d)    -> TMEM   (inter-chunk part; ~ = bf16 copy)
//   S += K'_c^T V_c           (d x d)      -> TMEM   (fp32 master state)
//   P  = Q'_c K'_c^T          (128 x 128)  -> TMEM
//   O += P~_c V_c             (P masked to tau <= t, rounded to bf16)
//   out = O / (q'.z_{c-1} + rowsum(P~_c) + eps)
//
// The denominator stays on the CUDA cores in fp32: z is a column sum of k' kept in shared memory,
// q'.z is formed while the features are computed, and the row sums of the masked fp32 scores
// while P is converted to the bf16 operand of the intra-chunk product.
//
// Kernel B is warp-specialised (896 threads, one CTA per SM):
//   warps 0-15  (producers):  RMSNorm, RoPE and ReLU of chunk c+1 while the tensor core works on
//                             chunk c. Raw q arrives by TMA in one of two q' buffers and q' is
//                             written back in place; k comes through registers two passes ahead
//                             and k' is held there until the single k' buffer is free. Features
//                             are the bulk of the CUDA-core work, so they get most of the warps;
//   warps 16-23 (converters): two per TMEM lane quarter (32 tile rows), half of the columns each:
//                             q'.z_{c-1} from the q' tile, P -> masked bf16 P~ written back into
//                             TMEM (the A operand of P~V) with the row sums of the masked scores,
//                             S -> S~ in shared memory, then the epilogue O / den from one of two
//                             O accumulators, staged in the chunk's v buffer;
//   warp 24     (issuer):     one thread issues the MMAs (P, then QS, KV, PV) and commits them to
//                             mbarriers;
//   warp 25     (TMA):        one thread loads raw q two chunks ahead (once both products and the
//                             converters have read the buffer), writes each staged output tile with
//                             TMA stores and loads the v tile of two chunks later into the freed
//                             buffer;
//   warps 26-27 (z helpers):  z_c = z_{c-1} + the column sums of the bf16 k' tile, into a ring of
//                             three slots that the converters read.
// Hand-offs are mbarriers: qfull[2] (TMA -> producers), full[2] (producers -> issuer, converters,
// helpers), vfull[2] (TMA -> issuer), empty[2] (both products and the converters' q'.z done with a
// q' buffer), p_done, kv_done, b_done (tensor core -> converters), kfree (k' read by the MMAs and
// the helpers), pconv / sconv (converters -> issuer: P~ and S~ written), staged[2] / ofree[2]
// (converters -> TMA thread / issuer), zfull[3] / zempty[3] (the z ring). Every ring has as many
// phases in flight as its depth, so no waiter can be lapped. Every wait is bounded; a wait that
// gives up sets RAPT_DEV_INTERNAL in the caller's status word and the CTA winds down.
//
// Sequence parallelism: a document is cut into segments of seg_len tokens. Kernel A computes the
// state increments (K'^T V and sum k') of the parts of the document that precede its last
// segment, in blocks of blk_len tokens (a segment holds blk_per_seg blocks, so that kernel A has
// enough CTAs to fill the GPU); kernel B runs one CTA per (document, head, segment) starting from
// S0 + the increments of the blocks before the segment (added in block order: deterministic). The
// last segment's CTA writes the final state. Kernel B is launched as a programmatic dependent of
// kernel A: its CTAs set up and compute their first features while kernel A finishes, and wait
// for it only where they read the increments.
#include <cuda.h>

#include <cstring>

#include "kernels.h"
#include "tc_utils.cuh"
#include "tc_features.cuh"
#include "tensor_map.h"

namespace rapt {
namespace {

using namespace feat;

// 16-byte shared-memory accesses as plain C++ (at byte offset off from the dynamic shared base), so
// that the compiler may schedule them freely; ordering with the tensor core and the TMA comes from
// the fences and barriers, which are compiler barriers.
__device__ __forceinline__ void st_shared16(uint8_t* sm, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(sm + off) = v;
}
__device__ __forceinline__ uint4 ld_shared16(const uint8_t* sm, uint32_t off) {
  return *reinterpret_cast<const uint4*>(sm + off);
}

constexpr int kC = 128;          // chunk length = MMA M
constexpr int kProd = 512;       // producer threads (16 warps)
constexpr int kConv = 256;       // converter threads of kernel B (8 warps, two per TMEM lane quarter)
constexpr int kHelp = 64;        // z helper threads of kernel B (2 warps)
constexpr int kThreadsB = kProd + kConv + 128;  // + issuer, store and z helper warps
constexpr int kWarpIssue = (kProd + kConv) / 32;  // kernel B's MMA issuer warp
constexpr int kWarpStore = kWarpIssue + 1;        // kernel B's TMA store / v load warp
constexpr int kThreadsA = kProd + 128;          // kernel A: producers + issuer warpgroup
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s: a tensor-core step that is not done by then never will be
constexpr uint32_t kDevInternal = 2u;
constexpr uint32_t kBarProd = 1, kBarConv = 2;   // named barriers of the producer / converter groups
constexpr uint32_t kBarHelp = 4;                 // the two z helper warps
constexpr uint32_t kBarQuarter = 5;              // 5..8: the two converter warps of a lane quarter

// Register splits (setmaxnreg draws on the launch allocation: threads x launch registers).
constexpr int kLaunchRegsB = 72, kRegsProdB = 80, kRegsConvB = 64, kRegsIssueB = 56;
static_assert(kProd * kRegsProdB + kConv * kRegsConvB + 128 * kRegsIssueB <= kThreadsB * kLaunchRegsB,
              "kernel B register split exceeds the launch allocation");
constexpr int kLaunchRegsA = 96, kRegsProdA = 96, kRegsIssueA = 96;
static_assert(kProd * kRegsProdA + 128 * kRegsIssueA <= kThreadsA * kLaunchRegsA,
              "kernel A register split exceeds the launch allocation");

// Producer mapping: a thread owns 8 consecutive elements (one 16-byte chunk, four RoPE pairs) of
// one token row.
template <int D>
struct Prod {
  static constexpr int TPR = D / 8;          // threads per row
  static constexpr int RPP = kProd / TPR;    // rows per pass
  static constexpr int NPASS = kC / RPP;     // passes per chunk
  static constexpr int WARPS = kProd / 32;
  static constexpr uint32_t TILE = (D / 64) * 16384;  // one 128-row bf16 tile of d columns
};

// Kernel B shared memory (byte offsets from a 1024-byte aligned base). With PAIR (D = 128), the
// tiles hold two heads of 64 (columns 0-63 and 64-127).
template <int D, bool PAIR = false>
struct LayB {
  static constexpr uint32_t TILE = Prod<D>::TILE;
  static constexpr uint32_t Q0 = 0, Q1 = TILE;                 // raw q (TMA), turned into q' in place
  static constexpr uint32_t V0 = 2 * TILE, V1 = 3 * TILE;      // v, then the staged output
  static constexpr uint32_t KS = 4 * TILE;                     // k' : 2 x 16 KB (d = 64: + zero block)
  static constexpr uint32_t SS = KS + 32768;                   // S~ : D/64 blocks of D rows x 128 B
  static constexpr uint32_t ZS = SS + (D / 64) * D * 128;      // z ring [3][D] fp32
  static constexpr uint32_t DI = ZS + 3 * D * 4;               // q'.z halves [2 buffers][2 halves][128]
  static constexpr uint32_t RS = DI + 2 * 2 * kC * 4;          // masked score row sums, same shape
  static constexpr uint32_t ZH = RS + 2 * 2 * kC * 4;          // helpers' partial column sums [64 / (D / 8)][D]
  static constexpr uint32_t TAB = ZH + (64 / (D / 8)) * D * 4;  // feature tables (FeatTab)
  // full[2] vfull[2] empty[2] p_done kv_done kfree pconv sconv b_done ofree[2] staged[2]
  // zfull[3] zempty[3] qfull[2]
  static constexpr uint32_t BAR = TAB + 8 * D * 4;
  static constexpr int NBAR = 24;
  static constexpr uint32_t MISC = BAR + NBAR * 8;             // TMEM base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  // TMEM columns: P (fp32 scores; the bf16 P~ is written over columns [0, 32) and [64, 96)), two
  // O accumulators, S. PAIR: the two heads' scores (P~ over the first 64 columns of each), one
  // O accumulator for both heads, S.
  static constexpr uint32_t TP = 0, TP1 = 128;
  static constexpr uint32_t TO0 = PAIR ? 256 : 128, TO1 = PAIR ? 256 : 128 + D;
  static constexpr uint32_t TS = PAIR ? 384 : 128 + 2 * D;
  static_assert(TS + D <= 512, "TMEM budget");
  static_assert(!PAIR || D == 128, "head pairs fill 128-column tiles");
  static_assert(BYTES <= 232448, "shared memory budget");
};

// Kernel A shared memory: a ring of kStagesA stages, each the raw k tile (TMA; turned into k' in
// place; d = 64 adds the zero block that pads k'^T to M = 128) and the v tile.
constexpr int kStagesA = 3;
template <int D>
struct LayA {
  static constexpr uint32_t TILE = Prod<D>::TILE;
  static constexpr uint32_t KT = 32768;                                // one k' stage
  static constexpr uint32_t K0 = 0;                                    // k' stages
  static constexpr uint32_t V0 = kStagesA * KT;                        // v stages
  static constexpr uint32_t ZP = V0 + kStagesA * TILE;                 // z partials [producer warps][D]
  static constexpr uint32_t TAB = ZP + Prod<D>::WARPS * D * 4;         // feature tables (FeatTab)
  static constexpr uint32_t BAR = TAB + 8 * D * 4;  // kfull[S] vfull[S] ready[S] free[S]
  static constexpr uint32_t MISC = BAR + 4 * kStagesA * 8;
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(BYTES <= 232448, "shared memory budget");
};

// Initial state of a segment for columns [c0, c0 + D/2) of the calling thread's TMEM lane er:
// S0 (if any) + the increments of the first nblk blocks, in block order, into the fp32 state in
// TMEM (tmem_s: lane and column base of S) and its bf16 copy S~ in shared memory (ss). Heads of DH
// (= D, or 64 for a pair of heads in a 128-wide tile): lane er is row er % DH of head er / DH (bh +
// er / DH, whose records start rec_head floats after the first head's), and the state is block
// diagonal: columns of the other head, and TMEM rows >= D of a single head, are zero. Eight
// columns at a time, with two blocks' loads in flight.
template <int D, int DH = D>
__device__ __forceinline__ void init_state(const PrefillArgs& a, const float* wsb, long rec_head,
                                           int nblk, long bh, int er, uint32_t tmem_s, uint32_t ss,
                                           int c0) {
  const int hh = DH == D ? 0 : er / DH, r = DH == D ? er : er % DH;
  const bool live = DH == D ? er < D : c0 / DH == hh;
  const float* wh = wsb + hh * rec_head;
#pragma unroll 1
  for (int j0 = c0; j0 < c0 + D / 2; j0 += 8) {
    const int jh = j0 - hh * DH;  // column within the head
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
    if (live) {
      if (a.S0 != nullptr) {
        const float4* src = reinterpret_cast<const float4*>(a.S0 + ((bh + hh) * DH + r) * DH + jh);
        const float4 x0 = src[0], x1 = src[1];
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
      }
      const float4* inc = reinterpret_cast<const float4*>(wh) + (jh / 4) * DH + r;
      constexpr long R4 = Rec<DH>::FLOATS / 4;
#pragma unroll 1
      for (int g = 0; g < nblk; g += 2) {
        const bool two = g + 1 < nblk;
        const float4 x0 = __ldcg(inc + g * R4), x1 = __ldcg(inc + g * R4 + DH);
        float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
        if (two) {
          y0 = __ldcg(inc + (g + 1) * R4);
          y1 = __ldcg(inc + (g + 1) * R4 + DH);
        }
        v[0] += x0.x; v[1] += x0.y; v[2] += x0.z; v[3] += x0.w;
        v[4] += x1.x; v[5] += x1.y; v[6] += x1.z; v[7] += x1.w;
        if (two) {
          v[0] += y0.x; v[1] += y0.y; v[2] += y0.z; v[3] += y0.w;
          v[4] += y1.x; v[5] += y1.y; v[6] += y1.z; v[7] += y1.w;
        }
      }
    }
    uint32_t u[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) u[e] = __float_as_uint(v[e]);
    tc::tmem_st8(tmem_s + j0, u);
    if (er < D) sts16(ss + static_cast<uint32_t>(j0 / 64) * (D * 128) + tc::sw128(er, (j0 % 64) / 8), pack8(v));
  }
}

// Scores of one group of 32 keys [col, col + 32) of the calling thread's tile row er (its TMEM lane):
// P (fp32, TMEM at tp + col) -> bf16 P~ pairs written back into TMEM at tp + dst (16 columns that
// this thread has already read; the A operand of the P~V product), masked to tau <= er on the
// diagonal group. The masked fp32 scores are added to rs.
__device__ __forceinline__ void convert_p_group(uint32_t tp, int col, int dst, int er, bool diag, float& rs) {
  uint32_t u[2][16];
  tc::tmem_ld16(tp + col, u[0]);
  tc::tmem_ld16(tp + col + 16, u[1]);
  tc::tmem_wait_ld();
  uint32_t w[16];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int tau = col + 16 * m + 2 * e;
      float x0 = __uint_as_float(u[m][2 * e]);
      float x1 = __uint_as_float(u[m][2 * e + 1]);
      if (diag) {
        x0 = tau <= er ? x0 : 0.f;
        x1 = tau + 1 <= er ? x1 : 0.f;
      }
      w[8 * m + e] = tc::pack_bf16x2(x0, x1);
      rs += x0 + x1;
    }
  }
  tc::tmem_st16(tp + dst, w);
}

// q'_er . z over the columns [hf D/2, (hf + 1) D/2) of row er of the swizzled bf16 q' tile at qb
// (fp32 products and sum; z is fp32 [D]).
template <int D>
__device__ __forceinline__ float qz_half(const uint8_t* qb, const float* z, int er, int hf) {
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    const int col = hf * (D / 2) + 8 * i;
    const uint4 x = *reinterpret_cast<const uint4*>(qb + (col / 64) * 16384 + tc::sw128(er, (col % 64) / 8));
    const float4 za = *reinterpret_cast<const float4*>(z + col);
    const float4 zb = *reinterpret_cast<const float4*>(z + col + 4);
    acc0 = fmaf(__uint_as_float(x.x << 16), za.x, acc0);
    acc1 = fmaf(__uint_as_float(x.x & 0xffff0000u), za.y, acc1);
    acc0 = fmaf(__uint_as_float(x.y << 16), za.z, acc0);
    acc1 = fmaf(__uint_as_float(x.y & 0xffff0000u), za.w, acc1);
    acc0 = fmaf(__uint_as_float(x.z << 16), zb.x, acc0);
    acc1 = fmaf(__uint_as_float(x.z & 0xffff0000u), zb.y, acc1);
    acc0 = fmaf(__uint_as_float(x.w << 16), zb.z, acc0);
    acc1 = fmaf(__uint_as_float(x.w & 0xffff0000u), zb.w, acc1);
  }
  return acc0 + acc1;
}

// ------------------------------------------------------------------------------------------------
// Kernel B: one CTA per (document, head, segment). With PAIR (d = 64 heads, D = 128), one CTA per
// (document, pair of heads 2h and 2h + 1, segment): the q, k, v and output tiles of the pair are
// the 128-column tiles of the [rows, H / 2, 128] view of the tensors; each head has its own
// RMSNorm, gains, scores, denominators and state (the state and S~ are block diagonal, so one
// product Q'S~ serves both heads), and the two P~V products write the two halves of O.
template <int D, bool PAIR>
__global__ void __launch_bounds__(kThreadsB, 1)
    prefill_tc_kernel(const TcArgs ta, const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_o) {
  using L = LayB<D, PAIR>;
  using PM = Prod<D>;
  constexpr int TPR = PM::TPR, RPP = PM::RPP, NPASS = PM::NPASS;
  constexpr int DH = PAIR ? D / 2 : D;  // head size
  constexpr int NH = PAIR ? 2 : 1;      // heads per CTA
  const PrefillArgs& a = ta.p;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int HV = a.H / NH;  // heads of the tile view
  const int seg = blockIdx.x % ta.nseg_max;
  const int h = (blockIdx.x / ta.nseg_max) % HV;  // view head: heads NH h .. NH h + NH - 1
  const int slot = blockIdx.x / (ta.nseg_max * HV);
  const int doc = ta.order != nullptr ? ta.order[slot] : slot;

  long row0;
  int n;
  const bool good = doc_bounds(a, doc, row0, n);
  if (!good && seg == 0 && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 1u);
  const int nseg_doc = n > 0 ? (n + ta.seg_len - 1) / ta.seg_len : 1;
  if (seg >= nseg_doc) return;  // uniform across the CTA, before any allocation
  const int seg_start = seg * ta.seg_len;
  const int seg_n = min(ta.seg_len, n - seg_start);  // 0 only for an empty document
  const int nchunks = (seg_n + kC - 1) / kC;
  const bool last_seg = seg == nseg_doc - 1;
  const long bh = static_cast<long>(doc) * a.H + NH * h;  // (document, head) index of the first head

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  if (base & 1023u) {  // the swizzled layouts need 1024-byte alignment
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevInternal);
    return;
  }
  float* zs = reinterpret_cast<float*>(smem + L::ZS);
  float* di = reinterpret_cast<float*>(smem + L::DI);
  float* rsm = reinterpret_cast<float*>(smem + L::RS);
  const uint32_t bar_full = base + L::BAR, bar_vfull = bar_full + 16, bar_empty = bar_full + 32;
  const uint32_t bar_p = bar_full + 48, bar_kv = bar_full + 56, bar_kfree = bar_full + 64;
  const uint32_t bar_pconv = bar_full + 72, bar_sconv = bar_full + 80, bar_b = bar_full + 88;
  const uint32_t bar_ofree = bar_full + 96, bar_staged = bar_full + 112;
  const uint32_t bar_zfull = bar_full + 128, bar_zempty = bar_full + 152, bar_qfull = bar_full + 176;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);

  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar_full + 8 * i, kProd);
      tc::mbar_init(bar_vfull + 8 * i, 1);
      tc::mbar_init(bar_empty + 8 * i, 1 + kConv);  // the MMAs' commit + the converters' q'.z reads
      tc::mbar_init(bar_ofree + 8 * i, kConv);
      tc::mbar_init(bar_staged + 8 * i, kConv);
      tc::mbar_init(bar_qfull + 8 * i, 1);
    }
    tc::mbar_init(bar_p, 1);
    tc::mbar_init(bar_kv, 1);
    tc::mbar_init(bar_kfree, 1 + kHelp);  // the MMAs' commit + the helpers' column sums
    tc::mbar_init(bar_pconv, kConv);
    tc::mbar_init(bar_sconv, kConv);
    tc::mbar_init(bar_b, 1);
    for (int i = 0; i < 3; ++i) {
      tc::mbar_init(bar_zfull + 8 * i, kHelp);
      tc::mbar_init(bar_zempty + 8 * i, kConv);
    }
    tc::mbar_fence_init();
    *s_abort = 0;
  }
  if (D == 64) {  // zero block that pads k'^T to M = 128 rows (read by the tensor core)
    for (int i = tid; i < 16384 / 16; i += kThreadsB) sts16(base + L::KS + 16384 + i * 16, make_uint4(0, 0, 0, 0));
    tc::fence_async_smem();
  }
  const FeatTab tab = feat_tab<D>(smem + L::TAB);
  fill_tab<D, DH>(tab, a, NH * h, RPP, tid, kThreadsB);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const long rec_head = ta.nblk_max * Rec<DH>::FLOATS;  // records of one (document, head)
  const float* wsb = ta.ws + bh * rec_head;
  const int nblk = seg * ta.blk_per_seg;  // increment blocks before this segment

  if (warp < kProd / 32) {
    // ============================================================ producers
    tc::regs_inc<kRegsProdB>();
    const int prow = tid / TPR, part = tid % TPR, e0 = 8 * part;
    const uint32_t cblk = static_cast<uint32_t>(e0 / 64) * 16384;  // 64-column block
    const int cidx = (e0 % 64) / 8;                                 // 16-byte chunk in the row

    // raw q arrives by TMA in the q' buffer (the transform overwrites it in place); k goes through
    // registers, two passes of loads in flight (the ring index p % RK needs NPASS % RK == 0)
    constexpr int RK = NPASS < 2 ? NPASS : 2;
    static_assert(NPASS % RK == 0, "k load ring");
    const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
    const int pos_base = a.pos_offset + seg_start;
    const long rstride = static_cast<long>(HV) * D;  // elements from one token row to the next
    const __nv_bfloat16* krow = kg + (row0 + seg_start + prow) * rstride + static_cast<long>(h) * D + e0;
    auto load = [&](int c, int p, uint4& xk) {
      if (c * kC + p * RPP + prow < seg_n) xk = ldg16(krow + static_cast<long>(c * kC + p * RPP) * rstride);
      else xk = make_uint4(0, 0, 0, 0);
    };
    Rot rot;  // RoPE cos / sin of this thread's current row
    // rotation by RPP positions (one pass further down the chunk): held in registers for one head
    // per CTA; re-read from the table each pass for a pair of heads (its producers have no
    // registers to spare)
    Rot step_held;
    if constexpr (!PAIR) tab_step(tab, e0 / 2, step_held);
    uint4 rk[RK];
    if (nchunks > 0) {
#pragma unroll
      for (int p = 0; p < RK; ++p) load(0, p, rk[p]);
    }
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      int bad = 0;
      // the raw q of this chunk (loaded once the buffer's previous q' had been read by both of its
      // products and by the converters)
      if (!tc::mbar_wait(bar_qfull + 8 * s, (c >> 1) & 1, kWaitCycles)) bad = 1;
      const uint32_t qb = base + (s ? L::Q1 : L::Q0), vb = base + (s ? L::V1 : L::V0);
      if (tid == 0 && c < 2) {
        // v rows of the first two chunks, straight into the swizzled operand (rows past the segment
        // are either other tokens or zero fill; their k' and P columns are zero); the store thread
        // loads the later chunks' v into the buffer once its output staging is done
        tc::mbar_arrive_expect_tx(bar_vfull + 8 * s, L::TILE);
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb)
          tc::tma_load_3d(vb + jb * 16384, &tmap_v, 64 * jb, h,
                          static_cast<int>(row0 + seg_start + c * kC), bar_vfull + 8 * s);
      }
      uint4 kreg[NPASS];
      // angles of the chunk's first row: exact every 8 chunks, otherwise one more step of the
      // incremental rotation from the previous chunk's last pass (RPP positions further down)
      if ((c & 7) == 0) {
        tab_rot_at(tab, pos_base + c * kC + prow, e0 / 2, rot);
      } else if constexpr (PAIR) {
        Rot st;
        tab_step(tab, e0 / 2, st);
        rot_step(rot, st);
      } else {
        rot_step(rot, step_held);
      }
      uint4 xq_next = ld_shared16(smem, qb - base + cblk + tc::sw128(prow, cidx));
#pragma unroll
      for (int p = 0; p < NPASS; ++p) {
        const uint4 xq = xq_next, xk = rk[p % RK];
        if (p + 1 < NPASS) xq_next = ld_shared16(smem, qb - base + cblk + tc::sw128((p + 1) * RPP + prow, cidx));
        if (p + RK < NPASS) load(c, p + RK, rk[p % RK]);
        else if (c + 1 < nchunks) load(c + 1, p + RK - NPASS, rk[p % RK]);
        const int r = p * RPP + prow;
        const bool valid = c * kC + r < seg_n;
        if (p > 0) {
          if constexpr (PAIR) {
            Rot st;
            tab_step(tab, e0 / 2, st);
            rot_step(rot, st);
          } else {
            rot_step(rot, step_held);
          }
        }
        Pairs fq = unpack_pairs(xq), fk = unpack_pairs(xk);
        const float rq2 = sumsq(fq), rk2 = sumsq(fk);
        // (the 16-byte chunks of one head of a row are TPR / NH consecutive lanes)
        const float sq = row_sum<TPR / NH>(rq2), sk = row_sum<TPR / NH>(rk2);
        const float rinvq = valid ? rsqrtf(sq * (1.0f / DH) + a.fa.eps_norm) : 0.f;
        const float rinvk = valid ? rsqrtf(sk * (1.0f / DH) + a.fa.eps_norm) : 0.f;
        {
          float2 g0[2], g1[2];
          split_load<D>(tab.gq, part, g0, g1);
          scale_gains(g0, g1, rinvq);
          rope_scaled(fq, g0, g1, rot);
          split_load<D>(tab.gk, part, g0, g1);
          scale_gains(g0, g1, rinvk);
          rope_scaled(fk, g0, g1, rot);
        }
        st_shared16(smem, qb - base + cblk + tc::sw128(r, cidx), pack_pairs_relu(fq));
        kreg[p] = pack_pairs_relu(fk);
      }
      // the single k' buffer is free once the previous chunk's MMAs have read it and the helpers
      // have summed its columns
      if (c >= 1 && !tc::mbar_wait(bar_kfree, (c - 1) & 1, kWaitCycles)) bad = 1;
#pragma unroll
      for (int p = 0; p < NPASS; ++p) st_shared16(smem, L::KS + cblk + tc::sw128(p * RPP + prow, cidx), kreg[p]);
      tc::fence_async_smem();
      tc::mbar_arrive(bar_full + 8 * s);
      if (bad) atomicExch(s_abort, 1);
      if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(s_abort))) break;
    }
  } else if (warp < (kProd + kConv) / 32) {
    // ============================================ converters (warps 16-23): two per lane quarter
    tc::regs_dec<kRegsConvB>();
    const int q4 = warp & 3;                       // TMEM lane quarter
    const int hf = (warp - kProd / 32) >> 2;       // half of the columns
    const int er = 32 * q4 + lane;                 // TMEM lane = tile row
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    const int j_lo = hf * (D / 2), j_hi = j_lo + D / 2;
    // initial state of this half of the columns: S (TMEM) and S~ (completion 0 of sconv)
    if (nblk > 0) tc::grid_dep_wait();
    init_state<D, DH>(a, wsb, rec_head, nblk, bh, er, tmem + tl + L::TS, base + L::SS, j_lo);
    tc::tmem_wait_st();
    tc::fence_async_smem();
    tc::fence_before_sync();
    tc::mbar_arrive(bar_sconv);

    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out);
    int bad = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1, zj = c % 3;
      // ---- q'_t . z_{c-1} over this half's columns, read before the q' buffer is released
      int ok = tc::mbar_wait(bar_full + 8 * s, (c >> 1) & 1, kWaitCycles);
      ok &= tc::mbar_wait(bar_zfull + 8 * zj, (c / 3) & 1, kWaitCycles);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;
      float dq = 0.f;
      if (!bad) dq = qz_half<D>(smem + (s ? L::Q1 : L::Q0), zs + zj * D, er, hf);
      di[(2 * s + hf) * kC + er] = dq;
      tc::mbar_arrive(bar_zempty + 8 * zj);
      tc::mbar_arrive(bar_empty + 8 * s);
      // ---- P -> masked bf16 P~ in TMEM, and the row sums of the masked fp32 scores
      ok = tc::mbar_wait(bar_p, c & 1, kWaitCycles);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;  // warp-uniform, so TMEM accesses stay converged
      tc::fence_after_sync();
      float rs = 0.f;
      if (!bad) {
        // Key groups of 32: left of this warp's rows (col < 32 q4) fully visible, col == 32 q4 the
        // diagonal, the rest above it (all zero). One head: this half's keys [64 hf, 64 hf + 64)
        // become the bf16 pairs in TMEM columns [64 hf, 64 hf + 32). A pair of heads: all 128 keys
        // of head hf's scores become the bf16 pairs in the first 64 of its columns (group g is
        // written over columns that group g - 1 or g itself has already read).
        constexpr int NG = PAIR ? 4 : 2;
        const uint32_t tp = tmem + tl + (PAIR ? (hf ? L::TP1 : L::TP) : L::TP);
#pragma unroll(PAIR ? 1 : NG)
        for (int g = 0; g < NG; ++g) {
          const int col = PAIR ? 32 * g : 64 * hf + 32 * g;
          const int dst = PAIR ? 16 * g : 64 * hf + 16 * g;
          if (col > 32 * q4) {  // warp-uniform: strictly above the diagonal
            uint32_t zero[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) zero[e] = 0u;
            tc::tmem_st16(tp + dst, zero);
          } else {
            convert_p_group(tp, col, dst, er, col == 32 * q4, rs);
          }
        }
        tc::tmem_wait_st();
      }
      rsm[(2 * s + hf) * kC + er] = rs;
      tc::fence_before_sync();
      tc::mbar_arrive(bar_pconv);
      // ---- S (the state after this chunk) -> bf16 S~, the operand of the next chunk's Q'S~
      ok = tc::mbar_wait(bar_kv, c & 1, kWaitCycles);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;
      tc::fence_after_sync();
      if (!bad && (PAIR ? (q4 >> 1) == hf : 32 * q4 < D)) {
#pragma unroll 1
        for (int j0 = j_lo; j0 < j_hi; j0 += 32) {
          uint32_t u[2][16];
          tc::tmem_ld16(tmem + tl + L::TS + j0, u[0]);
          tc::tmem_ld16(tmem + tl + L::TS + j0 + 16, u[1]);
          tc::tmem_wait_ld();
          const uint32_t blk = base + L::SS + static_cast<uint32_t>(j0 / 64) * (D * 128);
          const int cc = (j0 % 64) / 8;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(u[m][e]);
            st_shared16(smem, blk - base + tc::sw128(er, cc + 2 * m), pack8(v));
            st_shared16(smem, blk - base + tc::sw128(er, cc + 2 * m + 1), pack8(v + 8));
          }
        }
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(bar_sconv);
      // ---- out = O / (q'.z_{c-1} + rowsum(P) + eps), this half's columns
      ok = tc::mbar_wait(bar_b, c & 1, kWaitCycles);
      if (__any_sync(0xffffffffu, !ok)) bad = 1;
      // one head: the other half's q'.z and row sums are written (a pair: each half is one head)
      if (!PAIR) tc::named_sync(kBarQuarter + q4, 64);
      // A whole chunk is staged in its v buffer (free: v was read by the finished MMAs) in the box
      // layout of the output tensor map and written by TMA in full 128-byte lines; the ragged last
      // chunk of a document is written row by row (its tile would reach past it).
      const bool whole = c * kC + kC <= seg_n;
      const uint32_t ob = base + (s ? L::V1 : L::V0);
      if (!bad) {
        tc::fence_after_sync();
        const float den = PAIR ? di[(2 * s + hf) * kC + er] + rsm[(2 * s + hf) * kC + er] + a.eps_den
                               : di[(2 * s) * kC + er] + di[(2 * s + 1) * kC + er] +
                                     rsm[(2 * s) * kC + er] + rsm[(2 * s + 1) * kC + er] + a.eps_den;
        const uint32_t to = tmem + tl + (s ? L::TO1 : L::TO0);
        const float inv = 1.0f / den;
        const int lt = c * kC + er;
        __nv_bfloat16* orow = og + ((row0 + seg_start + lt) * HV + h) * D;
#pragma unroll 1
        for (int j0 = j_lo; j0 < j_hi; j0 += 32) {
          uint32_t u[2][16];
          tc::tmem_ld16(to + j0, u[0]);
          tc::tmem_ld16(to + j0 + 16, u[1]);
          tc::tmem_wait_ld();
          const uint32_t blk = ob + static_cast<uint32_t>(j0 / 64) * 16384;
          const int cc = (j0 % 64) / 8;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            float f[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(u[m][e]) * inv;
            if (whole) {
              st_shared16(smem, blk - base + tc::sw128(er, cc + 2 * m), pack8(f));
              st_shared16(smem, blk - base + tc::sw128(er, cc + 2 * m + 1), pack8(f + 8));
            } else if (lt < seg_n) {
              uint4* dst = reinterpret_cast<uint4*>(orow + j0 + 16 * m);
              dst[0] = pack8(f);
              dst[1] = pack8(f + 8);
            }
          }
        }
        if (whole) tc::fence_async_smem();
      }
      tc::fence_before_sync();
      tc::mbar_arrive(bar_staged + 8 * s);  // the store thread takes it from here
      tc::mbar_arrive(bar_ofree + (PAIR ? 0 : 8 * s));  // the O accumulator may take chunk c + 2 (a pair: c + 1)
      if (bad) atomicExch(s_abort, 1);
      if (group_sync_or(kBarConv, kConv, *s_abort)) break;
    }
    if (bad) atomicExch(s_abort, 1);
    if (last_seg && a.S_final != nullptr && !*s_abort && (PAIR ? (q4 >> 1) == hf : 32 * q4 < D)) {
      tc::fence_after_sync();
      const int hh = PAIR ? hf : 0, r = PAIR ? er % DH : er;  // the diagonal block of head hh
      for (int j0 = j_lo; j0 < j_hi; j0 += 16) {
        uint32_t u[16];
        tc::tmem_ld16(tmem + tl + L::TS + j0, u);
        tc::tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(a.S_final + ((bh + hh) * DH + r) * DH + j0 - hh * DH);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                               __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
      }
    }
  } else {
    tc::regs_dec<kRegsIssueB>();  // one call site for the whole warpgroup (warps 24-27)
  if (warp == kWarpIssue) {
    // ========================================================== MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t ID_P = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_QS = tc::idesc_bf16(128, D, false, true);
      constexpr uint32_t ID_KV = tc::idesc_bf16(128, D, true, true);
      constexpr uint32_t ID_PV = tc::idesc_bf16(128, DH, false, true);
      int ok = 1;
      // descriptors: k-major operands advance 32 bytes per K=16 step inside a 64-column block and
      // 16 KB per block; MN-major operands advance 2 KB (16 rows) per step
      const uint64_t d_ks_k = tc::desc_sw128(base + L::KS, 16, 1024);
      const uint64_t d_ks_mn = tc::desc_sw128(base + L::KS, 16384, 1024);
      const uint64_t d_ss = tc::desc_sw128(base + L::SS, D * 128, 1024);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c & 1, ph = (c >> 1) & 1;
        const uint32_t qb = base + (s ? L::Q1 : L::Q0), vb = base + (s ? L::V1 : L::V0);
        const uint32_t to = tmem + (s ? L::TO1 : L::TO0);
        const uint64_t d_q = tc::desc_sw128(qb, 16, 1024);
        const uint64_t d_v = tc::desc_sw128(vb, 16384, 1024);
        ok = tc::mbar_wait(bar_full + 8 * s, ph, kWaitCycles) &&
             tc::mbar_wait(bar_vfull + 8 * s, ph, kWaitCycles);
        if (!ok) break;
        tc::fence_after_sync();
        // P = Q' K'^T (the converters turn it into P~ while the next two products run); a pair of
        // heads: Q'_h K'_h^T over each head's 64 feature columns, into the head's own columns
#pragma unroll 1
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t kofs = static_cast<uint64_t>((k / 4) * 1024 + (k % 4) * 2);
          const uint32_t tp = tmem + (PAIR && k >= 4 ? L::TP1 : L::TP);
          tc::mma_bf16(tp, d_q + kofs, d_ks_k + kofs, ID_P, PAIR ? (k % 4) > 0 : k > 0);
        }
        tc::mma_commit(bar_p);
        // O = Q' S~_{c-1}, once S~ holds the state before this chunk and the O buffer is free
        ok = tc::mbar_wait(bar_sconv, c & 1, kWaitCycles) &&
             (PAIR ? (c < 1 || tc::mbar_wait(bar_ofree, (c - 1) & 1, kWaitCycles))
                   : (c < 2 || tc::mbar_wait(bar_ofree + 8 * s, ((c >> 1) + 1) & 1, kWaitCycles)));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t kofs = static_cast<uint64_t>((k / 4) * 1024 + (k % 4) * 2);
          tc::mma_bf16(to, d_q + kofs, d_ss + static_cast<uint64_t>(k) * 128, ID_QS, k > 0);
        }
        tc::mma_commit(bar_empty + 8 * s);  // q' of this chunk read by both of its products
        // S += K'^T V (the fp32 master state, never leaves TMEM)
#pragma unroll 1
        for (int k = 0; k < kC / 16; ++k) {
          tc::mma_bf16(tmem + L::TS, d_ks_mn + static_cast<uint64_t>(k) * 128,
                       d_v + static_cast<uint64_t>(k) * 128, ID_KV, 1u);
        }
        tc::mma_commit(bar_kv);
        tc::mma_commit(bar_kfree);
        // O += P~ V, with P~ read from TMEM (keys 16 k .. 16 k + 15 in columns 64 (k / 4) + 8 (k % 4);
        // a pair of heads: in columns 8 k of the head's scores, and each head's product takes its
        // own 64 columns of v and writes its own half of O)
        ok = tc::mbar_wait(bar_pconv, c & 1, kWaitCycles);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int hh = 0; hh < NH; ++hh) {
#pragma unroll 1
          for (int k = 0; k < kC / 16; ++k) {
            const uint32_t pa = PAIR ? tmem + (hh ? L::TP1 : L::TP) + 8 * k
                                     : tmem + L::TP + 64 * (k / 4) + 8 * (k % 4);
            tc::mma_bf16_ta(to + 64 * hh, pa, d_v + static_cast<uint64_t>(hh) * 1024 + static_cast<uint64_t>(k) * 128,
                            ID_PV, 1u);
          }
        }
        tc::mma_commit(bar_b);
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else if (warp == kWarpStore) {
    // ========================================================== output stores, v loads
    if (lane == 0) {
      // raw q of the first two chunks into the q' buffers
      for (int c = 0; c < 2 && c < nchunks; ++c) {
        tc::mbar_arrive_expect_tx(bar_qfull + 8 * c, L::TILE);
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb)
          tc::tma_load_3d(base + (c ? L::Q1 : L::Q0) + jb * 16384, &tmap_q, 64 * jb, h,
                          static_cast<int>(row0 + seg_start + c * kC), bar_qfull + 8 * c);
      }
      int ok = 1;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (c + 2 < nchunks) {
          // q' of chunk c has been read by both of its products and by the converters: the raw q of
          // chunk c + 2 goes into the same buffer
          ok = tc::mbar_wait(bar_empty + 8 * s, (c >> 1) & 1, kWaitCycles);
          if (!ok || *reinterpret_cast<volatile int*>(s_abort)) break;
          tc::mbar_arrive_expect_tx(bar_qfull + 8 * s, L::TILE);
#pragma unroll
          for (int jb = 0; jb < D / 64; ++jb)
            tc::tma_load_3d(base + (s ? L::Q1 : L::Q0) + jb * 16384, &tmap_q, 64 * jb, h,
                            static_cast<int>(row0 + seg_start + (c + 2) * kC), bar_qfull + 8 * s);
        }
        ok = tc::mbar_wait(bar_staged + 8 * s, (c >> 1) & 1, kWaitCycles);
        if (!ok || *reinterpret_cast<volatile int*>(s_abort)) break;
        const uint32_t ob = base + (s ? L::V1 : L::V0);
        if (c * kC + kC <= seg_n) {  // a whole chunk was staged
#pragma unroll
          for (int jb = 0; jb < D / 64; ++jb)
            tc::tma_store_3d(&tmap_o, ob + jb * 16384, 64 * jb, h,
                             static_cast<int>(row0 + seg_start + c * kC));
          tc::bulk_commit();
          tc::bulk_wait_read0();  // the buffer may be refilled once the store has read it
        }
        if (c + 2 < nchunks) {  // v of chunk c + 2 into the same buffer
          tc::mbar_arrive_expect_tx(bar_vfull + 8 * s, L::TILE);
#pragma unroll
          for (int jb = 0; jb < D / 64; ++jb)
            tc::tma_load_3d(ob + jb * 16384, &tmap_v, 64 * jb, h,
                            static_cast<int>(row0 + seg_start + (c + 2) * kC), bar_vfull + 8 * s);
        }
      }
      tc::bulk_wait0();
      if (!ok) atomicExch(s_abort, 1);
    }
  } else {
    // ========================================================== z helpers (warps 26-27)
    // z_c = z_{c-1} + the column sums of the bf16 k' tile of chunk c (the values the products
    // read); each z goes into a ring of three slots for the converters' q'.z. A helper sums one
    // 16-byte column chunk (8 columns) over one group of rows; the groups' partials are then added
    // in a fixed order by the owner of each column pair.
    constexpr int NCQ = D / 8, NRG = 64 / NCQ, RPG = kC / NRG;
    const int ht = tid - (kProd + kConv + 64);
    const int cq = ht % NCQ, rg = ht / NCQ;
    const bool own = ht < D / 2;  // the owner of columns 2 ht and 2 ht + 1
    float* zh = reinterpret_cast<float*>(smem + L::ZH);
    float z0 = 0.f, z1 = 0.f;
    if (own) {
      if (nblk > 0) tc::grid_dep_wait();
      const int hh = (2 * ht) / DH, cz = (2 * ht) % DH;  // head and its column
      if (a.z0 != nullptr) {
        z0 = a.z0[(bh + hh) * DH + cz];
        z1 = a.z0[(bh + hh) * DH + cz + 1];
      }
      const float* wz = wsb + hh * rec_head + Rec<DH>::Z + cz;
      for (int g = 0; g < nblk; ++g) {
        z0 += __ldcg(wz + g * Rec<DH>::FLOATS);
        z1 += __ldcg(wz + g * Rec<DH>::FLOATS + 1);
      }
      zs[2 * ht] = z0;  // slot 0: z before the segment, read by chunk 0
      zs[2 * ht + 1] = z1;
    }
    tc::mbar_arrive(bar_zfull);
    const uint8_t* kt = smem + L::KS + (cq / 8) * 16384;
    int bad = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1, zj = (c + 1) % 3;
      int ok = tc::mbar_wait(bar_full + 8 * s, (c >> 1) & 1, kWaitCycles);
      // the slot's previous z (chunk c - 2's) has been read by the converters
      if (c + 1 >= 3) ok &= tc::mbar_wait(bar_zempty + 8 * zj, ((c + 1) / 3 - 1) & 1, kWaitCycles);
      if (group_sync_or(kBarHelp, kHelp, !ok || *reinterpret_cast<volatile int*>(s_abort))) {
        bad = 1;
        break;
      }
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 8
      for (int r = rg * RPG; r < rg * RPG + RPG; ++r) {
        const uint4 x = *reinterpret_cast<const uint4*>(kt + tc::sw128(r, cq % 8));
        acc[0] += __uint_as_float(x.x << 16);
        acc[1] += __uint_as_float(x.x & 0xffff0000u);
        acc[2] += __uint_as_float(x.y << 16);
        acc[3] += __uint_as_float(x.y & 0xffff0000u);
        acc[4] += __uint_as_float(x.z << 16);
        acc[5] += __uint_as_float(x.z & 0xffff0000u);
        acc[6] += __uint_as_float(x.w << 16);
        acc[7] += __uint_as_float(x.w & 0xffff0000u);
      }
      tc::mbar_arrive(bar_kfree);  // done reading k' of chunk c
#pragma unroll
      for (int e = 0; e < 8; ++e) zh[rg * D + 8 * cq + e] = acc[e];
      tc::named_sync(kBarHelp, kHelp);
      if (own) {
#pragma unroll
        for (int g = 0; g < NRG; ++g) {
          z0 += zh[g * D + 2 * ht];
          z1 += zh[g * D + 2 * ht + 1];
        }
        zs[zj * D + 2 * ht] = z0;
        zs[zj * D + 2 * ht + 1] = z1;
      }
      tc::mbar_arrive(bar_zfull + 8 * zj);
    }
    if (bad) atomicExch(s_abort, 1);
    tc::named_sync(kBarHelp, kHelp);
    if (last_seg && a.z_final != nullptr && !*s_abort && own) {
      const int hh = (2 * ht) / DH, cz = (2 * ht) % DH;
      a.z_final[(bh + hh) * DH + cz] = z0;
      a.z_final[(bh + hh) * DH + cz + 1] = z1;
    }
  }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*s_abort) {
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevInternal);
    // a bounded chance for MMAs still in flight to land before TMEM is released
    if (tid == 0) tc::mbar_wait(bar_b, 0, kWaitCycles / 4);
    __syncthreads();
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// Kernel A: state increment (K'^T V and the column sums of k') of one block of blk_len tokens (every
// block before a document's last segment; in whole-document mode, every block of the document, for
// the bidirectional form and for the state of a shard). One thread streams the raw k and v tiles of
// the block's chunks by TMA into a ring of stages; 16 producer warps turn each k tile into k' in
// place (RMSNorm, RoPE, ReLU) and sum its columns; one thread accumulates K'^T V into TMEM, and the
// stage is refilled once its product has completed.
template <int D>
__global__ void __launch_bounds__(kThreadsA, 1)
    segment_state_kernel(const TcArgs ta, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v) {
  using L = LayA<D>;
  using PM = Prod<D>;
  constexpr int S = kStagesA;
  constexpr int TPR = PM::TPR, RPP = PM::RPP, NPASS = PM::NPASS;
  const PrefillArgs& a = ta.p;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tc::grid_launch_dependents();  // kernel B may start; it waits for this grid before reading ws
  const int blk = blockIdx.x % ta.nblk_max;
  const int h = (blockIdx.x / ta.nblk_max) % a.H;
  const int doc = blockIdx.x / (ta.nblk_max * a.H);
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);  // a malformed document has n = 0 and is skipped
  if (ta.whole_doc) {
    if (static_cast<long>(blk) * ta.blk_len >= n) return;  // past the document's end
  } else {
    const int nseg_doc = n > 0 ? (n + ta.seg_len - 1) / ta.seg_len : 1;
    if (blk >= (nseg_doc - 1) * ta.blk_per_seg) return;  // the last segment needs no increment
  }
  const int seg_start = blk * ta.blk_len;
  // a block before the last segment is full; in whole-document mode the last one may be ragged
  // (its missing rows are zeroed by the features: they add nothing)
  const int blk_n = min(ta.blk_len, n - seg_start);
  const int nchunks = (blk_n + kC - 1) / kC;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  if (base & 1023u) {
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevInternal);
    return;
  }
  float* zp = reinterpret_cast<float*>(smem + L::ZP);
  const uint32_t bar_kfull = base + L::BAR, bar_vfull = bar_kfull + 8 * S;
  const uint32_t bar_ready = bar_vfull + 8 * S, bar_free = bar_ready + 8 * S;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
  int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 4);

  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 128);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(bar_kfull + 8 * i, 1);
      tc::mbar_init(bar_vfull + 8 * i, 1);
      tc::mbar_init(bar_ready + 8 * i, kProd);
      tc::mbar_init(bar_free + 8 * i, 1);
    }
    tc::mbar_fence_init();
    *s_abort = 0;
    *reinterpret_cast<int*>(smem + L::MISC + 8) = 0;
  }
  if (D == 64) {
    for (int i = tid; i < S * 16384 / 16; i += kThreadsA) {
      const int st = i / (16384 / 16), j = i % (16384 / 16);
      sts16(base + L::K0 + st * L::KT + 16384 + j * 16, make_uint4(0, 0, 0, 0));
    }
    tc::fence_async_smem();  // (read by the tensor core)
  }
  const FeatTab tab = feat_tab<D>(smem + L::TAB);
  fill_tab<D>(tab, a, h, RPP, tid, kThreadsA);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const long bh = static_cast<long>(doc) * a.H + h;
  float* dst = ta.ws + (bh * ta.nblk_max + blk) * Rec<D>::FLOATS;

  if (warp < kProd / 32) {
    tc::regs_inc<kRegsProdA>();
    const int prow = tid / TPR, part = tid % TPR, e0 = 8 * part;
    const uint32_t cblk = static_cast<uint32_t>(e0 / 64) * 16384;
    const int cidx = (e0 % 64) / 8;
    float2 gk0[2], gk1[2];
    split_load<D>(tab.gk, part, gk0, gk1);
    Rot step;
    tab_step(tab, e0 / 2, step);
    const int pos_base = a.pos_offset + seg_start;
    Rot rot;
    float2 zca[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 zcb[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    int bad = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c % S;
      if (!tc::mbar_wait(bar_kfull + 8 * st, (c / S) & 1, kWaitCycles)) bad = 1;
      const uint32_t kb = base + L::K0 + st * L::KT + cblk;
      if ((c & 7) == 0) tab_rot_at(tab, pos_base + c * kC + prow, e0 / 2, rot);
      else rot_step(rot, step);
      uint4 xk_next = ld_shared16(smem, kb - base + tc::sw128(prow, cidx));
#pragma unroll
      for (int p = 0; p < NPASS; ++p) {
        const uint4 xk = xk_next;
        const int r = p * RPP + prow;
        if (p + 1 < NPASS) xk_next = ld_shared16(smem, kb - base + tc::sw128(r + RPP, cidx));
        const bool valid = c * kC + r < blk_n;
        if (p > 0) rot_step(rot, step);
        Pairs fk = unpack_pairs(xk);
        const float sk = row_sum<TPR>(sumsq(fk));
        float2 g0[2] = {gk0[0], gk0[1]}, g1[2] = {gk1[0], gk1[1]};
        scale_gains(g0, g1, valid ? rsqrtf(sk * (1.0f / D) + a.fa.eps_norm) : 0.f);
        rope_relu(fk, g0, g1, rot);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          zca[g] = __fadd2_rn(zca[g], fk.x0[g]);
          zcb[g] = __fadd2_rn(zcb[g], fk.x1[g]);
        }
        st_shared16(smem, kb - base + tc::sw128(r, cidx), pack_pairs(fk));
      }
      tc::fence_async_smem();
      tc::mbar_arrive(bar_ready + 8 * st);
      if (bad) atomicExch(s_abort, 1);
      if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(s_abort))) break;
    }
    // sums of k' over the block (fixed order: deterministic)
    float zc[8];
    pairs_to8(Pairs{{zca[0], zca[1]}, {zcb[0], zcb[1]}}, zc);
    warp_colsum<TPR>(zc);
    if (lane < TPR) {
      *reinterpret_cast<float4*>(zp + warp * D + e0) = make_float4(zc[0], zc[1], zc[2], zc[3]);
      *reinterpret_cast<float4*>(zp + warp * D + e0 + 4) = make_float4(zc[4], zc[5], zc[6], zc[7]);
    }
    tc::named_sync(kBarProd, kProd);
    if (tid < D && !*s_abort) {
      float z = 0.f;
#pragma unroll
      for (int w = 0; w < PM::WARPS; ++w) z += zp[w * D + tid];
      dst[Rec<D>::Z + tid] = z;
    }
  } else {
    tc::regs_dec<kRegsIssueA>();
    const int q4 = warp & 3;
    if (warp == kProd / 32 && lane == 0) {
      // ======================================================= MMA issue
      constexpr uint32_t ID_KV = tc::idesc_bf16(128, D, true, true);
      int ok = 1;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int st = c % S, ph = (c / S) & 1;
        ok = tc::mbar_wait(bar_ready + 8 * st, ph, kWaitCycles) &&
             tc::mbar_wait(bar_vfull + 8 * st, ph, kWaitCycles);
        if (!ok) break;
        tc::fence_after_sync();
        const uint64_t d_k = tc::desc_sw128(base + L::K0 + st * L::KT, 16384, 1024);
        const uint64_t d_v = tc::desc_sw128(base + L::V0 + st * L::TILE, 16384, 1024);
#pragma unroll 1
        for (int k = 0; k < kC / 16; ++k)
          tc::mma_bf16(tmem, d_k + static_cast<uint64_t>(k) * 128, d_v + static_cast<uint64_t>(k) * 128,
                       ID_KV, (c > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(bar_free + 8 * st);
      }
      // the last accumulation
      const int last = nchunks - 1;
      if (ok && last >= 0) ok = tc::mbar_wait(bar_free + 8 * (last % S), (last / S) & 1, kWaitCycles);
      if (!ok) atomicExch(s_abort, 1);
      *reinterpret_cast<volatile int*>(smem + L::MISC + 8) = 1;  // accumulation complete
    } else if (warp == kProd / 32 + 1 && lane == 0) {
      // ======================================================= TMA: raw k and v tiles of each chunk
      int ok = 1;
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % S;
        // the stage's previous chunk (c - S) has been consumed by its product
        if (c >= S) ok = tc::mbar_wait(bar_free + 8 * st, ((c / S) + 1) & 1, kWaitCycles);
        if (!ok || *reinterpret_cast<volatile int*>(s_abort)) break;
        const int row = static_cast<int>(row0 + seg_start + c * kC);
        tc::mbar_arrive_expect_tx(bar_kfull + 8 * st, L::TILE);
        tc::mbar_arrive_expect_tx(bar_vfull + 8 * st, L::TILE);
#pragma unroll
        for (int jb = 0; jb < D / 64; ++jb) {
          tc::tma_load_3d(base + L::K0 + st * L::KT + jb * 16384, &tmap_k, 64 * jb, h, row, bar_kfull + 8 * st);
          tc::tma_load_3d(base + L::V0 + st * L::TILE + jb * 16384, &tmap_v, 64 * jb, h, row, bar_vfull + 8 * st);
        }
      }
      if (!ok) atomicExch(s_abort, 1);
    }
    __syncwarp();
    // the issuer warpgroup copies the increment out of TMEM (one lane quarter per warp)
    const volatile int* done = reinterpret_cast<const volatile int*>(smem + L::MISC + 8);
    const long long t0 = clock64();
    while (*done == 0 && clock64() - t0 < kWaitCycles) {
    }
    const int go = __all_sync(0xffffffffu, *done != 0 && *s_abort == 0);
    if (go && 32 * q4 < D) {
      tc::fence_after_sync();
      const int er = 32 * q4 + lane;
      const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
      float4* d4 = reinterpret_cast<float4*>(dst) + er;
      for (int j0 = 0; j0 < D; j0 += 16) {
        uint32_t u[16];
        tc::tmem_ld16(tmem + tl + j0, u);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 4; ++e)
          __stcg(d4 + (j0 / 4 + e) * D, make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                                    __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3])));
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*s_abort && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevInternal);
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// The documents in order of decreasing length (ties by index): order[rank] = doc, one CTA; the
// lengths of a malformed cu_seqlens are clamped (the prefill kernel reports such documents).
__global__ void __launch_bounds__(1024) doc_order_kernel(const int32_t* cu, int N, int total, int* order) {
  extern __shared__ int lens[];
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int l = cu[i + 1] - cu[i];
    lens[i] = l < 0 ? 0 : (l > total ? total : l);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int li = lens[i];
    int rank = 0;
    for (int j = 0; j < N; ++j) rank += (lens[j] > li || (lens[j] == li && j < i)) ? 1 : 0;
    order[rank] = i;
  }
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
cudaError_t launch_state_d(const TcArgs& ta, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                           cudaStream_t stream) {
  static unsigned long long cfg_a = 0;
  cudaError_t e = set_smem(segment_state_kernel<D>, LayA<D>::BYTES, cfg_a);
  if (e != cudaSuccess) return e;
  const long grid = static_cast<long>(ta.p.n_docs) * ta.p.H * ta.nblk_max;
  if (grid == 0) return cudaSuccess;
  segment_state_kernel<D><<<static_cast<unsigned>(grid), kThreadsA, LayA<D>::BYTES, stream>>>(ta, tmap_k, tmap_v);
  note_launches(1);
  return cudaGetLastError();
}

// Kernel B with head size D (PAIR: two heads of 64 per CTA, tiles of the [rows, H / 2, 128] view),
// after kernel A (single heads of the tensors' own size) where segments need their start states.
template <int D, bool PAIR>
cudaError_t launch_tc_d(const TcArgs& ta, cudaStream_t stream) {
  constexpr int DT = PAIR ? 2 * D : D;  // tile width
  constexpr int NH = PAIR ? 2 : 1;
  static unsigned long long cfg_b = 0;
  cudaError_t e = set_smem(prefill_tc_kernel<DT, PAIR>, LayB<DT, PAIR>::BYTES, cfg_b);
  if (e != cudaSuccess) return e;
  const long units = static_cast<long>(ta.p.n_docs) * (ta.p.H / NH);
  if (units == 0) return cudaSuccess;
  CUtensorMap tmap_q, tmap_v, tmap_o;
  const bool rows = ta.p.v != nullptr && ta.p.total_rows > 0;
  if (rows) {
    const int hv = ta.p.H / NH;
    e = make_rows_map(&tmap_q, ta.p.q, ta.p.total_rows, hv, DT);
    if (e == cudaSuccess) e = make_rows_map(&tmap_v, ta.p.v, ta.p.total_rows, hv, DT);
    if (e == cudaSuccess) e = make_rows_map(&tmap_o, ta.p.out, ta.p.total_rows, hv, DT);
    if (e != cudaSuccess) return e;
  } else {
    memset(&tmap_q, 0, sizeof(tmap_q));  // no rows: the kernels issue no copy
    memset(&tmap_v, 0, sizeof(tmap_v));
    memset(&tmap_o, 0, sizeof(tmap_o));
  }
  const bool with_a = ta.nblk_max > 0;
  if (with_a) {
    CUtensorMap tmap_k, tmap_va;
    e = make_rows_map(&tmap_k, ta.p.k, ta.p.total_rows, ta.p.H, D);
    if (e == cudaSuccess) e = make_rows_map(&tmap_va, ta.p.v, ta.p.total_rows, ta.p.H, D);
    if (e == cudaSuccess) e = launch_state_d<D>(ta, tmap_k, tmap_va, stream);
    if (e != cudaSuccess) return e;
  }
  // kernel B as a programmatic dependent of kernel A (only then: it must not overlap anything else)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * ta.nseg_max));
  cfg.blockDim = dim3(kThreadsB);
  cfg.dynamicSmemBytes = LayB<DT, PAIR>::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = with_a ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<DT, PAIR>, ta, tmap_q, tmap_v, tmap_o);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(DType dt, int d) { return dt == DType::BF16 && (d == 64 || d == 128); }

TcPlan tc_plan(int n_docs, int H_heads, int max_seqlen, long total_tokens, int d, bool varlen) {
  // d = 64 with an even head count: kernel B takes the heads in pairs (one 128-wide tile), so it
  // has half the units, each costing about one d = 128 chunk per chunk; kernel A stays per head.
  const bool pair = d == 64 && H_heads % 2 == 0;
  const int H = pair ? H_heads / 2 : H_heads;  // kernel B units per document
  // Estimated time in units of one kernel-B chunk. Kernel B runs one CTA per SM (waves of 152
  // CTAs, each costing its chunks plus about one chunk of state set-up); a kernel-A chunk (k
  // features and one GEMM) costs about half a kernel-B chunk, also one CTA per SM. Documents are
  // assumed to share the tokens evenly, except that the longest one bounds the segment count.
  // More segments or blocks cost workspace, so a longer plan must be clearly (5 %) faster to win.
  TcPlan best{1, kC, 1, 0, false, 0, pair};
  const int chunks_max = max_seqlen > 0 ? (max_seqlen + kC - 1) / kC : 1;
  const double avg_chunks = n_docs > 0 ? static_cast<double>(total_tokens) / n_docs / kC : 0.0;
  double best_cost = 1e300;
  // One segment per document, with the longest units dispatched first: bounded by the longest
  // unit or by the total work spread over the SMs (plus a chunk of set-up). Documents of unequal
  // lengths (varlen) make the wave estimate of the split plans below optimistic, so this plan wins
  // whenever it is within reach.
  {
    const double total_chunks = static_cast<double>(H) * (static_cast<double>(total_tokens) / kC + 0.5 * n_docs);
    const double cost1 = (chunks_max > total_chunks / 152 ? chunks_max : total_chunks / 152) + 1.0;
    if (varlen && cost1 <= (pair ? 1.2 : 1.15) * (total_chunks / 152 + 1.0)) {
      best = TcPlan{1, chunks_max * kC, 1, 0, n_docs <= 1024, 0, pair};
      best_cost = 0.0;  // taken: no split plan below can beat the spread of the work
    }
  }
  for (int seg_chunks = chunks_max; seg_chunks >= 1; --seg_chunks) {
    const int nseg = (chunks_max + seg_chunks - 1) / seg_chunks;
    if (nseg > 64) break;
    const double segs_per_doc = avg_chunks > 0 ? static_cast<double>(static_cast<long>(
                                                      (avg_chunks + seg_chunks - 1e-9) / seg_chunks))
                                               : 1.0;
    const double items_b = static_cast<double>(H) * n_docs * (segs_per_doc > 1 ? segs_per_doc : 1.0);
    const double waves_b = static_cast<double>(static_cast<long>((items_b + 151) / 152));
    for (int f = 1; f <= 8 && nseg > 1; f *= 2) {
      if (seg_chunks % f != 0) break;
      const double items_a = (items_b - static_cast<double>(H) * n_docs) * f * (pair ? 2 : 1);
      const double waves_a = items_a > 0 ? static_cast<double>(static_cast<long>((items_a + 151) / 152)) : 0.0;
      const double cost = waves_b * (seg_chunks + 1.0) + waves_a * (0.5 * seg_chunks / f + 0.5);
      if (cost < 0.95 * best_cost) {
        best_cost = cost;
        best = TcPlan{nseg, seg_chunks * kC, f, 0, false, 0, pair};
      }
    }
    if (nseg == 1) {
      const double cost = waves_b * (seg_chunks + 1.0);
      if (cost < 0.95 * best_cost) {
        best_cost = cost;
        best = TcPlan{1, seg_chunks * kC, 1, 0, false, 0, pair};
      }
    }
  }
  const long units = static_cast<long>(n_docs) * H_heads;  // kernel A's records are per head
  const long rec = static_cast<long>(d) * (d + 1);
  best.ws_bytes = best.nseg_max > 1 ? static_cast<size_t>(units) * (best.nseg_max - 1) *
                                          best.blk_per_seg * rec * sizeof(float)
                                    : 0;
  if (best.sort_docs) {
    best.order_off = (best.ws_bytes + 255) / 256 * 256;
    best.ws_bytes = best.order_off + static_cast<size_t>(n_docs) * sizeof(int);
  }
  return best;
}

cudaError_t launch_state_tc(int d, const TcArgs& ta, cudaStream_t stream) {
  if (static_cast<long>(ta.p.n_docs) * ta.p.H * ta.nblk_max == 0 || ta.p.total_rows == 0) return cudaSuccess;
  CUtensorMap tmap_k, tmap_v;
  cudaError_t e = make_rows_map(&tmap_k, ta.p.k, ta.p.total_rows, ta.p.H, d);
  if (e == cudaSuccess) e = make_rows_map(&tmap_v, ta.p.v, ta.p.total_rows, ta.p.H, d);
  if (e != cudaSuccess) return e;
  return d == 128 ? launch_state_d<128>(ta, tmap_k, tmap_v, stream) : launch_state_d<64>(ta, tmap_k, tmap_v, stream);
}

cudaError_t launch_doc_order(const int32_t* cu_seqlens, int n_docs, int total_rows, int* order,
                             cudaStream_t stream) {
  if (n_docs <= 0) return cudaSuccess;
  doc_order_kernel<<<1, 1024, static_cast<size_t>(n_docs) * sizeof(int), stream>>>(cu_seqlens, n_docs,
                                                                               total_rows, order);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(int d, const PrefillArgs& a, const TcPlan& plan, float* ws,
                              cudaStream_t stream) {
  TcArgs ta{};
  ta.p = a;
  ta.ws = ws;
  ta.seg_len = plan.seg_len;
  ta.nseg_max = plan.nseg_max;
  ta.blk_per_seg = plan.blk_per_seg;
  ta.blk_len = plan.seg_len / plan.blk_per_seg;
  ta.nblk_max = (plan.nseg_max - 1) * plan.blk_per_seg;
  ta.order = nullptr;
  if (plan.sort_docs && a.cu_seqlens != nullptr && a.n_docs > 0) {
    int* order = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + plan.order_off);
    const cudaError_t e = launch_doc_order(a.cu_seqlens, a.n_docs, a.total_rows, order, stream);
    if (e != cudaSuccess) return e;
    ta.order = order;
  }
  if (d == 128) return launch_tc_d<128, false>(ta, stream);
  return plan.pair ? launch_tc_d<64, true>(ta, stream) : launch_tc_d<64, false>(ta, stream);
}

}  // namespace rapt
