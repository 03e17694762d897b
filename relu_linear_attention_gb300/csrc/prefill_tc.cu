// Chunked causal RLA-2 forward on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
// bf16 inputs, d in {64, 128}; fp32 accumulation and fp32 state.
//
// The method (08-rapt-algorithm.md §3): q' = ReLU(RoPE(RMSNorm(q))), k' likewise,
// S_t = S_{t-1} + k'_t v_t^T, z_t = z_{t-1} + k'_t, out_t = q'_t S_t / (q'_t . z_t + 1e-4),
// with the state restarting at every document (§2.2, §4.1). It is evaluated chunk by chunk
// (C = 128 tokens), the chunk-parallel form the page mentions (§1, §3), as four tile GEMMs per
// chunk, all bf16 x bf16 -> fp32 on the tensor cores:
//
//   P  = Q'_c K'_c^T                       (128 x 128)    -> TMEM
//   O  = Q'_c [S | z]~                     (128 x (d+16)) -> TMEM   carried-in state, bf16 copy
//   [S | z] += K'_c^T [V_c | 1]            (d x (d+16))   -> TMEM   fp32 master state
//   O += (P masked to tau <= t)~ [V_c | 1]                -> TMEM
//   out = O[:, :d] / (O[:, d] + eps)
//
// A column of ones appended to V makes the tensor core produce z (column d of the state), the
// inter-chunk denominator q'.z (column d of Q'[S|z]) and the intra-chunk row sums of P (column d
// of P[V|1]) in the same MMAs, so the denominator needs no CUDA-core reduction. (~ marks the bf16
// rounding of an MMA operand; the numerator and denominator use the same rounded weights.)
//
// Sequence parallelism: a document is cut into segments of seg_len tokens. Kernel A computes the
// state increment of every segment but the last (K'^T [V | 1] over the segment); kernel B runs one
// CTA per (document, head, segment) that starts from S0 + the increments of the earlier segments
// (summed in segment order: deterministic) and walks the segment's chunks. The last segment's CTA
// writes the final state.
#include "kernels.h"
#include "tc_utils.cuh"

namespace rapt {
namespace {

constexpr int kC = 128;        // chunk length = MMA M
constexpr int kThreads = 256;  // 8 warps: two per TMEM lane quarter
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s: an MMA that has not finished by then never will
constexpr uint32_t kDevTimeout = 2u;

template <int D>
struct TcCfg {
  static constexpr int NA = D + 16;       // [V | 1 0 ... 0] columns
  static constexpr int KB = D / 64;       // 64-column blocks of q', k', S rows
  static constexpr int VB = KB + 1;       // value blocks incl. the ones block
  static constexpr int TPR = D / 16;      // prologue threads per token row (16 elements each)
  static constexpr int RPP = kThreads / TPR;  // rows per prologue pass
  static constexpr int NPASS = kC / RPP;
  // shared-memory byte offsets from a 1024-byte aligned base
  static constexpr uint32_t QS = 0;                                    // q' : KB x 16 KB
  static constexpr uint32_t KS = QS + KB * 16384;                      // k' : KB x 16 KB (+ zero block if D = 64)
  static constexpr uint32_t KS_END = KS + 2 * 16384;                   // M = 128 view of k'^T
  static constexpr uint32_t PS = (D == 128) ? QS : KS_END;             // P~ : 2 x 16 KB (aliases q' at D = 128)
  static constexpr uint32_t VS = (D == 128) ? KS_END : PS + 2 * 16384; // [V | 1] : VB x 16 KB
  static constexpr uint32_t SS = VS + VB * 16384;                      // [S | z]~ : VB x (D rows x 128 B)
  static constexpr uint32_t CTRL = SS + VB * D * 128;                  // barriers, TMEM base, flags
  static constexpr uint32_t BYTES = CTRL + 64 + 1024;                  // + alignment slack
  // TMEM columns
  static constexpr uint32_t TP = 0, TO = 128, TS = 288;
  static_assert(TS + NA <= 512, "TMEM budget");
};

// Kernel A shared layout (k' and [V | 1] only).
template <int D>
struct TcCfgA {
  static constexpr int KB = D / 64, VB = KB + 1;
  static constexpr uint32_t KS = 0;
  static constexpr uint32_t VS = KS + 2 * 16384;
  static constexpr uint32_t CTRL = VS + VB * 16384;
  static constexpr uint32_t BYTES = CTRL + 64 + 1024;
};

struct TcArgs {
  PrefillArgs p;
  float* ws;     // segment increments [n_docs][H][nseg_max][D][D + 1]
  int seg_len;   // tokens per segment (multiple of kC)
  int nseg_max;  // segments per document slot in the grid
};

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[m]));
    f[2 * m] = g.x;
    f[2 * m + 1] = g.y;
  }
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void sts16(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Document bounds for a CTA; false if the document is malformed (reported, then skipped).
__device__ __forceinline__ bool doc_bounds(const PrefillArgs& a, int doc, long& row0, int& n) {
  if (a.cu_seqlens != nullptr) {
    const int s = a.cu_seqlens[doc];
    const int e = a.cu_seqlens[doc + 1];
    const int prev = doc > 0 ? a.cu_seqlens[doc - 1] : 0;
    const bool bad = s < 0 || e < s || prev > s || e > a.total_rows || (doc == 0 && s != 0) ||
                     (doc == a.n_docs - 1 && e != a.total_rows) || (e - s) > a.max_seqlen;
    if (bad) {
      row0 = 0;
      n = 0;
      return false;
    }
    row0 = s;
    n = e - s;
  } else {
    row0 = static_cast<long>(doc) * a.doc_len;
    n = a.doc_len;
  }
  return true;
}

// Features of 16 consecutive elements of one token row (this thread's part), for q and k at the
// same position: RMSNorm over the row (shuffle across the TPR threads of the row), RoPE, ReLU,
// rounded to bf16 and packed into 2 x 16 bytes each.
template <int D>
__device__ __forceinline__ void features16(const uint4 (&xq)[2], const uint4 (&xk)[2], bool valid,
                                           int pos, const float (&gq)[16], const float (&gk)[16],
                                           const float (&fhi)[8], const float (&flo)[8],
                                           float eps_norm, uint4 (&oq)[2], uint4 (&ok)[2]) {
  constexpr int TPR = TcCfg<D>::TPR;
  float fq[16], fk[16];
  unpack8(xq[0], fq);
  unpack8(xq[1], fq + 8);
  unpack8(xk[0], fk);
  unpack8(xk[1], fk + 8);
  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    sq = fmaf(fq[e], fq[e], sq);
    sk = fmaf(fk[e], fk[e], sk);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, off);
    sk += __shfl_xor_sync(0xffffffffu, sk, off);
  }
  const float rq = rsqrtf(sq * (1.0f / D) + eps_norm);
  const float rk = rsqrtf(sk * (1.0f / D) + eps_norm);
  uint32_t wq[8], wk[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float s, c;
    rope_sincos(pos, fhi[m], flo[m], s, c);
    const float q0 = fq[2 * m] * rq * gq[2 * m], q1 = fq[2 * m + 1] * rq * gq[2 * m + 1];
    const float k0 = fk[2 * m] * rk * gk[2 * m], k1 = fk[2 * m + 1] * rk * gk[2 * m + 1];
    const float qa = fmaxf(fmaf(q0, c, -q1 * s), 0.f), qb = fmaxf(fmaf(q0, s, q1 * c), 0.f);
    const float ka = fmaxf(fmaf(k0, c, -k1 * s), 0.f), kb = fmaxf(fmaf(k0, s, k1 * c), 0.f);
    wq[m] = valid ? tc::pack_bf16x2(qa, qb) : 0u;
    wk[m] = valid ? tc::pack_bf16x2(ka, kb) : 0u;
  }
  oq[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
  oq[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
  ok[0] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
  ok[1] = make_uint4(wk[4], wk[5], wk[6], wk[7]);
}

// Same for k only (kernel A).
template <int D>
__device__ __forceinline__ void features16_k(const uint4 (&xk)[2], bool valid, int pos,
                                             const float (&gk)[16], const float (&fhi)[8],
                                             const float (&flo)[8], float eps_norm, uint4 (&ok)[2]) {
  constexpr int TPR = TcCfg<D>::TPR;
  float fk[16];
  unpack8(xk[0], fk);
  unpack8(xk[1], fk + 8);
  float sk = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) sk = fmaf(fk[e], fk[e], sk);
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, off);
  const float rk = rsqrtf(sk * (1.0f / D) + eps_norm);
  uint32_t wk[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float s, c;
    rope_sincos(pos, fhi[m], flo[m], s, c);
    const float k0 = fk[2 * m] * rk * gk[2 * m], k1 = fk[2 * m + 1] * rk * gk[2 * m + 1];
    const float ka = fmaxf(fmaf(k0, c, -k1 * s), 0.f), kb = fmaxf(fmaf(k0, s, k1 * c), 0.f);
    wk[m] = valid ? tc::pack_bf16x2(ka, kb) : 0u;
  }
  ok[0] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
  ok[1] = make_uint4(wk[4], wk[5], wk[6], wk[7]);
}

// Column groups (16 columns each) of the [S | z] tile handled by a thread of half `hf`:
// half 0 takes columns [0, D/2) and the z block [D, D + 16), half 1 takes [D/2, D).
template <int D>
struct StateCols {
  static constexpr int N0 = D / 32 + 1;  // groups of half 0
  static constexpr int N1 = D / 32;      // groups of half 1
  static __device__ __forceinline__ int count(int hf) { return hf == 0 ? N0 : N1; }
  static __device__ __forceinline__ int col(int hf, int g) {
    return hf == 0 ? (g < D / 32 ? 16 * g : D) : D / 2 + 16 * g;
  }
};

// Writes 16 fp32 values (columns j0 .. j0+15 of state row i) as bf16 into the [S | z]~ operand.
template <int D>
__device__ __forceinline__ void store_state_bf16(uint32_t ss_base, int i, int j0, const float* v) {
  const int jb = j0 / 64, c = (j0 % 64) / 8;
  uint4 w0 = make_uint4(tc::pack_bf16x2(v[0], v[1]), tc::pack_bf16x2(v[2], v[3]),
                        tc::pack_bf16x2(v[4], v[5]), tc::pack_bf16x2(v[6], v[7]));
  uint4 w1 = make_uint4(tc::pack_bf16x2(v[8], v[9]), tc::pack_bf16x2(v[10], v[11]),
                        tc::pack_bf16x2(v[12], v[13]), tc::pack_bf16x2(v[14], v[15]));
  const uint32_t blk = ss_base + static_cast<uint32_t>(jb) * (D * 128);
  sts16(blk + tc::sw128(i, c), w0);
  sts16(blk + tc::sw128(i, c + 1), w1);
}

// ------------------------------------------------------------------------------------------------
// Kernel B: one CTA per (document, head, segment).
template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const TcArgs ta) {
  using Cfg = TcCfg<D>;
  constexpr int NA = Cfg::NA, TPR = Cfg::TPR, RPP = Cfg::RPP, NPASS = Cfg::NPASS;
  const PrefillArgs& a = ta.p;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % ta.nseg_max;
  const int h = (blockIdx.x / ta.nseg_max) % a.H;
  const int doc = blockIdx.x / (ta.nseg_max * a.H);

  long row0;
  int n;
  const bool good = doc_bounds(a, doc, row0, n);
  if (!good && seg == 0 && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 1u);
  const int nseg_doc = n > 0 ? (n + ta.seg_len - 1) / ta.seg_len : 1;
  if (seg >= nseg_doc) return;  // uniform across the CTA, before any allocation
  const int seg_start = seg * ta.seg_len;
  const int seg_n = min(ta.seg_len, n - seg_start);  // 0 only for an empty document
  const bool last_seg = seg == nseg_doc - 1;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar_a = base + Cfg::CTRL, bar_b = bar_a + 8;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(gbase + Cfg::CTRL + 16);
  int* s_abort = reinterpret_cast<int*>(gbase + Cfg::CTRL + 20);

  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar_a, 1);
    tc::mbar_init(bar_b, 1);
    tc::mbar_fence_init();
    *s_abort = 0;
  }
  // constant parts of the operands: the ones block of [V | 1] (column D of every row), and for
  // D = 64 the zero block that pads k'^T to M = 128
  for (int idx = tid; idx < 16384 / 16; idx += kThreads) {
    const int r = idx / 8, c = idx % 8;
    const uint32_t one = (c == 0) ? 0x3F80u : 0u;  // bf16 1.0 in the first element of chunk 0
    sts16(base + Cfg::VS + Cfg::KB * 16384 + tc::sw128(r, c), make_uint4(one, 0u, 0u, 0u));
    if (D == 64) sts16(base + Cfg::KS + 16384 + idx * 16, make_uint4(0u, 0u, 0u, 0u));
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  const int q4 = warp & 3, hf = warp >> 2;
  const int er = 32 * q4 + lane;  // TMEM lane / tile row owned in the epilogues
  const uint32_t tlane = static_cast<uint32_t>(32 * q4) << 16;
  const long bh = static_cast<long>(doc) * a.H + h;

  // ---- initial state: S0 + increments of the earlier segments -> TMEM (fp32) and [S|z]~ (bf16)
  {
    const float* wsb = ta.ws + (bh * ta.nseg_max) * static_cast<long>(D) * (D + 1);
    for (int g = 0; g < StateCols<D>::count(hf); ++g) {
      const int j0 = StateCols<D>::col(hf, g);
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = j0 + e;
        float x = 0.f;
        if (er < D && j <= D) {
          if (j < D) {
            if (a.S0 != nullptr) x = a.S0[(bh * D + er) * D + j];
          } else if (a.z0 != nullptr) {
            x = a.z0[bh * D + er];
          }
          for (int gs = 0; gs < seg; ++gs) x += wsb[(static_cast<long>(gs) * D + er) * (D + 1) + j];
        }
        v[e] = x;
      }
      uint32_t u[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(v[e]);
      tc::tmem_st16(tmem + tlane + Cfg::TS + j0, u);
      if (er < D) store_state_bf16<D>(base + Cfg::SS, er, j0, v);
    }
    tc::tmem_wait_st();
  }

  // ---- per-thread constants of the prologue
  const int prow = tid / TPR, part = tid % TPR;
  const int e0 = 16 * part;
  float gq[16], gk[16], fhi[8], flo[8];
  {
    const float* gqp = a.gamma_q + h * a.fa.gamma_stride;
    const float* gkp = a.gamma_k + h * a.fa.gamma_stride;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      gq[e] = gqp[e0 + e];
      gk[e] = gkp[e0 + e];
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      fhi[m] = a.fa.rope_hi[(e0 >> 1) + m];
      flo[m] = a.fa.rope_lo[(e0 >> 1) + m];
    }
  }
  const uint32_t pro_off = static_cast<uint32_t>(part / 4) * 16384;  // 64-column block
  const int pro_c = (part % 4) * 2;                                   // first 16-byte chunk
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v);
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.out);
  const int pos_base = a.pos_offset + seg_start;

  uint4 rq[NPASS][2], rk[NPASS][2], rv[NPASS][2];
  auto prefetch = [&](int t0) {
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
      const int lt = t0 + p * RPP + prow;
      if (lt < seg_n) {
        const long off = ((row0 + seg_start + lt) * a.H + h) * D + e0;
        rq[p][0] = ldg16(qg + off);
        rq[p][1] = ldg16(qg + off + 8);
        rk[p][0] = ldg16(kg + off);
        rk[p][1] = ldg16(kg + off + 8);
        rv[p][0] = ldg16(vg + off);
        rv[p][1] = ldg16(vg + off + 8);
      } else {
        rq[p][0] = rq[p][1] = rk[p][0] = rk[p][1] = rv[p][0] = rv[p][1] = make_uint4(0, 0, 0, 0);
      }
    }
  };

  constexpr uint32_t ID_P = tc::idesc_bf16(128, 128, false, false);
  constexpr uint32_t ID_QS = tc::idesc_bf16(128, NA, false, true);
  constexpr uint32_t ID_KV = tc::idesc_bf16(128, NA, true, true);
  constexpr uint32_t ID_PV = tc::idesc_bf16(128, NA, false, true);

  uint32_t phase_a = 0, phase_b = 0;
  bool aborted = false;
  uint32_t fail_bar = 0, fail_parity = 0;  // the wait that gave up, if any
  if (seg_n > 0) prefetch(0);

  for (int t0 = 0; t0 < seg_n; t0 += kC) {
    // ---- prologue: features of the chunk into q', k'; raw v into [V | 1]
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
      const int r = p * RPP + prow;
      const bool valid = t0 + r < seg_n;
      uint4 oq[2], ok[2];
      features16<D>(rq[p], rk[p], valid, pos_base + t0 + r, gq, gk, fhi, flo, a.fa.eps_norm, oq, ok);
      sts16(base + Cfg::QS + pro_off + tc::sw128(r, pro_c), oq[0]);
      sts16(base + Cfg::QS + pro_off + tc::sw128(r, pro_c + 1), oq[1]);
      sts16(base + Cfg::KS + pro_off + tc::sw128(r, pro_c), ok[0]);
      sts16(base + Cfg::KS + pro_off + tc::sw128(r, pro_c + 1), ok[1]);
      sts16(base + Cfg::VS + pro_off + tc::sw128(r, pro_c), rv[p][0]);
      sts16(base + Cfg::VS + pro_off + tc::sw128(r, pro_c + 1), rv[p][1]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    if (tid == 0) {
      tc::fence_after_sync();
      // P = Q' K'^T
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t off = (s / 4) * 16384 + (s % 4) * 32;
        tc::mma_bf16(tmem + Cfg::TP, tc::desc_sw128(base + Cfg::QS + off, 16, 1024),
                     tc::desc_sw128(base + Cfg::KS + off, 16, 1024), ID_P, s > 0);
      }
      // O = Q' [S | z]~   (carried-in state)
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t off = (s / 4) * 16384 + (s % 4) * 32;
        tc::mma_bf16(tmem + Cfg::TO, tc::desc_sw128(base + Cfg::QS + off, 16, 1024),
                     tc::desc_sw128(base + Cfg::SS + s * 2048, D * 128, 1024), ID_QS, s > 0);
      }
      // [S | z] += K'^T [V | 1]
#pragma unroll
      for (int s = 0; s < kC / 16; ++s) {
        tc::mma_bf16(tmem + Cfg::TS, tc::desc_sw128(base + Cfg::KS + s * 2048, 16384, 1024),
                     tc::desc_sw128(base + Cfg::VS + s * 2048, 16384, 1024), ID_KV, 1u);
      }
      tc::mma_commit(bar_a);
    }
    if (t0 + kC < seg_n) prefetch(t0 + kC);  // next chunk's loads overlap this chunk's work

    if (!tc::mbar_wait(bar_a, phase_a, kWaitCycles)) *s_abort = 1;
    __syncthreads();
    if (*s_abort) {
      aborted = true;
      fail_bar = bar_a;
      fail_parity = phase_a;
      break;
    }
    phase_a ^= 1;
    tc::fence_after_sync();

    // ---- P -> masked bf16 P~ ; [S | z] (after this chunk) -> bf16 [S | z]~ for the next chunk
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t u[16];
      tc::tmem_ld16(tmem + tlane + Cfg::TP + 64 * hf + 16 * m, u);
      tc::tmem_wait_ld();
      float f[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int tau = 64 * hf + 16 * m + e;
        f[e] = tau <= er ? __uint_as_float(u[e]) : 0.f;
      }
      const uint32_t blk = base + Cfg::PS + hf * 16384;
      sts16(blk + tc::sw128(er, 2 * m),
            make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]),
                       tc::pack_bf16x2(f[4], f[5]), tc::pack_bf16x2(f[6], f[7])));
      sts16(blk + tc::sw128(er, 2 * m + 1),
            make_uint4(tc::pack_bf16x2(f[8], f[9]), tc::pack_bf16x2(f[10], f[11]),
                       tc::pack_bf16x2(f[12], f[13]), tc::pack_bf16x2(f[14], f[15])));
    }
    if (32 * q4 < D) {  // warp-uniform: TMEM rows >= D hold the zero padding of k'^T
      for (int g = 0; g < StateCols<D>::count(hf); ++g) {
        const int j0 = StateCols<D>::col(hf, g);
        uint32_t u[16];
        tc::tmem_ld16(tmem + tlane + Cfg::TS + j0, u);
        tc::tmem_wait_ld();
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(u[e]);
        store_state_bf16<D>(base + Cfg::SS, er, j0, v);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    if (tid == 0) {
      tc::fence_after_sync();
      // O += P~ [V | 1]
#pragma unroll
      for (int s = 0; s < kC / 16; ++s) {
        const uint32_t off = (s / 4) * 16384 + (s % 4) * 32;
        tc::mma_bf16(tmem + Cfg::TO, tc::desc_sw128(base + Cfg::PS + off, 16, 1024),
                     tc::desc_sw128(base + Cfg::VS + s * 2048, 16384, 1024), ID_PV, 1u);
      }
      tc::mma_commit(bar_b);
    }
    if (!tc::mbar_wait(bar_b, phase_b, kWaitCycles)) *s_abort = 1;
    __syncthreads();
    if (*s_abort) {
      aborted = true;
      fail_bar = bar_b;
      fail_parity = phase_b;
      break;
    }
    phase_b ^= 1;
    tc::fence_after_sync();

    // ---- epilogue: out = O[:, :D] / (O[:, D] + eps)
    {
      uint32_t dz;
      tc::tmem_ld1(tmem + tlane + Cfg::TO + D, dz);
      tc::tmem_wait_ld();
      const float inv = 1.0f / (__uint_as_float(dz) + a.eps_den);
      const bool valid = t0 + er < seg_n;
      __nv_bfloat16* orow = og + ((row0 + seg_start + t0 + er) * a.H + h) * D + hf * (D / 2);
#pragma unroll
      for (int m = 0; m < D / 32; ++m) {
        uint32_t u[16];
        tc::tmem_ld16(tmem + tlane + Cfg::TO + hf * (D / 2) + 16 * m, u);
        tc::tmem_wait_ld();
        if (valid) {
          float f[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(u[e]) * inv;
          uint4* dst = reinterpret_cast<uint4*>(orow + 16 * m);
          dst[0] = make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]),
                              tc::pack_bf16x2(f[4], f[5]), tc::pack_bf16x2(f[6], f[7]));
          dst[1] = make_uint4(tc::pack_bf16x2(f[8], f[9]), tc::pack_bf16x2(f[10], f[11]),
                              tc::pack_bf16x2(f[12], f[13]), tc::pack_bf16x2(f[14], f[15]));
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
  }

  if (aborted) {
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevTimeout);
    // give the MMAs still in flight a bounded chance to land before TMEM is released
    tc::mbar_wait(fail_bar, fail_parity, kWaitCycles);
  } else if (last_seg && (a.S_final != nullptr || a.z_final != nullptr) && 32 * q4 < D) {
    // ---- final state of the document
    tc::fence_after_sync();
    for (int g = 0; g < StateCols<D>::count(hf); ++g) {
      const int j0 = StateCols<D>::col(hf, g);
      uint32_t u[16];
      tc::tmem_ld16(tmem + tlane + Cfg::TS + j0, u);
      tc::tmem_wait_ld();
      if (j0 < D) {
        if (a.S_final != nullptr) {
          float4* dst = reinterpret_cast<float4*>(a.S_final + (bh * D + er) * D + j0);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                 __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
        }
      } else if (a.z_final != nullptr) {
        a.z_final[bh * D + er] = __uint_as_float(u[0]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// Kernel A: state increment [S | z] of one segment (every segment but a document's last).
template <int D>
__global__ void __launch_bounds__(kThreads, 1) segment_state_kernel(const TcArgs ta) {
  using Cfg = TcCfg<D>;
  using CA = TcCfgA<D>;
  constexpr int NA = Cfg::NA, TPR = Cfg::TPR, RPP = Cfg::RPP, NPASS = Cfg::NPASS;
  const PrefillArgs& a = ta.p;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x % ta.nseg_max;
  const int h = (blockIdx.x / ta.nseg_max) % a.H;
  const int doc = blockIdx.x / (ta.nseg_max * a.H);
  long row0;
  int n;
  doc_bounds(a, doc, row0, n);  // a malformed document has n = 0 and is skipped
  const int nseg_doc = n > 0 ? (n + ta.seg_len - 1) / ta.seg_len : 1;
  if (seg >= nseg_doc - 1) return;  // the last segment's increment is not needed
  const int seg_start = seg * ta.seg_len;
  const int seg_n = ta.seg_len;  // a non-last segment is full

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar = base + CA::CTRL;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(gbase + CA::CTRL + 16);
  int* s_abort = reinterpret_cast<int*>(gbase + CA::CTRL + 20);

  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_fence_init();
    *s_abort = 0;
  }
  for (int idx = tid; idx < 16384 / 16; idx += kThreads) {
    const int r = idx / 8, c = idx % 8;
    const uint32_t one = (c == 0) ? 0x3F80u : 0u;
    sts16(base + CA::VS + CA::KB * 16384 + tc::sw128(r, c), make_uint4(one, 0u, 0u, 0u));
    if (D == 64) sts16(base + CA::KS + 16384 + idx * 16, make_uint4(0u, 0u, 0u, 0u));
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  const int prow = tid / TPR, part = tid % TPR;
  const int e0 = 16 * part;
  float gk[16], fhi[8], flo[8];
  {
    const float* gkp = a.gamma_k + h * a.fa.gamma_stride;
#pragma unroll
    for (int e = 0; e < 16; ++e) gk[e] = gkp[e0 + e];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      fhi[m] = a.fa.rope_hi[(e0 >> 1) + m];
      flo[m] = a.fa.rope_lo[(e0 >> 1) + m];
    }
  }
  const uint32_t pro_off = static_cast<uint32_t>(part / 4) * 16384;
  const int pro_c = (part % 4) * 2;
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v);
  const int pos_base = a.pos_offset + seg_start;

  uint4 rk[NPASS][2], rv[NPASS][2];
  auto prefetch = [&](int t0) {
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
      const int lt = t0 + p * RPP + prow;
      const long off = ((row0 + seg_start + lt) * a.H + h) * D + e0;
      rk[p][0] = ldg16(kg + off);
      rk[p][1] = ldg16(kg + off + 8);
      rv[p][0] = ldg16(vg + off);
      rv[p][1] = ldg16(vg + off + 8);
    }
  };
  constexpr uint32_t ID_KV = tc::idesc_bf16(128, NA, true, true);
  uint32_t phase = 0;
  bool aborted = false;
  prefetch(0);
  for (int t0 = 0; t0 < seg_n; t0 += kC) {
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
      const int r = p * RPP + prow;
      uint4 ok[2];
      features16_k<D>(rk[p], true, pos_base + t0 + r, gk, fhi, flo, a.fa.eps_norm, ok);
      sts16(base + CA::KS + pro_off + tc::sw128(r, pro_c), ok[0]);
      sts16(base + CA::KS + pro_off + tc::sw128(r, pro_c + 1), ok[1]);
      sts16(base + CA::VS + pro_off + tc::sw128(r, pro_c), rv[p][0]);
      sts16(base + CA::VS + pro_off + tc::sw128(r, pro_c + 1), rv[p][1]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int s = 0; s < kC / 16; ++s) {
        tc::mma_bf16(tmem, tc::desc_sw128(base + CA::KS + s * 2048, 16384, 1024),
                     tc::desc_sw128(base + CA::VS + s * 2048, 16384, 1024), ID_KV,
                     (t0 > 0 || s > 0) ? 1u : 0u);
      }
      tc::mma_commit(bar);
    }
    if (t0 + kC < seg_n) prefetch(t0 + kC);
    if (!tc::mbar_wait(bar, phase, kWaitCycles)) *s_abort = 1;
    __syncthreads();
    if (*s_abort) {
      aborted = true;
      break;
    }
    phase ^= 1;
  }

  const int q4 = warp & 3, hf = warp >> 2;
  const int er = 32 * q4 + lane;
  const uint32_t tlane = static_cast<uint32_t>(32 * q4) << 16;
  if (aborted) {
    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, kDevTimeout);
    tc::mbar_wait(bar, phase, kWaitCycles);
  } else if (32 * q4 < D) {
    tc::fence_after_sync();
    const long bh = static_cast<long>(doc) * a.H + h;
    float* dst = ta.ws + ((bh * ta.nseg_max + seg) * D + er) * static_cast<long>(D + 1);
    for (int g = 0; g < StateCols<D>::count(hf); ++g) {
      const int j0 = StateCols<D>::col(hf, g);
      uint32_t u[16];
      tc::tmem_ld16(tmem + tlane + j0, u);
      tc::tmem_wait_ld();
      if (j0 < D) {
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[j0 + e] = __uint_as_float(u[e]);
      } else {
        dst[D] = __uint_as_float(u[0]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
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
cudaError_t launch_tc_d(const TcArgs& ta, cudaStream_t stream) {
  static unsigned long long cfg_a = 0, cfg_b = 0;
  cudaError_t e = set_smem(prefill_tc_kernel<D>, TcCfg<D>::BYTES, cfg_b);
  if (e != cudaSuccess) return e;
  e = set_smem(segment_state_kernel<D>, TcCfgA<D>::BYTES, cfg_a);
  if (e != cudaSuccess) return e;
  const long units = static_cast<long>(ta.p.n_docs) * ta.p.H;
  if (units == 0) return cudaSuccess;
  if (ta.nseg_max > 1) {
    segment_state_kernel<D><<<static_cast<unsigned>(units * ta.nseg_max), kThreads, TcCfgA<D>::BYTES, stream>>>(ta);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  prefill_tc_kernel<D><<<static_cast<unsigned>(units * ta.nseg_max), kThreads, TcCfg<D>::BYTES, stream>>>(ta);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(DType dt, int d) { return dt == DType::BF16 && (d == 64 || d == 128); }

TcPlan tc_plan(int n_docs, int H, int max_seqlen, long total_tokens, int d) {
  // Estimated time in units of one kernel-B chunk. Kernel B runs one CTA per SM (waves of 152
  // CTAs, each CTA costing its chunks plus about one chunk of state set-up); a kernel-A chunk
  // (k features + one GEMM) costs about 0.4 of a kernel-B chunk and kernel A fits two CTAs per
  // SM. Documents are assumed to share the tokens evenly, except that the longest one bounds the
  // segment count. The segment length with the smallest estimate wins.
  TcPlan best{1, kC, 0};
  const int chunks_max = max_seqlen > 0 ? (max_seqlen + kC - 1) / kC : 1;
  const double avg_chunks = n_docs > 0 ? static_cast<double>(total_tokens) / n_docs / kC : 0.0;
  double best_cost = 1e300;
  for (int seg_chunks = chunks_max; seg_chunks >= 1; --seg_chunks) {
    const int nseg = (chunks_max + seg_chunks - 1) / seg_chunks;
    if (nseg > 64) break;
    const double segs_per_doc = avg_chunks > 0 ? static_cast<double>(static_cast<long>(
                                                      (avg_chunks + seg_chunks - 1e-9) / seg_chunks))
                                               : 1.0;
    const double items_b = static_cast<double>(H) * n_docs * (segs_per_doc > 1 ? segs_per_doc : 1.0);
    const double items_a = items_b - static_cast<double>(H) * n_docs;
    const double waves_b = static_cast<double>(static_cast<long>((items_b + 151) / 152));
    const double waves_a = items_a > 0 ? static_cast<double>(static_cast<long>((items_a + 303) / 304)) : 0.0;
    const double cost = waves_b * (seg_chunks + 1.0) + 0.4 * waves_a * seg_chunks;
    if (cost < 0.95 * best_cost) {  // more segments cost workspace: demand a clear gain
      best_cost = cost;
      best.nseg_max = nseg;
      best.seg_len = seg_chunks * kC;
    }
  }
  const long units = static_cast<long>(n_docs) * H;
  best.ws_bytes = best.nseg_max > 1
                      ? static_cast<size_t>(units) * best.nseg_max * d * (d + 1) * sizeof(float)
                      : 0;
  return best;
}

cudaError_t launch_prefill_tc(int d, const PrefillArgs& a, const TcPlan& plan, float* ws,
                              cudaStream_t stream) {
  TcArgs ta{};
  ta.p = a;
  ta.ws = ws;
  ta.seg_len = plan.seg_len;
  ta.nseg_max = plan.nseg_max;
  return d == 128 ? launch_tc_d<128>(ta, stream) : launch_tc_d<64>(ta, stream);
}

}  // namespace rapt
