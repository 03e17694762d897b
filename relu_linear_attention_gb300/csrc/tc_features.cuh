// Device helpers of the tensor-core RLA-2 kernels: the feature arithmetic of the producer threads
// (RMSNorm, RoPE and ReLU on packed fp32 pairs, 08-rapt-algorithm.md §1 and §3), the per-CTA
// feature tables in shared memory, document bounds and a few shared-memory accessors.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "tc_utils.cuh"

namespace rapt {
namespace feat {

// One increment record: K'^T V of a block as D/4 column groups of [D rows][4 columns] (the float4
// of row r and columns 4j..4j+3 at float4 index j * D + r, so that 32 threads reading their rows'
// same 4 columns read 512 contiguous bytes), then the block's column sums of k' (D floats).
template <int D>
struct Rec {
  static constexpr long FLOATS = static_cast<long>(D) * (D + 1);
  static constexpr long Z = static_cast<long>(D) * D;
};


__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts16(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]),
                    tc::pack_bf16x2(f[4], f[5]), tc::pack_bf16x2(f[6], f[7]));
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

// Document bounds; false if the document is malformed (then treated as empty).
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

// ---------------------------------------------------------------------------------------------
// Feature arithmetic on packed fp32 pairs. A thread's 8 elements are four RoPE pairs m = 0..3
// (elements 2m, 2m+1). They are held as two "structure of arrays" groups g = 0, 1 covering pairs
// 2g and 2g+1: x0[g] = (first element of pair 2g, first of pair 2g+1), x1[g] = the second
// elements, so every rotation step is one packed operation over two pairs.
struct Pairs {
  float2 x0[2], x1[2];
};

__device__ __forceinline__ Pairs unpack_pairs(const uint4& u) {
  // 32-bit word m of the 16 bytes holds pair m: element 2m in the low half, 2m+1 in the high half
  Pairs p;
  p.x0[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.y << 16));
  p.x1[0] = make_float2(__uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y & 0xffff0000u));
  p.x0[1] = make_float2(__uint_as_float(u.z << 16), __uint_as_float(u.w << 16));
  p.x1[1] = make_float2(__uint_as_float(u.z & 0xffff0000u), __uint_as_float(u.w & 0xffff0000u));
  return p;
}

__device__ __forceinline__ float sumsq(const Pairs& p) {
  float2 acc = __fmul2_rn(p.x0[0], p.x0[0]);
  acc = __ffma2_rn(p.x1[0], p.x1[0], acc);
  acc = __ffma2_rn(p.x0[1], p.x0[1], acc);
  acc = __ffma2_rn(p.x1[1], p.x1[1], acc);
  return acc.x + acc.y;
}

template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Per-thread RoPE constants: gains and the sin/cos of the current row's angles, in pair groups.
struct Rot {
  float2 c[2], s[2];  // cos / sin of pairs (2g, 2g+1)
};

// ReLU(RoPE(x * gamma * rinv)), in place (the gains come multiplied by the row's 1 / rms: RoPE is
// linear, so that is the same as normalising first): x0 <- first elements, x1 <- second elements
// of the rotated pairs.
__device__ __forceinline__ void rope_relu(Pairs& p, const float2 (&g0)[2], const float2 (&g1)[2],
                                          const Rot& r) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const float2 y0 = __fmul2_rn(p.x0[g], g0[g]);
    const float2 y1 = __fmul2_rn(p.x1[g], g1[g]);
    const float2 ns = make_float2(-r.s[g].x, -r.s[g].y);
    const float2 u = __ffma2_rn(y0, r.c[g], __fmul2_rn(y1, ns));   // y0 c - y1 s
    const float2 v = __ffma2_rn(y0, r.s[g], __fmul2_rn(y1, r.c[g]));  // y0 s + y1 c
    p.x0[g] = make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f));
    p.x1[g] = make_float2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f));
  }
}
// RoPE(x * gamma * rinv) in place, without the ReLU (pack_pairs_relu applies it while rounding).
__device__ __forceinline__ void rope_scaled(Pairs& p, const float2 (&g0)[2], const float2 (&g1)[2],
                                            const Rot& r) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const float2 y0 = __fmul2_rn(p.x0[g], g0[g]);
    const float2 y1 = __fmul2_rn(p.x1[g], g1[g]);
    const float2 ns = make_float2(-r.s[g].x, -r.s[g].y);
    p.x0[g] = __ffma2_rn(y0, r.c[g], __fmul2_rn(y1, ns));    // y0 c - y1 s
    p.x1[g] = __ffma2_rn(y0, r.s[g], __fmul2_rn(y1, r.c[g]));  // y0 s + y1 c
  }
}
__device__ __forceinline__ void scale_gains(float2 (&g0)[2], float2 (&g1)[2], float s) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    g0[g] = __fmul2_rn(g0[g], s2);
    g1[g] = __fmul2_rn(g1[g], s2);
  }
}

__device__ __forceinline__ uint4 pack_pairs(const Pairs& p) {
  return make_uint4(tc::pack_bf16x2(p.x0[0].x, p.x1[0].x), tc::pack_bf16x2(p.x0[0].y, p.x1[0].y),
                    tc::pack_bf16x2(p.x0[1].x, p.x1[1].x), tc::pack_bf16x2(p.x0[1].y, p.x1[1].y));
}

// max(0, x) of the pairs, rounded to bf16 and packed in element order (one conversion per pair).
__device__ __forceinline__ uint4 pack_pairs_relu(const Pairs& p) {
  return make_uint4(tc::pack_bf16x2_relu(p.x0[0].x, p.x1[0].x), tc::pack_bf16x2_relu(p.x0[0].y, p.x1[0].y),
                    tc::pack_bf16x2_relu(p.x0[1].x, p.x1[1].x), tc::pack_bf16x2_relu(p.x0[1].y, p.x1[1].y));
}

// Advances the angles by a fixed step (cos / sin of the step in `st`): one exact rotation.
__device__ __forceinline__ void rot_step(Rot& r, const Rot& st) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const float2 ns = make_float2(-r.s[g].x, -r.s[g].y);
    const float2 c = __ffma2_rn(r.c[g], st.c[g], __fmul2_rn(ns, st.s[g]));
    const float2 s = __ffma2_rn(r.s[g], st.c[g], __fmul2_rn(r.c[g], st.s[g]));
    r.c[g] = c;
    r.s[g] = s;
  }
}

// Column sums of the 8 per-thread values over the rows of a warp (lanes with equal lane % TPR).
template <int TPR>
__device__ __forceinline__ void warp_colsum(float* z) {
#pragma unroll
  for (int off = TPR; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] += __shfl_xor_sync(0xffffffffu, z[e], off);
}
__device__ __forceinline__ void pairs_to8(const Pairs& p, float* f) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    f[4 * g + 0] = p.x0[g].x;
    f[4 * g + 1] = p.x1[g].x;
    f[4 * g + 2] = p.x0[g].y;
    f[4 * g + 3] = p.x1[g].y;
  }
}

// Per-CTA feature constants in shared memory (8 * D floats), so that the producers need no
// registers for them and no lane-divergent reads of the kernel parameters: the gains of q and k,
// and for every RoPE pair the frequency (hi, lo turns) and the cos / sin of the rotation over
// one producer pass (RPP positions). Gains are stored "split": the first 4 of a thread's 8
// values for every thread part, then the last 4, so that a warp's 16-byte reads are contiguous
// (no bank conflicts); inside each 4 the order is (pair 0 first, pair 1 first, pair 0 second,
// pair 1 second), so that a 16-byte read lands directly on the float2 pairs the arithmetic uses.
// split_idx maps an element index to that layout.
struct FeatTab {
  float* gq;   // [D]
  float* gk;   // [D]
  float* fhi;  // [D/2]
  float* flo;  // [D/2]
  float* stc;  // [D/2] cos of the per-pass rotation
  float* sts;  // [D/2] sin
};
template <int D>
__device__ __forceinline__ FeatTab feat_tab(uint8_t* p) {
  float* f = reinterpret_cast<float*>(p);
  return FeatTab{f, f + D, f + 2 * D, f + 2 * D + D / 2, f + 3 * D, f + 3 * D + D / 2};
}
template <int D>
__device__ __forceinline__ int split_idx(int i) {
  return (i & 4) * (D / 8) + (i >> 3) * 4 + (((i & 1) << 1) | ((i >> 1) & 1));
}
// A row of D elements holds D / DH heads of DH elements (heads h, h + 1, ...: two heads of 64 in a
// 128-wide tile, or one head), each with its own gains and the same RoPE frequencies.
template <int D, int DH = D>
__device__ __forceinline__ void fill_tab(const FeatTab& t, const PrefillArgs& a, int h, int rpp,
                                         int tid, int nthreads) {
  for (int i = tid; i < D; i += nthreads) {
    const long gi = static_cast<long>(h + i / DH) * a.fa.gamma_stride + i % DH;
    t.gq[split_idx<D>(i)] = a.gamma_q[gi];
    t.gk[split_idx<D>(i)] = a.gamma_k[gi];
  }
  for (int j = tid; j < D / 2; j += nthreads) {
    const int jh = j % (DH / 2);
    t.fhi[j] = a.fa.rope_hi[jh];
    t.flo[j] = a.fa.rope_lo[jh];
    float sn, cs;
    rope_sincos(rpp, a.fa.rope_hi[jh], a.fa.rope_lo[jh], sn, cs);
    t.stc[j] = cs;
    t.sts[j] = sn;
  }
}
// Two float4 halves of a thread's 8 values in a split table, in pair groups.
template <int D>
__device__ __forceinline__ void split_load(const float* t, int part, float2 (&x0)[2], float2 (&x1)[2]) {
  const float4 a = *reinterpret_cast<const float4*>(t + 4 * part);
  const float4 b = *reinterpret_cast<const float4*>(t + D / 2 + 4 * part);
  x0[0] = make_float2(a.x, a.y);
  x1[0] = make_float2(a.z, a.w);
  x0[1] = make_float2(b.x, b.y);
  x1[1] = make_float2(b.z, b.w);
}
__device__ __forceinline__ void tab_step(const FeatTab& t, int j0, Rot& st) {
  const float4 c = *reinterpret_cast<const float4*>(t.stc + j0);
  const float4 sn = *reinterpret_cast<const float4*>(t.sts + j0);
  st.c[0] = make_float2(c.x, c.y);
  st.c[1] = make_float2(c.z, c.w);
  st.s[0] = make_float2(sn.x, sn.y);
  st.s[1] = make_float2(sn.z, sn.w);
}
__device__ __forceinline__ void tab_rot_at(const FeatTab& t, int pos, int j0, Rot& r) {
  const float4 hi = *reinterpret_cast<const float4*>(t.fhi + j0);
  const float4 lo = *reinterpret_cast<const float4*>(t.flo + j0);
  float s0, c0, s1, c1, s2, c2, s3, c3;
  rope_sincos(pos, hi.x, lo.x, s0, c0);
  rope_sincos(pos, hi.y, lo.y, s1, c1);
  rope_sincos(pos, hi.z, lo.z, s2, c2);
  rope_sincos(pos, hi.w, lo.w, s3, c3);
  r.c[0] = make_float2(c0, c1);
  r.c[1] = make_float2(c2, c3);
  r.s[0] = make_float2(s0, s1);
  r.s[1] = make_float2(s2, s3);
}


}  // namespace feat
}  // namespace rapt
