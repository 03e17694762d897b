// Shared helpers of the lockstep tensor-core kernels with d = 128 (the backward and the causal L2
// form): addressing of 128-byte-swizzled bf16 tiles (128 rows x 128 columns, or d rows), operand
// descriptors, TMEM row reads and state hand-over, sm_103a.
#pragma once

#include <cuda_bf16.h>

#include "tc_features.cuh"
#include "tc_utils.cuh"

namespace rapt {
namespace tct {

constexpr int kD = 128;
constexpr long long kWait = 2000000000LL;  // ~1 s of SM cycles

// Byte offset of 16-byte chunk m (0..15, 8 bf16 each) of row r in a 128-row tile of 128 columns.
__device__ __forceinline__ uint32_t tile_off(int r, int m) {
  return static_cast<uint32_t>(m >> 3) * 16384u + tc::sw128(r, m & 7);
}
// The same in a D-row tile (S~ / R~: rows = D).
__device__ __forceinline__ uint32_t dtile_off(int r, int m) {
  return static_cast<uint32_t>(m >> 3) * (kD * 128u) + tc::sw128(r, m & 7);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

// K-major operand descriptor of a 128-row tile, K step k (16 elements).
__device__ __forceinline__ uint64_t kmaj(uint32_t tile, int k) {
  return tc::desc_sw128(tile, 16, 1024) + static_cast<uint64_t>((k >> 2) * 1024 + (k & 3) * 2);
}
// K-major operand descriptor of a D-row tile (S~ / R~ as N x K).
__device__ __forceinline__ uint64_t kmaj_d(uint32_t tile, int k) {
  return tc::desc_sw128(tile, 16, 1024) + static_cast<uint64_t>((k >> 2) * (kD * 8) + (k & 3) * 2);
}
// MN-major operand descriptor (rows = K): 128-row tile (LBO 16 KB) or D-row tile (LBO D*128 B).
__device__ __forceinline__ uint64_t mnmaj(uint32_t tile, int k, uint32_t lbo) {
  return tc::desc_sw128(tile, lbo, 1024) + static_cast<uint64_t>(k) * 128;
}

// Reads 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t u[2][16];
  tc::tmem_ld16(taddr, u[0]);
  tc::tmem_ld16(taddr + 16, u[1]);
  tc::tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    v[e] = __uint_as_float(u[0][e]);
    v[16 + e] = __uint_as_float(u[1][e]);
  }
}

// Two such reads with both in flight before the one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, float (&va)[32], uint32_t tb, float (&vb)[32]) {
  uint32_t u[4][16];
  tc::tmem_ld16(ta, u[0]);
  tc::tmem_ld16(ta + 16, u[1]);
  tc::tmem_ld16(tb, u[2]);
  tc::tmem_ld16(tb + 16, u[3]);
  tc::tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    va[e] = __uint_as_float(u[0][e]);
    va[16 + e] = __uint_as_float(u[1][e]);
    vb[e] = __uint_as_float(u[2][e]);
    vb[16 + e] = __uint_as_float(u[3][e]);
  }
}

// 32 fp32 values as bf16 into row r, columns 32 g .. 32 g + 31 of a tile (tile_off or dtile_off).
template <bool DROWS>
__device__ __forceinline__ void store_row32(uint32_t tile, int r, int g, const float (&v)[32]) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t off = DROWS ? dtile_off(r, 4 * g + m) : tile_off(r, 4 * g + m);
    feat::sts16(tile + off, feat::pack8(v + 8 * m));
  }
}

// Waits for an mbarrier phase; returns false when the wait gave up.
__device__ __forceinline__ bool wait_mma(uint32_t bar, int parity) {
  const bool ok = tc::mbar_wait(bar, parity, kWait);
  tc::fence_after_sync();
  return ok;
}

// A state (S or R) into TMEM lane t (this thread's lane), columns 32 gw .. 32 gw + 31 (taddr points
// there), and its bf16 copy into row t of the D-row tile xs.
__device__ __forceinline__ void state_put(uint32_t taddr, uint32_t xs, int t, int gw,
                                          const float (&v)[32]) {
  uint32_t u[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(v[e]);
  tc::tmem_st16(taddr, u);
#pragma unroll
  for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(v[16 + e]);
  tc::tmem_st16(taddr + 16, u);
  tc::tmem_wait_st();
  store_row32<true>(xs, t, gw, v);
}

}  // namespace tct
}  // namespace rapt
