// Dense projection y = x W^T on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a: bf16
// operands, fp32 accumulation, bf16 result. The projections of the layer (08-rapt-algorithm.md §3:
// q = W_q x, k = W_k x, v = W_v x before the features; §4.2: the output projection w_o after the
// division) are plain GEMMs with x [M, K] and W [N, K] both row-major (K contiguous).
//
// One persistent CTA per SM walks 128 x 256 output tiles. Roles (192 threads):
//   warp 0      one thread streams 64-wide K blocks of x (128 x 64) and W (256 x 64) by TMA into a
//               ring of four stages (128-byte swizzle, the layout the tensor core reads);
//   warp 1      allocates 512 TMEM columns (two 256-column fp32 accumulators) and one thread issues
//               four 128 x 256 x 16 MMAs per K block, committing each stage back to the producer
//               and each finished tile to the epilogue;
//   warps 2-5   epilogue, one TMEM lane quarter each (warp w reads lanes 32 (w % 4) ..): 16 columns
//               at a time, rounded to bf16 and stored; the accumulator is handed back so the next
//               tile's MMAs overlap this tile's epilogue.
// The output may be split by columns into `nsplit` tensors of `split_n` columns each (the fused
// q | k | v projection writes three [M, split_n] tensors). Rows past M and columns past N are read
// as zero by TMA and never stored. Every wait is bounded (~1 s); a CTA whose wait gives up sets
// RAPT_DEV_INTERNAL in the optional status word and stops.
#include <cuda.h>

#include <cstring>

#include "kernels.h"
#include "tc_utils.cuh"
#include "tensor_map.h"

namespace rapt {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr long long kWait = 2000000000LL;  // ~1 s of SM cycles
constexpr uint32_t kA = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kB = kBN * kBK * 2;     // 32 KB
constexpr uint32_t kStage = kA + kB;
constexpr uint32_t kBar = kStages * kStage;              // full[S], empty[S], accf[2], acce[2]
constexpr uint32_t kMisc = kBar + (2 * kStages + 4) * 8;  // TMEM base, abort flag
constexpr uint32_t kSmem = kMisc + 16;
static_assert(kSmem <= 232448, "shared memory budget");

struct LinArgs {
  void* out[3];      // nsplit output tensors, each [M, split_n] bf16
  int nsplit;
  int split_n;
  int M, N, K;
  uint32_t* dev_status;
};

__device__ __forceinline__ void st_global16(void* p, const uint4& v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    linear_tc_kernel(const LinArgs a, const __grid_constant__ CUtensorMap tx,
                     const __grid_constant__ CUtensorMap tw) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = (a.M + kBM - 1) / kBM, nt = (a.N + kBN - 1) / kBN;
  const int ntiles = mt * nt;
  const int nk = (a.K + kBK - 1) / kBK;

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = tc::smem_u32(smem);
  const uint32_t bar_full = base + kBar, bar_empty = bar_full + 8 * kStages;
  const uint32_t bar_accf = bar_empty + 8 * kStages, bar_acce = bar_accf + 16;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kMisc);
  int* s_abort = reinterpret_cast<int*>(smem + kMisc + 4);
  const bool misaligned = (base & 1023u) != 0;  // uniform; the swizzled layout needs 1 KB

  if (warp == 1 && !misaligned) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 2 * kBN);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar_full + 8 * s, 1);
      tc::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bar_accf + 8 * b, 1);
      tc::mbar_init(bar_acce + 8 * b, 128);
    }
    tc::mbar_fence_init();
    *s_abort = misaligned ? 1 : 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const bool run = !*s_abort;

  if (warp == 0) {
    if (lane == 0 && run) {  // TMA producer
      long g = 0;
      int ok = 1;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int m0 = (t / nt) * kBM, n0 = (t % nt) * kBN;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = static_cast<int>(g % kStages);
          if (g >= kStages && !tc::mbar_wait(bar_empty + 8 * s, ((g / kStages) - 1) & 1, kWait)) {
            ok = 0;
            break;
          }
          const uint32_t st = base + s * kStage;
          tc::mbar_arrive_expect_tx(bar_full + 8 * s, kStage);
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
              "[%1, {%2, %3}], [%4];" ::"r"(st),
              "l"(reinterpret_cast<uint64_t>(&tx)), "r"(kb * kBK), "r"(m0), "r"(bar_full + 8 * s)
              : "memory");
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
              "[%1, {%2, %3}], [%4];" ::"r"(st + kA),
              "l"(reinterpret_cast<uint64_t>(&tw)), "r"(kb * kBK), "r"(n0), "r"(bar_full + 8 * s)
              : "memory");
        }
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && run) {  // MMA issuer
      constexpr uint32_t ID = tc::idesc_bf16(kBM, kBN, false, false);
      long g = 0;
      int ok = 1, i = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++i) {
        const int buf = i & 1;
        if (i >= 2 && !tc::mbar_wait(bar_acce + 8 * buf, ((i / 2) - 1) & 1, kWait)) {
          ok = 0;
          break;
        }
        tc::fence_after_sync();
        const uint32_t acc = tmem + buf * kBN;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = static_cast<int>(g % kStages);
          if (!tc::mbar_wait(bar_full + 8 * s, (g / kStages) & 1, kWait)) {
            ok = 0;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st = base + s * kStage;
          const uint64_t da = tc::desc_sw128(st, 16, 1024);
          const uint64_t db = tc::desc_sw128(st + kA, 16, 1024);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16(acc, da + 2 * k, db + 2 * k, ID, (kb > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(bar_empty + 8 * s);
        }
        if (ok) tc::mma_commit(bar_accf + 8 * buf);
      }
      if (!ok) atomicExch(s_abort, 1);
    }
  } else if (run) {  // epilogue warps 2-5
    const int quarter = warp & 3;
    const uint32_t tl = static_cast<uint32_t>(32 * quarter) << 16;
    int i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      const int ok = tc::mbar_wait(bar_accf + 8 * buf, (i / 2) & 1, kWait);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicExch(s_abort, 1);
        break;
      }
      tc::fence_after_sync();
      const int m0 = (t / nt) * kBM, n0 = (t % nt) * kBN;
      const int row = m0 + 32 * quarter + lane;
      const uint32_t acc = tmem + buf * kBN + tl;
#pragma unroll 1
      for (int j = 0; j < kBN; j += 16) {
        uint32_t u[16];
        tc::tmem_ld16(acc + j, u);
        tc::tmem_wait_ld();
        const int col = n0 + j;
        if (row < a.M && col < a.N) {
          uint4 lo, hi;
          lo.x = tc::pack_bf16x2(__uint_as_float(u[0]), __uint_as_float(u[1]));
          lo.y = tc::pack_bf16x2(__uint_as_float(u[2]), __uint_as_float(u[3]));
          lo.z = tc::pack_bf16x2(__uint_as_float(u[4]), __uint_as_float(u[5]));
          lo.w = tc::pack_bf16x2(__uint_as_float(u[6]), __uint_as_float(u[7]));
          hi.x = tc::pack_bf16x2(__uint_as_float(u[8]), __uint_as_float(u[9]));
          hi.y = tc::pack_bf16x2(__uint_as_float(u[10]), __uint_as_float(u[11]));
          hi.z = tc::pack_bf16x2(__uint_as_float(u[12]), __uint_as_float(u[13]));
          hi.w = tc::pack_bf16x2(__uint_as_float(u[14]), __uint_as_float(u[15]));
          const int which = col / a.split_n, c = col % a.split_n;
          void* ob = which == 0 ? a.out[0] : (which == 1 ? a.out[1] : a.out[2]);
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(ob) + static_cast<long>(row) * a.split_n + c;
          st_global16(o, lo);
          st_global16(o + 8, hi);
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(bar_acce + 8 * buf);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*s_abort && tid == 0 && a.dev_status != nullptr && !misaligned) atomicOr(a.dev_status, 2u);
  if (misaligned && tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, 2u);
  tc::fence_after_sync();
  if (warp == 1 && !misaligned) tc::tmem_dealloc(tmem, 2 * kBN);
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

}  // namespace

bool linear_shape_ok(int M, int N, int K, int split_n) {
  return M >= 0 && N > 0 && K > 0 && K % 8 == 0 && N % 16 == 0 && split_n > 0 && split_n % 16 == 0 &&
         N % split_n == 0 && N / split_n <= 3;
}

cudaError_t launch_linear_tc(const void* x, const void* w, void* const* outs, int M, int N, int K,
                             int split_n, uint32_t* dev_status, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (!linear_shape_ok(M, N, K, split_n)) return cudaErrorInvalidValue;
  CUtensorMap tx, tw;
  const uint64_t dx[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint64_t dw[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
  const uint64_t st[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t bx[2] = {kBK, kBM}, bw[2] = {kBK, kBN};
  cudaError_t e = encode_bf16_map(&tx, x, 2, dx, st, bx);
  if (e != cudaSuccess) return e;
  e = encode_bf16_map(&tw, w, 2, dw, st, bw);
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0;  // bit per device (idempotent; races are benign)
  if (dev < 64 && !((configured >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    configured |= 1ull << dev;
  }
  LinArgs a{};
  a.nsplit = N / split_n;
  for (int i = 0; i < a.nsplit; ++i) a.out[i] = outs[i];
  a.split_n = split_n;
  a.M = M; a.N = N; a.K = K;
  a.dev_status = dev_status;
  const long tiles = static_cast<long>((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const int grid = static_cast<int>(tiles < num_sms() ? tiles : num_sms());
  linear_tc_kernel<<<grid, kThreads, kSmem, stream>>>(a, tx, tw);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rapt
