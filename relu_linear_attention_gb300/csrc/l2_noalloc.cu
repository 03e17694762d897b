// rla_l2_fwd_noalloc: the original-RLA L2-denominator forward without any device allocation.
//
// Some callers cannot allocate device memory: a plugin of an inference engine that owns all
// device memory and passes the plugin only its inputs and outputs, or a latency-critical loop
// that must never call cudaMalloc (it can synchronise the device). For them the fp32 partial
// moments of the L2 kernels live in a fixed array compiled into the library, instead of a
// caller-provided workspace. The split count over tokens is lowered until the moments fit.
#include "../../include/rapt.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchFloats = RAPT_L2_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Scratch for the partial and reduced moments. Host code must not use this name as a pointer:
// on the host it is only a stand-in for the symbol, whose device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_l2_scratch[kScratchFloats];

// Device address of g_l2_scratch in the current device's context. It is looked up on every call
// (a lookup allocates nothing): a cached address would go stale once the context is destroyed and
// created again (cudaDeviceReset), because the module is then loaded anew and may move. The first
// call on a device loads the module (lazy loading), so make it before any stream capture.
rapt_status scratch_on_current_device(float** ptr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_l2_scratch) != cudaSuccess || p == nullptr) return RAPT_ERR_CUDA;
  *ptr = static_cast<float*>(p);
  return RAPT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" rapt_status rla_l2_fwd_noalloc(const void* q, const void* k, const void* v,
                                          rapt_dtype dtype, int32_t B, int32_t L, int32_t H,
                                          int32_t d, float eps, void* out, rapt_stream_t stream) {
  if (dtype != RAPT_F32 && dtype != RAPT_BF16) return RAPT_ERR_UNSUPPORTED;
  if (d != 16 && d != 32 && d != 64 && d != 128) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0) return RAPT_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * L * H * d >= (1LL << 31)) return RAPT_ERR_INVALID_ARG;
  if (!(eps > 0.f) || eps > 3.0e38f) return RAPT_ERR_INVALID_ARG;
  if (L == 0) return RAPT_OK;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return RAPT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RAPT_ERR_INVALID_ARG;
  if (out == q || out == k || out == v) return RAPT_ERR_INVALID_ARG;

  // Largest split count (at most the one rla_l2_fwd uses) whose moments fit the scratch array.
  int nsplit = rapt::l2_default_splits(B, L, H);
  while (nsplit > 1 &&
         rapt::l2_workspace_bytes_for_splits(B, H, d, nsplit) > RAPT_L2_NOALLOC_SCRATCH_BYTES)
    --nsplit;
  if (rapt::l2_workspace_bytes_for_splits(B, H, d, nsplit) > RAPT_L2_NOALLOC_SCRATCH_BYTES)
    return RAPT_ERR_WORKSPACE;

  float* scratch = nullptr;
  const rapt_status st = scratch_on_current_device(&scratch);
  if (st != RAPT_OK) return st;

  rapt::L2Args a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.ws = scratch;
  a.B = B; a.L = L; a.H = H; a.eps = eps;
  const rapt::DType dt = dtype == RAPT_F32 ? rapt::DType::F32 : rapt::DType::BF16;
  const cudaError_t e =
      rapt::launch_rla_l2_with_splits(dt, d, a, nsplit, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RAPT_OK : RAPT_ERR_CUDA;
}
