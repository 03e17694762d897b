// C ABI of the RLA-2 / RAPT library (declared in include/rapt.h): argument validation, feature
// constants, workspace sizing and kernel dispatch. Nothing here allocates device memory or
// synchronises; every launch goes to the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/rapt.h"
#include "kernels.h"

namespace {

using rapt::DType;

constexpr double kTwoPi = 6.283185307179586476925286766559;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool opt_aligned16(const void* p) { return p == nullptr || aligned16(p); }
bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }
bool supported_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool known_dtype(rapt_dtype t) { return t == RAPT_F32 || t == RAPT_BF16; }
DType to_dt(rapt_dtype t) { return t == RAPT_F32 ? DType::F32 : DType::BF16; }

// Common checks of the feature parameters and gains. Returns RAPT_OK or the error.
rapt_status check_features(const float* gq, const float* gk, const rapt_params& p, int d) {
  if (gq == nullptr || gk == nullptr) return RAPT_ERR_INVALID_ARG;
  if (!aligned16(gq) || !aligned16(gk)) return RAPT_ERR_INVALID_ARG;
  if (!finite_pos(p.eps_norm) || !finite_pos(p.eps_den) || !finite_pos(p.rope_base))
    return RAPT_ERR_INVALID_ARG;
  if (p.gamma_head_stride != 0 && p.gamma_head_stride != d) return RAPT_ERR_INVALID_ARG;
  return RAPT_OK;
}

// RoPE frequencies theta_j = base^(-2j/d) in turns per position, split hi + lo (double on host).
rapt::FeatureArgs make_features(const rapt_params& p, int d) {
  rapt::FeatureArgs fa{};
  fa.eps_norm = p.eps_norm;
  fa.gamma_stride = p.gamma_head_stride;
  for (int j = 0; j < d / 2; ++j) {
    const double f = std::pow(static_cast<double>(p.rope_base), -2.0 * j / d) / kTwoPi;
    const float hi = static_cast<float>(f);
    fa.rope_hi[j] = hi;
    fa.rope_lo[j] = static_cast<float>(f - static_cast<double>(hi));
  }
  return fa;
}

rapt_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RAPT_OK : RAPT_ERR_CUDA; }

bool fits_i32(long long x) { return x >= 0 && x < (1LL << 31); }

std::atomic<unsigned long long> g_launches{0};

}  // namespace

namespace rapt {
void note_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
unsigned long long launch_count() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace rapt

extern "C" {

rapt_params rapt_default_params(void) {
  rapt_params p;
  p.eps_norm = 1e-6f;
  p.rope_base = 10000.f;
  p.eps_den = 1e-4f;
  p.gamma_head_stride = 0;
  return p;
}

const char* rapt_status_string(rapt_status s) {
  switch (s) {
    case RAPT_OK: return "RAPT_OK";
    case RAPT_ERR_INVALID_ARG: return "RAPT_ERR_INVALID_ARG: invalid argument";
    case RAPT_ERR_UNSUPPORTED: return "RAPT_ERR_UNSUPPORTED: unsupported head size or dtype";
    case RAPT_ERR_WORKSPACE: return "RAPT_ERR_WORKSPACE: workspace missing or too small";
    case RAPT_ERR_CUDA: return "RAPT_ERR_CUDA: CUDA launch failed";
    default: return "RAPT: unknown status";
  }
}

int32_t rapt_abi_version(void) { return 10300; }

uint64_t rapt_launch_counter(void) { return rapt::launch_count(); }

size_t rapt_prefill_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || B < 1 || H < 1 || L < 0) return 0;
  if (!rapt::tc_supported(to_dt(dtype), d)) return 0;
  return rapt::tc_plan(B, H, L, static_cast<long>(B) * L, d, false).ws_bytes;
}

rapt_status rapt_prefill_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                             int32_t B, int32_t L, int32_t H, int32_t d,
                             const float* gamma_q, const float* gamma_k, rapt_params params,
                             int32_t pos_offset, const float* S0, const float* z0, void* out,
                             float* S_final, float* z_final, uint32_t* dev_status,
                             void* workspace, size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0 || pos_offset < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(pos_offset) + L)) return RAPT_ERR_INVALID_ARG;
  if (L > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(out) ||
      !opt_aligned16(S0) || !opt_aligned16(z0) || !opt_aligned16(S_final) || !opt_aligned16(z_final))
    return RAPT_ERR_INVALID_ARG;
  if (out != nullptr && (out == q || out == k || out == v)) return RAPT_ERR_INVALID_ARG;
  if ((S_final != nullptr && S_final == S0) || (z_final != nullptr && z_final == z0))
    return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_prefill_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;

  rapt::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.gamma_q = gamma_q; a.gamma_k = gamma_k;
  a.S0 = S0; a.z0 = z0; a.S_final = S_final; a.z_final = z_final;
  a.cu_seqlens = nullptr; a.dev_status = dev_status;
  a.n_docs = B; a.doc_len = L; a.total_rows = B * L; a.max_seqlen = L;
  a.H = H; a.pos_offset = pos_offset; a.eps_den = params.eps_den;
  a.fa = make_features(params, d);
  if (L == 0 && S_final == nullptr && z_final == nullptr) return RAPT_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rapt::tc_supported(to_dt(dtype), d))
    return from_cuda(rapt::launch_prefill_tc(d, a, rapt::tc_plan(B, H, L, static_cast<long>(B) * L, d, false),
                                             static_cast<float*>(workspace), s));
  return from_cuda(rapt::launch_prefill_simt(to_dt(dtype), d, a, s));
}

// ---- host buffers: batch rows pipelined over two copy streams and the compute stream

namespace {
size_t up16(size_t x) { return (x + 15) / 16 * 16; }
// Bytes of one batch row of a [B, L, H, d] tensor.
size_t host_row_bytes(int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  return static_cast<size_t>(L) * H * d * (dtype == RAPT_F32 ? 4 : 2);
}
// The events of one call (created and released by the call).
struct HostEvents {
  cudaEvent_t start = nullptr, in[2] = {nullptr, nullptr}, comp[2] = {nullptr, nullptr},
              out[2] = {nullptr, nullptr};
  cudaError_t create() {
    cudaError_t e = cudaSuccess;
    for (cudaEvent_t* ev : {&start, &in[0], &in[1], &comp[0], &comp[1], &out[0], &out[1]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    return e;
  }
  ~HostEvents() {  // a pending event is released once it completes
    for (cudaEvent_t ev : {start, in[0], in[1], comp[0], comp[1], out[0], out[1]})
      if (ev != nullptr) cudaEventDestroy(ev);
  }
};
}  // namespace

size_t rapt_prefill_host_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d,
                                        rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || B < 1 || H < 1 || L < 0) return 0;
  return 8 * up16(host_row_bytes(L, H, d, dtype)) + up16(rapt_prefill_workspace_size(1, L, H, d, dtype));
}

rapt_status rapt_prefill_fwd_host(const void* q, const void* k, const void* v, rapt_dtype dtype,
                                  int32_t B, int32_t L, int32_t H, int32_t d,
                                  const float* gamma_q, const float* gamma_k, rapt_params params,
                                  int32_t pos_offset, const float* S0, const float* z0, void* out,
                                  float* S_final, float* z_final, uint32_t* dev_status,
                                  void* workspace, size_t workspace_bytes, rapt_stream_t stream,
                                  rapt_stream_t copy_in, rapt_stream_t copy_out) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0 || pos_offset < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(pos_offset) + L)) return RAPT_ERR_INVALID_ARG;
  if (L > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (out != nullptr && (out == q || out == k || out == v)) return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(S0) || !opt_aligned16(z0) || !opt_aligned16(S_final) || !opt_aligned16(z_final))
    return RAPT_ERR_INVALID_ARG;
  if ((S_final != nullptr && S_final == S0) || (z_final != nullptr && z_final == z0))
    return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_prefill_host_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || workspace == nullptr || !aligned16(workspace)) return RAPT_ERR_WORKSPACE;
  if (L == 0)  // nothing to copy: the states only
    return rapt_prefill_fwd(nullptr, nullptr, nullptr, dtype, B, 0, H, d, gamma_q, gamma_k, params,
                            pos_offset, S0, z0, nullptr, S_final, z_final, dev_status, workspace,
                            workspace_bytes, stream);

  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaStream_t si = reinterpret_cast<cudaStream_t>(copy_in);
  const cudaStream_t so = reinterpret_cast<cudaStream_t>(copy_out);
  const size_t row = host_row_bytes(L, H, d, dtype), slot_stride = 4 * up16(row);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* ws_pre = ws + 2 * slot_stride;
  const size_t pre_bytes = workspace_bytes - 2 * slot_stride;
  const long sdd = static_cast<long>(H) * d * d, sd = static_cast<long>(H) * d;
  HostEvents ev;
  bool in_rec[2] = {false, false}, out_rec[2] = {false, false};  // events recorded per slot
  rapt_status fail = RAPT_OK;
  cudaError_t e = ev.create();
  if (e == cudaSuccess) e = cudaEventRecord(ev.start, s);  // after the work already on `stream`
  if (e == cudaSuccess) e = cudaStreamWaitEvent(si, ev.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(so, ev.start, 0);
  for (int32_t b = 0; b < B && e == cudaSuccess; ++b) {
    const int slot = b & 1;
    uint8_t* sl = ws + slot * slot_stride;
    uint8_t *qd = sl, *kd = sl + up16(row), *vd = sl + 2 * up16(row), *od = sl + 3 * up16(row);
    const size_t off = static_cast<size_t>(b) * row;
    // copy in (once the row two back has been computed: it read this slot's inputs)
    if (b >= 2) e = cudaStreamWaitEvent(si, ev.comp[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(qd, static_cast<const uint8_t*>(q) + off, row, cudaMemcpyDefault, si);
    if (e == cudaSuccess) e = cudaMemcpyAsync(kd, static_cast<const uint8_t*>(k) + off, row, cudaMemcpyDefault, si);
    if (e == cudaSuccess) e = cudaMemcpyAsync(vd, static_cast<const uint8_t*>(v) + off, row, cudaMemcpyDefault, si);
    if (e == cudaSuccess) e = cudaEventRecord(ev.in[slot], si);
    if (e == cudaSuccess) in_rec[slot] = true;
    // compute (once the row is in and the row two back has been copied out of this slot)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev.in[slot], 0);
    if (e == cudaSuccess && b >= 2) e = cudaStreamWaitEvent(s, ev.out[slot], 0);
    if (e != cudaSuccess) break;
    st = rapt_prefill_fwd(qd, kd, vd, dtype, 1, L, H, d, gamma_q, gamma_k, params, pos_offset,
                          S0 != nullptr ? S0 + b * sdd : nullptr, z0 != nullptr ? z0 + b * sd : nullptr,
                          od, S_final != nullptr ? S_final + b * sdd : nullptr,
                          z_final != nullptr ? z_final + b * sd : nullptr, dev_status, ws_pre,
                          pre_bytes, stream);
    if (st != RAPT_OK) {
      fail = st;
      break;
    }
    e = cudaEventRecord(ev.comp[slot], s);
    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(so, ev.comp[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + off, od, row, cudaMemcpyDefault, so);
    if (e == cudaSuccess) e = cudaEventRecord(ev.out[slot], so);
    if (e == cudaSuccess) out_rec[slot] = true;
  }
  // `stream` covers everything queued, also when a row failed: it waits for the last copies in
  // and out of both slots, so a caller that synchronises `stream` may then free the buffers
  for (int slot = 0; slot < 2; ++slot) {
    cudaError_t w = cudaSuccess;
    if (in_rec[slot]) w = cudaStreamWaitEvent(s, ev.in[slot], 0);
    if (w == cudaSuccess && out_rec[slot]) w = cudaStreamWaitEvent(s, ev.out[slot], 0);
    if (e == cudaSuccess) e = w;
  }
  if (fail != RAPT_OK) return fail;
  return from_cuda(e);
}

size_t rapt_varlen_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d, int32_t max_seqlen,
                                  rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || N < 1 || H < 1 || max_seqlen < 0 || T < 0) return 0;
  if (!rapt::tc_supported(to_dt(dtype), d)) return 0;
  return rapt::tc_plan(N, H, max_seqlen, T, d, true).ws_bytes;
}

rapt_status rapt_varlen_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                            int32_t T, int32_t H, int32_t d, const int32_t* cu_seqlens,
                            int32_t N, int32_t max_seqlen, const float* gamma_q,
                            const float* gamma_k, rapt_params params, const float* S0,
                            const float* z0, void* out, float* S_final, float* z_final,
                            uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                            rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (T < 0 || N < 1 || H < 1 || max_seqlen < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(T) * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(N) * H * 4)) return RAPT_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  if (T > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(out) ||
      !opt_aligned16(S0) || !opt_aligned16(z0) || !opt_aligned16(S_final) || !opt_aligned16(z_final))
    return RAPT_ERR_INVALID_ARG;
  if (out != nullptr && (out == q || out == k || out == v)) return RAPT_ERR_INVALID_ARG;
  if ((S_final != nullptr && S_final == S0) || (z_final != nullptr && z_final == z0))
    return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_varlen_workspace_size(T, N, H, d, max_seqlen, dtype);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;

  rapt::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.gamma_q = gamma_q; a.gamma_k = gamma_k;
  a.S0 = S0; a.z0 = z0; a.S_final = S_final; a.z_final = z_final;
  a.cu_seqlens = cu_seqlens; a.dev_status = dev_status;
  a.n_docs = N; a.doc_len = 0; a.total_rows = T; a.max_seqlen = max_seqlen;
  a.H = H; a.pos_offset = 0; a.eps_den = params.eps_den;
  a.fa = make_features(params, d);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rapt::tc_supported(to_dt(dtype), d))
    return from_cuda(rapt::launch_prefill_tc(d, a, rapt::tc_plan(N, H, max_seqlen, T, d, true),
                                             static_cast<float*>(workspace), s));
  return from_cuda(rapt::launch_prefill_simt(to_dt(dtype), d, a, s));
}

size_t rapt_bidir_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || B < 1 || H < 1 || L < 0) return 0;
  if (!rapt::tc_supported(to_dt(dtype), d) || L == 0) return 0;  // nothing runs for L = 0
  return rapt::bidir_plan(B, H, L, d).ws_bytes;
}

rapt_status rapt_bidir_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                           int32_t B, int32_t L, int32_t H, int32_t d,
                           const float* gamma_q, const float* gamma_k, rapt_params params,
                           int32_t pos_offset, void* out, uint32_t* dev_status,
                           void* workspace, size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0 || pos_offset < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(pos_offset) + L)) return RAPT_ERR_INVALID_ARG;
  if (L > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(out))
    return RAPT_ERR_INVALID_ARG;
  if (out != nullptr && (out == q || out == k || out == v)) return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_bidir_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;
  if (L == 0) return RAPT_OK;

  rapt::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.gamma_q = gamma_q; a.gamma_k = gamma_k;
  a.cu_seqlens = nullptr; a.dev_status = dev_status;
  a.n_docs = B; a.doc_len = L; a.total_rows = B * L; a.max_seqlen = L;
  a.H = H; a.pos_offset = pos_offset; a.eps_den = params.eps_den; a.bidir = 1;
  a.fa = make_features(params, d);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rapt::tc_supported(to_dt(dtype), d))
    return from_cuda(rapt::launch_bidir_tc(d, a, rapt::bidir_plan(B, H, L, d), workspace, s));
  return from_cuda(rapt::launch_prefill_simt(to_dt(dtype), d, a, s));
}

size_t rapt_bidir_varlen_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d,
                                        int32_t max_seqlen, rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || N < 1 || H < 1 || max_seqlen < 0 || T < 0) return 0;
  if (!rapt::tc_supported(to_dt(dtype), d) || T == 0) return 0;  // nothing runs for T = 0
  return rapt::bidir_plan(N, H, max_seqlen, d).ws_bytes;
}

rapt_status rapt_bidir_varlen_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                                  int32_t T, int32_t H, int32_t d, const int32_t* cu_seqlens,
                                  int32_t N, int32_t max_seqlen, const float* gamma_q,
                                  const float* gamma_k, rapt_params params, void* out,
                                  uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                                  rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (T < 0 || N < 1 || H < 1 || max_seqlen < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(T) * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(N) * H * 4)) return RAPT_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  if (T > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(out))
    return RAPT_ERR_INVALID_ARG;
  if (out != nullptr && (out == q || out == k || out == v)) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_bidir_varlen_workspace_size(T, N, H, d, max_seqlen, dtype);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;
  if (T == 0) return RAPT_OK;

  rapt::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.gamma_q = gamma_q; a.gamma_k = gamma_k;
  a.cu_seqlens = cu_seqlens; a.dev_status = dev_status;
  a.n_docs = N; a.doc_len = 0; a.total_rows = T; a.max_seqlen = max_seqlen;
  a.H = H; a.pos_offset = 0; a.eps_den = params.eps_den; a.bidir = 1;
  a.fa = make_features(params, d);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rapt::tc_supported(to_dt(dtype), d))
    return from_cuda(rapt::launch_bidir_tc(d, a, rapt::bidir_plan(N, H, max_seqlen, d), workspace, s));
  return from_cuda(rapt::launch_prefill_simt(to_dt(dtype), d, a, s));
}

namespace {

// Shared tail of the two backward entry points: checks, workspace carving, launch.
rapt_status backward_common(const void* q, const void* k, const void* v, const void* dout,
                            rapt_dtype dtype, int n_docs, int doc_len, long total_rows, int H,
                            int d, const int32_t* cu_seqlens, int max_seqlen, int pos_offset,
                            const float* gamma_q, const float* gamma_k, const rapt_params& params,
                            void* dq, void* dk, void* dv, float* dgamma_q, float* dgamma_k,
                            uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                            size_t need, rapt_stream_t stream) {
  if (total_rows > 0 && (q == nullptr || k == nullptr || v == nullptr || dout == nullptr ||
                         dq == nullptr || dk == nullptr || dv == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(dout) ||
      !opt_aligned16(dq) || !opt_aligned16(dk) || !opt_aligned16(dv) ||
      !opt_aligned16(dgamma_q) || !opt_aligned16(dgamma_k))
    return RAPT_ERR_INVALID_ARG;
  const void* ins[4] = {q, k, v, dout};
  const void* outs[5] = {dq, dk, dv, dgamma_q, dgamma_k};
  for (const void* o : outs) {
    if (o == nullptr) continue;
    for (const void* i : ins)
      if (o == i) return RAPT_ERR_INVALID_ARG;
  }
  if ((dq != nullptr && (dq == dk || dq == dv)) || (dk != nullptr && dk == dv) ||
      (dgamma_q != nullptr && dgamma_q == dgamma_k))
    return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int n_gain = params.gamma_head_stride != 0 ? H * d : d;
  if (total_rows == 0) {  // no token: the gain gradients are zero
    if (dgamma_q != nullptr &&
        cudaMemsetAsync(dgamma_q, 0, sizeof(float) * n_gain, s) != cudaSuccess)
      return RAPT_ERR_CUDA;
    if (dgamma_k != nullptr &&
        cudaMemsetAsync(dgamma_k, 0, sizeof(float) * n_gain, s) != cudaSuccess)
      return RAPT_ERR_CUDA;
    return RAPT_OK;
  }
  const bool tc = rapt::bwd_tc_supported(to_dt(dtype), d);
  const rapt::BwdPlan plan = rapt::bwd_plan(n_docs, H, max_seqlen, total_rows, d, tc);
  rapt::BwdArgs b{};
  rapt::PrefillArgs& a = b.p;
  a.q = q; a.k = k; a.v = v; a.out = nullptr;
  a.gamma_q = gamma_q; a.gamma_k = gamma_k;
  a.cu_seqlens = cu_seqlens; a.dev_status = dev_status;
  a.n_docs = n_docs; a.doc_len = doc_len; a.total_rows = static_cast<int>(total_rows);
  a.max_seqlen = max_seqlen; a.H = H; a.pos_offset = pos_offset; a.eps_den = params.eps_den;
  a.fa = make_features(params, d);
  b.dout = dout; b.dq = dq; b.dk = dk; b.dv = dv;
  b.dgamma_q = dgamma_q; b.dgamma_k = dgamma_k;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  b.rec_fwd = reinterpret_cast<float*>(w);
  b.rec_rev = reinterpret_cast<float*>(w + plan.off_rev);
  b.den = reinterpret_cast<float*>(w + plan.off_den);
  b.scl = reinterpret_cast<float*>(w + plan.off_scl);
  b.sst = reinterpret_cast<float*>(w + plan.off_sst);
  b.nst = reinterpret_cast<float*>(w + plan.off_nst);
  b.dgp_q = reinterpret_cast<float*>(w + plan.off_dgq);
  b.dgp_k = reinterpret_cast<float*>(w + plan.off_dgk);
  b.nseg = plan.nseg;
  b.seg_len = plan.seg_len;
  b.qf = w + plan.off_qf;
  b.kf = w + plan.off_kf;
  b.blk_per_seg = plan.blk_per_seg;
  b.rblk_per_seg = plan.rblk_per_seg;
  b.nblk_max = plan.nblk_max;
  b.dqf = w + plan.off_dqf;
  b.dkf = w + plan.off_dkf;
  b.chunks_max = plan.chunks_max;
  b.d = d;
  b.order = (tc && cu_seqlens != nullptr && n_docs > 1) ? reinterpret_cast<int*>(w + plan.off_order) : nullptr;
  if (tc) return from_cuda(rapt::launch_backward_tc(b, s));
  return from_cuda(rapt::launch_backward_simt(to_dt(dtype), d, b, s));
}

}  // namespace

size_t rapt_prefill_bwd_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d,
                                       rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || B < 1 || H < 1 || L < 1) return 0;
  return rapt::bwd_plan(B, H, L, static_cast<long>(B) * L, d,
                        rapt::bwd_tc_supported(to_dt(dtype), d)).ws_bytes;
}

rapt_status rapt_prefill_bwd(const void* q, const void* k, const void* v, const void* dout,
                             rapt_dtype dtype, int32_t B, int32_t L, int32_t H, int32_t d,
                             const float* gamma_q, const float* gamma_k, rapt_params params,
                             int32_t pos_offset, void* dq, void* dk, void* dv, float* dgamma_q,
                             float* dgamma_k, void* workspace, size_t workspace_bytes,
                             rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0 || pos_offset < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(pos_offset) + L)) return RAPT_ERR_INVALID_ARG;
  return backward_common(q, k, v, dout, dtype, B, L, static_cast<long>(B) * L, H, d, nullptr, L,
                         pos_offset, gamma_q, gamma_k, params, dq, dk, dv, dgamma_q, dgamma_k,
                         nullptr, workspace, workspace_bytes,
                         rapt_prefill_bwd_workspace_size(B, L, H, d, dtype), stream);
}

size_t rapt_varlen_bwd_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d,
                                      int32_t max_seqlen, rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || N < 1 || H < 1 || max_seqlen < 0 || T < 1)
    return 0;
  return rapt::bwd_plan(N, H, max_seqlen, T, d, rapt::bwd_tc_supported(to_dt(dtype), d)).ws_bytes;
}

rapt_status rapt_varlen_bwd(const void* q, const void* k, const void* v, const void* dout,
                            rapt_dtype dtype, int32_t T, int32_t H, int32_t d,
                            const int32_t* cu_seqlens, int32_t N, int32_t max_seqlen,
                            const float* gamma_q, const float* gamma_k, rapt_params params,
                            void* dq, void* dk, void* dv, float* dgamma_q, float* dgamma_k,
                            uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                            rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (T < 0 || N < 1 || H < 1 || max_seqlen < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(T) * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(N) * H * 4)) return RAPT_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return RAPT_ERR_INVALID_ARG;
  return backward_common(q, k, v, dout, dtype, N, 0, T, H, d, cu_seqlens, max_seqlen, 0, gamma_q,
                         gamma_k, params, dq, dk, dv, dgamma_q, dgamma_k, dev_status, workspace,
                         workspace_bytes,
                         rapt_varlen_bwd_workspace_size(T, N, H, d, max_seqlen, dtype), stream);
}

namespace {

rapt_status l2_causal_common(const void* q, const void* k, const void* v, rapt_dtype dtype,
                             int n_docs, int doc_len, long total_rows, int H, int d,
                             const int32_t* cu_seqlens, int max_seqlen, float eps, void* out,
                             uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                             size_t need, rapt_stream_t stream) {
  if (!std::isfinite(eps) || eps <= 0.f) return RAPT_ERR_INVALID_ARG;
  if (total_rows > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(out))
    return RAPT_ERR_INVALID_ARG;
  if (out != nullptr && (out == q || out == k || out == v)) return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;
  if (total_rows == 0) return RAPT_OK;
  if (rapt::l2c_tc_supported(to_dt(dtype), d)) {
    rapt::L2cTcArgs a{};
    a.q = q; a.k = k; a.v = v; a.out = out;
    a.cu_seqlens = cu_seqlens; a.dev_status = dev_status;
    a.n_docs = n_docs; a.doc_len = doc_len; a.total_rows = static_cast<int>(total_rows);
    a.max_seqlen = max_seqlen; a.H = H; a.eps = eps;
    if (cu_seqlens == nullptr) {
      const rapt::L2cPlan plan = rapt::l2c_tc_plan(n_docs, doc_len, H, d);
      a.nseg = plan.nseg;
      a.seg_len = plan.seg_len;
    } else {
      a.nseg = 1;
      a.seg_len = max_seqlen > 0 ? (max_seqlen + 127) / 128 * 128 : 128;
    }
    return from_cuda(rapt::launch_l2_causal_tc(d, a, workspace, reinterpret_cast<cudaStream_t>(stream)));
  }
  const rapt::L2cPlan plan = rapt::l2c_plan(n_docs, H, max_seqlen, d);
  rapt::L2cArgs b{};
  rapt::PrefillArgs& a = b.p;
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.cu_seqlens = cu_seqlens; a.dev_status = dev_status;
  a.n_docs = n_docs; a.doc_len = doc_len; a.total_rows = static_cast<int>(total_rows);
  a.max_seqlen = max_seqlen; a.H = H;
  b.eps = eps;
  b.rec = static_cast<float*>(workspace);
  b.nseg = plan.nseg;
  b.seg_len = plan.seg_len;
  return from_cuda(rapt::launch_l2_causal_simt(to_dt(dtype), d, b,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

size_t rla_l2_causal_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || B < 1 || H < 1 || L < 1) return 0;
  if (rapt::l2c_tc_supported(to_dt(dtype), d)) return rapt::l2c_tc_plan(B, L, H, d).ws_bytes;
  return rapt::l2c_plan(B, H, L, d).ws_bytes;
}

rapt_status rla_l2_causal_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                              int32_t B, int32_t L, int32_t H, int32_t d, float eps, void* out,
                              void* workspace, size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  return l2_causal_common(q, k, v, dtype, B, L, static_cast<long>(B) * L, H, d, nullptr, L, eps,
                          out, nullptr, workspace, workspace_bytes,
                          rla_l2_causal_workspace_size(B, L, H, d, dtype), stream);
}

size_t rla_l2_causal_varlen_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d,
                                           int32_t max_seqlen, rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || N < 1 || H < 1 || max_seqlen < 0 || T < 1)
    return 0;
  if (rapt::l2c_tc_supported(to_dt(dtype), d)) return rapt::l2c_tc_varlen_ws_bytes(N);
  return rapt::l2c_plan(N, H, max_seqlen, d).ws_bytes;
}

rapt_status rla_l2_causal_varlen_fwd(const void* q, const void* k, const void* v,
                                     rapt_dtype dtype, int32_t T, int32_t H, int32_t d,
                                     const int32_t* cu_seqlens, int32_t N, int32_t max_seqlen,
                                     float eps, void* out, uint32_t* dev_status, void* workspace,
                                     size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (T < 0 || N < 1 || H < 1 || max_seqlen < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(T) * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(N) * H * 4)) return RAPT_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return RAPT_ERR_INVALID_ARG;
  return l2_causal_common(q, k, v, dtype, N, 0, T, H, d, cu_seqlens, max_seqlen, eps, out,
                          dev_status, workspace, workspace_bytes,
                          rla_l2_causal_varlen_workspace_size(T, N, H, d, max_seqlen, dtype),
                          stream);
}

rapt_status rapt_linear_fwd(const void* x, const void* w, void* y, int32_t M, int32_t N,
                            int32_t K, uint32_t* dev_status, rapt_stream_t stream) {
  if (M < 0 || N < 1 || K < 1) return RAPT_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 16 != 0) return RAPT_ERR_UNSUPPORTED;
  if (!fits_i32(static_cast<long long>(M) * K) || !fits_i32(static_cast<long long>(N) * K) ||
      !fits_i32(static_cast<long long>(M) * N))
    return RAPT_ERR_INVALID_ARG;
  if (M > 0 && (x == nullptr || w == nullptr || y == nullptr)) return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(x) || !opt_aligned16(w) || !opt_aligned16(y)) return RAPT_ERR_INVALID_ARG;
  if (y != nullptr && (y == x || y == w)) return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  void* outs[1] = {y};
  return from_cuda(rapt::launch_linear_tc(x, w, outs, M, N, K, N, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

size_t rapt_layer_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, int32_t d_model) {
  if (!supported_d(d) || B < 1 || H < 1 || L < 0 || d_model < 1) return 0;
  const size_t act = up256(static_cast<size_t>(B) * L * H * d * 2);
  return 4 * act + rapt_prefill_workspace_size(B, L, H, d, RAPT_BF16);
}

rapt_status rapt_layer_fwd(const void* x, const void* w_qkv, const void* w_o, int32_t B,
                           int32_t L, int32_t H, int32_t d, int32_t d_model,
                           const float* gamma_q, const float* gamma_k, rapt_params params,
                           int32_t pos_offset, void* y, uint32_t* dev_status, void* workspace,
                           size_t workspace_bytes, rapt_stream_t stream) {
  if (!supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0 || d_model < 1 || pos_offset < 0) return RAPT_ERR_INVALID_ARG;
  if (d_model % 16 != 0) return RAPT_ERR_UNSUPPORTED;
  const long long T = static_cast<long long>(B) * L;
  if (!fits_i32(T * d_model) || !fits_i32(T * 3 * H * d) ||
      !fits_i32(static_cast<long long>(3) * H * d * d_model) ||
      !fits_i32(static_cast<long long>(pos_offset) + L))
    return RAPT_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || w_qkv == nullptr || w_o == nullptr || y == nullptr))
    return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(x) || !opt_aligned16(w_qkv) || !opt_aligned16(w_o) || !opt_aligned16(y))
    return RAPT_ERR_INVALID_ARG;
  if (y != nullptr && (y == x || y == w_qkv || y == w_o)) return RAPT_ERR_INVALID_ARG;
  if (dev_status != nullptr && !aligned4(dev_status)) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_layer_workspace_size(B, L, H, d, d_model);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
    return RAPT_ERR_WORKSPACE;
  if (T == 0) return RAPT_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wb = static_cast<uint8_t*>(workspace);
  const size_t act = up256(static_cast<size_t>(T) * H * d * 2);
  void* q = wb;
  void* k = wb + act;
  void* v = wb + 2 * act;
  void* attn = wb + 3 * act;
  void* pws = wb + 4 * act;
  // q | k | v = x W_qkv^T, split into three [T, H, d] tensors
  void* qkv[3] = {q, k, v};
  cudaError_t e = rapt::launch_linear_tc(x, w_qkv, qkv, static_cast<int>(T), 3 * H * d, d_model,
                                         H * d, dev_status, s);
  if (e != cudaSuccess) return RAPT_ERR_CUDA;
  st = rapt_prefill_fwd(q, k, v, RAPT_BF16, B, L, H, d, gamma_q, gamma_k, params, pos_offset,
                        nullptr, nullptr, attn, nullptr, nullptr, dev_status, pws,
                        workspace_bytes - 4 * act, stream);
  if (st != RAPT_OK) return st;
  // y = attn W_o^T
  void* outs[1] = {y};
  e = rapt::launch_linear_tc(attn, w_o, outs, static_cast<int>(T), d_model, H * d, d_model,
                             dev_status, s);
  return from_cuda(e);
}

rapt_status rapt_decode_step(const void* q, const void* k, const void* v, rapt_dtype dtype,
                             int32_t N, int32_t H, int32_t d, const int32_t* positions,
                             const float* gamma_q, const float* gamma_k, rapt_params params,
                             float* S, float* z, void* out, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (N < 1 || H < 1) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(N) * H * d * d)) return RAPT_ERR_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || positions == nullptr ||
      S == nullptr || z == nullptr)
    return RAPT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(S) ||
      !aligned16(z) || !aligned4(positions))
    return RAPT_ERR_INVALID_ARG;
  if (out == q || out == k || out == v) return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_q, gamma_k, params, d);
  if (st != RAPT_OK) return st;

  rapt::DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.out = out; a.positions = positions;
  a.gamma_q = gamma_q; a.gamma_k = gamma_k; a.S = S; a.z = z;
  a.N = N; a.H = H; a.eps_den = params.eps_den;
  a.fa = make_features(params, d);
  return from_cuda(rapt::launch_decode(to_dt(dtype), d, a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t rla_l2_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  if (B < 1 || L < 0 || H < 1 || !supported_d(d) || !known_dtype(dtype)) return 0;
  if (rapt::l2_tc_supported(to_dt(dtype), d)) return rapt::l2_tc_workspace_bytes(B, L, H, d);
  return rapt::l2_workspace_bytes(B, L, H, d);
}

rapt_status rla_l2_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                       int32_t B, int32_t L, int32_t H, int32_t d, float eps, void* out,
                       void* workspace, size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!finite_pos(eps)) return RAPT_ERR_INVALID_ARG;
  if (L == 0) return RAPT_OK;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return RAPT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RAPT_ERR_INVALID_ARG;
  if (out == q || out == k || out == v) return RAPT_ERR_INVALID_ARG;
  const size_t need = rla_l2_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || (need > 0 && workspace == nullptr) || !aligned16(workspace))
    return RAPT_ERR_WORKSPACE;

  rapt::L2Args a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.ws = static_cast<float*>(workspace);
  a.B = B; a.L = L; a.H = H; a.eps = eps;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (rapt::l2_tc_supported(to_dt(dtype), d)) return from_cuda(rapt::launch_rla_l2_tc(d, a, st));
  return from_cuda(rapt::launch_rla_l2(to_dt(dtype), d, a, st));
}

// ---- one sequence split across GPUs: shard state, start state, and the L2 path in two halves

size_t rapt_prefill_state_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d,
                                         rapt_dtype dtype) {
  if (!known_dtype(dtype) || !supported_d(d) || B < 1 || H < 1 || L < 0) return 0;
  return rapt::shard_state_plan(to_dt(dtype), B, L, H, d).ws_bytes;
}

rapt_status rapt_prefill_state(const void* k, const void* v, rapt_dtype dtype, int32_t B,
                               int32_t L, int32_t H, int32_t d, const float* gamma_k,
                               rapt_params params, int32_t pos_offset, float* S_inc, float* z_inc,
                               void* workspace, size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0 || pos_offset < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(pos_offset) + L)) return RAPT_ERR_INVALID_ARG;
  if (S_inc == nullptr || z_inc == nullptr || !aligned16(S_inc) || !aligned16(z_inc))
    return RAPT_ERR_INVALID_ARG;
  if (L > 0 && (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)))
    return RAPT_ERR_INVALID_ARG;
  rapt_status st = check_features(gamma_k, gamma_k, params, d);
  if (st != RAPT_OK) return st;
  const size_t need = rapt_prefill_state_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || workspace == nullptr || !aligned16(workspace))
    return RAPT_ERR_WORKSPACE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long n_bh = static_cast<long>(B) * H;
  if (L == 0) {  // an empty shard adds nothing: zero increments
    cudaError_t e = rapt::launch_state_prefix(nullptr, n_bh * d * d, 0, nullptr, S_inc, s);
    if (e == cudaSuccess) e = rapt::launch_state_prefix(nullptr, n_bh * d, 0, nullptr, z_inc, s);
    return from_cuda(e);
  }
  rapt::PrefillArgs a{};
  a.k = k; a.v = v;
  a.gamma_q = gamma_k; a.gamma_k = gamma_k;
  a.n_docs = B; a.doc_len = L; a.total_rows = B * L; a.max_seqlen = L;
  a.H = H; a.pos_offset = pos_offset; a.eps_den = params.eps_den;
  a.fa = make_features(params, d);
  const rapt::ShardPlan plan = rapt::shard_state_plan(to_dt(dtype), B, L, H, d);
  return from_cuda(rapt::launch_shard_state(to_dt(dtype), d, a, plan,
                                            static_cast<float*>(workspace), S_inc, z_inc, s));
}

rapt_status rapt_state_prefix(const float* S_parts, const float* z_parts, int32_t W, int32_t r,
                              int32_t B, int32_t H, int32_t d, const float* S0, const float* z0,
                              float* S_start, float* z_start, rapt_stream_t stream) {
  if (!supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || W < 1 || r < 0 || r > W) return RAPT_ERR_INVALID_ARG;
  if (S_start == nullptr || z_start == nullptr || !aligned16(S_start) || !aligned16(z_start))
    return RAPT_ERR_INVALID_ARG;
  if (r > 0 && (S_parts == nullptr || z_parts == nullptr)) return RAPT_ERR_INVALID_ARG;
  if (!opt_aligned16(S_parts) || !opt_aligned16(z_parts) || !opt_aligned16(S0) || !opt_aligned16(z0))
    return RAPT_ERR_INVALID_ARG;
  if (S_start == S_parts || z_start == z_parts) return RAPT_ERR_INVALID_ARG;
  const long n_bh = static_cast<long>(B) * H;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = rapt::launch_state_prefix(S_parts, n_bh * d * d, r, S0, S_start, s);
  if (e == cudaSuccess) e = rapt::launch_state_prefix(z_parts, n_bh * d, r, z0, z_start, s);
  return from_cuda(e);
}

size_t rla_l2_moments_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  if (B < 1 || L < 0 || H < 1 || !supported_d(d) || !known_dtype(dtype)) return 0;
  if (rapt::l2_tc_supported(to_dt(dtype), d)) return rapt::l2_tc_moments_ws_bytes(B, L, H, d);
  return rapt::l2_moments_ws_bytes(B, L, H, d);
}

rapt_status rla_l2_moments(const void* k, const void* v, rapt_dtype dtype, int32_t B, int32_t L,
                           int32_t H, int32_t d, float* M, void* workspace, size_t workspace_bytes,
                           rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (M == nullptr || !aligned16(M)) return RAPT_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long n_mat = static_cast<long>(B) * H * d * 2 * d;
  if (L == 0) return from_cuda(rapt::launch_state_prefix(nullptr, n_mat, 0, nullptr, M, s));
  if (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)) return RAPT_ERR_INVALID_ARG;
  const size_t need = rla_l2_moments_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || workspace == nullptr || !aligned16(workspace))
    return RAPT_ERR_WORKSPACE;
  rapt::L2Args a{};
  a.k = k; a.v = v;
  a.ws = static_cast<float*>(workspace);
  a.B = B; a.L = L; a.H = H; a.eps = 1.f;
  if (rapt::l2_tc_supported(to_dt(dtype), d)) return from_cuda(rapt::launch_l2_tc_moments_plain(d, a, M, s));
  return from_cuda(rapt::launch_l2_moments_plain(to_dt(dtype), d, a, M, s));
}

size_t rla_l2_readout_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype) {
  if (B < 1 || L < 0 || H < 1 || !supported_d(d) || !known_dtype(dtype)) return 0;
  if (rapt::l2_tc_supported(to_dt(dtype), d)) return rapt::l2_tc_readout_ws_bytes(B, H, d);
  return 0;
}

rapt_status rla_l2_readout(const void* q, const float* M, rapt_dtype dtype, int32_t B, int32_t L,
                           int32_t H, int32_t d, float eps, void* out, void* workspace,
                           size_t workspace_bytes, rapt_stream_t stream) {
  if (!known_dtype(dtype) || !supported_d(d)) return RAPT_ERR_UNSUPPORTED;
  if (B < 1 || H < 1 || L < 0) return RAPT_ERR_INVALID_ARG;
  if (!fits_i32(static_cast<long long>(B) * L * H * d)) return RAPT_ERR_INVALID_ARG;
  if (!finite_pos(eps)) return RAPT_ERR_INVALID_ARG;
  if (L == 0) return RAPT_OK;
  if (q == nullptr || M == nullptr || out == nullptr) return RAPT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(M) || !aligned16(out) || out == q) return RAPT_ERR_INVALID_ARG;
  const size_t need = rla_l2_readout_workspace_size(B, L, H, d, dtype);
  if (workspace_bytes < need || (need > 0 && workspace == nullptr) || !opt_aligned16(workspace))
    return RAPT_ERR_WORKSPACE;
  rapt::L2Args a{};
  a.q = q; a.out = out;
  a.ws = static_cast<float*>(workspace);
  a.B = B; a.L = L; a.H = H; a.eps = eps;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rapt::l2_tc_supported(to_dt(dtype), d)) return from_cuda(rapt::launch_l2_tc_readout_plain(d, a, M, s));
  return from_cuda(rapt::launch_l2_readout_plain(to_dt(dtype), d, a, M, s));
}

}  // extern "C"
