/*
 * rapt.h — C ABI of the GB300 (sm_103a) RLA-2 / RAPT causal ReLU linear attention library.
 *
 * The method (neuralnet.cpp page "线性注意力家族：RLA / RAPT / RLA-2 与 GPU 落地",
 * docs/development/08-rapt-algorithm.md):
 *   features (§1, §3, §4.2):  q' = ReLU(RoPE(RMSNorm(q))),  k' = ReLU(RoPE(RMSNorm(k))),  v untouched;
 *                              RMSNorm per (token, head) over d, no 1/sqrt(d) scale.
 *   state    (§3):             S_t = S_{t-1} + k'_t (x) v_t  (d x d),  z_t = z_{t-1} + k'_t,
 *                              reset at every document boundary (§2.2, §4.1).
 *   output   (§3):             out_t = q'_t S_t / (q'_t . z_t + eps_den),  eps_den = 1e-4.
 *   original RLA (§2.1):       out_t = sum_i s_ti v_i / (sqrt(sum_i s_ti^2) + 1e-6), non-causal,
 *                              s_ti = ReLU(q_t) . ReLU(k_i), no norm, no RoPE.
 *   decode (§4.2 forward_step): features of the new token, update the state first, then read out.
 *
 * RMSNorm:  x_hat = x * (mean_d(x^2) + eps_norm)^(-1/2) * gamma  (gamma fp32, statistics fp32;
 *           ruDNN README §7).  RoPE: adjacent pairs (2j, 2j+1) rotated by p * base^(-2j/d),
 *           (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a); p = 0-based position of the
 *           token inside its document (plus pos_offset for dense prefill).
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers (caller-owned; the library never frees or keeps them), except
 *     where a parameter says "host". Tensors are dense, contiguous, row-major in the layout named,
 *     and 16-byte aligned.
 *   - Layouts: dense "BSND" [B, L, H, d]; packed varlen "TND" [T, H, d]; decode [N, H, d].
 *     States are fp32 and key-major: S[..., i, j] = sum_t k'_t[i] v_t[j]  ([.., H, d, d]); z [.., H, d].
 *   - Output dtype = input dtype (bf16 results are rounded to nearest even).
 *   - Precision. fp32 inputs (and bf16 at d = 16 or 32): all arithmetic and all accumulation are
 *     fp32. bf16 inputs at d = 64 or 128: the products of the chunked form run on the tensor cores
 *     with bf16 operands and fp32 accumulation: q', k' and the masked in-chunk scores are rounded
 *     to bf16, and the state enters the inter-chunk product as a bf16 copy; the state itself, z,
 *     RMSNorm, RoPE and the Sum denominator stay fp32. The L2 readout (rla_l2_fwd) uses bf16 copies
 *     of its fp32 moments. Decode is fp32 throughout.
 *   - Inputs must be finite. Tiles are read whole, so a non-finite value anywhere in q, k or v
 *     may make any output of the same call non-finite.
 *   - d must be one of 16, 32, 64, 128 (d_v = d_k = d).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream), allocates no
 *     device memory and never synchronises. Every call but the tensor-core backward launches only
 *     on `stream`; the backward (bf16, d = 64 or 128) forks part of its work onto a stream of
 *     greater priority that it makes once per thread and device (with three events; remade after a
 *     device reset) and joins it back to `stream` before it returns, so work queued on `stream`
 *     after the call waits for all of it.
 *   - Host-checkable errors are returned before anything is launched and nothing is written:
 *     RAPT_ERR_INVALID_ARG (null required pointer, size <= 0 where > 0 is required, eps not
 *     finite or <= 0, misalignment, `out` aliasing an input), RAPT_ERR_UNSUPPORTED (d or dtype not
 *     supported), RAPT_ERR_WORKSPACE (workspace pointer null or smaller than the size query).
 *     RAPT_ERR_CUDA reports a failed launch (cudaGetLastError after the launch); the kernels may
 *     then not have run.
 *   - Optional outputs are skipped when their pointer is NULL; optional inputs count as zero.
 *   - Initial states are read only, never written (ruDNN README §8: the initial state is not
 *     overwritten in place). S_final / z_final may not alias S0 / z0.
 */
#ifndef RAPT_H
#define RAPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the CUDA runtime's stream handle); NULL = the legacy default stream. */
typedef struct CUstream_st* rapt_stream_t;

typedef enum rapt_status {
  RAPT_OK = 0,
  RAPT_ERR_INVALID_ARG = 1,
  RAPT_ERR_UNSUPPORTED = 2,
  RAPT_ERR_WORKSPACE = 3,
  RAPT_ERR_CUDA = 4
} rapt_status;

typedef enum rapt_dtype { RAPT_F32 = 0, RAPT_BF16 = 1 } rapt_dtype;

/* Device error word bits, OR-ed into a caller's `dev_status` word when one is given. */
#define RAPT_DEV_BAD_CU_SEQLENS 1u /* cu_seqlens not non-decreasing from 0 to T: bad documents skipped */
#define RAPT_DEV_INTERNAL 2u       /* a tensor-core wait gave up or smem was misaligned (never expected): outputs invalid */

/* Feature / denominator settings (08-rapt-algorithm.md §1, §3). */
typedef struct rapt_params {
  float eps_norm;            /* RMSNorm epsilon, inside the root; finite, > 0 (1e-6)             */
  float rope_base;           /* RoPE base; finite, > 1 (10000)                                    */
  float eps_den;             /* Sum-denominator epsilon; finite, > 0 (1e-4)                       */
  int32_t gamma_head_stride; /* 0: gamma_q / gamma_k are [d], shared by all heads;
                                d: they are [H, d] (a separate gain vector per head)             */
} rapt_params;

/* Defaults of the pages: eps_norm 1e-6, rope_base 1e4, eps_den 1e-4, shared gamma. */
rapt_params rapt_default_params(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char* rapt_status_string(rapt_status status);

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
int32_t rapt_abi_version(void);

/* Number of CUDA kernel launches this library has enqueued since it was loaded (all devices,
 * all threads; a relaxed atomic counter). Instrumentation only: lets a caller count the kernels
 * of a timed region by differencing two reads. */
uint64_t rapt_launch_counter(void);

/*
 * Dense causal RLA-2 prefill (08-rapt-algorithm.md §3, §4.2 forward).
 *   q, k, v   [B, L, H, d] of `dtype`; every batch row is one document.
 *   gamma_q, gamma_k  fp32 [d] or [H, d] (see rapt_params.gamma_head_stride).
 *   pos_offset        RoPE position of token 0 of every batch row (>= 0); token t sits at
 *                     pos_offset + t (for continuing a sequence whose state is in S0/z0).
 *   S0, z0    nullable fp32 [B, H, d, d], [B, H, d]: state carried in (NULL = zeros).
 *   out       [B, L, H, d] of `dtype`; must not alias q, k or v.
 *   S_final, z_final  nullable fp32 [B, H, d, d], [B, H, d]: state after token L-1.
 *   dev_status  nullable DEVICE uint32: RAPT_DEV_* bits are OR-ed in on a device-side error
 *               (the caller zeroes it; the library only sets bits).
 *   workspace / workspace_bytes: device scratch of at least rapt_prefill_workspace_size()
 *                     bytes, 16-byte aligned (may be NULL when that size is 0). Contents on
 *                     entry do not matter.
 * Requirements: B, H >= 1, L >= 0 (L = 0 only writes S_final/z_final), B*L*H*d < 2^31.
 * bf16 with d = 64 or 128 runs on the tensor cores (tcgen05); fp32, and bf16 with d = 16 or 32,
 * run on CUDA cores.
 */
size_t rapt_prefill_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rapt_prefill_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                             int32_t B, int32_t L, int32_t H, int32_t d,
                             const float* gamma_q, const float* gamma_k, rapt_params params,
                             int32_t pos_offset, const float* S0, const float* z0, void* out,
                             float* S_final, float* z_final, uint32_t* dev_status,
                             void* workspace, size_t workspace_bytes, rapt_stream_t stream);

/*
 * rapt_prefill_fwd with q, k, v and out in HOST memory (page-locked for full speed; any memory
 * the CUDA runtime can copy from works). The batch rows are pipelined: row b is copied in on
 * `copy_in` while row b - 1 is computed on `stream` and row b - 2 is copied out on `copy_out`, so
 * the host -> device copies, the device -> host copies and the kernels overlap. Each row is
 * computed by rapt_prefill_fwd with B = 1, so the result is that of rapt_prefill_fwd on each
 * batch row alone (the same values a B-row call gives up to the segment split of the plan).
 *   q, k, v   host [B, L, H, d] of `dtype`; out host [B, L, H, d] of `dtype`.
 *   gamma_q, gamma_k, S0, z0, S_final, z_final, dev_status: DEVICE pointers, as for
 *             rapt_prefill_fwd (S0 / z0 / S_final / z_final are [B, H, d, d] / [B, H, d]).
 *   workspace / workspace_bytes: device scratch of at least rapt_prefill_host_workspace_size()
 *             bytes, 16-byte aligned: two staging slots of a row's q, k, v and out, then the
 *             B = 1 prefill workspace. Contents on entry do not matter.
 *   stream, copy_in, copy_out: the compute stream and the two copy streams (they may be the
 *             same stream; then nothing overlaps). All three first wait for the work already
 *             queued on `stream`, and `stream` waits for the last copy out before the call
 *             returns, so synchronising `stream` makes out and the states complete. The call
 *             creates and releases its own CUDA events and allocates no memory.
 * Errors: as rapt_prefill_fwd (checked before anything is queued), RAPT_ERR_WORKSPACE, and
 * RAPT_ERR_CUDA if queuing a copy, an event or a kernel fails (work queued before the failure
 * stays queued).
 */
size_t rapt_prefill_host_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d,
                                        rapt_dtype dtype);
rapt_status rapt_prefill_fwd_host(const void* q, const void* k, const void* v, rapt_dtype dtype,
                                  int32_t B, int32_t L, int32_t H, int32_t d,
                                  const float* gamma_q, const float* gamma_k, rapt_params params,
                                  int32_t pos_offset, const float* S0, const float* z0, void* out,
                                  float* S_final, float* z_final, uint32_t* dev_status,
                                  void* workspace, size_t workspace_bytes, rapt_stream_t stream,
                                  rapt_stream_t copy_in, rapt_stream_t copy_out);

/*
 * Packed variable-length causal RLA-2 (08-rapt-algorithm.md §2.2, §4.1: the state restarts at
 * every document; RoPE positions restart at 0 in every document).
 *   q, k, v   [T, H, d] of `dtype`.
 *   cu_seqlens  DEVICE int32 [N + 1]: 0 = cu[0] <= cu[1] <= ... <= cu[N] = T; document n is
 *               tokens cu[n] .. cu[n+1]-1 (empty documents allowed).
 *   max_seqlen  host int: an upper bound on every document length (used to size the launch);
 *               a document longer than max_seqlen is an error reported through dev_status.
 *   S0, z0    nullable fp32 [N, H, d, d], [N, H, d]: per-document carried-in state.
 *   out       [T, H, d]; S_final, z_final nullable fp32 [N, H, d, d], [N, H, d] (an empty
 *             document's final state is its initial state).
 *   dev_status  nullable DEVICE uint32: bits RAPT_DEV_* are OR-ed in when cu_seqlens is
 *             malformed (the offending documents are skipped, never read out of bounds). The
 *             caller zeroes it; the library only sets bits.
 *   workspace   at least rapt_varlen_workspace_size(T, N, H, d, max_seqlen, dtype) bytes.
 * Requirements: T >= 0, N >= 1, H >= 1, T*H*d < 2^31.
 */
size_t rapt_varlen_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d, int32_t max_seqlen,
                                  rapt_dtype dtype);
rapt_status rapt_varlen_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                            int32_t T, int32_t H, int32_t d, const int32_t* cu_seqlens,
                            int32_t N, int32_t max_seqlen, const float* gamma_q,
                            const float* gamma_k, rapt_params params, const float* S0,
                            const float* z0, void* out, float* S_final, float* z_final,
                            uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                            rapt_stream_t stream);

/*
 * Backward of the causal forward (08-rapt-algorithm.md §4.2 "backward": one prefix scan and two
 * suffix scans, then back through ReLU, RoPE and RMSNorm). For an upstream gradient dout = dL/dout
 * it returns dL/dq, dL/dk, dL/dv and the gain gradients. With gnum_t = dout_t / den_t and
 * scale_t = -(dout_t . num_t) / den_t^2 (num_t, den_t the forward's numerator and denominator):
 *   dq'_t = S_t gnum_t + scale_t z_t,
 *   dk'_tau = sum_{t >= tau} q'_t (gnum_t . v_tau + scale_t),   dv_tau = sum_{t >= tau} s_{t,tau} gnum_t,
 * then dq, dk through the feature map (the gradient passes the ReLU where its input is > 0; RoPE
 * is undone by the inverse rotation; RMSNorm: dx = r gamma dy - x r^3 (sum gamma dy x) / d).
 * Sums run inside each document (the state restarts at document boundaries).
 *   q, k, v, dout  as the forward's inputs (same dtype and layout); dout is dL/dout.
 *   gamma_q, gamma_k, params, pos_offset: as for the forward call being differentiated.
 *   dq, dk, dv     outputs of the inputs' dtype and layout; none may alias an input or another.
 *   dgamma_q, dgamma_k  nullable fp32 outputs shaped like the gains ([d] when shared, summed over
 *                  every token and head; [H, d] when per head): written, not accumulated.
 *   workspace      at least the matching *_bwd_workspace_size() bytes, 16-byte aligned (state
 *                  increments of the segments the documents are cut into, den and scale of every
 *                  (token, head), and partial gain sums).
 *   dev_status     (varlen) as for rapt_varlen_fwd: malformed documents are skipped and their
 *                  gradients are not written.
 * The forward has no carried-in state here (S0 = z0 = 0: documents start fresh). The computation
 * is recomputed from q, k, v (no activations of the forward are kept). bf16 at d = 64 or 128 runs
 * the chunk products on the tensor cores (bf16 operands: q', k', dout, dout / den, the masked
 * scores and their gradient, the states' bf16 copies; fp32 accumulation, states, denominators and
 * feature backward); everything else is fp32 on the CUDA cores. bf16 outputs are rounded to
 * nearest even. Every sum has a fixed order: repeated calls give bitwise-identical results.
 */
size_t rapt_prefill_bwd_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rapt_prefill_bwd(const void* q, const void* k, const void* v, const void* dout,
                             rapt_dtype dtype, int32_t B, int32_t L, int32_t H, int32_t d,
                             const float* gamma_q, const float* gamma_k, rapt_params params,
                             int32_t pos_offset, void* dq, void* dk, void* dv, float* dgamma_q,
                             float* dgamma_k, void* workspace, size_t workspace_bytes,
                             rapt_stream_t stream);
size_t rapt_varlen_bwd_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d,
                                      int32_t max_seqlen, rapt_dtype dtype);
rapt_status rapt_varlen_bwd(const void* q, const void* k, const void* v, const void* dout,
                            rapt_dtype dtype, int32_t T, int32_t H, int32_t d,
                            const int32_t* cu_seqlens, int32_t N, int32_t max_seqlen,
                            const float* gamma_q, const float* gamma_k, rapt_params params,
                            void* dq, void* dk, void* dv, float* dgamma_q, float* dgamma_k,
                            uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                            rapt_stream_t stream);

/*
 * Causal original RLA with the L2 denominator (08-rapt-algorithm.md §2.1 closed form, eps outside
 * the root; §2.2 a query reads the accumulated causal state, which restarts at document
 * boundaries; §4.1 the prefix scan's A_t = sum k'k'^T state):
 *   q' = ReLU(q), k' = ReLU(k) (no norm, no RoPE),
 *   out_t = sum_{i<=t} s_ti v_i / (sqrt(sum_{i<=t} s_ti^2) + eps) = q'_t S_t / (sqrt(q'_t^T A_t q'_t) + eps).
 *   Dense:  q, k, v, out [B, L, H, d]; one document per batch row.
 *   Varlen: q, k, v, out [T, H, d]; cu_seqlens, N, max_seqlen and dev_status as for rapt_varlen_fwd.
 *   eps       finite, > 0 (1e-6 on the page).
 *   workspace at least the matching *_workspace_size() bytes, 16-byte aligned (the states K'^T V and
 *             K'^T K' of the segments the documents are cut into; may be NULL when that size is 0).
 * Dense bf16 with d = 128 runs on the tensor cores (bf16 operands, fp32 accumulation and states;
 * the products with the states use bf16 copies of them; the sum of squared scores is fp32 from the
 * exact bf16 features). Everything else (fp32, other d, varlen) is fp32 on CUDA cores. bf16
 * outputs are rounded to nearest even. Results are bitwise repeatable (fixed summation order).
 */
size_t rla_l2_causal_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rla_l2_causal_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                              int32_t B, int32_t L, int32_t H, int32_t d, float eps, void* out,
                              void* workspace, size_t workspace_bytes, rapt_stream_t stream);
size_t rla_l2_causal_varlen_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d,
                                           int32_t max_seqlen, rapt_dtype dtype);
rapt_status rla_l2_causal_varlen_fwd(const void* q, const void* k, const void* v,
                                     rapt_dtype dtype, int32_t T, int32_t H, int32_t d,
                                     const int32_t* cu_seqlens, int32_t N, int32_t max_seqlen,
                                     float eps, void* out, uint32_t* dev_status, void* workspace,
                                     size_t workspace_bytes, rapt_stream_t stream);

/*
 * Projection y = x W^T (the layer's linear maps: q = W_q x, k = W_k x, v = W_v x before the
 * features, 08-rapt-algorithm.md §3; the output projection w_o after the division, §4.2).
 *   x  [M, K] bf16, W [N, K] bf16 (row-major, K contiguous: a linear layer's weight), y [M, N] bf16.
 * Tensor cores (tcgen05), bf16 operands, fp32 accumulation, result rounded to nearest even.
 * Requirements: M >= 0, K % 8 == 0, N % 16 == 0; y must not alias x or W. dev_status (nullable,
 * DEVICE uint32) gets RAPT_DEV_INTERNAL if a tensor-core wait gave up (never expected).
 */
rapt_status rapt_linear_fwd(const void* x, const void* w, void* y, int32_t M, int32_t N,
                            int32_t K, uint32_t* dev_status, rapt_stream_t stream);

/*
 * One RAPT attention layer (08-rapt-algorithm.md §3, §4.2 forward): projections, the causal RLA-2
 * attention of rapt_prefill_fwd, output projection:
 *   [q | k | v] = x W_qkv^T   (x [B, L, d_model] bf16; W_qkv [3 H d, d_model] bf16 whose rows are
 *                              W_q, then W_k, then W_v, each H d rows in head-major order h d + j),
 *   a = RLA-2(q, k, v) per head ([B, L, H, d], features and denominator as for rapt_prefill_fwd,
 *       one document per batch row, RoPE position pos_offset + t),
 *   y = a W_o^T               (W_o [d_model, H d] bf16, y [B, L, d_model] bf16).
 * q, k, v and a are bf16 tensors in the workspace (rapt_layer_workspace_size() bytes, 16-byte
 * aligned): four [B, L, H, d] activations, then the attention's own workspace. The projections run
 * on the tensor cores; the attention as rapt_prefill_fwd with dtype bf16.
 * Requirements: d in {16, 32, 64, 128}, d_model % 16 == 0; y must not alias an input.
 */
size_t rapt_layer_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, int32_t d_model);
rapt_status rapt_layer_fwd(const void* x, const void* w_qkv, const void* w_o, int32_t B,
                           int32_t L, int32_t H, int32_t d, int32_t d_model,
                           const float* gamma_q, const float* gamma_k, rapt_params params,
                           int32_t pos_offset, void* y, uint32_t* dev_status, void* workspace,
                           size_t workspace_bytes, rapt_stream_t stream);

/*
 * Bidirectional (non-causal) RLA-2 (08-rapt-algorithm.md §4.1: in its causal=false mode the prefix
 * scan sums over the whole set; §4.2: the layer's bidirectional branch; formula and eps of §3).
 * Features as in the causal form; for each (document, head), S = sum_tau k'_tau v_tau^T and
 * z = sum_tau k'_tau over the WHOLE document, and out_t = q'_t S / (q'_t . z + eps_den).
 *   Dense:  q, k, v, out [B, L, H, d]; one document per batch row; token t at RoPE position
 *           pos_offset + t.
 *   Varlen: q, k, v, out [T, H, d]; cu_seqlens and max_seqlen as for rapt_varlen_fwd; RoPE
 *           positions restart at 0 in every document, and a document sees only its own tokens.
 *   dev_status  nullable DEVICE uint32, as for rapt_prefill_fwd / rapt_varlen_fwd.
 *   workspace   at least the matching *_workspace_size() bytes, 16-byte aligned (the fp32
 *               state K'^T V and sum k' of every block of every (document, head)).
 * There is no carried-in or final state: the state is the document's own.
 * Requirements as for the causal entry points. bf16 with d = 64 or 128 runs on the tensor cores
 * (bf16 GEMM operands, fp32 accumulation, fp32 denominator); fp32, and bf16 with d = 16 or 32,
 * run on CUDA cores in fp32 and need no workspace.
 */
size_t rapt_bidir_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rapt_bidir_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                           int32_t B, int32_t L, int32_t H, int32_t d,
                           const float* gamma_q, const float* gamma_k, rapt_params params,
                           int32_t pos_offset, void* out, uint32_t* dev_status,
                           void* workspace, size_t workspace_bytes, rapt_stream_t stream);
size_t rapt_bidir_varlen_workspace_size(int32_t T, int32_t N, int32_t H, int32_t d,
                                        int32_t max_seqlen, rapt_dtype dtype);
rapt_status rapt_bidir_varlen_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                                  int32_t T, int32_t H, int32_t d, const int32_t* cu_seqlens,
                                  int32_t N, int32_t max_seqlen, const float* gamma_q,
                                  const float* gamma_k, rapt_params params, void* out,
                                  uint32_t* dev_status, void* workspace, size_t workspace_bytes,
                                  rapt_stream_t stream);

/*
 * One decode step for N sequences (08-rapt-algorithm.md §4.2 forward_step): features of the new
 * token at positions[n]; S += k' v^T and z += k' IN PLACE; out = q' S / (q' . z + eps_den)
 * with the updated state (the new token sees itself, like the inclusive prefill).
 *   q, k, v    [N, H, d] of `dtype`.
 *   positions  DEVICE int32 [N], >= 0: RoPE position of each sequence's new token.
 *   S, z       fp32 [N, H, d, d], [N, H, d], read and updated in place.
 *   out        [N, H, d] of `dtype`.
 */
rapt_status rapt_decode_step(const void* q, const void* k, const void* v, rapt_dtype dtype,
                             int32_t N, int32_t H, int32_t d, const int32_t* positions,
                             const float* gamma_q, const float* gamma_k, rapt_params params,
                             float* S, float* z, void* out, rapt_stream_t stream);

/*
 * Original RLA, non-causal, L2 denominator (08-rapt-algorithm.md §2.1):
 *   q' = ReLU(q), k' = ReLU(k) (no norm, no RoPE); M_V = K'^T V, M_K = K'^T K' over all L tokens
 *   of each (batch row, head); out_t = q'_t M_V / (sqrt(q'_t^T M_K q'_t) + eps).
 *   q, k, v, out  [B, L, H, d] of `dtype`; eps finite, > 0 (1e-6).
 *   workspace     at least rla_l2_workspace_size() bytes (fp32 partial moments of the token
 *                 splits; on the tensor-core path also their sum as the bf16 readout operand).
 * bf16 with d = 64 or 128 runs on the tensor cores (tcgen05): [M_V | M_K] = K'^T [V | K'] and
 * q'[M_V | M_K] are GEMMs with bf16 operands and fp32 accumulation. fp32, and bf16 with d = 16 or
 * 32, run on CUDA cores in fp32.
 */
size_t rla_l2_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rla_l2_fwd(const void* q, const void* k, const void* v, rapt_dtype dtype,
                       int32_t B, int32_t L, int32_t H, int32_t d, float eps, void* out,
                       void* workspace, size_t workspace_bytes, rapt_stream_t stream);

/*
 * One sequence split across GPUs. The RLA-2 state is a sum over tokens (08-rapt-algorithm.md §3:
 * S_t = sum_{i<=t} k'_i v_i^T, z_t = sum_{i<=t} k'_i), which the page notes can be accumulated
 * chunk by chunk in parallel (§1, §3). A sequence cut into W consecutive shards of L tokens, shard
 * r on GPU r, is computed exactly as one sequence by:
 *   1. rapt_prefill_state on every shard: its increment (dS_r, dz_r) over its own tokens;
 *   2. an all-gather of the W increments (by the caller, e.g. NCCL; W * B * H * d * (d + 1) fp32);
 *   3. rapt_state_prefix: shard r's initial state S0 + dS_0 + ... + dS_{r-1} (rank order);
 *   4. rapt_prefill_fwd on shard r with that initial state and pos_offset = the global position of
 *      its first token (RoPE positions continue across shards).
 * The whole sequence's final state is rapt_state_prefix with r = W.
 *
 * rapt_prefill_state: S_inc[b, h] = sum_t k'_t v_t^T and z_inc[b, h] = sum_t k'_t over the L
 * tokens of batch row b (token t at RoPE position pos_offset + t); k' as in rapt_prefill_fwd
 * (gamma_k, params.eps_norm, params.rope_base, params.gamma_head_stride; eps_den unused).
 *   k, v          [B, L, H, d] of `dtype` (may be null when L == 0: the increments are zero).
 *   S_inc, z_inc  fp32 [B, H, d, d], [B, H, d] (written; key-major like every state).
 *   workspace     rapt_prefill_state_workspace_size() bytes (the per-block partial sums).
 * Precision: bf16 at d = 64 or 128 runs on the tensor cores (bf16 k' and v operands, fp32
 * accumulation, as the prefill's own state); otherwise fp32 arithmetic. Bitwise repeatable.
 */
size_t rapt_prefill_state_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d,
                                         rapt_dtype dtype);
rapt_status rapt_prefill_state(const void* k, const void* v, rapt_dtype dtype, int32_t B,
                               int32_t L, int32_t H, int32_t d, const float* gamma_k,
                               rapt_params params, int32_t pos_offset, float* S_inc, float* z_inc,
                               void* workspace, size_t workspace_bytes, rapt_stream_t stream);
/*
 * rapt_state_prefix: S_start = S0 + S_parts[0] + ... + S_parts[r-1] and the same for z, added in
 * rank order (fp32; deterministic).
 *   S_parts, z_parts  fp32 [W, B, H, d, d], [W, B, H, d]: the gathered shard increments (may be
 *                     null when r == 0).
 *   r                 0 <= r <= W: the number of leading shards to add.
 *   S0, z0            nullable fp32 [B, H, d, d], [B, H, d]: the state before shard 0.
 *   S_start, z_start  fp32 [B, H, d, d], [B, H, d] (written; must not alias the parts).
 */
rapt_status rapt_state_prefix(const float* S_parts, const float* z_parts, int32_t W, int32_t r,
                              int32_t B, int32_t H, int32_t d, const float* S0, const float* z0,
                              float* S_start, float* z_start, rapt_stream_t stream);

/*
 * The original RLA L2 path (rla_l2_fwd) in two halves, for a sequence whose L tokens are split
 * across GPUs: the moments M_V = K'^T V and M_K = K'^T K' are sums over tokens (08-rapt-algorithm.md
 * §2.1, §2.2), so each GPU computes its shard's moments with rla_l2_moments, the caller sums them
 * over the GPUs (an all-reduce of B * H * d * 2d fp32), and each GPU reads out its own queries with
 * rla_l2_readout. On one GPU, moments then readout equals rla_l2_fwd.
 *   rla_l2_moments:  M fp32 [B, H, d, 2d] (written): row i holds (M_V[i, 0..d), M_K[i, 0..d));
 *                    k' = ReLU(k). Workspace rla_l2_moments_workspace_size() (split partials).
 *                    L == 0 gives zero moments.
 *   rla_l2_readout:  out_t = q'_t M_V / (sqrt(q'_t^T M_K q'_t) + eps), q' = ReLU(q), for the L
 *                    queries of q [B, L, H, d] and the moments M [B, H, d, 2d] (read only).
 *                    Workspace rla_l2_readout_workspace_size() (bf16 at d = 64 or 128: the bf16
 *                    copy of M the tensor cores read; 0 otherwise).
 * Precision as rla_l2_fwd: fp32 moments; the tensor-core readout reads bf16 copies of them.
 */
size_t rla_l2_moments_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rla_l2_moments(const void* k, const void* v, rapt_dtype dtype, int32_t B, int32_t L,
                           int32_t H, int32_t d, float* M, void* workspace, size_t workspace_bytes,
                           rapt_stream_t stream);
size_t rla_l2_readout_workspace_size(int32_t B, int32_t L, int32_t H, int32_t d, rapt_dtype dtype);
rapt_status rla_l2_readout(const void* q, const float* M, rapt_dtype dtype, int32_t B, int32_t L,
                           int32_t H, int32_t d, float eps, void* out, void* workspace,
                           size_t workspace_bytes, rapt_stream_t stream);

/*
 * Allocation-free variant of rla_l2_fwd. The pages have no counterpart to this entry point: it
 * exists for callers that cannot allocate device memory at all, such as a plugin inside an
 * inference engine that owns every byte of device memory and hands the plugin only its input
 * and output buffers, or a latency-critical loop that must not call cudaMalloc (which can
 * synchronise the device) or grow a memory pool.
 *
 * Same arguments and result as rla_l2_fwd, minus the workspace: the fp32 partial moments live in
 * a fixed device array of RAPT_L2_NOALLOC_SCRATCH_BYTES compiled into the library (every GPU that
 * loads the library holds it until the process exits). The number of token splits is reduced
 * until the moments fit. It always runs the CUDA-core path with fp32 moments: for fp32 inputs and
 * bf16 at d = 16 or 32 its results equal rla_l2_fwd's up to fp32 summation order; for bf16 at
 * d = 64 or 128 (where rla_l2_fwd uses the tensor cores and bf16 copies of the moments) both stay
 * within the bf16 tolerance of the exact result.
 *   - Returns RAPT_ERR_WORKSPACE, before launching anything, when even one split does not fit:
 *     B * H * 2 * d * 2d * 4 bytes must not exceed RAPT_L2_NOALLOC_SCRATCH_BYTES (at d = 128,
 *     B * H <= 64).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress), so an address never outlives its context (after cudaDeviceReset the
 *     module is loaded again and the array may move). The first call on a device also loads the
 *     library's kernels there; make that first call before any stream capture.
 *   - Every call on a device uses the same array. Calls whose kernels overlap on the GPU (for
 *     example on two streams without ordering between them) race on it and give wrong results;
 *     serialise them. Nothing has to be cleared between calls: every element of the array that a
 *     call reads was written earlier in the same call.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define RAPT_L2_NOALLOC_SCRATCH_BYTES (16u << 20)
rapt_status rla_l2_fwd_noalloc(const void* q, const void* k, const void* v, rapt_dtype dtype,
                               int32_t B, int32_t L, int32_t H, int32_t d, float eps, void* out,
                               rapt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RAPT_H */
