// Internal launch interface between the C ABI (api.cu) and the kernel translation units.
// Host-side only; no torch types. Every launcher enqueues on `stream` and returns the
// cudaError_t of the launch (cudaGetLastError right after it).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace rapt {

enum class DType { F32 = 0, BF16 = 1 };

// Counts every kernel launch the library enqueues (read by rapt_launch_counter()).
void note_launches(unsigned n);
unsigned long long launch_count();

// One causal RLA-2 forward over a set of documents. Dense prefill is the special case of
// `n_docs` = B documents of `doc_len` = L tokens each (cu_seqlens == nullptr); varlen reads the
// document bounds from the device array cu_seqlens[n_docs + 1].
struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const float* gamma_q;
  const float* gamma_k;
  const float* S0;  // [n_docs, H, d, d] or null
  const float* z0;  // [n_docs, H, d] or null
  float* S_final;   // [n_docs, H, d, d] or null
  float* z_final;   // [n_docs, H, d] or null
  const int32_t* cu_seqlens;  // null for dense
  uint32_t* dev_status;       // null or device error word
  int n_docs;
  int doc_len;     // dense: tokens per document
  int total_rows;  // dense: B * L; varlen: T
  int max_seqlen;  // varlen: bound on any document length (dense: L)
  int H;
  int pos_offset;  // dense only (0 for varlen)
  float eps_den;
  int bidir;       // 0: causal; 1: bidirectional (every token sees its whole document; no S0 / z0)
  FeatureArgs fa;
};

cudaError_t launch_prefill_simt(DType dt, int d, const PrefillArgs& a, cudaStream_t stream);

// Backward of the causal forward (CUDA cores, fp32 arithmetic) over a set of documents described
// by `p` (p.out, S0/z0 and S_final/z_final unused): gradients of sum dout . out. Documents are cut
// into nseg segments of seg_len tokens; the workspace holds, at the offsets below, the prefix-state
// increments of the segments (from 0), their suffix-state increments, den and scale of every
// (token, head), and the per-(document, head, segment) gain partials of q and k.
struct BwdArgs {
  PrefillArgs p;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* dgamma_q;  // nullable
  float* dgamma_k;  // nullable
  float* rec_fwd;
  float* rec_rev;
  float* den;  // per (token, head): den_t, scale_t, sst_t, nst_t (see backward_simt.cu)
  float* scl;
  float* sst;
  float* nst;
  float* dgp_q;
  float* dgp_k;
  int nseg;
  int seg_len;
  // tensor-core path: the suffix-state increments (rec_rev) are per block of seg_len / rblk_per_seg
  // tokens, rblk_per_seg blocks per segment, nseg * rblk_per_seg records per (document, head)
  int rblk_per_seg;
  // tensor-core path: q', k' of every (token, head) in bf16 (written by pass A, read by pass B),
  // and the prefix-state increments in the prefill state kernel's record format (rec_fwd), in
  // blocks of seg_len / blk_per_seg tokens, nblk_max per (document, head)
  void* qf;
  void* kf;
  int blk_per_seg;
  int nblk_max;
  // tensor-core path: dq', dk' in bf16 (written by the passes, turned into dq, dk by the feature
  // kernel, whose gain partials are per (document, head, 128-token chunk): chunks_max per pair)
  void* dqf;
  void* dkf;
  int chunks_max;
  int d;  // head size of q, k, v and the gradients
  // tensor-core path, packed documents: the passes' CTA slots take the documents in order of
  // decreasing length (order[rank] = document, written by the doc-order kernel); nullable
  int* order;
};
struct BwdPlan {
  int nseg;
  int seg_len;
  int blk_per_seg;   // tensor-core path
  int rblk_per_seg;  // tensor-core path: suffix-state blocks per segment
  int nblk_max;      // tensor-core path
  int chunks_max;   // tensor-core path: 128-token chunks of the longest document
  size_t off_rev, off_den, off_scl, off_sst, off_nst, off_dgq, off_dgk, off_qf, off_kf, off_dqf,
      off_dkf, off_order;
  size_t ws_bytes;
};
// tc: the tensor-core path (128-token chunks; the workspace also holds its block-state records,
// q', k', dq', dk' and the document order).
BwdPlan bwd_plan(int n_docs, int H, int max_seqlen, long total_rows, int d, bool tc);
cudaError_t launch_backward_simt(DType dt, int d, const BwdArgs& b, cudaStream_t stream);
// The gain gradients from the per-(document, head, segment) partials (launched by both paths).
cudaError_t launch_bwd_gain(const BwdArgs& b, int d, cudaStream_t stream);
// Tensor-core backward (bf16, d = 64 or 128): the feature map, two passes, the feature backward,
// then the gains.
bool bwd_tc_supported(DType dt, int d);
cudaError_t launch_backward_tc(const BwdArgs& b, cudaStream_t stream);

// Causal original RLA (L2 denominator) on CUDA cores over the documents of `p` (features ReLU(q),
// ReLU(k); gammas, RoPE, states and eps_den unused). rec: the workspace, 2 d^2 floats (K'^T V, then
// K'^T K') per (document, head, segment).
struct L2cArgs {
  PrefillArgs p;
  float eps;
  float* rec;
  int nseg;
  int seg_len;
};
struct L2cPlan {
  int nseg;
  int seg_len;
  size_t ws_bytes;
};
L2cPlan l2c_plan(int n_docs, int H, int max_seqlen, int d);
cudaError_t launch_l2_causal_simt(DType dt, int d, const L2cArgs& b, cudaStream_t stream);

// y = x W^T on the tensor cores (bf16 in and out, fp32 accumulation): x [M, K], W [N, K] row-major.
// The N output columns are split into N / split_n (<= 3) tensors outs[i] of [M, split_n].
// Shapes: K % 8 == 0, N % 16 == 0, split_n % 16 == 0 and divides N. dev_status (nullable) gets
// RAPT_DEV_INTERNAL if a wait gave up.
bool linear_shape_ok(int M, int N, int K, int split_n);
cudaError_t launch_linear_tc(const void* x, const void* w, void* const* outs, int M, int N, int K,
                             int split_n, uint32_t* dev_status, cudaStream_t stream);

// Tensor-core (tcgen05) chunked prefill for bf16 and d in {64, 128}. Documents are cut into
// nseg_max segments of seg_len tokens; the state increments of every segment but a document's
// last are computed first, in blocks of seg_len / blk_per_seg tokens, and ws_bytes of workspace
// hold them.
// With sort_docs (varlen, one segment per document), the workspace ends with an int32 order of
// the documents by decreasing length at order_off, so that the longest (document, head) units
// are dispatched first. With pair (d = 64, even H), the prefill kernel takes the heads two at a
// time, as the 128-column tiles of the [rows, H / 2, 128] view.
struct TcPlan {
  int nseg_max;
  int seg_len;
  int blk_per_seg;
  size_t ws_bytes;
  bool sort_docs;
  size_t order_off;
  bool pair;
};
bool tc_supported(DType dt, int d);
TcPlan tc_plan(int n_docs, int H, int max_seqlen, long total_tokens, int d, bool varlen);
cudaError_t launch_prefill_tc(int d, const PrefillArgs& a, const TcPlan& plan, float* ws,
                              cudaStream_t stream);

// Arguments of the tensor-core state and prefill kernels.
struct TcArgs {
  PrefillArgs p;
  float* ws;        // increment records [n_docs][H][nblk_max] (K'^T V, then sum k'; D * (D + 1) floats)
  int seg_len;      // tokens per segment (multiple of blk_len)
  int nseg_max;     // segments per document slot in the grid of the prefill kernel
  int blk_len;      // tokens per increment block (multiple of 128)
  int blk_per_seg;  // seg_len / blk_len
  int nblk_max;     // increment blocks per document slot
  int whole_doc;    // 0: the blocks before each document's last segment, all full;
                    // 1: every block of the document, the last one possibly ragged
  const int* order; // nullable: prefill CTA slot -> document (longest first)
};
// The state increments of TcArgs' blocks (one launch; later launches may depend on it
// programmatically: it triggers its dependents at its start).
cudaError_t launch_state_tc(int d, const TcArgs& ta, cudaStream_t stream);

// Bidirectional (non-causal) RLA-2 over a set of documents on the tensor cores (bf16, d in
// {64, 128}): out_t = q'_t S_doc / (q'_t . z_doc + eps) with S_doc, z_doc over the whole document.
// Two launches; ws_bytes of workspace (the fp32 state records of the blocks).
struct BidirPlan {
  int blk_len;       // tokens per state block
  int nblk_max;      // state blocks per document slot
  int nsplit;        // readout CTAs per (document, head)
  int split_chunks;  // 128-token tiles per readout CTA
  size_t ws_bytes;
};
BidirPlan bidir_plan(int n_docs, int H, int max_seqlen, int d);
cudaError_t launch_bidir_tc(int d, const PrefillArgs& a, const BidirPlan& plan, void* ws,
                            cudaStream_t stream);

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const int32_t* positions;
  const float* gamma_q;
  const float* gamma_k;
  float* S;
  float* z;
  int N;
  int H;
  float eps_den;
  FeatureArgs fa;
};

cudaError_t launch_decode(DType dt, int d, const DecodeArgs& a, cudaStream_t stream);

struct L2Args {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* ws;  // partial moments, then the reduced moments
  int B;
  int L;
  int H;
  float eps;
};

size_t l2_workspace_bytes(int B, int L, int H, int d);
// The moments [K'^T V | K'^T K'] of every (batch row, head, split of split_len tokens) into a.ws as
// fp32 partials (bf16, d = 128; float4 (i, 4c .. 4c+3) of a split at index c * d + i, 2d columns).
// (d in {64, 128}; the moments kernel reads k and v of a.B rows of a.L tokens.)
cudaError_t launch_l2_moments_tc(int d, const L2Args& a, int nsplit, int split_len, cudaStream_t stream);
// Causal L2 on the tensor cores (bf16, d in {64, 128}), dense batch rows (doc_len tokens each,
// cu_seqlens null) or packed documents (cu_seqlens[n_docs + 1] on the device). Dense rows are cut
// into nseg segments of seg_len tokens that start from the moments of the splits before them
// (written by launch_l2_moments_tc into the workspace: l2c_tc_plan().ws_bytes); packed documents
// run one segment each (nseg = 1, seg_len >= max_seqlen), the longest first (their document order,
// l2c_tc_varlen_ws_bytes(n_docs) bytes, is the workspace).
struct L2cTcArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const float* ws;
  const int32_t* cu_seqlens;
  const int* order;
  uint32_t* dev_status;
  int n_docs;
  int doc_len;
  int total_rows;
  int max_seqlen;
  int H;
  float eps;
  int nseg;
  int seg_len;
};
bool l2c_tc_supported(DType dt, int d);
L2cPlan l2c_tc_plan(int B, int L, int H, int d);
size_t l2c_tc_varlen_ws_bytes(int n_docs);
cudaError_t launch_l2_causal_tc(int d, L2cTcArgs a, void* ws, cudaStream_t stream);
// The documents of cu_seqlens in order of decreasing length (ties by index) into order[n_docs]
// (n_docs <= 1024), one small launch.
cudaError_t launch_doc_order(const int32_t* cu_seqlens, int n_docs, int total_rows, int* order,
                             cudaStream_t stream);
cudaError_t launch_rla_l2(DType dt, int d, const L2Args& a, cudaStream_t stream);

// Split count launch_rla_l2 would choose, and the launch with an explicit split count
// (workspace of l2_workspace_bytes_for_splits() bytes at a.ws).
// Tensor-core L2 path (bf16, d in {64, 128}): three launches, workspace of
// l2_tc_workspace_bytes() bytes at a.ws (fp32 split partials, then the bf16 moment operands).
bool l2_tc_supported(DType dt, int d);
size_t l2_tc_workspace_bytes(int B, int L, int H, int d);
cudaError_t launch_rla_l2_tc(int d, const L2Args& a, cudaStream_t stream);

// The L2 path in two halves, for a sequence whose tokens are split across GPUs (the moments
// are sums over tokens, so the shards' moments add up): the moments [M_V | M_K] as plain fp32
// (row i, column j at i * 2d + j, per (batch row, head)), and the readout from such moments.
// CUDA-core path: moments workspace l2_moments_ws_bytes(), readout none.
size_t l2_moments_ws_bytes(int B, int L, int H, int d);
cudaError_t launch_l2_moments_plain(DType dt, int d, const L2Args& a, float* M, cudaStream_t stream);
cudaError_t launch_l2_readout_plain(DType dt, int d, const L2Args& a, const float* M, cudaStream_t stream);
// Tensor-core path (bf16, d in {64, 128}): workspaces l2_tc_moments_ws_bytes() (split partials)
// and l2_tc_readout_ws_bytes() (the bf16 operand image).
size_t l2_tc_moments_ws_bytes(int B, int L, int H, int d);
size_t l2_tc_readout_ws_bytes(int B, int H, int d);
cudaError_t launch_l2_tc_moments_plain(int d, const L2Args& a, float* M, cudaStream_t stream);
cudaError_t launch_l2_tc_readout_plain(int d, const L2Args& a, const float* M, cudaStream_t stream);

// One sequence split into consecutive shards (one per GPU): the state increment of a shard
// (sum of k' v^T and of k' over its tokens, per (batch row, head)), in blocks of blk_len tokens
// whose records (ws_bytes of workspace, the tensor-core state kernel's layout) are summed in
// block order into plain S [bh][d][d] and z [bh][d].
struct ShardPlan {
  bool tc;
  int blk_len;
  int nblk;
  size_t ws_bytes;
};
ShardPlan shard_state_plan(DType dt, int B, int L, int H, int d);
cudaError_t launch_shard_state(DType dt, int d, const PrefillArgs& a, const ShardPlan& p, float* ws,
                               float* S, float* z, cudaStream_t stream);
// out[i] = init[i] (0 if null) + parts[0][i] + ... + parts[r-1][i] over n floats (n % 4 == 0),
// parts holding consecutive arrays of n floats, added in rank order.
cudaError_t launch_state_prefix(const float* parts, long n, int r, const float* init, float* out,
                                cudaStream_t stream);

int l2_default_splits(int B, int L, int H);
size_t l2_workspace_bytes_for_splits(int B, int H, int d, int nsplit);
cudaError_t launch_rla_l2_with_splits(DType dt, int d, const L2Args& a, int nsplit,
                                      cudaStream_t stream);

}  // namespace rapt
