"""GPU parity of the causal original RLA (L2 denominator) against the fp64 oracle, through the C
ABI: rla_l2_causal_fwd / rla_l2_causal_varlen_fwd.

08-rapt-algorithm.md §2.1 (closed form, eps 1e-6 outside the root), §2.2 (causal state, reset at
document boundaries), §4.1 (the A = sum k'k'^T prefix state). Tolerance: max per-row relative error
1e-4 for fp32 tensors, 2e-2 for bf16 (fp32 arithmetic throughout). Shapes span one and many
segments per document, ragged last chunks, L = 1, empty and one-token documents, packed documents
of the varlen length mix, and the full size of the L2 workload (B=2, L=16384, H=16, d=128) on 512
rows of every head.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, draw, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

CASES = [
    # (B, L, H, d, dtype)
    (1, 64, 2, 16, "f32"),
    (2, 65, 2, 32, "f32"),
    (1, 200, 2, 64, "f32"),
    (1, 129, 1, 128, "f32"),
    (2, 63, 2, 16, "bf16"),
    (1, 1, 1, 128, "bf16"),
    (2, 300, 2, 64, "bf16"),
    (1, 1000, 3, 128, "bf16"),
    (3, 257, 5, 128, "f32"),
    (3, 128, 2, 128, "bf16"),   # one whole chunk per row
    (1, 256, 1, 128, "bf16"),   # two chunks, each its own segment
    (2, 4000, 1, 128, "bf16"),  # many chunks per segment, ragged last chunk
    (1, 5000, 2, 64, "bf16"),   # d = 64 on the tensor cores: many segments from the moments
    (3, 129, 4, 64, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dL%dH%dd%d-%s" % c)
def test_l2_causal_matches_oracle(cuda_device, lib, case):
    B, L, H, d, dtype = case
    q, k, v = draw(400 + L, (B, L, H, d), dtype)
    out = R.rla_l2_causal_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    torch.cuda.synchronize()
    ref = O.rla_l2_causal(widen(q, dtype), widen(k, dtype), widen(v, dtype), 1e-6)
    assert O.relative_error(to_host(out), ref)[0] <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_l2_causal_varlen_matches_oracle(cuda_device, lib, dtype, d):
    lens = [1, 0, 65, 130, 3, 0, 64, 257]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H = int(cu[-1]), 2
    q, k, v = draw(410 + d, (T, H, d), dtype)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = R.rla_l2_causal_varlen_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                     torch.from_numpy(cu).to(cuda_device), max_seqlen=max(lens),
                                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.rla_l2_causal_varlen(widen(q, dtype), widen(k, dtype), widen(v, dtype), cu, 1e-6)
    assert O.relative_error(to_host(out), ref)[0] <= TOL[dtype]


def test_l2_causal_full_size_sampled(cuda_device, lib):
    """The L2 workload's shapes (B=2, L=16384, H=16, d=128, bf16), causal, in the bench's launch
    configuration; the oracle evaluates 512 sampled rows (including the first and last and rows
    at segment starts) of every (batch row, head) pair, each row exact over its whole causal
    prefix."""
    w = syn.l2_bf16(seed=4)
    out = R.rla_l2_causal_fwd(*(to_dev(x, "bf16") for x in (w.q, w.k, w.v)))
    torch.cuda.synchronize()
    edges = [0, 1, 4095, 4096, 4097, 8191, 8192, 12288, 16383]
    rows = np.unique(np.concatenate([edges, syn.rng(5).integers(0, 16384, 512 - len(edges))]))
    ref = O.rla_l2_causal(syn.bf16_bits_to_f64(w.q), syn.bf16_bits_to_f64(w.k),
                          syn.bf16_bits_to_f64(w.v), 1e-6, rows=rows)
    got = to_host(out[:, torch.from_numpy(rows).to(out.device)])
    assert O.relative_error(got, ref[:, rows])[0] <= TOL["bf16"]


def test_l2_causal_varlen_many_documents(cuda_device, lib):
    """Packed documents of the varlen workload's length mix (U[128, 8192], d = 64, bf16) on the
    tensor cores: one CTA per (document, head), longest first; every document and row."""
    lens = syn.doc_lengths(syn.rng(12), 24000, 128, 8192)
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H, d = int(cu[-1]), 3, 64
    q, k, v = draw(430, (T, H, d), "bf16")
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = R.rla_l2_causal_varlen_fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                                     torch.from_numpy(cu).to(cuda_device),
                                     max_seqlen=int(lens.max()), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.rla_l2_causal_varlen(widen(q, "bf16"), widen(k, "bf16"), widen(v, "bf16"), cu, 1e-6)
    assert O.relative_error(to_host(out), ref)[0] <= TOL["bf16"]


def test_l2_causal_repeats_bitwise_and_bad_cu_seqlens(cuda_device, lib):
    q, k, v = draw(420, (2, 700, 3, 64), "bf16")
    args = [to_dev(x, "bf16") for x in (q, k, v)]
    first = R.rla_l2_causal_fwd(*args)
    for _ in range(3):
        assert torch.equal(first, R.rla_l2_causal_fwd(*args))
    # a decreasing cu_seqlens is reported, never read out of bounds (CUDA-core and tensor-core
    # paths)
    T = 100
    for dtype, d in (("f32", 16), ("bf16", 64)):
        qv, kv, vv = (to_dev(x, dtype) for x in draw(421, (T, 2, d), dtype))
        cu = torch.tensor([0, 60, 40, T], dtype=torch.int32, device=cuda_device)
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        R.rla_l2_causal_varlen_fwd(qv, kv, vv, cu, max_seqlen=T, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & 1, dtype
