"""GPU parity of the causal original RLA (L2 denominator) against the fp64 oracle, through the C
ABI: rla_l2_causal_fwd / rla_l2_causal_varlen_fwd.

08-rapt-algorithm.md §2.1 (closed form, eps 1e-6 outside the root), §2.2 (causal state, reset at
document boundaries), §4.1 (the A = sum k'k'^T prefix state). Tolerance: max per-row relative error
1e-4 for fp32 tensors, 2e-2 for bf16 (fp32 arithmetic throughout). Shapes span one and many
segments per document, ragged last chunks, L = 1, empty and one-token documents, and the full
size of the L2 workload (B=2, L=16384, H=16, d=128) on sampled rows.
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
    configuration; the oracle evaluates 512 sampled rows (including the first and last) of two
    (batch row, head) pairs, each row exact over its whole causal prefix."""
    w = syn.l2_bf16(seed=4)
    out = R.rla_l2_causal_fwd(*(to_dev(x, "bf16") for x in (w.q, w.k, w.v)))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 1, 16383], syn.rng(5).integers(0, 16384, 509)]))
    for b, h in [(0, 0), (1, 15)]:
        ref = O.rla_l2_causal(syn.bf16_bits_to_f64(w.q), syn.bf16_bits_to_f64(w.k),
                              syn.bf16_bits_to_f64(w.v), 1e-6, pairs=[(b, h)], rows=rows)
        got = to_host(out[b, torch.from_numpy(rows).to(out.device), h])
        assert O.relative_error(got, ref[b, rows, h])[0] <= TOL["bf16"]


def test_l2_causal_repeats_bitwise_and_bad_cu_seqlens(cuda_device, lib):
    q, k, v = draw(420, (2, 700, 3, 64), "bf16")
    args = [to_dev(x, "bf16") for x in (q, k, v)]
    first = R.rla_l2_causal_fwd(*args)
    for _ in range(3):
        assert torch.equal(first, R.rla_l2_causal_fwd(*args))
    # a decreasing cu_seqlens is reported, never read out of bounds
    T = 100
    qv, kv, vv = (to_dev(x, "f32") for x in draw(421, (T, 2, 16), "f32"))
    cu = torch.tensor([0, 60, 40, T], dtype=torch.int32, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    R.rla_l2_causal_varlen_fwd(qv, kv, vv, cu, max_seqlen=T, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
