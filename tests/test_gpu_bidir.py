"""GPU parity of the bidirectional (non-causal) RLA-2 entry points against the fp64 oracle.

08-rapt-algorithm.md §4.1 (causal=false: the sums over the whole document) and §4.2 (the
bidirectional branch), Sum denominator and eps of §3. Tolerance as for the causal form: max
per-row relative error 1e-4 for fp32 inputs, 2e-2 for bf16 inputs with fp32 accumulation.
The shapes cover several state blocks per document (the last one ragged), several readout CTAs
per document, CTAs that run through more tiles than their ring of q buffers, empty and one-token
documents, and the full size of the dense prefill workload on sampled rows.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, draw, gammas, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

DENSE_CASES = [
    # (B, L, H, d, dtype, per_head_gamma, pos_offset, pairs evaluated by the oracle or None = all)
    (1, 64, 2, 16, "f32", False, 0, None),
    (2, 65, 2, 32, "f32", True, 5, None),
    (1, 200, 2, 64, "f32", False, 0, None),
    (1, 129, 1, 128, "f32", True, 1000, None),
    (2, 63, 2, 16, "bf16", False, 0, None),
    (1, 1, 1, 128, "bf16", False, 0, None),
    (2, 257, 2, 64, "bf16", True, 0, None),
    (1, 130, 3, 128, "bf16", True, 17, None),
    (3, 384, 2, 128, "bf16", True, 0, None),
    (2, 3000, 3, 128, "bf16", True, 7, [(0, 0), (1, 2)]),        # 24 blocks, 24 readout CTAs
    (8, 2000, 16, 64, "bf16", True, 0, [(0, 0), (7, 15), (3, 9)]),  # 16 tiles per readout CTA
    (4, 1500, 16, 128, "bf16", True, 3, [(0, 0), (3, 15)]),      # ragged second block
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: "B%dL%dH%dd%d-%s" % c[:5])
def test_bidir_matches_oracle(cuda_device, lib, case):
    B, L, H, d, dtype, per_head, off, pairs = case
    q, k, v = draw(100 + L, (B, L, H, d), dtype)
    gq, gk = gammas(101, H, d, per_head)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = R.rapt_bidir_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev(gq), dev(gk),
                           pos_offset=off, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.rla2_bidir(widen(q, dtype), widen(k, dtype), widen(v, dtype), gq, gk, 1e-6, 1e4, 1e-4,
                       pos_offset=off, pairs=pairs)
    got = to_host(out)
    if pairs is not None:
        sel = tuple(np.array(pairs).T)
        got, ref = got[sel[0], :, sel[1]], ref[sel[0], :, sel[1]]
    err = O.relative_error(got, ref)[0]
    assert err <= TOL[dtype], "max row rel err %.3g" % err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_bidir_varlen_matches_oracle(cuda_device, lib, dtype, d):
    lens = [1, 0, 65, 130, 3, 0, 64, 257]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H = int(cu[-1]), 2
    q, k, v = draw(110 + d, (T, H, d), dtype)
    gq, gk = gammas(111, H, d, True)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = R.rapt_bidir_varlen_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev(cu),
                                  dev(gq), dev(gk), max_seqlen=max(lens), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.rla2_bidir_varlen(widen(q, dtype), widen(k, dtype), widen(v, dtype), cu, gq, gk)
    assert O.relative_error(to_host(out), ref)[0] <= TOL[dtype]


def test_bidir_varlen_long_documents(cuda_device, lib):
    """Documents of several blocks and readout CTAs each, packed back to back (a tile at the end
    of one document reaches into the next: its rows must not be written)."""
    lens = [1000, 5, 2100, 0, 700, 129]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H, d = int(cu[-1]), 4, 128
    q, k, v = draw(120, (T, H, d), "bf16")
    gq, gk = gammas(121, H, d, True)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    out = torch.full((T, H, d), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    R.rapt_bidir_varlen_fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), dev(cu),
                            dev(gq), dev(gk), max_seqlen=max(lens), out=out)
    torch.cuda.synchronize()
    ref = O.rla2_bidir_varlen(widen(q, "bf16"), widen(k, "bf16"), widen(v, "bf16"), cu, gq, gk,
                              heads=[0, 3])
    got = to_host(out)
    assert O.relative_error(got[:, [0, 3]], ref[:, [0, 3]])[0] <= TOL["bf16"]
    assert not np.isnan(got).any()  # every row of every document written


@pytest.mark.parametrize("dtype,d", [("f32", 16), ("bf16", 64)])
def test_bidir_varlen_malformed_cu_seqlens_reported(cuda_device, lib, dtype, d):
    T, H = 300, 1
    q, k, v = draw(130, (T, H, d), dtype)
    cu = np.array([0, 150, 100, 300], dtype=np.int32)  # document 1 has end < start
    g = np.ones(d, np.float32)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = R.rapt_bidir_varlen_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev(cu),
                                  dev(g), dev(g), max_seqlen=T, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    ref = O.rla2_bidir_varlen(widen(q, dtype)[:150], widen(k, dtype)[:150], widen(v, dtype)[:150],
                              np.array([0, 150], np.int32), g, g)
    assert O.relative_error(to_host(out)[:150], ref)[0] <= TOL[dtype]


def test_bidir_deterministic(cuda_device, lib):
    B, L, H, d = 2, 3000, 3, 128
    q, k, v = (to_dev(x, "bf16") for x in draw(140, (B, L, H, d), "bf16"))
    gq, gk = (torch.from_numpy(g).to(cuda_device) for g in gammas(141, H, d, True))
    a = R.rapt_bidir_fwd(q, k, v, gq, gk)
    b = R.rapt_bidir_fwd(q, k, v, gq, gk)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_bidir_full_size_sampled_rows(cuda_device, lib):
    """The dense prefill workload's size (B=4, L=4096, H=16, d=128, bf16, per-head gains) in the
    launch configuration the benchmark times; sampled rows of two (batch, head) pairs, each
    exact over all L keys."""
    w = syn.prefill_bf16()
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    out = R.rapt_bidir_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"),
                           dev(w.gamma_q), dev(w.gamma_k))
    torch.cuda.synchronize()
    rows = np.sort(syn.rng(150).choice(w.q.shape[1], 256, replace=False))
    pairs = [(0, 0), (3, 15)]
    ref = O.rla2_bidir(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"), w.gamma_q,
                       w.gamma_k, pairs=pairs, rows=rows)
    got = to_host(out)
    for b, h in pairs:
        assert O.relative_error(got[b, rows, h], ref[b, rows, h])[0] <= TOL["bf16"]
