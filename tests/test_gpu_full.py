"""Parity at the full workload sizes, in the launch configuration the bench times: the whole
output is computed on the GPU and sampled rows (every row exact over all visible keys) are
compared with the fp64 oracle. Rows cover chunk boundaries, the first and last tokens and
random positions."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _rows(n, seed, extra=24):
    base = [0, 1, 2, 63, 64, 65, 127, 128, 129, n // 2, n - 2, n - 1]
    r = syn.rng(seed).integers(0, n, size=extra).tolist()
    return np.array(sorted(set(x for x in base + r if 0 <= x < n)), dtype=np.int64)


def test_prefill_full_size(cuda_device, lib):
    w = syn.prefill_bf16()
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    out, Sf, zf = R.rapt_prefill_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"),
                                     dev(w.gamma_q), dev(w.gamma_k), final_state=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    pairs = [(0, 0), (1, 5), (2, 9), (3, 15)]
    rows = _rows(w.L, 1)
    ref, Sref, zref = O.rla2_prefill(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"),
                                     w.gamma_q, w.gamma_k, pairs=pairs, rows=rows)
    o = to_host(out)
    for b, h in pairs:
        assert O.relative_error(o[b, rows, h], ref[b, rows, h])[0] <= TOL["bf16"]
        assert O.relative_error(to_host(Sf[b, h]), Sref[b, h])[1] <= 2e-2
        assert O.relative_error(to_host(zf[b, h]), zref[b, h])[1] <= 2e-2


def test_varlen_full_size(cuda_device, lib):
    w = syn.varlen_bf16()
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out, _, _ = R.rapt_varlen_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"),
                                  dev(w.cu_seqlens), dev(w.gamma_q), dev(w.gamma_k),
                                  max_seqlen=int(w.lengths.max()), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    N = len(w.lengths)
    docs = sorted(set([0, N - 1, int(np.argmax(w.lengths)), int(np.argmin(w.lengths))]))
    heads = [0, 31]
    rows = {n: _rows(int(w.lengths[n]), 10 + n, 12) for n in docs}
    ref, _, _ = O.rla2_varlen(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"),
                              w.cu_seqlens, w.gamma_q, w.gamma_k, docs=docs, heads=heads,
                              rows_per_doc=rows)
    o = to_host(out)
    for n in docs:
        idx = w.cu_seqlens[n] + rows[n]
        for h in heads:
            assert O.relative_error(o[idx, h], ref[idx, h])[0] <= TOL["bf16"]


def test_decode_full_size(cuda_device, lib):
    """256 sequences x 32 heads, d=128: state prefilled from 512 tokens by the prefill entry
    point, then 64 decode steps; sampled (sequence, head) outputs vs the oracle's quadratic
    form over the whole history (the oracle never sees the GPU state)."""
    P, steps = 512, 64
    pre = syn.decode_prefix()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(cuda_device)
    g = dev(pre.gamma_q)
    _, S, z = R.rapt_prefill_fwd(to_dev(pre.q, "bf16"), to_dev(pre.k, "bf16"),
                                 to_dev(pre.v, "bf16"), g, g, final_state=True)
    sample = [(0, 0), (17, 3), (128, 16), (255, 31)]
    hist_k = {s: [widen(pre.k[s[0], :, s[1]], "bf16")] for s in sample}
    hist_v = {s: [widen(pre.v[s[0], :, s[1]], "bf16")] for s in sample}
    check_steps = {0, 1, 31, 63}
    for t in range(steps):
        tok = syn.decode_step_tokens(step=t)
        out = R.rapt_decode_step(to_dev(tok.q, "bf16"), to_dev(tok.k, "bf16"),
                                 to_dev(tok.v, "bf16"), dev(tok.positions), g, g, S, z)
        for s in sample:
            hist_k[s].append(widen(tok.k[s[0], s[1]], "bf16")[None])
            hist_v[s].append(widen(tok.v[s[0], s[1]], "bf16")[None])
        if t in check_steps:
            o = to_host(out)
            for (n, h) in sample:
                ref = O.rla2_decode_from_history(widen(tok.q[n, h], "bf16"),
                                                 np.concatenate(hist_k[(n, h)]),
                                                 np.concatenate(hist_v[(n, h)]), P + t,
                                                 pre.gamma_q, pre.gamma_k)
                assert O.relative_error(o[n, h], ref)[0] <= TOL["bf16"], (t, n, h)


def test_rla_l2_full_size(cuda_device, lib):
    w = syn.l2_bf16()
    out = R.rla_l2_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"), eps=w.eps)
    torch.cuda.synchronize()
    pairs = [(0, 0), (1, 7), (1, 15)]
    rows = _rows(w.L, 5)
    ref = O.rla_l2(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"), w.eps, pairs=pairs,
                   rows=rows)
    o = to_host(out)
    for b, h in pairs:
        assert O.relative_error(o[b, rows, h], ref[b, rows, h])[0] <= TOL["bf16"]
