"""Parity at the full workload sizes, in the launch configuration the bench times, against the
fp64 oracle: the whole output of the tiny fp32 workload, the 4096-token prefill (every batch
row, head and row, plus every final state), the packed varlen forward (every document, head and
row) and the decode workload (every sequence and head at steps 0, 31 and 63); for the 16384-token
L2 workload 1024 query rows of every (batch row, head), each exact over all 16384 keys. Each test
prints its largest per-row error (run pytest with -s to see it)."""

import os

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _report(name, err):
    print("%s: max per-row rel err %.3e" % (name, err))


def _dev(x, device):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def test_tiny_fp32_exact_workload(cuda_device, lib):
    """B=1, H=2, L=64, d=16, fp32, seed 0, gamma = 1: every output against the oracle and
    against the stored oracle output (tests/golden/tiny_fp32_out.txt)."""
    w = syn.tiny_fp32(0)
    out, Sf, zf = R.rapt_prefill_fwd(to_dev(w.q, "f32"), to_dev(w.k, "f32"), to_dev(w.v, "f32"),
                                     _dev(w.gamma_q, cuda_device), _dev(w.gamma_k, cuda_device),
                                     final_state=True)
    torch.cuda.synchronize()
    ref, Sref, zref = O.rla2_prefill(w.q, w.k, w.v, w.gamma_q, w.gamma_k)
    gold = np.loadtxt(os.path.join(GOLDEN, "tiny_fp32_out.txt")).reshape(ref.shape)
    o = to_host(out)
    err = O.relative_error(o, ref)[0]
    _report("tiny fp32", err)
    assert err <= TOL["f32"]
    assert O.relative_error(o, gold)[0] <= TOL["f32"]
    assert O.relative_error(to_host(Sf), Sref)[1] <= TOL["f32"]
    assert O.relative_error(to_host(zf), zref)[1] <= TOL["f32"]


def test_prefill_full_size(cuda_device, lib):
    """B=4, L=4096, H=16, d=128 bf16, per-head gains: all 64 (batch row, head) pairs, all rows,
    and the final state of every pair."""
    w = syn.prefill_bf16()
    out, Sf, zf = R.rapt_prefill_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"),
                                     _dev(w.gamma_q, cuda_device), _dev(w.gamma_k, cuda_device),
                                     final_state=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    ref, Sref, zref = O.rla2_prefill(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"),
                                     w.gamma_q, w.gamma_k)
    o = to_host(out)
    err = O.relative_error(o, ref)[0]
    _report("prefill B=4 L=4096 H=16 d=128", err)
    assert err <= TOL["bf16"]
    S_h, z_h = to_host(Sf), to_host(zf)
    for b in range(w.B):
        for h in range(w.H):
            assert O.relative_error(S_h[b, h], Sref[b, h])[1] <= TOL["bf16"], (b, h)
            assert O.relative_error(z_h[b, h], zref[b, h])[1] <= TOL["bf16"], (b, h)


def test_varlen_full_size(cuda_device, lib):
    """T=65536, H=32, d=64 bf16, documents U[128, 8192]: every document, head and row, and every
    document's final state."""
    w = syn.varlen_bf16()
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out, Sf, zf = R.rapt_varlen_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"),
                                    _dev(w.cu_seqlens, cuda_device), _dev(w.gamma_q, cuda_device),
                                    _dev(w.gamma_k, cuda_device), max_seqlen=int(w.lengths.max()),
                                    dev_status=status, final_state=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, Sref, zref = O.rla2_varlen(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"),
                                    w.cu_seqlens, w.gamma_q, w.gamma_k)
    o = to_host(out)
    err = O.relative_error(o, ref)[0]
    _report("varlen T=65536 H=32 d=64 (%d documents)" % len(w.lengths), err)
    assert err <= TOL["bf16"]
    S_h, z_h = to_host(Sf), to_host(zf)
    for n in range(len(w.lengths)):
        for h in range(w.H):
            assert O.relative_error(S_h[n, h], Sref[n, h])[1] <= TOL["bf16"], (n, h)
            assert O.relative_error(z_h[n, h], zref[n, h])[1] <= TOL["bf16"], (n, h)


def test_decode_full_size(cuda_device, lib):
    """256 sequences x 32 heads, d=128: the state is prefilled from 512 tokens by the prefill
    entry point, then 64 decode steps. Every (sequence, head) output at steps 0, 31 and 63 is
    compared with the oracle's own recurrence, started from its fp64 prefill of the same 512
    tokens (the oracle never sees the GPU state); step 63 of a few pairs is also checked against
    the quadratic form over the whole history."""
    P, steps, check = 512, 64, (0, 31, 63)
    pre = syn.decode_prefix()
    g = _dev(pre.gamma_q, cuda_device)
    _, S, z = R.rapt_prefill_fwd(to_dev(pre.q, "bf16"), to_dev(pre.k, "bf16"),
                                 to_dev(pre.v, "bf16"), g, g, final_state=True)
    toks = [syn.decode_step_tokens(step=t) for t in range(steps)]
    got = {}
    for t, tok in enumerate(toks):
        out = R.rapt_decode_step(to_dev(tok.q, "bf16"), to_dev(tok.k, "bf16"),
                                 to_dev(tok.v, "bf16"), _dev(tok.positions, cuda_device), g, g, S, z)
        if t in check:
            got[t] = to_host(out)
    torch.cuda.synchronize()
    del S, z

    # the oracle's state after the 512 prefix tokens (fp64), then its own decode recurrence
    N, H, d = pre.q.shape[0], pre.q.shape[2], pre.q.shape[3]
    S_ref, z_ref = np.empty((N, H, d, d)), np.empty((N, H, d))
    for n0 in range(0, N, 32):  # 32 sequences at a time (bounds the host memory)
        sl = slice(n0, n0 + 32)
        _, S_ref[sl], z_ref[sl] = O.rla2_prefill(widen(pre.q[sl], "bf16"), widen(pre.k[sl], "bf16"),
                                                 widen(pre.v[sl], "bf16"), pre.gamma_q, pre.gamma_k,
                                                 rows=np.array([P - 1]))
    worst = 0.0
    for t, tok in enumerate(toks):
        ref, S_ref, z_ref = O.rla2_decode_step(widen(tok.q, "bf16"), widen(tok.k, "bf16"),
                                               widen(tok.v, "bf16"), tok.positions, pre.gamma_q,
                                               pre.gamma_k, S_ref, z_ref)
        if t in check:
            err = O.relative_error(got[t], ref)[0]
            worst = max(worst, err)
            assert err <= TOL["bf16"], (t, err)
    _report("decode N=256 H=32 d=128 at steps %s" % (check,), worst)

    # the recurrence itself against the quadratic form over the history, at the last step
    t = steps - 1
    for n, h in [(0, 0), (77, 13), (255, 31)]:
        kh = np.concatenate([widen(pre.k[n, :, h], "bf16")] +
                            [widen(toks[s].k[n, h], "bf16")[None] for s in range(steps)])
        vh = np.concatenate([widen(pre.v[n, :, h], "bf16")] +
                            [widen(toks[s].v[n, h], "bf16")[None] for s in range(steps)])
        hist = O.rla2_decode_from_history(widen(toks[t].q[n, h], "bf16"), kh, vh, P + t,
                                          pre.gamma_q, pre.gamma_k)
        assert O.relative_error(ref[n, h], hist)[0] <= 1e-10
        assert O.relative_error(got[t][n, h], hist)[0] <= TOL["bf16"]


def test_rla_l2_full_size(cuda_device, lib):
    """B=2, L=16384, H=16, d=128 bf16, non-causal: 1024 query rows of every one of the 32
    (batch row, head) pairs (the first and last rows, chunk edges and random rows), each exact
    over all 16384 keys."""
    w = syn.l2_bf16()
    out = R.rla_l2_fwd(to_dev(w.q, "bf16"), to_dev(w.k, "bf16"), to_dev(w.v, "bf16"), eps=w.eps)
    torch.cuda.synchronize()
    edges = [0, 1, 127, 128, 129, w.L // 2, w.L - 129, w.L - 128, w.L - 2, w.L - 1]
    rand = syn.rng(5).choice(w.L, size=1024, replace=False).tolist()
    rows = np.array(sorted(set(rand) | set(edges)), dtype=np.int64)
    assert len(rows) >= 1024
    ref = O.rla_l2(widen(w.q, "bf16"), widen(w.k, "bf16"), widen(w.v, "bf16"), w.eps, rows=rows)
    o = to_host(out)
    err = O.relative_error(o[:, rows], ref[:, rows])[0]
    _report("rla_l2 B=2 L=16384 H=16 d=128 (%d rows per head)" % len(rows), err)
    assert err <= TOL["bf16"]
