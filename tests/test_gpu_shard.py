"""One sequence split into consecutive shards (the exchange step of a sequence spread over GPUs),
run here shard by shard on one GPU through the C ABI, against the fp64 oracle of the whole
sequence.

Causal RLA-2: every shard's state increment (rapt_prefill_state) equals the oracle's state of
the shard's own tokens; each shard started from the sum of the earlier increments
(rapt_state_prefix) and run by rapt_prefill_fwd reproduces the whole sequence's output; the sum of
all increments is the whole sequence's final state. The all-gather between the two steps is the
stacking of the increments here (on several GPUs: NCCL). Non-causal L2: the moments of the
shards (rla_l2_moments) add up to the whole sequence's moments, and the readout of every shard
from the summed moments (rla_l2_readout) reproduces rla_l2 over the whole sequence.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, draw, gammas, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R

pytestmark = pytest.mark.gpu

CASES = [
    # (B, shard L, W shards, H, d, dtype, per-head gains, with an initial state)
    (2, 300, 3, 3, 128, "bf16", True, False),
    (1, 1000, 2, 2, 128, "bf16", False, True),
    (2, 200, 4, 2, 64, "bf16", True, True),
    (1, 96, 3, 2, 32, "f32", False, True),
    (2, 77, 2, 1, 16, "bf16", True, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dL%dxW%dH%dd%d-%s" % c[:6])
def test_sharded_prefill_equals_whole_sequence(cuda_device, lib, case):
    B, Ls, W, H, d, dtype, per_head, with_s0 = case
    L = W * Ls
    q, k, v = draw(700 + d + W, (B, L, H, d), dtype)
    gq, gk = gammas(701, H, d, per_head)
    S0 = z0 = None
    if with_s0:
        rs = np.random.default_rng(702)
        S0 = rs.standard_normal((B, H, d, d)).astype(np.float32)
        z0 = np.abs(rs.standard_normal((B, H, d))).astype(np.float32) * 4.0
    dev = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(cuda_device)
    shard = lambda x, r: to_dev(np.ascontiguousarray(x[:, r * Ls:(r + 1) * Ls]), dtype)
    wq, wk, wv = (widen(x, dtype) for x in (q, k, v))

    # 1. every shard's increment, checked against the oracle's state of that shard alone
    incs = []
    for r in range(W):
        S_inc, z_inc = R.rapt_prefill_state(shard(k, r), shard(v, r), dev(gk), pos_offset=r * Ls)
        incs.append((S_inc, z_inc))
        _, Sr, zr = O.rla2_prefill(wq[:, r * Ls:(r + 1) * Ls], wk[:, r * Ls:(r + 1) * Ls],
                                   wv[:, r * Ls:(r + 1) * Ls], gq, gk, pos_offset=r * Ls,
                                   rows=np.array([0]))
        torch.cuda.synchronize()
        for b in range(B):
            for h in range(H):
                assert O.relative_error(to_host(S_inc[b, h]), Sr[b, h])[1] <= TOL[dtype], (r, b, h)
                assert O.relative_error(to_host(z_inc[b, h]), zr[b, h])[1] <= TOL[dtype], (r, b, h)
    # 2. the gathered increments (rank order)
    S_parts = torch.stack([s for s, _ in incs])
    z_parts = torch.stack([z for _, z in incs])
    # 3. + 4. every shard from its start state
    outs = []
    for r in range(W):
        S_start, z_start = R.rapt_state_prefix(S_parts, z_parts, r, S0=dev(S0), z0=dev(z0))
        out, _, _ = R.rapt_prefill_fwd(shard(q, r), shard(k, r), shard(v, r), dev(gq), dev(gk),
                                       pos_offset=r * Ls, S0=S_start, z0=z_start)
        outs.append(out)
    S_fin, z_fin = R.rapt_state_prefix(S_parts, z_parts, W, S0=dev(S0), z0=dev(z0))
    torch.cuda.synchronize()
    got = np.concatenate([to_host(o) for o in outs], axis=1)
    ref, Sref, zref = O.rla2_prefill(wq, wk, wv, gq, gk, S0=S0, z0=z0)
    assert O.relative_error(got, ref)[0] <= TOL[dtype]
    for b in range(B):
        for h in range(H):
            assert O.relative_error(to_host(S_fin[b, h]), Sref[b, h])[1] <= TOL[dtype]
            assert O.relative_error(to_host(z_fin[b, h]), zref[b, h])[1] <= TOL[dtype]


def test_state_prefix_adds_in_rank_order(cuda_device, lib):
    """rapt_state_prefix against plain sums of the parts, r = 0 (the initial state alone, or zeros)
    up to r = W, with and without an initial state."""
    W, B, H, d = 4, 2, 3, 32
    g = torch.Generator(device=cuda_device).manual_seed(7)
    S_parts = torch.randn((W, B, H, d, d), device=cuda_device, generator=g)
    z_parts = torch.randn((W, B, H, d), device=cuda_device, generator=g)
    S0 = torch.randn((B, H, d, d), device=cuda_device, generator=g)
    z0 = torch.randn((B, H, d), device=cuda_device, generator=g)
    for init in (False, True):
        for r in range(W + 1):
            S, z = R.rapt_state_prefix(S_parts, z_parts, r, S0=S0 if init else None,
                                       z0=z0 if init else None)
            eS = (S0.double() if init else torch.zeros_like(S0, dtype=torch.float64)) + \
                S_parts[:r].double().sum(0)
            ez = (z0.double() if init else torch.zeros_like(z0, dtype=torch.float64)) + \
                z_parts[:r].double().sum(0)
            assert torch.allclose(S.double(), eS, rtol=1e-6, atol=1e-5)
            assert torch.allclose(z.double(), ez, rtol=1e-6, atol=1e-5)


def test_empty_shard_adds_nothing(cuda_device, lib):
    k = torch.empty((2, 0, 2, 64), dtype=torch.bfloat16, device=cuda_device)
    g = torch.ones(64, device=cuda_device)
    S, z = R.rapt_prefill_state(k, k.clone(), g)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S) == 0 and torch.count_nonzero(z) == 0


def test_sharded_helper_without_process_group_is_the_whole_prefill(cuda_device, lib):
    """One rank: the helper's state call, exchange and prefill give the whole sequence."""
    B, L, H, d = 2, 500, 2, 128
    qn, kn, vn = draw(720, (B, L, H, d), "bf16")
    gqn, gkn = gammas(721, H, d, True)
    q, k, v = (to_dev(x, "bf16") for x in (qn, kn, vn))
    gq, gk = (torch.from_numpy(x).to(cuda_device) for x in (gqn, gkn))
    out, Sf, zf = R.rapt_prefill_fwd_sharded(q, k, v, gq, gk, final_state=True)
    torch.cuda.synchronize()
    ref, Sref, zref = O.rla2_prefill(widen(qn, "bf16"), widen(kn, "bf16"), widen(vn, "bf16"), gqn, gkn)
    assert O.relative_error(to_host(out), ref)[0] <= TOL["bf16"]
    for b in range(B):
        for h in range(H):
            assert O.relative_error(to_host(Sf[b, h]), Sref[b, h])[1] <= TOL["bf16"]
            assert O.relative_error(to_host(zf[b, h]), zref[b, h])[1] <= TOL["bf16"]


L2_CASES = [
    # (B, shard L, W shards, H, d, dtype)
    (2, 1000, 2, 4, 128, "bf16"),
    (1, 700, 3, 2, 64, "bf16"),
    (1, 300, 2, 3, 32, "f32"),
    (2, 150, 3, 2, 16, "bf16"),
]


@pytest.mark.parametrize("case", L2_CASES, ids=lambda c: "B%dL%dxW%dH%dd%d-%s" % c)
def test_l2_moments_then_readout_equals_whole_sequence(cuda_device, lib, case):
    B, Ls, W, H, d, dtype = case
    L = W * Ls
    q, k, v = draw(730 + d, (B, L, H, d), dtype)
    shard = lambda x, r: to_dev(np.ascontiguousarray(x[:, r * Ls:(r + 1) * Ls]), dtype)
    wq, wk, wv = (widen(x, dtype) for x in (q, k, v))
    Ms = [R.rla_l2_moments(shard(k, r), shard(v, r)) for r in range(W)]
    M = torch.stack(Ms).sum(0)  # the all-reduce of the shards' moments
    outs = [R.rla_l2_readout(shard(q, r), M, eps=1e-6) for r in range(W)]
    torch.cuda.synchronize()
    # the moments are the definitions M_V = sum relu(k) v^T, M_K = sum relu(k) relu(k)^T (§2.1)
    kf = np.maximum(wk, 0.0)
    for b in range(B):
        for h in range(H):
            MV = kf[b, :, h].T @ wv[b, :, h]
            MK = kf[b, :, h].T @ kf[b, :, h]
            Mh = to_host(M[b, h])
            assert O.relative_error(Mh[:, :d], MV)[1] <= 1e-5
            assert O.relative_error(Mh[:, d:], MK)[1] <= 1e-5
    got = np.concatenate([to_host(o) for o in outs], axis=1)
    ref = O.rla_l2(wq, wk, wv, 1e-6)
    assert O.relative_error(got, ref)[0] <= TOL[dtype]
    # one shard: moments then readout is rla_l2_fwd
    qa, ka, va = (to_dev(x, dtype) for x in (q, k, v))
    whole = R.rla_l2_fwd(qa, ka, va, eps=1e-6)
    two = R.rla_l2_readout(qa, R.rla_l2_moments(ka, va), eps=1e-6)
    torch.cuda.synchronize()
    assert O.relative_error(to_host(two), to_host(whole))[0] <= TOL[dtype]


def test_l2_empty_shard_gives_zero_moments(cuda_device, lib):
    k = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device=cuda_device)
    M = R.rla_l2_moments(k, k.clone())
    torch.cuda.synchronize()
    assert torch.count_nonzero(M) == 0
