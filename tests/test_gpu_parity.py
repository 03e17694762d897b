"""GPU parity of every entry point against the fp64 oracle, element by element, on seeded
inputs at sizes spanning several 64/128-token tiles with ragged tails, plus edge cases.

Tolerance (max per-row relative error, oracle.relative_error): 1e-4 for fp32 inputs,
2e-2 for bf16 inputs with fp32 accumulation.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, draw, gammas, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

PREFILL_CASES = [
    # (B, L, H, d, dtype, per_head_gamma, pos_offset, with_state)
    (1, 64, 2, 16, "f32", False, 0, False),
    (2, 1, 3, 16, "f32", False, 0, False),
    (2, 65, 2, 32, "f32", True, 5, True),
    (1, 200, 2, 64, "f32", False, 0, True),
    (1, 129, 1, 128, "f32", True, 1000, False),
    (2, 63, 2, 16, "bf16", False, 0, False),
    (2, 257, 2, 64, "bf16", True, 0, True),
    (1, 130, 3, 128, "bf16", True, 17, True),
    (3, 384, 2, 128, "bf16", True, 0, False),
    (1, 2, 1, 32, "bf16", False, 0, False),
    (2, 3000, 4, 64, "bf16", True, 5, True),   # heads in pairs, several segments per row
    (3, 200, 6, 64, "bf16", False, 9, False),  # heads in pairs, gains shared by the heads
    (1, 300, 3, 64, "bf16", False, 0, True),   # odd head count: one head per CTA
]


def _prefill_case(B, L, H, d, dtype, per_head, off, with_state, seed=0):
    q, k, v = draw(seed + 1, (B, L, H, d), dtype)
    gq, gk = gammas(seed + 2, H, d, per_head)
    S0 = z0 = None
    if with_state:
        S0, z0 = syn.random_state(seed + 3, (B, H, d, d), (B, H, d))
    return q, k, v, gq, gk, S0, z0


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "B%dL%dH%dd%d-%s" % c[:5])
def test_prefill_matches_oracle(cuda_device, lib, case):
    B, L, H, d, dtype, per_head, off, with_state = case
    q, k, v, gq, gk, S0, z0 = _prefill_case(*case)
    dev = lambda x: None if x is None else torch.from_numpy(x).to(cuda_device)
    out, Sf, zf = R.rapt_prefill_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                     dev(gq), dev(gk), pos_offset=off, S0=dev(S0), z0=dev(z0),
                                     final_state=True)
    torch.cuda.synchronize()
    ref, Sref, zref = O.rla2_prefill(widen(q, dtype), widen(k, dtype), widen(v, dtype), gq, gk,
                                     1e-6, 1e4, 1e-4, pos_offset=off, S0=S0, z0=z0)
    err = O.relative_error(to_host(out), ref)[0]
    assert err <= TOL[dtype], "max row rel err %.3g" % err
    # the carried state is fp32 in both dtypes; bf16 features bound its error (rel. to its scale)
    stol = 1e-4 if dtype == "f32" else 2e-2
    assert O.relative_error(to_host(Sf).reshape(-1, d), Sref.reshape(-1, d))[1] <= stol
    assert O.relative_error(to_host(zf), zref)[1] <= stol


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_varlen_matches_oracle(cuda_device, lib, dtype, d):
    lens = [1, 0, 65, 130, 3, 0, 64, 257]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H, N = int(cu[-1]), 2, len(lens)
    q, k, v = draw(10 + d, (T, H, d), dtype)
    gq, gk = gammas(11, H, d, True)
    S0, z0 = syn.random_state(12, (N, H, d, d), (N, H, d))
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out, Sf, zf = R.rapt_varlen_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                    dev(cu), dev(gq), dev(gk), max_seqlen=max(lens), S0=dev(S0),
                                    z0=dev(z0), final_state=True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, Sref, zref = O.rla2_varlen(widen(q, dtype), widen(k, dtype), widen(v, dtype), cu, gq, gk,
                                    S0=S0, z0=z0)
    assert O.relative_error(to_host(out), ref)[0] <= TOL[dtype]
    stol = 1e-4 if dtype == "f32" else 2e-2
    assert O.relative_error(to_host(Sf).reshape(-1, d), Sref.reshape(-1, d))[1] <= stol
    assert O.relative_error(to_host(zf), zref)[1] <= stol
    # empty documents carry their initial state through unchanged
    for n in (1, 5):
        assert torch.equal(Sf[n].cpu(), torch.from_numpy(S0[n]))
        assert torch.equal(zf[n].cpu(), torch.from_numpy(z0[n]))


def test_varlen_malformed_cu_seqlens_reported(cuda_device, lib):
    """A decreasing cu_seqlens entry is reported through dev_status; the bad documents are
    skipped (never read out of bounds) and the good ones are still computed."""
    T, H, d = 40, 1, 16
    q, k, v = draw(20, (T, H, d), "f32")
    cu = np.array([0, 10, 5, 40], dtype=np.int32)  # document 1 has end < start
    g = np.ones(d, np.float32)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = torch.zeros((T, H, d), device=cuda_device)
    R.rapt_varlen_fwd(dev(q), dev(k), dev(v), dev(cu), dev(g), dev(g), max_seqlen=T, out=out,
                      dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    ref, _, _ = O.rla2_varlen(q, k, v, np.array([0, 10], np.int32), g, g)
    assert O.relative_error(to_host(out)[:10], ref[:10])[0] <= 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_decode_step_matches_oracle(cuda_device, lib, dtype, d):
    N, H = 5, 3
    q, k, v = draw(30 + d, (N, H, d), dtype)
    gq, gk = gammas(31, H, d, d >= 64)
    S, z = syn.random_state(32, (N, H, d, d), (N, H, d))
    pos = np.array([0, 1, 7, 512, 8191], dtype=np.int32)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    Sd, zd = dev(S), dev(z)
    out = R.rapt_decode_step(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev(pos),
                             dev(gq), dev(gk), Sd, zd)
    torch.cuda.synchronize()
    ref, Sref, zref = O.rla2_decode_step(widen(q, dtype), widen(k, dtype), widen(v, dtype), pos,
                                         gq, gk, S, z)
    assert O.relative_error(to_host(out), ref)[0] <= TOL[dtype]
    np.testing.assert_allclose(to_host(Sd), Sref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(to_host(zd), zref, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_equals_prefill(cuda_device, lib, dtype):
    """KV-cache consistency (08-rapt-algorithm.md §4.4): prefill P tokens on the GPU, then
    decode the next tokens one by one; every decode output equals the oracle's prefill row."""
    N, P, steps, H, d = 3, 70, 5, 2, 64
    q, k, v = draw(40, (N, P + steps, H, d), dtype)
    gq, gk = gammas(41, H, d, True)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(cuda_device)
    _, S, z = R.rapt_prefill_fwd(to_dev(q[:, :P], dtype), to_dev(k[:, :P], dtype),
                                 to_dev(v[:, :P], dtype), dev(gq), dev(gk), final_state=True)
    ref, _, _ = O.rla2_prefill(widen(q, dtype), widen(k, dtype), widen(v, dtype), gq, gk)
    for t in range(steps):
        pos = dev(np.full(N, P + t, np.int32))
        o = R.rapt_decode_step(to_dev(q[:, P + t], dtype), to_dev(k[:, P + t], dtype),
                               to_dev(v[:, P + t], dtype), pos, dev(gq), dev(gk), S, z)
        torch.cuda.synchronize()
        assert O.relative_error(to_host(o), ref[:, P + t])[0] <= TOL[dtype]


@pytest.mark.parametrize("B,L,H,d,dtype", [
    (1, 1, 1, 16, "f32"), (2, 77, 2, 32, "f32"), (1, 300, 2, 64, "f32"), (1, 129, 1, 128, "f32"),
    (2, 65, 2, 16, "bf16"), (1, 1000, 2, 64, "bf16"), (2, 513, 2, 128, "bf16"),
])
def test_rla_l2_matches_oracle(cuda_device, lib, B, L, H, d, dtype):
    q, k, v = draw(50 + L, (B, L, H, d), dtype)
    out = R.rla_l2_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), eps=1e-6)
    torch.cuda.synchronize()
    ref = O.rla_l2(widen(q, dtype), widen(k, dtype), widen(v, dtype), 1e-6)
    assert O.relative_error(to_host(out), ref)[0] <= TOL[dtype]


@pytest.mark.parametrize("B,L,H,d", [(4, 3000, 16, 64), (1, 4100, 40, 128), (3, 2000, 7, 128)])
def test_rla_l2_tensor_core_splits(cuda_device, lib, B, L, H, d):
    """bf16 shapes where the tensor-core L2 path cuts every (batch row, head) into token splits of
    several 128-token tiles (the stage ring wraps), L not a multiple of 128 (the last tile reads
    zeros past L and stores nothing there), and several batch rows (no tile crosses into the next
    row). Sampled rows, including the first and the ragged last ones, of every (batch row, head)."""
    q, k, v = draw(80 + L, (B, L, H, d), "bf16")
    out = R.rla_l2_fwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), eps=1e-6)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(3), np.arange(L - 3, L),
                                     np.random.default_rng(L).integers(0, L, 40)]))
    ref = O.rla_l2(widen(q, "bf16"), widen(k, "bf16"), widen(v, "bf16"), 1e-6, rows=rows)
    got = to_host(out)[:, rows]
    assert O.relative_error(got, ref[:, rows])[0] <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_disjoint_supports_exact_zero(cuda_device, lib, dtype):
    """Scores are exactly 0 when the positive supports of q' and k' are disjoint
    (08-rapt-algorithm.md §1): the GPU must return exact zeros, in every entry point."""
    B, L, H, d = 2, 150, 2, 64
    q, k, v = draw(60, (B, L, H, d), dtype)
    mq = np.zeros(d, bool)
    mq[0::4] = mq[1::4] = True  # q lives in pairs 0, 2, 4, ...; k in pairs 1, 3, 5, ...
    zero = np.zeros((), dtype=q.dtype)
    q = np.where(mq, q, zero)
    k = np.where(~mq, k, zero)
    g = np.ones(d, np.float32)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(cuda_device)
    out, _, _ = R.rapt_prefill_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev(g),
                                   dev(g))
    o2 = R.rla_l2_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    assert torch.count_nonzero(o2).item() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_deterministic_repeats(cuda_device, lib, dtype):
    """Ten repeats of each entry point are bitwise identical (no float atomics)."""
    B, L, H, d = 2, 300, 2, 128
    q, k, v = (to_dev(x, dtype) for x in draw(70, (B, L, H, d), dtype))
    g = torch.ones(d, device=cuda_device)
    first = R.rapt_prefill_fwd(q, k, v, g, g, final_state=True)
    l2 = R.rla_l2_fwd(q, k, v)
    for _ in range(9):
        again = R.rapt_prefill_fwd(q, k, v, g, g, final_state=True)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
        assert torch.equal(l2, R.rla_l2_fwd(q, k, v))


def test_zero_length_prefill_writes_initial_state(cuda_device, lib):
    B, H, d = 2, 2, 32
    S0, z0 = syn.random_state(80, (B, H, d, d), (B, H, d))
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    q = torch.empty((B, 0, H, d), device=cuda_device)
    g = torch.ones(d, device=cuda_device)
    _, Sf, zf = R.rapt_prefill_fwd(q, q.clone(), q.clone(), g, g, S0=dev(S0), z0=dev(z0),
                                   final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(Sf.cpu(), torch.from_numpy(S0)) and torch.equal(zf.cpu(), torch.from_numpy(z0))
