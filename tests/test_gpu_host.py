"""GPU tests of rapt_prefill_fwd_host: q, k, v and out in host memory, batch rows pipelined over a
copy-in stream, the compute stream and a copy-out stream, through the C ABI.

The entry point computes every batch row with rapt_prefill_fwd at B = 1, so its output and final
states must equal, bit for bit, those of rapt_prefill_fwd called on each row's device copy; one
case also checks the result against the fp64 oracle (causal RLA-2, 08-rapt-algorithm.md §3).
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, to_host
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _inputs(seed, B, L, H, d, dtype):
    g = syn.rng(seed)
    x = [g.standard_normal((B, L, H, d)).astype(np.float32) for _ in range(3)]
    if dtype == torch.bfloat16:
        bits = [syn.f32_to_bf16_bits(a) for a in x]
        host = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory() for b in bits]
        exact = [syn.bf16_bits_to_f64(b) for b in bits]
    else:
        host = [torch.from_numpy(a).pin_memory() for a in x]
        exact = [a.astype(np.float64) for a in x]
    gq = syn.gamma_uniform(g, (H, d))
    gk = syn.gamma_uniform(g, (H, d))
    return host, exact, gq, gk


def _per_row(host, gq, gk, dev, **kw):
    """rapt_prefill_fwd on each batch row's device copy (the reference of the host entry)."""
    q, k, v = (t.to(dev) for t in host)
    outs, Ss, zs = [], [], []
    for b in range(q.shape[0]):
        S0 = kw.get("S0")
        z0 = kw.get("z0")
        o, S, z = R.rapt_prefill_fwd(q[b:b + 1].contiguous(), k[b:b + 1].contiguous(),
                                     v[b:b + 1].contiguous(), gq, gk, final_state=True,
                                     S0=None if S0 is None else S0[b:b + 1].contiguous(),
                                     z0=None if z0 is None else z0[b:b + 1].contiguous(),
                                     pos_offset=kw.get("pos_offset", 0))
        outs.append(o)
        Ss.append(S)
        zs.append(z)
    return torch.cat(outs), torch.cat(Ss), torch.cat(zs)


@pytest.mark.parametrize("B,L,H,d,dtype,streams", [
    (3, 300, 4, 128, torch.bfloat16, 3),   # tensor cores, ragged last chunk, three streams
    (2, 256, 2, 64, torch.bfloat16, 1),    # tensor cores d = 64, everything on one stream
    (3, 100, 3, 32, torch.float32, 3),     # CUDA cores
    (1, 129, 2, 128, torch.bfloat16, 3),   # a single row
])
def test_host_entry_equals_per_row_device_calls(cuda_device, lib, B, L, H, d, dtype, streams):
    host, _, gq, gk = _inputs(700 + L, B, L, H, d, dtype)
    dgq, dgk = (torch.from_numpy(a).to(cuda_device) for a in (gq, gk))
    ci = torch.cuda.Stream() if streams == 3 else None
    co = torch.cuda.Stream() if streams == 3 else None
    out, S, z = R.rapt_prefill_fwd_host(*host, dgq, dgk, final_state=True, copy_in=ci, copy_out=co)
    torch.cuda.current_stream().synchronize()
    ref_o, ref_S, ref_z = _per_row(host, dgq, dgk, cuda_device)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o.cpu())
    assert torch.equal(S, ref_S) and torch.equal(z, ref_z)


def test_host_entry_with_initial_state_and_offset(cuda_device, lib):
    B, L, H, d = 2, 200, 2, 128
    host, _, gq, gk = _inputs(711, B, L, H, d, torch.bfloat16)
    dgq, dgk = (torch.from_numpy(a).to(cuda_device) for a in (gq, gk))
    g = syn.rng(712)
    S0 = torch.from_numpy(np.abs(g.standard_normal((B, H, d, d))).astype(np.float32)).to(cuda_device)
    z0 = torch.from_numpy(np.abs(g.standard_normal((B, H, d))).astype(np.float32) * 10).to(cuda_device)
    out, S, z = R.rapt_prefill_fwd_host(*host, dgq, dgk, S0=S0, z0=z0, pos_offset=7,
                                        final_state=True, copy_in=torch.cuda.Stream(),
                                        copy_out=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    ref_o, ref_S, ref_z = _per_row(host, dgq, dgk, cuda_device, S0=S0, z0=z0, pos_offset=7)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o.cpu())
    assert torch.equal(S, ref_S) and torch.equal(z, ref_z)


def test_host_entry_matches_oracle(cuda_device, lib):
    B, L, H, d = 2, 160, 2, 64
    host, exact, gq, gk = _inputs(721, B, L, H, d, torch.bfloat16)
    dgq, dgk = (torch.from_numpy(a).to(cuda_device) for a in (gq, gk))
    out, _, _ = R.rapt_prefill_fwd_host(*host, dgq, dgk, copy_in=torch.cuda.Stream(),
                                        copy_out=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    ref = O.rla2_prefill(*exact, gq, gk)[0]
    assert O.relative_error(to_host(out), ref)[0] <= TOL["bf16"]


def test_host_entry_empty_sequence_writes_states(cuda_device, lib):
    B, H, d = 2, 2, 64
    q = torch.empty((B, 0, H, d), dtype=torch.bfloat16).pin_memory()
    g1 = torch.ones(d, device=cuda_device)
    S0 = torch.rand((B, H, d, d), device=cuda_device)
    z0 = torch.rand((B, H, d), device=cuda_device)
    out, S, z = R.rapt_prefill_fwd_host(q, q, q, g1, g1, S0=S0, z0=z0, final_state=True)
    torch.cuda.current_stream().synchronize()
    assert out.shape == q.shape
    assert torch.equal(S, S0) and torch.equal(z, z0)


def test_host_entry_full_size_equals_device_rows(cuda_device, lib):
    """The headline shapes B=4 L=4096 H=16 d=128 (the end-to-end bench's call)."""
    B, L, H, d = 4, 4096, 16, 128
    w = syn.prefill_bf16(seed=1)
    host = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
            for x in (w.q, w.k, w.v)]
    dgq, dgk = (torch.from_numpy(a).to(cuda_device) for a in (w.gamma_q, w.gamma_k))
    out, _, _ = R.rapt_prefill_fwd_host(*host, dgq, dgk, copy_in=torch.cuda.Stream(),
                                        copy_out=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    ref_o, _, _ = _per_row(host, dgq, dgk, cuda_device)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o.cpu())
