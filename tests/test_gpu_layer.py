"""GPU parity of the tensor-core projection (rapt_linear_fwd) and of one RAPT layer
(rapt_layer_fwd: q | k | v projection, causal RLA-2, output projection) against the fp64 oracle,
through the C ABI.

The projections are the layer's linear maps (08-rapt-algorithm.md §3: q = W_q x before the
features; §4.2: the output projection w_o). bf16 tensors, fp32 accumulation; tolerance: max
per-row relative error 2e-2 (bf16). Shapes cover exact tiles, ragged M and N tiles, a K tail
shorter than one 64-wide block, K = 8, one row, and a projection of the size the layer bench uses.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, to_dev, to_host
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _bf16(seed, shape, scale=1.0):
    """N(0, scale^2) rounded to bf16: (bit pattern for the device, exact fp64 values)."""
    x = syn.rng(seed).standard_normal(shape).astype(np.float32) * np.float32(scale)
    bits = syn.f32_to_bf16_bits(x)
    return bits, syn.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 272, 72), (1, 16, 8), (300, 48, 1000),
                                   (1000, 512, 256), (513, 1024, 136)])
def test_linear_matches_oracle(cuda_device, lib, M, N, K):
    xb, x = _bf16(500 + M, (M, K))
    wb, w = _bf16(501 + N, (N, K), 1.0 / np.sqrt(K))
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    y = R.rapt_linear_fwd(to_dev(xb, "bf16"), to_dev(wb, "bf16"), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert O.relative_error(to_host(y), O.linear(x, w))[0] <= TOL["bf16"]


def test_linear_large_sampled_rows_and_repeats(cuda_device, lib):
    """x [16384, 2048] W_qkv^T with W [6144, 2048]: the layer workload's q | k | v projection; the
    oracle checks 256 sampled rows (each exact over all of K); repeats are bitwise equal."""
    M, N, K = 16384, 6144, 2048
    xb, x = _bf16(510, (M, K))
    wb, w = _bf16(511, (N, K), 1.0 / np.sqrt(K))
    tx, tw = to_dev(xb, "bf16"), to_dev(wb, "bf16")
    y = R.rapt_linear_fwd(tx, tw)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, M - 1], syn.rng(512).integers(0, M, 254)]))
    got = to_host(y[torch.from_numpy(rows).to(y.device)])
    assert O.relative_error(got, x[rows] @ w.T)[0] <= TOL["bf16"]
    assert torch.equal(y, R.rapt_linear_fwd(tx, tw))


LAYER_CASES = [
    # (B, L, H, d, d_model, per_head_gamma, pos_offset)
    (2, 200, 2, 64, 128, True, 0),
    (1, 300, 4, 128, 512, False, 5),
    (1, 64, 2, 16, 32, True, 0),
    (2, 129, 3, 32, 96, False, 0),
]


@pytest.mark.parametrize("case", LAYER_CASES, ids=lambda c: "B%dL%dH%dd%ddm%d" % c[:5])
def test_layer_matches_oracle(cuda_device, lib, case):
    B, L, H, d, dm, per_head, off = case
    xb, x = _bf16(520 + L, (B, L, dm))
    wqb, wq = _bf16(521, (3 * H * d, dm), 1.0 / np.sqrt(dm))
    wob, wo = _bf16(522, (dm, H * d), 1.0 / np.sqrt(H * d))
    g = syn.rng(523)
    gshape = (H, d) if per_head else (d,)
    gq, gk = syn.gamma_uniform(g, gshape), syn.gamma_uniform(g, gshape)
    dev = lambda a: torch.from_numpy(a).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    y = R.rapt_layer_fwd(to_dev(xb, "bf16"), to_dev(wqb, "bf16"), to_dev(wob, "bf16"), dev(gq),
                         dev(gk), heads=H, pos_offset=off, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.rapt_layer(x, wq, wo, gq, gk, H, pos_offset=off)
    assert O.relative_error(to_host(y), ref)[0] <= TOL["bf16"]


def test_layer_long_sampled_rows(cuda_device, lib):
    """B=1, L=2048, H=8, d=128, d_model=1024 (two attention segments): 128 sampled rows."""
    B, L, H, d, dm = 1, 2048, 8, 128, 1024
    xb, x = _bf16(530, (B, L, dm))
    wqb, wq = _bf16(531, (3 * H * d, dm), 1.0 / np.sqrt(dm))
    wob, wo = _bf16(532, (dm, H * d), 1.0 / np.sqrt(H * d))
    g = syn.rng(533)
    gq, gk = syn.gamma_uniform(g, (H, d)), syn.gamma_uniform(g, (H, d))
    dev = lambda a: torch.from_numpy(a).to(cuda_device)
    y = R.rapt_layer_fwd(to_dev(xb, "bf16"), to_dev(wqb, "bf16"), to_dev(wob, "bf16"), dev(gq),
                         dev(gk), heads=H)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, L - 1], syn.rng(534).integers(0, L, 126)]))
    ref = O.rapt_layer(x, wq, wo, gq, gk, H, pairs_rows=(0, rows))
    got = to_host(y[0, torch.from_numpy(rows).to(y.device)])
    assert O.relative_error(got, ref[0, rows])[0] <= TOL["bf16"]
