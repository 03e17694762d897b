"""rla_l2_fwd_noalloc: the allocation-free L2-denominator entry point.

It serves callers that cannot allocate device memory (a plugin handed only its input and output
buffers by an engine that owns all device memory, or a hot loop that must not call cudaMalloc
because it can synchronise the device). Its scratch is a fixed array inside the library. These
tests call it through the C ABI on two calls in a row (different shapes and dtypes, so the second
call runs on whatever the first one left in the shared array) and compare each call's whole
output with the fp64 oracle, within the tolerance of the other parity tests.
"""

import ctypes

import pytest
import torch

import oracle as O
from gpu_helpers import TOL, draw, to_dev, to_host, widen
from relu_linear_attention_gb300 import _lib

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, out, eps=1e-6):
    B, L, H, d = q.shape
    dt = _lib.RAPT_BF16 if q.dtype == torch.bfloat16 else _lib.RAPT_F32
    st = lib.rla_l2_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                ctypes.c_void_p(v.data_ptr()), dt, B, L, H, d, eps,
                                ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_oracle_twice(cuda_device, lib):
    cases = [((2, 4096, 16, 128), "bf16"), ((1, 1000, 3, 64), "f32")]
    for i, (shape, dtype) in enumerate(cases):
        qn, kn, vn = draw(90 + i, shape, dtype)
        q, k, v = (to_dev(x, dtype) for x in (qn, kn, vn))
        out = torch.full_like(q, float("nan"))
        assert _noalloc(lib, q, k, v, out) == _lib.RAPT_OK
        torch.cuda.synchronize()
        ref = O.rla_l2(widen(qn, dtype), widen(kn, dtype), widen(vn, dtype), 1e-6)
        err = O.relative_error(to_host(out), ref)[0]
        assert err <= TOL[dtype], "call %d: max row rel err %.3g" % (i, err)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device, lib):
    # B * H * 2 * d * 2d * 4 bytes must fit RAPT_L2_NOALLOC_SCRATCH_BYTES: at d = 128, B*H <= 64
    need = 1 * 65 * 2 * 128 * 256 * 4
    assert need > _lib.RAPT_L2_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((1, 8, 65, 128), dtype=torch.bfloat16, device=cuda_device)
    out = torch.empty_like(q)
    assert _noalloc(lib, q, q.clone(), q.clone(), out) == _lib.RAPT_ERR_WORKSPACE
