"""Host-only checks of the C ABI: the library loads, exports every function that
include/rapt.h declares, and rejects bad arguments before touching the GPU.

Every call here fails validation on the host (or is a pure size query), so no CUDA work
is issued; these tests run without a GPU.
"""

import ctypes
import os
import re

import pytest

from relu_linear_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

FAKE = ctypes.c_void_p(0x7F0000001000)  # a 16-byte aligned non-null value, never dereferenced
FAKE_ODD = ctypes.c_void_p(0x7F0000001004)


def declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, re.M):
            name = m.group(1)
            if name not in ("if", "sizeof", "defined"):
                names.append(name)
    return sorted(set(names))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for fn in ("rapt_prefill_fwd", "rapt_varlen_fwd", "rapt_decode_step", "rla_l2_fwd"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), "librapt.so does not export %s" % name
        assert name in _lib.SIGNATURES, "binding has no signature for %s" % name


def test_defaults_and_strings(lib):
    p = lib.rapt_default_params()
    assert p.eps_norm == pytest.approx(1e-6) and p.rope_base == 1e4
    assert p.eps_den == pytest.approx(1e-4) and p.gamma_head_stride == 0
    assert lib.rapt_status_string(0) == b"RAPT_OK"
    for code in range(1, 5):
        assert lib.rapt_status_string(code).startswith(b"RAPT_ERR")
    assert lib.rapt_abi_version() >= 10000


def test_workspace_queries(lib):
    assert lib.rapt_prefill_workspace_size(4, 4096, 16, 128, 1) > 0
    assert lib.rapt_prefill_workspace_size(4, 4096, 16, 128, 0) == 0  # fp32: CUDA-core path
    assert lib.rapt_varlen_workspace_size(65536, 17, 32, 64, 8192, 1) > 0
    assert lib.rapt_varlen_workspace_size(65536, 17, 32, 16, 8192, 1) == 0
    ws = lib.rla_l2_workspace_size(2, 16384, 16, 128, 1)
    assert ws >= 2 * 16 * 128 * 256 * 4  # at least the reduced moments
    assert lib.rla_l2_workspace_size(2, 16384, 16, 48, 1) == 0


def _params(**kw):
    p = _lib.rapt_params(1e-6, 1e4, 1e-4, 0)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=1, B=1, L=8, H=1, d=16, gq=FAKE, gk=FAKE,
             p=_params(), off=0, S0=None, z0=None, out=ctypes.c_void_p(0x7F0000002000),
             Sf=None, zf=None, st=None, ws=None, wsb=0, s=None)
    a.update(kw)
    return lib.rapt_prefill_fwd(a["q"], a["k"], a["v"], a["dt"], a["B"], a["L"], a["H"], a["d"],
                                a["gq"], a["gk"], a["p"], a["off"], a["S0"], a["z0"], a["out"],
                                a["Sf"], a["zf"], a["st"], a["ws"], a["wsb"], a["s"])


@pytest.mark.parametrize("kw,code", [
    (dict(d=48), _lib.RAPT_ERR_UNSUPPORTED),
    (dict(d=256), _lib.RAPT_ERR_UNSUPPORTED),
    (dict(dt=7), _lib.RAPT_ERR_UNSUPPORTED),
    (dict(q=None), _lib.RAPT_ERR_INVALID_ARG),
    (dict(out=None), _lib.RAPT_ERR_INVALID_ARG),
    (dict(gq=None), _lib.RAPT_ERR_INVALID_ARG),
    (dict(B=0), _lib.RAPT_ERR_INVALID_ARG),
    (dict(L=-1), _lib.RAPT_ERR_INVALID_ARG),
    (dict(off=-3), _lib.RAPT_ERR_INVALID_ARG),
    (dict(q=FAKE_ODD), _lib.RAPT_ERR_INVALID_ARG),
    (dict(out=FAKE), _lib.RAPT_ERR_INVALID_ARG),          # aliases q
    (dict(p=_params(eps_den=0.0)), _lib.RAPT_ERR_INVALID_ARG),
    (dict(p=_params(eps_norm=float("nan"))), _lib.RAPT_ERR_INVALID_ARG),
    (dict(p=_params(rope_base=float("inf"))), _lib.RAPT_ERR_INVALID_ARG),
    (dict(p=_params(gamma_head_stride=3)), _lib.RAPT_ERR_INVALID_ARG),
    (dict(B=1 << 20, L=1 << 20), _lib.RAPT_ERR_INVALID_ARG),
    (dict(S0=FAKE, Sf=FAKE), _lib.RAPT_ERR_INVALID_ARG),   # final state aliases initial
    (dict(st=ctypes.c_void_p(0x7F0000001001)), _lib.RAPT_ERR_INVALID_ARG),
    (dict(d=128, L=4096, B=4, H=16), _lib.RAPT_ERR_WORKSPACE),  # tensor-core path needs one
])
def test_prefill_rejects_bad_arguments(lib, kw, code):
    assert _prefill(lib, **kw) == code


def test_varlen_rejects_bad_arguments(lib):
    out = ctypes.c_void_p(0x7F0000002000)

    def call(**kw):
        a = dict(cu=FAKE, N=2, T=16, msl=16, d=64, p=_params(), st=None)
        a.update(kw)
        return lib.rapt_varlen_fwd(FAKE, FAKE, FAKE, 1, a["T"], 2, a["d"], a["cu"], a["N"], a["msl"],
                                   FAKE, FAKE, a["p"], None, None, out, None, None, a["st"], None, 0,
                                   None)

    assert call(cu=None) == _lib.RAPT_ERR_INVALID_ARG
    assert call(N=0) == _lib.RAPT_ERR_INVALID_ARG
    assert call(T=-1) == _lib.RAPT_ERR_INVALID_ARG
    assert call(msl=-1) == _lib.RAPT_ERR_INVALID_ARG
    assert call(d=96) == _lib.RAPT_ERR_UNSUPPORTED
    assert call(cu=ctypes.c_void_p(0x7F0000001002)) == _lib.RAPT_ERR_INVALID_ARG
    assert call(p=_params(eps_den=-1.0)) == _lib.RAPT_ERR_INVALID_ARG


def test_decode_rejects_bad_arguments(lib):
    out = ctypes.c_void_p(0x7F0000002000)

    def call(**kw):
        a = dict(S=FAKE, z=FAKE, pos=FAKE, N=4, d=128, out=out)
        a.update(kw)
        return lib.rapt_decode_step(FAKE, FAKE, FAKE, 1, a["N"], 2, a["d"], a["pos"], FAKE, FAKE,
                                    _params(), a["S"], a["z"], a["out"], None)

    assert call(S=None) == _lib.RAPT_ERR_INVALID_ARG
    assert call(z=None) == _lib.RAPT_ERR_INVALID_ARG
    assert call(pos=None) == _lib.RAPT_ERR_INVALID_ARG
    assert call(N=0) == _lib.RAPT_ERR_INVALID_ARG
    assert call(d=8) == _lib.RAPT_ERR_UNSUPPORTED
    assert call(S=FAKE_ODD) == _lib.RAPT_ERR_INVALID_ARG
    assert call(out=FAKE) == _lib.RAPT_ERR_INVALID_ARG


def test_l2_rejects_bad_arguments(lib):
    out = ctypes.c_void_p(0x7F0000002000)

    def call(**kw):
        a = dict(eps=1e-6, ws=FAKE, wsb=1 << 40, d=128, L=64)
        a.update(kw)
        return lib.rla_l2_fwd(FAKE, FAKE, FAKE, 1, 1, a["L"], 2, a["d"], a["eps"], out, a["ws"],
                              a["wsb"], None)

    assert call(eps=0.0) == _lib.RAPT_ERR_INVALID_ARG
    assert call(eps=float("nan")) == _lib.RAPT_ERR_INVALID_ARG
    assert call(d=24) == _lib.RAPT_ERR_UNSUPPORTED
    assert call(ws=None) == _lib.RAPT_ERR_WORKSPACE
    assert call(wsb=16) == _lib.RAPT_ERR_WORKSPACE
    assert call(L=0) == _lib.RAPT_OK  # nothing to do, nothing launched


def test_bidir_rejects_bad_arguments(lib):
    out = ctypes.c_void_p(0x7F0000002000)

    def dense(**kw):
        a = dict(q=FAKE, B=1, L=8, d=16, dt=1, off=0, p=_params(), out=out, ws=None, wsb=0)
        a.update(kw)
        return lib.rapt_bidir_fwd(a["q"], FAKE, FAKE, a["dt"], a["B"], a["L"], 2, a["d"], FAKE, FAKE,
                                  a["p"], a["off"], a["out"], None, a["ws"], a["wsb"], None)

    assert dense(d=48) == _lib.RAPT_ERR_UNSUPPORTED
    assert dense(dt=5) == _lib.RAPT_ERR_UNSUPPORTED
    assert dense(q=None) == _lib.RAPT_ERR_INVALID_ARG
    assert dense(B=0) == _lib.RAPT_ERR_INVALID_ARG
    assert dense(off=-1) == _lib.RAPT_ERR_INVALID_ARG
    assert dense(out=FAKE) == _lib.RAPT_ERR_INVALID_ARG  # aliases q
    assert dense(q=FAKE_ODD) == _lib.RAPT_ERR_INVALID_ARG
    assert dense(p=_params(eps_den=0.0)) == _lib.RAPT_ERR_INVALID_ARG
    assert dense(d=128, L=4096) == _lib.RAPT_ERR_WORKSPACE  # the tensor-core path needs one
    assert dense(d=128, L=0) == _lib.RAPT_OK  # nothing to do, nothing launched

    def varlen(**kw):
        a = dict(cu=FAKE, N=2, T=16, msl=16, d=64)
        a.update(kw)
        return lib.rapt_bidir_varlen_fwd(FAKE, FAKE, FAKE, 1, a["T"], 2, a["d"], a["cu"], a["N"],
                                         a["msl"], FAKE, FAKE, _params(), out, None, None, 0, None)

    assert varlen(cu=None) == _lib.RAPT_ERR_INVALID_ARG
    assert varlen(N=0) == _lib.RAPT_ERR_INVALID_ARG
    assert varlen(msl=-1) == _lib.RAPT_ERR_INVALID_ARG
    assert varlen(d=96) == _lib.RAPT_ERR_UNSUPPORTED
    assert varlen() == _lib.RAPT_ERR_WORKSPACE
    assert lib.rapt_bidir_workspace_size(4, 4096, 16, 128, 1) > 0
    assert lib.rapt_bidir_workspace_size(4, 4096, 16, 128, 0) == 0  # fp32: CUDA-core path
    assert lib.rapt_bidir_varlen_workspace_size(65536, 17, 32, 64, 8192, 1) > 0


def test_shard_entry_points_reject_bad_arguments(lib):
    S = ctypes.c_void_p(0x7F0000003000)
    z = ctypes.c_void_p(0x7F0000004000)

    def state(**kw):
        a = dict(k=FAKE, B=2, L=256, d=128, dt=1, off=0, p=_params(), S=S, z=z, ws=FAKE, wsb=16)
        a.update(kw)
        return lib.rapt_prefill_state(a["k"], FAKE, a["dt"], a["B"], a["L"], 2, a["d"], FAKE,
                                      a["p"], a["off"], a["S"], a["z"], a["ws"], a["wsb"], None)

    assert state(d=48) == _lib.RAPT_ERR_UNSUPPORTED
    assert state(B=0) == _lib.RAPT_ERR_INVALID_ARG
    assert state(off=-1) == _lib.RAPT_ERR_INVALID_ARG
    assert state(S=None) == _lib.RAPT_ERR_INVALID_ARG
    assert state(z=FAKE_ODD) == _lib.RAPT_ERR_INVALID_ARG
    assert state(k=None) == _lib.RAPT_ERR_INVALID_ARG
    assert state(p=_params(eps_norm=-1.0)) == _lib.RAPT_ERR_INVALID_ARG
    assert state() == _lib.RAPT_ERR_WORKSPACE
    assert lib.rapt_prefill_state_workspace_size(2, 256, 2, 128, 1) >= 2 * 2 * 128 * 129 * 4
    assert lib.rapt_prefill_state_workspace_size(2, 256, 2, 48, 1) == 0

    def prefix(**kw):
        a = dict(W=4, r=2, d=64, out=S)
        a.update(kw)
        return lib.rapt_state_prefix(FAKE, FAKE_ODD if kw.get("odd") else FAKE, a["W"], a["r"], 2, 2,
                                     a["d"], None, None, a["out"], z, None)

    assert prefix(r=5) == _lib.RAPT_ERR_INVALID_ARG
    assert prefix(r=-1) == _lib.RAPT_ERR_INVALID_ARG
    assert prefix(W=0) == _lib.RAPT_ERR_INVALID_ARG
    assert prefix(d=40) == _lib.RAPT_ERR_UNSUPPORTED
    assert prefix(out=FAKE) == _lib.RAPT_ERR_INVALID_ARG  # aliases the parts
    assert prefix(odd=True) == _lib.RAPT_ERR_INVALID_ARG

    out = ctypes.c_void_p(0x7F0000002000)
    assert lib.rla_l2_moments(FAKE, FAKE, 1, 1, 64, 2, 128, None, FAKE, 1 << 40, None) == \
        _lib.RAPT_ERR_INVALID_ARG
    assert lib.rla_l2_moments(FAKE, FAKE, 1, 1, 64, 2, 128, S, FAKE, 16, None) == \
        _lib.RAPT_ERR_WORKSPACE
    assert lib.rla_l2_moments(FAKE, FAKE, 1, 1, 64, 2, 24, S, FAKE, 1 << 40, None) == \
        _lib.RAPT_ERR_UNSUPPORTED
    assert lib.rla_l2_readout(FAKE, S, 1, 1, 64, 2, 128, 0.0, out, FAKE, 1 << 40, None) == \
        _lib.RAPT_ERR_INVALID_ARG
    assert lib.rla_l2_readout(FAKE, S, 1, 1, 64, 2, 128, 1e-6, out, None, 0, None) == \
        _lib.RAPT_ERR_WORKSPACE
    assert lib.rla_l2_readout(FAKE, S, 1, 1, 0, 2, 128, 1e-6, out, None, 0, None) == _lib.RAPT_OK
    assert lib.rla_l2_readout_workspace_size(1, 64, 2, 128, 1) == 2 * 128 * 256 * 2
    assert lib.rla_l2_readout_workspace_size(1, 64, 2, 128, 0) == 0
