"""ctypes loader for the in-tree C-ABI library ``librapt.so`` (declared in include/rapt.h).

There is no fallback: if the library is missing or does not load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "librapt.so")

c_int32 = ctypes.c_int32
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p
c_float = ctypes.c_float

RAPT_OK = 0
RAPT_ERR_INVALID_ARG = 1
RAPT_ERR_UNSUPPORTED = 2
RAPT_ERR_WORKSPACE = 3
RAPT_ERR_CUDA = 4
RAPT_F32 = 0
RAPT_BF16 = 1
RAPT_DEV_BAD_CU_SEQLENS = 1
RAPT_DEV_INTERNAL = 2


class rapt_params(ctypes.Structure):
    _fields_ = [("eps_norm", c_float), ("rope_base", c_float), ("eps_den", c_float),
                ("gamma_head_stride", c_int32)]


# name -> (restype, argtypes), in the order of include/rapt.h
SIGNATURES = {
    "rapt_default_params": (rapt_params, []),
    "rapt_status_string": (ctypes.c_char_p, [c_int32]),
    "rapt_abi_version": (c_int32, []),
    "rapt_launch_counter": (ctypes.c_uint64, []),
    "rapt_prefill_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rapt_prefill_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                   c_int32, c_int32, c_int32, c_int32,
                                   c_void_p, c_void_p, rapt_params,
                                   c_int32, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rapt_prefill_host_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rapt_prefill_fwd_host": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                        c_int32, c_int32, c_int32, c_int32,
                                        c_void_p, c_void_p, rapt_params,
                                        c_int32, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                        c_void_p, c_void_p, c_void_p]),
    "rapt_varlen_workspace_size": (c_size_t, [c_int32] * 5 + [c_int32]),
    "rapt_varlen_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                  c_int32, c_int32, c_int32, c_void_p,
                                  c_int32, c_int32, c_void_p,
                                  c_void_p, rapt_params, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_size_t, c_void_p]),
    "rapt_prefill_bwd_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rapt_prefill_bwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                   c_int32, c_int32, c_int32, c_int32,
                                   c_void_p, c_void_p, rapt_params, c_int32,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_size_t, c_void_p]),
    "rapt_varlen_bwd_workspace_size": (c_size_t, [c_int32] * 5 + [c_int32]),
    "rapt_varlen_bwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                  c_int32, c_int32, c_int32, c_void_p, c_int32, c_int32,
                                  c_void_p, c_void_p, rapt_params,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_size_t, c_void_p]),
    "rla_l2_causal_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rla_l2_causal_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                    c_int32, c_int32, c_int32, c_int32, c_float, c_void_p,
                                    c_void_p, c_size_t, c_void_p]),
    "rla_l2_causal_varlen_workspace_size": (c_size_t, [c_int32] * 5 + [c_int32]),
    "rla_l2_causal_varlen_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                           c_int32, c_int32, c_int32, c_void_p, c_int32, c_int32,
                                           c_float, c_void_p, c_void_p, c_void_p, c_size_t,
                                           c_void_p]),
    "rapt_linear_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                  c_void_p, c_void_p]),
    "rapt_layer_workspace_size": (c_size_t, [c_int32] * 5),
    "rapt_layer_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                 c_int32, c_void_p, c_void_p, rapt_params, c_int32, c_void_p,
                                 c_void_p, c_void_p, c_size_t, c_void_p]),
    "rapt_bidir_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rapt_bidir_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                 c_int32, c_int32, c_int32, c_int32,
                                 c_void_p, c_void_p, rapt_params,
                                 c_int32, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rapt_bidir_varlen_workspace_size": (c_size_t, [c_int32] * 5 + [c_int32]),
    "rapt_bidir_varlen_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                        c_int32, c_int32, c_int32, c_void_p,
                                        c_int32, c_int32, c_void_p,
                                        c_void_p, rapt_params, c_void_p,
                                        c_void_p, c_void_p, c_size_t, c_void_p]),
    "rapt_decode_step": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                   c_int32, c_int32, c_int32, c_void_p,
                                   c_void_p, c_void_p, rapt_params,
                                   c_void_p, c_void_p, c_void_p, c_void_p]),
    "rla_l2_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rla_l2_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                             c_int32, c_int32, c_int32, c_int32, c_float, c_void_p,
                             c_void_p, c_size_t, c_void_p]),
    "rapt_prefill_state_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rapt_prefill_state": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                     c_int32, c_void_p, rapt_params, c_int32, c_void_p, c_void_p,
                                     c_void_p, c_size_t, c_void_p]),
    "rapt_state_prefix": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                    c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "rla_l2_moments_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rla_l2_moments": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
                                 c_void_p, c_void_p, c_size_t, c_void_p]),
    "rla_l2_readout_workspace_size": (c_size_t, [c_int32] * 4 + [c_int32]),
    "rla_l2_readout": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
                                 c_float, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rla_l2_fwd_noalloc": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32,
                                     c_int32, c_int32, c_int32, c_int32, c_float, c_void_p,
                                     c_void_p]),
}

RAPT_L2_NOALLOC_SCRATCH_BYTES = 16 << 20

_LIB = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load librapt.so once and attach the C signatures. Raises if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            "librapt.so is not built (%s); run `python -c 'import __graft_entry__ as g; g.build()'`"
            % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def status_string(code: int) -> str:
    return load().rapt_status_string(code).decode()


class RaptError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__("%s failed: %s" % (fn, status_string(code)))
        self.code = code


def check(fn: str, code: int) -> None:
    if code != RAPT_OK:
        raise RaptError(fn, code)
