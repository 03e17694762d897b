"""Thin PyTorch binding of the C ABI in include/rapt.h (same function names).

Argument marshalling only: shapes, dtypes, devices and contiguity of torch tensors are checked,
outputs / workspaces are allocated with torch when the caller does not pass them, and the raw
device pointers plus the current CUDA stream go to librapt.so. Every step of the computation runs
in the library's CUDA kernels; there is no CPU path and no fallback.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib

_DT = {torch.float32: _lib.RAPT_F32, torch.bfloat16: _lib.RAPT_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(name, t, dtype=None, shape=None):
    _need(t.is_cuda, "%s must be a CUDA tensor" % name)
    _need(t.is_contiguous(), "%s must be contiguous" % name)
    if dtype is not None:
        _need(t.dtype == dtype, "%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None:
        _need(tuple(t.shape) == tuple(shape), "%s must have shape %s, got %s"
              % (name, tuple(shape), tuple(t.shape)))


def make_params(eps_norm=1e-6, rope_base=1e4, eps_den=1e-4, gamma_head_stride=0):
    p = _lib.rapt_params()
    p.eps_norm, p.rope_base, p.eps_den = float(eps_norm), float(rope_base), float(eps_den)
    p.gamma_head_stride = int(gamma_head_stride)
    return p


def _gammas(gamma_q, gamma_k, H, d):
    for name, g in (("gamma_q", gamma_q), ("gamma_k", gamma_k)):
        _cuda_contig(name, g, torch.float32)
        _need(tuple(g.shape) in ((d,), (H, d)), "%s must be [d] or [H, d]" % name)
    _need(gamma_q.dim() == gamma_k.dim(), "gamma_q and gamma_k must have the same shape")
    return 0 if gamma_q.dim() == 1 else d


def _state(name, t, shape):
    if t is not None:
        _cuda_contig(name, t, torch.float32, shape)
    return t


def rapt_prefill_fwd(q, k, v, gamma_q, gamma_k, *, eps_norm=1e-6, rope_base=1e4, eps_den=1e-4,
                     pos_offset=0, S0=None, z0=None, out=None, final_state=False, S_final=None,
                     z_final=None, dev_status=None, workspace=None, stream=None):
    """Dense causal RLA-2 prefill; q, k, v [B, L, H, d] (fp32 or bf16). Returns
    (out, S_final, z_final); the final state is None unless requested or passed."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    stride = _gammas(gamma_q, gamma_k, H, d)
    _state("S0", S0, (B, H, d, d))
    _state("z0", z0, (B, H, d))
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    if final_state and S_final is None:
        S_final = torch.empty((B, H, d, d), device=q.device, dtype=torch.float32)
    if final_state and z_final is None:
        z_final = torch.empty((B, H, d), device=q.device, dtype=torch.float32)
    _state("S_final", S_final, (B, H, d, d))
    _state("z_final", z_final, (B, H, d))
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_prefill_workspace_size(B, L, H, d, _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], B, L, H, d,
                              _ptr(gamma_q), _ptr(gamma_k),
                              make_params(eps_norm, rope_base, eps_den, stride), int(pos_offset),
                              _ptr(S0), _ptr(z0), _ptr(out), _ptr(S_final), _ptr(z_final),
                              _ptr(dev_status), _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rapt_prefill_fwd", st)
    return out, S_final, z_final


def rapt_prefill_fwd_host(q, k, v, gamma_q, gamma_k, *, out=None, eps_norm=1e-6, rope_base=1e4,
                          eps_den=1e-4, pos_offset=0, S0=None, z0=None, final_state=False,
                          S_final=None, z_final=None, dev_status=None, workspace=None, device=None,
                          stream=None, copy_in=None, copy_out=None):
    """rapt_prefill_fwd with q, k, v and out in host memory (CPU tensors, page-locked for full
    speed): the batch rows are copied in, computed and copied out in a pipeline over three CUDA
    streams (copy_in and copy_out default to the compute stream, which then overlaps nothing).
    gammas and states are CUDA tensors. Returns (out, S_final, z_final); out is complete once
    `stream` (default: the current stream) is synchronised."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(not t.is_cuda, "%s must be a host tensor" % name)
        _need(t.is_contiguous() and t.dtype == q.dtype and tuple(t.shape) == tuple(q.shape),
              "%s must be contiguous with q's dtype and shape" % name)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    dev = gamma_q.device if device is None else torch.device(device)
    stride = _gammas(gamma_q, gamma_k, H, d)
    _state("S0", S0, (B, H, d, d))
    _state("z0", z0, (B, H, d))
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    _need(not out.is_cuda and out.is_contiguous() and out.dtype == q.dtype and
          tuple(out.shape) == tuple(q.shape), "out must be a contiguous host tensor like q")
    if final_state and S_final is None:
        S_final = torch.empty((B, H, d, d), device=dev, dtype=torch.float32)
    if final_state and z_final is None:
        z_final = torch.empty((B, H, d), device=dev, dtype=torch.float32)
    _state("S_final", S_final, (B, H, d, d))
    _state("z_final", z_final, (B, H, d))
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_prefill_host_workspace_size(B, L, H, d, _DT[q.dtype])
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.rapt_prefill_fwd_host(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], B, L, H, d,
                                   _ptr(gamma_q), _ptr(gamma_k),
                                   make_params(eps_norm, rope_base, eps_den, stride),
                                   int(pos_offset), _ptr(S0), _ptr(z0), _ptr(out), _ptr(S_final),
                                   _ptr(z_final), _ptr(dev_status), _ptr(workspace), ws_bytes,
                                   _stream(stream), _stream(copy_in if copy_in is not None else stream),
                                   _stream(copy_out if copy_out is not None else stream))
    _lib.check("rapt_prefill_fwd_host", st)
    return out, S_final, z_final


def rapt_varlen_fwd(q, k, v, cu_seqlens, gamma_q, gamma_k, *, max_seqlen, eps_norm=1e-6,
                    rope_base=1e4, eps_den=1e-4, S0=None, z0=None, out=None, final_state=False,
                    S_final=None, z_final=None, dev_status=None, workspace=None, stream=None):
    """Packed varlen causal RLA-2; q, k, v [T, H, d]; cu_seqlens int32 [N + 1] on the device.
    Returns (out, S_final, z_final)."""
    _need(q.dim() == 3, "q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    _cuda_contig("cu_seqlens", cu_seqlens, torch.int32)
    _need(cu_seqlens.dim() == 1 and cu_seqlens.numel() >= 2, "cu_seqlens must be [N + 1]")
    N = cu_seqlens.numel() - 1
    stride = _gammas(gamma_q, gamma_k, H, d)
    _state("S0", S0, (N, H, d, d))
    _state("z0", z0, (N, H, d))
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    if final_state and S_final is None:
        S_final = torch.empty((N, H, d, d), device=q.device, dtype=torch.float32)
    if final_state and z_final is None:
        z_final = torch.empty((N, H, d), device=q.device, dtype=torch.float32)
    _state("S_final", S_final, (N, H, d, d))
    _state("z_final", z_final, (N, H, d))
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_varlen_workspace_size(T, N, H, d, int(max_seqlen), _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], T, H, d, _ptr(cu_seqlens),
                             N, int(max_seqlen), _ptr(gamma_q), _ptr(gamma_k),
                             make_params(eps_norm, rope_base, eps_den, stride), _ptr(S0), _ptr(z0),
                             _ptr(out), _ptr(S_final), _ptr(z_final), _ptr(dev_status),
                             _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rapt_varlen_fwd", st)
    return out, S_final, z_final


def _bwd_outputs(q, gamma_q, dq, dk, dv, dgamma_q, dgamma_k, need_gains):
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _cuda_contig(name, t, q.dtype, q.shape)
    if need_gains:
        dgamma_q = torch.empty_like(gamma_q) if dgamma_q is None else dgamma_q
        dgamma_k = torch.empty_like(gamma_q) if dgamma_k is None else dgamma_k
    for name, t in (("dgamma_q", dgamma_q), ("dgamma_k", dgamma_k)):
        if t is not None:
            _cuda_contig(name, t, torch.float32, gamma_q.shape)
    return dq, dk, dv, dgamma_q, dgamma_k


def rapt_prefill_bwd(q, k, v, dout, gamma_q, gamma_k, *, eps_norm=1e-6, rope_base=1e4,
                     eps_den=1e-4, pos_offset=0, dq=None, dk=None, dv=None, dgamma_q=None,
                     dgamma_k=None, need_gains=True, workspace=None, stream=None):
    """Backward of the dense causal prefill: q, k, v, dout [B, L, H, d] (fp32 or bf16).
    Returns (dq, dk, dv, dgamma_q, dgamma_k); the gain gradients are None when need_gains is
    False and none is given."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    stride = _gammas(gamma_q, gamma_k, H, d)
    dq, dk, dv, dgamma_q, dgamma_k = _bwd_outputs(q, gamma_q, dq, dk, dv, dgamma_q, dgamma_k,
                                                  need_gains)
    lib = _lib.load()
    need = lib.rapt_prefill_bwd_workspace_size(B, L, H, d, _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_prefill_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _DT[q.dtype], B, L, H, d,
                              _ptr(gamma_q), _ptr(gamma_k),
                              make_params(eps_norm, rope_base, eps_den, stride), int(pos_offset),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgamma_q), _ptr(dgamma_k),
                              _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rapt_prefill_bwd", st)
    return dq, dk, dv, dgamma_q, dgamma_k


def rapt_varlen_bwd(q, k, v, dout, cu_seqlens, gamma_q, gamma_k, *, max_seqlen, eps_norm=1e-6,
                    rope_base=1e4, eps_den=1e-4, dq=None, dk=None, dv=None, dgamma_q=None,
                    dgamma_k=None, need_gains=True, dev_status=None, workspace=None, stream=None):
    """Backward of the packed varlen causal forward: q, k, v, dout [T, H, d]; cu_seqlens int32
    [N + 1] on the device. Returns (dq, dk, dv, dgamma_q, dgamma_k)."""
    _need(q.dim() == 3, "q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    _cuda_contig("cu_seqlens", cu_seqlens, torch.int32)
    _need(cu_seqlens.dim() == 1 and cu_seqlens.numel() >= 2, "cu_seqlens must be [N + 1]")
    N = cu_seqlens.numel() - 1
    stride = _gammas(gamma_q, gamma_k, H, d)
    dq, dk, dv, dgamma_q, dgamma_k = _bwd_outputs(q, gamma_q, dq, dk, dv, dgamma_q, dgamma_k,
                                                  need_gains)
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_varlen_bwd_workspace_size(T, N, H, d, int(max_seqlen), _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _DT[q.dtype], T, H, d,
                             _ptr(cu_seqlens), N, int(max_seqlen), _ptr(gamma_q), _ptr(gamma_k),
                             make_params(eps_norm, rope_base, eps_den, stride),
                             _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgamma_q), _ptr(dgamma_k),
                             _ptr(dev_status), _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rapt_varlen_bwd", st)
    return dq, dk, dv, dgamma_q, dgamma_k


def rla_l2_causal_fwd(q, k, v, *, eps=1e-6, out=None, workspace=None, stream=None):
    """Causal original RLA (L2 denominator): q, k, v [B, L, H, d] (fp32 or bf16). Returns out."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    lib = _lib.load()
    need = lib.rla_l2_causal_workspace_size(B, L, H, d, _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rla_l2_causal_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], B, L, H, d, float(eps),
                               _ptr(out), _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rla_l2_causal_fwd", st)
    return out


def rla_l2_causal_varlen_fwd(q, k, v, cu_seqlens, *, max_seqlen, eps=1e-6, out=None,
                             dev_status=None, workspace=None, stream=None):
    """Packed varlen causal original RLA: q, k, v [T, H, d]; cu_seqlens int32 [N + 1] on the
    device. Returns out."""
    _need(q.dim() == 3, "q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    _cuda_contig("cu_seqlens", cu_seqlens, torch.int32)
    _need(cu_seqlens.dim() == 1 and cu_seqlens.numel() >= 2, "cu_seqlens must be [N + 1]")
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rla_l2_causal_varlen_workspace_size(T, N, H, d, int(max_seqlen), _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rla_l2_causal_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], T, H, d,
                                      _ptr(cu_seqlens), N, int(max_seqlen), float(eps), _ptr(out),
                                      _ptr(dev_status), _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rla_l2_causal_varlen_fwd", st)
    return out


def rapt_linear_fwd(x, w, *, out=None, dev_status=None, stream=None):
    """y = x W^T on the tensor cores: x [M, K] bf16, w [N, K] bf16. Returns y [M, N] bf16."""
    _need(x.dim() == 2 and w.dim() == 2 and x.shape[1] == w.shape[1], "x [M, K], w [N, K]")
    M, K = x.shape
    N = w.shape[0]
    _cuda_contig("x", x, torch.bfloat16, x.shape)
    _cuda_contig("w", w, torch.bfloat16, w.shape)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda_contig("out", out, torch.bfloat16, (M, N))
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    st = _lib.load().rapt_linear_fwd(_ptr(x), _ptr(w), _ptr(out), M, N, K, _ptr(dev_status),
                                     _stream(stream))
    _lib.check("rapt_linear_fwd", st)
    return out


def rapt_layer_fwd(x, w_qkv, w_o, gamma_q, gamma_k, *, heads, eps_norm=1e-6, rope_base=1e4,
                   eps_den=1e-4, pos_offset=0, out=None, dev_status=None, workspace=None,
                   stream=None):
    """One RAPT attention layer: x [B, L, d_model] bf16, w_qkv [3 H d, d_model], w_o [d_model, H d].
    Returns y [B, L, d_model] bf16."""
    _need(x.dim() == 3, "x must be [B, L, d_model]")
    B, L, dm = x.shape
    H = int(heads)
    _need(w_qkv.dim() == 2 and w_qkv.shape[1] == dm and w_qkv.shape[0] % (3 * H) == 0,
          "w_qkv must be [3 H d, d_model]")
    d = w_qkv.shape[0] // (3 * H)
    _need(tuple(w_o.shape) == (dm, H * d), "w_o must be [d_model, H d]")
    for name, t in (("x", x), ("w_qkv", w_qkv), ("w_o", w_o)):
        _cuda_contig(name, t, torch.bfloat16, t.shape)
    stride = _gammas(gamma_q, gamma_k, H, d)
    if out is None:
        out = torch.empty_like(x)
    _cuda_contig("out", out, torch.bfloat16, x.shape)
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_layer_workspace_size(B, L, H, d, dm)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=x.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_layer_fwd(_ptr(x), _ptr(w_qkv), _ptr(w_o), B, L, H, d, dm, _ptr(gamma_q),
                            _ptr(gamma_k), make_params(eps_norm, rope_base, eps_den, stride),
                            int(pos_offset), _ptr(out), _ptr(dev_status), _ptr(workspace), ws_bytes,
                            _stream(stream))
    _lib.check("rapt_layer_fwd", st)
    return out


def rapt_bidir_fwd(q, k, v, gamma_q, gamma_k, *, eps_norm=1e-6, rope_base=1e4, eps_den=1e-4,
                   pos_offset=0, out=None, dev_status=None, workspace=None, stream=None):
    """Dense bidirectional (non-causal) RLA-2; q, k, v [B, L, H, d] (fp32 or bf16). Returns out."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    stride = _gammas(gamma_q, gamma_k, H, d)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_bidir_workspace_size(B, L, H, d, _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_bidir_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], B, L, H, d,
                            _ptr(gamma_q), _ptr(gamma_k),
                            make_params(eps_norm, rope_base, eps_den, stride), int(pos_offset),
                            _ptr(out), _ptr(dev_status), _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rapt_bidir_fwd", st)
    return out


def rapt_bidir_varlen_fwd(q, k, v, cu_seqlens, gamma_q, gamma_k, *, max_seqlen, eps_norm=1e-6,
                          rope_base=1e4, eps_den=1e-4, out=None, dev_status=None, workspace=None,
                          stream=None):
    """Packed varlen bidirectional RLA-2; q, k, v [T, H, d]; cu_seqlens int32 [N + 1] on the
    device. Returns out."""
    _need(q.dim() == 3, "q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    _cuda_contig("cu_seqlens", cu_seqlens, torch.int32)
    _need(cu_seqlens.dim() == 1 and cu_seqlens.numel() >= 2, "cu_seqlens must be [N + 1]")
    N = cu_seqlens.numel() - 1
    stride = _gammas(gamma_q, gamma_k, H, d)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    if dev_status is not None:
        _cuda_contig("dev_status", dev_status, torch.int32)
    lib = _lib.load()
    need = lib.rapt_bidir_varlen_workspace_size(T, N, H, d, int(max_seqlen), _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rapt_bidir_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], T, H, d,
                                   _ptr(cu_seqlens), N, int(max_seqlen), _ptr(gamma_q),
                                   _ptr(gamma_k), make_params(eps_norm, rope_base, eps_den, stride),
                                   _ptr(out), _ptr(dev_status), _ptr(workspace), ws_bytes,
                                   _stream(stream))
    _lib.check("rapt_bidir_varlen_fwd", st)
    return out


def rapt_decode_step(q, k, v, positions, gamma_q, gamma_k, S, z, *, eps_norm=1e-6, rope_base=1e4,
                     eps_den=1e-4, out=None, stream=None):
    """One decode step; q, k, v [N, H, d]; positions int32 [N]; S [N, H, d, d] and z [N, H, d]
    fp32 are updated in place. Returns out [N, H, d]."""
    _need(q.dim() == 3, "q must be [N, H, d]")
    N, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    _cuda_contig("positions", positions, torch.int32, (N,))
    stride = _gammas(gamma_q, gamma_k, H, d)
    _cuda_contig("S", S, torch.float32, (N, H, d, d))
    _cuda_contig("z", z, torch.float32, (N, H, d))
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    st = _lib.load().rapt_decode_step(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], N, H, d,
                                      _ptr(positions), _ptr(gamma_q), _ptr(gamma_k),
                                      make_params(eps_norm, rope_base, eps_den, stride),
                                      _ptr(S), _ptr(z), _ptr(out), _stream(stream))
    _lib.check("rapt_decode_step", st)
    return out


def rla_l2_fwd(q, k, v, *, eps=1e-6, out=None, workspace=None, stream=None):
    """Original RLA, non-causal, L2 denominator; q, k, v [B, L, H, d]. Returns out."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_contig(name, t, q.dtype, q.shape)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    lib = _lib.load()
    need = lib.rla_l2_workspace_size(B, L, H, d, _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rla_l2_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], B, L, H, d, float(eps), _ptr(out),
                        _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rla_l2_fwd", st)
    return out


# ---------------------------------------------------------------- one sequence split across GPUs
def rapt_prefill_state(k, v, gamma_k, *, eps_norm=1e-6, rope_base=1e4, pos_offset=0, S_inc=None,
                       z_inc=None, workspace=None, stream=None):
    """State increment of a shard: S_inc = sum_t k'_t v_t^T, z_inc = sum_t k'_t over the L tokens of
    every batch row of k, v [B, L, H, d] (token t at RoPE position pos_offset + t). Returns
    (S_inc [B, H, d, d], z_inc [B, H, d]) in fp32."""
    _need(k.dim() == 4, "k must be [B, L, H, d]")
    B, L, H, d = k.shape
    for name, t in (("k", k), ("v", v)):
        _cuda_contig(name, t, k.dtype, k.shape)
    _need(k.dtype in _DT, "dtype must be float32 or bfloat16")
    stride = _gammas(gamma_k, gamma_k, H, d)
    if S_inc is None:
        S_inc = torch.empty((B, H, d, d), device=k.device, dtype=torch.float32)
    if z_inc is None:
        z_inc = torch.empty((B, H, d), device=k.device, dtype=torch.float32)
    _state("S_inc", S_inc, (B, H, d, d))
    _state("z_inc", z_inc, (B, H, d))
    lib = _lib.load()
    need = lib.rapt_prefill_state_workspace_size(B, L, H, d, _DT[k.dtype])
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=k.device, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.rapt_prefill_state(_ptr(k), _ptr(v), _DT[k.dtype], B, L, H, d, _ptr(gamma_k),
                                make_params(eps_norm, rope_base, 1e-4, stride), int(pos_offset),
                                _ptr(S_inc), _ptr(z_inc), _ptr(workspace), ws_bytes,
                                _stream(stream))
    _lib.check("rapt_prefill_state", st)
    return S_inc, z_inc


def rapt_state_prefix(S_parts, z_parts, r, *, S0=None, z0=None, S_start=None, z_start=None,
                      stream=None):
    """S_start = S0 + S_parts[0] + ... + S_parts[r-1] (and z likewise), in rank order, for the
    gathered shard increments S_parts [W, B, H, d, d], z_parts [W, B, H, d]."""
    _need(S_parts.dim() == 5, "S_parts must be [W, B, H, d, d]")
    W, B, H, d, _ = S_parts.shape
    _cuda_contig("S_parts", S_parts, torch.float32)
    _cuda_contig("z_parts", z_parts, torch.float32, (W, B, H, d))
    _state("S0", S0, (B, H, d, d))
    _state("z0", z0, (B, H, d))
    if S_start is None:
        S_start = torch.empty((B, H, d, d), device=S_parts.device, dtype=torch.float32)
    if z_start is None:
        z_start = torch.empty((B, H, d), device=S_parts.device, dtype=torch.float32)
    _state("S_start", S_start, (B, H, d, d))
    _state("z_start", z_start, (B, H, d))
    st = _lib.load().rapt_state_prefix(_ptr(S_parts), _ptr(z_parts), W, int(r), B, H, d, _ptr(S0),
                                       _ptr(z0), _ptr(S_start), _ptr(z_start), _stream(stream))
    _lib.check("rapt_state_prefix", st)
    return S_start, z_start


def gather_shard_states(S_inc, z_inc, group=None):
    """All-gathers every rank's shard increment, in rank order: returns (S_parts [W, ...],
    z_parts [W, ...]). Without an initialised process group (or with one rank) W = 1."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return S_inc.unsqueeze(0), z_inc.unsqueeze(0)
    W = dist.get_world_size(group)
    out = []
    for t in (S_inc.contiguous(), z_inc.contiguous()):
        # gathered along the leading axis (rank r's tensor at rows [r n, (r + 1) n)), then viewed
        # as [W, ...]
        g = torch.empty((W * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        dist.all_gather_into_tensor(g, t, group=group)
        out.append(g.view((W,) + tuple(t.shape)))
    return out[0], out[1]


def shard_rank(group=None):
    """(rank, world size) of this process in ``group`` ((0, 1) without a process group)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return 0, 1
    return dist.get_rank(group), dist.get_world_size(group)


def rapt_prefill_fwd_sharded(q, k, v, gamma_q, gamma_k, *, group=None, eps_norm=1e-6,
                             rope_base=1e4, eps_den=1e-4, pos_offset=0, S0=None, z0=None,
                             out=None, final_state=False, stream=None):
    """Causal RLA-2 prefill of sequences split across the ranks of ``group``: rank r holds tokens
    [r L, (r + 1) L) of every batch row in q, k, v [B, L, H, d] (equal L on every rank; pos_offset
    is the position of rank 0's first token). One all-gather of the shard states is the only
    exchange. Returns (out, S_final, z_final) with the final state of the whole sequence when
    requested (the same on every rank)."""
    r, W = shard_rank(group)
    B, L, H, d = q.shape
    first = int(pos_offset) + r * L
    S_inc, z_inc = rapt_prefill_state(k, v, gamma_k, eps_norm=eps_norm, rope_base=rope_base,
                                      pos_offset=first, stream=stream)
    S_parts, z_parts = gather_shard_states(S_inc, z_inc, group)
    S_start, z_start = rapt_state_prefix(S_parts, z_parts, r, S0=S0, z0=z0, stream=stream)
    out, _, _ = rapt_prefill_fwd(q, k, v, gamma_q, gamma_k, eps_norm=eps_norm, rope_base=rope_base,
                                 eps_den=eps_den, pos_offset=first, S0=S_start, z0=z_start, out=out,
                                 stream=stream)
    S_fin = z_fin = None
    if final_state:
        S_fin, z_fin = rapt_state_prefix(S_parts, z_parts, W, S0=S0, z0=z0, stream=stream)
    return out, S_fin, z_fin


def rla_l2_moments(k, v, *, M=None, workspace=None, stream=None):
    """The moments [M_V | M_K] = K'^T [V | K'] (k' = ReLU(k)) over the L tokens of k, v
    [B, L, H, d]: fp32 [B, H, d, 2d]."""
    _need(k.dim() == 4, "k must be [B, L, H, d]")
    B, L, H, d = k.shape
    for name, t in (("k", k), ("v", v)):
        _cuda_contig(name, t, k.dtype, k.shape)
    _need(k.dtype in _DT, "dtype must be float32 or bfloat16")
    if M is None:
        M = torch.empty((B, H, d, 2 * d), device=k.device, dtype=torch.float32)
    _state("M", M, (B, H, d, 2 * d))
    lib = _lib.load()
    need = lib.rla_l2_moments_workspace_size(B, L, H, d, _DT[k.dtype])
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=k.device, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.rla_l2_moments(_ptr(k), _ptr(v), _DT[k.dtype], B, L, H, d, _ptr(M), _ptr(workspace),
                            ws_bytes, _stream(stream))
    _lib.check("rla_l2_moments", st)
    return M


def rla_l2_readout(q, M, *, eps=1e-6, out=None, workspace=None, stream=None):
    """out = q'M_V / (sqrt(q'^T M_K q') + eps), q' = ReLU(q), for q [B, L, H, d] and the moments
    M [B, H, d, 2d] (fp32)."""
    _need(q.dim() == 4, "q must be [B, L, H, d]")
    B, L, H, d = q.shape
    _cuda_contig("q", q, None, None)
    _need(q.dtype in _DT, "dtype must be float32 or bfloat16")
    _state("M", M, (B, H, d, 2 * d))
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype, q.shape)
    lib = _lib.load()
    need = lib.rla_l2_readout_workspace_size(B, L, H, d, _DT[q.dtype])
    if need > 0 and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.rla_l2_readout(_ptr(q), _ptr(M), _DT[q.dtype], B, L, H, d, float(eps), _ptr(out),
                            _ptr(workspace), ws_bytes, _stream(stream))
    _lib.check("rla_l2_readout", st)
    return out


def allreduce_moments(M, group=None):
    """Sums the moments over the ranks of ``group`` in place (the identity without one)."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(M, op=dist.ReduceOp.SUM, group=group)
    return M


def rla_l2_fwd_sharded(q, k, v, *, group=None, eps=1e-6, out=None, stream=None):
    """Non-causal L2 of sequences whose tokens are split across the ranks of ``group`` (rank r
    holds its own tokens of q, k, v [B, L, H, d]): the moments of every shard are summed by one
    all-reduce, then every rank reads out its own queries. Returns out for this rank's tokens."""
    M = rla_l2_moments(k, v, stream=stream)
    allreduce_moments(M, group)
    return rla_l2_readout(q, M, eps=eps, out=out, stream=stream)
