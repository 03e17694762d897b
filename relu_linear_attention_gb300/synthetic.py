"""Seeded synthetic inputs for RLA-2 / RAPT causal ReLU linear attention.

This module is the only code shared by the CUDA path's tests/bench and the fp64
oracle. It draws random numbers and rounds them to the storage dtype; it holds
none of the method's arithmetic (no norm, no rotation, no ReLU, no attention).

Every array is produced by numpy's PCG64 generator from integer keys, so the
same keys give the same bits on x86 and on Arm. Large tensors are drawn in fixed
blocks of 2^22 elements; block b of tensor t under seed s comes from its own
stream PCG64(SeedSequence([s, t, b])), so the blocks can be drawn by parallel
threads and the values do not depend on the thread count. bf16 values are
returned as their raw uint16 bit patterns (round-to-nearest-even from fp32); use
``bf16_bits_to_f64`` / ``bf16_bits_to_f32`` to widen them exactly.

Workload recipes (shapes and distributions follow the method's problem
statement: q, k, v ~ N(0, 1) per element, per-head RMSNorm gains near 1,
documents of a few hundred to a few thousand tokens):

* ``tiny_fp32``      B=1, H=2, L=64, d=16, fp32, seed 0, gamma = 1.
* ``prefill_bf16``   B=4, H=16, L=4096, d=128, bf16, gamma_q, gamma_k ~ U(0.8, 1.2)
                     of shape [H, d], drawn after q, k, v from the same stream.
* ``varlen_bf16``    T=65536, H=32, d=64, bf16, document lengths ~ U{128..8192}
                     drawn until they cover T, the last one truncated; gamma = 1.
* ``decode``         N=256, H=32, d=128; 512 prefill tokens per sequence, then one
                     new bf16 token per step at positions 512, 513, ...
* ``l2_bf16``        B=2, H=16, L=16384, d=128, bf16 (original RLA, no norm/RoPE).
"""

from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

_BLOCK = 1 << 22
_POOL = None

__all__ = [
    "rng",
    "normal_f32",
    "normal_blocks",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "bf16_bits_to_f64",
    "qkv",
    "gamma_uniform",
    "doc_lengths",
    "cu_seqlens_from_lengths",
    "Workload",
    "tiny_fp32",
    "prefill_bf16",
    "varlen_bf16",
    "decode_prefix",
    "decode_step_tokens",
    "l2_bf16",
    "random_state",
]


def rng(seed: int) -> np.random.Generator:
    """numpy PCG64 stream for ``seed``."""
    return np.random.Generator(np.random.PCG64(int(seed)))


def normal_f32(g: np.random.Generator, shape) -> np.ndarray:
    """Standard normal samples drawn by numpy directly in float32 (ziggurat)."""
    return g.standard_normal(size=shape, dtype=np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits.

    Inputs are finite by construction (normal samples), so NaN handling is not needed.
    """
    # For finite x the bit pattern is at most 0xFF7FFFFF, so adding 0x8000 stays inside uint32.
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    return bf16_bits_to_f32(b).astype(np.float64)


class Workload(dict):
    """A dict of named arrays plus scalar settings; attribute access for convenience."""

    __getattr__ = dict.__getitem__


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def normal_blocks(seed: int, tensor: int, shape, dtype: str = "f32") -> np.ndarray:
    """N(0, 1) samples of ``shape``; block b (2^22 elements, row-major order) is drawn from
    PCG64(SeedSequence([seed, tensor, b])). dtype "bf16" rounds each block to bf16 bits."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(b):
        lo, hi = b * _BLOCK, min(n, (b + 1) * _BLOCK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tensor), b])))
        x = g.standard_normal(size=hi - lo, dtype=np.float32)
        out[lo:hi] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    nb = (n + _BLOCK - 1) // _BLOCK
    if nb <= 1:
        for b in range(nb):
            fill(b)
    else:
        list(_pool().map(fill, range(nb)))
    return out.reshape(shape)


def qkv(seed: int, shape, dtype: str, first_tensor: int = 0):
    """q, k, v ~ N(0, 1) of ``shape`` (tensor keys first_tensor, +1, +2 under ``seed``).

    dtype "f32" returns float32 arrays; "bf16" returns uint16 bf16 bit patterns.
    """
    return tuple(normal_blocks(seed, first_tensor + i, shape, dtype) for i in range(3))


def gamma_uniform(g: np.random.Generator, shape, lo=0.8, hi=1.2) -> np.ndarray:
    """RMSNorm gains ~ U(lo, hi), float32."""
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def doc_lengths(g: np.random.Generator, total: int, lo: int, hi: int) -> np.ndarray:
    """Integer document lengths ~ U{lo..hi} drawn until they reach ``total``; the
    last one is truncated so that the lengths sum to exactly ``total``."""
    lens = []
    s = 0
    while s < total:
        n = int(g.integers(lo, hi + 1))
        n = min(n, total - s)
        lens.append(n)
        s += n
    return np.asarray(lens, dtype=np.int64)


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    """Prefix sums [0, l0, l0+l1, ...] as int32 (N+1 entries)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


def tiny_fp32(seed: int = 0) -> Workload:
    B, L, H, d = 1, 64, 2, 16
    q, k, v = qkv(seed, (B, L, H, d), "f32")
    return Workload(q=q, k=k, v=v, dtype="f32", B=B, L=L, H=H, d=d,
                    gamma_q=np.ones(d, np.float32), gamma_k=np.ones(d, np.float32),
                    eps_norm=1e-6, rope_base=1e4, eps_den=1e-4)


def prefill_bf16(seed: int = 1, B=4, L=4096, H=16, d=128) -> Workload:
    q, k, v = qkv(seed, (B, L, H, d), "bf16")
    g = rng(seed)
    gq = gamma_uniform(g, (H, d))
    gk = gamma_uniform(g, (H, d))
    return Workload(q=q, k=k, v=v, dtype="bf16", B=B, L=L, H=H, d=d,
                    gamma_q=gq, gamma_k=gk, eps_norm=1e-6, rope_base=1e4, eps_den=1e-4)


def varlen_bf16(seed: int = 2, T=65536, H=32, d=64, lo=128, hi=8192) -> Workload:
    lens = doc_lengths(rng(seed), T, lo, hi)
    q, k, v = qkv(seed, (T, H, d), "bf16")
    return Workload(q=q, k=k, v=v, dtype="bf16", T=T, H=H, d=d,
                    cu_seqlens=cu_seqlens_from_lengths(lens), lengths=lens,
                    gamma_q=np.ones(d, np.float32), gamma_k=np.ones(d, np.float32),
                    eps_norm=1e-6, rope_base=1e4, eps_den=1e-4)


def decode_prefix(seed: int = 3, N=256, P=512, H=32, d=128) -> Workload:
    """The P prefill tokens of every decode sequence, as a dense [N, P, H, d] batch."""
    q, k, v = qkv(seed, (N, P, H, d), "bf16")
    return Workload(q=q, k=k, v=v, dtype="bf16", B=N, L=P, H=H, d=d,
                    gamma_q=np.ones(d, np.float32), gamma_k=np.ones(d, np.float32),
                    eps_norm=1e-6, rope_base=1e4, eps_den=1e-4)


def decode_step_tokens(seed: int = 3, step: int = 0, N=256, H=32, d=128, P=512) -> Workload:
    """The new token of every sequence for decode step ``step`` (position P + step)."""
    q, k, v = qkv(seed, (N, H, d), "bf16", first_tensor=3 * (int(step) + 1))
    return Workload(q=q, k=k, v=v, dtype="bf16", N=N, H=H, d=d,
                    positions=np.full(N, P + step, dtype=np.int32))


def l2_bf16(seed: int = 4, B=2, L=16384, H=16, d=128) -> Workload:
    q, k, v = qkv(seed, (B, L, H, d), "bf16")
    return Workload(q=q, k=k, v=v, dtype="bf16", B=B, L=L, H=H, d=d, eps=1e-6)


def random_state(seed: int, shape_S, shape_z):
    """An arbitrary carried-over state for tests: S ~ N(0, 1) fp32, z ~ |N(0, 1)| * 4
    fp32 (z is a sum of non-negative features, so it is drawn non-negative)."""
    S = normal_blocks(seed, 100, shape_S)
    z = np.abs(normal_blocks(seed, 101, shape_z)) * np.float32(4.0)
    return S, z
