"""Helpers for GPU parity tests: seeded numpy inputs -> device tensors, outputs -> fp64."""

import numpy as np
import torch

from relu_linear_attention_gb300 import synthetic as syn

TOL = {"f32": 1e-4, "bf16": 2e-2}  # max per-row relative error vs the fp64 oracle


def to_dev(x, dtype, device="cuda"):
    """numpy fp32 array ("f32") or uint16 bf16 bit pattern ("bf16") -> device tensor."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device)


def widen(x, dtype):
    """The exact fp64 values of the stored inputs (what the oracle receives)."""
    return syn.bf16_bits_to_f64(x) if dtype == "bf16" else np.asarray(x, dtype=np.float64)


def to_host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def draw(seed, shape, dtype):
    return syn.qkv(seed, shape, dtype)


def gammas(seed, H, d, per_head):
    g = syn.rng(seed)
    shape = (H, d) if per_head else (d,)
    return syn.gamma_uniform(g, shape), syn.gamma_uniform(g, shape)
