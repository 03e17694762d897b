"""Plain fp64 backward of causal RLA-2 / RAPT (gradients of a scalar loss through the layer).

Test infrastructure only (see the package docstring). The loss is L = sum_t dout_t . out_t for a
given upstream gradient ``dout``; the functions return dL/dq, dL/dk, dL/dv and dL/dgamma_q,
dL/dgamma_k. The steps follow the order the RLA page (08-rapt-algorithm.md §4.2, "backward: one
prefix scan and two suffix scans") gives, each written here in its quadratic O(L^2) form:

1. the forward quantities of every query: num_t = sum_{tau<=t} s_{t,tau} v_tau and
   den_t = sum_{tau<=t} s_{t,tau} + eps (the main scan and the z-scan);
2. gnum_t = g_t / den_t and scale_t = -(g_t . num_t) / den_t^2, and the gradient of q'_t,
   sum_{tau<=t} k'_tau (v_tau . gnum_t + scale_t)  (= S_t gnum_t + scale_t z_t);
3. the suffix sums over the queries that see a key: dv_tau = sum_{t>=tau} s_{t,tau} gnum_t and
   dk'_tau = sum_{t>=tau} q'_t (gnum_t . v_tau + scale_t);
4. back through the feature map: the ReLU mask (select y > 0), the inverse RoPE rotation, then
   RMSNorm (gradients of the input and of the gain).

Every sum runs inside one document (the state restarts at document boundaries, §2.2, §4.1).
"""

from __future__ import annotations

import numpy as np

from .rla2 import _f64, _gamma_h, rmsnorm, rope_adjacent


def relu_bwd(y, dy):
    """Gradient through max(0, y): passes where y > 0, zero elsewhere (the page's select(Qp > 0))."""
    return np.where(_f64(y) > 0.0, _f64(dy), 0.0)


def rope_adjacent_bwd(dy, positions, base):
    """Gradient through the adjacent-pair RoPE: each pair's rotation is orthogonal, so the gradient
    is rotated back by the same angle (the transpose of the rotation = rotation by -a)."""
    return rope_adjacent(dy, -_f64(positions), base)


def rmsnorm_bwd(x, gamma, eps, dy):
    """Gradient through y = x * r * gamma, r = (mean(x^2) + eps)^(-1/2), over the last axis.

    Returns (dx, dgamma_rows) with dgamma_rows = dy * x * r per row (the caller sums the rows).
    d r / d x_i = -r^3 x_i / d, so dx = r gamma dy - x r^3 (sum_j gamma_j dy_j x_j) / d.
    """
    x, dy, g = _f64(x), _f64(dy), _f64(gamma)
    d = x.shape[-1]
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(eps))
    dot = np.sum(g * dy * x, axis=-1, keepdims=True)
    dx = r * g * dy - x * (r ** 3) * dot / d
    return dx, dy * x * r


def features_bwd(x, gamma, positions, eps_norm, rope_base, df):
    """Gradient through f = ReLU(RoPE(RMSNorm(x))) for one head: x, df [n, d], gamma [d].

    Returns (dx [n, d], dgamma [d]) (dgamma summed over the n rows).
    """
    x = _f64(x)
    y = rope_adjacent(rmsnorm(x, gamma, eps_norm), positions, rope_base)
    dy = relu_bwd(y, df)
    dyn = rope_adjacent_bwd(dy, positions, rope_base)
    dx, dg_rows = rmsnorm_bwd(x, gamma, eps_norm, dyn)
    return dx, dg_rows.sum(axis=0)


def rla2_causal_doc_bwd(qf, kf, v, dout, eps_den=1e-4):
    """Gradients of L = sum_t dout_t . out_t w.r.t. q', k' and v of one head of one document.

    qf, kf, v, dout: [n, d]. Quadratic form of steps 1-3 of the module docstring. Returns
    (dqf, dkf, dv), each [n, d].
    """
    qf, kf, v, g = _f64(qf), _f64(kf), _f64(v), _f64(dout)
    n = qf.shape[0]
    causal = np.arange(n)[None, :] <= np.arange(n)[:, None]  # [t, tau]: tau <= t
    s = np.where(causal, qf @ kf.T, 0.0)
    num = s @ v
    den = s.sum(axis=1) + float(eps_den)
    gnum = g / den[:, None]
    scale = -np.sum(g * num, axis=1) / den ** 2
    a = np.where(causal, gnum @ v.T + scale[:, None], 0.0)  # a[t, tau] = gnum_t . v_tau + scale_t
    dqf = a @ kf
    dkf = a.T @ qf
    dv = s.T @ gnum
    return dqf, dkf, dv


def rla2_prefill_bwd(q, k, v, dout, gamma_q, gamma_k, eps_norm=1e-6, rope_base=1e4,
                     eps_den=1e-4, pos_offset=0):
    """Backward of the dense causal prefill: q, k, v, dout [B, L, H, d]; token t of each batch row
    at RoPE position pos_offset + t; one document per batch row; no carried-in state.

    Returns (dq, dk, dv) [B, L, H, d] and (dgamma_q, dgamma_k) with gamma's shape ([d] shared by
    the heads: summed over heads too; [H, d]: per head).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, L, H, d = q.shape
    cu = np.arange(B + 1, dtype=np.int64) * L
    r = rla2_varlen_bwd(q.reshape(B * L, H, d), k.reshape(B * L, H, d), v.reshape(B * L, H, d),
                        dout.reshape(B * L, H, d), cu, gamma_q, gamma_k, eps_norm, rope_base,
                        eps_den, pos_offset=pos_offset)
    dq, dk, dv = (x.reshape(B, L, H, d) for x in r[:3])
    return dq, dk, dv, r[3], r[4]


def rla2_varlen_bwd(q, k, v, dout, cu_seqlens, gamma_q, gamma_k, eps_norm=1e-6, rope_base=1e4,
                    eps_den=1e-4, pos_offset=0):
    """Backward of the packed varlen causal prefill: q, k, v, dout [T, H, d]; document n spans
    tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 at RoPE positions pos_offset + 0, 1, ...

    Returns (dq, dk, dv) [T, H, d] and (dgamma_q, dgamma_k) shaped like the gains.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, H, d = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dgq = np.zeros(np.shape(gamma_q))
    dgk = np.zeros(np.shape(gamma_k))
    for n in range(len(cu) - 1):
        a, b = int(cu[n]), int(cu[n + 1])
        if b == a:
            continue
        pos = pos_offset + np.arange(b - a)
        for h in range(H):
            gq, gk = _gamma_h(gamma_q, h), _gamma_h(gamma_k, h)
            yq = rope_adjacent(rmsnorm(q[a:b, h], gq, eps_norm), pos, rope_base)
            yk = rope_adjacent(rmsnorm(k[a:b, h], gk, eps_norm), pos, rope_base)
            qf, kf = np.maximum(yq, 0.0), np.maximum(yk, 0.0)
            dqf, dkf, dv[a:b, h] = rla2_causal_doc_bwd(qf, kf, v[a:b, h], dout[a:b, h], eps_den)
            dq[a:b, h], gq_h = features_bwd(q[a:b, h], gq, pos, eps_norm, rope_base, dqf)
            dk[a:b, h], gk_h = features_bwd(k[a:b, h], gk, pos, eps_norm, rope_base, dkf)
            if dgq.ndim == 2:
                dgq[h] += gq_h
            else:
                dgq += gq_h
            if dgk.ndim == 2:
                dgk[h] += gk_h
            else:
                dgk += gk_h
    return dq, dk, dv, dgq, dgk
