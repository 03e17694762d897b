"""Plain fp64 definitions of RLA-2 / RAPT and of the original RLA (L2 denominator).

Test infrastructure only (see the package docstring). Every function takes
numpy arrays (any float dtype; they are widened to float64 first) and returns
float64 arrays. Layouts: dense [B, L, H, d]; packed varlen [T, H, d];
decode [N, H, d]; states S [.., H, d, d] key-major (S[i, j] = sum k'_i v_j)
and z [.., H, d].
"""

from __future__ import annotations

import numpy as np

_ROW_BLOCK = 1024  # rows of the score matrix formed at a time (memory bound only)


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def rmsnorm(x, gamma, eps):
    """RMSNorm over the last axis: x * (mean(x^2) + eps)^(-1/2) * gamma.

    ruDNN README §7 (statistics over the final axis, gamma a vector, eps finite
    and positive); candle "05-nn/layers", normalisation section (LayerNorm
    without mean subtraction and without bias). eps sits inside the root.
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * _f64(gamma)


def rope_adjacent(x, positions, base):
    """Rotary position embedding on adjacent pairs (2j, 2j+1).

    The pair is rotated by the angle p * theta_j with theta_j = base^(-2j/d):
    (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a). candle
    "05-nn/layers", rotary_emb section (interleaved pairing 2i / 2i+1); RAPT
    applies it to Q and K before the ReLU (08-rapt-algorithm.md §1, §3).

    x: [n, ..., d]; positions: [n] (one position per leading index).
    """
    x = _f64(x)
    d = x.shape[-1]
    j = np.arange(d // 2, dtype=np.float64)
    theta = float(base) ** (-2.0 * j / d)
    pos = _f64(positions).reshape((-1,) + (1,) * (x.ndim - 1))
    a = pos * theta  # broadcasts to [n, ..., d/2]
    c, s = np.cos(a), np.sin(a)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def relu(x):
    """Per-element max(0, x) (08-rapt-algorithm.md §1, §2.1: element-wise, not a norm)."""
    return np.maximum(_f64(x), 0.0)


def features(x, gamma, positions, eps_norm, rope_base):
    """q' = ReLU(RoPE(RMSNorm(x))) for tokens x: [n, H, d] at ``positions`` [n].

    08-rapt-algorithm.md §3 (RLA-2 core formula) and §4.2 (Q/K -> RMSNorm ->
    RoPE -> ReLU; V untouched). gamma: [d] shared by all heads or [H, d].
    """
    return relu(rope_adjacent(rmsnorm(x, gamma, eps_norm), positions, rope_base))


def rla2_causal_doc(qf, kf, v, eps_den=1e-4, S0=None, z0=None, rows=None):
    """RLA-2 causal output of one head of one document, quadratic form.

    out_t = (sum_{tau<=t} s_{t,tau} v_tau [+ q'_t S0])
            / (sum_{tau<=t} s_{t,tau} [+ q'_t . z0] + eps_den),  s = q'_t . k'_tau.
    08-rapt-algorithm.md §3 (S_t and z_t include token t; eps 1e-4) and §4.1
    (causal prefix i <= t within the same document).

    qf, kf, v: [n, d]. S0 [d, d], z0 [d] optional carried-in state. ``rows``:
    optional query indices to evaluate (default all). Returns (out, S_final,
    z_final) with S_final = S0 + K'^T V and z_final = z0 + sum K'.
    """
    qf, kf, v = _f64(qf), _f64(kf), _f64(v)
    n, d = qf.shape
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), v.shape[1]), dtype=np.float64)
    for r0 in range(0, len(rows), _ROW_BLOCK):
        rr = rows[r0:r0 + _ROW_BLOCK]
        hi = int(rr.max()) + 1 if len(rr) else 0
        s = qf[rr] @ kf[:hi].T  # [rows, hi]
        s = np.where(np.arange(hi)[None, :] <= rr[:, None], s, 0.0)
        num = s @ v[:hi]
        den = s.sum(axis=1)
        if S0 is not None:
            num = num + qf[rr] @ _f64(S0)
        if z0 is not None:
            den = den + qf[rr] @ _f64(z0)
        out[r0:r0 + len(rr)] = num / (den + float(eps_den))[:, None]
    S_final = kf.T @ v
    z_final = kf.sum(axis=0)
    if S0 is not None:
        S_final = S_final + _f64(S0)
    if z0 is not None:
        z_final = z_final + _f64(z0)
    return out, S_final, z_final


def rla2_recurrent_doc(qf, kf, v, eps_den=1e-4, S0=None, z0=None):
    """RLA-2 in recurrence form (self-check of the quadratic form only).

    S_t = S_{t-1} + k'_t v_t^T, z_t = z_{t-1} + k'_t, out_t = q'_t S_t / (q'_t . z_t + eps):
    08-rapt-algorithm.md §3.
    """
    qf, kf, v = _f64(qf), _f64(kf), _f64(v)
    n, d = qf.shape
    S = np.zeros((d, v.shape[1])) if S0 is None else _f64(S0).copy()
    z = np.zeros(d) if z0 is None else _f64(z0).copy()
    out = np.zeros((n, v.shape[1]))
    for t in range(n):
        S += np.outer(kf[t], v[t])
        z += kf[t]
        out[t] = (qf[t] @ S) / (qf[t] @ z + float(eps_den))
    return out, S, z


def _gamma_h(gamma, h):
    g = _f64(gamma)
    return g[h] if g.ndim == 2 else g


def rla2_prefill(q, k, v, gamma_q, gamma_k, eps_norm=1e-6, rope_base=1e4, eps_den=1e-4,
                 pos_offset=0, S0=None, z0=None, pairs=None, rows=None):
    """Dense causal RLA-2 prefill: q, k, v [B, L, H, d]; token t of each batch row is
    at RoPE position pos_offset + t; one document per batch row.

    S0, z0: optional [B, H, d, d], [B, H, d]. ``pairs``: optional list of (b, h) to
    evaluate (default all); ``rows``: optional query rows per pair.
    Returns (out [B, L, H, d] (NaN where not evaluated), S_final [B, H, d, d],
    z_final [B, H, d]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, L, H, d = q.shape
    out = np.full(q.shape[:3] + (v.shape[3],), np.nan)
    S_fin = np.full((B, H, d, v.shape[3]), np.nan)
    z_fin = np.full((B, H, d), np.nan)
    pos = pos_offset + np.arange(L)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        qf = features(q[b, :, h], _gamma_h(gamma_q, h), pos, eps_norm, rope_base)
        kf = features(k[b, :, h], _gamma_h(gamma_k, h), pos, eps_norm, rope_base)
        s0 = None if S0 is None else S0[b, h]
        zz = None if z0 is None else z0[b, h]
        rr = np.arange(L) if rows is None else np.asarray(rows)
        o, Sf, zf = rla2_causal_doc(qf, kf, v[b, :, h], eps_den, s0, zz, rows=rr)
        out[b, rr, h] = o
        S_fin[b, h] = Sf
        z_fin[b, h] = zf
    return out, S_fin, z_fin


def rla2_varlen(q, k, v, cu_seqlens, gamma_q, gamma_k, eps_norm=1e-6, rope_base=1e4,
                eps_den=1e-4, S0=None, z0=None, docs=None, heads=None, rows_per_doc=None):
    """Packed varlen causal RLA-2: q, k, v [T, H, d]; document n spans tokens
    cu_seqlens[n] .. cu_seqlens[n+1]-1. The state restarts at every document
    (08-rapt-algorithm.md §2.2 and §4.1) and RoPE positions restart at 0.
    S0, z0: optional per-document carried-in state [N, H, d, d], [N, H, d]
    (a separate state per sequence, ruDNN README §8).

    Returns (out [T, H, d], S_final [N, H, d, d], z_final [N, H, d]); an empty
    document's final state is its initial state (zeros if none).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    out = np.full(q.shape[:2] + (v.shape[2],), np.nan)
    S_fin = np.full((N, H, d, v.shape[2]), np.nan)
    z_fin = np.full((N, H, d), np.nan)
    docs = range(N) if docs is None else docs
    heads = range(H) if heads is None else heads
    for n in docs:
        a, b = int(cu[n]), int(cu[n + 1])
        pos = np.arange(b - a)
        for h in heads:
            s0 = None if S0 is None else S0[n, h]
            zz = None if z0 is None else z0[n, h]
            qf = features(q[a:b, h], _gamma_h(gamma_q, h), pos, eps_norm, rope_base)
            kf = features(k[a:b, h], _gamma_h(gamma_k, h), pos, eps_norm, rope_base)
            rr = np.arange(b - a) if rows_per_doc is None else np.asarray(rows_per_doc[n])
            o, Sf, zf = rla2_causal_doc(qf.reshape(b - a, d), kf.reshape(b - a, d),
                                        v[a:b, h], eps_den, s0, zz, rows=rr)
            out[a + rr, h] = o
            S_fin[n, h] = Sf  # an empty document leaves S0 (or zeros) unchanged
            z_fin[n, h] = zf
    return out, S_fin, z_fin


def rla2_decode_step(q, k, v, positions, gamma_q, gamma_k, S, z, eps_norm=1e-6,
                     rope_base=1e4, eps_den=1e-4):
    """One RLA-2 decode step (forward_step, 08-rapt-algorithm.md §4.2).

    For each sequence n and head h: features of the new token at positions[n];
    update the state first (S += k' v^T, z += k'), then read out
    q' S / (q' . z + eps). q, k, v: [N, H, d]; S [N, H, d, d]; z [N, H, d].
    Returns (out [N, H, d], S_new, z_new); the inputs are not modified.
    Every (sequence, head) is independent; the arrays hold all of them at once.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    pos = np.asarray(positions).reshape(-1)
    qf = features(q, gamma_q, pos, eps_norm, rope_base)  # [N, H, d]
    kf = features(k, gamma_k, pos, eps_norm, rope_base)
    S = _f64(S).copy()
    for n in range(S.shape[0]):  # one sequence at a time (bounds the temporary)
        S[n] += kf[n, :, :, None] * v[n, :, None, :]     # S[n, h, i, j] += k'_i v_j
    z = _f64(z) + kf
    num = (qf[..., None, :] @ S)[..., 0, :]              # q' S per (sequence, head)
    den = (qf * z).sum(axis=-1) + float(eps_den)
    return num / den[..., None], S, z


def rla2_decode_from_history(q_new, k_hist, v_hist, pos_new, gamma_q, gamma_k, eps_norm=1e-6,
                             rope_base=1e4, eps_den=1e-4):
    """Decode output of one head from the full token history, quadratic form.

    q_new: [d] raw query of the token at position pos_new; k_hist, v_hist:
    [pos_new + 1, d] raw keys / values of tokens 0..pos_new (the new token last).
    Equals the last row of the causal prefill over the history; needs no state.
    """
    P = k_hist.shape[0]
    pos = np.arange(P)
    qf = features(_f64(q_new)[None, None, :], gamma_q, np.array([pos_new]), eps_norm,
                  rope_base)[0, 0]
    kf = features(_f64(k_hist)[:, None, :], gamma_k, pos, eps_norm, rope_base)[:, 0]
    s = kf @ qf
    return (s @ _f64(v_hist)) / (s.sum() + float(eps_den))


def rla2_bidir_doc(qf, kf, v, eps_den=1e-4, rows=None):
    """Bidirectional (non-causal) RLA-2 output of one head of one document, quadratic form.

    out_t = sum_{tau in doc} s_{t,tau} v_tau / (sum_{tau in doc} s_{t,tau} + eps_den),
    s = q'_t . k'_tau: every token of the document is seen by every query.
    08-rapt-algorithm.md §4.1 (the prefix scan's causal=false mode: the sums over the whole set,
    one constant for every t) and §4.2 (the bidirectional branch of the Sum-denominator layer),
    with the RLA-2 Sum denominator and eps of §3. qf, kf, v: [n, d]; ``rows``: optional query
    indices (default all).
    """
    qf, kf, v = _f64(qf), _f64(kf), _f64(v)
    n = qf.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), v.shape[1]), dtype=np.float64)
    for r0 in range(0, len(rows), _ROW_BLOCK):
        rr = rows[r0:r0 + _ROW_BLOCK]
        s = qf[rr] @ kf.T  # [rows, n]
        out[r0:r0 + len(rr)] = (s @ v) / (s.sum(axis=1) + float(eps_den))[:, None]
    return out


def rla2_bidir(q, k, v, gamma_q, gamma_k, eps_norm=1e-6, rope_base=1e4, eps_den=1e-4,
               pos_offset=0, pairs=None, rows=None):
    """Dense bidirectional RLA-2: q, k, v [B, L, H, d], one sequence per batch row, token t at
    RoPE position pos_offset + t; features as in the causal form (08-rapt-algorithm.md §4.2).
    ``pairs`` / ``rows`` restrict the evaluation; other entries are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, L, H, d = q.shape
    out = np.full(q.shape[:3] + (v.shape[3],), np.nan)
    pos = pos_offset + np.arange(L)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    rr = np.arange(L) if rows is None else np.asarray(rows)
    for b, h in pairs:
        qf = features(q[b, :, h], _gamma_h(gamma_q, h), pos, eps_norm, rope_base)
        kf = features(k[b, :, h], _gamma_h(gamma_k, h), pos, eps_norm, rope_base)
        out[b, rr, h] = rla2_bidir_doc(qf, kf, v[b, :, h], eps_den, rows=rr)
    return out


def rla2_bidir_varlen(q, k, v, cu_seqlens, gamma_q, gamma_k, eps_norm=1e-6, rope_base=1e4,
                      eps_den=1e-4, docs=None, heads=None, rows_per_doc=None):
    """Packed varlen bidirectional RLA-2: q, k, v [T, H, d]; document n spans tokens
    cu_seqlens[n] .. cu_seqlens[n+1]-1, sees only itself and starts at RoPE position 0
    (the document boundary of 08-rapt-algorithm.md §2.2 and §4.1). Returns out [T, H, d].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.full(q.shape[:2] + (v.shape[2],), np.nan)
    docs = range(len(cu) - 1) if docs is None else docs
    heads = range(H) if heads is None else heads
    for n in docs:
        a, b = int(cu[n]), int(cu[n + 1])
        if b == a:
            continue
        pos = np.arange(b - a)
        rr = np.arange(b - a) if rows_per_doc is None else np.asarray(rows_per_doc[n])
        for h in heads:
            qf = features(q[a:b, h], _gamma_h(gamma_q, h), pos, eps_norm, rope_base)
            kf = features(k[a:b, h], _gamma_h(gamma_k, h), pos, eps_norm, rope_base)
            out[a + rr, h] = rla2_bidir_doc(qf, kf, v[a:b, h], eps_den, rows=rr)
    return out


def rla_l2(q, k, v, eps=1e-6, pairs=None, rows=None):
    """Original RLA, non-causal, L2 denominator (08-rapt-algorithm.md §2.1):

    out_t = sum_i s_ti v_i / (sqrt(sum_i s_ti^2) + eps), s_ti = ReLU(q_t) . ReLU(k_i),
    i over the whole sequence. q, k, v: [B, L, H, d]. ``pairs`` / ``rows``
    restrict the evaluation; other entries are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, L, H, d = q.shape
    out = np.full(q.shape[:3] + (v.shape[3],), np.nan)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    rr_all = np.arange(L) if rows is None else np.asarray(rows)
    for b, h in pairs:
        qf = relu(q[b, :, h])
        kf = relu(k[b, :, h])
        for r0 in range(0, len(rr_all), _ROW_BLOCK):
            rr = rr_all[r0:r0 + _ROW_BLOCK]
            s = qf[rr] @ kf.T
            num = s @ v[b, :, h]
            den = np.sqrt((s * s).sum(axis=1)) + float(eps)
            out[b, rr, h] = num / den[:, None]
    return out


def relative_error(y, r, zero_tol=1e-6):
    """Per-row max relative error: max over rows of ||y - r||_inf / ||r||_inf.

    Rows are the last axis. Rows whose reference is (almost) all zero
    (||r||_inf < zero_tol, every score 0) must have ||y||_inf <= zero_tol; such a
    row counts as error 0 when it does and as inf when it does not.
    Returns (max_row_error, global_error) where global_error is
    ||y - r||_inf / ||r||_inf over the whole array.
    """
    y = _f64(y)
    r = _f64(r)
    ry = np.abs(y - r).max(axis=-1)
    rn = np.abs(r).max(axis=-1)
    yn = np.abs(y).max(axis=-1)
    small = rn < zero_tol
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(small, np.where(yn <= zero_tol, 0.0, np.inf), ry / np.where(small, 1, rn))
    glob = float(np.abs(y - r).max() / max(np.abs(r).max(), 1e-300)) if r.size else 0.0
    return (float(rel.max()) if rel.size else 0.0), glob


def rla_l2_causal_doc(qf, kf, v, eps=1e-6, rows=None):
    """Causal original RLA (L2 denominator) of one head of one document, quadratic form.

    out_t = sum_{i<=t} s_ti v_i / (sqrt(sum_{i<=t} s_ti^2) + eps), s_ti = q'_t . k'_i: the §2.1
    closed form with the sums restricted to the causal prefix of the document (§2.2: a new query
    reads the accumulated state, which restarts only at document boundaries; §4.1: the prefix scan
    keeps A_t = sum_{i<=t} k'_i k'_i^T, whose quadratic form q'^T A_t q' is the denominator's sum of
    squares). qf, kf, v: [n, d]; ``rows``: optional query indices (default all).
    """
    qf, kf, v = _f64(qf), _f64(kf), _f64(v)
    n = qf.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), v.shape[1]), dtype=np.float64)
    for r0 in range(0, len(rows), _ROW_BLOCK):
        rr = rows[r0:r0 + _ROW_BLOCK]
        hi = int(rr.max()) + 1 if len(rr) else 0
        s = qf[rr] @ kf[:hi].T
        s = np.where(np.arange(hi)[None, :] <= rr[:, None], s, 0.0)
        out[r0:r0 + len(rr)] = (s @ v[:hi]) / (np.sqrt((s * s).sum(axis=1)) + float(eps))[:, None]
    return out


def rla_l2_causal_recurrent_doc(qf, kf, v, eps=1e-6):
    """The same in recurrence form (self-check only): S_t = S_{t-1} + k'_t v_t^T,
    A_t = A_{t-1} + k'_t k'_t^T, out_t = q'_t S_t / (sqrt(q'_t^T A_t q'_t) + eps)
    (08-rapt-algorithm.md §4.1, the A and B prefix states of the scan)."""
    qf, kf, v = _f64(qf), _f64(kf), _f64(v)
    n, d = qf.shape
    S = np.zeros((d, v.shape[1]))
    A = np.zeros((d, d))
    out = np.zeros((n, v.shape[1]))
    for t in range(n):
        S += np.outer(kf[t], v[t])
        A += np.outer(kf[t], kf[t])
        out[t] = (qf[t] @ S) / (np.sqrt(qf[t] @ A @ qf[t]) + float(eps))
    return out


def rla_l2_causal(q, k, v, eps=1e-6, pairs=None, rows=None):
    """Dense causal original RLA: q, k, v [B, L, H, d], one document per batch row; features
    ReLU(q), ReLU(k) with no norm and no RoPE (§2.1's global view Q' = ReLU(Q W_q)). ``pairs`` /
    ``rows`` restrict the evaluation; other entries are NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, L, H, d = q.shape
    out = np.full(q.shape[:3] + (v.shape[3],), np.nan)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    rr = np.arange(L) if rows is None else np.asarray(rows)
    for b, h in pairs:
        out[b, rr, h] = rla_l2_causal_doc(relu(q[b, :, h]), relu(k[b, :, h]), v[b, :, h], eps,
                                          rows=rr)
    return out


def rla_l2_causal_varlen(q, k, v, cu_seqlens, eps=1e-6, docs=None, heads=None):
    """Packed varlen causal original RLA: q, k, v [T, H, d]; document n spans tokens
    cu_seqlens[n] .. cu_seqlens[n+1]-1 and sees only itself (§2.2). Returns out [T, H, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.full(q.shape[:2] + (v.shape[2],), np.nan)
    docs = range(len(cu) - 1) if docs is None else docs
    heads = range(H) if heads is None else heads
    for n in docs:
        a, b = int(cu[n]), int(cu[n + 1])
        if b == a:
            continue
        for h in heads:
            out[a:b, h] = rla_l2_causal_doc(relu(q[a:b, h]), relu(k[a:b, h]), v[a:b, h], eps)
    return out


def linear(x, w):
    """y = x W^T (a linear map with weight W [N, K]; the layer's projections, 08-rapt-algorithm.md
    §3 q = W_q x and §4.2 the output projection w_o). A library matmul in fp64."""
    return _f64(x) @ _f64(w).T


def rapt_layer(x, w_qkv, w_o, gamma_q, gamma_k, H, eps_norm=1e-6, rope_base=1e4, eps_den=1e-4,
               pos_offset=0, pairs_rows=None):
    """One RAPT attention layer (08-rapt-algorithm.md §3 core formula with the projections, §4.2
    forward: projections, RMSNorm -> RoPE -> ReLU, the causal scan, the division, w_o).

    x [B, L, d_model]; w_qkv [3 H d, d_model] (rows: W_q, then W_k, then W_v, each head-major
    h d + j); w_o [d_model, H d]. Returns y [B, L, d_model]. ``pairs_rows``: optional (b, rows) to
    evaluate only those rows of batch row b (other entries NaN).
    """
    x = _f64(x)
    B, L, dm = x.shape
    d = _f64(w_qkv).shape[0] // (3 * H)
    bs = range(B) if pairs_rows is None else [pairs_rows[0]]
    y = np.full((B, L, _f64(w_o).shape[0]), np.nan)
    for b in bs:
        qkv = linear(x[b], w_qkv)  # [L, 3 H d]
        q = qkv[:, :H * d].reshape(1, L, H, d)
        k = qkv[:, H * d:2 * H * d].reshape(1, L, H, d)
        v = qkv[:, 2 * H * d:].reshape(1, L, H, d)
        rows = None if pairs_rows is None else np.asarray(pairs_rows[1])
        a, _, _ = rla2_prefill(q, k, v, gamma_q, gamma_k, eps_norm, rope_base, eps_den,
                               pos_offset=pos_offset, rows=rows)
        rr = np.arange(L) if rows is None else rows
        y[b, rr] = linear(a[0, rr].reshape(len(rr), H * d), w_o)
    return y
