"""Pins of the fp64 backward oracle (oracle/rla2_bwd.py) against what mathematics fixes, on the CPU.

The gradient of L = sum dout . out is pinned by central finite differences of two forward
definitions that share no code with the backward: the oracle's forward (rla2_prefill) and the
pure-Python brute force (tests/bruteforce.py, RoPE as a complex product). Further pins: Euler's
identity for the part of the output that is linear in v, the RMSNorm scale identity
x . dx = eps r^2 (y . dy), shared gains = the sum of per-head gains, and varlen = per-document
dense runs. test_oracle_bwd_mutations.py plants mistakes and checks that one of these fails.
"""

import numpy as np
import pytest

import bruteforce as BF
import oracle
from oracle import rla2_bwd as RB

EPS_N, BASE, EPS_D = 1e-6, 1e4, 1e-4


def _case(seed, B=1, L=7, H=2, d=8, per_head_gamma=True):
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.standard_normal((B, L, H, d)) for _ in range(4))
    shape = (H, d) if per_head_gamma else (d,)
    gq = rng.uniform(0.8, 1.2, shape)
    gk = rng.uniform(0.8, 1.2, shape)
    return q, k, v, g, gq, gk


def _loss_oracle(q, k, v, g, gq, gk, pos_offset):
    out, _, _ = oracle.rla2_prefill(q, k, v, gq, gk, EPS_N, BASE, EPS_D, pos_offset=pos_offset)
    return float(np.sum(out * g))


def _loss_brute(q, k, v, g, gq, gk, pos_offset):
    B, L, H, d = q.shape
    tot = 0.0
    for b in range(B):
        for h in range(H):
            ga = gq[h] if np.ndim(gq) == 2 else gq
            gb = gk[h] if np.ndim(gk) == 2 else gk
            qf = [BF.feature_row(q[b, t, h], ga, pos_offset + t, EPS_N, BASE) for t in range(L)]
            kf = [BF.feature_row(k[b, t, h], gb, pos_offset + t, EPS_N, BASE) for t in range(L)]
            out = BF.causal_head(qf, kf, [list(v[b, t, h]) for t in range(L)], EPS_D)
            for t in range(L):
                tot += BF.dot(out[t], list(g[b, t, h]))
    return tot


def _grads(q, k, v, g, gq, gk, pos_offset):
    return RB.rla2_prefill_bwd(q, k, v, g, gq, gk, EPS_N, BASE, EPS_D, pos_offset=pos_offset)


@pytest.mark.parametrize("which", range(5))
@pytest.mark.parametrize("per_head_gamma", [True, False])
def test_directional_derivative_matches_finite_difference(which, per_head_gamma):
    """<grad_x, u> = (L(x + h u) - L(x - h u)) / 2h for a random direction u of one input at a
    time (q, k, v, gamma_q, gamma_k), so a mistake in one gradient cannot hide behind another."""
    q, k, v, g, gq, gk = _case(10 + which, per_head_gamma=per_head_gamma)
    args = [q, k, v, gq, gk]
    grads = _grads(q, k, v, g, gq, gk, 3)
    rng = np.random.default_rng(99 + which)
    u = rng.standard_normal(args[which].shape)
    h = 1e-6

    def at(sign):
        a = [x.copy() for x in args]
        a[which] = a[which] + sign * h * u
        return _loss_oracle(a[0], a[1], a[2], g, a[3], a[4], 3)

    fd = (at(1) - at(-1)) / (2 * h)
    an = float(np.sum(grads[which] * u))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (which, fd, an)


def test_every_element_against_the_brute_force():
    """Per-element central differences of the independent pure-Python forward on a tiny case
    (two documents as batch rows, per-head gains, a RoPE offset)."""
    q, k, v, g, gq, gk = _case(5, B=2, L=4, H=1, d=4)
    grads = _grads(q, k, v, g, gq, gk, 2)
    h = 1e-6
    for which, x in enumerate([q, k, v, gq, gk]):
        for idx in np.ndindex(x.shape):
            a = [t.copy() for t in (q, k, v, gq, gk)]
            a[which][idx] += h
            lp = _loss_brute(a[0], a[1], a[2], g, a[3], a[4], 2)
            a[which][idx] -= 2 * h
            lm = _loss_brute(a[0], a[1], a[2], g, a[3], a[4], 2)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grads[which][idx]) <= 2e-6 * max(1.0, abs(fd)), (which, idx, fd,
                                                                               grads[which][idx])


def test_euler_identity_in_v():
    """out is homogeneous of degree 1 in v (the scores do not depend on v), so
    sum(dv * v) = sum(dout * out) exactly up to rounding."""
    q, k, v, g, gq, gk = _case(7, B=2, L=33, H=3, d=16)
    out, _, _ = oracle.rla2_prefill(q, k, v, gq, gk, EPS_N, BASE, EPS_D)
    dv = _grads(q, k, v, g, gq, gk, 0)[2]
    assert np.isclose(np.sum(dv * v), np.sum(g * out), rtol=1e-11, atol=1e-11)


def test_rmsnorm_scale_identity():
    """d/dalpha of RMSNorm(alpha x) at alpha = 1 is y * eps / (m + eps): hence
    x . dx = eps r^2 (y . dy) for every row (r = (m + eps)^-1/2, y the output)."""
    rng = np.random.default_rng(3)
    for eps in (1e-6, 0.3):
        x = rng.standard_normal((9, 16)) * rng.uniform(0.05, 3.0, (9, 1))
        gam = rng.uniform(0.5, 1.5, 16)
        dy = rng.standard_normal((9, 16))
        dx, _ = RB.rmsnorm_bwd(x, gam, eps, dy)
        y = oracle.rmsnorm(x, gam, eps)
        r2 = 1.0 / (np.mean(x * x, axis=1) + eps)
        assert np.allclose(np.sum(x * dx, axis=1), eps * r2 * np.sum(y * dy, axis=1),
                           rtol=1e-10, atol=1e-13)


def test_rope_backward_is_the_inverse_rotation():
    """<RoPE(x), w> = <x, RoPE_bwd(w)> (the adjoint) and RoPE_bwd(RoPE(x)) = x (orthogonality)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 2, 12))
    w = rng.standard_normal((6, 2, 12))
    pos = np.array([0, 1, 5, 77, 1000, 8191])
    fx = oracle.rope_adjacent(x, pos, BASE)
    assert np.isclose(np.sum(fx * w), np.sum(x * RB.rope_adjacent_bwd(w, pos, BASE)), rtol=1e-12)
    assert np.allclose(RB.rope_adjacent_bwd(fx, pos, BASE), x, atol=1e-12)


def test_shared_gain_is_the_sum_over_heads():
    q, k, v, g, gq, gk = _case(8, B=1, L=9, H=3, d=8, per_head_gamma=False)
    shared = _grads(q, k, v, g, gq, gk, 0)
    per = _grads(q, k, v, g, np.tile(gq, (3, 1)), np.tile(gk, (3, 1)), 0)
    for i in range(3):
        assert np.allclose(shared[i], per[i], rtol=1e-12, atol=1e-14)
    assert np.allclose(shared[3], per[3].sum(axis=0), rtol=1e-12)
    assert np.allclose(shared[4], per[4].sum(axis=0), rtol=1e-12)


def test_varlen_is_per_document_dense():
    """Packed documents (one empty, one of length 1) = separate dense runs; gains sum over them."""
    rng = np.random.default_rng(11)
    lens = [5, 0, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, d = int(cu[-1]), 2, 8
    q, k, v, g = (rng.standard_normal((T, H, d)) for _ in range(4))
    gq, gk = rng.uniform(0.8, 1.2, (H, d)), rng.uniform(0.8, 1.2, (H, d))
    dq, dk, dv, dgq, dgk = RB.rla2_varlen_bwd(q, k, v, g, cu, gq, gk, EPS_N, BASE, EPS_D)
    sq, sk = np.zeros_like(dgq), np.zeros_like(dgk)
    for n, L in enumerate(lens):
        if L == 0:
            continue
        a, b = int(cu[n]), int(cu[n + 1])
        r = RB.rla2_prefill_bwd(q[None, a:b], k[None, a:b], v[None, a:b], g[None, a:b], gq, gk,
                                EPS_N, BASE, EPS_D)
        assert np.allclose(dq[a:b], r[0][0], rtol=1e-12, atol=1e-14)
        assert np.allclose(dk[a:b], r[1][0], rtol=1e-12, atol=1e-14)
        assert np.allclose(dv[a:b], r[2][0], rtol=1e-12, atol=1e-14)
        sq += r[3]
        sk += r[4]
    assert np.allclose(dgq, sq, rtol=1e-12) and np.allclose(dgk, sk, rtol=1e-12)


def test_disjoint_supports_give_zero_key_and_query_gradients():
    """With every score exactly 0 (q' and k' on disjoint RoPE pairs) out = 0 for any v, so
    dq = dk = 0 and dv = 0 exactly; the value path has no other route."""
    L, H, d = 6, 1, 8
    rng = np.random.default_rng(2)
    q = np.zeros((1, L, H, d)); k = np.zeros((1, L, H, d))
    q[..., 0:4] = rng.standard_normal((1, L, H, 4))
    k[..., 4:8] = rng.standard_normal((1, L, H, 4))
    v, g = rng.standard_normal((1, L, H, d)), rng.standard_normal((1, L, H, d))
    gam = np.ones(d)
    dq, dk, dv, dgq, dgk = RB.rla2_prefill_bwd(q, k, v, g, gam, gam, EPS_N, BASE, EPS_D)
    for x in (dq, dk, dv, dgq, dgk):
        assert np.all(x == 0.0)
