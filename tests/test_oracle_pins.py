"""Pins of the fp64 oracle against what the pages and mathematics fix (CPU only).

Each test is chosen so that a plausible slip in the oracle (a dropped eps, an
exclusive instead of inclusive prefix, a wrong RoPE sign / pairing / frequency,
a transposed state, positions that do not restart per document) fails at least
one of them. Citations name the page ("08-rapt-algorithm.md" is the
neuralnet.cpp page on the RLA family) and its section.
"""

import json
import math
import os

import numpy as np
import pytest

import bruteforce as BF
import oracle as O
from relu_linear_attention_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(seed, shape, scale=1.0):
    return syn.rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- brute force


@pytest.mark.parametrize("L,d,H", [(1, 2, 1), (2, 4, 1), (5, 8, 2), (16, 8, 2), (16, 16, 1)])
@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_matches_bruteforce(L, d, H, with_state):
    """Causal RLA-2 (08-rapt-algorithm.md §3) vs a pure-Python brute force."""
    B = 2
    q, k, v = (_rand(s, (B, L, H, d)) for s in (1, 2, 3))
    gq = syn.rng(4).uniform(0.8, 1.2, (H, d))
    gk = syn.rng(5).uniform(0.8, 1.2, (H, d))
    S0 = _rand(6, (B, H, d, d)) if with_state else None
    z0 = np.abs(_rand(7, (B, H, d))) if with_state else None
    off = 7
    out, Sf, zf = O.rla2_prefill(q, k, v, gq, gk, 1e-6, 1e4, 1e-4, pos_offset=off, S0=S0, z0=z0)
    for b in range(B):
        for h in range(H):
            qf = [BF.feature_row(q[b, t, h], gq[h], off + t, 1e-6, 1e4) for t in range(L)]
            kf = [BF.feature_row(k[b, t, h], gk[h], off + t, 1e-6, 1e4) for t in range(L)]
            ref = BF.causal_head(qf, kf, v[b, :, h], 1e-4,
                                 None if S0 is None else S0[b, h], None if z0 is None else z0[b, h])
            np.testing.assert_allclose(out[b, :, h], np.array(ref), rtol=1e-10, atol=1e-12)
            # final state: S0 + sum_t k'_t v_t^T, z0 + sum_t k'_t  (key-major)
            Sref = np.zeros((d, d)) if S0 is None else S0[b, h].copy()
            zref = np.zeros(d) if z0 is None else z0[b, h].copy()
            for t in range(L):
                for i in range(d):
                    zref[i] += kf[t][i]
                    for j in range(d):
                        Sref[i, j] += kf[t][i] * v[b, t, h, j]
            np.testing.assert_allclose(Sf[b, h], Sref, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(zf[b, h], zref, rtol=1e-10, atol=1e-12)


def test_varlen_matches_bruteforce():
    """Packed documents: state reset and RoPE restart at every document
    (08-rapt-algorithm.md §2.2, §4.1); empty and length-1 documents included."""
    lens = [3, 0, 5, 1, 7]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H, d = int(cu[-1]), 2, 8
    q, k, v = (_rand(s, (T, H, d)) for s in (11, 12, 13))
    g = np.ones(d)
    out, Sf, zf = O.rla2_varlen(q, k, v, cu, g, g)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        for h in range(H):
            qf = [BF.feature_row(q[t, h], g, t - a, 1e-6, 1e4) for t in range(a, b)]
            kf = [BF.feature_row(k[t, h], g, t - a, 1e-6, 1e4) for t in range(a, b)]
            ref = BF.causal_head(qf, kf, v[a:b, h], 1e-4)
            if b > a:
                np.testing.assert_allclose(out[a:b, h], np.array(ref), rtol=1e-10, atol=1e-12)
            else:
                assert np.all(Sf[n, h] == 0) and np.all(zf[n, h] == 0)


@pytest.mark.parametrize("L,d", [(1, 4), (9, 8), (16, 16)])
def test_l2_matches_bruteforce(L, d):
    """Original RLA, L2 denominator, non-causal (08-rapt-algorithm.md §2.1)."""
    q, k, v = (_rand(s, (1, L, 1, d)) for s in (21, 22, 23))
    out = O.rla_l2(q, k, v, 1e-6)
    qf = [[max(0.0, x) for x in q[0, t, 0]] for t in range(L)]
    kf = [[max(0.0, x) for x in k[0, t, 0]] for t in range(L)]
    ref = BF.l2_head(qf, kf, v[0, :, 0], 1e-6)
    np.testing.assert_allclose(out[0, :, 0], np.array(ref), rtol=1e-10, atol=1e-12)


def test_decode_step_matches_bruteforce():
    """forward_step: features, update first, then read (08-rapt-algorithm.md §4.2)."""
    N, H, d, P = 3, 2, 8, 6
    g = syn.rng(30)
    kh, vh = g.standard_normal((P, N, H, d)), g.standard_normal((P, N, H, d))
    qn, kn, vn = (g.standard_normal((N, H, d)) for _ in range(3))
    gam = np.ones(d)
    # state of P history tokens, built by brute force
    S = np.zeros((N, H, d, d))
    z = np.zeros((N, H, d))
    for n in range(N):
        for h in range(H):
            for t in range(P):
                kf = BF.feature_row(kh[t, n, h], gam, t, 1e-6, 1e4)
                S[n, h] += np.outer(kf, vh[t, n, h])
                z[n, h] += kf
    pos = np.full(N, P, dtype=np.int32)
    out, S2, z2 = O.rla2_decode_step(qn, kn, vn, pos, gam, gam, S, z)
    for n in range(N):
        for h in range(H):
            qf = [BF.feature_row(qn[n, h], gam, P, 1e-6, 1e4)]
            kf_all = [BF.feature_row(kh[t, n, h], gam, t, 1e-6, 1e4) for t in range(P)]
            kf_all.append(BF.feature_row(kn[n, h], gam, P, 1e-6, 1e4))
            v_all = [vh[t, n, h] for t in range(P)] + [vn[n, h]]
            s = [BF.dot(qf[0], kk) for kk in kf_all]
            num = [sum(s[t] * v_all[t][j] for t in range(P + 1)) for j in range(d)]
            ref = [x / (sum(s) + 1e-4) for x in num]
            np.testing.assert_allclose(out[n, h], ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- identities


def test_quadratic_equals_recurrence():
    """Associativity (08-rapt-algorithm.md §1, §2.2): the O(L^2) sum and the state
    recurrence S_t = S_{t-1} + k'_t v_t^T agree to fp64 rounding."""
    L, d = 200, 16
    q, k, v = (_rand(s, (L, 1, d)) for s in (41, 42, 43))
    pos = np.arange(L)
    qf = O.features(q, np.ones(d), pos, 1e-6, 1e4)[:, 0]
    kf = O.features(k, np.ones(d), pos, 1e-6, 1e4)[:, 0]
    S0 = _rand(44, (d, d))
    z0 = np.abs(_rand(45, (d,)))
    a, Sa, za = O.rla2_causal_doc(qf, kf, v[:, 0], 1e-4, S0, z0)
    b, Sb, zb = O.rla2_recurrent_doc(qf, kf, v[:, 0], 1e-4, S0, z0)
    assert O.relative_error(a, b)[0] < 1e-12
    np.testing.assert_allclose(Sa, Sb, rtol=1e-12, atol=1e-11)
    np.testing.assert_allclose(za, zb, rtol=1e-12, atol=1e-12)


def test_disjoint_supports_give_exact_zero():
    """Scores are exactly 0 when the positive supports of q' and k' do not meet
    (08-rapt-algorithm.md §1, §2.2). q lives only in RoPE pairs {0, 2}, k only in
    pairs {1, 3}; RMSNorm and RoPE keep pair supports, so every score is 0 and the
    output is 0 / (0 + eps) = 0 exactly."""
    L, H, d = 12, 2, 8
    q, k, v = (_rand(s, (1, L, H, d)) for s in (51, 52, 53))
    q[..., 2:4] = 0.0
    q[..., 6:8] = 0.0
    k[..., 0:2] = 0.0
    k[..., 4:6] = 0.0
    out, _, _ = O.rla2_prefill(q, k, v, np.ones(d), np.ones(d), pos_offset=3)
    assert np.all(out == 0.0)
    out2 = O.rla_l2(q, k, v)
    assert np.all(out2 == 0.0)


def test_ones_value_gives_weights_in_unit_interval():
    """With v = 1 the output is sum(s) / (sum(s) + eps), the z-scan identity of
    forward step 2 (08-rapt-algorithm.md §4.2): equal in every component, in [0, 1)."""
    L, H, d = 40, 2, 16
    q, k = _rand(61, (1, L, H, d)), _rand(62, (1, L, H, d))
    v = np.ones((1, L, H, d))
    out, _, zf = O.rla2_prefill(q, k, v, np.ones(d), np.ones(d))
    assert np.all(out >= 0) and np.all(out < 1)
    assert np.all(np.ptp(out, axis=-1) < 1e-15)
    # explicit sum(s)/(sum(s)+eps) through z = sum k' (separate route)
    pos = np.arange(L)
    qf = O.features(q[0], np.ones(d), pos, 1e-6, 1e4)
    kf = O.features(k[0], np.ones(d), pos, 1e-6, 1e4)
    zc = np.cumsum(kf, axis=0)
    qz = np.einsum("thd,thd->th", qf, zc)
    np.testing.assert_allclose(out[0, :, :, 0], qz / (qz + 1e-4), rtol=1e-13)


def test_output_in_convex_hull_of_visible_values():
    """Non-negative weights summing to sum(s)/(sum(s)+eps) <= 1 (08-rapt-algorithm.md
    §2.3, §3): each output component lies in [min(0, min v), max(0, max v)] over the
    visible tokens."""
    L, H, d = 30, 1, 8
    q, k, v = (_rand(s, (1, L, H, d)) for s in (71, 72, 73))
    out, _, _ = O.rla2_prefill(q, k, v, np.ones(d), np.ones(d))
    for t in range(L):
        lo = np.minimum(0, v[0, :t + 1, 0].min(axis=0))
        hi = np.maximum(0, v[0, :t + 1, 0].max(axis=0))
        assert np.all(out[0, t, 0] >= lo - 1e-12) and np.all(out[0, t, 0] <= hi + 1e-12)


def test_single_token_closed_form():
    """L = 1: out = s / (s + eps) * v_0 with s = q'.k' (inclusive prefix, §3/§4.1)."""
    d = 8
    q, k, v = (_rand(s, (1, 1, 1, d)) for s in (81, 82, 83))
    out, _, _ = O.rla2_prefill(q, k, v, np.ones(d), np.ones(d), pos_offset=5)
    qf = O.features(q[0], np.ones(d), [5], 1e-6, 1e4)[0, 0]
    kf = O.features(k[0], np.ones(d), [5], 1e-6, 1e4)[0, 0]
    s = qf @ kf
    assert s > 0
    np.testing.assert_allclose(out[0, 0, 0], s / (s + 1e-4) * v[0, 0, 0], rtol=1e-14)


def test_constant_value_and_linearity():
    """Constant v = c gives c * sum(s) / (sum(s) + eps); the output is linear in v
    (the denominator does not involve v)."""
    L, H, d = 25, 2, 8
    q, k = _rand(91, (1, L, H, d)), _rand(92, (1, L, H, d))
    g = np.ones(d)
    ones, _, _ = O.rla2_prefill(q, k, np.ones((1, L, H, d)), g, g)
    c = -2.5
    oc, _, _ = O.rla2_prefill(q, k, np.full((1, L, H, d), c), g, g)
    np.testing.assert_allclose(oc, c * ones, rtol=1e-14)
    v1, v2 = _rand(93, (1, L, H, d)), _rand(94, (1, L, H, d))
    a, _, _ = O.rla2_prefill(q, k, v1, g, g)
    b, _, _ = O.rla2_prefill(q, k, v2, g, g)
    ab, _, _ = O.rla2_prefill(q, k, v1 + 3 * v2, g, g)
    np.testing.assert_allclose(ab, a + 3 * b, rtol=1e-12, atol=1e-13)


def test_rope_properties():
    """RoPE (candle "05-nn/layers", rotary_emb; RAPT applies it before ReLU):
    per-pair norm preserved, position 0 is the identity, scores depend only on the
    position difference, pair 0 turns by exactly p radians, and neighbouring pair
    frequencies have the constant ratio base^(-2/d)."""
    d, base = 16, 1e4
    x, y = _rand(101, (1, d)), _rand(102, (1, d))
    for p in (0, 1, 17, 4095):
        rx = O.rope_adjacent(x, [p], base)
        np.testing.assert_allclose(np.hypot(rx[0, 0::2], rx[0, 1::2]),
                                   np.hypot(x[0, 0::2], x[0, 1::2]), rtol=1e-13)
    np.testing.assert_array_equal(O.rope_adjacent(x, [0], base), x)
    s1 = O.rope_adjacent(x, [10], base)[0] @ O.rope_adjacent(y, [3], base)[0]
    s2 = O.rope_adjacent(x, [1007], base)[0] @ O.rope_adjacent(y, [1000], base)[0]
    np.testing.assert_allclose(s1, s2, rtol=1e-10)
    # measured angles of the unit vector e_{2j} at position 1
    e = np.zeros((d // 2, d))
    for j in range(d // 2):
        e[j, 2 * j] = 1.0
    r = O.rope_adjacent(e, np.ones(d // 2), base)
    ang = np.array([math.atan2(r[j, 2 * j + 1], r[j, 2 * j]) for j in range(d // 2)])
    assert ang[0] == pytest.approx(1.0, abs=1e-15)
    np.testing.assert_allclose(ang[1:] / ang[:-1], base ** (-2.0 / d), rtol=1e-12)
    # positive rotation sense: e_0 at position p = pi/2 / theta_0 lands on +e_1
    r90 = O.rope_adjacent(e[:1], [math.pi / 2], base)
    assert r90[0, 1] == pytest.approx(1.0) and abs(r90[0, 0]) < 1e-15


def test_rmsnorm_properties():
    """RMSNorm (ruDNN README §7; LayerNorm without mean and bias, candle notes):
    ||x_hat / gamma||^2 = d * m / (m + eps) with m = mean(x^2), and scale invariance
    up to the eps term."""
    d = 64
    x = _rand(111, (5, d))
    gam = syn.rng(112).uniform(0.8, 1.2, d)
    eps = 1e-6
    y = O.rmsnorm(x, gam, eps)
    m = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sum((y / gam) ** 2, axis=1), d * m / (m + eps), rtol=1e-13)
    y3 = O.rmsnorm(3.0 * x, gam, eps)
    np.testing.assert_allclose(y3, y, rtol=1e-5)
    # eps dominates a tiny vector: x = 1e-5 everywhere -> x / sqrt(1e-10 + 1e-6)
    t = O.rmsnorm(np.full((1, 4), 1e-5), np.ones(4), 1e-6)
    np.testing.assert_allclose(t, 1e-5 / math.sqrt(1e-10 + 1e-6), rtol=1e-14)


def test_l2_identity_and_bound():
    """Original RLA (08-rapt-algorithm.md §2.1, §2.2): by associativity the numerator is
    q'(K'^T V) and sum_i s_i^2 = q'^T (K'^T K') q'; with v = 1 the output is
    sum(s) / (||s||_2 + eps) <= sqrt(L)."""
    B, L, H, d = 1, 64, 2, 16
    q, k, v = (_rand(s, (B, L, H, d)) for s in (121, 122, 123))
    out = O.rla_l2(q, k, v, 1e-6)
    for h in range(H):
        qf, kf = np.maximum(q[0, :, h], 0), np.maximum(k[0, :, h], 0)
        MV, MK = kf.T @ v[0, :, h], kf.T @ kf
        num = qf @ MV
        den = np.sqrt(np.einsum("ti,ij,tj->t", qf, MK, qf)) + 1e-6
        assert O.relative_error(out[0, :, h], num / den[:, None])[0] < 1e-12
    o1 = O.rla_l2(q, k, np.ones_like(v), 1e-6)
    assert np.all(o1 <= math.sqrt(L) + 1e-12) and np.all(o1 >= 0)


def test_varlen_equals_concatenated_dense_runs():
    """Packing documents changes nothing: each document's rows equal a dense run of
    that document alone with positions from 0 (state reset §2.2; carried state per
    sequence, ruDNN README §8)."""
    lens = [17, 1, 0, 33]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H, d = int(cu[-1]), 2, 16
    q, k, v = (_rand(s, (T, H, d)) for s in (131, 132, 133))
    gq = syn.rng(134).uniform(0.8, 1.2, (H, d))
    N = len(lens)
    S0 = _rand(135, (N, H, d, d))
    z0 = np.abs(_rand(136, (N, H, d)))
    out, Sf, zf = O.rla2_varlen(q, k, v, cu, gq, gq, S0=S0, z0=z0)
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        o, S1, z1 = O.rla2_prefill(q[None, a:b], k[None, a:b], v[None, a:b], gq, gq,
                                   S0=S0[n:n + 1], z0=z0[n:n + 1])
        np.testing.assert_array_equal(out[a:b], o[0])
        np.testing.assert_array_equal(Sf[n], S1[0])
        np.testing.assert_array_equal(zf[n], z1[0])
    assert np.array_equal(Sf[2], S0[2]) and np.array_equal(zf[2], z0[2])


def test_decode_equals_prefill():
    """KV-cache consistency (08-rapt-algorithm.md §4.4, rapt_smoke_test): decode steps
    from the prefill state reproduce the prefill rows; the history form agrees."""
    N, P, steps, H, d = 2, 9, 4, 2, 8
    Lt = P + steps
    q, k, v = (_rand(s, (N, Lt, H, d)) for s in (141, 142, 143))
    g = syn.rng(144).uniform(0.8, 1.2, (H, d))
    full, _, _ = O.rla2_prefill(q, k, v, g, g)
    _, S, z = O.rla2_prefill(q[:, :P], k[:, :P], v[:, :P], g, g)
    for t in range(steps):
        pos = np.full(N, P + t, np.int32)
        o, S, z = O.rla2_decode_step(q[:, P + t], k[:, P + t], v[:, P + t], pos, g, g, S, z)
        assert O.relative_error(o, full[:, P + t])[0] < 1e-12
    for n in range(N):
        for h in range(H):
            oh = O.rla2_decode_from_history(q[n, Lt - 1, h], k[n, :, h], v[n, :, h], Lt - 1,
                                            g[h], g[h])
            assert O.relative_error(oh, full[n, Lt - 1, h])[0] < 1e-12


def test_relative_error_metric():
    r = np.array([[1.0, -2.0], [0.0, 0.0]])
    assert O.relative_error(r, r) == (0.0, 0.0)
    y = np.array([[1.0, -2.2], [0.0, 0.0]])
    assert O.relative_error(y, r)[0] == pytest.approx(0.1)
    y2 = np.array([[1.0, -2.0], [1e-3, 0.0]])
    assert O.relative_error(y2, r)[0] == math.inf


# ---------------------------------------------------------------- golden values


def test_page_constants():
    """The constants the pages fix, stored with their citations."""
    with open(os.path.join(GOLDEN, "page_constants.json")) as f:
        c = json.load(f)
    import inspect

    assert inspect.signature(O.rla2_prefill).parameters["eps_den"].default == c["rla2_eps_den"]["value"]
    assert inspect.signature(O.rla_l2).parameters["eps"].default == c["rla_l2_eps"]["value"]
    assert c["rla2_eps_den"]["value"] == 1e-4 and c["rla_l2_eps"]["value"] == 1e-6


def test_tiny_fp32_golden_regression():
    """Output of the tiny fp32 workload (B=1, H=2, L=64, d=16, seed 0), stored by
    tests/golden/make_golden.py, which calls only the oracle and the generator."""
    w = syn.tiny_fp32(0)
    out, _, _ = O.rla2_prefill(w.q, w.k, w.v, w.gamma_q, w.gamma_k, w.eps_norm, w.rope_base,
                               w.eps_den)
    ref = np.loadtxt(os.path.join(GOLDEN, "tiny_fp32_out.txt")).reshape(out.shape)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- bidirectional (non-causal)


@pytest.mark.parametrize("L,d,H", [(1, 2, 1), (5, 8, 2), (16, 8, 2), (16, 16, 1)])
def test_bidir_matches_bruteforce(L, d, H):
    """Non-causal RLA-2 (08-rapt-algorithm.md §4.1 causal=false, §3 Sum denominator) vs a
    pure-Python brute force in which every query sees every token."""
    B = 2
    q, k, v = (_rand(s, (B, L, H, d)) for s in (41, 42, 43))
    gq = syn.rng(44).uniform(0.8, 1.2, (H, d))
    gk = syn.rng(45).uniform(0.8, 1.2, (H, d))
    off = 3
    out = O.rla2_bidir(q, k, v, gq, gk, 1e-6, 1e4, 1e-4, pos_offset=off)
    for b in range(B):
        for h in range(H):
            qf = [BF.feature_row(q[b, t, h], gq[h], off + t, 1e-6, 1e4) for t in range(L)]
            kf = [BF.feature_row(k[b, t, h], gk[h], off + t, 1e-6, 1e4) for t in range(L)]
            ref = BF.bidir_head(qf, kf, v[b, :, h], 1e-4)
            np.testing.assert_allclose(out[b, :, h], np.array(ref), rtol=1e-10, atol=1e-12)


def test_bidir_last_row_is_causal_last_row():
    """The inclusive causal prefix of the last token covers the whole sequence (§4.1 "i <= t"),
    so the two modes agree exactly there and nowhere is the bidirectional row a causal one."""
    B, L, H, d = 2, 40, 2, 16
    q, k, v = (_rand(s, (B, L, H, d)) for s in (51, 52, 53))
    g = np.ones(d)
    bi = O.rla2_bidir(q, k, v, g, g)
    ca, _, _ = O.rla2_prefill(q, k, v, g, g)
    np.testing.assert_allclose(bi[:, -1], ca[:, -1], rtol=1e-12, atol=1e-14)
    assert np.abs(bi[:, 0] - ca[:, 0]).max() > 1e-3  # the first query sees the future


def test_bidir_key_order_invariance():
    """Sums over the whole set: reordering the (k', v) rows together changes nothing; reordering
    the queries reorders the output rows."""
    n, d = 33, 16
    qf = np.abs(_rand(61, (n, d)))
    kf = np.abs(_rand(62, (n, d)))
    v = _rand(63, (n, d))
    ref = O.rla2_bidir_doc(qf, kf, v)
    perm = syn.rng(64).permutation(n)
    np.testing.assert_allclose(O.rla2_bidir_doc(qf, kf[perm], v[perm]), ref, rtol=1e-12)
    np.testing.assert_allclose(O.rla2_bidir_doc(qf[perm], kf, v), ref[perm], rtol=1e-12)


def test_bidir_constant_v_closed_form():
    """v == 1: out = sum(s) / (sum(s) + eps), in [0, 1), equal across the row."""
    n, d = 20, 8
    qf = np.abs(_rand(71, (n, d)))
    kf = np.abs(_rand(72, (n, d)))
    out = O.rla2_bidir_doc(qf, kf, np.ones((n, 4)))
    ssum = (qf @ kf.T).sum(axis=1)
    np.testing.assert_allclose(out[:, 0], ssum / (ssum + 1e-4), rtol=1e-13)
    assert np.all(out >= 0) and np.all(out < 1) and np.all(out == out[:, :1])


def test_bidir_varlen_matches_dense_docs():
    """Packed documents see only themselves and restart RoPE at 0 (§2.2, §4.1)."""
    lens = [4, 0, 9, 1]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H, d = int(cu[-1]), 2, 8
    q, k, v = (_rand(s, (T, H, d)) for s in (81, 82, 83))
    g = syn.rng(84).uniform(0.8, 1.2, (H, d))
    out = O.rla2_bidir_varlen(q, k, v, cu, g, g)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        if b == a:
            continue
        ref = O.rla2_bidir(q[None, a:b], k[None, a:b], v[None, a:b], g, g)[0]
        np.testing.assert_allclose(out[a:b], ref, rtol=1e-13)
