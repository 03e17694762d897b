"""Pins of the causal original-RLA oracle (L2 denominator over the causal prefix; CPU only).

08-rapt-algorithm.md §2.1 (the L2-denominator closed form, eps 1e-6 outside the root, features
ReLU(q), ReLU(k)), §2.2 (a query reads the accumulated causal state, reset at document
boundaries) and §4.1 (the prefix scan's A_t = sum k'k'^T state). The last part of the file plants
mistakes in the oracle and checks that a pin catches each.
"""

import math

import numpy as np
import pytest

import bruteforce as BF
import oracle as O
import oracle.rla2 as R
from relu_linear_attention_gb300 import synthetic as syn


def _rand(seed, shape):
    return syn.rng(seed).standard_normal(shape)


def _relu_rows(x):
    return [[float(e) if e > 0 else 0.0 for e in row] for row in x]


@pytest.mark.parametrize("L,d,H", [(1, 2, 1), (2, 4, 1), (7, 8, 2), (16, 8, 2), (16, 16, 1)])
def test_matches_bruteforce(L, d, H):
    q, k, v = (_rand(s, (2, L, H, d)) for s in (21, 22, 23))
    out = O.rla_l2_causal(q, k, v, 1e-6)
    for b in range(2):
        for h in range(H):
            ref = BF.l2_causal_head(_relu_rows(q[b, :, h]), _relu_rows(k[b, :, h]), v[b, :, h], 1e-6)
            np.testing.assert_allclose(out[b, :, h], np.array(ref), rtol=1e-10, atol=1e-12)


def test_quadratic_equals_recurrence_with_the_a_state():
    q, k, v = (_rand(s, (300, 16)) for s in (24, 25, 26))
    qf, kf = np.maximum(q, 0), np.maximum(k, 0)
    a = O.rla_l2_causal_doc(qf, kf, v, 1e-6)
    b = O.rla_l2_causal_recurrent_doc(qf, kf, v, 1e-6)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_last_row_is_the_noncausal_row():
    q, k, v = (_rand(s, (1, 50, 2, 8)) for s in (27, 28, 29))
    c = O.rla_l2_causal(q, k, v, 1e-6)
    nc = O.rla_l2(q, k, v, 1e-6)
    np.testing.assert_allclose(c[:, -1], nc[:, -1], rtol=1e-12, atol=1e-14)
    # and row 0 sees only token 0: s v_0 / (|s| + eps)
    s = np.maximum(q[0, 0], 0) @ np.maximum(k[0, 0], 0).T
    for h in range(2):
        np.testing.assert_allclose(c[0, 0, h], s[h, h] * v[0, 0, h] / (abs(s[h, h]) + 1e-6),
                                   rtol=1e-12)


def test_homogeneity_in_q():
    """out(alpha q') with eps equals out(q') with eps / alpha: numerator and the L2 norm of the
    scores are both of degree 1 in q' (eps sits outside the root)."""
    q, k, v = (_rand(s, (40, 8)) for s in (30, 31, 32))
    qf, kf = np.maximum(q, 0), np.maximum(k, 0)
    for alpha in (1e-3, 0.5, 7.0):
        np.testing.assert_allclose(O.rla_l2_causal_doc(alpha * qf, kf, v, 1e-2),
                                   O.rla_l2_causal_doc(qf, kf, v, 1e-2 / alpha), rtol=1e-12)


def test_v_one_bound():
    """v == 1: out_t = sum s / (|s|_2 + eps) <= sqrt(t + 1) (Cauchy-Schwarz); equal keys make the
    scores equal and reach sqrt(t + 1) |s| / (|s| + eps)."""
    q, k = _rand(33, (30, 8)), _rand(34, (30, 8))
    qf, kf = np.maximum(q, 0), np.maximum(k, 0)
    out = O.rla_l2_causal_doc(qf, kf, np.ones((30, 1)), 1e-6)[:, 0]
    assert np.all(out <= np.sqrt(np.arange(1, 31)) + 1e-12) and np.all(out >= 0)
    keq = np.tile(kf[:1], (30, 1))
    out = O.rla_l2_causal_doc(qf, keq, np.ones((30, 1)), 1e-6)[:, 0]
    s = qf @ kf[0]
    t = np.arange(30)
    np.testing.assert_allclose(out, (t + 1) * s / (np.sqrt(t + 1) * s + 1e-6), rtol=1e-12)


def test_disjoint_supports_give_exact_zeros():
    d = 8
    q, k, v = np.zeros((20, d)), np.zeros((20, d)), _rand(35, (20, d))
    q[:, :4] = np.abs(_rand(36, (20, 4)))
    k[:, 4:] = np.abs(_rand(37, (20, 4)))
    assert np.all(O.rla_l2_causal_doc(q, k, v, 1e-6) == 0.0)


def test_varlen_is_per_document_dense():
    lens = [5, 0, 1, 12]
    cu = syn.cu_seqlens_from_lengths(lens)
    T = int(cu[-1])
    q, k, v = (_rand(s, (T, 2, 8)) for s in (38, 39, 40))
    out = O.rla_l2_causal_varlen(q, k, v, cu, 1e-6)
    for n, L in enumerate(lens):
        if L == 0:
            continue
        a, b = int(cu[n]), int(cu[n + 1])
        ref = O.rla_l2_causal(q[None, a:b], k[None, a:b], v[None, a:b], 1e-6)[0]
        np.testing.assert_array_equal(out[a:b], ref)


# ---------------------------------------------------------------- planted mistakes

def _variant(kind):
    def f(qf, kf, v, eps=1e-6, rows=None):
        qf, kf, v = (np.asarray(x, np.float64) for x in (qf, kf, v))
        n = qf.shape[0]
        s = qf @ kf.T
        if kind == "exclusive":
            s = np.where(np.arange(n)[None, :] < np.arange(n)[:, None], s, 0.0)
        elif kind != "noncausal":
            s = np.where(np.arange(n)[None, :] <= np.arange(n)[:, None], s, 0.0)
        if kind == "eps_inside":
            den = np.sqrt((s * s).sum(1) + eps)
        elif kind == "sum_den":
            den = s.sum(1) + eps
        else:
            den = np.sqrt((s * s).sum(1)) + eps
        out = (s @ v) / den[:, None]
        return out if rows is None else out[np.asarray(rows)]
    return f


PINS = [
    lambda: [test_matches_bruteforce(*c) for c in [(7, 8, 2), (16, 8, 2)]],
    test_last_row_is_the_noncausal_row,
    test_homogeneity_in_q,
    test_v_one_bound,
]


@pytest.mark.parametrize("kind", ["exclusive", "noncausal", "eps_inside", "sum_den"])
def test_a_pin_catches_the_mistake(kind, monkeypatch):
    monkeypatch.setattr(R, "rla_l2_causal_doc", _variant(kind))
    caught = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, kind


# ---------------------------------------------------------------- the layer (projections)

def _layer_case(seed, B=1, L=20, H=2, d=8):
    dm = H * d
    x = _rand(seed, (B, L, dm))
    gq = syn.rng(seed + 1).uniform(0.8, 1.2, (H, d))
    gk = syn.rng(seed + 2).uniform(0.8, 1.2, (H, d))
    return x, gq, gk, dm


def test_layer_with_identity_projections_is_the_attention():
    x, gq, gk, dm = _layer_case(50)
    eye = np.eye(dm)
    y = O.rapt_layer(x, np.vstack([eye, eye, eye]), eye, gq, gk, 2, pos_offset=3)
    q = x.reshape(1, 20, 2, 8)
    a, _, _ = O.rla2_prefill(q, q, q, gq, gk, 1e-6, 1e4, 1e-4, pos_offset=3)
    np.testing.assert_allclose(y, a.reshape(1, 20, dm), rtol=1e-12, atol=1e-14)


def test_layer_with_diagonal_projections():
    """W_qkv = [diag(a); diag(b); diag(c)] and W_o = diag(e) reduce the layer to the attention of
    the element-wise scaled inputs, scaled by e: this fixes the q | k | v order of the rows (the
    three scalings differ, and RMSNorm keeps a per-element scaling) and the head-major columns."""
    x, gq, gk, dm = _layer_case(51)
    a, b, c, e = (syn.rng(60 + i).uniform(0.2, 2.0, dm) for i in range(4))
    y = O.rapt_layer(x, np.vstack([np.diag(a), np.diag(b), np.diag(c)]), np.diag(e), gq, gk, 2)
    sh = (1, 20, 2, 8)
    att, _, _ = O.rla2_prefill((x * a).reshape(sh), (x * b).reshape(sh), (x * c).reshape(sh),
                               gq, gk, 1e-6, 1e4, 1e-4)
    np.testing.assert_allclose(y, att.reshape(1, 20, dm) * e, rtol=1e-12, atol=1e-14)
    swapped, _, _ = O.rla2_prefill((x * b).reshape(sh), (x * a).reshape(sh), (x * c).reshape(sh),
                                   gq, gk, 1e-6, 1e4, 1e-4)
    assert not np.allclose(y, swapped.reshape(1, 20, dm) * e, rtol=1e-6)


def test_layer_output_projection_permutes():
    x, gq, gk, dm = _layer_case(54)
    w = _rand(55, (3 * dm, dm))
    perm = syn.rng(56).permutation(dm)
    base = O.rapt_layer(x, w, np.eye(dm), gq, gk, 2)
    np.testing.assert_allclose(O.rapt_layer(x, w, np.eye(dm)[perm], gq, gk, 2), base[..., perm],
                               rtol=1e-12, atol=1e-14)
    # sampled rows agree with the full evaluation
    part = O.rapt_layer(x, w, np.eye(dm), gq, gk, 2, pairs_rows=(0, [0, 7, 19]))
    np.testing.assert_allclose(part[0, [0, 7, 19]], base[0, [0, 7, 19]], rtol=1e-12)
