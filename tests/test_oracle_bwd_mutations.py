"""Plants plausible mistakes in the backward oracle (on the CPU, via monkeypatch) and checks that
the pins in test_oracle_bwd.py catch each one. Nothing here touches a GPU."""

import numpy as np
import pytest

import oracle.rla2_bwd as RB
import test_oracle_bwd as P

_orig_doc = RB.rla2_causal_doc_bwd
_orig_rms = RB.rmsnorm_bwd
_orig_rope_adj = RB.rope_adjacent


def _doc_variant(drop_scale=False, flip_scale=False, exclusive_keys=False, unmasked_dv=False):
    def f(qf, kf, v, dout, eps_den=1e-4):
        qf, kf, v, g = (np.asarray(x, np.float64) for x in (qf, kf, v, dout))
        n = qf.shape[0]
        causal = np.arange(n)[None, :] <= np.arange(n)[:, None]
        s = np.where(causal, qf @ kf.T, 0.0)
        num = s @ v
        den = s.sum(axis=1) + eps_den
        gnum = g / den[:, None]
        scale = -np.sum(g * num, axis=1) / den ** 2
        if drop_scale:
            scale = 0.0 * scale
        if flip_scale:
            scale = -scale
        a = np.where(causal, gnum @ v.T + scale[:, None], 0.0)
        dqf = a @ kf
        mk = np.arange(n)[None, :] < np.arange(n)[:, None] if exclusive_keys else causal
        dkf = np.where(mk, a, 0.0).T @ qf
        dv = (qf @ kf.T).T @ gnum if unmasked_dv else s.T @ gnum
        return dqf, dkf, dv
    return f


def _rms_no_cubic(x, gamma, eps, dy):
    x, dy, g = np.asarray(x, np.float64), np.asarray(dy, np.float64), np.asarray(gamma, np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return r * g * dy, dy * x * r


def _rms_dgamma_without_r(x, gamma, eps, dy):
    dx, dg = _orig_rms(x, gamma, eps, dy)
    x = np.asarray(x, np.float64)
    return dx, np.asarray(dy, np.float64) * x


def _rms_cubic_without_d(x, gamma, eps, dy):
    x, dy, g = np.asarray(x, np.float64), np.asarray(dy, np.float64), np.asarray(gamma, np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    dot = np.sum(g * dy * x, axis=-1, keepdims=True)
    return r * g * dy - x * r ** 3 * dot, dy * x * r


def _rope_bwd_forward_direction(dy, positions, base):
    return _orig_rope_adj(dy, np.asarray(positions, np.float64), base)


PINS = [
    lambda: [P.test_directional_derivative_matches_finite_difference(w, True) for w in range(5)],
    P.test_every_element_against_the_brute_force,
    P.test_euler_identity_in_v,
    P.test_rmsnorm_scale_identity,
    P.test_rope_backward_is_the_inverse_rotation,
]

MUTANTS = {
    "dropped denominator term": ("rla2_causal_doc_bwd", _doc_variant(drop_scale=True)),
    "denominator term with the wrong sign": ("rla2_causal_doc_bwd", _doc_variant(flip_scale=True)),
    "exclusive suffix for the keys": ("rla2_causal_doc_bwd", _doc_variant(exclusive_keys=True)),
    "value gradient without the causal mask": ("rla2_causal_doc_bwd", _doc_variant(unmasked_dv=True)),
    "RMSNorm backward without the r^3 term": ("rmsnorm_bwd", _rms_no_cubic),
    "RMSNorm r^3 term without 1/d": ("rmsnorm_bwd", _rms_cubic_without_d),
    "gain gradient without the 1/rms factor": ("rmsnorm_bwd", _rms_dgamma_without_r),
    "RoPE backward rotating forward": ("rope_adjacent_bwd", _rope_bwd_forward_direction),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_a_pin_catches_the_mistake(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(RB, attr, fn)
    caught = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, "no pin caught: " + name


def test_unmutated_oracle_passes_every_pin():
    for pin in PINS:
        pin()
