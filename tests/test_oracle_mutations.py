"""Plants plausible mistakes in the oracle (on the CPU, via monkeypatch) and checks
that the pins in test_oracle_pins.py catch each one. Nothing here touches a GPU."""

import numpy as np
import pytest

import oracle
import oracle.rla2 as R
import test_oracle_pins as P

_orig_rope = R.rope_adjacent
_orig_rmsnorm = R.rmsnorm
_orig_causal = R.rla2_causal_doc
_orig_features = R.features
_orig_bidir = R.rla2_bidir_doc


def rope_wrong_sign(x, positions, base):
    return _orig_rope(x, -np.asarray(positions, dtype=np.float64), base)


def rope_half_split(x, positions, base):
    # pairs (i, i + d/2) instead of (2i, 2i+1)
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    perm = np.empty(d, dtype=np.int64)
    perm[0::2] = np.arange(d // 2)
    perm[1::2] = np.arange(d // 2) + d // 2
    y = _orig_rope(x[..., perm], positions, base)
    out = np.empty_like(y)
    out[..., perm] = y
    return out


def rope_wrong_freq(x, positions, base):
    # theta_j = base^(-j/d): emulate by a square-rooted base
    return _orig_rope(x, positions, np.sqrt(base))


def rmsnorm_eps_outside(x, gamma, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * np.asarray(gamma)


def causal_exclusive(qf, kf, v, eps_den=1e-4, S0=None, z0=None, rows=None):
    qf, kf, v = (np.asarray(a, np.float64) for a in (qf, kf, v))
    n = qf.shape[0]
    s = qf @ kf.T
    s = np.where(np.arange(n)[None, :] < np.arange(n)[:, None], s, 0.0)
    num, den = s @ v, s.sum(1)
    if S0 is not None:
        num = num + qf @ S0
    if z0 is not None:
        den = den + qf @ z0
    out = num / (den + eps_den)[:, None]
    rows = np.arange(n) if rows is None else rows
    Sf = kf.T @ v + (0 if S0 is None else S0)
    zf = kf.sum(0) + (0 if z0 is None else z0)
    return out[rows], Sf, zf


def causal_no_eps(qf, kf, v, eps_den=1e-4, S0=None, z0=None, rows=None):
    return _orig_causal(qf, kf, v, 0.0, S0, z0, rows)


def causal_transposed_state(qf, kf, v, eps_den=1e-4, S0=None, z0=None, rows=None):
    return _orig_causal(qf, kf, v, eps_den, None if S0 is None else np.asarray(S0).T, z0, rows)


def bidir_causal_mask(qf, kf, v, eps_den=1e-4, rows=None):
    # the non-causal form with the causal mask left in
    return _orig_causal(qf, kf, v, eps_den, rows=rows)[0]


def bidir_no_eps(qf, kf, v, eps_den=1e-4, rows=None):
    return _orig_bidir(qf, kf, v, 0.0, rows)


def bidir_l2_den(qf, kf, v, eps_den=1e-4, rows=None):
    # the original RLA's L2 denominator in place of the Sum denominator
    qf, kf, v = (np.asarray(a, np.float64) for a in (qf, kf, v))
    s = qf @ kf.T
    out = (s @ v) / (np.sqrt((s * s).sum(1)) + eps_den)[:, None]
    return out if rows is None else out[np.asarray(rows)]


def features_no_relu(x, gamma, positions, eps_norm, rope_base):
    return R.rope_adjacent(R.rmsnorm(x, gamma, eps_norm), positions, rope_base)


MUTANTS = {
    "rope_wrong_sign": ("rope_adjacent", rope_wrong_sign),
    "rope_half_split": ("rope_adjacent", rope_half_split),
    "rope_wrong_freq": ("rope_adjacent", rope_wrong_freq),
    "rmsnorm_eps_outside": ("rmsnorm", rmsnorm_eps_outside),
    "causal_exclusive": ("rla2_causal_doc", causal_exclusive),
    "causal_no_eps": ("rla2_causal_doc", causal_no_eps),
    "causal_transposed_state": ("rla2_causal_doc", causal_transposed_state),
    "features_no_relu": ("features", features_no_relu),
    "bidir_causal_mask": ("rla2_bidir_doc", bidir_causal_mask),
    "bidir_no_eps": ("rla2_bidir_doc", bidir_no_eps),
    "bidir_l2_den": ("rla2_bidir_doc", bidir_l2_den),
}


def _pins():
    return [
        lambda: P.test_prefill_matches_bruteforce(5, 8, 2, True),
        lambda: P.test_prefill_matches_bruteforce(1, 2, 1, False),
        P.test_varlen_matches_bruteforce,
        P.test_disjoint_supports_give_exact_zero,
        P.test_single_token_closed_form,
        P.test_rope_properties,
        P.test_rmsnorm_properties,
        P.test_decode_equals_prefill,
        lambda: P.test_bidir_matches_bruteforce(5, 8, 2),
        P.test_bidir_key_order_invariance,
        P.test_bidir_constant_v_closed_form,
    ]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(R, attr, fn)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    caught = 0
    with np.errstate(all="ignore"):
        for pin in _pins():
            try:
                pin()
            except AssertionError:
                caught += 1
    assert caught > 0, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_the_same_pins():
    for pin in _pins():
        pin()
