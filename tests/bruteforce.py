"""Independent brute force for tiny RLA-2 / RLA cases: pure Python, float64, literal loops.

Written separately from ``oracle/`` (shares no code with it) so that the two can
pin each other on L <= 16. RoPE is applied here as a complex multiplication
(x_{2j} + i x_{2j+1}) * exp(i p theta_j), the textbook statement of the rotation,
instead of the oracle's cos/sin form; RMSNorm is an explicit sum.
"""

import cmath
import math


def feature_row(x, gamma, p, eps_norm, base):
    d = len(x)
    ms = 0.0
    for xi in x:
        ms += float(xi) * float(xi)
    ms /= d
    r = 1.0 / math.sqrt(ms + eps_norm)
    y = [float(x[i]) * r * float(gamma[i]) for i in range(d)]
    f = [0.0] * d
    for j in range(d // 2):
        theta = base ** (-(2.0 * j) / d)
        c = complex(y[2 * j], y[2 * j + 1]) * cmath.exp(1j * p * theta)
        f[2 * j] = c.real if c.real > 0 else 0.0
        f[2 * j + 1] = c.imag if c.imag > 0 else 0.0
    return f


def dot(a, b):
    s = 0.0
    for i in range(len(a)):
        s += a[i] * b[i]
    return s


def causal_head(qf, kf, v, eps_den, S0=None, z0=None):
    """qf, kf, v: lists of rows. Returns output rows of the inclusive causal form."""
    n = len(qf)
    dv = len(v[0]) if n else 0
    out = []
    for t in range(n):
        num = [0.0] * dv
        den = 0.0
        for tau in range(t + 1):
            s = dot(qf[t], kf[tau])
            for j in range(dv):
                num[j] += s * float(v[tau][j])
            den += s
        if S0 is not None:
            for j in range(dv):
                for i in range(len(qf[t])):
                    num[j] += qf[t][i] * float(S0[i][j])
        if z0 is not None:
            den += dot(qf[t], [float(x) for x in z0])
        out.append([num[j] / (den + eps_den) for j in range(dv)])
    return out


def l2_head(qf, kf, v, eps):
    n = len(qf)
    dv = len(v[0])
    out = []
    for t in range(n):
        num = [0.0] * dv
        ss = 0.0
        for i in range(n):
            s = dot(qf[t], kf[i])
            ss += s * s
            for j in range(dv):
                num[j] += s * float(v[i][j])
        out.append([num[j] / (math.sqrt(ss) + eps) for j in range(dv)])
    return out


def bidir_head(qf, kf, v, eps_den):
    """Every query sees every token of the sequence (non-causal Sum denominator)."""
    n = len(qf)
    dv = len(v[0]) if n else 0
    out = []
    for t in range(n):
        num = [0.0] * dv
        den = 0.0
        for tau in range(n):
            s = dot(qf[t], kf[tau])
            for j in range(dv):
                num[j] += s * float(v[tau][j])
            den += s
        out.append([num[j] / (den + eps_den) for j in range(dv)])
    return out


def l2_causal_head(qf, kf, v, eps):
    """Causal L2 denominator: query t sees keys 0..t; out = sum s v / (sqrt(sum s^2) + eps)."""
    n = len(qf)
    dv = len(v[0]) if n else 0
    out = []
    for t in range(n):
        num = [0.0] * dv
        ss = 0.0
        for i in range(t + 1):
            s = dot(qf[t], kf[i])
            ss += s * s
            for j in range(dv):
                num[j] += s * float(v[i][j])
        out.append([num[j] / (math.sqrt(ss) + eps) for j in range(dv)])
    return out
