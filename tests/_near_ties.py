"""Inputs that sit on the quantizer's decision boundaries.

Each generator returns binary32 values placed within one binary32 rounding
of a boundary where the quantizer takes an integer decision: the outlier
threshold |x - mu| = sigma * s, the midpoints k + 1/2 of an affine code, the
fp16 / e4m3 / e2m1 rounding midpoints of a scale or a code, and the fp16
midpoint of a Lloyd-Max centroid.  There the decision depends on the
precision it is taken in: the quantizer is defined in fp64, and binary32
arithmetic can land on the other side.  The exact decisions are computed here
with rational arithmetic (fractions.Fraction), which is what the oracle's
fp64 results must match and what the CUDA path must reproduce bit for bit.

These are test inputs only: nothing here quantizes a cache.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

F32 = np.float32


def f32_neighbours(r: float, k: int = 1):
    """The binary32 values nearest to r: round(r) and k steps either side."""
    x = F32(r)
    out = [x]
    lo = hi = x
    for _ in range(k):
        lo = np.nextafter(lo, F32(-np.inf))
        hi = np.nextafter(hi, F32(np.inf))
        out += [lo, hi]
    return out


# ----------------------------------------------------------------------------- outlier threshold
def exact_outliers(x, sigma: int = 3):
    """Exact decisions |x_i - mu| > sigma * s (mu the mean, s the unbiased
    standard deviation) over rationals: (x_i - mu)^2 > sigma^2 s^2."""
    xs = [Fraction(float(v)) for v in x]
    n = len(xs)
    mu = sum(xs) / n
    var = sum((v - mu) ** 2 for v in xs) / (n - 1)
    return np.array([(v - mu) ** 2 > sigma * sigma * var for v in xs])


def outlier_tie_vector(rng, n: int, which: int, pick: int, scale: float = 1.0, big=(), side: int = 1):
    """A binary32 vector of n values whose element `which` is one of the binary32
    neighbours (pick in 0..2) of a value that puts it exactly on the threshold
    |x - mu| = 3 s (mu, s computed with that element included): the root
    above the others' mean (side = 1) or below it (side = -1)."""
    y = (rng.standard_normal(n) * scale).astype(F32)
    for c in big:
        y[c] = F32(y[c] * 8)
    y[which] = 0
    A = float(np.sum(y.astype(np.float64)))
    Q = float(np.sum(y.astype(np.float64) ** 2))
    # with x in place: (n-1) ((n-1) x - A)^2 = 9 n^2 Q - 9 n A^2 + 9 n (n-1) x^2 - 18 n A x
    a = (n - 1) ** 3 - 9 * n * (n - 1)
    b = -2 * (n - 1) ** 2 * A + 18 * n * A
    c = (n - 1) * A * A - 9 * n * n * Q + 9 * n * A * A
    r = math.sqrt(b * b - 4 * a * c)
    roots = sorted([(-b - r) / (2 * a), (-b + r) / (2 * a)])
    y[which] = f32_neighbours(roots[1] if side > 0 else roots[0])[pick]
    return y


# ----------------------------------------------------------------------------- affine codes (INT4 groups, ASYM3 channels)
def fp16_rne(q: Fraction) -> float:
    """fp16 round-to-nearest-even of a rational, via its correctly rounded fp64
    value (53 bits is far more than the 11 fp16 keeps, and the quotients here
    are never within 2^-53 of an fp16 midpoint without being on it)."""
    return float(np.float16(float(q)))


def affine_scale(mn, mx, levels: int):
    """(S, m) as fp16 values: S = fp16((mx - mn) / levels), m = fp16(mn)."""
    S = fp16_rne((Fraction(float(mx)) - Fraction(float(mn))) / levels)
    return S, float(np.float16(float(mn)))


def exact_affine_code(x, m: float, S: float, qmax: int) -> int:
    """clamp(round-half-even((x - m) / S), 0, qmax) over rationals."""
    r = (Fraction(float(x)) - Fraction(m)) / Fraction(S)
    q = round(r)    # Python rounds a Fraction half to even
    return max(0, min(qmax, q))


def affine_tie_values(rng, n: int, levels: int, n_ties: int, s_tie: bool):
    """n binary32 values in (-1, 1) (no 3-sigma outlier can occur: every
    deviation is below 2 while 3 s exceeds 1.7 for such spreads) with n_ties
    of them moved onto binary32 neighbours of the code midpoints
    m + (k + 1/2) S.  With s_tie, max - min is chosen so that (max - min) /
    levels lies within a binary32 rounding of an fp16 midpoint."""
    while True:
        v = rng.uniform(-1, 1, n).astype(F32)
        if s_tie:
            # an fp16 midpoint of the scale's binade, then max = min + levels * midpoint (nudged)
            S0 = float(np.float16(float(v.max() - v.min()) / levels))
            up = float(np.nextafter(np.float16(S0), np.float16(np.inf)))
            mid = (S0 + up) / 2
            i_mn, i_mx = int(np.argmin(v)), int(np.argmax(v))
            v[i_mx] = f32_neighbours(float(v[i_mn]) + levels * mid)[int(rng.integers(0, 3))]
            if not (v[i_mx] >= v).all():
                continue
        mn, mx = v.min(), v.max()
        S, m = affine_scale(mn, mx, levels)
        if S == 0:
            continue
        idx = [i for i in rng.permutation(n) if v[i] != mn and v[i] != mx][:n_ties]
        for i in idx:
            k = int(rng.integers(0, levels))
            cand = f32_neighbours(m + (k + 0.5) * S)[int(rng.integers(0, 3))]
            if mn < cand < mx:
                v[i] = cand
        if v.min() == mn and v.max() == mx and not exact_outliers(v).any():
            return v


# ----------------------------------------------------------------------------- e4m3 / e2m1 rounding
def e4m3_values():
    """The finite non-negative e4m3 magnitudes in increasing order."""
    vals = set()
    for e in range(16):
        for mnt in range(8):
            if e == 15 and mnt == 7:
                continue
            vals.add(mnt / 8 * 2.0 ** -6 if e == 0 else (1 + mnt / 8) * 2.0 ** (e - 7))
    return sorted(vals)


E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1_tie_block(rng, scale_tie: bool):
    """16 binary32 values: with scale_tie, amax / 6 within a binary32 rounding of
    an e4m3 midpoint; the other values on binary32 neighbours of s * (e2m1
    midpoint), s the scale that amax gives."""
    ev = e4m3_values()
    while True:
        if scale_tie:
            i = int(rng.integers(40, 100))
            mid = (ev[i] + ev[i + 1]) / 2
            amax = f32_neighbours(6 * mid)[int(rng.integers(0, 3))]
        else:
            amax = F32(rng.uniform(0.5, 40))
        q = Fraction(float(amax)) / 6
        s = e4m3_rne(q)
        if s == 0:
            continue
        x = np.zeros(16, F32)
        x[0] = amax if rng.integers(0, 2) else -amax
        for j in range(1, 16):
            k = int(rng.integers(0, 7))
            mid = (E2M1[k] + E2M1[k + 1]) / 2
            cand = f32_neighbours(s * mid)[int(rng.integers(0, 3))]
            if abs(cand) <= abs(amax):
                x[j] = cand if rng.integers(0, 2) else -cand
        return rng.permutation(x)


def e4m3_rne(q: Fraction) -> float:
    """e4m3 (bias 7, 3 mantissa bits, satfinite at 448) of a non-negative rational,
    ties to even, by exact comparison with the midpoints."""
    ev = e4m3_values()
    if q >= 448:
        return 448.0
    for a, b in zip(ev[:-1], ev[1:]):
        if q <= b:
            mid = Fraction(a) + (Fraction(b) - Fraction(a)) / 2
            if q < mid:
                return a
            if q > mid:
                return b
            # tie: the even code (mantissa LSB 0)
            return a if ev.index(a) % 2 == 0 else b
    return 448.0


def fp8_tie_page(rng, D: int):
    """16 x D binary32 values for an FP8 tier page (s = fp32(amax / 448)): most
    values on binary32 neighbours of s * (e4m3 midpoint)."""
    ev = e4m3_values()
    amax = F32(rng.uniform(1, 60))
    s = float(F32(float(amax) / 448.0))
    x = (rng.standard_normal((16, D)) * float(amax) / 4).astype(F32)
    x = np.clip(x, -amax, amax)
    x[0, 0] = amax
    for t in range(16):
        for c in range(D):
            if (t, c) == (0, 0) or rng.random() < 0.3:
                continue
            i = int(rng.integers(0, len(ev) - 1))
            cand = f32_neighbours(s * (ev[i] + ev[i + 1]) / 2)[int(rng.integers(0, 3))]
            if abs(cand) <= amax:
                x[t, c] = cand if rng.integers(0, 2) else -cand
    return x


# ----------------------------------------------------------------------------- Lloyd-Max centroids on fp16 midpoints
def fp16_midpoint_near(v: float) -> float:
    h = np.float16(v)
    up = np.nextafter(h, np.float16(np.inf))
    return (float(h) + float(up)) / 2


def lloyd_tie_channel(rng, n: int = 16):
    """n binary32 values in four tight, evenly spread clusters (so the linspace
    start puts one centroid in each and the fit converges to the cluster
    means).  Each cluster is three copies of an fp16 midpoint M and one value
    one binary32 step above or below it: its mean, M +- ulp(M) / 4, is not a
    binary32 number; a binary32 sum rounds it onto M itself (a rounding tie,
    resolved to the even fp16), fp64 keeps it and rounds away from the tie."""
    base = rng.uniform(-4, -2)
    gap = rng.uniform(1.5, 2.5)
    vals, means = [], []
    for j in range(4):
        M = fp16_midpoint_near(base + j * gap)
        step = np.nextafter(F32(M), F32(np.inf) if rng.integers(0, 2) else F32(-np.inf))
        cl = [F32(M)] * (n // 4 - 1) + [step]
        vals += cl
        means.append(sum(Fraction(float(v)) for v in cl) / len(cl))
    return rng.permutation(np.array(vals, F32)), means
