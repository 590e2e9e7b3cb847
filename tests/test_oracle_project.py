"""Pins for the oracle's K/V projection (the input of the fused projection +
append path): brute force on tiny shapes, a closed form with selection
weights, and linearity -- each would catch a transposed operand, a wrong
head / channel index or a dropped term."""
import itertools

import numpy as np

import oracle


def _brute(x, w, Hkv, D):
    B, T, E = x.shape
    out = np.zeros((B, T, Hkv, D))
    for b, i, h, j in itertools.product(range(B), range(T), range(Hkv), range(D)):
        s = 0.0
        for e in range(E):
            s += float(x[b, i, e]) * float(w[h * D + j, e])
        out[b, i, h, j] = s
    return out


def test_projection_matches_brute_force_on_tiny_shapes():
    rng = np.random.default_rng(5)
    B, T, E, Hkv, D = 2, 3, 5, 2, 3          # hidden != Hkv * D, so a transposed weight cannot fit
    x = rng.integers(-4, 5, (B, T, E)).astype(np.float32)
    wk = rng.integers(-3, 4, (Hkv * D, E)).astype(np.float32)
    wv = rng.integers(-3, 4, (Hkv * D, E)).astype(np.float32)
    k, v = oracle.project_kv(x, wk, wv, Hkv, D)
    np.testing.assert_array_equal(k, _brute(x, wk, Hkv, D))   # small integers: exact
    np.testing.assert_array_equal(v, _brute(x, wv, Hkv, D))


def test_selection_weights_copy_input_features():
    # row h*D + j of w_k selects input feature perm[h*D + j]: k is x gathered by perm
    rng = np.random.default_rng(9)
    B, T, Hkv, D = 2, 4, 2, 8
    E = Hkv * D + 3
    x = rng.standard_normal((B, T, E))
    perm = rng.permutation(E)[:Hkv * D]
    wk = np.zeros((Hkv * D, E))
    wk[np.arange(Hkv * D), perm] = 1.0
    wv = 2.0 * wk
    k, v = oracle.project_kv(x, wk, wv, Hkv, D)
    np.testing.assert_array_equal(k, x[:, :, perm].reshape(B, T, Hkv, D))
    np.testing.assert_array_equal(v, 2.0 * x[:, :, perm].reshape(B, T, Hkv, D))


def test_projection_is_linear_in_the_input():
    rng = np.random.default_rng(11)
    B, T, E, Hkv, D = 1, 6, 32, 2, 4
    x1 = rng.integers(-8, 9, (B, T, E)).astype(np.float64)
    x2 = rng.integers(-8, 9, (B, T, E)).astype(np.float64)
    w = rng.integers(-5, 6, (Hkv * D, E)).astype(np.float64)
    k1, _ = oracle.project_kv(x1, w, w, Hkv, D)
    k2, _ = oracle.project_kv(x2, w, w, Hkv, D)
    k12, v12 = oracle.project_kv(x1 + x2, w, w, Hkv, D)
    np.testing.assert_array_equal(k12, k1 + k2)
    np.testing.assert_array_equal(v12, k12)
