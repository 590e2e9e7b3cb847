"""Bit-exact parity of the CUDA quantizer with the fp64 oracle on inputs placed
within one binary32 rounding of every decision boundary (tests/_near_ties.py):
outlier thresholds, affine-code and scale midpoints, e4m3 / e2m1 midpoints,
and Lloyd-Max centroids a quarter binary32 step off an fp16 midpoint.  The
kernels take these decisions in binary32 with a certified error bound and
fall back to fp64 where the bound does not settle them; a wrong bound or a
fallback that differs from the definition shows up here as a differing byte.
"""
import numpy as np
import pytest
import torch

import _near_ties as nt
from _kvq_pairs import Pair
from sub_byte_quantized_kvq_gb300 import kvq

pytestmark = pytest.mark.gpu

F32 = np.float32


def _outlier_rows(rng, T, D, big):
    return np.stack([nt.outlier_tie_vector(rng, D, int(rng.integers(0, D)), t % 3, scale=float(rng.uniform(0.2, 5)),
                                           big=big, side=1 if rng.integers(0, 2) else -1) for t in range(T)])


def _lloyd_rows(rng, T, D):
    return np.stack([nt.lloyd_tie_channel(rng, T)[0] for _ in range(D)], 1)


def _affine_rows(rng, T, D, levels):
    return np.stack([nt.affine_tie_values(rng, T, levels, T // 3, s_tie=c % 3 == 0) for c in range(D)], 1)


def _page_stream(rng, fmt, npages, D, tiers_row):
    """[npages * 16, D] binary32 rows for one (sequence, kv head, K|V): pages
    cycle through outlier ties, Lloyd ties and affine ties (groups of four
    pages for the group format); FP8 tier pages carry e4m3 midpoints."""
    big = tuple(sorted(rng.choice(D, 4, replace=False).tolist()))
    out = []
    if fmt == kvq.KVQ_FMT_CB2_GROUP4:
        for g in range(npages // 4):
            kind = g % 2
            out.append(_outlier_rows(rng, 64, D, big) if kind == 0 else _lloyd_rows(rng, 64, D))
        return np.concatenate(out)
    for p in range(npages):
        if tiers_row is not None and tiers_row[p]:
            out.append(nt.fp8_tie_page(rng, D))
            continue
        kind = p % 3
        if kind == 0 and fmt != kvq.KVQ_FMT_CB2_STATIC:
            out.append(_outlier_rows(rng, 16, D, big))
        elif kind == 2 and fmt == kvq.KVQ_FMT_ASYM3_OUTLIER:
            out.append(_affine_rows(rng, 16, D, 7))
        else:
            out.append(_lloyd_rows(rng, 16, D))
    return np.concatenate(out)


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_CB2_OUTLIER, kvq.KVQ_FMT_TIERED, kvq.KVQ_FMT_ASYM3_OUTLIER,
                                 kvq.KVQ_FMT_CB2_GROUP4, kvq.KVQ_FMT_CB2_STATIC])
@pytest.mark.parametrize("D", [64, 128])
def test_page_formats_bit_exact_on_decision_boundaries(fmt, D):
    rng = np.random.default_rng(100 + fmt + D)
    B, Hkv = 2, 2
    npages = 8 if fmt == kvq.KVQ_FMT_CB2_GROUP4 else 6
    tiers = None
    if fmt == kvq.KVQ_FMT_TIERED:
        tiers = np.zeros((B, npages), bool)
        tiers[:, 1::3] = True
    pair = Pair(fmt, B, Hkv, D, npages, seed=7, tiers=tiers)
    T = 16 * npages
    kv = np.zeros((2, B, T, Hkv, D), F32)
    for r in range(2):
        for b in range(B):
            for h in range(Hkv):
                kv[r, b, :, h] = _page_stream(rng, fmt, npages, D, None if tiers is None else tiers[b])
    k, v = torch.from_numpy(kv[0]), torch.from_numpy(kv[1])
    pair.append(k[:, :21], v[:, :21])      # a staged partial page first, then the rest
    pair.append(k[:, 21:].contiguous(), v[:, 21:].contiguous())
    pair.assert_cache_equal()


@pytest.mark.parametrize("D", [64, 128])
def test_int4_bit_exact_on_decision_boundaries(D):
    rng = np.random.default_rng(200 + D)
    B, Hkv, T = 2, 2, 40
    pair = Pair(kvq.KVQ_FMT_INT4_G32, B, Hkv, D, 3, seed=8)
    kv = np.zeros((2, B, T, Hkv, D), F32)
    for idx in np.ndindex(2, B, T, Hkv):
        groups = []
        for g in range(D // 32):
            if (idx[2] + g) % 3 == 0:
                groups.append(nt.outlier_tie_vector(rng, 32, int(rng.integers(0, 32)), idx[2] % 3,
                                                    scale=float(rng.uniform(0.2, 5)), side=1 if g % 2 else -1))
            else:
                groups.append(nt.affine_tie_values(rng, 32, 15, 10, s_tie=(idx[2] + g) % 3 == 1))
        kv[idx] = np.concatenate(groups)
    pair.append(torch.from_numpy(kv[0]), torch.from_numpy(kv[1]))
    pair.assert_cache_equal()


@pytest.mark.parametrize("D", [64, 128])
def test_e2m1_bit_exact_on_decision_boundaries(D):
    rng = np.random.default_rng(300 + D)
    B, Hkv, T = 2, 2, 40
    pair = Pair(kvq.KVQ_FMT_FP4_E2M1_S16, B, Hkv, D, 3, seed=9)
    kv = np.zeros((2, B, T, Hkv, D), F32)
    for idx in np.ndindex(2, B, T, Hkv):
        kv[idx] = np.concatenate([nt.e2m1_tie_block(rng, scale_tie=(idx[2] + s) % 2 == 0) for s in range(D // 16)])
    pair.append(torch.from_numpy(kv[0]), torch.from_numpy(kv[1]))
    pair.assert_cache_equal()


def coarse_grid_kv(rng, B, T, Hkv, D, step, tiny):
    """K, V float32 [2, B, T, Hkv, D] on multiples of `step` in [-2, 2] with one
    outlier channel; `tiny` puts a value of 2^-30 in row 3 of every page, so
    the values span more than 24 bits and no cell sum is exact in binary32."""
    levels = np.arange(-2.0, 2.0 + step, step, dtype=F32)
    kv = rng.choice(levels, size=(2, B, T, Hkv, D)).astype(F32)
    kv[:, :, :, :, 5] *= 8.0   # an outlier channel
    if tiny:
        kv[:, :, 3::16] = F32(2.0 ** -30)
    return kv


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_CB2_OUTLIER, kvq.KVQ_FMT_CB2_GROUP4, kvq.KVQ_FMT_CB2_STATIC])
@pytest.mark.parametrize("step", [0.25, 0.125])
@pytest.mark.parametrize("tiny", [False, True])
def test_lloyd_on_a_coarse_value_grid_bit_exact(fmt, step, tiny):
    """Values on a coarse grid (multiples of `step` in [-2, 2], plus a few
    large ones): a value often sits exactly on the midpoint of two cell means
    or at the same distance from both.  The binary32 margin cannot settle
    such rows; they take the fp64 distances of the definition, from exact
    binary32 sums or (tiny: the sums are inexact) from fp64 means of the
    cells, and the cache must match the oracle bit for bit."""
    rng = np.random.default_rng(int(400 + 1000 * step) + fmt + 7 * tiny)
    B, Hkv, D = 2, 2, 128
    npages = 8
    pair = Pair(fmt, B, Hkv, D, npages, seed=11)
    T = 16 * npages
    kv = coarse_grid_kv(rng, B, T, Hkv, D, step, tiny)
    k, v = torch.from_numpy(kv[0]), torch.from_numpy(kv[1])
    dt = torch.bfloat16 if not tiny else torch.float32   # the grid is exact in bf16; 2^-30 rows need fp32
    pair.append(k[:, :37].contiguous(), v[:, :37].contiguous(), dtype=dt)
    pair.append(k[:, 37:].contiguous(), v[:, 37:].contiguous(), dtype=dt)
    pair.assert_cache_equal()
