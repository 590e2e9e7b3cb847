"""Pins for the oracle's quantizers against closed forms, exact library
statistics, brute force and the error bounds the formats imply.

Sources:
  "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression",
  Paradigm 2 (outlier isolation; 4-centroid codebook via k-means, the
  compress_kv_head listing's linspace start and argmin assignment).
  "The Sub-10ms Barrier: Fusing Sparse MoE Routing with FP4 KV-Cache
  Quantization", section 2 (S = (max - min) / (2^b - 1); E2M1).
  "Hierarchical Token Gating and Tiered KV-Cache Paging", section 2 (FP8 tier).
"""
import itertools
import statistics
from fractions import Fraction

import numpy as np
import pytest

import oracle

R_K, R_V = 0, 1


# ------------------------------------------------------------------ outliers
def test_outlier_rule_matches_exact_statistics():
    """Decisions (taken in fp64) equal those from Python's exact-rational mean
    and variance of the same values, with no band skipped (the fp64 rounding
    of the statistics is far below these margins; inputs placed on the
    threshold itself are in test_oracle_near_ties.py)."""
    rng = np.random.default_rng(0)
    checked = 0
    for trial in range(300):
        n = [32, 64, 128][trial % 3]
        x = rng.standard_normal(n)
        x[rng.integers(0, n, 3)] *= rng.uniform(2, 12)
        x = x.astype(np.float32).astype(np.float64)
        mask, k = oracle.outlier_mask(x, 3.0, cap=n)
        xs = [Fraction(float(v)) for v in x]
        mu = sum(xs) / n
        var = sum((v - mu) ** 2 for v in xs) / (n - 1)
        for i, v in enumerate(xs):
            assert mask[i] == ((v - mu) ** 2 > 9 * var)
            checked += 1
    assert checked > 20000


@pytest.mark.parametrize("n", [32, 64, 128])
def test_outlier_count_bound(n):
    """k outliers need k*9*s^2 < (n-1)*s^2: at most ceil((n-1)/9)-1 of them."""
    assert oracle.kmax(n) == {32: 3, 64: 6, 128: 14}[n]
    rng = np.random.default_rng(n)
    worst = 0
    for _ in range(500):
        x = rng.standard_normal(n)
        m = rng.integers(1, n // 4)
        x[:m] += rng.choice([-1, 1], m) * rng.uniform(5, 50, m)
        _, k = oracle.outlier_mask(x, 3.0, cap=n)   # uncapped
        worst = max(worst, k)
        assert k <= oracle.kmax(n)
    # closed form: k equal spikes over n-k zeros are all outliers iff
    # (1 - k/n)^2 > 9 k (n-k) / (n (n-1)), i.e. (n-k)(n-1) > 9 k n
    for k in range(1, n // 2):
        x = np.zeros(n)
        x[:k] = 1.0
        mask, got = oracle.outlier_mask(x, 3.0, cap=n)
        expect = (n - k) * (n - 1) > 9 * k * n
        assert got == (k if expect else 0) and (mask[:k].all() == expect)


def test_outlier_special_cases():
    assert oracle.outlier_mask(np.full(128, 2.5))[1] == 0          # s == 0
    assert oracle.outlier_mask(np.arange(128.0))[1] == 0           # uniform ramp: max dev 1.7 s
    x = np.zeros(128)
    x[5] = 100.0
    m, k = oracle.outlier_mask(x)
    assert k == 1 and m[5]


# ------------------------------------------------------------------ Lloyd-Max
def _brute_optimum(v):
    """Minimum squared distortion over all partitions of sorted values into at
    most 4 contiguous cells (optimal 1-D quantizer cells are intervals)."""
    s = np.sort(v)
    n = len(s)
    best = np.inf
    for k in range(1, min(4, n) + 1):
        for cuts in itertools.combinations(range(1, n), k - 1):
            edges = (0,) + cuts + (n,)
            d = sum(((s[a:b] - s[a:b].mean()) ** 2).sum() for a, b in zip(edges[:-1], edges[1:]))
            best = min(best, d)
    return best


def _distortion(v, c):
    return sum(min((float(x) - float(cj)) ** 2 for cj in c) for x in v)


def test_lloyd_never_beats_brute_force_and_hits_it_on_clusters():
    rng = np.random.default_rng(1)
    for trial in range(120):
        n = int(rng.integers(1, 13))
        v = (rng.standard_normal(n) * rng.uniform(0.1, 5)).astype(np.float32).astype(np.float64)
        c, _, _, _ = oracle.lloyd4(v)
        opt = _brute_optimum(v)
        assert _distortion(v, c) >= opt - 1e-5 * max(opt, 1e-6)
    # evenly spaced, well separated clusters: the linspace start puts one
    # centroid in each cluster's cell, so Lloyd reaches the global optimum
    for trial in range(40):
        centers = rng.uniform(-20, 20) + rng.uniform(5, 20) * np.arange(4)
        v = np.concatenate([cc + rng.uniform(-0.5, 0.5, 4) for cc in centers]).astype(np.float32).astype(np.float64)
        rng.shuffle(v)
        c, _, _, _ = oracle.lloyd4(v)
        opt = _brute_optimum(v)
        assert abs(_distortion(v, c) - opt) <= 1e-5 * max(opt, 1e-3)


def test_lloyd_fixed_point_and_codes():
    rng = np.random.default_rng(2)
    for _ in range(200):
        n = int(rng.integers(1, 17))
        v = rng.standard_normal(n).astype(np.float32).astype(np.float64)
        c, c16, codes, passes = oracle.lloyd4(v, iters=64)
        # converged: each non-empty cell's centroid is the mean of its members
        assign = np.array([int(np.argmin(np.abs(x - c.astype(np.float64)))) for x in v])
        for j in range(4):
            if (assign == j).any():
                assert abs(float(c[j]) - v[assign == j].mean()) <= 1e-5 * max(1, abs(float(c[j])))
        # final codes: nearest fp16 centroid, first index on ties (numpy argmin's rule)
        cf = np.array([oracle.fp16_decode(h) for h in c16])
        assert (codes == np.array([int(np.argmin(np.abs(x - cf))) for x in v])).all()
        assert all(h == np.array(float(cj), np.float64).astype(np.float16).view(np.uint16) for h, cj in zip(c16, c))


def test_lloyd_special_cases():
    c, c16, codes, _ = oracle.lloyd4(np.full(16, 1.25))
    assert (c == 1.25).all() and (codes == 0).all()
    c, c16, codes, _ = oracle.lloyd4(np.array([]))
    assert (c16 == 0).all()
    # linspace start (as the listing) on 4 equally spaced points is already optimal
    c, _, codes, passes = oracle.lloyd4(np.array([0.0, 1.0, 2.0, 3.0]))
    assert list(c) == [0, 1, 2, 3] and list(codes) == [0, 1, 2, 3] and passes == 2


# ------------------------------------------------------------------ per-format error bounds
def _ulp16(x):
    return float(np.spacing(np.float16(abs(x)))) if np.isfinite(np.float16(abs(x))) else np.inf


def test_int4_group_bounds():
    """Non-outliers: |x - xh| <= S/2 + |m - mn| + fp32 rounding; outliers exact fp16."""
    rng = np.random.default_rng(3)
    D = 64
    for trial in range(60):
        x = rng.standard_normal(D).astype(np.float32) * rng.uniform(0.01, 10)
        x[rng.integers(0, D, 2)] *= 10
        blk = np.zeros(oracle.block_stride(oracle.BLK_INT4, D), np.uint8)
        t = int(rng.integers(0, 16))
        oracle.quantize_token(oracle.BLK_INT4, D, x, t, blk, role=trial % 2)
        xh = oracle.dequantize_block(oracle.BLK_INT4, D, blk, role=trial % 2)[t]
        for g in range(D // 32):
            seg = x[32 * g:32 * g + 32].astype(np.float64)
            mask, _ = oracle.outlier_mask(seg, 3.0)
            assert mask.sum() <= 3
            norm = seg[~mask]
            S = float(np.float16((norm.max() - norm.min()) / 15))
            m = float(np.float16(norm.min()))
            for i in range(32):
                c = 32 * g + i
                if mask[i]:
                    assert xh[c] == np.float32(np.float16(seg[i]))
                else:
                    bound = S / 2 + abs(m - norm.min()) + 2 * _ulp16(S) * 15 + 1e-6 * abs(seg[i])
                    assert abs(xh[c] - seg[i]) <= bound + 1e-7


def test_e2m1_block_bounds():
    rng = np.random.default_rng(4)
    D = 128
    for trial in range(40):
        x = (rng.standard_t(4, D) / np.sqrt(2)).astype(np.float32) * rng.uniform(0.001, 100)
        blk = np.zeros(oracle.block_stride(oracle.BLK_E2M1, D), np.uint8)
        oracle.quantize_token(oracle.BLK_E2M1, D, x, 7, blk, role=trial % 2)
        xh = oracle.dequantize_block(oracle.BLK_E2M1, D, blk, role=trial % 2)[7]
        for s in range(D // 16):
            seg = x[16 * s:16 * s + 16].astype(np.float64)
            amax = np.abs(seg).max()
            sc = oracle.e4m3_decode(oracle.e4m3_encode(float(np.float32(amax / 6))))
            for i in range(16):
                r = seg[i] / sc
                # half the local grid spacing, plus the saturation loss when s rounded down
                spacing = 0.5 if abs(r) < 2 else (1.0 if abs(r) < 4 else 2.0)
                bound = sc * spacing / 2 + max(0.0, amax - 6 * sc) + 1e-6 * abs(seg[i])
                assert abs(xh[16 * s + i] - seg[i]) <= bound


def test_fp8_page_bounds():
    rng = np.random.default_rng(5)
    D = 128
    for trial in range(10):
        x = rng.standard_normal((16, D)).astype(np.float32) * rng.uniform(0.01, 50)
        blk = oracle.quantize_page(oracle.BLK_FP8, D, x, role=trial % 2)
        xh = oracle.dequantize_block(oracle.BLK_FP8, D, blk, role=trial % 2)
        s = np.float32(np.abs(x).max() / np.float32(448))
        rel = np.abs(xh - x) / np.maximum(np.abs(x), 2.0 ** -6 * s)
        assert rel.max() <= 2.0 ** -4 + 1e-6           # 3 mantissa bits: half-ulp = 2^-4 relative


def test_cb2_page_properties():
    rng = np.random.default_rng(6)
    D = 128
    for trial in range(8):
        x = rng.standard_normal((16, D)).astype(np.float32)
        x[:, rng.choice(D, 4, replace=False)] *= 8
        role = trial % 2
        blk = oracle.quantize_page(oracle.BLK_CB2, D, x, role=role)
        xh = oracle.dequantize_block(oracle.BLK_CB2, D, blk, role=role)
        masks = np.array([oracle.outlier_mask(x[t].astype(np.float64))[0] for t in range(16)])
        # side-list grouped by channel: header {n_ch, total}, then one 20-byte
        # record {channel, 0, token mask, 16 e4m3 values} per channel holding
        # an outlier, channels ascending; values 0 where the token is not one
        chans = np.nonzero(masks.any(0))[0]
        hdr = blk[12 * D:]
        n = len(chans)
        assert hdr[0] == n and hdr[1] == masks.sum()
        for i, c in enumerate(chans):
            rec = hdr[4 + 20 * i:24 + 20 * i]
            assert rec[0] == c and rec[1] == 0
            assert int(rec[2]) | (int(rec[3]) << 8) == sum(1 << t for t in range(16) if masks[t, c])
            for t in range(16):
                want = oracle.e4m3_encode(float(x[t, c])) if masks[t, c] else 0
                assert rec[4 + t] == want
        assert not hdr[4 + 20 * n:].any()
        # outliers reproduced exactly as e4m3
        for t, c in zip(*np.nonzero(masks)):
            assert xh[t, c] == oracle.e4m3_decode(oracle.e4m3_encode(float(x[t, c])))
        # non-outliers: the stored value is the nearest of the channel's 4 fp16 centroids
        for c in range(D):
            vals = x[~masks[:, c], c].astype(np.float64)
            cents, c16, _, _ = oracle.lloyd4(vals)
            cf = np.array([oracle.fp16_decode(h) for h in c16])
            for t in np.nonzero(~masks[:, c])[0]:
                assert abs(float(xh[t, c]) - float(x[t, c])) <= np.abs(cf - float(x[t, c])).min()
                assert xh[t, c] in cf


def test_cb2_outlier_rate_near_page_claim():
    """cb2_4k data (4 of 128 channels x8): about 2.2 outliers per token (1.7%),
    consistent with the 'under 1.8%' volume the first page reports."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4000, 128))
    x[:, [3, 40, 77, 120]] *= 8
    k = np.mean([oracle.outlier_mask(r)[1] for r in x])
    assert 1.9 < k < 2.5 and k / 128 < 0.02


# ------------------------------------------------------------------ layout
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("role", [R_K, R_V])
def test_fragment_positions_are_a_bijection(D, role):
    seen = set()
    for t in range(16):
        for c in range(D):
            lane, s, k = oracle.frag_pos(role, t, c)
            assert 0 <= lane < 32 and 0 <= k < 8 and s == c // 16
            seen.add((lane, s, k))
    assert len(seen) == 16 * D


@pytest.mark.parametrize("fmt", [oracle.BLK_INT4, oracle.BLK_E2M1, oracle.BLK_CB2, oracle.BLK_FP8])
def test_block_strides_aligned(fmt):
    for D in (64, 128):
        assert oracle.block_stride(fmt, D) % 128 == 0
    assert oracle.block_stride(oracle.BLK_CB2, 128) == 4224
    assert oracle.block_stride(oracle.BLK_E2M1, 128) == 1152


# ----------------------------------------------------------------------------- CB2 with a static fp16 channel mask
def test_select_static_matches_brute_force():
    """Top-n_s channels by max |x| over the calibration tokens, ties to the lower
    channel, ascending ("The Sub-10ms Barrier", Key Production Engineering
    Takeaways, item 2: top 1% channels by absolute magnitude stay in FP16)."""
    rng = np.random.default_rng(11)
    for trial in range(6):
        t, Hkv, D, n_s = int(rng.integers(1, 40)), 3, (64, 128)[trial % 2], int(rng.integers(1, 9))
        x = rng.standard_normal((t, Hkv, D)).astype(np.float32)
        if trial >= 3:   # ties: quantize magnitudes coarsely
            x = np.round(x * 2) / 2
        got = oracle.select_static(x, n_s)
        score = np.abs(x).max(0)                     # [Hkv, D]
        for h in range(Hkv):
            order = sorted(range(D), key=lambda c: (-score[h, c], c))
            assert list(got[h]) == sorted(order[:n_s])


def test_cb2_static_page_properties():
    rng = np.random.default_rng(12)
    for trial in range(6):
        D = (64, 128)[trial % 2]
        role = (trial // 2) % 2
        x = rng.standard_normal((16, D)).astype(np.float32)
        n_s = 1 + trial % 3
        ch = np.sort(rng.choice(D, n_s, replace=False))
        x[:, ch] *= 20
        x[3, (ch[0] + 1) % D] = 40.0      # a large value outside the mask gets no special treatment
        blk = oracle.quantize_page_static(D, x, ch, role=role)
        xh = oracle.dequantize_block(oracle.BLK_CB2S, D, blk, role=role)
        hdr = blk[12 * D:]
        assert hdr[0] == n_s and list(hdr[1:1 + n_s]) == list(ch) and not hdr[1 + n_s:16].any()
        for i, c in enumerate(ch):
            for t in range(16):
                h16 = int(hdr[16 + 32 * i + 2 * t]) | (int(hdr[17 + 32 * i + 2 * t]) << 8)
                assert h16 == oracle.fp16_encode(float(x[t, c]))
                assert xh[t, c] == oracle.fp16_decode(h16)
        assert not hdr[16 + 32 * n_s:].any()
        # the same codes and codebook as a CB2 page of the other channels, fitted over all 16 values
        for c in range(D):
            if c in ch:
                continue
            _, c16, codes, _ = oracle.lloyd4(x[:, c].astype(np.float64))
            cf = np.array([oracle.fp16_decode(h) for h in c16])
            for t in range(16):
                assert abs(float(xh[t, c]) - float(x[t, c])) <= np.abs(cf - float(x[t, c])).min()
                assert xh[t, c] in cf
        # static channels carry code 0 and an all-zero codebook in the 2-bit planes
        plain = blk.copy()
        plain[12 * D:] = 0
        plain[12 * D] = 0
        xz = oracle.dequantize_block(oracle.BLK_CB2, D, plain, role=role)
        assert (xz[:, ch] == 0).all()


def test_cb2_static_cache_round_trip():
    """Appends in ragged chunks give the same cache as one prefill (pages are
    quantized once complete, from fp32 staging); dequantize returns fp16 values
    on the static channels."""
    rng = np.random.default_rng(13)
    B, Hkv, D, P = 2, 2, 64, 4
    x = rng.standard_normal((2, B, 50, Hkv, D)).astype(np.float32)
    st = np.zeros((Hkv, 2, 2), np.uint8)
    st[:, :, 0], st[:, :, 1] = 3, 40
    x[..., 3] *= 15
    a = oracle.OracleCache(oracle.FMT_CB2S, B, Hkv, D, P, B * P, static_channels=st)
    b = oracle.OracleCache(oracle.FMT_CB2S, B, Hkv, D, P, B * P, static_channels=st)
    a.append(x[0], x[1])
    for t0, t1 in ((0, 7), (7, 16), (16, 33), (33, 50)):
        b.append(x[0][:, t0:t1], x[1][:, t0:t1])
    # staging rows past the partial page's 2 tokens are stale in the chunked cache and never read
    assert (a.pool == b.pool).all() and (a.staging[:, :, :, :2] == b.staging[:, :, :, :2]).all()
    for role in (0, 1):
        got = a.dequantize(1, 1, role, 0, 48)
        want = np.array([[oracle.fp16_decode(oracle.fp16_encode(float(v))) for v in row] for row in x[role][1, :48, 1][:, [3, 40]]])
        assert (got[:, [3, 40]] == want).all()


# ----------------------------------------------------------------------------- ASYM3 (3-bit asymmetric + outliers)
def _a3_code(blk, D, role, t, c):
    """3-bit code of (t, c), unpacked from the documented bit positions."""
    lane, s, k = oracle.frag_pos(role, t, c)
    NS = D // 16
    x = int.from_bytes(bytes(blk[4 * (lane * (NS // 2) + s // 2):][:4]), "little")
    y = int.from_bytes(bytes(blk[4 * D + 4 * (lane * (NS // 4) + s // 4):][:4]), "little")
    bx = 8 * (s % 2) + 16 * (k % 2) + 2 * (k // 2)
    by = 4 * (s % 4) + 16 * (k % 2) + k // 2
    return ((x >> bx) & 3) | (((y >> by) & 1) << 2)


def test_a3_page_matches_the_recipe():
    """Per channel over its non-outliers, in fp64: S = fp16((max-min)/7),
    m = fp16(min), q = clamp(rint((x-m)/S), 0, 7); outlier slots hold 0; the
    side-list is CB2's for the same page; a code stands for fp16(q*S + m)
    ("Sub-5ms MoE Inference", Sub-Byte KV-Cache Quantization: asymmetric 3-bit
    packing with dynamic outlier preservation)."""
    rng = np.random.default_rng(21)
    for trial in range(6):
        D = (64, 128)[trial % 2]
        role = (trial // 2) % 2
        x = rng.standard_normal((16, D)).astype(np.float32)
        x[:, rng.choice(D, 3, replace=False)] *= 8
        if trial == 5:
            x[:, 7] = 0.25          # a constant channel: S = 0, every code 0
        blk = oracle.quantize_page(oracle.BLK_A3, D, x, role=role)
        cb2 = oracle.quantize_page(oracle.BLK_CB2, D, x, role=role)
        assert (blk[10 * D:10 * D + 4 + 20 * D] == cb2[12 * D:12 * D + 4 + 20 * D]).all()
        masks = np.array([oracle.outlier_mask(x[t])[0] for t in range(16)])
        xh = oracle.dequantize_block(oracle.BLK_A3, D, blk, role=role)
        for c in range(D):
            keep = ~masks[:, c]
            vals = x[keep, c]
            S16 = oracle.fp16_encode(float(Fraction(float(vals.max())) - Fraction(float(vals.min()))) / 7) \
                if keep.any() else 0
            m16 = oracle.fp16_encode(float(vals.min())) if keep.any() else 0
            rho = (16 * (c // 16) + 4 * ((c % 8) // 2) + 2 * ((c % 16) // 8) + c % 2 if role == 0
                   else 16 * (c // 16) + 2 * (c % 8) + (c % 16) // 8)
            assert int(blk[6 * D + 2 * rho]) | (int(blk[6 * D + 2 * rho + 1]) << 8) == S16
            assert int(blk[8 * D + 2 * rho]) | (int(blk[8 * D + 2 * rho + 1]) << 8) == m16
            S, m = np.float32(oracle.fp16_decode(S16)), np.float32(oracle.fp16_decode(m16))
            for t in range(16):
                q = _a3_code(blk, D, role, t, c)
                if masks[t, c] or S == 0:
                    assert q == 0
                else:
                    r = (Fraction(float(x[t, c])) - Fraction(float(m))) / Fraction(float(S))
                    assert q == max(0, min(7, round(r)))
                want = oracle.fp16_decode(oracle.fp16_encode(q * float(S) + float(m)))
                if masks[t, c]:
                    want = oracle.e4m3_decode(oracle.e4m3_encode(float(x[t, c])))
                assert xh[t, c] == np.float32(want)
                if not masks[t, c]:   # half a step plus the fp16 rounding of the level
                    assert abs(float(xh[t, c]) - float(x[t, c])) <= float(S) / 2 + abs(want) * 2.0 ** -11 + 1e-7


def test_a3_cache_chunking_independent():
    rng = np.random.default_rng(22)
    B, Hkv, D, P = 2, 2, 128, 4
    x = rng.standard_normal((2, B, 50, Hkv, D)).astype(np.float32)
    x[..., 9] *= 10
    a = oracle.OracleCache(oracle.FMT_A3, B, Hkv, D, P, B * P)
    b = oracle.OracleCache(oracle.FMT_A3, B, Hkv, D, P, B * P)
    a.append(x[0], x[1])
    for t0, t1 in ((0, 5), (5, 16), (16, 40), (40, 50)):
        b.append(x[0][:, t0:t1], x[1][:, t0:t1])
    assert (a.pool == b.pool).all() and (a.staging[:, :, :, :2] == b.staging[:, :, :, :2]).all()
    assert (a.dequantize(0, 1, 1, 0, 50) == b.dequantize(0, 1, 1, 0, 50)).all()


# ----------------------------------------------------------------------------- CB2 with a codebook per group of 4 pages
def test_cb2_group_matches_the_recipe():
    """One codebook per (group of 4 pages, channel), fitted like CB2's over the
    non-outliers of all 64 tokens ("Hierarchical Token Routing and Sub-2-Bit
    Non-Linear KV Compression", 2. Centroid Vector Quantization for Residuals:
    k-means per head-group block).  It lives in the group's first page; every
    page's side-list is the CB2 side-list of its own 16 tokens."""
    rng = np.random.default_rng(31)
    for trial in range(4):
        D = (64, 128)[trial % 2]
        role = trial // 2
        x = rng.standard_normal((64, D)).astype(np.float32)
        x[:, rng.choice(D, 4, replace=False)] *= 8
        blks = oracle.quantize_group(D, x, role=role)
        masks = np.array([oracle.outlier_mask(x[t])[0] for t in range(64)])
        assert not blks[1:, :8 * D].any()
        for p in range(4):
            page = oracle.quantize_page(oracle.BLK_CB2, D, x[16 * p:16 * p + 16], role=role)
            assert (blks[p, 12 * D:] == page[12 * D:]).all()
        xh = np.concatenate([oracle.dequantize_group_page(D, blks[p], blks[0], role=role) for p in range(4)])
        for c in range(D):
            keep = ~masks[:, c]
            _, c16, _, _ = oracle.lloyd4(x[keep, c].astype(np.float64))
            cf = np.array([oracle.fp16_decode(h) for h in c16])
            for t in range(64):
                if masks[t, c]:
                    assert xh[t, c] == oracle.e4m3_decode(oracle.e4m3_encode(float(x[t, c])))
                else:
                    assert xh[t, c] in cf
                    assert abs(float(xh[t, c]) - float(x[t, c])) <= np.abs(cf - float(x[t, c])).min()


def test_cb2_group_cache_chunking_and_staging():
    """A group is quantized when its 64th token arrives, from fp32 staging;
    before that dequantize returns the staged values exactly."""
    rng = np.random.default_rng(32)
    B, Hkv, D, P = 2, 2, 64, 12
    x = rng.standard_normal((2, B, 150, Hkv, D)).astype(np.float32)
    x[..., 5] *= 8
    a = oracle.OracleCache(oracle.FMT_CB2G, B, Hkv, D, P, B * P)
    b = oracle.OracleCache(oracle.FMT_CB2G, B, Hkv, D, P, B * P)
    a.append(x[0], x[1])
    for t0, t1 in ((0, 30), (30, 64), (64, 65), (65, 140), (140, 150)):
        b.append(x[0][:, t0:t1], x[1][:, t0:t1])
    assert (a.pool == b.pool).all()
    assert (a.staging[:, :, :, :150 - 128] == b.staging[:, :, :, :150 - 128]).all()
    for role in (0, 1):
        got = a.dequantize(1, 0, role, 0, 150)
        assert (got[128:] == x[role][1, 128:150, 0]).all()          # the partial group, from staging
        blk = a.pool.reshape(-1, a.stride)
        pt = a.page_table.view(np.uint32)
        cb = blk[(pt[1, 4] * Hkv + 0) * 2 + role]
        for p in range(4, 8):                                        # the second group, from blocks
            page = blk[(pt[1, p] * Hkv + 0) * 2 + role]
            assert (got[16 * p:16 * p + 16] == oracle.dequantize_group_page(D, page, cb, role=role)).all()
