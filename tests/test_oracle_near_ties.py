"""The oracle's quantizer decisions are fp64 decisions: pinned against exact
rational arithmetic on inputs placed within one binary32 rounding of each
decision boundary (tests/_near_ties.py), where binary32 arithmetic goes to the
wrong side in a good share of the cases.

Each test except the E2M1 one also counts how often a binary32 evaluation
of the same rule disagrees with the exact decision on the same inputs: that
count must be positive, so a quantizer computed in binary32 could not pass
the test.  (E2M1 divides by an e4m3 scale, a divisor of four significant
bits, and on these inputs the binary32 quotient never lands on the wrong
side; the test pins exactness only.)

Sources: "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression",
1. Dynamic Outlier Isolation (the 3-sigma rule over a head vector) and
2. Centroid Vector Quantization for Residuals (the 4-centroid fit); "The
Sub-10ms Barrier", 2. FP4/INT4 KV-Cache Quantization (S = (max - min) /
(2^b - 1), E2M1 with a scale per block); "Hierarchical Token Gating and Tiered
KV-Cache Paging", 2. Entropy-Guided Tiered KV-Cache Quantization (FP8 pages).
"""
from fractions import Fraction

import numpy as np

import _near_ties as nt
import oracle

F32 = np.float32


def _f32_outliers(x):
    """The same rule in binary32 with sequential sums (what the test must catch)."""
    n = len(x)
    s = F32(0)
    for v in x:
        s = F32(s + v)
    mu = F32(s / F32(n))
    ss = F32(0)
    for v in x:
        d = F32(v - mu)
        ss = F32(ss + F32(d * d))
    thr = F32(3) * F32(np.sqrt(F32(ss / F32(n - 1))))
    return np.abs((x - mu).astype(F32)) > thr


def test_outlier_decisions_are_exact_on_the_threshold():
    rng = np.random.default_rng(40)
    wrong32 = 0
    for t in range(240):
        n = (32, 64, 128)[t % 3]
        x = nt.outlier_tie_vector(rng, n, int(rng.integers(0, n)), t % 3, scale=float(rng.uniform(0.1, 20)),
                                  big=(1, 9, 40) if n == 128 else (), side=1 if t % 2 else -1)
        exact = nt.exact_outliers(x)
        mask, _ = oracle.outlier_mask(x, 3.0, cap=n)
        assert (mask == exact).all(), t
        wrong32 += (_f32_outliers(x) != exact).any()
    assert wrong32 > 10


def test_outlier_decisions_exact_on_random_vectors():
    """No skip band: random vectors (margins far above fp64 rounding) agree exactly."""
    rng = np.random.default_rng(41)
    for trial in range(200):
        n = (32, 64, 128)[trial % 3]
        x = rng.standard_normal(n).astype(F32)
        x[rng.integers(0, n, 3)] *= F32(rng.uniform(2, 12))
        mask, _ = oracle.outlier_mask(x, 3.0, cap=n)
        assert (mask == nt.exact_outliers(x)).all()


def _int4_codes(blk, D, role, t):
    codes = np.zeros(D, int)
    for c in range(D):
        lane, s, k = oracle.frag_pos(role, t, c)
        byte = blk[4 * (D // 16) * lane + 4 * s + k // 2]
        codes[c] = (byte >> (4 * (k % 2))) & 0xF
    return codes


def test_int4_scales_and_codes_are_exact_on_midpoints():
    rng = np.random.default_rng(42)
    D = 64
    wrong32 = 0
    for trial in range(60):
        x = np.concatenate([nt.affine_tie_values(rng, 32, 15, 12, s_tie=(trial + g) % 2 == 0) for g in range(2)])
        role, t = trial % 2, int(rng.integers(0, 16))
        blk = np.zeros(oracle.block_stride(oracle.BLK_INT4, D), np.uint8)
        oracle.quantize_token(oracle.BLK_INT4, D, x, t, blk, role=role)
        codes = _int4_codes(blk, D, role, t)
        assert blk[10 * D + t] == 0                              # no outliers in these groups
        for g in range(2):
            seg = x[32 * g:32 * g + 32]
            S, m = nt.affine_scale(seg.min(), seg.max(), 15)
            sz = blk[8 * D + 4 * (t * 2 + g):][:4]
            assert int(sz[0]) | (int(sz[1]) << 8) == int(np.float16(S).view(np.uint16))
            assert int(sz[2]) | (int(sz[3]) << 8) == int(np.float16(m).view(np.uint16))
            S32 = np.float16(F32(F32(seg.max() - seg.min()) / F32(15))).astype(np.float64)
            wrong32 += S32 != S
            for i in range(32):
                q = nt.exact_affine_code(seg[i], m, S, 15)
                assert codes[32 * g + i] == q
                q32 = int(np.clip(np.rint(F32(F32(seg[i] - F32(m)) / F32(S))), 0, 15))
                wrong32 += q32 != q
    assert wrong32 > 10


def test_asym3_scales_and_codes_are_exact_on_midpoints():
    rng = np.random.default_rng(43)
    D = 64
    wrong32 = 0
    for trial in range(8):
        role = trial % 2
        x = np.stack([nt.affine_tie_values(rng, 16, 7, 6, s_tie=(trial + c) % 3 == 0) for c in range(D)], 1)
        blk = oracle.quantize_page(oracle.BLK_A3, D, x, role=role)
        assert blk[10 * D] == 0                                  # no outliers
        xh = oracle.dequantize_block(oracle.BLK_A3, D, blk, role=role)
        for c in range(D):
            S, m = nt.affine_scale(x[:, c].min(), x[:, c].max(), 7)
            for t in range(16):
                q = nt.exact_affine_code(x[t, c], m, S, 7)
                want = float(np.float16(q * S + m))             # fp16(q S + m), one rounding
                assert xh[t, c] == F32(want), (trial, t, c)
                q32 = int(np.clip(np.rint(F32(F32(x[t, c] - F32(m)) / F32(S))), 0, 7))
                wrong32 += q32 != q
    assert wrong32 > 10


def test_e2m1_scales_and_codes_are_exact_on_midpoints():
    rng = np.random.default_rng(44)
    D = 128
    for trial in range(30):
        x = np.concatenate([nt.e2m1_tie_block(rng, scale_tie=(trial + s) % 2 == 0) for s in range(D // 16)])
        blk = np.zeros(oracle.block_stride(oracle.BLK_E2M1, D), np.uint8)
        oracle.quantize_token(oracle.BLK_E2M1, D, x, 5, blk, role=trial % 2)
        xh = oracle.dequantize_block(oracle.BLK_E2M1, D, blk, role=trial % 2)[5]
        for s in range(D // 16):
            seg = x[16 * s:16 * s + 16]
            amax = np.abs(seg).max()
            sc = nt.e4m3_rne(Fraction(float(amax)) / 6)
            for i in range(16):
                r = abs(Fraction(float(seg[i]))) / Fraction(sc)
                k = min(range(8), key=lambda j: (abs(Fraction(nt.E2M1[j]) - r), j % 2))   # nearest, ties to even
                want = (-1 if seg[i] < 0 else 1) * nt.E2M1[k] * sc
                assert xh[16 * s + i] == F32(want), (trial, s, i)


def test_fp8_page_codes_are_exact_on_midpoints():
    rng = np.random.default_rng(45)
    D = 128
    wrong32 = 0
    for trial in range(4):
        x = nt.fp8_tie_page(rng, D)
        blk = oracle.quantize_page(oracle.BLK_FP8, D, x, role=trial % 2)
        xh = oracle.dequantize_block(oracle.BLK_FP8, D, blk, role=trial % 2)
        s = F32(float(np.abs(x).max()) / 448.0)              # the stored scale: fp32 of the fp64 quotient
        for t in range(16):
            for c in range(D):
                mag = nt.e4m3_rne(abs(Fraction(float(x[t, c]))) / Fraction(float(s)))
                want = F32((-1 if x[t, c] < 0 else 1) * mag) * s
                assert xh[t, c] == want, (trial, t, c)
                mag32 = nt.e4m3_rne(abs(Fraction(float(F32(x[t, c] / s)))))
                wrong32 += mag32 != mag
    assert wrong32 > 10


def test_lloyd_centroids_round_from_their_exact_means():
    """Four tight clusters whose means lie a quarter binary32 step off an fp16
    midpoint: the fit converges to the cluster means and stores each rounded
    once from its exact value (a binary32 mean lands on the midpoint and
    rounds to the even neighbour instead)."""
    rng = np.random.default_rng(46)
    wrong32 = 0
    for trial in range(60):
        v, means = nt.lloyd_tie_channel(rng)
        _, c16, codes, _ = oracle.lloyd4(v)
        for j in range(4):
            assert int(c16[j]) == int(np.float16(float(means[j])).view(np.uint16)), (trial, j)
        # binary32 means (members in order) round differently on some channel
        for j in range(4):
            cl = [F32(x) for x in v if abs(float(x) - float(means[j])) < 0.5]
            s = F32(0)
            for x in cl:
                s = F32(s + x)
            wrong32 += np.float16(F32(s / F32(len(cl)))) != np.float16(float(means[j]))
        # final codes: the nearest stored centroid
        cf = np.array([oracle.fp16_decode(int(h)) for h in c16])
        assert (codes == np.array([int(np.argmin(np.abs(float(x) - cf))) for x in v])).all()
    assert wrong32 > 10


def test_lloyd_centroids_equal_the_rounded_exact_means():
    """At convergence each non-empty cell's fp64 centroid is its members' exact
    mean rounded once to fp64 (the sums of these binary32 values are exact in
    fp64), and each stored centroid is that value rounded to fp16."""
    rng = np.random.default_rng(47)
    for trial in range(150):
        n = int(rng.integers(2, 17))
        v = (rng.standard_normal(n) * rng.uniform(0.01, 30)).astype(F32)
        c, c16, codes, passes = oracle.lloyd4(v, iters=64)
        assert passes < 64
        cf = np.array([oracle.fp16_decode(int(h)) for h in c16])
        assign = [int(np.argmin(np.abs(float(x) - c))) for x in v]
        for j in range(4):
            mem = [Fraction(float(x)) for x, a in zip(v, assign) if a == j]
            if mem:
                assert c[j] == float(sum(mem) / len(mem))
            assert c16[j] == np.float16(c[j]).view(np.uint16)
        # final codes by exact comparison, the lower index on ties
        for x, q in zip(v, codes):
            d = [abs(Fraction(float(x)) - Fraction(float(cj))) for cj in cf]
            assert q == min(range(4), key=lambda j: (d[j], j))
