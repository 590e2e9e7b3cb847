"""Pins for the oracle's scalar number formats, against library routines and
the format definitions (not against the oracle itself).

fp16  : numpy.float16 (IEEE binary16, round-to-nearest-even)
e4m3  : torch.float8_e4m3fn casting (the dtype the compress_kv_head listing of
        "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression"
        stores its outliers in)
e2m1  : the bit layout "The Sub-10ms Barrier: Fusing Sparse MoE Routing with
        FP4 KV-Cache Quantization" gives (1 sign, 2 exponent, 1 mantissa bit)
bf16  : torch.bfloat16
"""
import numpy as np
import pytest
import torch

import oracle


def _sweep(n=20000, seed=0):
    rng = np.random.default_rng(seed)
    mags = np.exp(rng.uniform(np.log(1e-9), np.log(1e6), n))
    vals = mags * rng.choice([-1.0, 1.0], n)
    return vals


def test_fp16_encode_matches_numpy():
    vals = list(_sweep())
    # exact ties between neighbouring fp16 values, subnormals, overflow edge
    for h in range(0, 0x7C00, 97):
        a = float(np.array(h, np.uint16).view(np.float16))
        b = float(np.array(h + 1, np.uint16).view(np.float16))
        vals += [(a + b) / 2, -(a + b) / 2, a]
    vals += [65504.0, 65519.99, 65520.0, 1e5, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 0.0, -0.0]
    for v in vals:
        want = int(np.array(v, np.float64).astype(np.float16).view(np.uint16))
        assert oracle.fp16_encode(v) == want, (v, hex(want))


def test_fp16_decode_all_finite_codes():
    for h in range(0, 0x10000, 7):
        f = np.array(h, np.uint16).view(np.float16)
        if not np.isfinite(f):
            continue
        assert oracle.fp16_decode(h) == float(f)


def test_e4m3_encode_matches_torch_cast():
    vals = np.concatenate([_sweep(seed=1), _sweep(seed=2) * 1e-3])
    vals = vals[np.abs(vals) <= 464.0].astype(np.float32)   # torch yields NaN past the last tie
    codes = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, c in zip(vals, codes):
        assert oracle.e4m3_encode(float(v)) == int(c), (v, c)


def test_e4m3_ties_and_saturation():
    # every midpoint between adjacent codes rounds to the even mantissa, as torch does
    mids = []
    for c in range(0, 0x7E):
        a, b = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mids.append((a + b) / 2)
    t = torch.tensor(mids, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    assert [oracle.e4m3_encode(m) for m in mids] == t
    # satfinite reading: beyond 448 clamps instead of producing NaN
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-1e9) == 0xFE


def test_e4m3_roundtrip_all_codes():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        v = oracle.e4m3_decode(c)
        assert oracle.e4m3_encode(v) == c
        assert v == float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])


def test_e2m1_table_from_definition():
    # value = (-1)^s * 2^(e-1) * (1 + m/2) for e > 0, (-1)^s * m/2 for e == 0
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = 2.0 ** (e - 1) * (1 + m / 2) if e else m / 2
        assert oracle.e2m1_decode(code) == (-mag if s else mag)
    assert sorted({abs(oracle.e2m1_decode(c)) for c in range(16)}) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


@pytest.mark.parametrize("x,expect", [
    (0.25, 0.0), (0.26, 0.5), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
    (5.0, 4.0), (5.01, 6.0), (6.0, 6.0), (100.0, 6.0), (-0.75, -1.0), (-5.0, -4.0), (0.7, 0.5),
])
def test_e2m1_round_to_nearest_even(x, expect):
    # ties go to the code with an even mantissa bit; saturate at 6
    assert oracle.e2m1_decode(oracle.e2m1_encode(x)) == expect


def test_e2m1_nearest_property():
    grid = np.array(sorted({oracle.e2m1_decode(c) for c in range(16)}))
    for v in np.linspace(-7, 7, 2801):
        got = oracle.e2m1_decode(oracle.e2m1_encode(v))
        d = np.abs(grid - np.clip(v, -6, 6))
        assert abs(got - np.clip(v, -6, 6)) == d.min()


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 0x10000, 13, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    for b, f in zip(bits, t):
        if np.isfinite(f):
            assert oracle.bf16_decode(int(b)) == float(f)
