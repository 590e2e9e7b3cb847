"""Pins for the oracle's attention, paged cache and byte accounting.

Attention ("Hardware-Kernel Fusion" of "Hierarchical Token Routing and
Sub-2-Bit Non-Linear KV Compression"; the flash-decoding phase of "The
Sub-10ms Barrier"): checked against scipy's softmax with numpy matmuls on tiny
shapes, and against the special cases that have closed forms.

Byte accounting: "Total KV Cache Size per Token = 2 x L x H x D x Precision"
("The Bottleneck: Why Standard MoE Inference Stalls" on the first page) and the
75% traffic cut from FP16 to 4-bit ("2. FP4/INT4 KV-Cache Quantization" on the
fourth page).
"""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from sub_byte_quantized_kvq_gb300 import synth


def _rand_attn(rng, G, N, D):
    q = rng.standard_normal((G, D))
    k = rng.standard_normal((N, D)).astype(np.float32)
    v = rng.standard_normal((N, D)).astype(np.float32)
    return q, k, v


@pytest.mark.parametrize("G,N,D", [(1, 1, 8), (4, 7, 16), (8, 33, 64), (2, 100, 128)])
def test_attention_matches_scipy(G, N, D):
    rng = np.random.default_rng(G * 1000 + N)
    q, k, v = _rand_attn(rng, G, N, D)
    scale = 1 / np.sqrt(D)
    p = scipy.special.softmax(scale * (q @ k.astype(np.float64).T), axis=-1)
    ref = p @ v.astype(np.float64)
    got = oracle.attention(q, k, v, scale)
    assert np.abs(got - ref).max() < 1e-12
    assert np.abs(p.sum(-1) - 1).max() < 1e-12


def test_attention_closed_forms():
    rng = np.random.default_rng(9)
    G, N, D = 4, 50, 32
    q, k, v = _rand_attn(rng, G, N, D)
    # constant V rows -> that constant
    vc = np.tile(rng.standard_normal(D).astype(np.float32), (N, 1))
    assert np.abs(oracle.attention(q, k, vc, 0.3) - vc[0]).max() < 1e-12
    # Q = 0 -> uniform weights -> mean of V
    assert np.abs(oracle.attention(np.zeros((G, D)), k, v, 0.3) - v.astype(np.float64).mean(0)).max() < 1e-12
    # a single token -> that token's V
    assert np.abs(oracle.attention(q, k[:1], v[:1], 0.3) - v[0]).max() == 0
    # empty context -> zeros (the library's convention)
    assert (oracle.attention(q, k[:0], v[:0], 0.3) == 0).all()
    # huge logits do not overflow (max subtracted): one dominant token
    k2 = k.copy()
    k2[17] = 1000 * q[0] / np.linalg.norm(q[0])
    out = oracle.attention(q[:1], k2, v, 1.0)
    assert np.abs(out[0] - v[17]).max() < 1e-12


# ------------------------------------------------------------------ paged cache
def _small_kv(seed, B, T, Hkv, D, factor=6.0):
    w = synth.Workload("t", 0, B, Hkv, Hkv, D, T, "normal", 2, factor)
    ks, vs = [], []
    for b in range(B):
        k, v = synth.workload_kv(w, seed, b, 0, T)
        ks.append(k.numpy())
        vs.append(v.numpy())
    return np.stack(ks), np.stack(vs)


@pytest.mark.parametrize("fmt", [oracle.FMT_INT4, oracle.FMT_E2M1, oracle.FMT_CB2, oracle.FMT_TIERED])
def test_append_chunking_invariance(fmt):
    """The cache a sequence ends up with does not depend on how its tokens
    were split into append calls (prefill vs token-by-token vs ragged)."""
    B, Hkv, D, T, P = 2, 2, 64, 53, 4
    k, v = _small_kv(1, B, T, Hkv, D)
    tiers = np.zeros((B, P), bool)
    if fmt == oracle.FMT_TIERED:
        tiers[:, 1] = True
    pt, nm, nt = synth.page_table(3, B, P, True, tiers)

    def mk():
        return oracle.OracleCache(fmt, B, Hkv, D, P, nm, nt, page_table=pt)
    a = mk()
    assert a.append(k, v) == 0
    b = mk()
    for t in range(T):
        assert b.append(k[:, t:t + 1], v[:, t:t + 1]) == 0
    c = mk()
    pos = 0
    for step in [5, 16, 1, 20, 11]:
        assert c.append(k[:, pos:pos + step], v[:, pos:pos + step]) == 0
        pos += step
    for x in (b, c):
        assert (x.pool == a.pool).all() and (x.tier_pool == a.tier_pool).all()
        assert (x.seq_lens == a.seq_lens).all()
        full = (T // 16) * 16
        assert (x.staging[..., :T - full, :] == a.staging[..., :T - full, :]).all()


def test_ragged_append_and_capacity():
    B, Hkv, D, P = 3, 1, 64, 2
    k, v = _small_kv(2, B, 20, Hkv, D)
    pt, nm, _ = synth.page_table(0, B, P, False)
    c = oracle.OracleCache(oracle.FMT_CB2, B, Hkv, D, P, nm, page_table=pt)
    assert c.append(k, v, t_per_seq=np.array([20, 0, 7])) == 0
    assert list(c.seq_lens) == [20, 0, 7]
    # 20 + 20 > 32 slots: sequence 0 overflows and is skipped, the others proceed
    assert c.append(k, v, t_per_seq=np.array([20, 3, 1])) == 1
    assert list(c.seq_lens) == [20, 3, 8]


def test_dequantized_cache_round_trip_and_placement_invariance():
    """Attention over the paged cache equals plain attention over the
    dequantized values, and does not depend on where pages live."""
    B, Hkv, G, D, T = 2, 2, 4, 64, 70
    P = 5
    k, v = _small_kv(4, B, T, Hkv, D)
    q = synth.queries_bf16(0, B, Hkv * G, D).view(torch.int16).numpy().view(np.uint16)
    outs = []
    for shuffled in (False, True):
        pt, nm, _ = synth.page_table(11, B, P, shuffled)
        c = oracle.OracleCache(oracle.FMT_CB2, B, Hkv, D, P, nm, page_table=pt)
        c.append(k, v)
        out = c.decode(q, 0.125)
        for b in range(B):
            for h in range(Hkv):
                kd, vd = c.dequantize(b, h, 0, 0, T), c.dequantize(b, h, 1, 0, T)
                qd = np.array([[oracle.bf16_decode(x) for x in row] for row in q[b, h * G:(h + 1) * G]])
                assert np.abs(out[b, h * G:(h + 1) * G] - oracle.attention(qd, kd, vd, 0.125)).max() == 0
                # the staged tail (last T % 16 tokens) is kept exactly
                assert (kd[64:] == k[b, 64:, h]).all()
        outs.append(out)
    assert (outs[0] == outs[1]).all()


# ------------------------------------------------------------------ byte accounting
def test_kv_bytes_per_token_formula_and_page_claims():
    # 2 x L x H x D x bytes; the first page's 80-layer GQA model, batch 64, 32k
    # context in FP16 needs "over 180 GB" (H and D are not given; 8 x 128 is the
    # common GQA shape and gives 687 GB)
    per_tok = 2 * 80 * 8 * 128 * 2
    assert per_tok * 64 * 32768 / 1e9 > 180
    # FP16 -> 4-bit codes: the code plane is 25% of FP16 ("reduces memory traffic by 75%")
    D = 128
    fp16_bytes = 16 * D * 2
    assert 16 * D // 2 == fp16_bytes // 4
    # with metadata: INT4 g32 with fp16 S and m is 4 + 32/32 = 5 bits per value,
    # E2M1 with one e4m3 scale per 16 values is 4 + 8/16 = 4.5 bits
    assert (16 * D // 2 + 16 * (D // 32) * 4) * 8 / (16 * D) == 5.0
    assert (16 * D // 2 + 16 * (D // 16)) * 8 / (16 * D) == 4.5
