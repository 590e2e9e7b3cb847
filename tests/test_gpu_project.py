"""K/V projection fused with quantize-on-append (kvq_project_append): the
projected values it hands back agree with the oracle's fp64 projection within
the fp32-accumulation bound, and the cache it writes is bit-identical to the
oracle appending those same values -- every format, both head dims, ragged
appends that span several 128-row tiles, a staged tail from an earlier
append, and an append that starts mid-group."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_quantized_kvq_gb300 import kvq, synth

from _kvq_pairs import ORACLE_FMT, Pair, make_kv

pytestmark = pytest.mark.gpu

FORMATS = [kvq.KVQ_FMT_INT4_G32, kvq.KVQ_FMT_FP4_E2M1_S16, kvq.KVQ_FMT_CB2_OUTLIER, kvq.KVQ_FMT_TIERED,
           kvq.KVQ_FMT_CB2_STATIC, kvq.KVQ_FMT_ASYM3_OUTLIER, kvq.KVQ_FMT_CB2_GROUP4]


def assert_projection_close(got, x, w, which, Hkv, D, t_per_seq):
    """|got - exact| <= hidden * 2^-23 * sum_e |x_e w_e|: bf16 products are exact in
    fp32, so the only error is the fp32 accumulation over `hidden` terms."""
    xf, wf = x.float().numpy().astype(np.float64), w.float().numpy().astype(np.float64)
    exact = oracle.project_kv(xf, wf, wf, Hkv, D)[0]
    mag = np.matmul(np.abs(xf), np.abs(wf).T).reshape(exact.shape)
    bound = x.shape[2] * 2.0 ** -23 * mag + 1e-30
    for b in range(x.shape[0]):
        n = x.shape[1] if t_per_seq is None else t_per_seq[b]
        err = np.abs(got[b, :n] - exact[b, :n])
        assert (err <= bound[b, :n]).all(), f"{which} seq {b}: max err {err.max():.3e}"
        assert (got[b, n:] == 0).all(), f"{which} seq {b}: rows past the append were written"


def tiers_for(fmt, B, P):
    if fmt != kvq.KVQ_FMT_TIERED:
        return None
    t = np.zeros((B, P), bool)
    t[:, 1::3] = True
    return t


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("fmt", FORMATS)
def test_project_append_matches_oracle(fmt, D):
    B, Hkv, P, hidden = 2, 2, 24, 256
    pair = Pair(fmt, B, Hkv, D, P, seed=3, tiers=tiers_for(fmt, B, P))
    x, wk, wv = synth.projection_inputs(3, B, 200, hidden, Hkv, D)
    # a ragged first append, then one that spans two tiles (more than 8 pages / 2 groups)
    for sl, tps in [(slice(0, 37), [37, 21]), (slice(37, 200), [163, 150])]:
        xs = x[:, sl].contiguous()
        k, v = pair.project(xs, wk, wv, tps)
        assert_projection_close(k, xs, wk, "K", Hkv, D, tps)
        assert_projection_close(v, xs, wv, "V", Hkv, D, tps)
        pair.assert_cache_equal()


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_CB2_OUTLIER, kvq.KVQ_FMT_CB2_GROUP4, kvq.KVQ_FMT_INT4_G32])
def test_project_after_plain_append_uses_the_staged_tail(fmt):
    B, Hkv, D, P, hidden = 2, 2, 128, 16, 128
    pair = Pair(fmt, B, Hkv, D, P, seed=4)
    k0, v0 = synth.kv_tokens(4, 0, 0, 27, Hkv, D, "normal", np.zeros((2, Hkv, 0), np.int64), 1.0)
    pair.append(torch.stack([k0, k0 * 0.5]), torch.stack([v0, v0 * 0.5]), t_per_seq=[27, 9])
    pair.assert_cache_equal()
    x, wk, wv = synth.projection_inputs(4, B, 120, hidden, Hkv, D)
    pair.project(x, wk, wv, [120, 101])
    pair.assert_cache_equal()
    # and a plain append after the projected one
    k1, v1 = synth.kv_tokens(5, 0, 0, 30, Hkv, D, "normal", np.zeros((2, Hkv, 0), np.int64), 1.0)
    pair.append(torch.stack([k1, k1]), torch.stack([v1, v1]), t_per_seq=[30, 11])
    pair.assert_cache_equal()


def test_project_single_token_decode_appends():
    B, Hkv, D, P, hidden = 3, 2, 128, 4, 64
    pair = Pair(kvq.KVQ_FMT_CB2_OUTLIER, B, Hkv, D, P, seed=6)
    x, wk, wv = synth.projection_inputs(6, B, 40, hidden, Hkv, D)
    for t in range(40):
        pair.project(x[:, t:t + 1].contiguous(), wk, wv, [1, 1 if t % 3 else 0, 1])
    pair.assert_cache_equal()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("fmt", FORMATS)
def test_project_one_token_appends_every_format(fmt, D):
    """One-token appends (the decode-time shape: one row per sequence, a
    cluster of CTAs splitting the hidden dimension): 19 sequences (one
    32-row cluster, three of its four row tiles used), positions ragged so
    that pages and the first 64-token group complete on different steps,
    sequences that skip a step, hidden 4096 (16 slices of 256 columns)."""
    B, Hkv, P, hidden = 19, 2, 5, 4096
    pair = Pair(fmt, B, Hkv, D, P, seed=13, tiers=tiers_for(fmt, B, P))
    k0, v0 = make_kv(13, B, 62, Hkv, D)
    pair.append(k0, v0, t_per_seq=[57 + b % 6 for b in range(B)])
    pair.assert_cache_equal()
    x, wk, wv = synth.projection_inputs(13, B, 9, hidden, Hkv, D)
    for t in range(9):
        tps = [0 if (b + t) % 5 == 0 else 1 for b in range(B)]
        xt = x[:, t:t + 1].contiguous()
        k, v = pair.project(xt, wk, wv, tps)
        assert_projection_close(k, xt, wk, "K", Hkv, D, tps)
        assert_projection_close(v, xt, wv, "V", Hkv, D, tps)
    pair.assert_cache_equal()


@pytest.mark.parametrize("hidden", [32, 96, 992, 8192, 32768])
def test_project_one_token_cluster_sizes(hidden):
    """hidden 32 / 96 (one CTA: a 32-column step past the 64-column stages),
    992 (one CTA: fifteen stages and a 32-column step), 8192 (16 CTAs of 512
    columns), 32768 (too wide for a cluster's slices: the tile kernel)."""
    B, Hkv, D, P = 9, 2, 128, 2
    pair = Pair(kvq.KVQ_FMT_CB2_OUTLIER, B, Hkv, D, P, seed=15)
    x, wk, wv = synth.projection_inputs(15, B, 17, hidden, Hkv, D)
    for t in range(17):
        xt = x[:, t:t + 1].contiguous()
        k, v = pair.project(xt, wk, wv)
        assert_projection_close(k, xt, wk, "K", Hkv, D, None)
        assert_projection_close(v, xt, wv, "V", Hkv, D, None)
    pair.assert_cache_equal()


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_INT4_G32, kvq.KVQ_FMT_TIERED])
def test_project_one_token_many_sequences(fmt):
    """40 sequences: clusters of 32 rows (a full one and one holding 8)."""
    B, Hkv, D, P, hidden = 40, 2, 128, 2, 1024
    pair = Pair(fmt, B, Hkv, D, P, seed=16, tiers=tiers_for(fmt, B, P))
    x, wk, wv = synth.projection_inputs(16, B, 17, hidden, Hkv, D)
    for t in range(17):
        tps = [0 if (b * 7 + t) % 9 == 0 else 1 for b in range(B)]
        xt = x[:, t:t + 1].contiguous()
        k, v = pair.project(xt, wk, wv, tps)
        assert_projection_close(k, xt, wk, "K", Hkv, D, tps)
        assert_projection_close(v, xt, wv, "V", Hkv, D, tps)
    pair.assert_cache_equal()


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_FP4_E2M1_S16, kvq.KVQ_FMT_CB2_OUTLIER])
def test_project_one_token_full_size(fmt):
    """The decode shapes' per-step append: 16 sequences, 8 kv heads, head_dim
    128, hidden 8192 (E2M1) or 4096 (CB2), 17 steps so that every sequence
    completes a page on the 16th."""
    B, Hkv, D, P = 16, 8, 128, 2
    hidden = 8192 if fmt == kvq.KVQ_FMT_FP4_E2M1_S16 else 4096
    pair = Pair(fmt, B, Hkv, D, P, seed=14)
    x, wk, wv = synth.projection_inputs(14, B, 17, hidden, Hkv, D)
    for t in range(17):
        xt = x[:, t:t + 1].contiguous()
        k, v = pair.project(xt, wk, wv)
        if t in (0, 15, 16):
            assert_projection_close(k, xt, wk, "K", Hkv, D, None)
            assert_projection_close(v, xt, wv, "V", Hkv, D, None)
    pair.assert_cache_equal()


def test_project_rejects_bad_arguments():
    pair = Pair(kvq.KVQ_FMT_INT4_G32, 1, 1, 64, 4, seed=0)
    x, wk, wv = synth.projection_inputs(0, 1, 4, 64, 1, 64)
    L = kvq.lib()
    import ctypes
    c, cc = ctypes.byref(pair.gpu.cfg), ctypes.byref(pair.gpu.c)
    xp, kp, vp = x.cuda(), wk.cuda(), wv.cuda()
    assert L.kvq_project_append(c, cc, xp.data_ptr(), 48, kp.data_ptr(), vp.data_ptr(), 4, None, None, None) == \
        kvq.KVQ_ERR_INVALID_ARG   # hidden not a multiple of 32
    assert L.kvq_project_append(c, cc, xp.data_ptr() + 2, 64, kp.data_ptr(), vp.data_ptr(), 4, None, None, None) == \
        kvq.KVQ_ERR_INVALID_ARG   # misaligned x
    assert L.kvq_project_append(c, cc, xp.data_ptr(), 64, kp.data_ptr(), vp.data_ptr(), 4 * 16 + 1, None, None,
                                None) == kvq.KVQ_ERR_CAPACITY
    assert L.kvq_project_append(c, cc, xp.data_ptr(), 64, kp.data_ptr(), vp.data_ptr(), 0, None, None, None) == \
        kvq.KVQ_OK


def test_project_full_size_prefill_sampled():
    """The long-context shape's prefill chunk (4 sequences x 4096 tokens, 8 kv
    heads, head_dim 128, hidden 4096 = 32 query heads x 128) through the fused
    path: sampled projected rows against the oracle's fp64 projection, and
    sampled blocks bit-exact against the oracle quantizing the returned rows."""
    B, Hkv, D, T, hidden = 4, 8, 128, 4096, 4096
    P = T // 16
    c = kvq.QuantizedKVCache(kvq.KVQ_FMT_CB2_OUTLIER, B, Hkv, D, P, B * P, 0, device="cuda")
    x, wk, wv = synth.projection_inputs(12, B, T, hidden, Hkv, D, device="cuda")
    kv_out = torch.empty((2, B, T, Hkv, D), dtype=torch.float32, device="cuda")
    kvq.kvq_project_append(c, x, wk, wv, None, kv_out)
    torch.cuda.synchronize()
    assert c.status_word() == 0
    assert (c.seq_lens.cpu().numpy() == T).all()
    rng = np.random.default_rng(0)
    wk_c, wv_c = wk.cpu(), wv.cpu()
    for b, t in zip(rng.integers(0, B, 24), rng.integers(0, T, 24)):
        xr = x[b:b + 1, t:t + 1].cpu()
        for role, w in ((0, wk_c), (1, wv_c)):
            assert_projection_close(kv_out[role, b:b + 1, t:t + 1].cpu().numpy(), xr, w, "KV"[role], Hkv, D, None)
    pool = c.pool.cpu().numpy()
    pt = c.page_table.cpu().numpy()
    stride = oracle.block_stride(oracle.BLK_CB2, D)
    for b, pg, h, role in zip(rng.integers(0, B, 12), rng.integers(0, P, 12), rng.integers(0, Hkv, 12),
                              rng.integers(0, 2, 12)):
        rows = kv_out[role, b, 16 * pg:16 * pg + 16, h].cpu().numpy()
        exp = oracle.quantize_page(oracle.BLK_CB2, D, rows, role=int(role))
        phys = int(pt[b, pg]) & 0x7FFFFFFF
        off = ((phys * Hkv + h) * 2 + role) * stride
        np.testing.assert_array_equal(pool[off:off + stride], exp[:stride])


@pytest.mark.parametrize("hidden", [32, 96, 160])
def test_project_hidden_not_a_multiple_of_the_stage_width(hidden):
    """hidden a multiple of 32 but not of the 64-column stage: the last stage's
    boxes run past the matrices and read zeros."""
    B, Hkv, D, P = 2, 2, 128, 8
    pair = Pair(kvq.KVQ_FMT_FP4_E2M1_S16, B, Hkv, D, P, seed=8)
    x, wk, wv = synth.projection_inputs(8, B, 50, hidden, Hkv, D)
    k, v = pair.project(x, wk, wv, [50, 33])
    assert_projection_close(k, x, wk, "K", Hkv, D, [50, 33])
    assert_projection_close(v, x, wv, "V", Hkv, D, [50, 33])
    pair.assert_cache_equal()


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_CB2_OUTLIER, kvq.KVQ_FMT_INT4_G32])
def test_project_bad_page_entry_is_flagged_and_skipped(fmt):
    """A page-table entry outside the pool: the fused path skips that sequence
    (seq_lens unchanged, nothing written for it), flags KVQ_STATUS_BAD_PAGE,
    and appends the other sequences exactly as the oracle does."""
    B, Hkv, D, P, hidden = 2, 2, 128, 4, 128
    pair = Pair(fmt, B, Hkv, D, P, seed=9)
    x, wk, wv = synth.projection_inputs(9, B, 40, hidden, Hkv, D)
    pt = pair.gpu.page_table.clone()
    pair.gpu.page_table[0, 1] = pair.gpu.cfg.num_pages + 5      # sequence 0 names a page outside the pool
    kv_out = torch.zeros((2, B, 40, Hkv, D), dtype=torch.float32, device="cuda")
    kvq.kvq_project_append(pair.gpu, x.cuda(), wk.cuda(), wv.cuda(), None, kv_out)
    torch.cuda.synchronize()
    assert pair.gpu.status_word() & kvq.KVQ_STATUS_BAD_PAGE
    assert pair.gpu.seq_lens.cpu().tolist() == [0, 40]
    assert (kv_out[:, 0] == 0).all()                                 # the skipped sequence produced nothing
    pair.gpu.page_table.copy_(pt)
    pair.gpu.status.zero_()
    kv = kv_out.cpu().numpy()
    pair.ref.append(kv[0], kv[1], np.array([0, 40], np.int32))      # the oracle appends sequence 1 only
    pair.assert_cache_equal()


def test_project_capacity_overflow_is_flagged():
    B, Hkv, D, P, hidden = 2, 1, 64, 2, 64
    pair = Pair(kvq.KVQ_FMT_FP4_E2M1_S16, B, Hkv, D, P, seed=10)
    x, wk, wv = synth.projection_inputs(10, B, 20, hidden, Hkv, D)
    pair.project(x, wk, wv)
    pair.assert_cache_equal()
    kvq.kvq_project_append(pair.gpu, x.cuda(), wk.cuda(), wv.cuda(), torch.tensor([20, 12], dtype=torch.int32,
                                                                                     device="cuda"))
    torch.cuda.synchronize()
    assert pair.gpu.status_word() & kvq.KVQ_STATUS_CAPACITY          # 40 tokens > 32 slots for sequence 0
    assert pair.gpu.seq_lens.cpu().tolist() == [20, 32]


@pytest.mark.parametrize("fmt", FORMATS)
def test_project_end_to_end_against_the_oracles_own_projection(fmt):
    """End to end from x and the weights: the oracle projects with its own fp64
    product (rounded once to fp32, the quantizer's input precision) and
    quantizes that, while the fused GPU path projects on the tensor cores
    (fp32 accumulation) and quantizes in the same kernel.  The two quantizer
    inputs differ only within the fp32 accumulation bound, so a decision can
    differ only where those inputs straddle it.  Such a straddle moves an
    element by a quantization step; everything else moves by no more than the
    inputs do (a staged tail row, an FP8 page's scale): the elements that move
    by more than 1e-5 of their size are counted and bounded (0.2% of the
    elements), and the GPU's
    attention over its cache must lie within 2e-3, plus the straddles' own
    effect on the exact attention, of the oracle's attention over the
    oracle's cache."""
    B, Hkv, D, P, hidden, T = 2, 2, 128, 24, 256, 200
    tps = [200, 143]
    pair = Pair(fmt, B, Hkv, D, P, seed=21, tiers=tiers_for(fmt, B, P))
    x, wk, wv = synth.projection_inputs(21, B, T, hidden, Hkv, D)
    kg, vg = pair.project(x, wk, wv, tps)           # GPU cache, and the oracle fed the GPU's own K / V
    pair.assert_cache_equal()
    k64, v64 = oracle.project_kv(x.float().numpy(), wk.float().numpy(), wv.float().numpy(), Hkv, D)
    own = oracle.OracleCache(ORACLE_FMT[fmt], B, Hkv, D, P, pair.ref.cfg.num_pages, pair.ref.cfg.num_tier_pages,
                             page_table=pair.pt, static_channels=pair.ref.static_ch.copy())
    own.append(k64.astype(np.float32), v64.astype(np.float32), np.array(tps, np.int32))
    n_diff = n_all = 0
    for b in range(B):
        for h in range(Hkv):
            for role in range(2):
                a = own.dequantize(b, h, role, 0, tps[b])
                g = pair.ref.dequantize(b, h, role, 0, tps[b])
                n_diff += int((np.abs(a - g) > 1e-5 * np.maximum(np.abs(a), np.abs(g)) + 1e-6).sum())
                n_all += a.size
    assert n_diff <= 0.002 * n_all, f"{n_diff} of {n_all} dequantized elements differ"
    q = synth.queries_bf16(21, B, 4 * Hkv, D, device="cuda")
    out = kvq.kvq_decode_attention(pair.gpu, q, D ** -0.5, T, out_dtype=torch.float32)
    torch.cuda.synchronize()
    qb = q.cpu().view(torch.int16).numpy().view(np.uint16)
    exp_own = own.decode(qb, D ** -0.5)
    exp_gpu_inputs = pair.ref.decode(qb, D ** -0.5)
    err = np.abs(out.cpu().numpy() - exp_own)
    assert (err <= 2e-3 + np.abs(exp_own - exp_gpu_inputs)).all(), f"max err {err.max():.3e}"
