"""Parity of the CUDA path (called through the C ABI) with the CPU oracle on
small seeded inputs that span several pages, ragged lengths and partial tails.

Bar: packed caches (codes, scales, codebooks, outlier lists, tier pages,
staging, seq_lens) and kvq_dequantize are bit-exact; decode attention is within
max-abs 2e-3 of the fp64 oracle (fp32 output), plus half a bf16 ulp of the
reference for bf16 output."""
import numpy as np
import pytest
import torch

from _kvq_pairs import Pair, assert_attention_close, make_kv
from sub_byte_quantized_kvq_gb300 import kvq

pytestmark = pytest.mark.gpu

CB2S, A3, CB2G = kvq.KVQ_FMT_CB2_STATIC, kvq.KVQ_FMT_ASYM3_OUTLIER, kvq.KVQ_FMT_CB2_GROUP4
INT4, E2M1, CB2, TIERED = (kvq.KVQ_FMT_INT4_G32, kvq.KVQ_FMT_FP4_E2M1_S16, kvq.KVQ_FMT_CB2_OUTLIER,
                           kvq.KVQ_FMT_TIERED)
FORMATS_D = [(INT4, 64), (INT4, 128), (E2M1, 64), (E2M1, 128), (CB2, 64), (CB2, 128), (TIERED, 64), (TIERED, 128),
             (CB2S, 64), (CB2S, 128), (A3, 64), (A3, 128), (CB2G, 64), (CB2G, 128)]
IDS = [f"{['int4', 'e2m1', 'cb2', 'tiered', 'cb2s', 'a3', 'cb2g'][f]}-d{d}" for f, d in FORMATS_D]


def _tiers(fmt, B, P):
    t = np.zeros((B, P), bool)
    if fmt == TIERED:
        t[:, 1::3] = True
    return t


def _dist(fmt):
    return ("student_t4", 0, 1.0) if fmt == E2M1 else ("normal", 4, 8.0)


@pytest.mark.parametrize("fmt,D", FORMATS_D, ids=IDS)
@pytest.mark.parametrize("pattern", ["prefill", "tokens", "ragged", "prefill_bf16", "prefill_f16"])
def test_quantize_append_bit_exact(fmt, D, pattern):
    B, Hkv, P = 3, 2, 8
    pair = Pair(fmt, B, Hkv, D, P, seed=1, tiers=_tiers(fmt, B, P))
    dist, n_out, factor = _dist(fmt)
    T = 100 if pattern.startswith("prefill") else 40
    k, v = make_kv(5, B, T if pattern != "ragged" else 120, Hkv, D, dist, n_out, factor)
    if pattern == "prefill":
        pair.append(k, v)
    elif pattern == "prefill_bf16":
        pair.append(k, v, dtype=torch.bfloat16)
    elif pattern == "prefill_f16":
        pair.append(k, v, dtype=torch.float16)
    elif pattern == "tokens":
        for t in range(T):
            pair.append(k[:, t:t + 1], v[:, t:t + 1])
    else:
        pos = np.zeros(B, int)
        for tps in ([20, 5, 0], [3, 17, 9], [16, 16, 16], [1, 0, 31], [40, 2, 15]):
            Tc = max(tps)
            kc = torch.zeros((B, Tc, Hkv, D))
            vc = torch.zeros((B, Tc, Hkv, D))
            for b in range(B):
                kc[b, :tps[b]] = k[b, pos[b]:pos[b] + tps[b]]
                vc[b, :tps[b]] = v[b, pos[b]:pos[b] + tps[b]]
                pos[b] += tps[b]
            assert pair.append(kc, vc, t_per_seq=tps) == 0
    pair.assert_cache_equal()


@pytest.mark.parametrize("fmt", [INT4, E2M1, CB2])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_append_unaligned_inputs(fmt, dtype):
    """K / V that start one element past a 16-byte boundary: the quantizers
    fall back to element loads and still match the oracle bit for bit."""
    B, Hkv, D, P, T = 2, 2, 128, 8, 70
    pair = Pair(fmt, B, Hkv, D, P, seed=21)
    dist, n_out, factor = _dist(fmt)
    k, v = make_kv(21, B, T, Hkv, D, dist, n_out, factor)
    kd, vd = k.to(dtype), v.to(dtype)
    n = kd.numel()
    kb = torch.zeros(n + 1, dtype=dtype, device="cuda")
    vb = torch.zeros(n + 1, dtype=dtype, device="cuda")
    kb[1:] = kd.reshape(-1).cuda()
    vb[1:] = vd.reshape(-1).cuda()
    ku, vu = kb[1:].view(kd.shape), vb[1:].view(vd.shape)
    assert ku.data_ptr() % 16 != 0 and vu.data_ptr() % 16 != 0
    kvq.kvq_quantize_append(pair.gpu, ku, vu, torch.tensor([T, 37], dtype=torch.int32, device="cuda"))
    pair.ref.append(kd.float().numpy(), vd.float().numpy(), np.array([T, 37], np.int32))
    pair.assert_cache_equal()


@pytest.mark.parametrize("fmt,D", FORMATS_D, ids=IDS)
def test_dequantize_bit_exact(fmt, D):
    B, Hkv, P = 2, 2, 7
    pair = Pair(fmt, B, Hkv, D, P, seed=2, tiers=_tiers(fmt, B, P))
    k, v = make_kv(6, B, 83, Hkv, D, *_dist(fmt))
    pair.append(k, v, t_per_seq=[83, 50])
    for b, L in enumerate([83, 50]):
        for h in range(Hkv):
            for role in (0, 1):
                got = kvq.kvq_dequantize(pair.gpu, b, h, role, 0, L).cpu().numpy()
                exp = pair.ref.dequantize(b, h, role, 0, L)
                np.testing.assert_array_equal(got.view(np.int32), exp.view(np.int32))
                got = kvq.kvq_dequantize(pair.gpu, b, h, role, 5, 37).cpu().numpy()
                np.testing.assert_array_equal(got.view(np.int32), exp[5:37].view(np.int32))


@pytest.mark.parametrize("fmt,D", FORMATS_D, ids=IDS)
@pytest.mark.parametrize("G", [1, 4, 8, 16])
def test_decode_attention_parity(fmt, D, G):
    B, Hkv, P = 3, 2, 14
    lens = [209, 77, 1]
    pair = Pair(fmt, B, Hkv, D, P, seed=3, tiers=_tiers(fmt, B, P))
    k, v = make_kv(7, B, max(lens), Hkv, D, *_dist(fmt))
    pair.append(k, v, t_per_seq=lens)
    for splits in (0, 1, 5):
        for od in (torch.float32, torch.bfloat16):
            got, exp = pair.decode(Hkv * G, seed=splits, num_splits=splits, out_dtype=od)
            assert_attention_close(got, exp, od)
    assert pair.gpu.status_word() == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4])
@pytest.mark.parametrize("dist", ["normal", "student_t4"])
def test_decode_cuda_cores_parity(D, G, dist):
    """KVQ_DECODE_CUDA_CORES: the CB2 pages' QK^T and PV as fp32 FMAs (G <= 4),
    against the oracle with the same bar as the tensor-core path; heavy tails
    give side-lists longer than the prefetched records."""
    B, Hkv, P = 3, 2, 14
    lens = [209, 77, 1]
    pair = Pair(CB2, B, Hkv, D, P, seed=21)
    k, v = make_kv(22, B, max(lens), Hkv, D, *((dist, 4, 8.0) if dist == "normal" else (dist, 0, 1.0)))
    pair.append(k, v, t_per_seq=lens)
    pair.gpu.cfg.decode_math = kvq.KVQ_DECODE_CUDA_CORES
    for splits in (0, 1, 5):
        for od in (torch.float32, torch.bfloat16):
            got, exp = pair.decode(Hkv * G, seed=splits, num_splits=splits, out_dtype=od)
            assert_attention_close(got, exp, od)
    assert pair.gpu.status_word() == 0


def test_decode_cuda_cores_token_by_token_and_fallback():
    """The CUDA-core path after single-token appends (partial pages from
    staging, page boundaries); a group size it does not cover (G = 8) runs the
    tensor-core kernel, bit for bit."""
    B, Hkv, D, P = 2, 2, 128, 4
    pair = Pair(CB2, B, Hkv, D, P, seed=23)
    k, v = make_kv(24, B, 40, Hkv, D)
    pair.gpu.cfg.decode_math = kvq.KVQ_DECODE_CUDA_CORES
    for t in range(40):
        pair.append(k[:, t:t + 1], v[:, t:t + 1])
        if t in (0, 15, 16, 31, 32, 39):
            got, exp = pair.decode(Hkv * 4, seed=t)
            assert_attention_close(got, exp)
    # the two-stage calls run the same CUDA-core kernel
    from sub_byte_quantized_kvq_gb300 import synth
    cache, Hq, L = pair.gpu, Hkv * 4, 40
    q = synth.queries_bf16(6, B, Hq, D, device="cuda")
    ws = kvq.alloc_workspace(cache, Hq, L, 3)
    one = kvq.kvq_decode_attention(cache, q, D ** -0.5, L, 3, out_dtype=torch.float32, workspace=ws)
    two = torch.empty_like(one)
    kvq.kvq_decode_split(cache, q, D ** -0.5, L, ws, 3)
    kvq.kvq_decode_combine(cache, Hq, L, ws, two, 3)
    torch.cuda.synchronize()
    assert torch.equal(one, two)
    cc, _ = pair.decode(Hkv * 8, seed=5)
    pair.gpu.cfg.decode_math = kvq.KVQ_DECODE_TENSOR_CORES
    tc, exp = pair.decode(Hkv * 8, seed=5)
    np.testing.assert_array_equal(cc, tc)
    assert_attention_close(tc, exp)


@pytest.mark.parametrize("fmt", [INT4, E2M1, CB2, TIERED, CB2S, A3, CB2G])
def test_fused_merge_matches_split_then_combine(fmt):
    """kvq_decode_attention merges the splits inside its one launch (the last
    CTA of each (sequence, kv head) to arrive); kvq_decode_split followed by
    kvq_decode_combine does it in a second kernel with the same arithmetic.
    The results are identical, and repeated calls on one workspace work (the
    arrival counters return to zero)."""
    B, Hkv, D, P, G = 3, 2, 128, 14, 4
    lens = [209, 77, 1]
    pair = Pair(fmt, B, Hkv, D, P, seed=9, tiers=_tiers(fmt, B, P))
    k, v = make_kv(10, B, max(lens), Hkv, D, *_dist(fmt))
    pair.append(k, v, t_per_seq=lens)
    cache, Hq, L = pair.gpu, Hkv * G, max(lens)
    from sub_byte_quantized_kvq_gb300 import synth
    q = synth.queries_bf16(4, B, Hq, D, device="cuda")
    for S in (1, 2, 5, 14):
        ws = kvq.alloc_workspace(cache, Hq, L, S)
        two = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_split(cache, q, D ** -0.5, L, ws, S)
        kvq.kvq_decode_combine(cache, Hq, L, ws, two, S)
        for _ in range(3):
            one = kvq.kvq_decode_attention(cache, q, D ** -0.5, L, S, out_dtype=torch.float32, workspace=ws)
            torch.cuda.synchronize()
            assert torch.equal(one, two), f"S={S}"
        assert (ws.view(torch.int32)[:B * Hkv] == 0).all()   # the arrival counters, at the start
    assert cache.status_word() == 0


def test_one_workspace_across_call_shapes():
    """The arrival counters sit at the workspace's start whatever the call's
    shape, so one workspace (sized for the largest call) serves calls with
    other split counts, query heads and lengths; each gives the result of a
    fresh workspace, bit for bit."""
    B, Hkv, D, P = 3, 2, 128, 14
    lens = [209, 77, 130]
    pair = Pair(CB2, B, Hkv, D, P, seed=31)
    k, v = make_kv(32, B, max(lens), Hkv, D)
    pair.append(k, v, t_per_seq=lens)
    cache = pair.gpu
    from sub_byte_quantized_kvq_gb300 import synth
    calls = ((4, 5, 224), (4, 1, 224), (8, 14, 224), (4, 5, 213), (8, 0, 224), (4, 14, 213))
    big = max(kvq.kvq_decode_workspace_bytes(cache, Hkv * G, L, S) for G, S, L in calls)
    ws = torch.zeros((big + 15) // 16 * 4, dtype=torch.float32, device="cuda")
    for G, S, L in calls:
        q = synth.queries_bf16(G + S, B, Hkv * G, D, device="cuda")
        shared = kvq.kvq_decode_attention(cache, q, D ** -0.5, L, S, out_dtype=torch.float32, workspace=ws)
        fresh = kvq.kvq_decode_attention(cache, q, D ** -0.5, L, S, out_dtype=torch.float32,
                                         workspace=kvq.alloc_workspace(cache, Hkv * G, L, S))
        torch.cuda.synchronize()
        assert torch.equal(shared, fresh), (G, S, L)
        assert (ws.view(torch.int32)[:B * Hkv] == 0).all()
    assert cache.status_word() == 0


@pytest.mark.parametrize("fmt", [CB2, TIERED, A3, CB2G])
@pytest.mark.parametrize("D,dist", [(64, "student_t4"), (128, "student_t4"), (128, "normal")])
def test_decode_side_lists_longer_than_prefetch(fmt, D, dist):
    """The decode kernel gets the first six side-list records (channels) with
    each block and copies further ones from global memory six at a time.
    Heavy tails, or no dominant outlier channels, spread the outliers over many
    channels and make blocks with more than six common."""
    B, Hkv, P, G = 2, 2, 10, 8
    lens = [150, 97]
    pair = Pair(fmt, B, Hkv, D, P, seed=12, tiers=_tiers(fmt, B, P))
    k, v = make_kv(13, B, max(lens), Hkv, D, dist, 0, 1.0)
    pair.append(k, v, t_per_seq=lens)
    blocks = pair.ref.pool.reshape(-1, pair.ref.stride)
    nch = blocks[:, (10 if fmt == A3 else 12) * D].astype(np.int64)
    assert (nch > 6).sum() >= 2 and (nch > 12).sum() >= (2 if dist == "student_t4" else 0)
    for splits in (0, 3):
        for od in (torch.float32, torch.bfloat16):
            got, exp = pair.decode(Hkv * G, seed=splits, num_splits=splits, out_dtype=od)
            assert_attention_close(got, exp, od)
    assert pair.gpu.status_word() == 0


@pytest.mark.parametrize("fmt", [INT4, E2M1, CB2, TIERED, CB2S, A3, CB2G])
def test_decode_after_token_by_token_appends(fmt):
    """Decode after every single-token append (the serving loop), crossing page boundaries."""
    B, Hkv, D, P, G = 2, 2, 128, 4, 4
    pair = Pair(fmt, B, Hkv, D, P, seed=4, tiers=_tiers(fmt, B, P))
    k, v = make_kv(8, B, 40, Hkv, D, *_dist(fmt))
    for t in range(40):
        pair.append(k[:, t:t + 1], v[:, t:t + 1])
        if t in (0, 14, 15, 16, 31, 32, 39):
            got, exp = pair.decode(Hkv * G, seed=t)
            assert_attention_close(got, exp)


def test_empty_and_single_token_sequences():
    B, Hkv, D, P = 3, 1, 128, 3
    pair = Pair(CB2, B, Hkv, D, P, seed=5)
    k, v = make_kv(9, B, 33, Hkv, D)
    pair.append(k, v, t_per_seq=[0, 1, 33])
    got, exp = pair.decode(4, num_splits=2)
    assert (got[0] == 0).all() and (exp[0] == 0).all()
    assert_attention_close(got, exp)
    # one cached token: the output is that token's V row (as stored: fp32 staging)
    np.testing.assert_allclose(got[1], np.broadcast_to(v[1, 0, 0].numpy(), got[1].shape), atol=1e-6)


@pytest.mark.parametrize("fmt", [INT4, CB2])
def test_constant_and_extreme_values(fmt):
    """Constant pages (zero std: no outliers, degenerate codebooks) and outliers
    far beyond the e4m3 range (both sides saturate at 448) stay bit-exact."""
    B, Hkv, D, P = 2, 1, 64, 3
    pair = Pair(fmt, B, Hkv, D, P, seed=6)
    k = torch.full((B, 48, Hkv, D), 0.75)
    v = torch.full((B, 48, Hkv, D), -1.5)
    k[1, :, 0, 3] = 3000.0 * torch.linspace(-1, 1, 48)
    v[1, :, 0, 9] = 1e4
    pair.append(k, v)
    pair.assert_cache_equal()
    got, exp = pair.decode(4, scale=1e-4)
    assert_attention_close(got, exp, tol=2e-3 * max(1.0, float(np.abs(exp).max()) / 100))


def test_bad_page_entry_is_flagged_and_skipped():
    B, Hkv, D, P = 2, 1, 128, 4
    pair = Pair(CB2, B, Hkv, D, P, seed=7, extra_pages=0)
    k, v = make_kv(10, B, 40, Hkv, D)
    pt = pair.gpu.page_table.clone()
    pair.gpu.page_table[0, 1] = pair.gpu.cfg.num_pages + 5      # sequence 0 names a page outside the pool
    kvq.kvq_quantize_append(pair.gpu, k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert pair.gpu.status_word() & kvq.KVQ_STATUS_BAD_PAGE
    assert pair.gpu.seq_lens.cpu().tolist() == [0, 40]          # sequence 0 skipped, 1 appended
    pair.gpu.page_table.copy_(pt)
    pair.gpu.status.zero_()


@pytest.mark.parametrize("fmt", [CB2, TIERED, E2M1])
def test_decode_bad_page_entry_is_flagged_and_skipped(fmt):
    """A page-table entry outside its pool at decode time: the page is skipped
    (its tokens do not take part), KVQ_STATUS_BAD_PAGE is set, and the other
    pages still give a finite softmax over the rest of the sequence."""
    B, Hkv, D, P = 2, 2, 128, 6
    pair = Pair(fmt, B, Hkv, D, P, seed=12, tiers=_tiers(fmt, B, P))
    k, v = make_kv(12, B, 96, Hkv, D, *_dist(fmt))
    pair.append(k, v)
    pt = pair.gpu.page_table.clone()
    pair.gpu.page_table[1, 2] = pair.gpu.cfg.num_pages + 3
    q = torch.ones((B, 4 * Hkv, D), dtype=torch.bfloat16, device="cuda")
    out = kvq.kvq_decode_attention(pair.gpu, q, D ** -0.5, 96, 2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pair.gpu.status_word() & kvq.KVQ_STATUS_BAD_PAGE
    assert torch.isfinite(out).all()
    pair.gpu.page_table.copy_(pt)
    pair.gpu.status.zero_()
    good = kvq.kvq_decode_attention(pair.gpu, q, D ** -0.5, 96, 2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pair.gpu.status_word() == 0
    assert torch.equal(out[0], good[0])          # the other sequence is untouched


def test_capacity_overflow_matches_oracle():
    B, Hkv, D, P = 2, 1, 64, 2
    pair = Pair(E2M1, B, Hkv, D, P, seed=8)
    k, v = make_kv(11, B, 20, Hkv, D, "student_t4", 0, 1.0)
    pair.append(k, v)
    bad = pair.append(k, v, t_per_seq=[20, 12])     # 40 > 32 slots for sequence 0
    assert bad == 1
    torch.cuda.synchronize()
    assert pair.gpu.status_word() & kvq.KVQ_STATUS_CAPACITY
    pair.gpu.status.zero_()
    pair.assert_cache_equal()


def test_seq_longer_than_max_seq_len_is_flagged():
    B, Hkv, D, P = 1, 1, 128, 4
    pair = Pair(CB2, B, Hkv, D, P, seed=9)
    k, v = make_kv(12, B, 50, Hkv, D)
    pair.append(k, v)
    q = torch.zeros((1, 4, D), dtype=torch.bfloat16, device="cuda")
    kvq.kvq_decode_attention(pair.gpu, q, 0.1, 32)
    torch.cuda.synchronize()
    assert pair.gpu.status_word() & kvq.KVQ_STATUS_SEQ_TOO_LONG


def test_workspace_and_argument_errors():
    pair = Pair(CB2, 1, 2, 128, 2, seed=10)
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention(pair.gpu, q, 0.1, 32, workspace=ws)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE
    with pytest.raises(kvq.KVQError) as e:   # 3 query heads do not divide over 2 kv heads
        kvq.kvq_decode_attention(pair.gpu, torch.zeros((1, 3, 128), dtype=torch.bfloat16, device="cuda"), 0.1, 32)
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt,D", [(CB2, 128), (TIERED, 128), (E2M1, 128), (INT4, 64), (CB2S, 128), (A3, 64),
                                   (CB2G, 128)])
def test_decode_query_of_extreme_magnitude(fmt, D):
    """Query heads far outside fp16's comfortable range: components near 1e5
    (above fp16's 65504), heads whose largest component is 1e-6 (below fp16's
    normal range), and a head mixing both scales.  Each head's query is
    brought into fp16 range by a power of two folded into its score scale,
    so the result stays within the attention tolerance of the fp64 oracle."""
    B, Hkv, G, P = 2, 2, 8, 10
    pair = Pair(fmt, B, Hkv, D, P, seed=31, tiers=_tiers(fmt, B, P))
    k, v = make_kv(31, B, 150, Hkv, D, *_dist(fmt))
    pair.append(k, v, t_per_seq=[150, 97])
    rng = np.random.default_rng(31)
    q = rng.standard_normal((B, Hkv * G, D))
    q[:, 0] *= 1e5 / 4            # components up to ~1e5
    q[:, 1] *= 1e-6               # tiny head
    q[:, 2, :4] = [3e4, -5e4, 2e-7, 1.0]
    q[:, 3] *= 3e-5 / 4
    q[:, 9] = 0.0                 # an all-zero head: uniform attention
    qt = torch.from_numpy(q).float().to(torch.bfloat16)
    qbits = qt.view(torch.int16).numpy().view(np.uint16)
    for od in (torch.float32, torch.bfloat16):
        out = kvq.kvq_decode_attention(pair.gpu, qt.cuda(), D ** -0.5, 150, 3, out_dtype=od)
        torch.cuda.synchronize()
        exp = pair.ref.decode(qbits, D ** -0.5)
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert_attention_close(got, exp, od)
