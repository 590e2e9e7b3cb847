"""kvq_decode_attention_noalloc: decode attention for callers that may not
allocate device memory while they decode (it keeps the split partials in a
scratch array built into the library instead of a caller workspace).

Checked through the C ABI against kvq_decode_attention, the entry point that
takes a workspace, on two calls in a row (the second call reuses a scratch
that still holds the first call's partials), and on a run of calls whose
shapes differ, within the tolerance the parity tests use (max-abs 2e-3, fp32
output).  This file is collected last so that a
run stopping at its first failure has already run every other test; it builds
its own cache, so it also passes alone in a fresh process.
"""
import pytest
import torch

from sub_byte_quantized_kvq_gb300 import kvq, synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _cache(fmt, B=3, Hkv=2, G=4, D=128, lens=(209, 77, 1), P=14):
    w = synth.Workload("noalloc", fmt, B, Hkv, Hkv * G, D, max(lens), "normal", 4, 8.0)
    pt, nm, _ = synth.page_table(5, B, P, True)
    cache = kvq.QuantizedKVCache(fmt, B, Hkv, D, P, nm, page_table=torch.from_numpy(pt), device="cuda")
    ks, vs = zip(*[synth.workload_kv(w, 3, b, 0, max(lens)) for b in range(B)])
    kvq.kvq_quantize_append(cache, torch.stack(ks).cuda(), torch.stack(vs).cuda(),
                            torch.tensor(lens, dtype=torch.int32, device="cuda"))
    q = synth.queries_bf16(7, B, Hkv * G, D, device="cuda")
    return cache, q, max(lens)


@pytest.mark.parametrize("fmt", [kvq.KVQ_FMT_CB2_OUTLIER, kvq.KVQ_FMT_FP4_E2M1_S16])
@pytest.mark.parametrize("splits", [0, 5])
def test_noalloc_matches_workspace_entry_point_on_two_calls(fmt, splits):
    cache, q, L = _cache(fmt)
    scale = q.shape[-1] ** -0.5
    ref = kvq.kvq_decode_attention(cache, q, scale, L, splits, out_dtype=torch.float32)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_decode_attention_noalloc(cache, q, scale, L, splits, out=out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert (out - ref).abs().max().item() <= TOL
    assert cache.status_word() == 0


def test_noalloc_bf16_output_and_other_query():
    cache, q, L = _cache(kvq.KVQ_FMT_CB2_OUTLIER)
    scale = q.shape[-1] ** -0.5
    for seed in (11, 12):   # two calls in a row with different queries
        qq = synth.queries_bf16(seed, q.shape[0], q.shape[1], q.shape[2], device="cuda")
        ref = kvq.kvq_decode_attention(cache, qq, scale, L, 3, out_dtype=torch.float32)
        out = kvq.kvq_decode_attention_noalloc(cache, qq, scale, L, 3, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        bound = TOL + 0.5 * 2.0 ** (torch.floor(torch.log2(ref.abs().clamp_min(2.0 ** -126))) - 7)
        assert ((out.float() - ref).abs() <= bound).all()


def test_noalloc_rejects_partials_larger_than_its_scratch():
    cache, q, L = _cache(kvq.KVQ_FMT_CB2_OUTLIER)
    splits = 4000   # 3 x 8 x 4000 rows x 520 bytes, far beyond the 16 MiB scratch
    assert kvq.kvq_decode_workspace_bytes(cache, q.shape[1], L, splits) > kvq.NOALLOC_SCRATCH_BYTES
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention_noalloc(cache, q, 0.1, L, splits, out=out)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == 0).all()   # nothing was launched


def test_noalloc_shape_changes_between_calls():
    """The scratch is shared by every cache: its arrival counters sit at the
    start, one per (sequence, kv head) of the calling cache.  Run splits 5,
    then 1, then a cache with more (sequence, kv head) pairs, then the first
    again: every call must still merge its splits and match the workspace
    entry point."""
    a, qa, La = _cache(kvq.KVQ_FMT_CB2_OUTLIER)
    b, qb, Lb = _cache(kvq.KVQ_FMT_CB2_OUTLIER, B=5, Hkv=3, G=2, lens=(33, 160, 16, 95, 200), P=16)
    scale = qa.shape[-1] ** -0.5
    for cache, q, L, splits in ((a, qa, La, 5), (a, qa, La, 1), (b, qb, Lb, 7), (b, qb, Lb, 2), (a, qa, La, 5),
                                (a, qa, La, 0)):
        ref = kvq.kvq_decode_attention(cache, q, scale, L, splits, out_dtype=torch.float32)
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_decode_attention_noalloc(cache, q, scale, L, splits, out=out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"splits {splits}: output not written"
        assert (out - ref).abs().max().item() <= TOL
    assert a.status_word() == 0 and b.status_word() == 0
