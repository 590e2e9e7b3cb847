"""Parity at the full sizes of the benchmark workloads, in the launch
configuration bench.py times (the workload's split count, bf16 output), on
sampled (sequence, kv head) units the oracle can compute one by one.

For each sampled unit the sequence's K/V chunks are drawn again from the same
seeded device generator, quantized by the oracle on its own (one kv head), and
compared with the GPU cache block by block (bit-exact) and with the GPU decode
output (max-abs 2e-3 plus half a bf16 ulp)."""
import numpy as np
import pytest
import torch

import oracle
from _kvq_pairs import ORACLE_FMT, assert_attention_close
from sub_byte_quantized_kvq_gb300 import kvq, synth, workloads

pytestmark = pytest.mark.gpu

SEED = 0


def _static_mask(built, dev):
    """The oracle's own choice of the static channels from the same calibration values."""
    w = built.w
    kc, vc = workloads.calibration_kv(w, built.seed, dev)
    n = w.static_channels
    return np.stack([oracle.select_static(kc.cpu().numpy(), n), oracle.select_static(vc.cpu().numpy(), n)], 1)


def _oracle_unit(built, b, h, dev):
    w = built.w
    tiers = built.tiers[b:b + 1]
    pt, nm, nt = synth.page_table(SEED, 1, w.pages, False, tiers)
    st = _static_mask(built, dev)[h:h + 1] if w.fmt == synth.FMT_CB2S else None
    ref = oracle.OracleCache(ORACLE_FMT[w.fmt], 1, 1, w.D, w.pages, max(nm, 1), nt, page_table=pt,
                             static_channels=st)
    for t0, T in workloads.chunks(w.N):
        k, v = workloads.seq_kv(w, built.seed, b, t0, T, dev)
        ref.append(k[:, h:h + 1].cpu().numpy()[None], v[:, h:h + 1].cpu().numpy()[None])
    return ref, pt


def _gpu_block(built, phys_entry, h, role):
    c, w = built.cache, built.w
    u = int(phys_entry) & 0xFFFFFFFF
    tier, phys = u >> 31, u & 0x7FFFFFFF
    pool, stride = (c.tier_pool, c.block_bytes(1)) if tier else (c.pool, c.block_bytes(0))
    off = ((phys * w.Hkv + h) * 2 + role) * stride
    return pool[off:off + stride].cpu().numpy()


def _ref_block(ref, entry, role):
    u = int(entry) & 0xFFFFFFFF
    tier, phys = u >> 31, u & 0x7FFFFFFF
    pool, stride = (ref.tier_pool, ref.tier_stride) if tier else (ref.pool, ref.stride)
    off = (phys * 2 + role) * stride
    return pool[off:off + stride]


@pytest.mark.parametrize("name", ["tiny_int4", "cb2_4k", "fp4_32k", "tiered_32k", "longctx_128k", "static_4k",
                                  "a3_4k", "group_4k"])
def test_full_size_workload_sampled(name):
    w = synth.WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    built = workloads.build(w, seed=SEED, device=dev)
    q = synth.queries_bf16(SEED, w.B, w.Hq, w.D, device=dev)
    scale = w.D ** -0.5
    out16 = kvq.kvq_decode_attention(built.cache, q, scale, w.N, w.splits, out_dtype=torch.bfloat16)
    out32 = kvq.kvq_decode_attention(built.cache, q, scale, w.N, w.splits, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert built.cache.status_word() == 0
    assert built.cache.seq_lens.cpu().tolist() == [w.N] * w.B
    if w.fmt == synth.FMT_CB2S:
        np.testing.assert_array_equal(built.cache.static_mask.cpu().numpy(), _static_mask(built, dev))
    qbits = q.cpu().view(torch.int16).numpy().view(np.uint16)
    rng = np.random.default_rng(1)
    units = sorted({(0, 0), (w.B - 1, w.Hkv - 1)})
    for b, h in units:
        ref, pt = _oracle_unit(built, b, h, dev)
        pages = sorted({0, w.pages - 1, w.pages // 2, *rng.integers(0, w.pages, 6).tolist()})
        for p in pages:
            for role in (0, 1):
                got = _gpu_block(built, built.page_table[b, p], h, role)
                exp = _ref_block(ref, pt[0, p], role)
                assert (got == exp).all(), f"{name}: block (seq {b}, page {p}, head {h}, role {role}) differs"
        exp = ref.decode(qbits[b:b + 1, h * w.G:(h + 1) * w.G], scale)[0]
        assert_attention_close(out32[b, h * w.G:(h + 1) * w.G].cpu().numpy(), exp, torch.float32)
        assert_attention_close(out16[b, h * w.G:(h + 1) * w.G].float().cpu().numpy(), exp, torch.bfloat16)
