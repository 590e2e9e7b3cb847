"""Pins for what bench.py's figures rest on, checked on the CPU.

1. bench.step_bytes (the algorithmic bytes every GB/s figure divides) equals
   the bytes an oracle cache of the same small workload actually holds, for
   every format.  The count here is independent of bench.py: it walks each
   block the decode step reads (page table, tier bit, the partial tail that
   stays in staging), parses the block by the layout (side-list records,
   per-token outlier slots, static channels), and checks that no nonzero byte
   of the block lies outside the sections it counts.
2. synth.tier_pages (which pages of the tiered workload are FP8) against a
   brute-force ranking: the ceil(10%) pages with the largest synthetic mass,
   ties to the lower page index ("Hierarchical Token Gating and Tiered
   KV-Cache Paging", 2. Entropy-Guided Tiered KV-Cache Quantization: the pages
   carrying the largest cumulative attention weight go to the FP8 tier).
3. The source hash that keys the stored DRAM traffic record ignores comments
   and layout but not code (a stale record reads as traffic null).
"""
import math

import numpy as np
import pytest

import bench
import oracle
from sub_byte_quantized_kvq_gb300 import synth

FORMATS = [synth.FMT_INT4, synth.FMT_E2M1, synth.FMT_CB2, synth.FMT_TIERED, synth.FMT_CB2S, synth.FMT_A3,
           synth.FMT_CB2G]


def _held(fmt_blk, D, blk, n_static=0):
    """Bytes block `blk` holds by the layout, after checking that every byte
    outside the counted sections is zero and that the side-list parses."""
    used = np.zeros(blk.size, bool)
    if fmt_blk in (oracle.BLK_CB2, oracle.BLK_A3, oracle.BLK_CB2G):
        side = {oracle.BLK_CB2: 12 * D, oracle.BLK_A3: 10 * D, oracle.BLK_CB2G: 12 * D}[fmt_blk]
        n_ch, total = int(blk[side]), int(blk[side + 1])
        last, outl = -1, 0
        for i in range(n_ch):
            rec = blk[side + 4 + 20 * i: side + 24 + 20 * i]
            ch, mask = int(rec[0]), int(rec[2]) | (int(rec[3]) << 8)
            assert ch > last and ch < D and mask != 0 and rec[1] == 0
            assert all(rec[4 + t] == 0 for t in range(16) if not mask >> t & 1)   # values only at outliers
            last, outl = ch, outl + bin(mask).count("1")
        assert outl == total
        used[:side + 4 + 20 * n_ch] = True
        held = int(used.sum())
        if fmt_blk == oracle.BLK_CB2G:
            held -= 8 * D             # the group codebook: counted once per group, by the caller
    elif fmt_blk == oracle.BLK_FP8:
        used[:16 * D + 4] = True
        held = 16 * D + 4
    elif fmt_blk == oracle.BLK_E2M1:
        used[:9 * D] = True
        held = 9 * D
    elif fmt_blk == oracle.BLK_CB2S:
        used[:12 * D + 16 + 32 * n_static] = True
        assert int(blk[12 * D]) == n_static
        held = 12 * D + 16 + 32 * n_static
    else:   # INT4: codes, scale/zero, counts, then only the slots each token's count covers
        cap = 3 * (D // 32)
        used[:10 * D + 16] = True
        held = 10 * D + 16
        for t in range(16):
            cnt = int(blk[10 * D + t])
            assert cnt <= cap
            used[10 * D + 16 + t * cap: 10 * D + 16 + t * cap + cnt] = True
            v0 = 10 * D + 16 + 16 * cap + 2 * t * cap
            used[v0: v0 + 2 * cnt] = True
            held += 3 * cnt
    assert not blk[~used].any(), "block holds nonzero bytes outside the counted sections"
    return held


def _oracle_cache(fmt, B, Hkv, D, N, seed=2):
    pages = (N + 15) // 16
    tiers = None
    if fmt == synth.FMT_TIERED:
        tiers = synth.tier_pages(seed, B, N, 0.25, 1.1)
    pt, nm, nt = synth.page_table(seed, B, pages, True, tiers)
    n_s = 2 if fmt == synth.FMT_CB2S else 0
    st = None
    w = synth.Workload("acct", fmt, B, Hkv, 2 * Hkv, D, N, "normal", 4, 8.0)
    ks, vs = zip(*[synth.workload_kv(w, seed, b, 0, N) for b in range(B)])
    k, v = np.stack([x.numpy() for x in ks]), np.stack([x.numpy() for x in vs])
    if fmt == synth.FMT_CB2S:
        st = np.stack([oracle.select_static(k[0, :64], n_s), oracle.select_static(v[0, :64], n_s)], 1)
    ref = oracle.OracleCache(fmt, B, Hkv, D, pages, max(nm, 1), nt, page_table=pt, static_channels=st)
    ref.append(k, v)
    return ref, pt, tiers, n_s


@pytest.mark.parametrize("N", [208, 200])
@pytest.mark.parametrize("fmt", FORMATS)
def test_step_bytes_equal_what_the_cache_holds(fmt, N):
    B, Hkv, Hq, D = 2, 2, 4, 128
    ref, pt, tiers, n_s = _oracle_cache(fmt, B, Hkv, D, N)
    main = oracle.BLK_CB2 if fmt == synth.FMT_TIERED else fmt
    pool = ref.pool.reshape(-1, ref.stride)
    tpool = ref.tier_pool[:-1].reshape(-1, ref.tier_stride) if ref.tier_pool.size > 1 else None
    paged = fmt in (synth.FMT_CB2, synth.FMT_TIERED, synth.FMT_CB2S, synth.FMT_A3, synth.FMT_CB2G)
    unit = 64 if fmt == synth.FMT_CB2G else 16
    n_blocks_read = N // unit * (unit // 16) if paged else -(-N // 16)
    expect = 0
    for b in range(B):
        for p in range(n_blocks_read):
            u = int(pt[b, p]) & 0xFFFFFFFF
            for h in range(Hkv):
                for role in range(2):
                    if u >> 31:
                        expect += _held(oracle.BLK_FP8, D, tpool[((u & 0x7FFFFFFF) * Hkv + h) * 2 + role])
                    else:
                        blk = pool[(u * Hkv + h) * 2 + role]
                        expect += _held(main, D, blk, n_s)
                        if fmt == synth.FMT_CB2G and p % 4 == 0:
                            expect += 8 * D      # the group's codebook, in its first page
                            assert blk[:8 * D].any()
                        elif fmt == synth.FMT_CB2G:
                            assert not blk[:8 * D].any()
    staged = N - N // unit * unit if paged else 0
    expect += staged * D * 4 * 2 * B * Hkv               # fp32 tail rows of K and V
    expect += 2 * B * Hq * D * 2                         # Q and the output, bf16
    meta = bench.block_meta(fmt, D, pool)
    got = bench.step_bytes(fmt, D, Hkv, Hq, B, N, pt, meta, n_s)
    assert got["step"] == expect
    assert got["split_kernel"] == expect - B * Hq * D * 2


def test_tier_pages_is_the_top_tenth_by_mass():
    B, N, frac, s = 3, 16 * 57 + 5, 0.10, 1.1
    got = synth.tier_pages(11, B, N, frac, s)
    pages = -(-N // 16)
    k = math.ceil(frac * pages)
    assert got.shape == (B, pages) and (got.sum(1) == k).all()
    for b in range(B):
        rank = np.random.default_rng([11, 104729, b]).permutation(N) + 1
        mass = [sum(float(r) ** -s for r in rank[16 * p: 16 * p + 16]) for p in range(pages)]
        # brute force: page p is chosen iff fewer than k pages beat it (heavier, or as heavy and lower)
        for p in range(pages):
            beats = sum(1 for o in range(pages) if mass[o] > mass[p] or (mass[o] == mass[p] and o < p))
            assert got[b, p] == (beats < k), (b, p)


def test_tier_pages_ties_go_to_the_lower_page():
    # s = 0: every position weighs 1, so all full pages tie and the last (partial) page is lightest
    got = synth.tier_pages(0, 1, 16 * 20 + 3, 0.10, 0.0)
    assert np.nonzero(got[0])[0].tolist() == [0, 1, 2]



def test_source_hash_ignores_comments_not_code():
    base = 'asm("mov.u32 %0, %%globaltimer; // kept");\nconstexpr float kTh = 8.0f;\n'
    assert bench.code_only(base) == bench.code_only("// a note\n" + base.replace(";\n", ";   /* x\n y */\n\n"))
    assert "// kept" in bench.code_only(base)                      # string literals are code
    assert bench.code_only(base) != bench.code_only(base.replace("8.0f", "7.0f"))
