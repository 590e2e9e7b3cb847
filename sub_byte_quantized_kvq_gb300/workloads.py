"""Build a quantized cache on the GPU for one of the synthetic workloads
(synth.WORKLOADS): page table (shuffled / tiered as the workload says), then a
chunked prefill through kvq_quantize_append.  Inputs come from synth's seeded
generators, drawn on the device chunk by chunk, so any chunk can be drawn again
for a sampled check."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import kvq, synth

PREFILL_CHUNK = 4096


@dataclasses.dataclass
class Built:
    w: synth.Workload
    cache: kvq.QuantizedKVCache
    page_table: np.ndarray   # int32 [B, pages]
    tiers: np.ndarray        # bool [B, pages]
    num_pages: int
    num_tier_pages: int
    seed: int


def chunks(N: int, chunk: int = PREFILL_CHUNK):
    t0 = 0
    while t0 < N:
        yield t0, min(chunk, N - t0)
        t0 += chunk


def seq_kv(w: synth.Workload, seed: int, b: int, t0: int, T: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """K, V float32 [T, Hkv, D] of tokens [t0, t0 + T) of sequence b (one prefill chunk)."""
    return synth.workload_kv(w, seed, b, t0, T, device=device)


def calibration_kv(w: synth.Workload, seed: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """K, V [t, Hkv, D] the static channel mask is chosen from: sequence 0's first tokens."""
    return seq_kv(w, seed, 0, 0, min(w.N, synth.CALIBRATION_TOKENS), device)


def build(w: synth.Workload, seed: int = 0, device="cuda", in_dtype=torch.float32) -> Built:
    pages = w.pages
    tiers = synth.tier_pages(seed, w.B, w.N, w.tier_frac, w.zipf_s) if w.tier_frac > 0 else np.zeros((w.B, pages), bool)
    pt, n_main, n_tier = synth.page_table(seed, w.B, pages, w.shuffled, tiers)
    cache = kvq.QuantizedKVCache(w.fmt, w.B, w.Hkv, w.D, pages, max(n_main, 1), n_tier,
                                 page_table=torch.from_numpy(pt), device=device, static_channels=w.static_channels)
    if w.fmt == synth.FMT_CB2S:   # the static channel mask, from calibration tokens
        kc, vc = calibration_kv(w, seed, device)
        kvq.kvq_select_static_channels(cache, kc.to(in_dtype).contiguous(), vc.to(in_dtype).contiguous())
    for t0, T in chunks(w.N):
        k = torch.empty((w.B, T, w.Hkv, w.D), dtype=in_dtype, device=device)
        v = torch.empty_like(k)
        for b in range(w.B):
            kb, vb = seq_kv(w, seed, b, t0, T, device)
            k[b].copy_(kb)
            v[b].copy_(vb)
        kvq.kvq_quantize_append(cache, k, v)
    return Built(w, cache, pt, tiers, max(n_main, 1), n_tier, seed)
