"""Seeded synthetic inputs for the quantized-KV decode path.

This module only draws random inputs: it holds none of the method's arithmetic
(no quantization, no attention) and is the one piece of code that both the CUDA
path's tests/benchmarks and the CPU oracle consume.

Workloads (shapes and distributions of the five cases the library is measured
on; no public dataset is involved, these stand in for real KV caches):

  tiny_int4      B1  Hkv1 Hq4  D64  N256     INT4 g32, N(0,1) K/V with channels
                 {0, 1} scaled x10 (two channels of one 32-group), fp16 outliers
  cb2_4k         B8  Hkv8 Hq32 D128 N4096    2-bit codebook + e4m3 outliers,
                 N(0,1) with 4 of 128 channels x8
  fp4_32k        B16 Hkv8 Hq64 D128 N32768   E2M1 + e4m3/16, Student-t(4)/sqrt(2)
  tiered_32k     B64 Hkv8 Hq64 D128 N32768   shuffled page table; the 10% of
                 pages with the largest Zipf(1.1) mass are FP8 pages, the rest
                 as cb2_4k
  longctx_128k   B4  Hkv8 Hq32 D128 N131072  2-bit codebook, 1% (=1) outlier
                 channel x10, 64 splits
  static_4k      B8  Hkv8 Hq32 D128 N4096    2-bit codebook with a static fp16
                 channel mask (2 = ceil(1% of 128) channels per K|V and head,
                 chosen from sequence 0's first 256 tokens), 1 channel x10
  a3_4k          B8  Hkv8 Hq32 D128 N4096    3-bit asymmetric codes + e4m3
                 outliers, data as cb2_4k
  group_4k       B8  Hkv8 Hq32 D128 N4096    2-bit codebook per group of 4
                 pages + e4m3 outliers, data as cb2_4k

Every generator takes an explicit seed; per-sequence data is drawn from a
generator seeded by (seed, sequence) so one sequence of a large workload can be
regenerated on its own (for sampled checks against the oracle).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

FMT_INT4, FMT_E2M1, FMT_CB2, FMT_TIERED, FMT_CB2S, FMT_A3, FMT_CB2G = 0, 1, 2, 3, 4, 5, 6
CALIBRATION_TOKENS = 256   # static channel mask: chosen from sequence 0's first tokens
TIER_BIT = 1 << 31


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    fmt: int
    B: int
    Hkv: int
    Hq: int
    D: int
    N: int
    dist: str                 # "normal" or "student_t4"
    n_outlier_channels: int   # channels scaled by `factor` per (K|V, head)
    factor: float
    fixed_channels: tuple = ()   # explicit outlier channels (overrides random choice)
    shuffled: bool = False
    tier_frac: float = 0.0
    zipf_s: float = 1.1
    splits: int = 0              # 0 = library heuristic
    static_channels: int = 0     # FMT_CB2S: fp16 channels per (K|V, head)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def pages(self) -> int:
        return (self.N + 15) // 16


WORKLOADS = {
    "tiny_int4": Workload("tiny_int4", FMT_INT4, 1, 1, 4, 64, 256, "normal", 2, 10.0, fixed_channels=(0, 1)),
    "cb2_4k": Workload("cb2_4k", FMT_CB2, 8, 8, 32, 128, 4096, "normal", 4, 8.0),
    "fp4_32k": Workload("fp4_32k", FMT_E2M1, 16, 8, 64, 128, 32768, "student_t4", 0, 1.0),
    "tiered_32k": Workload("tiered_32k", FMT_TIERED, 64, 8, 64, 128, 32768, "normal", 4, 8.0, shuffled=True,
                           tier_frac=0.10),
    "longctx_128k": Workload("longctx_128k", FMT_CB2, 4, 8, 32, 128, 131072, "normal", 1, 10.0, splits=64),
    "static_4k": Workload("static_4k", FMT_CB2S, 8, 8, 32, 128, 4096, "normal", 1, 10.0, static_channels=2),
    "a3_4k": Workload("a3_4k", FMT_A3, 8, 8, 32, 128, 4096, "normal", 4, 8.0),
    "group_4k": Workload("group_4k", FMT_CB2G, 8, 8, 32, 128, 4096, "normal", 4, 8.0),
}


def outlier_channels(seed: int, Hkv: int, D: int, n: int, fixed=()) -> np.ndarray:
    """[2 (K|V), Hkv, n] channel indices, drawn once per (K|V, head)."""
    if fixed:
        return np.broadcast_to(np.array(fixed, np.int64), (2, Hkv, len(fixed))).copy()
    rng = np.random.default_rng([seed, 7919])
    out = np.zeros((2, Hkv, n), np.int64)
    for r in range(2):
        for h in range(Hkv):
            out[r, h] = np.sort(rng.choice(D, size=n, replace=False))
    return out


def kv_tokens(seed: int, b: int, t0: int, T: int, Hkv: int, D: int, dist: str, channels: np.ndarray,
              factor: float, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """K, V float32 [T, Hkv, D] for tokens [t0, t0+T) of sequence b."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(b) * 7_919 + int(t0) // 16)
    out = []
    for r in range(2):
        x = torch.randn((T, Hkv, D), generator=g, device=device, dtype=torch.float32)
        if dist == "student_t4":
            # Student-t with 4 dof: N / sqrt(chi2_4 / 4); chi2_4 = sum of 4 squared normals.
            z = torch.randn((T, Hkv, D, 4), generator=g, device=device, dtype=torch.float32)
            chi2 = (z * z).sum(-1)
            x = x / torch.sqrt(chi2 / 4.0) / math.sqrt(2.0)   # variance nu/(nu-2) = 2 -> 1
        if channels.size:
            scale = torch.ones((Hkv, D), device=device, dtype=torch.float32)
            for h in range(Hkv):
                scale[h, torch.as_tensor(channels[r, h], device=device)] = factor
            x = x * scale
        out.append(x)
    return out[0], out[1]


def workload_kv(w: Workload, seed: int, b: int, t0: int, T: int, device="cpu"):
    ch = outlier_channels(seed, w.Hkv, w.D, w.n_outlier_channels, w.fixed_channels)
    return kv_tokens(seed, b, t0, T, w.Hkv, w.D, w.dist, ch, w.factor, device)


def projection_inputs(seed: int, B: int, T: int, hidden: int, Hkv: int, D: int, n_out: int = 4,
                      factor: float = 8.0, device="cpu"):
    """Layer input x bf16 [B, T, hidden] ~ N(0, 1) and K / V projection weights
    bf16 [Hkv * D, hidden] ~ N(0, 1 / hidden) (so projected values are about
    unit variance), the weight rows of n_out channels per (K|V, head) scaled by
    `factor` so the projected K / V carry outlier channels like the workloads'."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 131 + 7)
    x = torch.randn((B, T, hidden), generator=g, dtype=torch.float32).to(torch.bfloat16)
    ch = outlier_channels(seed, Hkv, D, n_out)
    ws = []
    for r in range(2):
        w = torch.randn((Hkv, D, hidden), generator=g, dtype=torch.float32) * hidden ** -0.5
        for h in range(Hkv):
            w[h, torch.as_tensor(ch[r, h])] *= factor
        ws.append(w.reshape(Hkv * D, hidden).to(torch.bfloat16))
    return x.to(device), ws[0].to(device), ws[1].to(device)


def queries_bf16(seed: int, B: int, Hq: int, D: int, device="cpu") -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 31 + 17)
    return torch.randn((B, Hq, D), generator=g, dtype=torch.float32).to(torch.bfloat16).to(device)


def tier_pages(seed: int, B: int, N: int, frac: float, s: float) -> np.ndarray:
    """bool [B, pages]: the ceil(frac * pages) pages with the largest synthetic
    attention mass.  Mass of a position = rank^(-s) with rank a seeded random
    permutation of 1..N (a Zipf-distributed stand-in for cumulative attention
    weight); page mass = sum over its tokens; ties go to the lower page index."""
    pages = (N + 15) // 16
    k = math.ceil(frac * pages)
    out = np.zeros((B, pages), bool)
    for b in range(B):
        rng = np.random.default_rng([seed, 104729, b])
        rank = rng.permutation(N) + 1
        w = rank.astype(np.float64) ** (-s)
        wp = np.zeros(pages * 16)
        wp[:N] = w
        mass = wp.reshape(pages, 16).sum(1)
        order = np.lexsort((np.arange(pages), -mass))
        out[b, order[:k]] = True
    return out


def page_table(seed: int, B: int, pages_per_seq: int, shuffled: bool, tiers: np.ndarray | None = None):
    """int32 [B, pages_per_seq] page table plus the pool sizes it needs.

    Main-pool pages and tier-pool pages are numbered separately; a tier page's
    entry carries bit 31.  With `shuffled`, physical indices are a seeded
    permutation (pages of a sequence scattered through the pool)."""
    rng = np.random.default_rng([seed, 15485863])
    tiers = np.zeros((B, pages_per_seq), bool) if tiers is None else tiers
    n_tier = int(tiers.sum())
    n_main = B * pages_per_seq - n_tier
    main_ids = rng.permutation(n_main) if shuffled else np.arange(n_main)
    tier_ids = rng.permutation(n_tier) if shuffled else np.arange(n_tier)
    pt = np.zeros((B, pages_per_seq), np.int64)
    mi = ti = 0
    for b in range(B):
        for p in range(pages_per_seq):
            if tiers[b, p]:
                pt[b, p] = tier_ids[ti] | TIER_BIT
                ti += 1
            else:
                pt[b, p] = main_ids[mi]
                mi += 1
    return pt.astype(np.uint32).view(np.int32), n_main, n_tier
