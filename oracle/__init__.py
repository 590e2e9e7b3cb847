"""CPU oracle for the sub-byte quantized KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline
and reference legs) may import this package.  It shares no code with the CUDA
path.  The arithmetic lives in ``kvq_oracle.c`` (plain C, everything in fp64:
the quantizer's statistics, fits and decisions and the attention, compiled
with ``-ffp-contract=off``); this module compiles it with gcc, loads it with ctypes
and keeps a numpy model of the paged cache (pools, page table, staging tail,
sequence lengths) that mirrors the layout the library documents.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_INT4, FMT_E2M1, FMT_CB2, FMT_TIERED, FMT_CB2S, FMT_A3, FMT_CB2G = 0, 1, 2, 3, 4, 5, 6
BLK_INT4, BLK_E2M1, BLK_CB2, BLK_FP8, BLK_CB2S, BLK_A3, BLK_CB2G = 0, 1, 2, 3, 4, 5, 6
GROUP_PAGES = 4   # pages per CB2 group codebook
TIER_BIT = 1 << 31


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -march flags: it runs on x86 and Arm)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("pages_per_seq_max", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("num_tier_pages", ctypes.c_int32),
                ("iters", ctypes.c_int32), ("sigma", ctypes.c_double),
                ("n_static", ctypes.c_int32), ("static_ch", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, D_ = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            sig = {
                "or_fp16_encode": (ctypes.c_uint16, [D_]), "or_fp16_decode": (D_, [ctypes.c_uint16]),
                "or_e4m3_encode": (ctypes.c_uint8, [D_]), "or_e4m3_decode": (D_, [ctypes.c_uint8]),
                "or_e2m1_encode": (ctypes.c_uint8, [D_]), "or_e2m1_decode": (D_, [ctypes.c_uint8]),
                "or_bf16_decode": (D_, [ctypes.c_uint16]),
                "or_kmax": (I, [I]),
                "or_outlier_mask": (I, [P, I, D_, I, P]),
                "or_lloyd4": (I, [P, I, I, P, P, P]),
                "or_block_stride": (I, [I, I]),
                "or_frag_pos": (None, [I, I, I, P, P, P]),
                "or_quantize_token": (None, [I, I, D_, I, I, P, P]),
                "or_quantize_page": (None, [I, I, D_, I, I, P, P]),
                "or_quantize_page_static": (None, [I, I, I, P, P, I, P]),
                "or_select_static": (None, [P, I, I, I, I, P]),
                "or_quantize_group": (None, [I, D_, I, I, P, P]),
                "or_dequantize_group_page": (None, [I, P, P, I, I, P]),
                "or_dequantize_block": (None, [I, I, P, I, I, P]),
                "or_append": (I, [P, P, P, P, P, P, P, P, I, P]),
                "or_dequantize_range": (None, [P, P, P, P, P, P, I, I, I, I, I, P]),
                "or_attention": (None, [I, I, I, P, P, P, D_, P]),
                "or_decode": (None, [P, P, P, P, P, P, P, I, D_, P, I, I, I]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------- scalar codecs
def fp16_encode(v: float) -> int: return int(lib().or_fp16_encode(float(v)))
def fp16_decode(h: int) -> float: return float(lib().or_fp16_decode(int(h)))
def e4m3_encode(v: float) -> int: return int(lib().or_e4m3_encode(float(v)))
def e4m3_decode(b: int) -> float: return float(lib().or_e4m3_decode(int(b)))
def e2m1_encode(v: float) -> int: return int(lib().or_e2m1_encode(float(v)))
def e2m1_decode(b: int) -> float: return float(lib().or_e2m1_decode(int(b)))
def bf16_decode(h: int) -> float: return float(lib().or_bf16_decode(int(h)))
def kmax(n: int) -> int: return int(lib().or_kmax(n))
def block_stride(blk_fmt: int, D: int) -> int: return int(lib().or_block_stride(blk_fmt, D))


def outlier_mask(x, sigma: float = 3.0, cap: int | None = None):
    """fp64 outlier rule over x (taken as float32, the values a cache receives)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    m = np.zeros(x.size, dtype=np.uint8)
    n = lib().or_outlier_mask(_p(x), x.size, sigma, kmax(x.size) if cap is None else cap, _p(m))
    return m.astype(bool), int(n)


def lloyd4(v, iters: int = 16):
    """fp64 Lloyd-Max fit of v (taken as float32, the values a cache receives).
    Returns (fp64 centroids before fp16 rounding, fp16 bits, codes, passes)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    c = np.zeros(4, np.float64)
    c16 = np.zeros(4, np.uint16)
    codes = np.zeros(max(v.size, 1), np.uint8)
    passes = lib().or_lloyd4(_p(v), v.size, iters, _p(c), _p(c16), _p(codes))
    return c, c16, codes[:v.size], int(passes)


def frag_pos(role: int, t: int, c: int):
    a, b, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    lib().or_frag_pos(role, t, c, ctypes.byref(a), ctypes.byref(b), ctypes.byref(k))
    return a.value, b.value, k.value


def quantize_token(blk_fmt: int, D: int, x, t: int, blk: np.ndarray, role: int = 0, sigma: float = 3.0):
    x = np.ascontiguousarray(x, dtype=np.float32)
    lib().or_quantize_token(blk_fmt, D, sigma, role, t, _p(x), _p(blk))


def quantize_page(blk_fmt: int, D: int, x, role: int = 0, sigma: float = 3.0, iters: int = 16) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(16, D)
    blk = np.zeros(block_stride(blk_fmt, D), np.uint8)
    lib().or_quantize_page(blk_fmt, D, sigma, iters, role, _p(x), _p(blk))
    return blk


def quantize_page_static(D: int, x, channels, role: int = 0, iters: int = 16) -> np.ndarray:
    """CB2 page with static fp16 channels `channels` (ascending, at most 8)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(16, D)
    ch = np.ascontiguousarray(channels, dtype=np.uint8)
    blk = np.zeros(block_stride(BLK_CB2S, D), np.uint8)
    lib().or_quantize_page_static(D, iters, role, _p(x), _p(ch), len(ch), _p(blk))
    return blk


def select_static(x, n_s: int) -> np.ndarray:
    """x: float [t, Hkv, D] calibration values -> uint8 [Hkv, n_s] static channels."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    t, Hkv, D = x.shape
    out = np.zeros((Hkv, n_s), np.uint8)
    lib().or_select_static(_p(x), t, Hkv, D, n_s, _p(out))
    return out


def quantize_group(D: int, x, role: int = 0, sigma: float = 3.0, iters: int = 16) -> np.ndarray:
    """CB2 group of 4 pages from x [64, D] -> uint8 [4, stride] (codebook in block 0)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(64, D)
    blks = np.zeros((4, block_stride(BLK_CB2G, D)), np.uint8)
    lib().or_quantize_group(D, sigma, iters, role, _p(x), _p(blks))
    return blks


def dequantize_group_page(D: int, codes_blk: np.ndarray, codebook_blk: np.ndarray, role: int = 0,
                          ntok: int = 16) -> np.ndarray:
    out = np.zeros((16, D), np.float32)
    lib().or_dequantize_group_page(D, _p(np.ascontiguousarray(codes_blk)), _p(np.ascontiguousarray(codebook_blk)),
                                   role, ntok, _p(out))
    return out[:ntok]


def dequantize_block(blk_fmt: int, D: int, blk: np.ndarray, role: int = 0, ntok: int = 16) -> np.ndarray:
    out = np.zeros((16, D), np.float32)
    lib().or_dequantize_block(blk_fmt, D, _p(np.ascontiguousarray(blk)), role, ntok, _p(out))
    return out[:ntok]


def attention(q, k, v, scale: float) -> np.ndarray:
    """Plain fp64 attention of G query rows q[G][D] over k, v [N][D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    G, D = q.shape
    out = np.zeros((G, D), np.float64)
    lib().or_attention(G, D, k.shape[0], _p(q), _p(k), _p(v), float(scale), _p(out))
    return out


# ----------------------------------------------------------------------------- paged cache model
def project_kv(x, w_k, w_v, Hkv: int, D: int):
    """The appended tokens' K and V as the attention projection of the layer
    input ("Sub-5ms MoE Inference: Sub-Byte KV Quantization and Expert
    Pipelining at Scale", Engineering Real-Time Autonomous Workflows, item 1,
    which fuses this projection with the KV-cache write):
        k[b, i, h, j] = sum_e x[b, i, e] * w_k[h * D + j, e]   (likewise v)
    in fp64.  x [B, T, hidden], w_k / w_v [Hkv * D, hidden] (a linear layer's
    output-major weight).  Returns (k, v) float64 [B, T, Hkv, D]."""
    x = np.asarray(x, np.float64)
    out = []
    for w in (w_k, w_v):
        w = np.asarray(w, np.float64)
        out.append(np.matmul(x, w.T).reshape(x.shape[0], x.shape[1], Hkv, D))
    return out[0], out[1]


class OracleCache:
    """numpy model of the paged, quantized cache (same layout as the library's)."""

    def __init__(self, fmt: int, num_seqs: int, num_kv_heads: int, head_dim: int, pages_per_seq_max: int,
                 num_pages: int, num_tier_pages: int = 0, sigma: float = 3.0, lloyd_iters: int = 16,
                 page_table: np.ndarray | None = None, static_channels: np.ndarray | None = None):
        # static_channels (format 4): uint8 [Hkv, 2, n_s], ascending per (head, role)
        self.static_ch = (np.zeros((num_kv_heads, 2, 1), np.uint8) if static_channels is None
                          else np.ascontiguousarray(static_channels, dtype=np.uint8))
        self.cfg = _Cfg(fmt, num_seqs, num_kv_heads, head_dim, pages_per_seq_max, num_pages,
                        num_tier_pages, lloyd_iters, sigma, self.static_ch.shape[-1], _p(self.static_ch))
        self.fmt, self.B, self.Hkv, self.D = fmt, num_seqs, num_kv_heads, head_dim
        main = BLK_CB2 if fmt == FMT_TIERED else fmt   # FMT_CB2S blocks are BLK_CB2S
        self.stride = block_stride(main, head_dim)
        self.tier_stride = block_stride(BLK_FP8, head_dim)
        self.pool = np.zeros(num_pages * num_kv_heads * 2 * self.stride, np.uint8)
        self.tier_pool = np.zeros(max(num_tier_pages, 0) * num_kv_heads * 2 * self.tier_stride + 1, np.uint8)
        if page_table is None:
            page_table = np.arange(num_seqs * pages_per_seq_max, dtype=np.int64).reshape(num_seqs, -1) % max(num_pages, 1)
        self.page_table = np.ascontiguousarray(page_table.astype(np.uint32).view(np.int32))
        self.seq_lens = np.zeros(num_seqs, np.int32)
        rows = 16 * GROUP_PAGES if fmt == FMT_CB2G else 16
        self.staging = np.zeros((num_seqs, num_kv_heads, 2, rows, head_dim), np.float32)

    def _args(self):
        return (ctypes.byref(self.cfg), _p(self.pool), _p(self.tier_pool), _p(self.page_table))

    def append(self, k_new, v_new, t_per_seq=None) -> int:
        """k_new, v_new: float32 [B, T, Hkv, D] -> number of sequences skipped."""
        k_new = np.ascontiguousarray(k_new, dtype=np.float32)
        v_new = np.ascontiguousarray(v_new, dtype=np.float32)
        tps = None if t_per_seq is None else np.ascontiguousarray(t_per_seq, dtype=np.int32)
        return int(lib().or_append(*self._args(), _p(self.seq_lens), _p(self.staging), _p(k_new), _p(v_new),
                                   k_new.shape[1], _p(tps)))

    def dequantize(self, b: int, h: int, role: int, t0: int, t1: int) -> np.ndarray:
        out = np.zeros((max(t1 - t0, 0), self.D), np.float32)
        lib().or_dequantize_range(*self._args(), _p(self.seq_lens), _p(self.staging), b, h, role, t0, t1,
                                  _p(out))
        return out

    def decode(self, q_bf16_bits: np.ndarray, scale: float, units=None, nthreads: int = 1) -> np.ndarray:
        """q_bf16_bits: uint16 [B, Hq, D] (bf16 bit patterns) -> fp64 [B, Hq, D]."""
        q = np.ascontiguousarray(q_bf16_bits, dtype=np.uint16)
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D), np.float64)
        u0, u1 = (0, B * self.Hkv) if units is None else units
        lib().or_decode(*self._args(), _p(self.seq_lens), _p(self.staging), _p(q), Hq, float(scale), _p(out),
                        u0, u1, nthreads)
        return out
