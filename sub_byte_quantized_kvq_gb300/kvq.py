"""Thin Python binding of the C ABI in include/kvq.h (argument marshalling only).

Every step of the path runs in the CUDA library ``_build/libkvq.so``; torch
supplies device memory and streams.  If the library is missing the calls raise
``KVQError`` -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

KVQ_FMT_INT4_G32, KVQ_FMT_FP4_E2M1_S16, KVQ_FMT_CB2_OUTLIER, KVQ_FMT_TIERED, KVQ_FMT_CB2_STATIC = 0, 1, 2, 3, 4
KVQ_FMT_ASYM3_OUTLIER, KVQ_FMT_CB2_GROUP4 = 5, 6
KVQ_BF16, KVQ_F16, KVQ_F32 = 0, 1, 2
KVQ_DECODE_AUTO, KVQ_DECODE_TENSOR_CORES, KVQ_DECODE_CUDA_CORES = 0, 1, 2
KVQ_TIER_BIT = 1 << 31
KVQ_STATUS_BAD_PAGE, KVQ_STATUS_CAPACITY, KVQ_STATUS_SEQ_TOO_LONG, KVQ_STATUS_TIMEOUT = 1, 2, 4, 8
KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE, KVQ_ERR_CAPACITY, KVQ_ERR_CUDA = range(6)

_DTYPE = {torch.bfloat16: KVQ_BF16, torch.float16: KVQ_F16, torch.float32: KVQ_F32}


class KVQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = kvq_status_string(status) if _lib is not None else str(status)
        if status == KVQ_ERR_CUDA and _lib is not None:   # the runtime's own error name
            msg += f" {_lib.kvq_cuda_error_name(_lib.kvq_last_cuda_error()).decode()}"
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


class kvq_config(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("pages_per_seq_max", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("num_tier_pages", ctypes.c_int32), ("format", ctypes.c_int32), ("lloyd_iters", ctypes.c_int32),
                ("sigma", ctypes.c_double), ("static_channels", ctypes.c_int32),
                ("decode_math", ctypes.c_int32)]


class kvq_cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("tier_pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("staging", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("static_mask", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()
EXPORTS = ("kvq_block_bytes", "kvq_cache_bytes", "kvq_quantize_append", "kvq_project_append",
           "kvq_decode_workspace_bytes",
           "kvq_decode_num_splits", "kvq_decode_split", "kvq_decode_combine", "kvq_decode_attention",
           "kvq_decode_attention_noalloc", "kvq_select_static_channels", "kvq_dequantize", "kvq_status_string",
           "kvq_last_cuda_error", "kvq_cuda_error_name", "kvq_version")


def lib() -> ctypes.CDLL:
    """Load libkvq.so (built by __graft_entry__.build() / sub_byte_quantized_kvq_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise KVQError(-1, f"CUDA library not built: {LIB_PATH} is missing")
            L = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            pcfg, pcache = ctypes.POINTER(kvq_config), ctypes.POINTER(kvq_cache)
            sig = {
                "kvq_block_bytes": (I, [pcfg, I, ctypes.POINTER(S)]),
                "kvq_cache_bytes": (I, [pcfg, ctypes.POINTER(S), ctypes.POINTER(S), ctypes.POINTER(S)]),
                "kvq_quantize_append": (I, [pcfg, pcache, P, P, I, I, P, P]),
                "kvq_project_append": (I, [pcfg, pcache, P, I, P, P, I, P, P, P]),
                "kvq_decode_workspace_bytes": (I, [pcfg, I, I, I, ctypes.POINTER(S)]),
                "kvq_decode_num_splits": (I, [pcfg, I, I, ctypes.POINTER(I)]),
                "kvq_decode_split": (I, [pcfg, pcache, P, I, ctypes.c_float, I, I, P, S, P]),
                "kvq_decode_combine": (I, [pcfg, I, I, I, P, S, P, I, P]),
                "kvq_decode_attention": (I, [pcfg, pcache, P, I, ctypes.c_float, I, I, P, I, P, S, P]),
                "kvq_decode_attention_noalloc": (I, [pcfg, pcache, P, I, ctypes.c_float, I, I, P, I, P]),
                "kvq_select_static_channels": (I, [pcfg, P, P, I, I, P, P]),
                "kvq_dequantize": (I, [pcfg, pcache, I, I, I, I, I, P, P]),
                "kvq_status_string": (ctypes.c_char_p, [I]),
                "kvq_last_cuda_error": (I, []),
                "kvq_cuda_error_name": (ctypes.c_char_p, [I]),
                "kvq_version": (ctypes.c_char_p, []),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != KVQ_OK:
        raise KVQError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


def kvq_version() -> str:
    return lib().kvq_version().decode()


class QuantizedKVCache:
    """Device buffers of one paged, quantized cache (allocated with torch)."""

    def __init__(self, fmt: int, num_seqs: int, num_kv_heads: int, head_dim: int, pages_per_seq_max: int,
                 num_pages: int, num_tier_pages: int = 0, sigma: float = 3.0, lloyd_iters: int = 16,
                 page_table: torch.Tensor | None = None, device="cuda", static_channels: int = 0,
                 decode_math: int = KVQ_DECODE_AUTO):
        """static_channels (KVQ_FMT_CB2_STATIC): fp16 channels per (kv head, K|V);
        fill `static_mask` ([Hkv, 2, n]) before the first append, e.g. with
        kvq_select_static_channels.  decode_math: KVQ_DECODE_* (cfg.decode_math
        may be changed between calls)."""
        self.cfg = kvq_config(num_seqs, num_kv_heads, head_dim, pages_per_seq_max, num_pages, num_tier_pages, fmt,
                              lloyd_iters, sigma, static_channels, decode_math)
        pb, tb, sb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().kvq_cache_bytes(ctypes.byref(self.cfg), ctypes.byref(pb), ctypes.byref(tb), ctypes.byref(sb)),
               "kvq_cache_bytes")
        self.device = torch.device(device)
        self.pool = torch.zeros(pb.value, dtype=torch.uint8, device=self.device)
        self.tier_pool = torch.zeros(tb.value, dtype=torch.uint8, device=self.device) if tb.value else None
        self.staging = torch.zeros(sb.value // 4, dtype=torch.float32, device=self.device) if sb.value else None
        if page_table is None:
            page_table = torch.arange(num_seqs * pages_per_seq_max, dtype=torch.int64).view(num_seqs, -1) % num_pages
        self.page_table = torch.as_tensor(page_table).to(torch.int32).to(self.device).contiguous()
        self.seq_lens = torch.zeros(num_seqs, dtype=torch.int32, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.static_mask = (torch.zeros((num_kv_heads, 2, static_channels), dtype=torch.uint8, device=self.device)
                            if fmt == KVQ_FMT_CB2_STATIC else None)
        self.c = kvq_cache(self.pool.data_ptr(), self.tier_pool.data_ptr() if self.tier_pool is not None else None,
                           self.page_table.data_ptr(), self.seq_lens.data_ptr(),
                           self.staging.data_ptr() if self.staging is not None else None, self.status.data_ptr(),
                           self.static_mask.data_ptr() if self.static_mask is not None else None)

    @property
    def head_dim(self) -> int:
        return self.cfg.head_dim

    def block_bytes(self, tier: int = 0) -> int:
        return kvq_block_bytes(self.cfg, tier)

    def status_word(self) -> int:
        return int(self.status.item()) & 0xFFFFFFFF


def kvq_block_bytes(cfg: kvq_config, tier: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(lib().kvq_block_bytes(ctypes.byref(cfg), tier, ctypes.byref(n)), "kvq_block_bytes")
    return n.value


def kvq_quantize_append(cache: QuantizedKVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                        t_per_seq: torch.Tensor | None = None, stream=None):
    """k_new, v_new: [num_seqs, t_new, Hkv, D] bf16/f16/f32 on the cache's device."""
    assert k_new.shape == v_new.shape and k_new.dtype == v_new.dtype and k_new.is_contiguous() and v_new.is_contiguous()
    assert k_new.dim() == 4 and k_new.shape[0] == cache.cfg.num_seqs
    if t_per_seq is not None:
        t_per_seq = t_per_seq.to(torch.int32).contiguous()
    _check(lib().kvq_quantize_append(ctypes.byref(cache.cfg), ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new),
                                     _DTYPE[k_new.dtype], k_new.shape[1], _ptr(t_per_seq), _stream(stream)),
           "kvq_quantize_append")


def kvq_project_append(cache: QuantizedKVCache, x: torch.Tensor, w_k: torch.Tensor, w_v: torch.Tensor,
                       t_per_seq: torch.Tensor | None = None, kv_out: torch.Tensor | None = None, stream=None):
    """x: bf16 [num_seqs, t_new, hidden]; w_k, w_v: bf16 [Hkv * D, hidden].  K = x w_k^T and
    V = x w_v^T are projected on the tensor cores and quantized into the cache in one kernel.
    kv_out: optional fp32 [2, num_seqs, t_new, Hkv, D] that receives the projected K and V."""
    cfg = cache.cfg
    assert x.dtype == torch.bfloat16 and w_k.dtype == torch.bfloat16 and w_v.dtype == torch.bfloat16
    assert x.is_contiguous() and w_k.is_contiguous() and w_v.is_contiguous()
    assert x.dim() == 3 and x.shape[0] == cfg.num_seqs
    hidden = x.shape[2]
    assert w_k.shape == (cfg.num_kv_heads * cfg.head_dim, hidden) and w_v.shape == w_k.shape
    if kv_out is not None:
        assert kv_out.dtype == torch.float32 and kv_out.is_contiguous()
        assert kv_out.shape == (2, cfg.num_seqs, x.shape[1], cfg.num_kv_heads, cfg.head_dim)
    if t_per_seq is not None:
        t_per_seq = t_per_seq.to(torch.int32).contiguous()
    _check(lib().kvq_project_append(ctypes.byref(cfg), ctypes.byref(cache.c), _ptr(x), hidden, _ptr(w_k), _ptr(w_v),
                                    x.shape[1], _ptr(t_per_seq), _ptr(kv_out), _stream(stream)),
           "kvq_project_append")


def kvq_decode_num_splits(cache: QuantizedKVCache, num_q_heads: int, max_seq_len: int) -> int:
    n = ctypes.c_int32()
    _check(lib().kvq_decode_num_splits(ctypes.byref(cache.cfg), num_q_heads, max_seq_len, ctypes.byref(n)),
           "kvq_decode_num_splits")
    return n.value


def kvq_decode_workspace_bytes(cache: QuantizedKVCache, num_q_heads: int, max_seq_len: int,
                               num_splits: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(lib().kvq_decode_workspace_bytes(ctypes.byref(cache.cfg), num_q_heads, max_seq_len, num_splits,
                                            ctypes.byref(n)), "kvq_decode_workspace_bytes")
    return n.value


def kvq_decode_attention(cache: QuantizedKVCache, q: torch.Tensor, softmax_scale: float, max_seq_len: int,
                         num_splits: int = 0, out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q: [num_seqs, Hq, D] bf16 -> out [num_seqs, Hq, D] (bf16 or f32)."""
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    Hq = q.shape[1]
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(cache, Hq, max_seq_len, num_splits)
    _check(lib().kvq_decode_attention(ctypes.byref(cache.cfg), ctypes.byref(cache.c), _ptr(q), Hq,
                                      float(softmax_scale), max_seq_len, num_splits, _ptr(out), _DTYPE[out.dtype],
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "kvq_decode_attention")
    return out


def kvq_select_static_channels(cache: QuantizedKVCache, k: torch.Tensor, v: torch.Tensor, stream=None):
    """Fill cache.static_mask from calibration values k, v [t, Hkv, D] (device)."""
    assert k.shape == v.shape and k.dim() == 3 and k.dtype == v.dtype and k.is_contiguous() and v.is_contiguous()
    _check(lib().kvq_select_static_channels(ctypes.byref(cache.cfg), _ptr(k), _ptr(v), _DTYPE[k.dtype], k.shape[0],
                                            _ptr(cache.static_mask), _stream(stream)), "kvq_select_static_channels")
    return cache.static_mask


def alloc_workspace(cache: QuantizedKVCache, num_q_heads: int, max_seq_len: int, num_splits: int = 0) -> torch.Tensor:
    nbytes = kvq_decode_workspace_bytes(cache, num_q_heads, max_seq_len, num_splits)
    # zeroed once: its head holds the fused split merge's arrival counters
    return torch.zeros((nbytes + 15) // 16 * 4, dtype=torch.float32, device=cache.device)


def kvq_decode_split(cache: QuantizedKVCache, q: torch.Tensor, softmax_scale: float, max_seq_len: int,
                     workspace: torch.Tensor, num_splits: int = 0, stream=None):
    """Stage 1 of kvq_decode_attention: split partials into `workspace`."""
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    _check(lib().kvq_decode_split(ctypes.byref(cache.cfg), ctypes.byref(cache.c), _ptr(q), q.shape[1],
                                  float(softmax_scale), max_seq_len, num_splits, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)), "kvq_decode_split")


def kvq_decode_combine(cache: QuantizedKVCache, num_q_heads: int, max_seq_len: int, workspace: torch.Tensor,
                       out: torch.Tensor, num_splits: int = 0, stream=None) -> torch.Tensor:
    """Stage 2 of kvq_decode_attention: merge the split partials into `out`."""
    _check(lib().kvq_decode_combine(ctypes.byref(cache.cfg), num_q_heads, max_seq_len, num_splits, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(out), _DTYPE[out.dtype],
                                    _stream(stream)), "kvq_decode_combine")
    return out


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def kvq_decode_attention_noalloc(cache: QuantizedKVCache, q: torch.Tensor, softmax_scale: float, max_seq_len: int,
                                 num_splits: int = 0, out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                                 stream=None) -> torch.Tensor:
    """kvq_decode_attention without a workspace, for callers that may not
    allocate device memory while they decode (the library's own fixed scratch
    holds the split partials).  `out` should be passed by such callers; it is
    allocated here only as a convenience when omitted.  Concurrent calls on
    different streams share that scratch and must be serialised."""
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    st = lib().kvq_decode_attention_noalloc(ctypes.byref(cache.cfg), ctypes.byref(cache.c), _ptr(q), q.shape[1],
                                            float(softmax_scale), max_seq_len, num_splits, _ptr(out),
                                            _DTYPE[out.dtype], _stream(stream))
    if st == KVQ_ERR_WORKSPACE:
        need = kvq_decode_workspace_bytes(cache, q.shape[1], max_seq_len, num_splits)
        raise KVQError(st, f"kvq_decode_attention_noalloc: split partials need {need} bytes, more than the "
                           f"{NOALLOC_SCRATCH_BYTES}-byte built-in scratch")
    _check(st, "kvq_decode_attention_noalloc")
    return out


def kvq_dequantize(cache: QuantizedKVCache, seq: int, kv_head: int, which: int, tok_begin: int, tok_end: int,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Values tokens [tok_begin, tok_end) of (seq, kv_head, K=0 / V=1) stand for, fp32 [n, D]."""
    if out is None:
        out = torch.empty((max(tok_end - tok_begin, 0), cache.head_dim), dtype=torch.float32, device=cache.device)
    _check(lib().kvq_dequantize(ctypes.byref(cache.cfg), ctypes.byref(cache.c), seq, kv_head, which, tok_begin,
                                tok_end, _ptr(out), _stream(stream)), "kvq_dequantize")
    return out
