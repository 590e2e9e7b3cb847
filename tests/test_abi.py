"""The C-ABI library builds, loads and exports every function include/kvq.h
declares; host-side validation and sizing work without a GPU (no compute call
is made here)."""
import ctypes
import os
import re
import shutil

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def kvq():
    from sub_byte_quantized_kvq_gb300 import build
    build.build()
    from sub_byte_quantized_kvq_gb300 import kvq as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvq):
    names = declared_functions()
    assert len(names) >= 9
    L = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(L, n), f"{n} declared in kvq.h but not exported"
    assert set(kvq.EXPORTS) == set(names)


def _cfg(kvq, fmt=2, D=128, **kw):
    c = kvq.kvq_config(4, 8, D, 16, 64, 0, fmt, 16, 3.0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_block_sizes_agree_with_oracle_layout(kvq):
    for fmt, blk in [(0, oracle.BLK_INT4), (1, oracle.BLK_E2M1), (2, oracle.BLK_CB2)]:
        for D in (64, 128):
            assert kvq.kvq_block_bytes(_cfg(kvq, fmt, D)) == oracle.block_stride(blk, D)
    for D in (64, 128):
        c = _cfg(kvq, 3, D, num_tier_pages=4)
        assert kvq.kvq_block_bytes(c, 0) == oracle.block_stride(oracle.BLK_CB2, D)
        assert kvq.kvq_block_bytes(c, 1) == oracle.block_stride(oracle.BLK_FP8, D)


def test_cache_bytes(kvq):
    L = kvq.lib()
    c = _cfg(kvq, 3, 128, num_tier_pages=5)
    p, t, s = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert L.kvq_cache_bytes(ctypes.byref(c), ctypes.byref(p), ctypes.byref(t), ctypes.byref(s)) == 0
    assert p.value == 64 * 8 * 2 * 4224 and t.value == 5 * 8 * 2 * 2176 and s.value == 4 * 8 * 2 * 16 * 128 * 4
    c = _cfg(kvq, 1, 64)
    assert L.kvq_cache_bytes(ctypes.byref(c), ctypes.byref(p), ctypes.byref(t), ctypes.byref(s)) == 0
    assert s.value == 0 and t.value == 0


def test_invalid_arguments_rejected_before_launch(kvq):
    L = kvq.lib()
    n = ctypes.c_size_t()
    assert L.kvq_block_bytes(None, 0, ctypes.byref(n)) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_block_bytes(ctypes.byref(_cfg(kvq, 7)), 0, ctypes.byref(n)) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_block_bytes(ctypes.byref(_cfg(kvq, 2, 96)), 0, ctypes.byref(n)) == kvq.KVQ_ERR_UNSUPPORTED
    assert L.kvq_block_bytes(ctypes.byref(_cfg(kvq, 2, sigma=2.0)), 0, ctypes.byref(n)) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_block_bytes(ctypes.byref(_cfg(kvq, 2, num_tier_pages=3)), 0, ctypes.byref(n)) == kvq.KVQ_ERR_INVALID_ARG
    for bad in (-1, 3):
        assert L.kvq_block_bytes(ctypes.byref(_cfg(kvq, 2, decode_math=bad)), 0, ctypes.byref(n)) == \
            kvq.KVQ_ERR_INVALID_ARG
    for ok in (kvq.KVQ_DECODE_AUTO, kvq.KVQ_DECODE_TENSOR_CORES, kvq.KVQ_DECODE_CUDA_CORES):
        assert L.kvq_block_bytes(ctypes.byref(_cfg(kvq, 0, decode_math=ok)), 0, ctypes.byref(n)) == kvq.KVQ_OK
    cache = kvq.kvq_cache()   # all-null cache
    c = _cfg(kvq)
    assert L.kvq_quantize_append(ctypes.byref(c), ctypes.byref(cache), None, None, 0, 1, None, None) == \
        kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_project_append(ctypes.byref(c), ctypes.byref(cache), None, 64, None, None, 1, None, None, None) == \
        kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(ctypes.byref(c), ctypes.byref(cache), None, 32, ctypes.c_float(0.1), 16, 0, None, 0,
                                  None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequantize(ctypes.byref(c), ctypes.byref(cache), 0, 0, 0, 0, 1, None, None) == kvq.KVQ_ERR_INVALID_ARG
    # workspace size with an explicit split count is pure host arithmetic
    assert L.kvq_decode_workspace_bytes(ctypes.byref(c), 32, 4096, 8, ctypes.byref(n)) == 0
    assert n.value == 256 + 4 * 32 * 8 * (128 * 4 + 8)   # one arrival counter per (seq, kv head), padded; partials
    assert L.kvq_decode_workspace_bytes(ctypes.byref(c), 30, 4096, 8, ctypes.byref(n)) == kvq.KVQ_ERR_INVALID_ARG


def test_projection_size_limits_before_launch(kvq):
    """kvq_project_append refuses sizes its launch cannot express before it
    touches any buffer (the pointers here are never dereferenced)."""
    L = kvq.lib()
    fake = ctypes.c_void_p(1 << 20)   # 16-byte aligned, never read
    c = _cfg(kvq, 0, 128, num_seqs=1, pages_per_seq_max=600000, num_pages=600000)
    cache = kvq.kvq_cache(fake, None, fake, fake, None, fake, None)   # INT4: no staging
    args = lambda t: (ctypes.byref(c), ctypes.byref(cache), fake, 4096, fake, fake, t, None, None, None)
    assert L.kvq_project_append(*args(65535 * 128 - 1023)) == kvq.KVQ_ERR_UNSUPPORTED   # grid rows
    assert L.kvq_project_append(*args(600000 * 16 + 1)) == kvq.KVQ_ERR_CAPACITY
    c.num_seqs = 300
    assert L.kvq_project_append(*args(7200000)) == kvq.KVQ_ERR_UNSUPPORTED   # 2^31 TMA rows
    assert L.kvq_project_append(*args(0)) == kvq.KVQ_OK                      # nothing to do
    assert L.kvq_project_append(ctypes.byref(c), ctypes.byref(cache), fake, 4010, fake, fake, 16, None, None,
                                None) == kvq.KVQ_ERR_INVALID_ARG              # hidden not a multiple of 32


def test_status_strings_and_version(kvq):
    for s in range(7):
        assert kvq.kvq_status_string(s)
    assert kvq.kvq_status_string(99) == "unknown status"
    assert re.fullmatch(r"\d+\.\d+\.\d+", kvq.kvq_version())


def test_cuda_error_accessors(kvq):
    """kvq_last_cuda_error is per thread (0 on a thread that has seen no
    KVQ_ERR_CUDA) and kvq_cuda_error_name maps runtime codes to their names;
    neither needs a GPU."""
    import threading
    L = kvq.lib()
    seen = []
    t = threading.Thread(target=lambda: seen.append(L.kvq_last_cuda_error()))
    t.start()
    t.join()
    assert seen == [0]
    assert L.kvq_cuda_error_name(0).decode() == "cudaSuccess"
    assert L.kvq_cuda_error_name(1).decode() == "cudaErrorInvalidValue"
    assert L.kvq_cuda_error_name(2).decode() == "cudaErrorMemoryAllocation"
