"""Helpers for the GPU parity tests: the same seeded inputs go through the CUDA
path (via the C ABI binding) and through the CPU oracle."""
import numpy as np
import torch

import oracle
from sub_byte_quantized_kvq_gb300 import kvq, synth

ORACLE_FMT = {kvq.KVQ_FMT_CB2_STATIC: oracle.FMT_CB2S, kvq.KVQ_FMT_ASYM3_OUTLIER: oracle.FMT_A3,
              kvq.KVQ_FMT_CB2_GROUP4: oracle.FMT_CB2G,
              kvq.KVQ_FMT_INT4_G32: oracle.FMT_INT4, kvq.KVQ_FMT_FP4_E2M1_S16: oracle.FMT_E2M1,
              kvq.KVQ_FMT_CB2_OUTLIER: oracle.FMT_CB2, kvq.KVQ_FMT_TIERED: oracle.FMT_TIERED}


def make_kv(seed, B, T, Hkv, D, dist="normal", n_out=4, factor=8.0, fixed=()):
    w = synth.Workload("t", 0, B, Hkv, Hkv, D, T, dist, n_out, factor, fixed_channels=fixed)
    ks, vs = zip(*[synth.workload_kv(w, seed, b, 0, T) for b in range(B)])
    return torch.stack(ks), torch.stack(vs)


class Pair:
    """A GPU cache and an oracle cache built from identical inputs."""

    def __init__(self, fmt, B, Hkv, D, P, seed=0, shuffled=True, tiers=None, extra_pages=0, sigma=3.0, iters=16,
                 static_channels=0):
        self.fmt, self.B, self.Hkv, self.D, self.P = fmt, B, Hkv, D, P
        if fmt == kvq.KVQ_FMT_CB2_STATIC and static_channels == 0:
            static_channels = -(-D // 100)   # ceil(1% of D)
        self.calibrated = fmt != kvq.KVQ_FMT_CB2_STATIC
        pt, nm, nt = synth.page_table(seed, B, P, shuffled, tiers)
        nm += extra_pages
        self.pt = pt
        self.gpu = kvq.QuantizedKVCache(fmt, B, Hkv, D, P, nm, nt, sigma=sigma, lloyd_iters=iters,
                                        page_table=torch.from_numpy(pt), device="cuda",
                                        static_channels=static_channels)
        st = np.zeros((Hkv, 2, max(static_channels, 1)), np.uint8)
        self.ref = oracle.OracleCache(ORACLE_FMT[fmt], B, Hkv, D, P, nm, nt, sigma=sigma, lloyd_iters=iters,
                                      page_table=pt, static_channels=st)

    def calibrate(self, k, v, dtype=torch.float32):
        """Static channel mask from calibration values k, v (CPU float32 [t, Hkv, D]):
        the GPU selects it, the oracle selects it independently; they must agree."""
        kd, vd = k.to(dtype), v.to(dtype)
        got = kvq.kvq_select_static_channels(self.gpu, kd.cuda().contiguous(), vd.cuda().contiguous())
        torch.cuda.synchronize()
        n = self.gpu.cfg.static_channels
        exp = np.stack([oracle.select_static(kd.float().numpy(), n), oracle.select_static(vd.float().numpy(), n)], 1)
        np.testing.assert_array_equal(got.cpu().numpy(), exp)
        self.ref.static_ch[...] = exp      # the oracle's config points at this array
        self.calibrated = True
        return exp

    def append(self, k, v, t_per_seq=None, dtype=torch.float32):
        """k, v: float32 CPU [B, T, Hkv, D]; the GPU gets them in `dtype`, the
        oracle gets the same values (rounded to `dtype`) as float32."""
        kd, vd = k.to(dtype), v.to(dtype)
        if not self.calibrated:   # static mask from the first append's first tokens of sequence 0
            n = min(k.shape[1], 64)
            self.calibrate(k[0, :n], v[0, :n], dtype)
        tps = None if t_per_seq is None else torch.as_tensor(t_per_seq, dtype=torch.int32)
        kvq.kvq_quantize_append(self.gpu, kd.cuda().contiguous(), vd.cuda().contiguous(),
                                None if tps is None else tps.cuda())
        bad = self.ref.append(kd.float().numpy(), vd.float().numpy(), None if tps is None else tps.numpy())
        return bad

    def project(self, x, w_k, w_v, t_per_seq=None):
        """x: bf16 CPU [B, T, hidden], w_k / w_v: bf16 CPU [Hkv * D, hidden].  The GPU
        projects and appends in one kernel and hands back the fp32 K / V it
        quantized; the oracle appends those same values.  Returns the GPU's
        (k, v) float32 [B, T, Hkv, D] (rows past t_per_seq[b] zero)."""
        B, T = x.shape[0], x.shape[1]
        if not self.calibrated:   # static mask from the oracle's projection of sequence 0's first tokens
            n = min(T, 64)
            kc, vc = oracle.project_kv(x[:1, :n].float().numpy(), w_k.float().numpy(), w_v.float().numpy(),
                                       self.Hkv, self.D)
            self.calibrate(torch.from_numpy(kc[0]).float(), torch.from_numpy(vc[0]).float())
        tps = None if t_per_seq is None else torch.as_tensor(t_per_seq, dtype=torch.int32)
        kv_out = torch.zeros((2, B, T, self.Hkv, self.D), dtype=torch.float32, device="cuda")
        kvq.kvq_project_append(self.gpu, x.cuda().contiguous(), w_k.cuda().contiguous(), w_v.cuda().contiguous(),
                               None if tps is None else tps.cuda(), kv_out)
        torch.cuda.synchronize()
        kv = kv_out.cpu().numpy()
        self.ref.append(kv[0], kv[1], None if tps is None else tps.numpy())
        return kv[0], kv[1]

    def assert_cache_equal(self):
        torch.cuda.synchronize()
        assert self.gpu.status_word() == 0, hex(self.gpu.status_word())
        np.testing.assert_array_equal(self.gpu.seq_lens.cpu().numpy(), self.ref.seq_lens)
        gp = self.gpu.pool.cpu().numpy()
        if not (gp == self.ref.pool).all():
            stride = self.ref.stride
            diff = np.nonzero(gp != self.ref.pool)[0]
            blk = diff[0] // stride
            raise AssertionError(f"pool differs at {len(diff)} bytes; first in block {blk} "
                                 f"(phys {blk // (2 * self.Hkv)}, head {(blk // 2) % self.Hkv}, role {blk % 2}) "
                                 f"offset {diff[0] % stride}: gpu {gp[diff[0]]:#x} oracle {self.ref.pool[diff[0]]:#x}")
        if self.gpu.tier_pool is not None:
            np.testing.assert_array_equal(self.gpu.tier_pool.cpu().numpy(), self.ref.tier_pool[:-1])
        if self.gpu.staging is not None:
            np.testing.assert_array_equal(self.gpu.staging.cpu().numpy(), self.ref.staging.reshape(-1))

    def decode(self, Hq, seed=0, scale=None, max_seq_len=None, num_splits=0, out_dtype=torch.float32):
        scale = self.D ** -0.5 if scale is None else scale
        max_seq_len = int(self.ref.seq_lens.max()) if max_seq_len is None else max_seq_len
        q = synth.queries_bf16(seed, self.B, Hq, self.D, device="cuda")
        out = kvq.kvq_decode_attention(self.gpu, q, scale, max_seq_len, num_splits, out_dtype=out_dtype)
        torch.cuda.synchronize()
        exp = self.ref.decode(q.cpu().view(torch.int16).numpy().view(np.uint16), scale)
        return out.float().cpu().numpy(), exp


def bf16_half_ulp(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def assert_attention_close(got, exp, out_dtype=torch.float32, tol=2e-3):
    """max-abs <= 2e-3 in fp32 output; bf16 output adds half a bf16 ulp of the reference."""
    err = np.abs(got - exp)
    bound = tol + (bf16_half_ulp(exp) if out_dtype == torch.bfloat16 else 0.0)
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} outputs outside tolerance; max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    return float(err.max())
