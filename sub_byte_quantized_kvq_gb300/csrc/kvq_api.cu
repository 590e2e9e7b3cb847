// kvq_api.cu -- the C ABI (include/kvq.h): argument validation, sizing queries,
// the split heuristic, and the debug dequantization kernel.
#include <cmath>

#include "kvq_project.cuh"

namespace kvq {
// The CUDA runtime's error behind the last KVQ_ERR_CUDA this thread saw.
thread_local int g_last_cuda_error = 0;
kvq_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KVQ_OK;
  g_last_cuda_error = (int)e;
  return KVQ_ERR_CUDA;
}

// ----------------------------------------------------------------------------- debug dequantization
// One thread per (token, channel) of the requested range; values are exactly
// the ones the codes stand for (INT4: fmaf(q, S, m); E2M1: e2m1 * scale;
// CB2: fp16 centroid or e4m3 outlier; FP8: e4m3 * scale in fp32; staging tail: as stored).
__device__ __forceinline__ float dq_e4m3(uint32_t b) {
  uint32_t d;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(d) : "r"(b & 0xFFu));
  return __half2float(__ushort_as_half((unsigned short)(d & 0xFFFFu)));
}
__device__ __forceinline__ float dq_e2m1(uint32_t nib) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  return (nib & 8u) ? -mag[nib & 7u] : mag[nib & 7u];
}
__device__ __forceinline__ float dq_f16(uint32_t bits) {
  return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}

struct DequantArgs {
  const uint8_t* pool;
  const uint8_t* tier_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const float* staging;
  uint32_t* status;
  float* out;
  int Hkv, D, ppsm, num_pages, num_tier_pages, fmt, seq, head, role, t0, t1;
};

// The value an outlier side-list (CB2, ASYM3) gives (t, c), else v.
__device__ __forceinline__ float side_list_value(const uint8_t* hdr, int D, int t, int c, float v) {
  const int n_ch = min((int)hdr[0], D);  // a corrupt side-list never reads past its block
  for (int i = 0; i < n_ch; ++i) {
    const uint8_t* rec = hdr + 4 + 20 * i;
    const uint32_t tm = rec[2] | (rec[3] << 8);
    if (rec[0] == c && (tm >> t & 1u)) v = dq_e4m3(rec[4 + t]);
  }
  return v;
}

__global__ void dequantize_kernel(const DequantArgs a) {
  const int D = a.D, NS = D / 16;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)(a.t1 - a.t0) * D) return;
  const int pos = a.t0 + (int)(idx / D), c = (int)(idx % D);
  const int t = pos % kPage, pg = pos / kPage;
  const int L = a.seq_lens[a.seq];
  const bool group = a.fmt == KVQ_FMT_CB2_GROUP4;
  const bool paged = a.fmt == KVQ_FMT_CB2_OUTLIER || a.fmt == KVQ_FMT_TIERED || a.fmt == KVQ_FMT_CB2_STATIC ||
                     a.fmt == KVQ_FMT_ASYM3_OUTLIER || group;
  // tokens not yet in a block: the partial last page, or for the group format the partial last group
  const int unit = group ? kPage * kGroupPages : kPage;
  float v = 0.f;
  if (pos >= L || pg >= a.ppsm) {
    v = 0.f;
  } else if (paged && (pos / unit + 1) * unit > L) {
    v = a.staging[((((size_t)a.seq * a.Hkv + a.head) * 2 + a.role) * unit + pos % unit) * D + c];
  } else if (group) {
    // codes of this page, codebook of the group's first page
    const int32_t* row = a.page_table + (size_t)a.seq * a.ppsm;
    const uint32_t u = (uint32_t)row[pg], u0 = (uint32_t)row[(pg / kGroupPages) * kGroupPages];
    if ((u >> 31) || (u0 >> 31) || u >= (uint32_t)a.num_pages || u0 >= (uint32_t)a.num_pages) {
      atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
      a.out[idx] = 0.f;
      return;
    }
    const size_t stride = (size_t)block_stride(kBlkCb2g, D);
    const uint8_t* blk = a.pool + (((size_t)u * a.Hkv + a.head) * 2 + a.role) * stride;
    const uint8_t* cbk = a.pool + (((size_t)u0 * a.Hkv + a.head) * 2 + a.role) * stride;
    const FragPos p = frag_pos(a.role, t, c);
    const uint8_t* cw = blk + cb2g_code_off(D) + 2 * NS * p.lane + 2 * p.step;
    const uint32_t q = ((cw[0] | (cw[1] << 8)) >> (4 * (p.slot & 3) + 2 * (p.slot >> 2))) & 3u;
    const uint8_t* cb = cbk + 8 * cb2_slot(a.role, c);
    v = dq_f16(cb[q] | (cb[4 + q] << 8));
    v = side_list_value(blk + cb2_out_off(D), D, t, c, v);
  } else {
    const uint32_t u = (uint32_t)a.page_table[(size_t)a.seq * a.ppsm + pg], phys = u & 0x7FFFFFFFu;
    const bool tier = (u >> 31) != 0;
    const bool ok = tier ? (a.fmt == KVQ_FMT_TIERED && phys < (uint32_t)a.num_tier_pages) : phys < (uint32_t)a.num_pages;
    if (!ok) {
      atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
      a.out[idx] = 0.f;
      return;
    }
    const int bf = tier ? kBlkFp8 : (a.fmt == KVQ_FMT_TIERED ? kBlkCb2 : a.fmt);
    const size_t stride = (size_t)block_stride(bf, D);
    const uint8_t* blk = (tier ? a.tier_pool : a.pool) + (((size_t)phys * a.Hkv + a.head) * 2 + a.role) * stride;
    const FragPos p = frag_pos(a.role, t, c);
    if (bf == kBlkInt4) {
      const uint32_t q = (blk[4 * NS * p.lane + 4 * p.step + p.slot / 2] >> (4 * (p.slot & 1))) & 0xFu;
      const uint8_t* sz = blk + int4_sz_off(D) + 4 * (t * (D / 32) + c / 32);
      v = fmaf((float)q, dq_f16(sz[0] | (sz[1] << 8)), dq_f16(sz[2] | (sz[3] << 8)));
      const int cap = int4_cap(D), cnt = blk[int4_cnt_off(D) + t];
      for (int i = 0; i < cnt && i < cap; ++i)
        if (blk[int4_ch_off(D) + t * cap + i] == c) {
          const uint8_t* vp = blk + int4_val_off(D) + 2 * (t * cap + i);
          v = dq_f16(vp[0] | (vp[1] << 8));
        }
    } else if (bf == kBlkE2m1) {
      const uint32_t q = (blk[4 * NS * p.lane + 4 * p.step + p.slot / 2] >> (4 * (p.slot & 1))) & 0xFu;
      v = dq_e2m1(q) * dq_e4m3(blk[e2m1_sc_off(D) + 16 * (c / 16) + t]);
    } else if (bf == kBlkCb2 || bf == kBlkCb2s) {
      const uint32_t w = blk[2 * NS * p.lane + 2 * p.step] | (blk[2 * NS * p.lane + 2 * p.step + 1] << 8);
      const uint32_t q = (w >> (4 * (p.slot & 3) + 2 * (p.slot >> 2))) & 3u;
      const uint8_t* cb = blk + cb2_cb_off(D) + 8 * cb2_slot(a.role, c);
      v = dq_f16(cb[q] | (cb[4 + q] << 8));
      if (bf == kBlkCb2s) {   // static fp16 channels
        const uint8_t* hdr = blk + cb2s_hdr_off(D);
        const int n_s = min((int)hdr[0], kMaxStatic);
        for (int i = 0; i < n_s; ++i)
          if (hdr[1 + i] == c) {
            const uint8_t* vp = blk + cb2s_val_off(D) + 32 * i + 2 * t;
            v = dq_f16(vp[0] | (vp[1] << 8));
          }
      } else {
        v = side_list_value(blk + cb2_out_off(D), D, t, c, v);
      }
    } else if (bf == kBlkA3) {
      uint32_t vx, vy;
      memcpy(&vx, blk + 4 * (p.lane * (NS / 2) + p.step / 2), 4);
      memcpy(&vy, blk + a3_hi_off(D) + 4 * (p.lane * (NS / 4) + p.step / 4), 4);
      const int bx = 8 * (p.step % 2) + 16 * (p.slot % 2) + 2 * (p.slot / 2);
      const int by = 4 * (p.step % 4) + 16 * (p.slot % 2) + p.slot / 2;
      const uint32_t q = ((vx >> bx) & 3u) | (((vy >> by) & 1u) << 2);
      const int r = a3_rho(a.role, c);
      const uint8_t* sp = blk + a3_s_off(D) + 2 * r;
      const uint8_t* mp = blk + a3_m_off(D) + 2 * r;
      // fp16(q * S + m): one rounding of the exact value (fp16 fused multiply-add)
      v = __half2float(__hfma(__float2half_rn((float)q), __ushort_as_half((unsigned short)(sp[0] | (sp[1] << 8))),
                              __ushort_as_half((unsigned short)(mp[0] | (mp[1] << 8)))));
      v = side_list_value(blk + a3_out_off(D), D, t, c, v);
    } else {
      float s;
      memcpy(&s, blk + fp8_sc_off(D), 4);
      v = __fmul_rn(dq_e4m3(blk[8 * NS * p.lane + 8 * p.step + p.slot]), s);
    }
  }
  a.out[idx] = v;
}

cudaError_t dequantize_launch(const kvq_config& cfg, const kvq_cache& cache, int seq, int head, int role, int t0,
                              int t1, float* out, cudaStream_t st) {
  DequantArgs a;
  a.pool = static_cast<const uint8_t*>(cache.pool);
  a.tier_pool = static_cast<const uint8_t*>(cache.tier_pool);
  a.page_table = cache.page_table;
  a.seq_lens = cache.seq_lens;
  a.staging = cache.staging;
  a.status = cache.status;
  a.out = out;
  a.Hkv = cfg.num_kv_heads;
  a.D = cfg.head_dim;
  a.ppsm = cfg.pages_per_seq_max;
  a.num_pages = cfg.num_pages;
  a.num_tier_pages = cfg.num_tier_pages;
  a.fmt = cfg.format;
  a.seq = seq;
  a.head = head;
  a.role = role;
  a.t0 = t0;
  a.t1 = t1;
  const long long n = (long long)(t1 - t0) * cfg.head_dim;
  if (n <= 0) return cudaSuccess;
  dequantize_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- validation
static bool cfg_ok(const kvq_config* c) {
  if (!c) return false;
  if (c->num_seqs <= 0 || c->num_kv_heads <= 0 || c->pages_per_seq_max <= 0 || c->num_pages <= 0) return false;
  if (c->format < KVQ_FMT_INT4_G32 || c->format > KVQ_FMT_CB2_GROUP4) return false;
  if (c->format == KVQ_FMT_CB2_STATIC && (c->static_channels < 1 || c->static_channels > kMaxStatic)) return false;
  if (c->num_tier_pages < 0 || (c->format != KVQ_FMT_TIERED && c->num_tier_pages != 0)) return false;
  if (!(c->sigma >= 3.0) || !std::isfinite(c->sigma)) return false;
  if (c->lloyd_iters < 1 || c->lloyd_iters > 64) return false;
  if (c->decode_math < KVQ_DECODE_AUTO || c->decode_math > KVQ_DECODE_CUDA_CORES) return false;
  if (c->num_seqs > 65535 || c->num_kv_heads > 32767) return false;  // grid dimensions
  return true;
}
static bool dim_supported(const kvq_config* c) { return c->head_dim == 64 || c->head_dim == 128; }
static bool paged_format(int f) {
  return f == KVQ_FMT_CB2_OUTLIER || f == KVQ_FMT_TIERED || f == KVQ_FMT_CB2_STATIC || f == KVQ_FMT_ASYM3_OUTLIER ||
         f == KVQ_FMT_CB2_GROUP4;
}
static bool cache_ok(const kvq_config* c, const kvq_cache* k) {
  if (!k || !k->pool || !k->page_table || !k->seq_lens || !k->status) return false;
  if (paged_format(c->format) && !k->staging) return false;
  if (c->format == KVQ_FMT_CB2_STATIC && !k->static_mask) return false;
  if (c->format == KVQ_FMT_TIERED && c->num_tier_pages > 0 && !k->tier_pool) return false;
  return true;
}
static int main_blk(const kvq_config* c) { return c->format == KVQ_FMT_TIERED ? kBlkCb2 : c->format; }

static int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Splits per (sequence, kv head): the smallest count whose grid fills at least
// 90% of its last wave of resident CTA slots (so no nearly empty final wave),
// keeping at least 2 pages per warp in each split; otherwise the count with the
// best last-wave fill.
// Workspace layout: the fused merge's arrival counters u32 [B][Hkv] first
// (padded to 256 bytes), then part_o fp32 [B][Hq][S][D] and part_ml float2
// [B][Hq][S].  The counters' place depends only on the cache's (sequence, kv
// head) count, so calls of any shape (splits, query heads, length) can share
// a workspace: each call's last CTAs leave the counters at zero.
static size_t partials_offset(const kvq_config* c) {
  return ((size_t)c->num_seqs * c->num_kv_heads * sizeof(uint32_t) + 255) / 256 * 256;
}
static size_t partials_bytes(const kvq_config* c, int num_q_heads, int S) {
  const size_t rows = (size_t)c->num_seqs * num_q_heads * S;
  return rows * c->head_dim * sizeof(float) + rows * sizeof(float2);
}

// The decode math a call runs: CUDA cores only where that path exists
// (CB2, G <= 4); AUTO takes the tensor cores.
static int decode_math(const kvq_config* c, int G) {
  const bool cc_ok = c->format == KVQ_FMT_CB2_OUTLIER && G <= 4;
  return cc_ok && c->decode_math == KVQ_DECODE_CUDA_CORES ? KVQ_DECODE_CUDA_CORES : KVQ_DECODE_TENSOR_CORES;
}

static int auto_splits(const kvq_config* c, int G, int max_seq_len) {
  const long long pages = (max_seq_len + kPage - 1) / kPage;
  const long long units = (long long)c->num_seqs * c->num_kv_heads;
  const int per_sm = decode_ctas_per_sm(c->format, c->head_dim, G, decode_math(c, G));
  const long long slots = (long long)num_sms() * (per_sm > 0 ? per_sm : 1);
  long long smax = pages / (2 * kWarpsPerCta);
  if (smax < 1) smax = 1;
  if (smax > 256) smax = 256;
  long long best = 1;
  double best_fill = -1.0;
  for (long long s = 1; s <= smax; ++s) {
    const long long ctas = units * s;
    const long long waves = (ctas + slots - 1) / slots;
    const double fill = (double)ctas / (double)(waves * slots);
    if (fill >= 0.9) return (int)s;
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = s;
    }
  }
  return (int)best;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

kvq_status kvq_block_bytes(const kvq_config* cfg, int32_t tier, size_t* bytes) {
  if (!cfg_ok(cfg) || !bytes || (tier != 0 && tier != 1)) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg)) return KVQ_ERR_UNSUPPORTED;
  *bytes = (size_t)block_stride(tier ? kBlkFp8 : main_blk(cfg), cfg->head_dim);
  return KVQ_OK;
}

kvq_status kvq_cache_bytes(const kvq_config* cfg, size_t* pool_bytes, size_t* tier_pool_bytes, size_t* staging_bytes) {
  if (!cfg_ok(cfg) || !pool_bytes || !tier_pool_bytes || !staging_bytes) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg)) return KVQ_ERR_UNSUPPORTED;
  const size_t per_page = (size_t)cfg->num_kv_heads * 2;
  *pool_bytes = (size_t)cfg->num_pages * per_page * block_stride(main_blk(cfg), cfg->head_dim);
  *tier_pool_bytes = (size_t)cfg->num_tier_pages * per_page * block_stride(kBlkFp8, cfg->head_dim);
  const int rows = cfg->format == KVQ_FMT_CB2_GROUP4 ? kPage * kGroupPages : kPage;
  *staging_bytes = paged_format(cfg->format) ? (size_t)cfg->num_seqs * cfg->num_kv_heads * 2 * rows * cfg->head_dim * sizeof(float) : 0;
  return KVQ_OK;
}

static void fill_append_args(const kvq_config* cfg, const kvq_cache* cache, int32_t t_new, const int32_t* t_per_seq,
                             AppendArgs& a) {
  a.pool = static_cast<uint8_t*>(cache->pool);
  a.tier_pool = static_cast<uint8_t*>(cache->tier_pool);
  a.page_table = cache->page_table;
  a.seq_lens = cache->seq_lens;
  a.staging = cache->staging;
  a.status = cache->status;
  a.kv[0] = a.kv[1] = nullptr;
  a.in_dtype = KVQ_F32;
  a.t_new = t_new;
  a.t_per_seq = t_per_seq;
  a.B = cfg->num_seqs;
  a.Hkv = cfg->num_kv_heads;
  a.ppsm = cfg->pages_per_seq_max;
  a.num_pages = cfg->num_pages;
  a.num_tier_pages = cfg->num_tier_pages;
  a.fmt = cfg->format;
  a.iters = cfg->lloyd_iters;
  a.sigma = cfg->sigma;
  a.static_mask = cache->static_mask;
  a.n_static = cfg->format == KVQ_FMT_CB2_STATIC ? cfg->static_channels : 0;
}

kvq_status kvq_quantize_append(const kvq_config* cfg, const kvq_cache* cache, const void* k_new, const void* v_new,
                               kvq_dtype in_dtype, int32_t t_new, const int32_t* t_per_seq, void* stream) {
  if (!cfg_ok(cfg) || !cache_ok(cfg, cache) || !k_new || !v_new || t_new < 0) return KVQ_ERR_INVALID_ARG;
  if (in_dtype != KVQ_BF16 && in_dtype != KVQ_F16 && in_dtype != KVQ_F32) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg)) return KVQ_ERR_UNSUPPORTED;
  if (t_new == 0) return KVQ_OK;
  if ((long long)t_new > (long long)cfg->pages_per_seq_max * kPage) return KVQ_ERR_CAPACITY;
  AppendArgs a;
  fill_append_args(cfg, cache, t_new, t_per_seq, a);
  a.kv[0] = k_new;
  a.kv[1] = v_new;
  a.in_dtype = in_dtype;
  return cuda_status(append_launch(a, cfg->head_dim, static_cast<cudaStream_t>(stream)));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status kvq_project_append(const kvq_config* cfg, const kvq_cache* cache, const void* x, int32_t hidden,
                              const void* w_k, const void* w_v, int32_t t_new, const int32_t* t_per_seq,
                              float* kv_out, void* stream) {
  if (!cfg_ok(cfg) || !cache_ok(cfg, cache) || !x || !w_k || !w_v || t_new < 0) return KVQ_ERR_INVALID_ARG;
  if (hidden <= 0 || hidden % 32 || !aligned16(x) || !aligned16(w_k) || !aligned16(w_v) || !aligned16(kv_out))
    return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg)) return KVQ_ERR_UNSUPPORTED;
  if (t_new == 0) return KVQ_OK;
  if ((long long)t_new > (long long)cfg->pages_per_seq_max * kPage) return KVQ_ERR_CAPACITY;
  if ((long long)cfg->num_seqs * t_new >= (1ll << 31)) return KVQ_ERR_UNSUPPORTED;   // TMA row coordinates are int32
  if (t_new > 65535 * 128 - 1024) return KVQ_ERR_UNSUPPORTED;   // 128-row tiles in the grid's y dimension
  ProjArgs p;
  fill_append_args(cfg, cache, t_new, t_per_seq, p.a);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w[0] = static_cast<const __nv_bfloat16*>(w_k);
  p.w[1] = static_cast<const __nv_bfloat16*>(w_v);
  p.hidden = hidden;
  p.kv_out = kv_out;
  return cuda_status(project_append_launch(p, cfg->head_dim, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_num_splits(const kvq_config* cfg, int32_t num_q_heads, int32_t max_seq_len,
                                 int32_t* num_splits) {
  if (!cfg_ok(cfg) || !num_splits || num_q_heads <= 0 || max_seq_len < 0) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % cfg->num_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg) || num_q_heads / cfg->num_kv_heads > 16) return KVQ_ERR_UNSUPPORTED;
  *num_splits = auto_splits(cfg, num_q_heads / cfg->num_kv_heads, max_seq_len);
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t num_q_heads, int32_t max_seq_len,
                                      int32_t num_splits, size_t* bytes) {
  if (!cfg_ok(cfg) || !bytes || num_q_heads <= 0 || max_seq_len < 0 || num_splits < 0) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % cfg->num_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg) || num_q_heads / cfg->num_kv_heads > 16) return KVQ_ERR_UNSUPPORTED;
  int S = num_splits;
  if (S == 0) S = auto_splits(cfg, num_q_heads / cfg->num_kv_heads, max_seq_len);
  *bytes = partials_offset(cfg) + partials_bytes(cfg, num_q_heads, S);
  return KVQ_OK;
}

}  // extern "C"

namespace kvq {
// Validate a decode request and fill the split kernel's arguments (partials
// only: out == nullptr).
static kvq_status decode_prepare(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t num_q_heads,
                                 float softmax_scale, int32_t max_seq_len, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, DecodeArgs& a) {
  if (!cfg_ok(cfg) || !cache_ok(cfg, cache) || !q || !workspace) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cfg->num_kv_heads || max_seq_len < 0 || num_splits < 0)
    return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 16) return KVQ_ERR_INVALID_ARG;
  const int G = num_q_heads / cfg->num_kv_heads;
  if (!dim_supported(cfg) || G > 16) return KVQ_ERR_UNSUPPORTED;
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_bytes(cfg, num_q_heads, max_seq_len, num_splits, &need);
  if (st != KVQ_OK) return st;
  if (workspace_bytes < need) return KVQ_ERR_WORKSPACE;
  const int S = num_splits ? num_splits : auto_splits(cfg, G, max_seq_len);
  if (S > kMaxSplits) return KVQ_ERR_CAPACITY;
  const int cap_len = cfg->pages_per_seq_max * kPage;
  const int len = max_seq_len < cap_len ? max_seq_len : cap_len;
  const int pages = (len + kPage - 1) / kPage;
  a.pool = static_cast<const uint8_t*>(cache->pool);
  a.tier_pool = static_cast<const uint8_t*>(cache->tier_pool);
  a.page_table = cache->page_table;
  a.seq_lens = cache->seq_lens;
  a.staging = cache->staging;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + partials_offset(cfg));
  a.part_ml = reinterpret_cast<float2*>(a.part_o + (size_t)cfg->num_seqs * num_q_heads * S * cfg->head_dim);
  a.status = cache->status;
  a.B = cfg->num_seqs;
  a.Hkv = cfg->num_kv_heads;
  a.Hq = num_q_heads;
  a.G = G;
  a.ppsm = cfg->pages_per_seq_max;
  a.num_pages = cfg->num_pages;
  a.num_tier_pages = cfg->num_tier_pages;
  a.S = S;
  a.pps = pages > 0 ? (pages + S - 1) / S : 1;
  if (cfg->format == KVQ_FMT_CB2_GROUP4) a.pps = (a.pps + kGroupPages - 1) / kGroupPages * kGroupPages;   // whole groups
  a.max_seq_len = len;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = nullptr;
  a.out_dtype = KVQ_F32;
  a.arrivals = static_cast<uint32_t*>(workspace);
  a.static_mask = cache->static_mask;
  a.n_static = cfg->format == KVQ_FMT_CB2_STATIC ? cfg->static_channels : 0;
  a.math = decode_math(cfg, G);
  return KVQ_OK;
}
}  // namespace kvq

extern "C" {

kvq_status kvq_decode_split(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t num_q_heads,
                            float softmax_scale, int32_t max_seq_len, int32_t num_splits, void* workspace,
                            size_t workspace_bytes, void* stream) {
  DecodeArgs a;
  kvq_status st = decode_prepare(cfg, cache, q, num_q_heads, softmax_scale, max_seq_len, num_splits, workspace,
                                 workspace_bytes, a);
  if (st != KVQ_OK) return st;
  return cuda_status(decode_split_launch(a, cfg->format, cfg->head_dim, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_combine(const kvq_config* cfg, int32_t num_q_heads, int32_t max_seq_len, int32_t num_splits,
                              const void* workspace, size_t workspace_bytes, void* out, kvq_dtype out_dtype,
                              void* stream) {
  if (!cfg_ok(cfg) || !workspace || !out || num_q_heads <= 0 || num_q_heads % cfg->num_kv_heads || max_seq_len < 0 ||
      num_splits < 0)
    return KVQ_ERR_INVALID_ARG;
  if (out_dtype != KVQ_BF16 && out_dtype != KVQ_F32) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 16) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg) || num_q_heads / cfg->num_kv_heads > 16) return KVQ_ERR_UNSUPPORTED;
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_bytes(cfg, num_q_heads, max_seq_len, num_splits, &need);
  if (st != KVQ_OK) return st;
  if (workspace_bytes < need) return KVQ_ERR_WORKSPACE;
  const int S = num_splits ? num_splits : auto_splits(cfg, num_q_heads / cfg->num_kv_heads, max_seq_len);
  const float* part_o = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + partials_offset(cfg));
  const float2* part_ml = reinterpret_cast<const float2*>(part_o + (size_t)cfg->num_seqs * num_q_heads * S * cfg->head_dim);
  if (S > kMaxSplits) return KVQ_ERR_CAPACITY;
  return cuda_status(decode_combine_launch(part_o, part_ml, cfg->num_seqs, cfg->num_kv_heads, num_q_heads, S,
                                           cfg->head_dim, out, out_dtype, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t num_q_heads,
                                float softmax_scale, int32_t max_seq_len, int32_t num_splits, void* out,
                                kvq_dtype out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (!out || (out_dtype != KVQ_BF16 && out_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  DecodeArgs a;
  kvq_status st = decode_prepare(cfg, cache, q, num_q_heads, softmax_scale, max_seq_len, num_splits, workspace,
                                 workspace_bytes, a);
  if (st != KVQ_OK) return st;
  a.out = out;   // one launch: the split kernel's last CTA per (sequence, kv head) merges the splits
  a.out_dtype = out_dtype;
  return cuda_status(decode_split_launch(a, cfg->format, cfg->head_dim, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace kvq {
kvq_status decode_attention_zeroing_counters(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                             int32_t num_q_heads, float softmax_scale, int32_t max_seq_len,
                                             int32_t num_splits, void* out, kvq_dtype out_dtype, void* workspace,
                                             size_t workspace_bytes, cudaStream_t st) {
  if (!out || (out_dtype != KVQ_BF16 && out_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  DecodeArgs a;
  kvq_status s = decode_prepare(cfg, cache, q, num_q_heads, softmax_scale, max_seq_len, num_splits, workspace,
                                workspace_bytes, a);
  if (s != KVQ_OK) return s;
  a.out = out;
  a.out_dtype = out_dtype;
  const kvq_status zs = cuda_status(cudaMemsetAsync(a.arrivals, 0, (size_t)a.B * a.Hkv * sizeof(uint32_t), st));
  if (zs != KVQ_OK) return zs;
  return cuda_status(decode_split_launch(a, cfg->format, cfg->head_dim, st));
}
}  // namespace kvq

extern "C" {

kvq_status kvq_select_static_channels(const kvq_config* cfg, const void* k, const void* v, kvq_dtype in_dtype,
                                      int32_t t, uint8_t* mask, void* stream) {
  if (!cfg_ok(cfg) || cfg->format != KVQ_FMT_CB2_STATIC || !k || !v || !mask || t < 1) return KVQ_ERR_INVALID_ARG;
  if (in_dtype != KVQ_BF16 && in_dtype != KVQ_F16 && in_dtype != KVQ_F32) return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg)) return KVQ_ERR_UNSUPPORTED;
  return cuda_status(select_static_launch(k, v, in_dtype, t, cfg->num_kv_heads, cfg->head_dim, cfg->static_channels,
                                          mask, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_cache* cache, int32_t seq, int32_t kv_head, int32_t which,
                          int32_t tok_begin, int32_t tok_end, float* out, void* stream) {
  if (!cfg_ok(cfg) || !cache_ok(cfg, cache) || !out) return KVQ_ERR_INVALID_ARG;
  if (seq < 0 || seq >= cfg->num_seqs || kv_head < 0 || kv_head >= cfg->num_kv_heads || (which != 0 && which != 1))
    return KVQ_ERR_INVALID_ARG;
  if (tok_begin < 0 || tok_end < tok_begin || (long long)tok_end > (long long)cfg->pages_per_seq_max * kPage)
    return KVQ_ERR_INVALID_ARG;
  if (!dim_supported(cfg)) return KVQ_ERR_UNSUPPORTED;
  return cuda_status(dequantize_launch(*cfg, *cache, seq, kv_head, which, tok_begin, tok_end, out,
                                       static_cast<cudaStream_t>(stream)));
}

int32_t kvq_last_cuda_error(void) { return g_last_cuda_error; }

const char* kvq_cuda_error_name(int32_t error) { return cudaGetErrorName(static_cast<cudaError_t>(error)); }

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CAPACITY: return "size exceeds the layout's capacity";
    case KVQ_ERR_CUDA: return "CUDA runtime error";
    case KVQ_ERR_TIMEOUT: return "timed out";
  }
  return "unknown status";
}

const char* kvq_version(void) { return "0.1.0"; }

}  // extern "C"
