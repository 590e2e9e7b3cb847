// kvq_quantize.cu -- quantize-on-append into the paged cache.  The quantizer's
// decisions (outlier tests, Lloyd-Max, INT4 codes) are taken in binary32 in a
// fixed order; the file is compiled with --fmad=false so no multiply-add is
// fused and codes are bit-identical to the CPU reference.
//
// "The Sub-10ms Barrier: Fusing Sparse MoE Routing with FP4 KV-Cache
// Quantization", section 2 ("Outlier Isolation and Block-wise Quantization"):
// asymmetric INT4 per 32-group, S = (max - min) / (2^b - 1), and FP4 E2M1;
// scales are computed as tokens are inserted.
// "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression",
// Paradigm 2: outliers beyond sigma standard deviations (mean / unbiased std
// along head_dim) kept in FP8 E4M3; the rest mapped to a 4-centroid codebook
// fitted by k-means (Lloyd-Max in one dimension) from a linspace start,
// assignment by nearest centroid with the first index winning ties.
// "Hierarchical Token Gating and Tiered KV-Cache Paging", section 2: FP8 pages
// for the tier named by the page table.
//
// One append = up to three launches on the caller's stream:
//   1. quantize: per-token formats write every new token into its block;
//      page formats quantize each page the append completes (from fp32
//      staging + the new tokens);
//   2. (page formats) copy the new tokens of the final partial page into
//      staging -- after 1, which may still be reading the old staging rows;
//   3. advance seq_lens and raise status bits -- after 1 and 2, which read it.
#include "kvq_internal.cuh"

namespace kvq {

enum { kSeqOk = 0, kSeqNothing = 1, kSeqCapacity = 2, kSeqBadPage = 3 };

// Decide, identically in every launch, whether sequence b's append proceeds.
__device__ int seq_append_state(const AppendArgs& a, int b, int& start, int& n) {
  start = a.seq_lens[b];
  n = a.t_per_seq ? a.t_per_seq[b] : a.t_new;
  if (n <= 0) return kSeqNothing;
  if (n > a.t_new || start < 0 || (long long)start + n > (long long)a.ppsm * kPage) return kSeqCapacity;
  // a completed CB2 group rewrites all of its pages, including earlier ones
  const int first = a.fmt == KVQ_FMT_CB2_GROUP4 ? (start / (kPage * kGroupPages)) * kGroupPages : start / kPage;
  for (int pg = first; pg <= (start + n - 1) / kPage; ++pg) {
    const uint32_t u = (uint32_t)a.page_table[(size_t)b * a.ppsm + pg], phys = u & 0x7FFFFFFFu;
    const bool ok = (u >> 31) ? (a.fmt == KVQ_FMT_TIERED && phys < (uint32_t)a.num_tier_pages)
                              : phys < (uint32_t)a.num_pages;
    if (!ok) return kSeqBadPage;
  }
  return kSeqOk;
}

__device__ __forceinline__ float load_in(const AppendArgs& a, int role, int b, int t, int h, int c, int D) {
  const size_t i = (((size_t)b * a.t_new + t) * a.Hkv + h) * D + c;
  if (a.in_dtype == KVQ_F32) return static_cast<const float*>(a.kv[role])[i];
  if (a.in_dtype == KVQ_F16) return __half2float(static_cast<const __half*>(a.kv[role])[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(a.kv[role])[i]);
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(x));
  return (uint8_t)(r & 0xFFu);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
  uint32_t d;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(d) : "r"((uint32_t)v));
  return __half2float(__ushort_as_half((unsigned short)(d & 0xFFFFu)));
}
__device__ __forceinline__ uint8_t f32_to_e2m1(float x) {
  uint32_t r;
  asm("{ .reg .b8 t; .reg .b16 w; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; mov.b16 w, {t, t}; cvt.u32.u16 %0, w; }"
      : "=r"(r)
      : "f"(0.f), "f"(x));
  return (uint8_t)(r & 0xFu);
}
__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Outlier mask of one vector (binary32, ascending order): |x - mu| > sigma * s,
// s the unbiased standard deviation; at most kmax kept (lowest indices).
__device__ int outlier_mask(const float* x, int n, int stride, float sigma, int kmax, uint8_t* mask, int mstride) {
  float sum = 0.f;
  for (int i = 0; i < n; ++i) sum += x[i * stride];
  const float mu = __fdiv_rn(sum, (float)n);
  float ss = 0.f;
  for (int i = 0; i < n; ++i) {
    const float d = x[i * stride] - mu;
    ss += d * d;
  }
  const float thr = sigma * __fsqrt_rn(__fdiv_rn(ss, (float)(n - 1)));
  int k = 0;
  for (int i = 0; i < n; ++i) {
    int out = fabsf(x[i * stride] - mu) > thr;
    if (out && k >= kmax) out = 0;
    mask[i * mstride] = (uint8_t)out;
    k += out;
  }
  return k;
}

__device__ __forceinline__ int nearest4(float v, const float* c) {
  int best = 0;
  float bd = fabsf(v - c[0]);
  for (int j = 1; j < 4; ++j) {
    const float d = fabsf(v - c[j]);
    if (d < bd) { bd = d; best = j; }
  }
  return best;
}

// Lloyd-Max 4-centroid fit of v[0..n) (n <= NMAX) in binary32; fp16 centroids and codes.
template <int NMAX>
__device__ void lloyd4(const float* v, int n, int iters, uint16_t* c16, uint8_t* codes) {
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  if (n > 0) {
    float mn = v[0], mx = v[0];
    for (int i = 1; i < n; ++i) { mn = v[i] < mn ? v[i] : mn; mx = v[i] > mx ? v[i] : mx; }
    const float h = __fdiv_rn(mx - mn, 3.0f);
    c[0] = mn; c[1] = mn + h; c[2] = mn + 2.0f * h; c[3] = mx;
    uint8_t a[NMAX], prev[NMAX];
    bool have_prev = false;
    for (int it = 0; it < iters; ++it) {
      bool same = have_prev;
      for (int i = 0; i < n; ++i) {
        a[i] = (uint8_t)nearest4(v[i], c);
        same = same && a[i] == prev[i];
      }
      if (same) break;
      for (int j = 0; j < 4; ++j) {
        float s = 0.f;
        int cnt = 0;
        for (int i = 0; i < n; ++i)
          if (a[i] == j) { s += v[i]; ++cnt; }
        if (cnt > 0) c[j] = __fdiv_rn(s, (float)cnt);
      }
      for (int i = 0; i < n; ++i) prev[i] = a[i];
      have_prev = true;
    }
  }
  float cf[4];
  for (int j = 0; j < 4; ++j) { c16[j] = f32_to_f16_bits(c[j]); cf[j] = f16_bits_to_f32(c16[j]); }
  for (int i = 0; i < n; ++i) codes[i] = (uint8_t)nearest4(v[i], cf);
}

// Element (t, c) held by fragment (lane, step, slot) -- the inverse of frag_pos.
__device__ __forceinline__ void frag_inverse(int role, int lane, int s, int k, int& t, int& c) {
  if (role == 0) {
    t = (lane >> 2) + 8 * ((k >> 1) & 1);
    c = 16 * s + 2 * (lane & 3) + (k & 1) + 8 * (k >> 2);
  } else {
    c = 16 * s + (lane >> 2) + 8 * ((k >> 1) & 1);
    t = 2 * (lane & 3) + (k & 1) + 8 * (k >> 2);
  }
}

// ----------------------------------------------------------------------------- per-token formats
// INT4 group-32 quantization of token slot t by one warp (lane g < D/32 owns group g).
template <int D>
__device__ void quantize_token_int4(const float* x, int t, uint8_t (*codes)[D], uint8_t* blk, double sigma, int lane) {
  constexpr int NG = D / 32, CAP = int4_cap(D);
  uint8_t mask[32];
  int cnt = 0;
  if (lane < NG) {
    const float* xg = x + 32 * lane;
    outlier_mask(xg, 32, 1, (float)sigma, kmax_outliers(32), mask, 1);
    bool have = false;
    float mn = 0.f, mx = 0.f;
    for (int i = 0; i < 32; ++i) {
      if (mask[i]) continue;
      const float v = xg[i];
      if (!have || v < mn) mn = v;
      if (!have || v > mx) mx = v;
      have = true;
    }
    const uint16_t S16 = have ? f32_to_f16_bits(__fdiv_rn(mx - mn, 15.0f)) : 0;
    const uint16_t m16 = have ? f32_to_f16_bits(mn) : 0;
    const float S = f16_bits_to_f32(S16), m = f16_bits_to_f32(m16);
    for (int i = 0; i < 32; ++i) {
      uint8_t q = 0;
      if (mask[i]) {
        ++cnt;
      } else if (S != 0.f) {
        float r = rintf(__fdiv_rn(xg[i] - m, S));
        r = r < 0.f ? 0.f : (r > 15.f ? 15.f : r);
        q = (uint8_t)r;
      }
      codes[t][32 * lane + i] = q;
    }
    uint8_t* sz = blk + int4_sz_off(D) + 4 * (t * NG + lane);
    *reinterpret_cast<uint16_t*>(sz) = S16;
    *reinterpret_cast<uint16_t*>(sz + 2) = m16;
  }
  // entries of group g go after those of groups < g (ascending channel order)
  int off = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, off, d);
    if (lane >= d) off += y;
  }
  const int total = __shfl_sync(0xffffffffu, off, NG - 1);
  off -= cnt;
  uint8_t* chans = blk + int4_ch_off(D) + t * CAP;
  uint16_t* vals = reinterpret_cast<uint16_t*>(blk + int4_val_off(D)) + t * CAP;
  if (lane < NG) {
    for (int i = 0; i < 32; ++i)
      if (mask[i]) {
        chans[off] = (uint8_t)(32 * lane + i);
        vals[off] = __half_as_ushort(__float2half_rn(x[32 * lane + i]));
        ++off;
      }
  }
  for (int i = total + lane; i < CAP; i += 32) {
    chans[i] = 0;
    vals[i] = 0;
  }
  if (lane == 0) blk[int4_cnt_off(D) + t] = (uint8_t)total;
}

// E2M1 quantization of token slot t by one warp (lane s < D/16 owns 16 channels).
template <int D>
__device__ void quantize_token_e2m1(const float* x, int t, uint8_t (*codes)[D], uint8_t* blk, int lane) {
  if (lane >= D / 16) return;
  const float* xs = x + 16 * lane;
  float amax = 0.f;
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(xs[i]));
  const uint8_t s8 = f32_to_e4m3(__fdiv_rn(amax, 6.0f));
  const float sc = e4m3_to_f32(s8);
  for (int i = 0; i < 16; ++i) codes[t][16 * lane + i] = sc != 0.f ? f32_to_e2m1(__fdiv_rn(xs[i], sc)) : 0;
  blk[e2m1_sc_off(D) + 16 * lane + t] = s8;
}

template <int BF, int D>
__global__ void __launch_bounds__(256) append_token_kernel(const AppendArgs a) {
  constexpr int kStride = block_stride(BF, D), NS = D / 16;
  __shared__ __align__(16) uint8_t blk[kStride];
  __shared__ uint8_t codes[16][D];
  __shared__ float xs[16][D];
  const int j = blockIdx.x, h = blockIdx.y >> 1, role = blockIdx.y & 1, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, pg = start / kPage + j;
  if (pg * kPage >= end) return;
  const int lo = max(start, pg * kPage), hi = min(end, pg * kPage + kPage);
  const uint32_t phys = (uint32_t)a.page_table[(size_t)b * a.ppsm + pg] & 0x7FFFFFFFu;
  uint8_t* gblk = a.pool + (((size_t)phys * a.Hkv + h) * 2 + role) * kStride;

  for (int i = tid; i < kStride / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(blk)[i] = reinterpret_cast<const uint4*>(gblk)[i];
  for (int i = tid; i < (hi - lo) * D; i += blockDim.x) {
    const int tt = i / D, c = i - tt * D;
    xs[(lo % kPage) + tt][c] = load_in(a, role, b, lo + tt - start, h, c, D);
  }
  __syncthreads();
  for (int i = tid; i < 32 * NS * 8; i += blockDim.x) {
    const int ln = i / (NS * 8), s = (i / 8) % NS, k = i % 8;
    int t, c;
    frag_inverse(role, ln, s, k, t, c);
    codes[t][c] = (blk[4 * NS * ln + 4 * s + k / 2] >> (4 * (k & 1))) & 0xF;
  }
  __syncthreads();
  for (int tt = warp; tt < hi - lo; tt += nwarps) {
    const int t = (lo % kPage) + tt;
    if (BF == kBlkInt4) quantize_token_int4<D>(xs[t], t, codes, blk, a.sigma, lane);
    else quantize_token_e2m1<D>(xs[t], t, codes, blk, lane);
  }
  __syncthreads();
  for (int i = tid; i < 32 * NS; i += blockDim.x) {
    const int ln = i / NS, s = i % NS;
    uint32_t word = 0;
    for (int k = 0; k < 8; ++k) {
      int t, c;
      frag_inverse(role, ln, s, k, t, c);
      word |= (uint32_t)codes[t][c] << (4 * k);
    }
    *reinterpret_cast<uint32_t*>(blk + 4 * NS * ln + 4 * s) = word;
  }
  __syncthreads();
  for (int i = tid; i < kStride / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gblk)[i] = reinterpret_cast<const uint4*>(blk)[i];
}

// ----------------------------------------------------------------------------- page formats
// Outlier side-list of one page (CB2, ASYM3, CB2 group) from its mask and
// values [16][D], built by one warp: lane l owns channels [l*D/32, (l+1)*D/32);
// one 20-byte record {channel, 0, token mask, 16 e4m3 values} per channel
// with an outlier, channels ascending, after {n_ch, total}.  Zeros come from
// the block clear.
template <int D>
__device__ void build_side_list(const uint8_t (*mask)[D], const float (*xs)[D], uint8_t* hdr, int lane) {
  constexpr int CPL = D / 32;
  uint32_t tm[CPL];
  int nch = 0, nval = 0;
  for (int k = 0; k < CPL; ++k) {
    const int c = lane * CPL + k;
    uint32_t m = 0;
    for (int t = 0; t < 16; ++t) m |= (uint32_t)mask[t][c] << t;
    tm[k] = m;
    nch += m != 0;
    nval += __popc(m);
  }
  int ich = nch, ival = nval;
  for (int d = 1; d < 32; d <<= 1) {
    const int a1 = __shfl_up_sync(0xffffffffu, ich, d), a2 = __shfl_up_sync(0xffffffffu, ival, d);
    if (lane >= d) { ich += a1; ival += a2; }
  }
  const int tot_ch = __shfl_sync(0xffffffffu, ich, 31), tot_val = __shfl_sync(0xffffffffu, ival, 31);
  int ci = ich - nch;
  for (int k = 0; k < CPL; ++k) {
    if (!tm[k]) continue;
    const int c = lane * CPL + k;
    uint8_t* rec = hdr + 4 + 20 * ci;
    rec[0] = (uint8_t)c;
    rec[1] = 0;
    rec[2] = (uint8_t)(tm[k] & 0xFF);
    rec[3] = (uint8_t)(tm[k] >> 8);
    for (int t = 0; t < 16; ++t)
      if (tm[k] >> t & 1u) rec[4 + t] = f32_to_e4m3(xs[t][c]);
    ++ci;
  }
  if (lane == 0) {
    hdr[0] = (uint8_t)tot_ch;
    hdr[1] = (uint8_t)tot_val;
  }
}

// 2-bit codes [16][D] -> the block's lane-major code words (CB2 layout).
template <int D>
__device__ __forceinline__ void pack_cb2_codes(const uint8_t (&codes)[16][D], uint8_t* blk, int role, int tid) {
  constexpr int NS = D / 16;
  for (int i = tid; i < 32 * NS; i += blockDim.x) {
    const int ln = i / NS, s = i % NS;
    uint32_t word = 0;
    for (int k = 0; k < 8; ++k) {
      int t, c;
      frag_inverse(role, ln, s, k, t, c);
      word |= (uint32_t)codes[t][c] << (4 * (k & 3) + 2 * (k >> 2));
    }
    *reinterpret_cast<uint16_t*>(blk + 2 * NS * ln + 2 * s) = (uint16_t)word;
  }
}

// 3-bit codes [16][D] -> the block's two ASYM3 code planes (include/kvq.h):
// one thread per (lane, 4-step group) builds one high-bit word and two
// low-bit words.
template <int D>
__device__ __forceinline__ void pack_a3_codes(const uint8_t (&codes)[16][D], uint8_t* blk, int role, int tid) {
  constexpr int NS = D / 16, NG = NS / 4;
  for (int i = tid; i < 32 * NG; i += blockDim.x) {
    const int ln = i / NG, grp = i % NG;
    uint32_t lo[2] = {0u, 0u}, hi = 0u;
    for (int ss = 0; ss < 4; ++ss) {
      const int s = 4 * grp + ss;
      for (int k = 0; k < 8; ++k) {
        int t, c;
        frag_inverse(role, ln, s, k, t, c);
        const uint32_t q = codes[t][c];
        lo[ss >> 1] |= (q & 3u) << (8 * (s % 2) + 16 * (k % 2) + 2 * (k / 2));
        hi |= ((q >> 2) & 1u) << (4 * (s % 4) + 16 * (k % 2) + k / 2);
      }
    }
    uint32_t* xw = reinterpret_cast<uint32_t*>(blk) + ln * (NS / 2) + 2 * grp;
    xw[0] = lo[0];
    xw[1] = lo[1];
    reinterpret_cast<uint32_t*>(blk + a3_hi_off(D))[ln * NG + grp] = hi;
  }
}

template <int D>
__global__ void __launch_bounds__(128) append_page_kernel(const AppendArgs a) {
  constexpr int NS = D / 16;
  constexpr int kCb2 = block_stride(kBlkCb2, D), kFp8 = block_stride(kBlkFp8, D);
  constexpr int kBlk = kCb2 > kFp8 ? kCb2 : kFp8;
  __shared__ float xs[16][D];
  __shared__ uint8_t mask[16][D];
  __shared__ uint8_t codes[16][D];
  __shared__ __align__(16) uint8_t blk[kBlk];
  __shared__ int cnt[16];
  __shared__ float red[4];
  const int j = blockIdx.x, h = blockIdx.y >> 1, role = blockIdx.y & 1, b = blockIdx.z;
  const int tid = threadIdx.x;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, pg = start / kPage + j;
  if (pg * kPage + kPage > end) return;  // only pages this append completes
  const uint32_t u = (uint32_t)a.page_table[(size_t)b * a.ppsm + pg], phys = u & 0x7FFFFFFFu;
  const bool tier = (u >> 31) != 0;
  const bool stat = a.fmt == KVQ_FMT_CB2_STATIC;
  const int stride = tier ? kFp8
                   : stat ? block_stride(kBlkCb2s, D)
                   : a.fmt == KVQ_FMT_ASYM3_OUTLIER ? block_stride(kBlkA3, D) : kCb2;
  uint8_t* gblk = (tier ? a.tier_pool : a.pool) + (((size_t)phys * a.Hkv + h) * 2 + role) * stride;
  const float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * kPage * D;

  for (int i = tid; i < 16 * D; i += blockDim.x) {
    const int t = i / D, c = i - t * D, pos = pg * kPage + t;
    xs[t][c] = pos < start ? stg[t * D + c] : load_in(a, role, b, pos - start, h, c, D);
  }
  for (int i = tid; i < kBlk / 16; i += blockDim.x) reinterpret_cast<uint4*>(blk)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  if (tier) {
    float amax = 0.f;
    for (int i = tid; i < 16 * D; i += blockDim.x) amax = fmaxf(amax, fabsf(xs[i / D][i % D]));
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float s = __fdiv_rn(amax, 448.0f);
    for (int i = tid; i < 16 * D; i += blockDim.x) {
      const int t = i / D, c = i - t * D;
      const FragPos p = frag_pos(role, t, c);
      blk[8 * NS * p.lane + 8 * p.step + p.slot] = s != 0.f ? f32_to_e4m3(__fdiv_rn(xs[t][c], s)) : 0;
    }
    if (tid == 0) *reinterpret_cast<float*>(blk + fp8_sc_off(D)) = s;
  } else if (stat) {
    // static fp16 channels (all tokens); every other channel: codebook over all 16 values
    const uint8_t* chs = a.static_mask + ((size_t)h * 2 + role) * a.n_static;
    if (tid < D) mask[0][tid] = 0;
    __syncthreads();
    if (tid < a.n_static) mask[0][chs[tid] & (D - 1)] = 1;
    __syncthreads();
    if (tid < D) {
      const int c = tid;
      if (mask[0][c]) {
        for (int t = 0; t < 16; ++t) codes[t][c] = 0;   // all-zero centroids from the block clear
      } else {
        float v[16];
        uint8_t cc[16];
        uint16_t c16[4];
        for (int t = 0; t < 16; ++t) v[t] = xs[t][c];
        lloyd4<16>(v, 16, a.iters, c16, cc);
        for (int t = 0; t < 16; ++t) codes[t][c] = cc[t];
        uint8_t* cbp = blk + cb2_cb_off(D) + 8 * cb2_slot(role, c);
        for (int jj = 0; jj < 4; ++jj) {
          cbp[jj] = (uint8_t)(c16[jj] & 0xFF);
          cbp[4 + jj] = (uint8_t)(c16[jj] >> 8);
        }
      }
    }
    if (tid < a.n_static) {
      const int c = chs[tid] & (D - 1);
      blk[cb2s_hdr_off(D) + 1 + tid] = (uint8_t)c;
      for (int t = 0; t < 16; ++t)
        *reinterpret_cast<uint16_t*>(blk + cb2s_val_off(D) + 32 * tid + 2 * t) = f32_to_f16_bits(xs[t][c]);
    }
    if (tid == 0) blk[cb2s_hdr_off(D)] = (uint8_t)a.n_static;
    __syncthreads();
    pack_cb2_codes<D>(codes, blk, role, tid);
  } else {
    // CB2 or ASYM3: per-token outliers, then per channel a codebook (CB2) or an
    // 8-level affine grid (ASYM3) over the non-outliers
    const bool a3 = a.fmt == KVQ_FMT_ASYM3_OUTLIER;
    if (tid < 16) cnt[tid] = outlier_mask(&xs[tid][0], D, 1, (float)a.sigma, kmax_outliers(D), &mask[tid][0], 1);
    __syncthreads();
    if (tid < D && a3) {
      const int c = tid;
      bool have = false;
      float mn = 0.f, mx = 0.f;
      for (int t = 0; t < 16; ++t) {
        if (mask[t][c]) continue;
        const float v = xs[t][c];
        if (!have || v < mn) mn = v;
        if (!have || v > mx) mx = v;
        have = true;
      }
      const uint16_t S16 = have ? f32_to_f16_bits(__fdiv_rn(mx - mn, 7.0f)) : 0;
      const uint16_t m16 = have ? f32_to_f16_bits(mn) : 0;
      const float S = f16_bits_to_f32(S16), m = f16_bits_to_f32(m16);
      for (int t = 0; t < 16; ++t) {
        uint8_t q = 0;
        if (!mask[t][c] && S != 0.f) {
          float r = rintf(__fdiv_rn(xs[t][c] - m, S));
          r = fminf(fmaxf(r, 0.f), 7.f);
          q = (uint8_t)r;
        }
        codes[t][c] = q;
      }
      const int r = a3_rho(role, c);
      *reinterpret_cast<uint16_t*>(blk + a3_s_off(D) + 2 * r) = S16;
      *reinterpret_cast<uint16_t*>(blk + a3_m_off(D) + 2 * r) = m16;
    } else if (tid < D) {
      const int c = tid;
      float v[16];
      uint8_t cc[16];
      uint16_t c16[4];
      int nv = 0;
      for (int t = 0; t < 16; ++t)
        if (!mask[t][c]) v[nv++] = xs[t][c];
      lloyd4<16>(v, nv, a.iters, c16, cc);
      nv = 0;
      for (int t = 0; t < 16; ++t) codes[t][c] = mask[t][c] ? 0 : cc[nv++];
      uint8_t* cbp = blk + cb2_cb_off(D) + 8 * cb2_slot(role, c);
      for (int jj = 0; jj < 4; ++jj) {
        cbp[jj] = (uint8_t)(c16[jj] & 0xFF);
        cbp[4 + jj] = (uint8_t)(c16[jj] >> 8);
      }
    }
    if (tid < 32) build_side_list<D>(mask, xs, blk + (a3 ? a3_out_off(D) : cb2_out_off(D)), tid);
    __syncthreads();
    if (a3) pack_a3_codes<D>(codes, blk, role, tid);
    else pack_cb2_codes<D>(codes, blk, role, tid);
  }
  __syncthreads();
  for (int i = tid; i < stride / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gblk)[i] = reinterpret_cast<const uint4*>(blk)[i];
}

// CB2 group format: each group of 4 pages (64 tokens) this append completes,
// from fp32 staging + the new tokens: outliers per token, one codebook per
// channel over the group's non-outliers in token order (in the group's first
// page), codes and side-list per page.  One CTA per (group, kv head x role,
// sequence); dynamic shared memory holds the values, masks, codes and the
// four blocks.
template <int D>
__global__ void __launch_bounds__(128) append_group_kernel(const AppendArgs a) {
  constexpr int GT = kPage * kGroupPages, kStride = block_stride(kBlkCb2g, D);
  extern __shared__ __align__(16) uint8_t gsm[];
  float(*xs)[D] = reinterpret_cast<float(*)[D]>(gsm);
  uint8_t(*mask)[D] = reinterpret_cast<uint8_t(*)[D]>(gsm + GT * D * 4);
  uint8_t(*codes)[D] = reinterpret_cast<uint8_t(*)[D]>(gsm + GT * D * 5);
  uint8_t* blk = gsm + GT * D * 6;   // 4 blocks of kStride bytes
  const int j = blockIdx.x, h = blockIdx.y >> 1, role = blockIdx.y & 1, b = blockIdx.z;
  const int tid = threadIdx.x;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, gr = start / GT + j;
  if (gr * GT + GT > end) return;  // only groups this append completes
  const float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * GT * D;
  for (int i = tid; i < GT * D; i += blockDim.x) {
    const int t = i / D, c = i - t * D, pos = gr * GT + t;
    xs[t][c] = pos < start ? stg[t * D + c] : load_in(a, role, b, pos - start, h, c, D);
  }
  for (int i = tid; i < kGroupPages * kStride / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(blk)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid < GT) outlier_mask(&xs[tid][0], D, 1, (float)a.sigma, kmax_outliers(D), &mask[tid][0], 1);
  __syncthreads();
  if (tid < D) {
    const int c = tid;
    float v[GT];
    uint8_t cc[GT];
    uint16_t c16[4];
    int nv = 0;
    for (int t = 0; t < GT; ++t)
      if (!mask[t][c]) v[nv++] = xs[t][c];
    lloyd4<GT>(v, nv, a.iters, c16, cc);
    nv = 0;
    for (int t = 0; t < GT; ++t) codes[t][c] = mask[t][c] ? 0 : cc[nv++];
    uint8_t* cbp = blk + 8 * cb2_slot(role, c);   // the codebook sits at the start of the group's first block
    for (int jj = 0; jj < 4; ++jj) {
      cbp[jj] = (uint8_t)(c16[jj] & 0xFF);
      cbp[4 + jj] = (uint8_t)(c16[jj] >> 8);
    }
  }
  // one warp per page builds its side-list
  {
    const int w = tid >> 5;
    build_side_list<D>(mask + 16 * w, xs + 16 * w, blk + w * kStride + cb2_out_off(D), tid & 31);
  }
  __syncthreads();
  for (int p = 0; p < kGroupPages; ++p)
    pack_cb2_codes<D>(*reinterpret_cast<const uint8_t(*)[16][D]>(&codes[16 * p][0]), blk + p * kStride + cb2g_code_off(D),
                      role, tid);
  __syncthreads();
  for (int p = 0; p < kGroupPages; ++p) {
    const uint32_t u = (uint32_t)a.page_table[(size_t)b * a.ppsm + gr * kGroupPages + p];
    uint8_t* gblk = a.pool + (((size_t)(u & 0x7FFFFFFFu) * a.Hkv + h) * 2 + role) * kStride;
    for (int i = tid; i < kStride / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(gblk)[i] = reinterpret_cast<const uint4*>(blk + p * kStride)[i];
  }
}

template <int D>
constexpr size_t group_smem_bytes() {
  return (size_t)kPage * kGroupPages * D * 6 + (size_t)kGroupPages * block_stride(kBlkCb2g, D);
}

// New tokens of the final partial page (the final partial group for the CB2
// group format) -> fp32 staging (after the page / group kernel).
__global__ void __launch_bounds__(256) append_stage_kernel(const AppendArgs a, int D) {
  const int h = blockIdx.x >> 1, role = blockIdx.x & 1, b = blockIdx.y;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int rows = a.fmt == KVQ_FMT_CB2_GROUP4 ? kPage * kGroupPages : kPage;
  const int end = start + n;
  if (end % rows == 0) return;
  const int lo = max(start, (end / rows) * rows);
  float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * rows * D;
  for (int i = threadIdx.x; i < (end - lo) * D; i += blockDim.x) {
    const int tt = i / D, c = i - tt * D, pos = lo + tt;
    stg[(pos % rows) * D + c] = load_in(a, role, b, pos - start, h, c, D);
  }
}

// Advance seq_lens and report skipped sequences (after every other launch read them).
__global__ void append_finish_kernel(const AppendArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.B) return;
  int start, n;
  const int st = seq_append_state(a, b, start, n);
  if (st == kSeqOk) a.seq_lens[b] = start + n;
  else if (st == kSeqCapacity) atomicOr(a.status, KVQ_STATUS_CAPACITY);
  else if (st == kSeqBadPage) atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
}

// Static channel mask of CB2_STATIC: one CTA per (kv head, K|V); thread c
// takes max_t |x[t][h][c]|, then n_s argmax passes (ties to the lower channel)
// and an ascending write-out.
__global__ void __launch_bounds__(128) select_static_kernel(const void* k, const void* v, int in_dtype, int t, int Hkv,
                                                            int D, int n_s, uint8_t* mask) {
  __shared__ float score[128];
  __shared__ uint8_t taken[128];
  const int h = blockIdx.x >> 1, role = blockIdx.x & 1, c = threadIdx.x;
  const void* x = role ? v : k;
  if (c < D) {
    float m = 0.f;
    for (int i = 0; i < t; ++i) {
      const size_t idx = ((size_t)i * Hkv + h) * D + c;
      const float val = in_dtype == KVQ_F32   ? static_cast<const float*>(x)[idx]
                        : in_dtype == KVQ_F16 ? __half2float(static_cast<const __half*>(x)[idx])
                                              : __bfloat162float(static_cast<const __nv_bfloat16*>(x)[idx]);
      m = fmaxf(m, fabsf(val));
    }
    score[c] = m;
    taken[c] = 0;
  }
  __syncthreads();
  if (c == 0) {
    for (int k2 = 0; k2 < n_s; ++k2) {
      int best = -1;
      for (int j = 0; j < D; ++j)
        if (!taken[j] && (best < 0 || score[j] > score[best])) best = j;
      taken[best] = 1;
    }
    uint8_t* out = mask + ((size_t)h * 2 + role) * n_s;
    int n = 0;
    for (int j = 0; j < D; ++j)
      if (taken[j]) out[n++] = (uint8_t)j;
  }
}

cudaError_t select_static_launch(const void* k, const void* v, int in_dtype, int t, int Hkv, int D, int n_s,
                                 uint8_t* mask, cudaStream_t st) {
  select_static_kernel<<<Hkv * 2, 128, 0, st>>>(k, v, in_dtype, t, Hkv, D, n_s, mask);
  return cudaGetLastError();
}

template <int D>
static cudaError_t append_launch_d(const AppendArgs& a, cudaStream_t st) {
  const int pages_max = (a.t_new + kPage - 1) / kPage + 1;
  const dim3 grid(pages_max, a.Hkv * 2, a.B);
  if (a.fmt == KVQ_FMT_INT4_G32) append_token_kernel<kBlkInt4, D><<<grid, 256, 0, st>>>(a);
  else if (a.fmt == KVQ_FMT_FP4_E2M1_S16) append_token_kernel<kBlkE2m1, D><<<grid, 256, 0, st>>>(a);
  else if (a.fmt == KVQ_FMT_CB2_GROUP4) {
    constexpr size_t smem = group_smem_bytes<D>();
    if (smem > 48 * 1024) {
      const cudaError_t e =
          cudaFuncSetAttribute(append_group_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    const int groups_max = a.t_new / (kPage * kGroupPages) + 2;
    append_group_kernel<D><<<dim3(groups_max, a.Hkv * 2, a.B), 128, smem, st>>>(a);
    append_stage_kernel<<<dim3(a.Hkv * 2, a.B), 256, 0, st>>>(a, D);
  } else {
    append_page_kernel<D><<<grid, 128, 0, st>>>(a);
    append_stage_kernel<<<dim3(a.Hkv * 2, a.B), 256, 0, st>>>(a, D);
  }
  append_finish_kernel<<<(a.B + 127) / 128, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t append_launch(const AppendArgs& a, int D, cudaStream_t st) {
  return D == 64 ? append_launch_d<64>(a, st) : append_launch_d<128>(a, st);
}

}  // namespace kvq
