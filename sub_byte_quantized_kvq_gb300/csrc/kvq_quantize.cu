// kvq_quantize.cu -- quantize-on-append into the paged cache.  The quantizer
// is defined in fp64 (statistics, Lloyd-Max fit, scales and codes, each result
// rounded once to its stored format).  Every decision is first taken in
// binary32 together with a bound on how far that arithmetic can be from the
// fp64 one; where the bound does not separate the two sides of the decision
// (a value within rounding of a threshold, a Lloyd cell boundary or a
// rounding midpoint) the unit is recomputed in fp64 in the definition's own
// order, so codes are bit-identical to the fp64 definition while fp64 runs
// only on those rare units.  Compiled with --fmad=false: no multiply-add is
// fused in either precision.
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
// One append = two launches on the caller's stream:
//   1. quantize: per-token formats write every new token into its block;
//      page formats quantize each page (group) the append completes, from
//      fp32 staging + the new tokens, and the CTA of the append's first page
//      (the only one that reads staged rows) then stages the new tokens of
//      the final partial page;
//   2. advance seq_lens and raise status bits -- after 1, which reads them.
//
// The K/V projection fused with the append (kvq_project_append) is here too:
// a tcgen05 tile kernel for prefill chunks and a thread-block-cluster split-K
// kernel for one-token appends, both ending in the same per-unit quantizers
// (token_block_update, page_quantize, group_quantize) as the append kernels.
#include "kvq_project.cuh"

namespace kvq {

enum { kSeqOk = 0, kSeqNothing = 1, kSeqCapacity = 2, kSeqBadPage = 3 };

// The part of the append decision that needs no page-table check: kSeqOk
// means pages [first, last] must still be checked.
__device__ __forceinline__ int seq_append_head(const AppendArgs& a, int b, int& start, int& n, int& first, int& last) {
  start = a.seq_lens[b];
  n = a.t_per_seq ? a.t_per_seq[b] : a.t_new;
  if (n <= 0) return kSeqNothing;
  if (n > a.t_new || start < 0 || (long long)start + n > (long long)a.ppsm * kPage) return kSeqCapacity;
  // a completed CB2 group rewrites all of its pages, including earlier ones
  first = a.fmt == KVQ_FMT_CB2_GROUP4 ? (start / (kPage * kGroupPages)) * kGroupPages : start / kPage;
  last = (start + n - 1) / kPage;
  return kSeqOk;
}
__device__ __forceinline__ bool page_entry_ok(const AppendArgs& a, int b, int pg) {
  const uint32_t u = (uint32_t)a.page_table[(size_t)b * a.ppsm + pg], phys = u & 0x7FFFFFFFu;
  return (u >> 31) ? (a.fmt == KVQ_FMT_TIERED && phys < (uint32_t)a.num_tier_pages) : phys < (uint32_t)a.num_pages;
}

// Decide, identically in every launch, whether sequence b's append proceeds.
// Every thread of the CTA calls it together: they share the page-table checks
// (one strided pass) and agree on the answer.
__device__ int seq_append_state(const AppendArgs& a, int b, int& start, int& n) {
  int first = 0, last = -1;
  const int st = seq_append_head(a, b, start, n, first, last);
  int bad = 0;
  for (int pg = first + (int)threadIdx.x; pg <= last; pg += (int)blockDim.x) bad |= !page_entry_ok(a, b, pg);
  if (st != kSeqOk) return st;
  return __syncthreads_or(bad) ? kSeqBadPage : kSeqOk;
}
// The same decision taken by one thread alone.
__device__ int seq_append_state_1(const AppendArgs& a, int b, int& start, int& n) {
  int first = 0, last = -1;
  const int st = seq_append_head(a, b, start, n, first, last);
  if (st != kSeqOk) return st;
  for (int pg = first; pg <= last; ++pg)
    if (!page_entry_ok(a, b, pg)) return kSeqBadPage;
  return kSeqOk;
}

// Channels [c, c + 8) of new token t (c a multiple of 8) as fp32 into dst[0..8):
// one or two 16-byte loads when the input is 16-byte aligned (then every such
// run is, D being a multiple of 8), else element loads.
__device__ __forceinline__ void load_in8(const AppendArgs& a, int role, int b, int t, int h, int c, int D, float* dst) {
  const size_t i = (((size_t)b * a.t_new + t) * a.Hkv + h) * D + c;
  const bool vec = (reinterpret_cast<uintptr_t>(a.kv[role]) & 15u) == 0;
  if (a.in_dtype == KVQ_F32) {
    const float* p = static_cast<const float*>(a.kv[role]) + i;
    if (vec) {
      const float4 u = reinterpret_cast<const float4*>(p)[0], w = reinterpret_cast<const float4*>(p)[1];
      dst[0] = u.x; dst[1] = u.y; dst[2] = u.z; dst[3] = u.w;
      dst[4] = w.x; dst[5] = w.y; dst[6] = w.z; dst[7] = w.w;
    } else {
      for (int j = 0; j < 8; ++j) dst[j] = p[j];
    }
    return;
  }
  const uint16_t* p = static_cast<const uint16_t*>(a.kv[role]) + i;
  uint16_t hv[8];
  if (vec) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
    for (int j = 0; j < 4; ++j) { hv[2 * j] = (uint16_t)(w4[j] & 0xFFFFu); hv[2 * j + 1] = (uint16_t)(w4[j] >> 16); }
  } else {
    for (int j = 0; j < 8; ++j) hv[j] = p[j];
  }
  for (int j = 0; j < 8; ++j)
    dst[j] = a.in_dtype == KVQ_F16 ? __half2float(__ushort_as_half(hv[j])) : __uint_as_float((uint32_t)hv[j] << 16);
}

// 16-byte asynchronous global -> shared copies, committed and waited for per thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

// ----------------------------------------------------------------------------- certified decisions
// Unit roundoff of binary32, and the relative nudge used to test a rounding
// decision: a binary32 result r within relative error 3u of the exact value
// rounds to the same code as the exact value (and as the fp64 value, which is
// far closer) whenever r * (1 - kNudge) and r * (1 + kNudge) round to the same
// code, rounding being monotone (the nudged products are themselves rounded,
// by at most u, so they still enclose r (1 +- 5u)).
constexpr float kU = 5.9604645e-08f;      // 2^-24
constexpr float kNudge = 4.76837158e-07f; // 2^-21

// Round |a| (finite, >= 0) to the grid of a binary format with `mbits`
// mantissa bits and smallest normal exponent emin, ties to even, in fp64:
// quantum 2^(max(e, emin) - mbits) for a in [2^e, 2^(e+1)).  The result is a
// grid point, exact in binary32 for the formats used here (fp16, e4m3, e2m1),
// so a conversion of it from binary32 is exact (or saturates / overflows as
// the format does).
__device__ __noinline__ double grid_round64(double a, int mbits, int emin) {
  if (a == 0.0) return 0.0;
  int e = ilogb(a);
  if (e < emin) e = emin;
  const double q = ldexp(1.0, e - mbits);
  return rint(a / q) * q;
}
__device__ __noinline__ uint16_t f16_from_f64(double v) {
  const float r = (float)grid_round64(fabs(v), 10, -14);
  return (uint16_t)(f32_to_f16_bits(r) | (signbit(v) ? 0x8000u : 0u));
}
__device__ __noinline__ uint8_t e4m3_from_f64(double v) {
  const float r = (float)grid_round64(fabs(v), 3, -6);
  return (uint8_t)(f32_to_e4m3(r) | (signbit(v) ? 0x80u : 0u));
}
__device__ __noinline__ uint8_t e2m1_from_f64(double v) {
  const float r = (float)grid_round64(fabs(v), 1, 0);
  return (uint8_t)(f32_to_e2m1(r) | (signbit(v) ? 0x8u : 0u));
}

// The fp64 side of each certified rounding below (called only when the
// binary32 result cannot be certified; kept out of line so the common path
// holds no fp64 state).
__device__ __noinline__ uint16_t f16_of_quotient64(float a, float b) { return f16_from_f64((double)a / (double)b); }
__device__ __noinline__ uint16_t f16_of_range64(float mx, float mn, float div) {
  return f16_from_f64(((double)mx - (double)mn) / (double)div);
}
__device__ __noinline__ uint8_t e4m3_of_quotient64(float a, float b) { return e4m3_from_f64((double)a / (double)b); }
__device__ __noinline__ uint8_t e2m1_of_quotient64(float a, float b) { return e2m1_from_f64((double)a / (double)b); }
__device__ __noinline__ uint32_t affine_code64(float x, float m, float S, float qmax) {
  const double r = rint(((double)x - (double)m) / (double)S);
  return (uint32_t)fmin(fmax(r, 0.0), (double)qmax);
}

// Whether the binary32 quotient r = fl(a / b) is exact: then it is the fp64
// quotient too, and any rounding of it (ties included) agrees with the
// definition.  The residual a - r b is exact in one fused multiply-add.
__device__ __forceinline__ bool quotient_exact(float r, float a, float b) { return __fmaf_rn(-r, b, a) == 0.f; }
// Whether the binary32 difference d = fl(x - m) is exact (TwoSum error term).
__device__ __forceinline__ bool difference_exact(float d, float x, float m) {
  const float bb = d - x;
  return (x - (d - bb)) + (-m - bb) == 0.f;
}

// fp16 bits of q = a / b, q's fp64 value rounded once (a, b binary32): the
// binary32 quotient when it is exact or the nudge cannot change its rounding,
// else fp64.
__device__ __forceinline__ uint16_t f16_of_quotient(float a, float b) {
  const float r = __fdiv_rn(a, b);
  const uint16_t h = f32_to_f16_bits(r);
  if (f32_to_f16_bits(r * (1.f - kNudge)) == h && f32_to_f16_bits(r * (1.f + kNudge)) == h) return h;
  if (quotient_exact(r, a, b)) return h;
  return f16_of_quotient64(a, b);
}
// fp16 bits of (mx - mn) / div (the affine formats' scale S), the same way;
// the binary32 value carries two roundings (the difference, the quotient).
__device__ __forceinline__ uint16_t f16_of_range(float mx, float mn, float div) {
  const float d = mx - mn, r = __fdiv_rn(d, div);
  const uint16_t h = f32_to_f16_bits(r);
  if (f32_to_f16_bits(r * (1.f - kNudge)) == h && f32_to_f16_bits(r * (1.f + kNudge)) == h) return h;
  if (difference_exact(d, mx, mn) && quotient_exact(r, d, div)) return h;
  return f16_of_range64(mx, mn, div);
}
// e4m3 / e2m1 code of a / b, the same way.
__device__ __forceinline__ uint8_t e4m3_of_quotient(float a, float b) {
  const float r = __fdiv_rn(a, b);
  const uint8_t c = f32_to_e4m3(r);
  if (f32_to_e4m3(r * (1.f - kNudge)) == c && f32_to_e4m3(r * (1.f + kNudge)) == c) return c;
  if (quotient_exact(r, a, b)) return c;
  return e4m3_of_quotient64(a, b);
}
__device__ __forceinline__ uint8_t e2m1_of_quotient(float a, float b) {
  const float r = __fdiv_rn(a, b);
  const uint8_t c = f32_to_e2m1(r);
  if (f32_to_e2m1(r * (1.f - kNudge)) == c && f32_to_e2m1(r * (1.f + kNudge)) == c) return c;
  if (quotient_exact(r, a, b)) return c;
  return e2m1_of_quotient64(a, b);
}
// Affine code clamp(rint((x - m) / S), 0, qmax) (S, m fp16 values, S != 0)
// with the quotient in fp64: (x - m) and the division are each rounded once in
// binary32 (relative error <= 2u + u^2, no cancellation term since x and m are
// exact inputs), so the nudge test certifies the binary32 code; so does an
// exact difference and quotient (a tie then resolves to even in both).
__device__ __forceinline__ uint32_t affine_code(float x, float m, float S, float qmax) {
  const float d = x - m, r = __fdiv_rn(d, S);
  const float c = fminf(fmaxf(rintf(r), 0.f), qmax);
  const float lo = fminf(fmaxf(rintf(r * (1.f - kNudge)), 0.f), qmax);
  const float hi = fminf(fmaxf(rintf(r * (1.f + kNudge)), 0.f), qmax);
  if (lo == c && hi == c) return (uint32_t)c;
  if (difference_exact(d, x, m) && quotient_exact(r, d, S)) return (uint32_t)c;
  return affine_code64(x, m, S, qmax);
}

// The outlier decisions of outlier_decide below, in fp64 in the definition's
// order (ascending sums, strict comparison).
__device__ __noinline__ void outlier_decide64(const float* x, int n, int stride, double sigma, int kmax,
                                              uint32_t* bits) {
  double sum64 = 0.0;
  for (int i = 0; i < n; ++i) sum64 += (double)x[i * stride];
  const double mu64 = sum64 / (double)n;
  double ss64 = 0.0;
  for (int i = 0; i < n; ++i) {
    const double d = (double)x[i * stride] - mu64;
    ss64 += d * d;
  }
  const double thr64 = sigma * sqrt(ss64 / (double)(n - 1));
  int k = 0;
  for (int w = 0; w < (n + 31) / 32; ++w) {
    uint32_t m = 0;
    for (int j = 0; j < 32 && 32 * w + j < n; ++j) {
      int out = fabs((double)x[(32 * w + j) * stride] - mu64) > thr64;
      if (out && k >= kmax) out = 0;
      m |= (uint32_t)out << j;
      k += out;
    }
    bits[w] = m;
  }
}

// Outlier decisions of one vector x[i * stride], i < n <= 128, as bits
// (bit i % 32 of bits[i / 32]): x_i is an outlier iff |x_i - mu| > sigma * s,
// mu the mean and s the unbiased standard deviation, at most kmax kept (the
// lowest indices).  Defined in fp64 with ascending-index sums.  The binary32
// pass (sequential sums) stays within E = 2 n (2 + sigma) u max|x| of the
// exact |x_i - mu| - sigma s for every i (mean: (n + 1) u max|x|; s: the
// deviation errors plus n u s from the sum of squares, s <= 2 max|x|), and
// the fp64 pass within 1e-12 of that; when some |x_i - mu| - sigma s is not
// farther than E from 0 the vector is decided again in fp64.
__device__ __noinline__ void outlier_decide(const float* x, int n, int stride, double sigma, int kmax, uint32_t* bits) {
  const float sg = (float)sigma;
  float sum = 0.f, amax = 0.f;
  const float v0 = x[0];
  bool cst = true;   // every value equal (no NaN)
  for (int i = 0; i < n; ++i) {
    const float v = x[i * stride];
    sum += v;
    amax = fmaxf(amax, fabsf(v));
    cst = cst && v == v0;
  }
  if (cst) {   // a constant vector: its mean is the value itself in either precision, so no outliers
    for (int w = 0; w < (n + 31) / 32; ++w) bits[w] = 0u;
    return;
  }
  const float mu = __fdiv_rn(sum, (float)n);
  float ss = 0.f;
  for (int i = 0; i < n; ++i) {
    const float d = x[i * stride] - mu;
    ss += d * d;
  }
  const float thr = sg * __fsqrt_rn(__fdiv_rn(ss, (float)(n - 1)));
  const float E = 2.f * (float)n * (2.f + sg) * kU * amax;
  bool sure = true;
  int k = 0;
  for (int w = 0; w < (n + 31) / 32; ++w) {
    uint32_t m = 0;
    for (int j = 0; j < 32 && 32 * w + j < n; ++j) {
      const float f = fabsf(x[(32 * w + j) * stride] - mu);
      sure = sure && fabsf(f - thr) > E;   // false for a NaN anywhere: decided in fp64
      int out = f > thr;
      if (out && k >= kmax) out = 0;
      m |= (uint32_t)out << j;
      k += out;
    }
    bits[w] = m;
  }
  if (!sure) outlier_decide64(x, n, stride, sigma, kmax, bits);
}

// Outlier mask of one vector as bytes mask[i * mstride] (see outlier_decide).
__device__ int outlier_mask(const float* x, int n, int stride, double sigma, int kmax, uint8_t* mask, int mstride) {
  uint32_t bits[4];
  outlier_decide(x, n, stride, sigma, kmax, bits);
  int k = 0;
  for (int i = 0; i < n; ++i) {
    const int out = (bits[i >> 5] >> (i & 31)) & 1u;
    mask[i * mstride] = (uint8_t)out;
    k += out;
  }
  return k;
}

// The same decisions for one row of D values as bits: bit c % 32 of
// bits[c / 32] is set for an outlier channel c.
template <int D>
__device__ void outlier_bits(const float* x, double sigma, int kmax, uint32_t* bits) {
  outlier_decide(x, D, 1, sigma, kmax, bits);
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
// Nearest of four centroids (lowest index on ties) and whether the choice is
// certain: the runner-up is farther by more than E.
__device__ __forceinline__ int nearest4_sure(float v, const float* c, float E, bool& sure) {
  int best = 0;
  float bd = fabsf(v - c[0]), sd = INFINITY;
  for (int j = 1; j < 4; ++j) {
    const float d = fabsf(v - c[j]);
    if (d < bd) { sd = bd; bd = d; best = j; }
    else sd = fminf(sd, d);
  }
  sure = sure && sd - bd > E;
  return best;
}

// Lloyd-Max 4-centroid fit of the values x[r * xs] of the rows r < NROWS set
// in `keep`, taken in row order, exactly as defined (fp64): linspace(min, max,
// 4) start, nearest centroid (lowest index on ties), at most `iters`
// assignment passes, stop when an assignment repeats, centroid = mean of its
// values (an empty cell keeps its centroid), centroids rounded once to fp16,
// codes = the nearest fp16 centroid.
template <int NROWS>
__device__ __noinline__ void lloyd4_rows64(const float* x, int xs, uint64_t keep, int iters, uint16_t* c16,
                                           uint32_t (&code)[(NROWS + 15) / 16]) {
  constexpr int NW = (NROWS + 15) / 16;
  double c[4] = {0.0, 0.0, 0.0, 0.0};
  for (int w = 0; w < NW; ++w) code[w] = 0u;
  auto near64 = [](double v, const double* cc) {
    int best = 0;
    double bd = fabs(v - cc[0]);
    for (int j = 1; j < 4; ++j) {
      const double d = fabs(v - cc[j]);
      if (d < bd) { bd = d; best = j; }
    }
    return best;
  };
  if (keep) {
    bool have = false;
    double mn = 0.0, mx = 0.0;
    for (int r = 0; r < NROWS; ++r) {
      if (!(keep >> r & 1u)) continue;
      const double v = x[r * xs];
      if (!have) { mn = v; mx = v; have = true; }
      mn = v < mn ? v : mn;
      mx = v > mx ? v : mx;
    }
    const double h = (mx - mn) / 3.0;
    c[0] = mn; c[1] = mn + h; c[2] = mn + 2.0 * h; c[3] = mx;
    uint32_t prev[NW], a[NW];
    bool have_prev = false;
    for (int it = 0; it < iters; ++it) {
      for (int w = 0; w < NW; ++w) a[w] = 0u;
      for (int r = 0; r < NROWS; ++r)
        if (keep >> r & 1u) a[r >> 4] |= (uint32_t)near64((double)x[r * xs], c) << (2 * (r & 15));
      bool same = have_prev;
      for (int w = 0; w < NW; ++w) same = same && a[w] == prev[w];
      if (same) break;
      for (int jj = 0; jj < 4; ++jj) {
        double sum = 0.0;
        int cnt = 0;
        for (int r = 0; r < NROWS; ++r)
          if ((keep >> r & 1u) && ((a[r >> 4] >> (2 * (r & 15))) & 3u) == (uint32_t)jj) {
            sum += (double)x[r * xs];
            ++cnt;
          }
        if (cnt > 0) c[jj] = sum / (double)cnt;
      }
      for (int w = 0; w < NW; ++w) prev[w] = a[w];
      have_prev = true;
    }
  }
  double cf[4];
  for (int jj = 0; jj < 4; ++jj) {
    c16[jj] = f16_from_f64(c[jj]);
    cf[jj] = (double)f16_bits_to_f32(c16[jj]);
  }
  for (int r = 0; r < NROWS; ++r)
    if (keep >> r & 1u) code[r >> 4] |= (uint32_t)near64((double)x[r * xs], cf) << (2 * (r & 15));
}

// Exponent of the lowest set bit of binary32 v != 0 (v is a multiple of 2^e).
__device__ __forceinline__ int low_bit_exp(float v) {
  const uint32_t u = __float_as_uint(v);
  const int ef = (int)((u >> 23) & 0xFFu);
  const uint32_t m = (u & 0x7FFFFFu) | (ef ? 0x800000u : 0u);
  return (ef ? ef : 1) - 150 + (__ffs((int)m) - 1);
}

// Whether v's four distances |v - c_j| decide alike in binary32 and fp64: each
// c_j is its exact value (a binary32 mean that is the exact mean, or an input
// value) and each subtraction is exact, so both precisions compare the same
// exact numbers, ties included.
__device__ __forceinline__ bool distances_exact(float v, const float* c, const bool* cx) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 4; ++j) ok = ok && cx[j] && difference_exact(v - c[j], v, c[j]);
  return ok;
}

// The fp64 mean of the rows of `keep` whose code in `asg` is j, summed in row
// order (the definition's order).
template <int NROWS>
__device__ __noinline__ double cell_mean64(const float* x, int xs, uint64_t keep, const uint32_t* asg, int j) {
  double sum = 0.0;
  int cnt = 0;
  for (int r = 0; r < NROWS; ++r)
    if ((keep >> r & 1u) && ((asg[r >> 4] >> (2 * (r & 15))) & 3u) == (uint32_t)j) {
      sum += (double)x[r * xs];
      ++cnt;
    }
  return sum / (double)cnt;
}
// The nearest of four fp16 centroids to v by fp64 distances (lowest index on ties).
__device__ __noinline__ int nearest4_64(float v, const float* cf) {
  int best = 0;
  double bd = fabs((double)v - (double)cf[0]);
  for (int j = 1; j < 4; ++j) {
    const double d = fabs((double)v - (double)cf[j]);
    if (d < bd) { bd = d; best = j; }
  }
  return best;
}

// Centroid j's fp64 value as the definition computes it, given its source: a
// linspace point (from the min mn and max mx), or the mean of a cell whose
// sum `sum` of `cnt` values is exact in binary32 (so the fp64 sum, in any
// order, is the same number).
__device__ __noinline__ double centroid64(int j, float mn, float mx, bool lin, float sum, int cnt) {
  if (lin) {
    const double h = ((double)mx - (double)mn) / 3.0;
    return j == 0 ? (double)mn : j == 1 ? (double)mn + h : j == 2 ? (double)mn + 2.0 * h : (double)mx;
  }
  return (double)sum / (double)cnt;
}
// fp16 bits of the mean of the rows of `keep` whose code in `asg` is j, when
// a compensated (TwoSum) binary32 evaluation settles its rounding; 0xFFFF
// (a NaN pattern no mean produces here) when it does not.  The sum is kept
// as hi + lo (within n^2 u^2 max|value| of the exact sum), the mean as q1 +
// d with q1 = hi / n and d = (hi - q1 n + lo) / n (the first residual exact),
// so q1 + d is within 4 u |d| + 4 n u^2 max|value| of the exact mean, which
// is far closer to it than to any fp16 rounding boundary except in an exact
// tie; the side of the boundary is the sign of (q1 - b) + d, whose first
// difference is exact (q1 and b are close).  The fp64 mean lies as close.
template <int NROWS>
__device__ __noinline__ uint16_t cell_mean_f16_tight(const float* x, int xs, uint64_t keep, const uint32_t* asg,
                                                     int j) {
  float hi = 0.f, lo = 0.f, m = 0.f;
  int n = 0;
  for (int r = 0; r < NROWS; ++r)
    if ((keep >> r & 1u) && ((asg[r >> 4] >> (2 * (r & 15))) & 3u) == (uint32_t)j) {
      const float v = x[r * xs];
      const float sm = hi + v, bb = sm - hi;
      lo += (hi - (sm - bb)) + (v - bb);
      hi = sm;
      m = fmaxf(m, fabsf(v));
      ++n;
    }
  const float fn = (float)n;
  const float q1 = __fdiv_rn(hi, fn);
  const float d = __fdiv_rn(__fmaf_rn(-q1, fn, hi) + lo, fn);
  const float mean = q1 + d;
  const float tol = 4.f * kU * fabsf(d) + 4.f * fn * kU * kU * m;
  const float e = kU * fabsf(mean) + tol;
  const uint16_t h = f32_to_f16_bits(mean);
  const uint16_t lo16 = f32_to_f16_bits(mean - e), hi16 = f32_to_f16_bits(mean + e);
  if (lo16 == h && hi16 == h) return h;
  const float vl = f16_bits_to_f32(lo16), vh = f16_bits_to_f32(hi16);
  if (!isfinite(vl) || !isfinite(vh)) return 0xFFFFu;
  // one fp16 boundary b inside [mean - e, mean + e]: which side is the mean on?
  const float b = (vl + vh) * 0.5f;
  if (f32_to_f16_bits(b) != lo16 && f32_to_f16_bits(b) != hi16) return 0xFFFFu;   // not adjacent
  const float t = (q1 - b) + d;
  if (t > tol) return hi16;
  if (t < -tol) return lo16;
  return 0xFFFFu;
}

// Final codes of the rows of `rows` that the midpoint count did not settle:
// nearest fp16 centroid by a distance margin, exact distances, else fp64.
// (Rare; out of line so that it takes no registers from the fit's loop.)
template <int NROWS>
__device__ __noinline__ void lloyd_fix_codes(const float* x, int xs, uint64_t rows, const float* cf, bool flat,
                                             float cmax, uint32_t* code) {
  const bool cfx[4] = {true, true, true, true};
  for (int r = 0; r < NROWS; ++r) {
    if (!(rows >> r & 1u)) continue;
    const float v = x[r * xs];
    const float ef = flat ? -1.f : 4.f * kU * (fabsf(v) + cmax);
    bool ok = true;
    uint32_t q = (uint32_t)nearest4_sure(v, cf, ef, ok);
    if (!ok && !distances_exact(v, cf, cfx)) q = (uint32_t)nearest4_64(v, cf);
    code[r >> 4] = (code[r >> 4] & ~(3u << (2 * (r & 15)))) | (q << (2 * (r & 15)));
  }
}

// State of one channel's binary32 fit that the rare paths need: the values'
// range, the bound E, and per centroid its source (a linspace point, or the
// binary32 sum and count of the cell it was last the mean of).
struct LloydState {
  float c[4];
  float sumc[4];
  int cntc[4];
  bool lin[4];
  float mn, mx, amax, E;
  int sums_exact;   // -1: not yet known; else whether every partial sum of the values is exact
};

// Whether every partial sum of at most NROWS of the kept values is exact in
// binary32 (and so in fp64): they are multiples of 2^elo (the lowest set bit
// of any value) below NROWS * max|x|, so exact if that spans at most 24 bits.
template <int NROWS>
__device__ __noinline__ bool sums_exact_of(const float* x, int xs, uint64_t keep, float amax) {
  if (amax == 0.f) return true;
  int elo = 1000;
  for (int r = 0; r < NROWS; ++r)
    if (keep >> r & 1u) {
      const float v = x[r * xs];
      if (v != 0.f) elo = min(elo, low_bit_exp(v));
    }
  int eh = 0;
  frexpf(amax * (float)NROWS, &eh);
  return eh - elo <= 24;
}
// fp16 bits of sum / cnt rounded once (ties to even), for a sum that is
// exact in binary32: the binary32 quotient is within one rounding of the
// mean, so the answer is its fp16 rounding or a neighbour, and which side of
// a neighbouring midpoint b the mean lies on is the sign of sum - b cnt, which
// one fused multiply-add gives exactly (b cnt is exact; the result is rounded
// once, keeping its sign, and is zero only on a tie).  The fp64 mean is never
// closer to b than a binary32 ulp of the sum unless it equals b, so rounding
// it to fp64 first (the definition) picks the same fp16 value.  0xFFFF for
// the largest fp16 values (left to fp64).
__device__ __forceinline__ uint16_t f16_of_exact_mean(float sum, int cnt) {
  const float fc = (float)cnt, as = fabsf(sum);
  uint16_t h = f32_to_f16_bits(__fdiv_rn(as, fc));
  if (h >= 0x7BFFu) return 0xFFFFu;
  const float vh = f16_bits_to_f32(h);
  const float bh = (vh + f16_bits_to_f32((uint16_t)(h + 1))) * 0.5f;
  const float rh = __fmaf_rn(-bh, fc, as);
  if (rh > 0.f || (rh == 0.f && (h & 1u))) {
    h = (uint16_t)(h + 1);
  } else if (h > 0) {
    const float bl = (f16_bits_to_f32((uint16_t)(h - 1)) + vh) * 0.5f;
    const float rl = __fmaf_rn(-bl, fc, as);
    if (rl < 0.f || (rl == 0.f && (h & 1u))) h = (uint16_t)(h - 1);
  }
  return (uint16_t)(h | (sum < 0.f ? 0x8000u : 0u));
}

// Whether centroid j is exactly its fp64 value.
template <int NROWS>
__device__ __forceinline__ bool centroid_exact(LloydState& S, const float* x, int xs, uint64_t keep, int j) {
  if (S.lin[j]) return j == 0 || j == 3 || S.mn == S.mx;
  if (S.sums_exact < 0) S.sums_exact = sums_exact_of<NROWS>(x, xs, keep, S.amax);
  return S.sums_exact && quotient_exact(S.c[j], S.sumc[j], (float)S.cntc[j]);
}

// The rows of `rows` whose binary32 assignment was not certified by the
// midpoint margin (all kept rows when the centroids are not strictly
// sorted), assigned again: by distances with a margin, by exact distances,
// else in fp64 from the centroids' fp64 values (from exact binary32 sums, or
// recomputed from the cells the previous pass formed; a centroid formed in an
// earlier pass leaves the fit unsure).  Rebuilds the assignment words and the four
// sums and counts in row order.  Returns false when a row is left unsure.
// (Rare; out of line like lloyd_fix_codes.)
// The fp64 nearest centroid of v (lowest index on ties) among those within
// 2E of the binary32 best, each candidate's fp64 value recomputed as the
// definition forms it: a linspace point from the range, or the fp64 mean, in
// row order, of the values the previous pass assigned to it (`prev`; that
// pass matched the definition).  -1 when a candidate was last formed in an
// earlier pass (its cell is no longer at hand).
template <int NROWS>
__device__ __noinline__ int nearest4_by_cells64(float v, const LloydState& S, const float* x, int xs, uint64_t keep,
                                                const uint32_t* prev, const bool* lastf) {
  float bd = INFINITY;
  for (int j = 0; j < 4; ++j) bd = fminf(bd, fabsf(v - S.c[j]));
  int best = -1;
  double b64 = 0.0;
  for (int j = 0; j < 4; ++j) {
    if (fabsf(v - S.c[j]) > bd + 2.f * S.E) continue;
    double c;
    if (S.lin[j]) c = centroid64(j, S.mn, S.mx, true, 0.f, 1);
    else if (lastf[j]) c = cell_mean64<NROWS>(x, xs, keep, prev, j);
    else return -1;
    const double d = fabs((double)v - c);
    if (best < 0 || d < b64) { b64 = d; best = j; }
  }
  return best;
}

template <int NROWS>
__device__ __noinline__ bool lloyd_fix_rows(LloydState& S, const float* x, int xs, uint64_t keep, uint64_t rows,
                                            uint32_t* a, float* sum, int* cnt, const uint32_t* prev,
                                            const bool* lastf) {
  constexpr int NW = (NROWS + 15) / 16;
  bool cx[4] = {false, false, false, false}, have_cx = false, have64 = false;
  double c64[4] = {0.0, 0.0, 0.0, 0.0};
  bool sure = true, changed = false;
  for (uint64_t m = rows; m; m &= m - 1) {
    const int r = __ffsll((long long)m) - 1;
    const float v = x[r * xs];
    bool ok = true;
    uint32_t j = (uint32_t)nearest4_sure(v, S.c, S.E, ok);
    if (!ok && !have_cx) {
      for (int jj = 0; jj < 4; ++jj) cx[jj] = centroid_exact<NROWS>(S, x, xs, keep, jj);
      have_cx = true;
    }
    if (!ok && !distances_exact(v, S.c, cx)) {
      if (S.sums_exact < 0) S.sums_exact = sums_exact_of<NROWS>(x, xs, keep, S.amax);
      if (S.sums_exact) {
        if (!have64) {   // the four fp64 centroids as centroid64 forms them, at once (independent divisions)
          const double h = ((double)S.mx - (double)S.mn) / 3.0;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            c64[jj] = S.lin[jj] ? (jj == 0 ? (double)S.mn : jj == 1 ? (double)S.mn + h : jj == 2 ? (double)S.mn + 2.0 * h
                                                                                         : (double)S.mx)
                                : (double)S.sumc[jj] / (double)S.cntc[jj];
          have64 = true;
        }
        // the fp64 nearest (lowest index on ties) among the centroids whose
        // binary32 distance is within 2E of the binary32 best: the others are
        // farther in fp64 as well (each distance is within E / 2 of its fp64 value)
        float bd = INFINITY;
        for (int jj = 0; jj < 4; ++jj) bd = fminf(bd, fabsf(v - S.c[jj]));
        int best = -1;
        double b64 = 0.0;
        for (int jj = 0; jj < 4; ++jj) {
          if (fabsf(v - S.c[jj]) > bd + 2.f * S.E) continue;
          const double d = fabs((double)v - c64[jj]);
          if (best < 0 || d < b64) { b64 = d; best = jj; }
        }
        j = (uint32_t)best;
      } else {   // inexact sums: the candidates' fp64 means from their cells
        const int jc = nearest4_by_cells64<NROWS>(v, S, x, xs, keep, prev, lastf);
        if (jc >= 0) j = (uint32_t)jc;
        else sure = false;
      }
    }
    changed |= ((a[r >> 4] >> (2 * (r & 15))) & 3u) != j;
    a[r >> 4] = (a[r >> 4] & ~(3u << (2 * (r & 15)))) | (j << (2 * (r & 15)));
  }
  if (!changed) return sure;   // the pass's own sums and counts stand
  for (int jj = 0; jj < 4; ++jj) { sum[jj] = 0.f; cnt[jj] = 0; }
  for (int r = 0; r < NROWS; ++r)
    if (keep >> r & 1u) {
      const uint32_t j = (a[r >> 4] >> (2 * (r & 15))) & 3u;
      sum[j] += x[r * xs];
      ++cnt[j];
    }
  (void)NW;
  return sure;
}

// The same fit, run in binary32 with a bound: while the assignments agree, a
// centroid is the mean of the same values in either precision, and a binary32
// mean of cnt values lies within cnt u max|x| of the fp64 one (a sum of cnt
// terms, then one division); the linspace points lie within 4 u max|x|.
// Centroids stay sorted (the linspace start is, and the means of cells cut at
// midpoints keep the order; an empty cell's centroid lies between its
// neighbours' cells).  With strictly sorted centroids the nearest one (lowest
// index on ties) is the number of midpoints (c_j + c_j+1) / 2 a value
// exceeds, and a value farther than E = 2 (NROWS + 4) u max|x| from every
// binary32 midpoint is assigned as fp64 would.  The other rows (all rows if
// the centroids are not strictly sorted) are assigned again out of line
// (lloyd_fix_rows); a row that neither a margin, exact distances nor fp64
// centroids settle sends the channel to lloyd4_rows64.  The fp16 rounding of
// each final centroid is checked over +-2 (cnt + 2) u max|x| around it, then
// from a compensated mean of its cell, then done in fp64.  Each final code
// counts the exact midpoints of the sorted fp16 centroids it exceeds (one
// fp64 comparison where it lies within 2^-45 of one), or, unsorted, is taken
// like an assignment.  Values are read from shared memory on every pass;
// assignments are packed 16 to a word, so the fit holds few registers.
template <int NROWS>
__device__ __forceinline__ void lloyd4_rows(const float* x, int xs, uint64_t keep, int iters, uint16_t* c16,
                                            uint32_t (&code)[(NROWS + 15) / 16]) {
  constexpr int NW = (NROWS + 15) / 16;
  LloydState S;
#pragma unroll
  for (int j = 0; j < 4; ++j) { S.c[j] = 0.f; S.sumc[j] = 0.f; S.cntc[j] = 1; S.lin[j] = false; }
  S.mn = S.mx = S.amax = S.E = 0.f;
  S.sums_exact = -1;
  bool last[4] = {false, false, false, false};   // centroid j was formed in the last update
#pragma unroll
  for (int w = 0; w < NW; ++w) code[w] = 0u;
  bool sure = true, flat = false;
  uint32_t prev[NW];
  bool have_prev = false;
  if (keep) {
    bool have = false;
    float mn = 0.f, mx = 0.f;
    int elo = 1000;   // lowest set bit of any nonzero value
    for (int r = 0; r < NROWS; ++r) {
      if (!(keep >> r & 1u)) continue;
      const float v = x[r * xs];
      if (!have) { mn = v; mx = v; have = true; }
      mn = v < mn ? v : mn;
      mx = v > mx ? v : mx;
      if (v != 0.f) elo = min(elo, low_bit_exp(v));
    }
    S.mn = mn;
    S.mx = mx;
    S.amax = fmaxf(fabsf(mn), fabsf(mx));
    {   // whether every partial sum of the values is exact (as sums_exact_of;
        // taken here for every fit: the rare paths that need it would
        // otherwise stall their warp on a separate pass over the rows)
      int eh = 0;
      frexpf(S.amax * (float)NROWS, &eh);
      S.sums_exact = S.amax == 0.f || eh - elo <= 24;
    }
    // one value repeated: all centroids equal it in either precision and
    // every assignment is centroid 0; no margin to check
    flat = mn == mx;
    S.E = flat ? -1.f : 2.f * (float)(NROWS + 4) * kU * S.amax;
    const float h = __fdiv_rn(mx - mn, 3.0f);
    S.c[0] = mn; S.c[1] = mn + h; S.c[2] = mn + 2.0f * h; S.c[3] = mx;
    S.lin[0] = S.lin[1] = S.lin[2] = S.lin[3] = true;
    for (int it = 0; it < iters; ++it) {
      // one pass assigns every value and sums each centroid's members in row
      // order (four independent sums: adding +0.0 to the others changes none
      // of them, a sum that starts at +0.0 never being -0.0)
      const bool srt = S.c[0] < S.c[1] && S.c[1] < S.c[2] && S.c[2] < S.c[3];
      const float m0 = (S.c[0] + S.c[1]) * 0.5f, m1 = (S.c[1] + S.c[2]) * 0.5f, m2 = (S.c[2] + S.c[3]) * 0.5f;
      uint32_t a[NW];
#pragma unroll
      for (int w = 0; w < NW; ++w) a[w] = 0u;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      int cnt[4] = {0, 0, 0, 0};
      uint64_t unc = 0;
      for (int r = 0; r < NROWS; ++r) {
        if (!(keep >> r & 1u)) continue;
        const float v = x[r * xs];
        const uint32_t j = (uint32_t)(v > m0) + (uint32_t)(v > m1) + (uint32_t)(v > m2);
        const float mg = fminf(fminf(fabsf(v - m0), fabsf(v - m1)), fabsf(v - m2));
        unc |= (uint64_t)(!(mg > S.E)) << r;
        a[r >> 4] |= j << (2 * (r & 15));
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          sum[jj] += j == (uint32_t)jj ? v : 0.f;
          cnt[jj] += j == (uint32_t)jj;
        }
      }
      if (!srt) unc = keep;
      if (unc) sure = lloyd_fix_rows<NROWS>(S, x, xs, keep, unc, a, sum, cnt, prev, last) && sure;
      bool same = have_prev;
#pragma unroll
      for (int w = 0; w < NW; ++w) same = same && a[w] == prev[w];
      if (same) break;
      // centroid j = the mean of its values
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        last[jj] = cnt[jj] > 0;
        if (cnt[jj] > 0) {
          S.c[jj] = __fdiv_rn(sum[jj], (float)cnt[jj]);
          S.lin[jj] = false;
          S.sumc[jj] = sum[jj];
          S.cntc[jj] = cnt[jj];
        }
      }
#pragma unroll
      for (int w = 0; w < NW; ++w) prev[w] = a[w];
      have_prev = true;
    }
  }
  if (!sure) {   // an assignment neither bound nor exact sums settle: the whole fit in fp64
    lloyd4_rows64<NROWS>(x, xs, keep, iters, c16, code);
    return;
  }
  float cf[4];
  for (int jj = 0; jj < 4; ++jj) {
    c16[jj] = f32_to_f16_bits(S.c[jj]);
    // a mean of cnt values: within cnt u max|x| (linspace points: 4 u max|x|)
    const float ec = flat ? 0.f : 2.f * (float)((S.lin[jj] ? 2 : S.cntc[jj]) + 2) * kU * S.amax;
    const float e = fmaxf(ec, fabsf(S.c[jj]) * kNudge);
    bool ok = f32_to_f16_bits(S.c[jj] - e) == c16[jj] && f32_to_f16_bits(S.c[jj] + e) == c16[jj];
    if (!ok) ok = centroid_exact<NROWS>(S, x, xs, keep, jj);
    if (!ok && !S.lin[jj] && S.sums_exact == 1) {   // an exact sum: its mean rounded exactly
      const uint16_t hm = f16_of_exact_mean(S.sumc[jj], S.cntc[jj]);
      if (hm != 0xFFFFu) {
        c16[jj] = hm;
        ok = true;
      }
    }
    if (!ok && !S.lin[jj] && !S.sums_exact && last[jj]) {   // a compensated mean of its cell
      const uint16_t hm = cell_mean_f16_tight<NROWS>(x, xs, keep, prev, jj);
      if (hm != 0xFFFFu) {
        c16[jj] = hm;
        ok = true;
      }
    }
    if (!ok) {
      if (S.lin[jj] || S.sums_exact) {
        c16[jj] = f16_from_f64(centroid64(jj, S.mn, S.mx, S.lin[jj], S.sumc[jj], S.cntc[jj]));
      } else if (last[jj]) {
        c16[jj] = f16_from_f64(cell_mean64<NROWS>(x, xs, keep, prev, jj));
      } else {   // not a mean of the last cells and its sum not kept exactly: refit in fp64
        lloyd4_rows64<NROWS>(x, xs, keep, iters, c16, code);
        return;
      }
    }
    cf[jj] = f16_bits_to_f32(c16[jj]);
  }
  // final codes: the midpoints of strictly sorted fp16 centroids are exact in
  // binary32 when their sums are (checked); fp64 compares |x - c_j| exactly
  // unless x lies within its rounding (2^-45 of |x| + max|c|) of a midpoint
  const bool fsrt = cf[0] < cf[1] && cf[1] < cf[2] && cf[2] < cf[3];
  const float s0 = cf[0] + cf[1], s1 = cf[1] + cf[2], s2 = cf[2] + cf[3];
  const bool bex = fsrt && difference_exact(s0, cf[0], -cf[1]) && difference_exact(s1, cf[1], -cf[2]) &&
                   difference_exact(s2, cf[2], -cf[3]);
  const float b0 = s0 * 0.5f, b1 = s1 * 0.5f, b2 = s2 * 0.5f;
  const float cmax = fmaxf(fmaxf(fabsf(cf[0]), fabsf(cf[1])), fmaxf(fabsf(cf[2]), fabsf(cf[3])));
  uint64_t unc = 0;
  for (int r = 0; r < NROWS; ++r)
    if (keep >> r & 1u) {
      const float v = x[r * xs];
      const uint32_t q = (uint32_t)(v > b0) + (uint32_t)(v > b1) + (uint32_t)(v > b2);
      const float mg = fminf(fminf(fabsf(v - b0), fabsf(v - b1)), fabsf(v - b2));
      unc |= (uint64_t)(!(mg > 2.8421709e-14f * (fabsf(v) + cmax))) << r;   // 2^-45
      code[r >> 4] |= q << (2 * (r & 15));
    }
  if (!bex) unc = keep;
  if (unc) lloyd_fix_codes<NROWS>(x, xs, unc, cf, flat, cmax, code);
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
// Byte of a block's code words (fragment order, see frag_inverse) that holds
// the 4-bit codes of K channels c, c + 1 (c even) of token t -- low, high
// nibble -- and the byte that holds tokens t, t + 1 (t even) of V channel c.
__device__ __forceinline__ int code_byte_k(int NS, int t, int c) {
  const int cc = c & 15;
  return 4 * NS * (4 * (t & 7) + ((cc & 7) >> 1)) + 4 * (c >> 4) + (t >> 3) + 2 * (cc >> 3);
}
__device__ __forceinline__ int code_byte_v(int NS, int t, int c) {
  const int cc = c & 15;
  return 4 * NS * (4 * (cc & 7) + ((t & 7) >> 1)) + 4 * (c >> 4) + 2 * (t >> 3) + (cc >> 3);
}

// Store the NC codes of one lane -- token t, channels c0 .. c0 + NC, code i at
// bits 4 (i % 8) of nb[i / 8] -- into the block's code words.  Tokens outside
// [lo, hi) keep their codes.  K bytes belong to one token.  A V byte holds an
// even token and the next one: the even token's lane (always in the same
// pass, whose first token is even) writes it, with its partner's codes (the
// lane pd above, fetched by shuffle) or the kept nibble for a token outside
// [lo, hi).  Every lane of the warp calls this (the shuffle).
template <int NC>
__device__ __forceinline__ void store_codes(uint8_t* blk, int role, int NS, int t, int c0, int lo, int hi,
                                            const uint32_t (&nb)[NC / 8], int pd) {
  const bool act = t >= lo && t < hi;
  if (role == 0) {
    if (act)
#pragma unroll
      for (int i = 0; i < NC; i += 2) blk[code_byte_k(NS, t, c0 + i)] = (uint8_t)(nb[i >> 3] >> (4 * (i & 7)));
    return;
  }
  uint32_t pn[NC / 8];
#pragma unroll
  for (int w = 0; w < NC / 8; ++w) pn[w] = __shfl_down_sync(0xffffffffu, nb[w], pd);
  if (!(t & 1)) {
    const bool pact = t + 1 >= lo && t + 1 < hi;
    if (!act && !pact) return;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      uint8_t* p = blk + code_byte_v(NS, t, c0 + i);
      const uint32_t lo4 = act ? (nb[i >> 3] >> (4 * (i & 7))) & 0xFu : *p & 0xFu;
      const uint32_t hi4 = pact ? (pn[i >> 3] >> (4 * (i & 7))) & 0xFu : *p >> 4;
      *p = (uint8_t)(lo4 | (hi4 << 4));
    }
  }
}

// INT4 group-32 quantization of token slots [t0, t0 + 32 / NG) by one warp (NG
// = D / 32 groups): lane s * NG + g owns group g of slot t0 + s; slots outside
// [lo, hi) compute on slot lo (a row the caller wrote) and store nothing.
// t0 < hi.  Channel c of a row sits at xs[t][c + GP * (c / 32)].
template <int D, int XS, int GP>
__device__ void quantize_tokens_int4(const float (*xs)[XS], int t0, int lo, int hi, uint8_t* blk, int role,
                                     double sigma, int lane) {
  constexpr int NG = D / 32, CAP = int4_cap(D);
  const int g = lane % NG, t = t0 + lane / NG;
  const bool act = t >= lo && t < hi;
  const float* xg = xs[act ? t : lo] + (32 + GP) * g;
  uint8_t mask[32];
  outlier_mask(xg, 32, 1, sigma, kmax_outliers(32), mask, 1);
  bool have = false;
  float mn = 0.f, mx = 0.f;
  for (int i = 0; i < 32; ++i) {
    if (mask[i]) continue;
    const float v = xg[i];
    if (!have || v < mn) mn = v;
    if (!have || v > mx) mx = v;
    have = true;
  }
  const uint16_t S16 = have ? f16_of_range(mx, mn, 15.0f) : 0;
  const uint16_t m16 = have ? f32_to_f16_bits(mn) : 0;
  const float S = f16_bits_to_f32(S16), m = f16_bits_to_f32(m16);
  int cnt = 0;
  uint32_t nb[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    uint32_t q = 0;
    if (mask[i]) {
      ++cnt;
    } else if (S != 0.f) {
      q = affine_code(xg[i], m, S, 15.f);
    }
    nb[i >> 3] |= q << (4 * (i & 7));
  }
  store_codes<32>(blk, role, D / 16, t, 32 * g, lo, hi, nb, NG);
  // entries of group g go after those of groups < g of the same token (ascending channel order)
  int off = cnt;
#pragma unroll
  for (int d = 1; d < NG; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, off, d, NG);
    if (g >= d) off += y;
  }
  const int total = __shfl_sync(0xffffffffu, off, NG - 1, NG);
  off -= cnt;
  if (!act) return;
  uint8_t* sz = blk + int4_sz_off(D) + 4 * (t * NG + g);
  *reinterpret_cast<uint16_t*>(sz) = S16;
  *reinterpret_cast<uint16_t*>(sz + 2) = m16;
  uint8_t* chans = blk + int4_ch_off(D) + t * CAP;
  uint16_t* vals = reinterpret_cast<uint16_t*>(blk + int4_val_off(D)) + t * CAP;
  for (int i = 0; i < 32; ++i)
    if (mask[i]) {
      chans[off] = (uint8_t)(32 * g + i);
      vals[off] = __half_as_ushort(__float2half_rn(xg[i]));
      ++off;
    }
  for (int i = total + g; i < CAP; i += NG) {
    chans[i] = 0;
    vals[i] = 0;
  }
  if (g == 0) blk[int4_cnt_off(D) + t] = (uint8_t)total;
}

// E2M1 quantization of token slots [t0, t0 + 32 / NS) by one warp (NS = D / 16
// scale groups): lane s * NS + g owns channels [16 g, 16 g + 16) of slot
// t0 + s; slots outside [lo, hi) compute on slot lo (a row the caller wrote)
// and store nothing.  Channel c of a row sits at xs[t][c + GP * (c / 32)].
template <int D, int XS, int GP>
__device__ void quantize_tokens_e2m1(const float (*xs)[XS], int t0, int lo, int hi, uint8_t* blk, int role,
                                     int lane) {
  constexpr int NS = D / 16;
  const int g = lane % NS, t = t0 + lane / NS;
  const bool act = t >= lo && t < hi;
  const float* x = xs[act ? t : lo] + 16 * g + GP * (g >> 1);
  float amax = 0.f;
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint8_t s8 = e4m3_of_quotient(amax, 6.0f);
  const float sc = e4m3_to_f32(s8);
  // binary32 codes, certified or flagged; the flagged ones (rare) are taken
  // again in fp64 after the loop, so the unrolled loop holds no call
  uint32_t nb[2] = {0u, 0u}, unsure = 0u;
  if (sc != 0.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float r = __fdiv_rn(x[i], sc);
      const uint8_t c = f32_to_e2m1(r);
      const bool sure = (f32_to_e2m1(r * (1.f - kNudge)) == c && f32_to_e2m1(r * (1.f + kNudge)) == c) ||
                        quotient_exact(r, x[i], sc);
      unsure |= (uint32_t)!sure << i;
      nb[i >> 3] |= (uint32_t)c << (4 * (i & 7));
    }
  }
  while (unsure) {
    const int i = __ffs(unsure) - 1;
    unsure &= unsure - 1u;
    const uint32_t c = e2m1_of_quotient64(x[i], sc), sh = 4 * (i & 7);
    if (i < 8) nb[0] = (nb[0] & ~(0xFu << sh)) | (c << sh);
    else nb[1] = (nb[1] & ~(0xFu << sh)) | (c << sh);
  }
  store_codes<16>(blk, role, NS, t, 16 * g, lo, hi, nb, NS);
  if (act) blk[e2m1_sc_off(D) + 16 * g + t] = s8;
}

// Threads [0, n) of a group of a CTA (tid is the index within the group, n a
// multiple of 32) that synchronise on named barrier `bar`; bar 0 with
// n = blockDim.x is the whole CTA.
struct Grp {
  int tid, n, bar;
  __device__ __forceinline__ void sync() const { asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(n) : "memory"); }
};
__device__ __forceinline__ Grp whole_cta() { return Grp{(int)threadIdx.x, (int)blockDim.x, 0}; }

// Per-token formats: re-quantize token slots [lo, hi) of one block from rows
// xs[slot] (row stride XS); the other slots keep their codes and metadata.
// blk (the block's bytes) is the group's scratch; the caller's writes of xs
// come before the call.  Channel c of a row sits at xs[slot][c + GP * (c /
// 32)]: GP = 1 pads each 32-channel group so that the lanes of a warp, one
// group each, read distinct banks.
template <int BF, int D, int XS, int GP = 0>
__device__ void token_block_update(const AppendArgs& a, int role, const float (*xs)[XS], int lo, int hi, uint8_t* gblk,
                                   uint8_t* blk, const Grp& g) {
  constexpr int kStride = block_stride(BF, D);
  const int lane = g.tid & 31, warp = g.tid >> 5, nw = g.n >> 5;
  // a block whose 16 slots are all rewritten keeps nothing of its old
  // contents: start it from zeros (its padding included) instead of a copy
  if (lo > 0 || hi < kPage) {
    for (int i = g.tid; i < kStride / 16; i += g.n)
      reinterpret_cast<uint4*>(blk)[i] = reinterpret_cast<const uint4*>(gblk)[i];
  } else {
    for (int i = g.tid; i < kStride / 16; i += g.n) reinterpret_cast<uint4*>(blk)[i] = make_uint4(0, 0, 0, 0);
  }
  g.sync();
  // passes start at an even slot, so the two tokens of a V code byte share a warp
  constexpr int TPW = 32 / (BF == kBlkInt4 ? D / 32 : D / 16);   // token slots per warp pass (even)
  for (int t0 = (lo & ~1) + warp * TPW; t0 < hi; t0 += nw * TPW) {
    if (BF == kBlkInt4) quantize_tokens_int4<D, XS, GP>(xs, t0, lo, hi, blk, role, a.sigma, lane);
    else quantize_tokens_e2m1<D, XS, GP>(xs, t0, lo, hi, blk, role, lane);
  }
  g.sync();
  for (int i = g.tid; i < kStride / 16; i += g.n)
    reinterpret_cast<uint4*>(gblk)[i] = reinterpret_cast<const uint4*>(blk)[i];
  g.sync();   // the scratch may be reused by the next call
}

// Pages one CTA of the per-token append handles: enough that every warp has
// tokens (a warp quantizes 32 / (D / 32) INT4 or 32 / (D / 16) E2M1 tokens per
// pass, and a page holds 16).
template <int BF>
__host__ __device__ constexpr int token_ppc() { return BF == kBlkInt4 ? 4 : 2; }

// Whether the per-token append prefetches its next pages (E2M1: measured 8%
// faster; INT4, whose CTAs already keep every warp busy, lost a resident CTA
// per SM to the buffer and ran 25% slower), and the page groups (of token_ppc
// pages) one CTA then takes in turn.
template <int BF>
__host__ __device__ constexpr bool token_pipe() { return BF == kBlkE2m1; }
constexpr int kTokenIters = 4;
// Dynamic shared memory of append_token_kernel<BF, D> for input elements of
// es bytes: per page, 16 staged rows of D + D / 32 floats, the block's bytes
// and (prefetching) the next page's raw input rows.
template <int BF, int D>
constexpr size_t token_smem_bytes(int es) {
  return (size_t)token_ppc<BF>() * (16 * (D + D / 32) * 4 + block_stride(BF, D) + (token_pipe<BF>() ? 16 * D * es : 0));
}

// Eight input elements (es bytes each, in_dtype) at p as fp32.
__device__ __forceinline__ void raw8_to_f32(const uint8_t* p, int in_dtype, float* dst) {
  if (in_dtype == KVQ_F32) {
    const float4 u = reinterpret_cast<const float4*>(p)[0], w = reinterpret_cast<const float4*>(p)[1];
    dst[0] = u.x; dst[1] = u.y; dst[2] = u.z; dst[3] = u.w;
    dst[4] = w.x; dst[5] = w.y; dst[6] = w.z; dst[7] = w.w;
    return;
  }
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
  for (int j = 0; j < 4; ++j)
    for (int k = 0; k < 2; ++k) {
      const uint16_t hv = (uint16_t)(w4[j] >> (16 * k));
      dst[2 * j + k] = in_dtype == KVQ_F16 ? __half2float(__ushort_as_half(hv)) : __uint_as_float((uint32_t)hv << 16);
    }
}

// A CTA's thread groups each take one page of a group of PPC pages, for
// page groups blockIdx.x, + gridDim.x, ... of the append; when prefetching,
// the next group's input rows are copied (cp.async) into shared memory while
// the current one is quantized.
template <int BF, int D>
__global__ void __launch_bounds__(256, BF == kBlkInt4 ? 4 : 5) append_token_kernel(const AppendArgs a) {
  // rows padded by one float per 32 channels: with D + D / 32 floats a row, the
  // lanes of a quantizing warp (each on its own token and channel group) read
  // 32 distinct banks
  constexpr int kStride = block_stride(BF, D), PPC = token_ppc<BF>(), GT = 256 / PPC, XS = D + D / 32;
  static_assert(kStride % 16 == 0, "per-page blocks must stay 16-byte aligned");
  extern __shared__ __align__(16) uint8_t tsm[];
  const int h = blockIdx.y >> 1, role = blockIdx.y & 1, b = blockIdx.z;
  const int grp = (int)threadIdx.x / GT;           // one thread group (its own named barrier) per page
  const Grp g{(int)threadIdx.x % GT, GT, 1 + grp};
  const int es = a.in_dtype == KVQ_F32 ? 4 : 2;
  float(*xs)[XS] = reinterpret_cast<float(*)[XS]>(tsm) + grp * 16;
  uint8_t* blk = tsm + PPC * 16 * XS * 4 + grp * kStride;
  uint8_t* raw = tsm + PPC * (16 * XS * 4 + kStride) + grp * 16 * D * es;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, p0 = start / kPage, np = (end - 1) / kPage - p0 + 1;   // the append's pages
  const int ngr = (np + PPC - 1) / PPC;
  const bool vec = token_pipe<BF>() && (reinterpret_cast<uintptr_t>(a.kv[role]) & 15u) == 0;   // 16-byte copies
  const uint8_t* src = static_cast<const uint8_t*>(a.kv[role]);
  auto issue = [&](int gi) {   // the group's page of page group gi -> raw
    const int pg = p0 + gi * PPC + grp;
    if (vec && gi < ngr && pg - p0 < np) {
      const int lo = max(start, pg * kPage), hi = min(end, pg * kPage + kPage);
      for (int i = g.tid; i < (hi - lo) * (D / 8); i += g.n) {
        const int tt = i / (D / 8), c = 8 * (i - tt * (D / 8));
        const uint8_t* sp = src + ((((size_t)b * a.t_new + (lo + tt - start)) * a.Hkv + h) * D + c) * es;
        const uint32_t d = smem_u32(raw + ((lo % kPage + tt) * D + c) * es);
        cp_async16(d, sp);
        if (es == 4) cp_async16(d + 16, sp + 16);
      }
    }
    cp_async_commit();
  };
  issue((int)blockIdx.x);
  for (int gi = (int)blockIdx.x; gi < ngr; gi += (int)gridDim.x) {
    const int pg = p0 + gi * PPC + grp;
    const bool mine = pg - p0 < np;   // uniform within the group
    const int lo = max(start, pg * kPage), hi = min(end, pg * kPage + kPage);
    cp_async_wait<0>();
    g.sync();   // the group's copies of this page have landed
    if (mine)
      for (int i = g.tid; i < (hi - lo) * (D / 8); i += g.n) {
        const int tt = i / (D / 8), c = 8 * (i - tt * (D / 8)), slot = lo % kPage + tt;
        if (vec) raw8_to_f32(raw + (slot * D + c) * es, a.in_dtype, &xs[slot][c + c / 32]);
        else load_in8(a, role, b, lo + tt - start, h, c, D, &xs[slot][c + c / 32]);
      }
    g.sync();   // raw is free for the next page's copies
    issue(gi + (int)gridDim.x);
    if (!mine) continue;
    const uint32_t phys = (uint32_t)a.page_table[(size_t)b * a.ppsm + pg] & 0x7FFFFFFFu;
    token_block_update<BF, D, XS, 1>(a, role, xs, lo % kPage, lo % kPage + (hi - lo),
                                     a.pool + (((size_t)phys * a.Hkv + h) * 2 + role) * kStride, blk, g);
  }
  cp_async_wait<0>();
}

// ----------------------------------------------------------------------------- page formats
// Outlier side-list of one page (CB2, ASYM3, CB2 group) from its mask and
// values [16][D] (row stride XS), built by one warp: lane l owns channels
// [l*D/32, (l+1)*D/32); one 20-byte record {channel, 0, token mask, 16 e4m3
// values} per channel with an outlier, channels ascending, after {n_ch,
// total}.  Zeros come from the block clear.
template <int D, int XS>
__device__ void build_side_list(const uint8_t (*mask)[D], const float (*xs)[XS], uint8_t* hdr, int lane) {
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
__device__ __forceinline__ void pack_cb2_codes(const uint8_t (*codes)[D], uint8_t* blk, int role, const Grp& g) {
  constexpr int NS = D / 16;
  for (int i = g.tid; i < 32 * NS; i += g.n) {
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
__device__ __forceinline__ void pack_a3_codes(const uint8_t (*codes)[D], uint8_t* blk, int role, const Grp& g) {
  constexpr int NS = D / 16, NG = NS / 4;
  for (int i = g.tid; i < 32 * NG; i += g.n) {
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

// Bytes of the block buffer a page quantization needs (CB2, CB2_STATIC, ASYM3 or an FP8 tier block).
template <int D>
__host__ __device__ constexpr int page_blk_bytes() {
  return block_stride(kBlkCb2, D) > block_stride(kBlkFp8, D) ? block_stride(kBlkCb2, D) : block_stride(kBlkFp8, D);
}

// Shared scratch of one page quantization.
template <int D>
struct PageWs {
  uint8_t (*mask)[D];   // [16][D]
  uint8_t (*codes)[D];  // [16][D]
  uint8_t* blk;         // page_blk_bytes<D>(), 16-byte aligned
  float* red;           // one float per warp of the group
};

// Page formats: quantize the 16 tokens xs[16] (row stride XS) of one page into
// the block named by page-table entry u (tier bit, physical page) and store it.
// The caller's writes of xs come before the call.
template <int D, int XS>
__device__ void page_quantize(const AppendArgs& a, int h, int role, uint32_t u, const float (*xs)[XS],
                              const PageWs<D>& ws, const Grp& g, const uint32_t* rbits = nullptr) {
  constexpr int NS = D / 16, kBlk = page_blk_bytes<D>();
  constexpr int kCb2 = block_stride(kBlkCb2, D), kFp8 = block_stride(kBlkFp8, D);
  uint8_t(*mask)[D] = ws.mask;
  uint8_t(*codes)[D] = ws.codes;
  uint8_t* blk = ws.blk;
  const int tid = g.tid;
  const uint32_t phys = u & 0x7FFFFFFFu;
  const bool tier = (u >> 31) != 0;
  const bool stat = a.fmt == KVQ_FMT_CB2_STATIC;
  const int stride = tier ? kFp8
                   : stat ? block_stride(kBlkCb2s, D)
                   : a.fmt == KVQ_FMT_ASYM3_OUTLIER ? block_stride(kBlkA3, D) : kCb2;
  uint8_t* gblk = (tier ? a.tier_pool : a.pool) + (((size_t)phys * a.Hkv + h) * 2 + role) * stride;

  for (int i = tid; i < kBlk / 16; i += g.n) reinterpret_cast<uint4*>(blk)[i] = make_uint4(0, 0, 0, 0);
  g.sync();

  if (tier) {
    float amax = 0.f;
    for (int i = tid; i < 16 * D; i += g.n) amax = fmaxf(amax, fabsf(xs[i / D][i % D]));
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((tid & 31) == 0) ws.red[tid >> 5] = amax;
    g.sync();
    amax = 0.f;
    for (int w = 0; w < g.n / 32; ++w) amax = fmaxf(amax, ws.red[w]);
    const float s = __fdiv_rn(amax, 448.0f);
    for (int i = tid; i < 16 * D; i += g.n) {
      const int t = i / D, c = i - t * D;
      const FragPos p = frag_pos(role, t, c);
      blk[8 * NS * p.lane + 8 * p.step + p.slot] = s != 0.f ? e4m3_of_quotient(xs[t][c], s) : 0;
    }
    if (tid == 0) *reinterpret_cast<float*>(blk + fp8_sc_off(D)) = s;
  } else if (stat) {
    // static fp16 channels (all tokens); every other channel: codebook over all 16 values
    const uint8_t* chs = a.static_mask + ((size_t)h * 2 + role) * a.n_static;
    if (tid < D) mask[0][tid] = 0;
    g.sync();
    if (tid < a.n_static) mask[0][chs[tid] & (D - 1)] = 1;
    g.sync();
    if (tid < D) {
      const int c = tid;
      if (mask[0][c]) {
        for (int t = 0; t < 16; ++t) codes[t][c] = 0;   // all-zero centroids from the block clear
      } else {
        uint32_t cc[1];
        uint16_t c16[4];
        lloyd4_rows<16>(&xs[0][c], XS, 0xFFFFull, a.iters, c16, cc);
        for (int t = 0; t < 16; ++t) codes[t][c] = (cc[0] >> (2 * t)) & 3u;
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
    g.sync();
    pack_cb2_codes<D>(codes, blk, role, g);
  } else {
    // CB2 or ASYM3: per-token outliers, then per channel a codebook (CB2) or an
    // 8-level affine grid (ASYM3) over the non-outliers
    const bool a3 = a.fmt == KVQ_FMT_ASYM3_OUTLIER;
    if (rbits) {   // decisions taken beforehand (outlier_bits), one row of D / 32 words per token
      for (int i = tid; i < 16 * D; i += g.n)
        mask[i / D][i % D] = (uint8_t)((rbits[(i / D) * (D / 32) + (i % D) / 32] >> (i % 32)) & 1u);
    } else if (tid < 16) {
      outlier_mask(&xs[tid][0], D, 1, a.sigma, kmax_outliers(D), &mask[tid][0], 1);
    }
    g.sync();
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
      const uint16_t S16 = have ? f16_of_range(mx, mn, 7.0f) : 0;
      const uint16_t m16 = have ? f32_to_f16_bits(mn) : 0;
      const float S = f16_bits_to_f32(S16), m = f16_bits_to_f32(m16);
      for (int t = 0; t < 16; ++t) {
        uint8_t q = 0;
        if (!mask[t][c] && S != 0.f) q = (uint8_t)affine_code(xs[t][c], m, S, 7.f);
        codes[t][c] = q;
      }
      const int r = a3_rho(role, c);
      *reinterpret_cast<uint16_t*>(blk + a3_s_off(D) + 2 * r) = S16;
      *reinterpret_cast<uint16_t*>(blk + a3_m_off(D) + 2 * r) = m16;
    } else if (tid < D) {
      const int c = tid;
      uint32_t cc[1];
      uint16_t c16[4];
      uint64_t keep = 0;
      for (int t = 0; t < 16; ++t) keep |= (uint64_t)(mask[t][c] == 0) << t;
      lloyd4_rows<16>(&xs[0][c], XS, keep, a.iters, c16, cc);
      for (int t = 0; t < 16; ++t) codes[t][c] = (cc[0] >> (2 * t)) & 3u;
      uint8_t* cbp = blk + cb2_cb_off(D) + 8 * cb2_slot(role, c);
      for (int jj = 0; jj < 4; ++jj) {
        cbp[jj] = (uint8_t)(c16[jj] & 0xFF);
        cbp[4 + jj] = (uint8_t)(c16[jj] >> 8);
      }
    }
    if (tid < 32) build_side_list<D, XS>(mask, xs, blk + (a3 ? a3_out_off(D) : cb2_out_off(D)), tid);
    g.sync();
    if (a3) pack_a3_codes<D>(codes, blk, role, g);
    else pack_cb2_codes<D>(codes, blk, role, g);
  }
  g.sync();
  for (int i = tid; i < stride / 16; i += g.n)
    reinterpret_cast<uint4*>(gblk)[i] = reinterpret_cast<const uint4*>(blk)[i];
  g.sync();   // the scratch may be reused by the next call
}

// New tokens of the final partial page (the final partial group for the CB2
// group format) -> fp32 staging.  Run by the CTA of the append's first page
// (first group) after it has read the staged rows: no other CTA reads them.
__device__ void stage_tail(const AppendArgs& a, int b, int h, int role, int start, int n, int rows, int D) {
  const int end = start + n;
  if (end % rows == 0) return;
  const int lo = max(start, (end / rows) * rows);
  float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * rows * D;
  for (int i = threadIdx.x; i < (end - lo) * (D / 8); i += blockDim.x) {
    const int tt = i / (D / 8), c = 8 * (i - tt * (D / 8)), pos = lo + tt;
    float v[8];
    load_in8(a, role, b, pos - start, h, c, D, v);
    for (int j = 0; j < 8; ++j) stg[(pos % rows) * D + c + j] = v[j];
  }
}

template <int D>
__global__ void __launch_bounds__(128, 8) append_page_kernel(const AppendArgs a) {
  __shared__ __align__(16) float xs[16][D];
  __shared__ uint8_t mask[16][D];
  __shared__ uint8_t codes[16][D];
  __shared__ __align__(16) uint8_t blk[page_blk_bytes<D>()];
  __shared__ float red[4];
  const int j = blockIdx.x, h = blockIdx.y >> 1, role = blockIdx.y & 1, b = blockIdx.z;
  const int tid = threadIdx.x;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, pg = start / kPage + j;
  const bool full = pg * kPage + kPage <= end;   // quantize only the pages this append completes
  if (!full && j != 0) return;
  if (full) {
    const uint32_t u = (uint32_t)a.page_table[(size_t)b * a.ppsm + pg];
    const float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * kPage * D;
    for (int i = tid; i < 16 * (D / 8); i += blockDim.x) {
      const int t = i / (D / 8), c = 8 * (i - t * (D / 8)), pos = pg * kPage + t;
      if (pos < start) {
        for (int jj = 0; jj < 8; ++jj) xs[t][c + jj] = stg[t * D + c + jj];
      } else {
        load_in8(a, role, b, pos - start, h, c, D, &xs[t][c]);
      }
    }
    page_quantize<D, D>(a, h, role, u, xs, PageWs<D>{mask, codes, blk, red}, whole_cta());   // ends with a barrier
  }
  if (j == 0) stage_tail(a, b, h, role, start, n, kPage, D);
}

// Shared scratch of one CB2 group quantization.
template <int D>
struct GroupWs {
  uint32_t* rbits;      // [64][D / 32] outlier decisions of the group's tokens (bit c % 32 of word c / 32)
  uint32_t (*cc)[4];    // [D][4] the 64 tokens' 2-bit codes of each channel, token t at bits 2 (t % 16) of word t / 16
  uint8_t* blk;         // kGroupPages blocks
};

// Outlier side-list of page p of a group (CB2 record layout, see
// build_side_list) from the group's outlier bits: lane l owns channels
// [l*D/32, (l+1)*D/32).
template <int D, int XS>
__device__ void build_side_list_bits(const uint32_t* rbits, const float (*xs)[XS], uint8_t* hdr, int lane) {
  constexpr int CPL = D / 32;
  uint32_t tm[CPL];
  int nch = 0, nval = 0;
  for (int k = 0; k < CPL; ++k) {
    const int c = lane * CPL + k;
    uint32_t m = 0;
    for (int t = 0; t < 16; ++t) m |= ((rbits[t * (D / 32) + c / 32] >> (c % 32)) & 1u) << t;
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

// Page p's 2-bit codes (word p of every channel's packed codes) -> the block's
// lane-major code words (CB2 layout).
template <int D>
__device__ __forceinline__ void pack_cb2_codes_packed(const uint32_t (*cc)[4], int p, uint8_t* blk, int role,
                                                      const Grp& g) {
  constexpr int NS = D / 16;
  for (int i = g.tid; i < 32 * NS; i += g.n) {
    const int ln = i / NS, s = i % NS;
    uint32_t word = 0;
    for (int k = 0; k < 8; ++k) {
      int t, c;
      frag_inverse(role, ln, s, k, t, c);
      word |= ((cc[c][p] >> (2 * t)) & 3u) << (4 * (k & 3) + 2 * (k >> 2));
    }
    *reinterpret_cast<uint16_t*>(blk + 2 * NS * ln + 2 * s) = (uint16_t)word;
  }
}

// CB2 group format: quantize the 64 tokens xs[64] (row stride XS) of group gr
// of the sequence whose page-table row is pt: outliers per token, one codebook
// per channel over the group's non-outliers in token order (in the group's
// first page), codes and side-list per page.  have_bits: ws.rbits already
// holds the tokens' outlier decisions (else they are taken here).
template <int D, int XS>
__device__ void group_quantize(const AppendArgs& a, int h, int role, const int32_t* pt, int gr, const float (*xs)[XS],
                               const GroupWs<D>& ws, const Grp& g, bool have_bits) {
  constexpr int GT = kPage * kGroupPages, kStride = block_stride(kBlkCb2g, D), NWD = D / 32;
  uint8_t* blk = ws.blk;
  const int tid = g.tid;
  for (int i = tid; i < kGroupPages * kStride / 16; i += g.n)
    reinterpret_cast<uint4*>(blk)[i] = make_uint4(0, 0, 0, 0);
  g.sync();   // also orders the caller's writes of xs before the reads below
  if (!have_bits) {
    if (tid < GT) outlier_bits<D>(&xs[tid][0], a.sigma, kmax_outliers(D), ws.rbits + tid * NWD);
    g.sync();
  }
  if (tid < D) {
    const int c = tid;
    uint32_t cc[GT / 16];
    uint16_t c16[4];
    uint64_t keep = 0;
    for (int t = 0; t < GT; ++t) keep |= (uint64_t)(((ws.rbits[t * NWD + c / 32] >> (c % 32)) & 1u) ^ 1u) << t;
    lloyd4_rows<GT>(&xs[0][c], XS, keep, a.iters, c16, cc);
    for (int w = 0; w < GT / 16; ++w) ws.cc[c][w] = cc[w];
    uint8_t* cbp = blk + 8 * cb2_slot(role, c);   // the codebook sits at the start of the group's first block
    for (int jj = 0; jj < 4; ++jj) {
      cbp[jj] = (uint8_t)(c16[jj] & 0xFF);
      cbp[4 + jj] = (uint8_t)(c16[jj] >> 8);
    }
  }
  // one warp per page builds its side-list
  for (int w = tid >> 5; w < kGroupPages; w += g.n >> 5)
    build_side_list_bits<D, XS>(ws.rbits + 16 * w * NWD, xs + 16 * w, blk + w * kStride + cb2_out_off(D), tid & 31);
  g.sync();
  for (int p = 0; p < kGroupPages; ++p) pack_cb2_codes_packed<D>(ws.cc, p, blk + p * kStride + cb2g_code_off(D), role, g);
  g.sync();
  for (int p = 0; p < kGroupPages; ++p) {
    const uint32_t u = (uint32_t)pt[gr * kGroupPages + p];
    uint8_t* gblk = a.pool + (((size_t)(u & 0x7FFFFFFFu) * a.Hkv + h) * 2 + role) * kStride;
    for (int i = tid; i < kStride / 16; i += g.n)
      reinterpret_cast<uint4*>(gblk)[i] = reinterpret_cast<const uint4*>(blk + p * kStride)[i];
  }
  g.sync();   // the scratch may be reused by the next call
}

// Shared memory of the standalone group kernel: the group's values, their
// outlier bits, the packed codes and the four blocks.
template <int D>
constexpr size_t group_smem_bytes() {
  return (size_t)kPage * kGroupPages * D * 4 + (size_t)kPage * kGroupPages * (D / 32) * 4 + (size_t)D * 16 +
         (size_t)kGroupPages * block_stride(kBlkCb2g, D);
}

// CB2 group format: each group of 4 pages (64 tokens) this append completes,
// from fp32 staging + the new tokens.  One CTA per (group, kv head x role,
// sequence).
template <int D>
__global__ void __launch_bounds__(128, 4) append_group_kernel(const AppendArgs a) {
  constexpr int GT = kPage * kGroupPages;
  extern __shared__ __align__(16) uint8_t gsm[];
  float(*xs)[D] = reinterpret_cast<float(*)[D]>(gsm);
  uint32_t* rbits = reinterpret_cast<uint32_t*>(gsm + GT * D * 4);
  uint32_t(*cc)[4] = reinterpret_cast<uint32_t(*)[4]>(gsm + GT * D * 4 + GT * (D / 32) * 4);
  uint8_t* blk = gsm + GT * D * 4 + GT * (D / 32) * 4 + D * 16;   // 4 blocks
  const int j = blockIdx.x, h = blockIdx.y >> 1, role = blockIdx.y & 1, b = blockIdx.z;
  const int tid = threadIdx.x;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, gr = start / GT + j;
  const bool full = gr * GT + GT <= end;   // quantize only the groups this append completes
  if (!full && j != 0) return;
  if (full) {
    const float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * GT * D;
    for (int i = tid; i < GT * (D / 8); i += blockDim.x) {
      const int t = i / (D / 8), c = 8 * (i - t * (D / 8)), pos = gr * GT + t;
      if (pos < start) {
        for (int jj = 0; jj < 8; ++jj) xs[t][c + jj] = stg[t * D + c + jj];
      } else {
        load_in8(a, role, b, pos - start, h, c, D, &xs[t][c]);
      }
    }
    group_quantize<D, D>(a, h, role, a.page_table + (size_t)b * a.ppsm, gr, xs, GroupWs<D>{rbits, cc, blk},
                         whole_cta(), false);   // ends with a barrier
  }
  if (j == 0) stage_tail(a, b, h, role, start, n, GT, D);
}

// Advance seq_lens and report skipped sequences (after every other launch read them).
__global__ void __launch_bounds__(128) append_finish_kernel(const AppendArgs a) {
  const int b = blockIdx.x;   // one CTA per sequence
  int start, n;
  const int st = seq_append_state(a, b, start, n);
  if (threadIdx.x != 0) return;
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
  if (a.fmt == KVQ_FMT_INT4_G32 || a.fmt == KVQ_FMT_FP4_E2M1_S16) {
    const bool i4 = a.fmt == KVQ_FMT_INT4_G32;
    const int es = a.in_dtype == KVQ_F32 ? 4 : 2;
    const auto kern = i4 ? append_token_kernel<kBlkInt4, D> : append_token_kernel<kBlkE2m1, D>;
    const size_t smem = i4 ? token_smem_bytes<kBlkInt4, D>(es) : token_smem_bytes<kBlkE2m1, D>(es);
    const int ppc = i4 ? token_ppc<kBlkInt4>() : token_ppc<kBlkE2m1>();
    const int groups_max = (pages_max + ppc - 1) / ppc, iters = i4 ? 1 : kTokenIters;
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    kern<<<dim3((groups_max + iters - 1) / iters, a.Hkv * 2, a.B), 256, smem, st>>>(a);
  }
  else if (a.fmt == KVQ_FMT_CB2_GROUP4) {
    constexpr size_t smem = group_smem_bytes<D>();
    if (smem > 48 * 1024) {
      const cudaError_t e =
          cudaFuncSetAttribute(append_group_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    const int groups_max = a.t_new / (kPage * kGroupPages) + 2;
    append_group_kernel<D><<<dim3(groups_max, a.Hkv * 2, a.B), 128, smem, st>>>(a);
  } else {
    append_page_kernel<D><<<grid, 128, 0, st>>>(a);
  }
  append_finish_kernel<<<a.B, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t append_launch(const AppendArgs& a, int D, cudaStream_t st) {
  return D == 64 ? append_launch_d<64>(a, st) : append_launch_d<128>(a, st);
}

// ----------------------------------------------------------------------------- fused projection + append
// K = x W_k^T and V = x W_v^T for the appended tokens, computed on the 5th
// generation tensor cores (tcgen05.mma, fp32 accumulators in tensor memory)
// and handed straight to the quantizer of the cache's format: the projected
// K/V never reach global memory ("Sub-5ms MoE Inference: Sub-Byte KV
// Quantization and Expert Pipelining at Scale", Engineering Real-Time
// Autonomous Workflows, item 1: the attention projection and the KV-cache
// write in one kernel).
//
// One CTA (512 threads) per (kv head, tile of 128 sequence positions,
// sequence) computes K and V together (N = 2 D accumulator columns).  Two
// CTAs holding neighbouring tiles of the same kv head form a cluster and share
// each MMA (tcgen05.mma.cta_group::2, M = 256): each stages its own x rows but
// only one of the two weight matrices, so a stage is 32 KB instead of 48 and
// three fit where two did (the pair's mainloop measured 1.2x the single CTA's
// rate).  The kv heads are the grid's fastest dimension, so the CTAs that read
// the same x rows run at about the same time and all but the first find them
// in L2 (measured 2-5% faster than tiles first).  Tile
// rows are whole pages (4-page groups for the CB2 group format), so each block
// is written by one CTA.  Warp 0 streams the operands with TMA (one 2-D box
// per unit of x rows, one per weight matrix; 128-byte swizzle, 64 hidden
// columns per stage) into a ring of shared-memory stages; warp 1 (of the
// pair's even CTA) issues the MMAs of each stage and commits it back to both
// producers; the other warps sleep on the accumulator's mbarrier.  The
// epilogue reads each CTA's own accumulators with tcgen05.ld into an fp32 tile
// in shared memory and runs the same per-token / per-page / per-group
// quantizers as kvq_quantize_append.  Where a cluster launch is refused, one
// CTA per tile does the same work alone (M = 128, both weight matrices).
namespace tc {
// Shared-memory matrix descriptor, K-major with 128-byte swizzle: rows of
// 128 bytes, 8-row atoms 1024 bytes apart (stride byte offset), leading byte
// offset unused (1), descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: bf16 A and B (K-major), fp32 accumulator, M x N
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accumulate) {
  asm volatile("{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem),
               "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// CTA pairs (cta_group::2): an M = 256 MMA issued by the pair's even CTA reads
// A rows 0..127 and B rows 0..N/2-1 from its own shared memory and A rows
// 128..255, B rows N/2..N-1 from the odd CTA's, at the same offsets; D rows
// 0..127 land in the even CTA's tensor memory, 128..255 in the odd CTA's.
__device__ __forceinline__ void mma_pair(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accumulate) {
  asm volatile("{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem),
               "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate));
}
// Arrives on the mbarrier at `bar`'s offset in both CTAs of the pair once the
// issuing thread's earlier MMAs are complete.
__device__ __forceinline__ void commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((unsigned short)3)
      : "memory");
}
// Shared-memory address of the same location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 fp32 columns of the calling warp's 32 tensor-memory lanes.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
// 2-D TMA load of one box (x = column in elements, y = row; rows outside the
// tensor read as zeros) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same into this CTA's shared memory, completing on the mbarrier at
// cluster address `bar` (the pair's even CTA's).
__device__ __forceinline__ void tma2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
}  // namespace tc

// Fused projection plan: a tile is kPM rows (sequence positions, whole units
// of U rows: pages, or 4-page groups for the CB2 group format) x N = 2 D
// columns (K then V of one kv head) in TMEM; the hidden dimension streams
// through S stages of kPK columns (A: kPM rows, B: N / CG rows, 128 bytes
// each).  CG = 2: two CTAs of a cluster share each MMA (M = 256, the two
// tiles' rows), and each stages one of the two weight matrices.
enum { kProjInt4 = 0, kProjE2m1 = 1, kProjPage = 2, kProjGroup = 3 };
constexpr int kPM = 128, kPK = 64, kPThreads = 512;

template <int KIND, int D, int CG = 1>
struct ProjPlan {
  static constexpr int U = KIND == kProjGroup ? kPage * kGroupPages : kPage;  // rows of one unit
  static constexpr int SPT = kPM / U;                                         // units per tile
  static constexpr int NB = KIND == kProjGroup ? 2 : 4;                       // unit groups working at once
  static constexpr int GS = kPThreads / NB;                                   // threads per unit group
  static constexpr int N = 2 * D;                                             // TMEM columns: K | V
  static constexpr int XS = D + 4;  // row stride of the fp32 tile: rows start 4 banks apart
  static constexpr int S = CG == 2 ? (D == 128 ? 3 : 4) : (D == 128 ? 2 : 3);   // operand stages
  static constexpr int A_BYTES = kPM * kPK * 2, B_BYTES = N / CG * kPK * 2, STAGE = A_BYTES + B_BYTES;
  // a unit group's scratch: the block (per-token formats); the block, mask and
  // codes, and per-warp partials (pages); the 4 blocks and 2-bit codes (groups)
  static constexpr int WS = KIND == kProjInt4   ? block_stride(kBlkInt4, D)
                          : KIND == kProjE2m1   ? block_stride(kBlkE2m1, D)
                          : KIND == kProjPage   ? page_blk_bytes<D>() + 32 * D + 64
                                                : kGroupPages * block_stride(kBlkCb2g, D) + 16 * D;
  static constexpr int WSR = (WS + 127) / 128 * 128;
  static constexpr int EPI = kPM * XS * 4 + NB * WSR;   // the epilogue's fp32 tile and scratch
  static constexpr int R0 = S * STAGE > EPI ? S * STAGE : EPI;
  static constexpr int SMEM = 1024 + R0 + kPM * 4 + kPM * D / 8 + (2 * S + 1) * 8 + 16;   // 1024: alignment slack
};

#define KVQ_PLAN_FITS(K, D_)                                                                          \
  static_assert(ProjPlan<K, D_>::SMEM <= 227 * 1024 && ProjPlan<K, D_>::N <= 256 &&                     \
                    ProjPlan<K, D_>::STAGE % 1024 == 0 && ProjPlan<K, D_>::A_BYTES % 1024 == 0 &&      \
                    ProjPlan<K, D_, 2>::SMEM <= 113 * 1024 && ProjPlan<K, D_, 2>::STAGE % 1024 == 0,   \
                "fused projection plan does not fit")
KVQ_PLAN_FITS(kProjInt4, 64);
KVQ_PLAN_FITS(kProjInt4, 128);
KVQ_PLAN_FITS(kProjE2m1, 64);
KVQ_PLAN_FITS(kProjE2m1, 128);
KVQ_PLAN_FITS(kProjPage, 64);
KVQ_PLAN_FITS(kProjPage, 128);
KVQ_PLAN_FITS(kProjGroup, 64);
KVQ_PLAN_FITS(kProjGroup, 128);
#undef KVQ_PLAN_FITS

// Two CTAs per SM (64 registers a thread, a few spilled): one CTA's
// quantization epilogue then runs beside the other's MMAs; one CTA per SM
// measured 1.1-1.7x slower on every format.
template <int KIND, int D, int CG>
__global__ void __launch_bounds__(kPThreads, 2) project_append_kernel(const __grid_constant__ ProjArgs p) {
  using P = ProjPlan<KIND, D, CG>;
  constexpr int U = P::U, SPT = P::SPT, NB = P::NB, GS = P::GS, N = P::N, XS = P::XS, S = P::S;
  extern __shared__ __align__(1024) uint8_t psm_raw[];
  const AppendArgs& a = p.a;
  // grid (Hkv, tiles, B); pairs: (2 Hkv, tile pairs, B) in clusters of two
  // along x, the cluster's CTAs holding tiles 2y and 2y + 1 of kv head x / 2
  const int h = CG == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int tile = CG == 2 ? 2 * (int)blockIdx.y + (int)(blockIdx.x & 1) : (int)blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int start, n;
  if (seq_append_state(a, b, start, n) != kSeqOk) return;
  const int end = start + n, first = start / U, last = (end - 1) / U, nu = last - first + 1;
  const int32_t* pt = a.page_table + (size_t)b * a.ppsm;
  // Unit in slot s of tile t, or -1.  Tile 0 holds both the first unit
  // (which reads the staged rows) and the last (which writes them), so no
  // other CTA touches this sequence's staging.
  auto unit_at = [&](int t, int s) -> int {
    if (nu <= SPT) return t == 0 && s < nu ? first + s : -1;
    if (t == 0) return s < SPT - 1 ? first + s : last;
    const int u = first + (SPT - 1) + SPT * (t - 1) + s;
    return u < last ? u : -1;
  };
  auto unit_of = [&](int s) { return unit_at(tile, s); };
  // CTA pairs: cluster rank = tile & 1; a CTA without units still stages its
  // weight half for its partner
  const uint32_t rank = CG == 2 ? tc::cluster_rank() : 0u;
  const int peer_tile = tile ^ 1;
  const bool active = unit_of(0) >= 0;
  if (!active && (CG == 1 || unit_at(peer_tile, 0) < 0)) return;   // both CTAs of a pair leave together

  // 1024-byte aligned base: the swizzled stages need it
  uint8_t* psm = psm_raw + (((smem_u32(psm_raw) + 1023u) & ~1023u) - smem_u32(psm_raw));
  float(*xs)[XS] = reinterpret_cast<float(*)[XS]>(psm);   // the fp32 tile, once the stages are done
  uint8_t* ws = psm + kPM * XS * 4;
  int* rowtok = reinterpret_cast<int*>(psm + P::R0);
  uint32_t* rbits = reinterpret_cast<uint32_t*>(rowtok + kPM);   // [kPM][D / 32] outlier decisions of the tile's rows
  uint64_t* full = reinterpret_cast<uint64_t*>(rbits + kPM * D / 32);   // [S]: a stage's bytes have landed
  uint64_t* empty = full + S;                                    // [S]: a stage's MMAs are done
  uint64_t* done = empty + S;                                    // every MMA is done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);

  for (int r = tid; r < kPM; r += kPThreads) {
    const int u = unit_of(r / U), pos = u * U + r % U;
    rowtok[r] = u >= 0 && pos >= start && pos < end ? pos - start : -1;
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    if constexpr (CG == 2) {   // one warp of each CTA of the pair, together
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)), "r"(N)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)), "r"(N)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc::fence_before();
  if constexpr (CG == 2) tc::cluster_sync();   // the partner's barriers are initialised before any copy
  else __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const int nk = (p.hidden + kPK - 1) / kPK;
  bool ok = true;

  if (tid == 0) {
    // producer: stage kc = the x rows of every unit of the tile (one box per
    // unit; rows of other sequences or past the end are never used) and the
    // K | V weight rows of head h, hidden columns [kPK kc, kPK kc + kPK)
    int nvalid = 0, nvalid_peer = 0;
    for (int s = 0; s < SPT; ++s) {
      nvalid += unit_of(s) >= 0;
      nvalid_peer += CG == 2 && unit_at(peer_tile, s) >= 0;
    }
    // pairs: the even CTA's barrier counts the bytes of both CTAs' copies
    const uint32_t bytes = CG == 2 ? (uint32_t)((nvalid + nvalid_peer) * U * kPK * 2 + 2 * P::B_BYTES)
                                   : (uint32_t)(nvalid * U * kPK * 2 + P::B_BYTES);
    for (int kc = 0; kc < nk && ok; ++kc) {
      const int s = kc % S;
      if (kc >= S && !mbar_wait_bounded(&empty[s], (kc / S - 1) & 1, kWaitLimitNs)) ok = false;
      if (!ok) break;
      uint8_t* st = psm + s * P::STAGE;
      if constexpr (CG == 2) {
        const uint32_t fb = tc::map_rank(&full[s], 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[s], bytes);
        for (int sl = 0; sl < SPT; ++sl) {
          const int u = unit_of(sl);
          if (u >= 0) tc::tma2d_pair(st + sl * U * kPK * 2, &p.tm_x, kPK * kc, b * a.t_new + (u * U - start), fb);
        }
        tc::tma2d_pair(st + P::A_BYTES, &p.tm_w[rank], kPK * kc, h * D, fb);
      } else {
        mbar_arrive_expect_tx(&full[s], bytes);
        for (int sl = 0; sl < SPT; ++sl) {
          const int u = unit_of(sl);
          if (u >= 0) tc::tma2d(st + sl * U * kPK * 2, &p.tm_x, kPK * kc, b * a.t_new + (u * U - start), &full[s]);
        }
        tc::tma2d(st + P::A_BYTES, &p.tm_w[0], kPK * kc, h * D, &full[s]);
        tc::tma2d(st + P::A_BYTES + D * kPK * 2, &p.tm_w[1], kPK * kc, h * D, &full[s]);
      }
    }
  } else if (tid == 32 && CG == 2 && rank == 0) {
    // MMA issuer of the pair: M = 256 over both CTAs' stages, each stage
    // handed back to both producers on completion
    const uint32_t idesc = tc::idesc_bf16(2 * kPM, N);
    for (int kc = 0; kc < nk && ok; ++kc) {
      const int s = kc % S;
      if (!mbar_wait_bounded(&full[s], (kc / S) & 1, kWaitLimitNs)) { ok = false; break; }
      tc::fence_after();
      const uint32_t sa = smem_u32(psm + s * P::STAGE), sb = sa + P::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kPK / 16; ++kk)
        tc::mma_pair(tmem, tc::desc_sw128(sa + 32 * kk), tc::desc_sw128(sb + 32 * kk), idesc, (kc | kk) != 0);
      tc::commit_pair(&empty[s]);
    }
    tc::commit_pair(done);
  } else if (tid == 32 && CG == 1) {
    // MMA issuer: kPK / 16 MMAs per stage, the stage handed back on completion
    const uint32_t idesc = tc::idesc_bf16(kPM, N);
    for (int kc = 0; kc < nk && ok; ++kc) {
      const int s = kc % S;
      if (!mbar_wait_bounded(&full[s], (kc / S) & 1, kWaitLimitNs)) { ok = false; break; }
      tc::fence_after();
      const uint32_t sa = smem_u32(psm + s * P::STAGE), sb = sa + P::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kPK / 16; ++kk)
        tc::mma(tmem, tc::desc_sw128(sa + 32 * kk), tc::desc_sw128(sb + 32 * kk), idesc, (kc | kk) != 0);
      tc::commit(&empty[s]);
    }
    tc::commit(done);
  }
  // everyone: sleep until the accumulators are complete
  {
    bool got = false;
    const uint64_t t0 = global_timer_ns();
    while (!(got = mbar_try_wait_sleep(done, 0, 1000000u)))
      if (global_timer_ns() - t0 > kWaitLimitNs) break;
    ok = ok && got;
  }
  const bool all_ok = __syncthreads_and(ok) != 0;
  tc::fence_after();
  if (all_ok && active) {
    const int grp = warp / (GS / 32);
    const Grp g{tid % GS, GS, 1 + grp};
    uint8_t* gws = ws + grp * P::WSR;
    for (int role = 0; role < 2; ++role) {
      // accumulators of this role -> xs: warp w reads TMEM lanes (tile rows)
      // 32 (w % 4) .. and 32 columns from 32 (w / 4)
      const int q = warp & 3, cc = warp >> 2, r = 32 * q + lane;
      if (32 * cc < D) {
        float v[32];
        tc::ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(role * D + 32 * cc), v);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(&xs[r][32 * cc + 4 * j]) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        const int tt = rowtok[r];
        if (p.kv_out && tt >= 0) {
          float4* o = reinterpret_cast<float4*>(p.kv_out + ((((size_t)role * a.B + b) * a.t_new + tt) * a.Hkv + h) * D +
                                                32 * cc);
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      __syncthreads();
      if (KIND >= kProjPage && tile == 0) {   // the first unit's earlier tokens come from staging
        const int pre = start - first * U;
        const float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * U * D;
        for (int i = tid; i < pre * D; i += kPThreads) xs[i / D][i % D] = stg[i];
        __syncthreads();
      }
      // per-token outlier decisions of every row at once (one thread per row)
      const bool pre_bits = KIND >= kProjPage && a.fmt != KVQ_FMT_CB2_STATIC;
      if (pre_bits) {
        for (int r = tid; r < kPM; r += kPThreads) outlier_bits<D>(xs[r], a.sigma, kmax_outliers(D), rbits + r * (D / 32));
        __syncthreads();
      }
      for (int s = grp; s < SPT; s += NB) {
        const int u = unit_of(s);
        if (u < 0) continue;
        const int lo = max(start, u * U) - u * U, hi = min(end, u * U + U) - u * U;   // new rows of the unit
        const float(*xu)[XS] = xs + s * U;
        if constexpr (KIND == kProjInt4 || KIND == kProjE2m1) {
          constexpr int BF = KIND == kProjInt4 ? kBlkInt4 : kBlkE2m1, kStride = block_stride(BF, D);
          const uint32_t phys = (uint32_t)pt[u] & 0x7FFFFFFFu;
          token_block_update<BF, D, XS>(a, role, xu, lo, hi, a.pool + (((size_t)phys * a.Hkv + h) * 2 + role) * kStride,
                                        gws, g);
        } else if (u * U + U <= end) {   // the append completes the unit
          if constexpr (KIND == kProjPage) {
            constexpr int kB = page_blk_bytes<D>();
            const PageWs<D> pw{reinterpret_cast<uint8_t(*)[D]>(gws + kB), reinterpret_cast<uint8_t(*)[D]>(gws + kB + 16 * D),
                               gws, reinterpret_cast<float*>(gws + kB + 32 * D)};
            page_quantize<D, XS>(a, h, role, (uint32_t)pt[u], xu, pw, g, pre_bits ? rbits + s * U * (D / 32) : nullptr);
          } else {
            constexpr int kB = kGroupPages * block_stride(kBlkCb2g, D);
            const GroupWs<D> gw{rbits + s * U * (D / 32), reinterpret_cast<uint32_t(*)[4]>(gws + kB), gws};
            group_quantize<D, XS>(a, h, role, pt, u, xu, gw, g, true);
          }
        } else {   // the final partial unit: its new rows wait in staging
          float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * U * D;
          for (int i = g.tid; i < (hi - lo) * D; i += g.n) {
            const int t = lo + i / D, c = i % D;
            stg[t * D + c] = xu[t][c];
          }
        }
      }
      __syncthreads();
    }
  } else if (tid == 0 && !all_ok) {
    atomicOr(a.status, KVQ_STATUS_TIMEOUT);
  }
  tc::fence_before();
  if constexpr (CG == 2) {   // both CTAs are done with their tensor memory and the partner's stages
    tc::cluster_sync();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(N) : "memory");
  } else {
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(N) : "memory");
  }
  if (tid == 0 && all_ok) {   // after a timeout a late arrival may still be pending: leave them
    for (int s = 0; s < S; ++s) {
      mbar_inval(&full[s]);
      mbar_inval(&empty[s]);
    }
    mbar_inval(done);
  }
}

// ----------------------------------------------------------------------------- one-token fused projection
// A one-token append (decode time) has one row per sequence: as a 128-row
// tcgen05 tile it would stream a head's whole weight for each sequence.  Here
// the rows of up to 16 sequences share one pass over the weights, the hidden
// dimension is split across the CTAs of a thread-block cluster (each streams
// its slice of the head's K | V weight rows straight from HBM into mma.sync
// fragments), the partial sums meet in distributed shared memory in rank
// order, and each (sequence, K|V) row is then quantized by one thread group of
// the cluster exactly as in the tile kernel's epilogue.
namespace small {
constexpr int kMaxRows = 32;   // sequences per cluster: 16 (two n8 tiles) or 32 (four)
constexpr int kThreads = 256;  // 8 warps; two 128-thread groups in the epilogue
constexpr int kMaxSlice = 1024;   // hidden columns one CTA stages (R rows of bf16: 32 or 64 KB)

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// fp32 at shared address `a` of cluster CTA `rank`
__device__ __forceinline__ float ld_cluster_f32(uint32_t a, uint32_t rank) {
  uint32_t r;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Rows of one quantization unit and the epilogue scratch of one thread group;
// R sequences per cluster.
template <int KIND, int D, int R>
struct Plan {
  static constexpr int U = KIND == kProjGroup ? kPage * kGroupPages : kPage;
  static constexpr int XS = D + 4;
  static constexpr int XB = U * XS * 4;   // the unit's fp32 rows
  static constexpr int WS = KIND == kProjInt4   ? block_stride(kBlkInt4, D)
                          : KIND == kProjE2m1   ? block_stride(kBlkE2m1, D)
                          : KIND == kProjPage   ? page_blk_bytes<D>() + 32 * D + 64
                                                : kGroupPages * block_stride(kBlkCb2g, D) + U * (D / 32) * 4 + D * 16;
  static constexpr int EW = (XB + WS + 127) / 128 * 128;
  static constexpr int PART = R * 2 * D * 4;   // fp32 partial sums [row][K | V channel]
  // weight ring: a stage is RK hidden columns of the CTA's 2D weight rows; a
  // thread copies its own 16-byte pieces and reads back only those
  static constexpr int MPW = 2 * D / 16 / 8, RK = 64, NSTG = D == 128 ? 4 : 6;
  static constexpr int WSTG = (RK / 32) * MPW * 2 * 512, STAGE = 8 * WSTG, RING = NSTG * STAGE;
  static constexpr int smem(int slice) {
    return PART + (R * slice * 2 + RING > 2 * EW ? R * slice * 2 + RING : 2 * EW) + 4 * R;
  }
};

static_assert(Plan<kProjGroup, 128, kMaxRows>::smem(kMaxSlice) <= 227 * 1024 &&
                  Plan<kProjPage, 128, kMaxRows>::smem(kMaxSlice) <= 227 * 1024 &&
                  Plan<kProjInt4, 128, kMaxRows>::smem(kMaxSlice) <= 227 * 1024 &&
                  Plan<kProjGroup, 64, kMaxRows>::smem(kMaxSlice) <= 227 * 1024,
              "one-token projection plan does not fit");

template <int KIND, int D, int R>
__global__ void __launch_bounds__(kThreads, 1) project_one_kernel(const ProjArgs p, int slice) {
  using P = Plan<KIND, D, R>;
  constexpr int U = P::U, XS = P::XS, N = 2 * D;
  extern __shared__ __align__(128) uint8_t osm[];
  const AppendArgs& a = p.a;
  float(*part)[N] = reinterpret_cast<float(*)[N]>(osm);
  uint8_t* region = osm + P::PART;   // x slice and weight ring, then the epilogue scratch
  int* rstart = reinterpret_cast<int*>(osm + P::smem(slice) - 4 * R);   // [R], -1 = skip
  const uint32_t rank = cluster_rank();
  const int h = blockIdx.y, b0 = blockIdx.z * R;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q4 = lane & 3;

  // partial[row][oc] = sum over this slice of x[row][k] * W[oc][k].  The
  // A fragment (16 output channels x 16 k) and the B fragment (16 k x 8
  // rows) of lane (g, q) take the same 8 consecutive k of a 32-column step
  // from one 16-byte piece each: k order inside a step is permuted alike on
  // both sides, so the products pair up.  The weights stream through a ring
  // of cp.async stages (nothing held in registers while in flight).
  constexpr int MPW = P::MPW, RK = P::RK, NSTG = P::NSTG;
  const size_t k0 = (size_t)rank * slice;
  const __nv_bfloat16* wrow[MPW][2];
#pragma unroll
  for (int m = 0; m < MPW; ++m) {
    const int oc = 16 * (warp * MPW + m), role = oc / D, c = oc % D;
    wrow[m][0] = p.w[role] + (size_t)(h * D + c + g) * p.hidden + k0 + 8 * q4;
    wrow[m][1] = wrow[m][0] + (size_t)8 * p.hidden;
  }
  __nv_bfloat16* xsl = reinterpret_cast<__nv_bfloat16*>(region);
  const uint32_t ring_s = smem_u32(region + R * slice * 2) + warp * P::WSTG + 16 * lane;
  const int nst = slice / RK;
  auto issue = [&](int st) {
    if (st < nst) {
      const uint32_t d = ring_s + (st % NSTG) * P::STAGE;
#pragma unroll
      for (int u = 0; u < RK / 32; ++u)
#pragma unroll
        for (int m = 0; m < MPW; ++m)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) cp_async16(d + ((u * MPW + m) * 2 + hf) * 512, wrow[m][hf] + st * RK + 32 * u);
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int st = 0; st < NSTG - 1; ++st) issue(st);

  // x[b][0][rank * slice ...] of the tile's rows
  for (int i = tid; i < R * slice / 8; i += kThreads) {
    const int r = i / (slice / 8), c = 8 * (i - r * (slice / 8));
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (b0 + r < a.B) v = *reinterpret_cast<const uint4*>(p.x + (size_t)(b0 + r) * a.t_new * p.hidden + k0 + c);
    *reinterpret_cast<uint4*>(xsl + r * slice + c) = v;
  }
  __syncthreads();
  // which rows append a token (one thread per row; every CTA of the cluster
  // decides the same; read only after the cluster barrier below): the first
  // warp takes these dependent loads while its copies are in flight
  if (tid < R) {
    int start = -1, n = 0;
    const bool ok = b0 + tid < a.B && seq_append_state_1(a, b0 + tid, start, n) == kSeqOk;
    rstart[tid] = ok ? start : -1;
  }

  constexpr int NT = R / 8;   // n8 tiles of rows
  const int ntl = min(NT, (a.B - b0 + 7) / 8);   // the ones holding a sequence
  float acc[MPW][NT][4];
#pragma unroll
  for (int m = 0; m < MPW; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[m][nt][0] = acc[m][nt][1] = acc[m][nt][2] = acc[m][nt][3] = 0.f;
  const uint32_t xa = smem_u32(xsl) + 2 * (g * slice + 8 * q4);
  auto step = [&](int kk, const uint4 (&wa)[MPW], const uint4 (&wb)[MPW]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt > 0 && nt >= ntl) break;   // uniform
      const uint4 x = lds128(xa + 2 * (8 * nt * slice + kk));
#pragma unroll
      for (int m = 0; m < MPW; ++m) {
        mma_bf16(acc[m][nt], wa[m].x, wb[m].x, wa[m].y, wb[m].y, x.x, x.y);
        mma_bf16(acc[m][nt], wa[m].z, wb[m].z, wa[m].w, wb[m].w, x.z, x.w);
      }
    }
  };
#pragma unroll 1
  for (int st = 0; st < nst; ++st) {
    issue(st + NSTG - 1);
    cp_async_wait<NSTG - 1>();   // stage st has landed (groups complete in order)
    const uint32_t d = ring_s + (st % NSTG) * P::STAGE;
#pragma unroll
    for (int u = 0; u < RK / 32; ++u) {
      uint4 wa[MPW], wb[MPW];
#pragma unroll
      for (int m = 0; m < MPW; ++m) {
        wa[m] = lds128(d + ((u * MPW + m) * 2) * 512);
        wb[m] = lds128(d + ((u * MPW + m) * 2 + 1) * 512);
      }
      step(st * RK + 32 * u, wa, wb);
    }
  }
  cp_async_wait<0>();
  if (slice % RK) {   // a last 32-column step
    const int kk = nst * RK;
    uint4 wa[MPW], wb[MPW];
#pragma unroll
    for (int m = 0; m < MPW; ++m) {
      wa[m] = ldg_stream(wrow[m][0] + kk);
      wb[m] = ldg_stream(wrow[m][1] + kk);
    }
    step(kk, wa, wb);
  }
  // accumulator (channel g | g + 8 of the m tile, row 2q | 2q + 1 of the n tile)
#pragma unroll
  for (int m = 0; m < MPW; ++m) {
    const int oc = 16 * (warp * MPW + m) + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = 8 * nt + 2 * q4;
      part[r][oc] = acc[m][nt][0];
      part[r + 1][oc] = acc[m][nt][1];
      part[r][oc + 8] = acc[m][nt][2];
      part[r + 1][oc + 8] = acc[m][nt][3];
    }
  }
  cluster_sync();   // every partial is visible cluster-wide; the x slices are dead

  // units (row, K|V): unit 2 rank + grp, then + 2 * cluster size ...
  const int grp = tid >> 7;
  const Grp gp{tid & 127, 128, 1 + grp};
  uint8_t* ew = region + grp * P::EW;
  float(*xs)[XS] = reinterpret_cast<float(*)[XS]>(ew);
  uint8_t* ws = ew + P::XB;
  const int nrank = (int)gridDim.x;
  // channel c of row r, role: the sum over the cluster's slices in rank order
  // (all remote loads in flight at once), also written to kv_out
  auto row_sum = [&](int r, int role, int c) {
    const uint32_t ad = smem_u32(&part[r][role * D + c]);
    float pv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) pv[q] = q < nrank ? ld_cluster_f32(ad, (uint32_t)q) : 0.f;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (q < nrank) v += pv[q];
    if (p.kv_out) p.kv_out[((((size_t)role * a.B + b0 + r) * a.t_new) * a.Hkv + h) * D + c] = v;
    return v;
  };
  if constexpr (KIND == kProjPage || KIND == kProjGroup) {
    // rows that only wait in staging (their unit is not complete): the whole
    // CTA at once, rows rank, rank + cluster size, ...
    const int nr = (R - (int)rank + nrank - 1) / nrank;
    for (int i = tid; i < nr * 2 * D; i += kThreads) {
      const int c = i % D, role = (i / D) & 1, r = (int)rank + nrank * (i / (2 * D)), pos = rstart[r];
      if (pos < 0 || pos % U == U - 1) continue;
      const float v = row_sum(r, role, c);
      a.staging[((((size_t)(b0 + r) * a.Hkv + h) * 2 + role) * U + pos % U) * D + c] = v;
    }
  }
  for (int unit = 2 * (int)rank + grp; unit < 2 * R; unit += 2 * nrank) {
    const int r = unit >> 1, role = unit & 1, b = b0 + r, pos = rstart[r];
    if (pos < 0) continue;   // uniform within the group
    const int32_t* ptb = a.page_table + (size_t)b * a.ppsm;
    const int slot = pos % U;
    if ((KIND == kProjPage || KIND == kProjGroup) && slot < U - 1) continue;   // staged above
    const float v = gp.tid < D ? row_sum(r, role, gp.tid) : 0.f;
    if constexpr (KIND == kProjInt4 || KIND == kProjE2m1) {
      constexpr int BF = KIND == kProjInt4 ? kBlkInt4 : kBlkE2m1, kStride = block_stride(BF, D);
      if (gp.tid < D) xs[slot][gp.tid] = v;
      const uint32_t phys = (uint32_t)ptb[pos / U] & 0x7FFFFFFFu;
      token_block_update<BF, D, XS>(a, role, xs, slot, slot + 1, a.pool + (((size_t)phys * a.Hkv + h) * 2 + role) * kStride,
                                    ws, gp);
    } else {   // the row completes its unit
      const float* stg = a.staging + (((size_t)b * a.Hkv + h) * 2 + role) * U * D;
      for (int i = gp.tid; i < (U - 1) * D; i += gp.n) xs[i / D][i % D] = stg[i];
      if (gp.tid < D) xs[U - 1][gp.tid] = v;
      if constexpr (KIND == kProjPage) {
        constexpr int kB = page_blk_bytes<D>();
        const PageWs<D> pw{reinterpret_cast<uint8_t(*)[D]>(ws + kB), reinterpret_cast<uint8_t(*)[D]>(ws + kB + 16 * D), ws,
                           reinterpret_cast<float*>(ws + kB + 32 * D)};
        page_quantize<D, XS>(a, h, role, (uint32_t)ptb[pos / U], xs, pw, gp);
      } else {
        constexpr int kB = kGroupPages * block_stride(kBlkCb2g, D);
        const GroupWs<D> gw{reinterpret_cast<uint32_t*>(ws + kB), reinterpret_cast<uint32_t(*)[4]>(ws + kB + U * (D / 32) * 4),
                            ws};
        group_quantize<D, XS>(a, h, role, ptb, pos / U, xs, gw, gp, false);
      }
    }
    gp.sync();   // the scratch is reused by the group's next unit
  }
  cluster_sync();   // no CTA leaves while another may still read its partials
}

// Cluster size for a one-token projection of `hidden` columns: the largest of
// 16, 8, 4, 2, 1 that splits hidden into 32-column multiples of at most
// kMaxSlice columns; 0 when none does.
inline int cluster_for(int hidden) {
  for (int cs = 16; cs >= 1; cs >>= 1)
    if (hidden % (32 * cs) == 0 && hidden / cs <= kMaxSlice) return cs;
  return 0;
}

// Launches with clusters of cs CTAs; with one_wave, only when every cluster
// can be resident at once (else cudaErrorLaunchOutOfResources, nothing launched).
// `enqueued` tells whether the projection kernel itself went onto the stream:
// an error after that point must reach the caller, not start another launch.
template <int KIND, int D, int R>
cudaError_t launch_r(ProjArgs& p, int cs, bool one_wave, cudaStream_t st, bool& enqueued) {
  enqueued = false;
  const int slice = p.hidden / cs;
  const size_t smem = (size_t)Plan<KIND, D, R>::smem(slice);
  auto kern = project_one_kernel<KIND, D, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && cs > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)cs, (unsigned)p.a.Hkv, (unsigned)((p.a.B + R - 1) / R));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  e = cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (nclusters < 1 || (one_wave && (long long)nclusters < (long long)cfg.gridDim.y * cfg.gridDim.z))
    return cudaErrorLaunchOutOfResources;
  e = cudaLaunchKernelEx(&cfg, kern, p, slice);
  if (e != cudaSuccess) return e;
  enqueued = true;
  append_finish_kernel<<<p.a.B, 128, 0, st>>>(p.a);
  return cudaGetLastError();
}

// 16 sequences per cluster, or 32 (the weights streamed half as often) when
// there are more than 16.
template <int KIND, int D>
cudaError_t launch(ProjArgs& p, int cs, bool one_wave, cudaStream_t st, bool& enqueued) {
  return p.a.B > 16 ? launch_r<KIND, D, 32>(p, cs, one_wave, st, enqueued)
                    : launch_r<KIND, D, 16>(p, cs, one_wave, st, enqueued);
}
}  // namespace small

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Row-major bf16 [rows][cols] matrix, boxes of 64 columns x box_rows rows, 128-byte swizzle.
static bool encode_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows}, strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kPK, box_rows}, es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, int D>
static cudaError_t project_launch_k(ProjArgs& p, cudaStream_t st) {
  using P = ProjPlan<KIND, D>;
  if (p.a.t_new == 1) {   // one token per sequence: the cluster split-K kernel
    // the widest split (within the slice limit) whose clusters are all
    // resident at once; failing that, the widest that launches at all
    for (int pass = 0; pass < 2; ++pass)
      for (int cs = small::cluster_for(p.hidden); cs >= 1; cs >>= 1) {
        if (p.hidden % (32 * cs) || p.hidden / cs > small::kMaxSlice) break;
        bool enqueued = false;
        const cudaError_t e = small::launch<KIND, D>(p, cs, pass == 0, st, enqueued);
        if (e == cudaSuccess || enqueued) return e;   // once enqueued, never launch the projection again
        (void)cudaGetLastError();   // refused: a narrower cluster, else the tile kernel
      }
  }
  if (!encode_rows(&p.tm_x, p.x, (uint64_t)p.a.B * p.a.t_new, (uint64_t)p.hidden, (uint32_t)P::U) ||
      !encode_rows(&p.tm_w[0], p.w[0], (uint64_t)p.a.Hkv * D, (uint64_t)p.hidden, (uint32_t)D) ||
      !encode_rows(&p.tm_w[1], p.w[1], (uint64_t)p.a.Hkv * D, (uint64_t)p.hidden, (uint32_t)D))
    return cudaErrorInvalidValue;
  const int units_max = (p.a.t_new + 2 * P::U - 2) / P::U;   // units a span of t_new positions can touch
  const int tiles = (units_max + P::SPT - 1) / P::SPT;
  // CTA pairs first (clusters of two CTAs, one tile each, sharing each MMA);
  // if the pair kernel cannot launch, the one-CTA kernel
  {
    using P2 = ProjPlan<KIND, D, 2>;
    auto kern = project_append_kernel<KIND, D, 2>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P2::SMEM);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2u * (unsigned)p.a.Hkv, (unsigned)((tiles + 1) / 2), (unsigned)p.a.B);
      cfg.blockDim = dim3(kPThreads);
      cfg.dynamicSmemBytes = P2::SMEM;
      cfg.stream = st;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int nclusters = 0;
      e = cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg);
      if (e == cudaSuccess && nclusters >= 1) {
        e = cudaLaunchKernelEx(&cfg, kern, p);
        if (e != cudaSuccess) return e;
        append_finish_kernel<<<p.a.B, 128, 0, st>>>(p.a);
        return cudaGetLastError();
      }
    }
    (void)cudaGetLastError();
  }
  const cudaError_t e =
      cudaFuncSetAttribute(project_append_kernel<KIND, D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.a.Hkv, tiles, p.a.B);
  project_append_kernel<KIND, D, 1><<<grid, kPThreads, P::SMEM, st>>>(p);
  append_finish_kernel<<<p.a.B, 128, 0, st>>>(p.a);
  return cudaGetLastError();
}

template <int D>
static cudaError_t project_launch_d(ProjArgs& p, cudaStream_t st) {
  switch (p.a.fmt) {
    case KVQ_FMT_INT4_G32: return project_launch_k<kProjInt4, D>(p, st);
    case KVQ_FMT_FP4_E2M1_S16: return project_launch_k<kProjE2m1, D>(p, st);
    case KVQ_FMT_CB2_GROUP4: return project_launch_k<kProjGroup, D>(p, st);
    default: return project_launch_k<kProjPage, D>(p, st);
  }
}

cudaError_t project_append_launch(ProjArgs& p, int D, cudaStream_t st) {
  return D == 64 ? project_launch_d<64>(p, st) : project_launch_d<128>(p, st);
}

}  // namespace kvq
