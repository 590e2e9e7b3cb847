/*
 * kvq_oracle.c -- plain, slow, fp64 CPU oracle for the sub-byte quantized KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load this library.  It shares no code, header,
 * table or constant with the CUDA path; it re-derives every step from the pages:
 *
 *   [P1] "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression",
 *        section "Paradigm 2: Sub-2-Bit Non-Linear KV-Cache Quantization"
 *        (1. Dynamic Outlier Isolation; 2. Centroid Vector Quantization for
 *        Residuals; the compress_kv_head listing) and "Hardware-Kernel Fusion".
 *   [P2] "Hierarchical Token Gating and Tiered KV-Cache Paging",
 *        section "2. Entropy-Guided Tiered KV-Cache Quantization".
 *   [P3] "Sub-5ms MoE Inference: Sub-Byte KV Quantization and Expert Pipelining
 *        at Scale", section "Sub-Byte KV-Cache Quantization" (FP16 outlier tensor).
 *   [P4] "The Sub-10ms Barrier: Fusing Sparse MoE Routing with FP4 KV-Cache
 *        Quantization", section "2. FP4/INT4 KV-Cache Quantization"
 *        (block-wise asymmetric quantization, E2M1, the scale formula).
 *
 * Everything is fp64 (IEEE binary64): the quantizer's statistics and decisions
 * (outlier tests, the Lloyd-Max fit and its assignments, INT4 / 3-bit scales
 * and codes, E2M1 and FP8 scales and codes) and the attention.  Inputs are the
 * binary32 values the cache receives, converted exactly; results are rounded
 * once, to the stored format.  Reductions run in ascending index order;
 * compile with -ffp-contract=off so no multiply-add is fused.  Where the pages
 * leave a step open, the reading taken is stated next to the code.
 *
 * Every function here is pinned by tests/test_oracle_*.py against something
 * other than itself (library routines, closed forms, brute force, invariants).
 * Pinning status per function is listed in the tests; nothing here is
 * "parity unpinned" except the byte layout of a block, which is a definition
 * of this library (not of the pages) and is pinned only as a bijection.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Scalar number formats.                                                     */
/*                                                                            */
/* One generic routine rounds a real number (given as a double) to a binary   */
/* floating format with `mbits` mantissa bits, exponent bias `bias` and a     */
/* smallest normal exponent emin = 1 - bias, using round-to-nearest-even,     */
/* exactly as IEEE 754 defines it: pick the binade of |v|, clamp it to emin   */
/* (subnormals share the emin quantum), divide by the quantum (exact: a power */
/* of two), round the quotient to the nearest integer with ties to even       */
/* (rint in the default rounding mode), multiply back.                        */
/* ------------------------------------------------------------------------- */

static double round_to_format(double a /* >= 0, finite */, int mbits, int emin)
{
    if (a == 0.0) return 0.0;
    int ex;
    frexp(a, &ex);               /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;              /* a in [2^e, 2^(e+1)) */
    if (e < emin) e = emin;      /* subnormal range uses the emin quantum */
    double quantum = ldexp(1.0, e - mbits);
    double r = rint(a / quantum);    /* exact division; rint = ties-to-even */
    return r * quantum;
}

/* Bits of a rounded, representable magnitude v in the format. */
static uint32_t magnitude_bits(double v, int mbits, int bias)
{
    int emin = 1 - bias;
    if (v == 0.0) return 0;
    if (v < ldexp(1.0, emin)) {                 /* subnormal: exponent field 0 */
        double m = v / ldexp(1.0, emin - mbits);
        return (uint32_t)m;
    }
    int ex;
    frexp(v, &ex);
    int e = ex - 1;
    double m = v / ldexp(1.0, e - mbits) - ldexp(1.0, mbits);
    return ((uint32_t)(e + bias) << mbits) | (uint32_t)m;
}

static double bits_to_magnitude(uint32_t bits, int mbits, int bias)
{
    uint32_t ef = bits >> mbits, mf = bits & ((1u << mbits) - 1u);
    if (ef == 0) return ldexp((double)mf, 1 - bias - mbits);
    return ldexp((double)((1u << mbits) + mf), (int)ef - bias - mbits);
}

/* IEEE binary16: 5 exponent bits, bias 15, 10 mantissa bits, overflow -> inf. */
EXPORT uint16_t or_fp16_encode(double v)
{
    uint16_t s = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return 0x7E00u;
    double r = isinf(a) ? INFINITY : round_to_format(a, 10, -14);
    if (r > 65504.0) return s | 0x7C00u;
    return s | (uint16_t)magnitude_bits(r, 10, 15);
}

EXPORT double or_fp16_decode(uint16_t h)
{
    double sgn = (h & 0x8000u) ? -1.0 : 1.0;
    uint32_t ef = (h >> 10) & 0x1Fu;
    if (ef == 0x1F) return (h & 0x3FFu) ? NAN : sgn * INFINITY;
    return sgn * bits_to_magnitude(h & 0x7FFFu, 10, 15);
}

/* OCP FP8 E4M3 ("e4m3fn", the torch.float8_e4m3fn format named by [P1]'s
 * listing): bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, the
 * largest finite magnitude is 448.  Conversion saturates to +-448 (satfinite);
 * NaN is never produced from a finite input. */
EXPORT uint8_t or_e4m3_encode(double v)
{
    uint8_t s = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    double r = isinf(a) ? 448.0 : round_to_format(a, 3, -6);
    if (r > 448.0) r = 448.0;
    return s | (uint8_t)magnitude_bits(r, 3, 7);
}

EXPORT double or_e4m3_decode(uint8_t b)
{
    double sgn = (b & 0x80u) ? -1.0 : 1.0;
    if ((b & 0x7Fu) == 0x7Fu) return NAN;
    return sgn * bits_to_magnitude(b & 0x7Fu, 3, 7);
}

/* FP4 E2M1 as [P4] defines it (1 sign, 2 exponent, 1 mantissa bit): bias 1,
 * magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; saturating at 6. */
EXPORT uint8_t or_e2m1_encode(double v)
{
    uint8_t s = signbit(v) ? 0x8u : 0u;
    double a = fabs(v);
    double r = isinf(a) ? 6.0 : round_to_format(a, 1, 0);
    if (r > 6.0) r = 6.0;
    return s | (uint8_t)magnitude_bits(r, 1, 1);
}

EXPORT double or_e2m1_decode(uint8_t b)
{
    double sgn = (b & 0x8u) ? -1.0 : 1.0;
    return sgn * bits_to_magnitude(b & 0x7u, 1, 1);
}

/* bfloat16 -> real: the top 16 bits of an IEEE binary32. */
EXPORT double or_bf16_decode(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* The binary32 value nearest to the fp64 quotient a / b (one rounding to
 * binary32 of the fp64 quotient; 53 >= 2*24 + 2 bits, so for binary32 inputs
 * this double rounding equals a single correct rounding of the exact
 * quotient). */
static float f32_of_quotient(float a, float b) { return (float)((double)a / (double)b); }

/* ------------------------------------------------------------------------- */
/* Outlier isolation ([P1] "1. Dynamic Outlier Isolation" and the             */
/* compress_kv_head listing; [P3] outlier channels; [P4] "Channel-Outlier     */
/* Isolation").  For one vector x[0..n) (a token's head vector, or one        */
/* 32-value group for INT4), in fp64:                                         */
/*   mu  = (sum x) / n                    ascending index                     */
/*   s   = sqrt( sum (x - mu)^2 / (n-1) ) unbiased, as torch's .std()         */
/*   x_i is an outlier  iff  |x_i - mu| > sigma * s   (strict, as the listing)*/
/* Reading: sigma = 3 (the pages print 3.5 in the text and "> 3 Sigma" in the */
/* flowchart; the workloads use 3).  Since k outliers need                    */
/* k*sigma^2*s^2 < (n-1)*s^2, at most kmax = ceil((n-1)/sigma^2)-1 exist for  */
/* sigma >= 3; if rounding ever produced more, only the kmax lowest indices   */
/* are kept (this never happens on real data; stated so both sides agree).    */
/* ------------------------------------------------------------------------- */

EXPORT int or_kmax(int n) /* capacity at sigma = 3 */
{
    int k = (n - 1 + 8) / 9 - 1;     /* ceil((n-1)/9) - 1 */
    return k < 0 ? 0 : k;
}

EXPORT int or_outlier_mask(const float* x, int n, double sigma, int kmax, uint8_t* mask)
{
    double sum = 0.0;
    for (int i = 0; i < n; ++i) sum += (double)x[i];
    double mu = sum / (double)n;
    double ss = 0.0;
    for (int i = 0; i < n; ++i) {
        double d = (double)x[i] - mu;
        ss += d * d;
    }
    double s = sqrt(ss / (double)(n - 1));
    double thr = sigma * s;
    int k = 0;
    for (int i = 0; i < n; ++i) {
        int out = fabs((double)x[i] - mu) > thr;
        if (out && k >= kmax) out = 0;
        mask[i] = (uint8_t)out;
        k += out;
    }
    return k;
}

/* ------------------------------------------------------------------------- */
/* 2-bit non-uniform codebook ([P1] "2. Centroid Vector Quantization for      */
/* Residuals": a 4-centroid codebook fitted by k-means; the listing starts    */
/* the centroids at linspace(min, max, 4) and assigns by argmin distance).    */
/* In one dimension k-means is the Lloyd-Max iteration (fp64):                */
/*   c = (mn, mn+h, mn+2h, mx) with h = (mx-mn)/3                             */
/*   repeat up to `iters` times:                                              */
/*     a = nearest-centroid assignment (ties -> lower index, argmin's rule)   */
/*     stop if a equals the previous assignment                               */
/*     c_j = mean of the values assigned to j (ascending order); an empty    */
/*           cell keeps its centroid                                          */
/*   centroids are stored as fp16 (one round-to-nearest-even of the fp64      */
/*   value); final code = nearest fp16 centroid, ties -> lower index.         */
/* n == 0 (every value of the channel is an outlier) gives four zero          */
/* centroids.  Returns the number of assignment passes made.                  */
/* ------------------------------------------------------------------------- */

static int nearest4(double v, const double* c)
{
    int best = 0;
    double bd = fabs(v - c[0]);
    for (int j = 1; j < 4; ++j) {
        double d = fabs(v - c[j]);
        if (d < bd) { bd = d; best = j; }
    }
    return best;
}

EXPORT int or_lloyd4(const float* v, int n, int iters, double* c_out, uint16_t* c16_out, uint8_t* codes_out)
{
    double c[4] = {0.0, 0.0, 0.0, 0.0};
    int passes = 0;
    if (n > 0) {
        double mn = v[0], mx = v[0];
        for (int i = 1; i < n; ++i) {
            if (v[i] < mn) mn = v[i];
            if (v[i] > mx) mx = v[i];
        }
        double h = (mx - mn) / 3.0;
        c[0] = mn;
        c[1] = mn + h;
        c[2] = mn + 2.0 * h;
        c[3] = mx;
        uint8_t prev[64], a[64];
        int have_prev = 0;
        for (int it = 0; it < iters; ++it) {
            for (int i = 0; i < n; ++i) a[i] = (uint8_t)nearest4((double)v[i], c);
            ++passes;
            if (have_prev && memcmp(a, prev, (size_t)n) == 0) break;
            for (int j = 0; j < 4; ++j) {
                double sum = 0.0;
                int cnt = 0;
                for (int i = 0; i < n; ++i)
                    if (a[i] == j) { sum += (double)v[i]; ++cnt; }
                if (cnt > 0) c[j] = sum / (double)cnt;
            }
            memcpy(prev, a, (size_t)n);
            have_prev = 1;
        }
    }
    double c16[4];
    for (int j = 0; j < 4; ++j) {
        uint16_t h = or_fp16_encode(c[j]);
        if (c16_out) c16_out[j] = h;
        c16[j] = or_fp16_decode(h);
        if (c_out) c_out[j] = c[j];
    }
    if (codes_out)
        for (int i = 0; i < n; ++i) codes_out[i] = (uint8_t)nearest4((double)v[i], c16);
    return passes;
}

/* ------------------------------------------------------------------------- */
/* Block layout (a definition of this library, not of the pages).             */
/*                                                                            */
/* A block is one (page of 16 tokens, kv head, K-or-V) slice of the cache.    */
/* Element (t, c) -- token t in 0..15, channel c in 0..D-1 -- is stored at a  */
/* "fragment position" (lane in 0..31, step s = c/16, slot k in 0..7) that    */
/* depends on the role (K or V).  With j = c % 16:                            */
/*   K: lane = 4*(t%8) + (j%8)/2,  k = 2*((t/8) + 2*(j/8)) + j%2              */
/*   V: lane = 4*(j%8) + (t%8)/2,  k = 2*((j/8) + 2*(t/8)) + t%2              */
/* Per-format byte layouts (D = head_dim, NS = D/16 steps):                   */
/*  INT4_G32  codes  [0, 8D)     lane-major, 4*NS B/lane, step s = u32 at 4s, */
/*                               slot k = bits 4k..4k+3                       */
/*            scale/zero at 8D   [t][D/32] x {S fp16, m fp16}                 */
/*            counts    at 10D   u8[16] outliers per token                    */
/*            channels  at 10D+16        u8 [16][cap], cap = 3*D/32           */
/*            values    at 10D+16+16cap  fp16 [16][cap]                       */
/*  E2M1_S16  codes  [0, 8D)     as INT4 (slot k = e2m1 nibble)               */
/*            scales at 8D       e4m3 [NS][16] (step-major, token minor)      */
/*  CB2       codes  [0, 4D)     lane-major, 2*NS B/lane, step s = u16 at 2s, */
/*                               slot k = bits 4*(k%4) + 2*(k/4)              */
/*            codebook at 4D     8 B per slot sigma(c): u32 L (byte j = low   */
/*                               byte of fp16 centroid j), u32 H (high bytes) */
/*                               K: sigma(c) = c                              */
/*                               V: sigma(c) = 16*(c/16) + 2*(c%8) + (c%16)/8 */
/*            outliers at 12D    u8 n_ch (channels holding an outlier),       */
/*                               u8 total (outliers), 2 zero bytes; then n_ch */
/*                               20-byte records, channels ascending:         */
/*                               {u8 channel, 0, u16 token mask, u8 value[16]}*/
/*                               value[t] = e4m3 of the outlier at token t,   */
/*                               0 where t is not an outlier of the channel   */
/*                               (record i at 4 + 20*i; K and V alike)        */
/*  CB2 static codes, codebook   as CB2; the static channels have code 0 and  */
/*  (f4)                         an all-zero codebook                         */
/*            at 12D             u8 n_s, u8 channel[n_s] (ascending), zeros  */
/*                               to 12D + 16                                  */
/*            at 12D + 16        fp16 value(i, t) at 12D + 16 + 32*i + 2*t of */
/*                               static channel i (K and V alike)             */
/*  ASYM3     codes  [0, 6D)     3-bit codes at the fragment positions, in    */
/*  (f3)                         two planes: low 2 bits in u32 words X, lane  */
/*                               l's word j (steps 2j, 2j+1) at 4*(l*NS/2+j), */
/*                               slot k of step s at bit 8*(s%2) + 16*(k%2) + */
/*                               2*(k/2); high bit in u32 words Y at 4D +      */
/*                               4*(l*NS/4 + s/4), bit 4*(s%4) + 16*(k%2) +   */
/*                               k/2                                          */
/*            S at 6D, m at 8D   fp16 per channel c at +2*rho(c):             */
/*                               x = fp16(q*S + m); K: rho(c) = 16*(c/16) +   */
/*                               4*((c%8)/2) + 2*((c%16)/8) + c%2, V: rho(c)  */
/*                               = 16*(c/16) + 2*(c%8) + (c%16)/8             */
/*            outliers at 10D    as CB2's side-list (records at 10D + 4 + 20i)*/
/*  CB2 group codebook [0, 8D)   as CB2's codebook, fitted over a group of 4  */
/*  (f1)                         pages (64 tokens); only the group's first    */
/*                               page holds it (zeros in the other three)     */
/*            codes  [8D, 12D)   as CB2's codes                               */
/*            outliers at 12D    as CB2's side-list (per page)                */
/*  FP8 tier  codes  [0, 16D)    lane-major, 8*NS B/lane, step s at 8s,       */
/*                               slot k = byte k (e4m3)                       */
/*            scale at 16D       fp32                                         */
/* Bytes not listed are zero.  Strides are rounded up to 128 B ([P4] "Align   */
/* Page Sizes with Memory Bus Lines").                                        */
/* ------------------------------------------------------------------------- */

enum { OR_INT4 = 0, OR_E2M1 = 1, OR_CB2 = 2, OR_FP8 = 3, OR_CB2S = 4, OR_A3 = 5, OR_CB2G = 6 };
enum { OR_GROUP = 4 };   /* pages per CB2 group codebook */
enum { OR_MAX_STATIC = 8 };

static int round128(int x) { return (x + 127) / 128 * 128; }

EXPORT int or_block_stride(int fmt, int D)
{
    int cap = 3 * (D / 32);
    switch (fmt) {
    case OR_INT4: return round128(10 * D + 16 + 48 * cap);
    case OR_E2M1: return round128(9 * D);
    case OR_CB2:  return round128(12 * D + 4 + 20 * D);
    case OR_FP8:  return round128(16 * D + 16);
    case OR_CB2S: return round128(12 * D + 16 + 32 * OR_MAX_STATIC);
    case OR_A3:   return round128(10 * D + 4 + 20 * D);
    case OR_CB2G: return round128(12 * D + 4 + 20 * D);
    }
    return -1;
}

EXPORT void or_frag_pos(int role, int t, int c, int* lane, int* step, int* slot)
{
    int j = c % 16;
    *step = c / 16;
    if (role == 0) {
        *lane = 4 * (t % 8) + (j % 8) / 2;
        *slot = 2 * ((t / 8) + 2 * (j / 8)) + j % 2;
    } else {
        *lane = 4 * (j % 8) + (t % 8) / 2;
        *slot = 2 * ((j / 8) + 2 * (t / 8)) + t % 2;
    }
}

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void put_f32(uint8_t* p, float f) { memcpy(p, &f, 4); }
static float get_f32(const uint8_t* p) { float f; memcpy(&f, p, 4); return f; }

/* nibble (4-bit) code at element (t, c) for INT4 / E2M1 */
static void nib_set(uint8_t* blk, int D, int role, int t, int c, uint8_t code)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    int byte = 4 * (D / 16) * lane + 4 * s + k / 2;
    int sh = 4 * (k % 2);
    blk[byte] = (uint8_t)((blk[byte] & ~(0xF << sh)) | ((code & 0xF) << sh));
}
static uint8_t nib_get(const uint8_t* blk, int D, int role, int t, int c)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    int byte = 4 * (D / 16) * lane + 4 * s + k / 2;
    return (uint8_t)((blk[byte] >> (4 * (k % 2))) & 0xF);
}

/* 2-bit code at element (t, c) for CB2 */
static void cb2_code_set(uint8_t* blk, int D, int role, int t, int c, uint8_t code)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    uint8_t* w = blk + 2 * (D / 16) * lane + 2 * s;
    uint16_t v = get_u16(w);
    int bit = 4 * (k % 4) + 2 * (k / 4);
    v = (uint16_t)((v & ~(3u << bit)) | ((unsigned)(code & 3) << bit));
    put_u16(w, v);
}
static uint8_t cb2_code_get(const uint8_t* blk, int D, int role, int t, int c)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    uint16_t v = get_u16(blk + 2 * (D / 16) * lane + 2 * s);
    return (uint8_t)((v >> (4 * (k % 4) + 2 * (k / 4))) & 3u);
}

/* ASYM3 per-channel S / m position (layout above). */
static int a3_rho(int role, int c)
{
    if (role == 0) return 16 * (c / 16) + 4 * ((c % 8) / 2) + 2 * ((c % 16) / 8) + c % 2;
    return 16 * (c / 16) + 2 * (c % 8) + (c % 16) / 8;
}

/* ASYM3 3-bit codes (layout above). */
static void a3_code_set(uint8_t* blk, int D, int role, int t, int c, uint8_t q)
{
    int lane, s, k, NS = D / 16;
    or_frag_pos(role, t, c, &lane, &s, &k);
    uint8_t* x = blk + 4 * (lane * (NS / 2) + s / 2);
    uint8_t* y = blk + 4 * D + 4 * (lane * (NS / 4) + s / 4);
    int bx = 8 * (s % 2) + 16 * (k % 2) + 2 * (k / 2), by = 4 * (s % 4) + 16 * (k % 2) + k / 2;
    uint32_t vx, vy;
    memcpy(&vx, x, 4);
    memcpy(&vy, y, 4);
    vx = (vx & ~(3u << bx)) | ((uint32_t)(q & 3) << bx);
    vy = (vy & ~(1u << by)) | ((uint32_t)((q >> 2) & 1) << by);
    memcpy(x, &vx, 4);
    memcpy(y, &vy, 4);
}
static uint8_t a3_code_get(const uint8_t* blk, int D, int role, int t, int c)
{
    int lane, s, k, NS = D / 16;
    or_frag_pos(role, t, c, &lane, &s, &k);
    uint32_t vx, vy;
    memcpy(&vx, blk + 4 * (lane * (NS / 2) + s / 2), 4);
    memcpy(&vy, blk + 4 * D + 4 * (lane * (NS / 4) + s / 4), 4);
    int bx = 8 * (s % 2) + 16 * (k % 2) + 2 * (k / 2), by = 4 * (s % 4) + 16 * (k % 2) + k / 2;
    return (uint8_t)(((vx >> bx) & 3u) | (((vy >> by) & 1u) << 2));
}

static int cb2_slot(int role, int c);
/* CB2 codes / centroids relative to explicit section bases (CB2 group pages). */
static void code2_set(uint8_t* codes, int D, int role, int t, int c, uint8_t code)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    uint8_t* w = codes + 2 * (D / 16) * lane + 2 * s;
    uint16_t v = get_u16(w);
    int bit = 4 * (k % 4) + 2 * (k / 4);
    v = (uint16_t)((v & ~(3u << bit)) | ((unsigned)(code & 3) << bit));
    put_u16(w, v);
}
static uint8_t code2_get(const uint8_t* codes, int D, int role, int t, int c)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    uint16_t v = get_u16(codes + 2 * (D / 16) * lane + 2 * s);
    return (uint8_t)((v >> (4 * (k % 4) + 2 * (k / 4))) & 3u);
}
static void cent_set(uint8_t* cb, int role, int c, int j, uint16_t h)
{
    uint8_t* p = cb + 8 * cb2_slot(role, c);
    p[j] = (uint8_t)(h & 0xFF);
    p[4 + j] = (uint8_t)(h >> 8);
}
static uint16_t cent_get(const uint8_t* cb, int role, int c, int j)
{
    const uint8_t* p = cb + 8 * cb2_slot(role, c);
    return (uint16_t)(p[j] | (p[4 + j] << 8));
}

static int cb2_slot(int role, int c)
{
    if (role == 0) return c;
    return 16 * (c / 16) + 2 * (c % 8) + (c % 16) / 8;
}
static void cb2_cent_set(uint8_t* blk, int D, int role, int c, int j, uint16_t h)
{
    uint8_t* p = blk + 4 * D + 8 * cb2_slot(role, c);
    p[j] = (uint8_t)(h & 0xFF);
    p[4 + j] = (uint8_t)(h >> 8);
}
static uint16_t cb2_cent_get(const uint8_t* blk, int D, int role, int c, int j)
{
    const uint8_t* p = blk + 4 * D + 8 * cb2_slot(role, c);
    return (uint16_t)(p[j] | (p[4 + j] << 8));
}

/* e4m3 byte at element (t, c) for the FP8 tier */
static int fp8_byte(int D, int role, int t, int c)
{
    int lane, s, k;
    or_frag_pos(role, t, c, &lane, &s, &k);
    return 8 * (D / 16) * lane + 8 * s + k;
}

/* ------------------------------------------------------------------------- */
/* Per-token quantizers (INT4 group-32 and E2M1 scale-16), [P4] "Outlier      */
/* Isolation and Block-wise Quantization":                                    */
/*   q = Round(Clamp(x/S + Z, min, max)),  S = (max(X) - min(X)) / (2^b - 1)  */
/* INT4 reading (asymmetric, b = 4, group of 32 along head_dim, FP16 outlier  */
/* side-list as in [P3]'s "FP16 Outlier Tensor"):                             */
/*   outliers: 3-sigma rule over the 32 values of the group                   */
/*   mn, mx over the group's non-outliers; S = fp16((mx - mn) / 15),          */
/*   m = fp16(mn) (the zero point stored as the group minimum: x = q*S + m is */
/*   the same affine map as (q - Z)*S with Z = -mn/S);                        */
/*   q = clamp(rint((x - m) / S), 0, 15) in fp64 from the stored S, m;        */
/*   S == 0 gives q = 0; outlier slots hold q = 0 and the value as fp16.      */
/* E2M1 reading (one e4m3 scale per 16 values, no outliers):                  */
/*   s = e4m3(amax / 6); q = e2m1(x / s) (quotients in fp64, rounded once to  */
/*   the format); s == 0 gives q = 0.                                         */
/* ------------------------------------------------------------------------- */

static void quantize_token_int4(const float* x, int D, double sigma, int role, int t, uint8_t* blk)
{
    int cap = 3 * (D / 32), cnt = 0;
    uint8_t* counts = blk + 10 * D;
    uint8_t* chans = blk + 10 * D + 16;
    uint8_t* vals = blk + 10 * D + 16 + 16 * cap;
    for (int i = 0; i < cap; ++i) { chans[t * cap + i] = 0; put_u16(vals + 2 * (t * cap + i), 0); }
    for (int g = 0; g < D / 32; ++g) {
        const float* v = x + 32 * g;
        uint8_t mask[32];
        or_outlier_mask(v, 32, sigma, or_kmax(32), mask);
        int have = 0;
        float mn = 0.0f, mx = 0.0f;
        for (int i = 0; i < 32; ++i) {
            if (mask[i]) continue;
            if (!have || v[i] < mn) mn = v[i];
            if (!have || v[i] > mx) mx = v[i];
            have = 1;
        }
        uint16_t S16 = 0, m16 = 0;
        if (have) { S16 = or_fp16_encode(((double)mx - (double)mn) / 15.0); m16 = or_fp16_encode((double)mn); }
        double S = or_fp16_decode(S16), m = or_fp16_decode(m16);
        for (int i = 0; i < 32; ++i) {
            int c = 32 * g + i;
            uint8_t q = 0;
            if (mask[i]) {
                chans[t * cap + cnt] = (uint8_t)c;
                put_u16(vals + 2 * (t * cap + cnt), or_fp16_encode((double)v[i]));
                ++cnt;
            } else if (S != 0.0) {
                double r = rint(((double)v[i] - m) / S);
                if (r < 0.0) r = 0.0;
                if (r > 15.0) r = 15.0;
                q = (uint8_t)r;
            }
            nib_set(blk, D, role, t, c, q);
        }
        uint8_t* sz = blk + 8 * D + 4 * (t * (D / 32) + g);
        put_u16(sz, S16);
        put_u16(sz + 2, m16);
    }
    counts[t] = (uint8_t)cnt;
}

static void quantize_token_e2m1(const float* x, int D, int role, int t, uint8_t* blk)
{
    for (int s = 0; s < D / 16; ++s) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(x[16 * s + i]);
            if (a > amax) amax = a;
        }
        uint8_t s8 = or_e4m3_encode((double)amax / 6.0);
        double sc = or_e4m3_decode(s8);
        for (int i = 0; i < 16; ++i) {
            uint8_t q = 0;
            if (sc != 0.0) q = or_e2m1_encode((double)x[16 * s + i] / sc);
            nib_set(blk, D, role, t, 16 * s + i, q);
        }
        blk[8 * D + 16 * s + t] = s8;
    }
}

/* ------------------------------------------------------------------------- */
/* Page quantizers (all 16 tokens of a page at once).                          */
/* CB2 ([P1]): per token, outliers by the 3-sigma rule over the whole head    */
/* vector (the listing takes mean/std along head_dim); per channel, the       */
/* Lloyd-Max codebook of the page's non-outlier values; codes at outlier      */
/* slots are 0; the side-list keeps (channel, e4m3(x)) sorted by (token,      */
/* channel) with a per-token count.                                           */
/* FP8 tier ([P2] "Tier 1 (High-Precision FP8)"): one fp32 scale per block,   */
/* s = f32(amax / 448) (the fp64 quotient rounded to binary32, the stored     */
/* scale); q = e4m3(x / s) with the quotient in fp64; s == 0 gives q = 0.     */
/* ------------------------------------------------------------------------- */

static void write_side_list(const float* x, int D, uint8_t mask[16][128], uint8_t* hdr);

static void quantize_page_cb2(const float* x, int D, double sigma, int iters, int role, uint8_t* blk)
{
    memset(blk, 0, (size_t)or_block_stride(OR_CB2, D));
    uint8_t mask[16][128];
    int kmax = or_kmax(D);
    for (int t = 0; t < 16; ++t) or_outlier_mask(x + t * D, D, sigma, kmax, mask[t]);
    for (int c = 0; c < D; ++c) {
        float v[16];
        uint8_t codes[16];
        uint16_t c16[4];
        int n = 0;
        for (int t = 0; t < 16; ++t)
            if (!mask[t][c]) v[n++] = x[t * D + c];
        or_lloyd4(v, n, iters, NULL, c16, codes);
        for (int j = 0; j < 4; ++j) cb2_cent_set(blk, D, role, c, j, c16[j]);
        n = 0;
        for (int t = 0; t < 16; ++t)
            cb2_code_set(blk, D, role, t, c, mask[t][c] ? 0 : codes[n++]);
    }
    write_side_list(x, D, mask, blk + 12 * D);
}

/* The outlier side-list of a page (CB2, ASYM3): one 20-byte record {channel,
 * 0, token mask, 16 e4m3 values (0 where the token is not an outlier)} for
 * each channel holding an outlier, channels ascending, after {n_ch, total}. */
static void write_side_list(const float* x, int D, uint8_t mask[16][128], uint8_t* hdr)
{
    int n_ch = 0, total = 0;
    for (int c = 0; c < D; ++c) {
        unsigned tmask = 0;
        for (int t = 0; t < 16; ++t)
            if (mask[t][c]) tmask |= 1u << t;
        if (!tmask) continue;
        uint8_t* rec = hdr + 4 + 20 * n_ch;
        rec[0] = (uint8_t)c;
        rec[1] = 0;
        put_u16(rec + 2, (uint16_t)tmask);
        for (int t = 0; t < 16; ++t)
            if (mask[t][c]) {
                rec[4 + t] = or_e4m3_encode((double)x[t * D + c]);
                ++total;
            }
        ++n_ch;
    }
    hdr[0] = (uint8_t)n_ch;
    hdr[1] = (uint8_t)total;
}

/* ASYM3 ([P3] "Sub-Byte KV-Cache Quantization": asymmetric 3-bit packing with
 * dynamic outlier preservation).  Outliers as CB2 (sigma rule per token over
 * the head vector, e4m3 side-list).  Per channel, over its non-outliers in
 * fp64 (the INT4 recipe with 8 levels): S = fp16((max - min) / 7),
 * m = fp16(min), q = clamp(rint((x - m) / S), 0, 7) (q = 0 when S == 0 or the
 * channel has no non-outlier); outlier slots hold q = 0.  The value a code
 * stands for is fp16(q * S + m), one rounding of the exact value. */
static void quantize_page_a3(const float* x, int D, double sigma, int role, uint8_t* blk)
{
    memset(blk, 0, (size_t)or_block_stride(OR_A3, D));
    uint8_t mask[16][128];
    int kmax = or_kmax(D);
    for (int t = 0; t < 16; ++t) or_outlier_mask(x + t * D, D, sigma, kmax, mask[t]);
    for (int c = 0; c < D; ++c) {
        int have = 0;
        float mn = 0.0f, mx = 0.0f;
        for (int t = 0; t < 16; ++t) {
            if (mask[t][c]) continue;
            float v = x[t * D + c];
            if (!have || v < mn) mn = v;
            if (!have || v > mx) mx = v;
            have = 1;
        }
        uint16_t S16 = 0, m16 = 0;
        if (have) { S16 = or_fp16_encode(((double)mx - (double)mn) / 7.0); m16 = or_fp16_encode((double)mn); }
        double S = or_fp16_decode(S16), m = or_fp16_decode(m16);
        put_u16(blk + 6 * D + 2 * a3_rho(role, c), S16);
        put_u16(blk + 8 * D + 2 * a3_rho(role, c), m16);
        for (int t = 0; t < 16; ++t) {
            uint8_t q = 0;
            if (!mask[t][c] && S != 0.0) {
                double r = rint(((double)x[t * D + c] - m) / S);
                if (r < 0.0) r = 0.0;
                if (r > 7.0) r = 7.0;
                q = (uint8_t)r;
            }
            a3_code_set(blk, D, role, t, c, q);
        }
    }
    write_side_list(x, D, mask, blk + 10 * D);
}

/* CB2 with a codebook per group of 4 pages ([P1] "2. Centroid Vector          */
/* Quantization for Residuals": k-means "per head-group block").  Outliers as */
/* CB2, per token; per channel, Lloyd-Max (as CB2) over the non-outliers of   */
/* all 64 tokens of the group, in token order; codes of every page from that  */
/* one codebook (0 at outliers); the side-list per page.  x: float [64][D];   */
/* blk[p] receives page p of the group.                                       */
static void quantize_group_cb2g(const float* x, int D, double sigma, int iters, int role, uint8_t* const blk[4])
{
    int n_tok = 16 * OR_GROUP;
    for (int p = 0; p < OR_GROUP; ++p) memset(blk[p], 0, (size_t)or_block_stride(OR_CB2G, D));
    uint8_t mask[64][128];
    int kmax = or_kmax(D);
    for (int t = 0; t < n_tok; ++t) or_outlier_mask(x + t * D, D, sigma, kmax, mask[t]);
    for (int c = 0; c < D; ++c) {
        float v[64];
        uint8_t codes[64];
        uint16_t c16[4];
        int n = 0;
        for (int t = 0; t < n_tok; ++t)
            if (!mask[t][c]) v[n++] = x[t * D + c];
        or_lloyd4(v, n, iters, NULL, c16, codes);
        for (int j = 0; j < 4; ++j) cent_set(blk[0], role, c, j, c16[j]);
        n = 0;
        for (int t = 0; t < n_tok; ++t)
            code2_set(blk[t / 16] + 8 * D, D, role, t % 16, c, mask[t][c] ? 0 : codes[n++]);
    }
    for (int p = 0; p < OR_GROUP; ++p) write_side_list(x + (size_t)16 * p * D, D, &mask[16 * p], blk[p] + 12 * D);
}

/* Dequantize page `codes_blk` of a CB2 group whose codebook lives in `cb_blk`. */
EXPORT void or_dequantize_group_page(int D, const uint8_t* codes_blk, const uint8_t* cb_blk, int role, int ntok,
                                     float* out)
{
    for (int t = 0; t < ntok; ++t)
        for (int c = 0; c < D; ++c)
            out[t * D + c] = (float)or_fp16_decode(cent_get(cb_blk, role, c, code2_get(codes_blk + 8 * D, D, role, t, c)));
    const uint8_t* hdr = codes_blk + 12 * D;
    int n_ch = hdr[0];
    for (int i = 0; i < n_ch; ++i) {
        const uint8_t* rec = hdr + 4 + 20 * i;
        unsigned tmask = get_u16(rec + 2);
        for (int t = 0; t < 16 && t < ntok; ++t)
            if (tmask & (1u << t)) out[t * D + rec[0]] = (float)or_e4m3_decode(rec[4 + t]);
    }
}

/* Single-group entry point for the pins: x float [64][D] -> 4 blocks. */
EXPORT void or_quantize_group(int D, double sigma, int iters, int role, const float* x, uint8_t* blocks)
{
    size_t stride = (size_t)or_block_stride(OR_CB2G, D);
    uint8_t* const blk[4] = {blocks, blocks + stride, blocks + 2 * stride, blocks + 3 * stride};
    quantize_group_cb2g(x, D, sigma, iters, role, blk);
}

static void quantize_page_fp8(const float* x, int D, int role, uint8_t* blk)
{
    memset(blk, 0, (size_t)or_block_stride(OR_FP8, D));
    float amax = 0.0f;
    for (int i = 0; i < 16 * D; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = f32_of_quotient(amax, 448.0f);
    for (int t = 0; t < 16; ++t)
        for (int c = 0; c < D; ++c) {
            uint8_t q = 0;
            if (s != 0.0f) q = or_e4m3_encode((double)x[t * D + c] / (double)s);
            blk[fp8_byte(D, role, t, c)] = q;
        }
    put_f32(blk + 16 * D, s);
}

/* CB2 with a static FP16 channel mask ([P4] "Key Production Engineering     */
/* Takeaways", item 2: the top 1% channels by absolute magnitude stay in      */
/* FP16).  No per-token outlier detection: every other channel gets the CB2   */
/* codebook fitted over all 16 of its values; the n_s static channels keep    */
/* fp16(x) for every token (code 0, all-zero centroids).                      */
static void quantize_page_cb2s(const float* x, int D, int iters, int role, const uint8_t* ch, int n_s, uint8_t* blk)
{
    memset(blk, 0, (size_t)or_block_stride(OR_CB2S, D));
    uint8_t is_static[128] = {0};
    for (int i = 0; i < n_s; ++i) is_static[ch[i] & (D - 1)] = 1;
    for (int c = 0; c < D; ++c) {
        if (is_static[c]) continue;   /* codes 0 and zero centroids from the clear */
        float v[16];
        uint8_t codes[16];
        uint16_t c16[4];
        for (int t = 0; t < 16; ++t) v[t] = x[t * D + c];
        or_lloyd4(v, 16, iters, NULL, c16, codes);
        for (int j = 0; j < 4; ++j) cb2_cent_set(blk, D, role, c, j, c16[j]);
        for (int t = 0; t < 16; ++t) cb2_code_set(blk, D, role, t, c, codes[t]);
    }
    uint8_t* hdr = blk + 12 * D;
    hdr[0] = (uint8_t)n_s;
    for (int i = 0; i < n_s; ++i) {
        int c = ch[i] & (D - 1);
        hdr[1 + i] = (uint8_t)c;
        for (int t = 0; t < 16; ++t) put_u16(hdr + 16 + 32 * i + 2 * t, or_fp16_encode((double)x[t * D + c]));
    }
}

/* The n_s static channels of one (head, role): the channels with the largest */
/* max_t |x[t][c]| over the calibration tokens, ties to the lower channel,    */
/* written in ascending channel order.  x is float [t][Hkv][D].               */
EXPORT void or_select_static(const float* x, int t, int Hkv, int D, int n_s, uint8_t* out /* [Hkv][n_s] */)
{
    for (int h = 0; h < Hkv; ++h) {
        float score[128];
        uint8_t taken[128] = {0};
        for (int c = 0; c < D; ++c) {
            float m = 0.0f;
            for (int i = 0; i < t; ++i) {
                float a = fabsf(x[((size_t)i * Hkv + h) * D + c]);
                if (a > m) m = a;
            }
            score[c] = m;
        }
        for (int k = 0; k < n_s; ++k) {
            int best = -1;
            for (int c = 0; c < D; ++c)
                if (!taken[c] && (best < 0 || score[c] > score[best])) best = c;
            taken[best] = 1;
        }
        int k = 0;
        for (int c = 0; c < D; ++c)
            if (taken[c]) out[(size_t)h * n_s + k++] = (uint8_t)c;
    }
}

/* Dequantize tokens [0, ntok) of a block to fp32 (values the codes stand for;
 * every one is exactly representable in fp32 as computed here). */
EXPORT void or_dequantize_block(int fmt, int D, const uint8_t* blk, int role, int ntok, float* out)
{
    for (int t = 0; t < ntok; ++t) {
        for (int c = 0; c < D; ++c) {
            double xv = 0.0;
            if (fmt == OR_INT4) {
                const uint8_t* sz = blk + 8 * D + 4 * (t * (D / 32) + c / 32);
                double S = or_fp16_decode(get_u16(sz)), m = or_fp16_decode(get_u16(sz + 2));
                xv = (double)nib_get(blk, D, role, t, c) * S + m;   /* exact; one rounding below */
            } else if (fmt == OR_E2M1) {
                double sc = or_e4m3_decode(blk[8 * D + 16 * (c / 16) + t]);
                xv = or_e2m1_decode(nib_get(blk, D, role, t, c)) * sc;
            } else if (fmt == OR_CB2 || fmt == OR_CB2S) {
                xv = or_fp16_decode(cb2_cent_get(blk, D, role, c, cb2_code_get(blk, D, role, t, c)));
            } else if (fmt == OR_A3) {
                double S = or_fp16_decode(get_u16(blk + 6 * D + 2 * a3_rho(role, c)));
                double m = or_fp16_decode(get_u16(blk + 8 * D + 2 * a3_rho(role, c)));
                xv = or_fp16_decode(or_fp16_encode((double)a3_code_get(blk, D, role, t, c) * S + m));   /* exact, then fp16 */
            } else {
                xv = or_e4m3_decode(blk[fp8_byte(D, role, t, c)]) * (double)get_f32(blk + 16 * D);
            }
            out[t * D + c] = (float)xv;
        }
        if (fmt == OR_INT4) {
            int cap = 3 * (D / 32);
            int cnt = blk[10 * D + t];
            for (int i = 0; i < cnt && i < cap; ++i) {
                int c = blk[10 * D + 16 + t * cap + i];
                out[t * D + c] = (float)or_fp16_decode(get_u16(blk + 10 * D + 16 + 16 * cap + 2 * (t * cap + i)));
            }
        }
    }
    if (fmt == OR_CB2S) {   /* the static channels hold their fp16 values */
        const uint8_t* hdr = blk + 12 * D;
        int n_s = hdr[0] < OR_MAX_STATIC ? hdr[0] : OR_MAX_STATIC;
        for (int i = 0; i < n_s; ++i)
            for (int t = 0; t < ntok; ++t)
                out[t * D + (hdr[1 + i] & (D - 1))] = (float)or_fp16_decode(get_u16(hdr + 16 + 32 * i + 2 * t));
    }
    if (fmt == OR_CB2 || fmt == OR_A3) {
        const uint8_t* hdr = blk + (fmt == OR_CB2 ? 12 : 10) * D;
        int n_ch = hdr[0];
        for (int i = 0; i < n_ch; ++i) {
            const uint8_t* rec = hdr + 4 + 20 * i;
            unsigned tmask = get_u16(rec + 2);
            for (int t = 0; t < 16 && t < ntok; ++t)
                if (tmask & (1u << t))
                    out[t * D + rec[0]] = (float)or_e4m3_decode(rec[4 + t]);
        }
    }
}

/* Single-block entry points used by the pinning tests. */
EXPORT void or_quantize_token(int fmt, int D, double sigma, int role, int t, const float* x, uint8_t* blk)
{
    if (fmt == OR_INT4) quantize_token_int4(x, D, sigma, role, t, blk);
    else quantize_token_e2m1(x, D, role, t, blk);
}
EXPORT void or_quantize_page_static(int D, int iters, int role, const float* x, const uint8_t* ch, int n_s,
                                    uint8_t* blk)
{
    quantize_page_cb2s(x, D, iters, role, ch, n_s, blk);
}
EXPORT void or_quantize_page(int fmt, int D, double sigma, int iters, int role, const float* x, uint8_t* blk)
{
    if (fmt == OR_CB2) quantize_page_cb2(x, D, sigma, iters, role, blk);
    else if (fmt == OR_A3) quantize_page_a3(x, D, sigma, role, blk);
    else quantize_page_fp8(x, D, role, blk);
}

/* ------------------------------------------------------------------------- */
/* Paged cache ([P2] "Paged Attention Memory Engine", [P4] PagedAttention     */
/* takeaway).  Pages hold 16 tokens.  page_table[b][p] names the physical     */
/* page of logical page p of sequence b; for the tiered format bit 31 says    */
/* the page lives in the FP8 tier pool ([P2] "Dual-Tier Paged Compression    */
/* Protocol").  Pool layout: block (phys, head, role) at                      */
/* ((phys * Hkv + head) * 2 + role) * stride.                                 */
/* Per-token formats quantize every token when it arrives.  The CB2 group    */
/* format keeps the partial last group in staging [B][Hkv][2][64][D] and      */
/* quantizes a group when its 64th token arrives.  Page formats keep          */
/* the partial last page in fp32 staging [B][Hkv][2][16][D] and quantize a    */
/* page when its 16th token arrives (reading: the pages never discuss partial */
/* pages; page statistics stay fixed once written).                           */
/* ------------------------------------------------------------------------- */

typedef struct {
    int32_t fmt;            /* 0 INT4, 1 E2M1, 2 CB2, 3 TIERED (CB2 + FP8 tier), 4 CB2 static, 5 ASYM3,
                               6 CB2 group (codebook per 4 pages) */
    int32_t B, Hkv, D, pages_per_seq_max, num_pages, num_tier_pages;
    int32_t iters;
    double sigma;
    int32_t n_static;              /* format 4: static channels per (head, role) */
    const uint8_t* static_ch;      /* format 4: [Hkv][2][n_static] */
} or_cfg;

static int page_fmt(const or_cfg* c) { return c->fmt == 3 ? OR_CB2 : c->fmt; }
static int is_paged(const or_cfg* c)
{
    return c->fmt == OR_CB2 || c->fmt == 3 || c->fmt == OR_CB2S || c->fmt == OR_A3 || c->fmt == OR_CB2G;
}
/* fp32 staging rows per (sequence, head, role): the partial page, or for the
 * group format the partial group. */
static int stg_rows(const or_cfg* c) { return c->fmt == OR_CB2G ? 16 * OR_GROUP : 16; }

static int entry_ok(const or_cfg* c, int32_t e)
{
    uint32_t u = (uint32_t)e;
    int tier = (u >> 31) & 1;
    int32_t phys = (int32_t)(u & 0x7FFFFFFFu);
    if (tier) return c->fmt == 3 && phys < c->num_tier_pages;
    return phys < c->num_pages;
}

static uint8_t* block_ptr(const or_cfg* c, uint8_t* pool, uint8_t* tier_pool, int32_t e, int h, int role)
{
    uint32_t u = (uint32_t)e;
    size_t phys = u & 0x7FFFFFFFu;
    if ((u >> 31) & 1)
        return tier_pool + ((phys * c->Hkv + h) * 2 + role) * (size_t)or_block_stride(OR_FP8, c->D);
    return pool + ((phys * c->Hkv + h) * 2 + role) * (size_t)or_block_stride(page_fmt(c), c->D);
}

static float* staging_row(const or_cfg* c, float* staging, int b, int h, int role, int t)
{
    return staging + ((((size_t)b * c->Hkv + h) * 2 + role) * stg_rows(c) + t) * c->D;
}

/* Append t_new tokens (or t_per_seq[b] <= t_new of them) to every sequence.
 * kv[role] is float [B][t_new][Hkv][D].  Returns the number of sequences
 * skipped because the append overflows the page table or names a bad page. */
EXPORT int or_append(const or_cfg* c, uint8_t* pool, uint8_t* tier_pool, const int32_t* page_table,
                     int32_t* seq_lens, float* staging, const float* k_new, const float* v_new,
                     int t_new, const int32_t* t_per_seq)
{
    int bad = 0, D = c->D;
    const float* src[2] = {k_new, v_new};
    for (int b = 0; b < c->B; ++b) {
        int start = seq_lens[b];
        int n = t_per_seq ? t_per_seq[b] : t_new;
        int end = start + n;
        if (n <= 0) continue;
        if (end > c->pages_per_seq_max * 16 || n > t_new) { ++bad; continue; }
        int ok = 1;
        int first_pg = c->fmt == OR_CB2G ? (start / 64) * OR_GROUP : start / 16;   /* a group writes all its pages */
        for (int pg = first_pg; pg <= (end - 1) / 16; ++pg)
            if (!entry_ok(c, page_table[(size_t)b * c->pages_per_seq_max + pg])) ok = 0;
        if (!ok) { ++bad; continue; }
        for (int h = 0; h < c->Hkv; ++h)
            for (int role = 0; role < 2; ++role) {
                const float* in = src[role];
#define IN_ROW(pos) (in + (((size_t)b * t_new + (size_t)((pos) - start)) * c->Hkv + h) * D)
                if (c->fmt == OR_CB2G) {
                    for (int gr = start / 64; gr <= (end - 1) / 64; ++gr) {
                        int lo = start > gr * 64 ? start : gr * 64;
                        int hi = end < gr * 64 + 64 ? end : gr * 64 + 64;
                        if (hi == gr * 64 + 64) {   /* the group completes: quantize its 4 pages */
                            float* x = (float*)malloc(sizeof(float) * 64 * D);
                            for (int t = 0; t < 64; ++t) {
                                int pos = gr * 64 + t;
                                const float* r = pos < start ? staging_row(c, staging, b, h, role, t) : IN_ROW(pos);
                                memcpy(x + t * D, r, sizeof(float) * D);
                            }
                            uint8_t* blks[4];
                            for (int q = 0; q < OR_GROUP; ++q)
                                blks[q] = block_ptr(c, pool, tier_pool,
                                                    page_table[(size_t)b * c->pages_per_seq_max + gr * OR_GROUP + q], h, role);
                            quantize_group_cb2g(x, D, c->sigma, c->iters, role, blks);
                            free(x);
                        } else {
                            for (int pos = lo; pos < hi; ++pos)
                                memcpy(staging_row(c, staging, b, h, role, pos % 64), IN_ROW(pos), sizeof(float) * D);
                        }
                    }
                    continue;
                }
                for (int pg = start / 16; pg <= (end - 1) / 16; ++pg) {
                    int32_t e = page_table[(size_t)b * c->pages_per_seq_max + pg];
                    uint8_t* blk = block_ptr(c, pool, tier_pool, e, h, role);
                    int lo = start > pg * 16 ? start : pg * 16;
                    int hi = end < pg * 16 + 16 ? end : pg * 16 + 16;
                    if (c->fmt == OR_INT4 || c->fmt == OR_E2M1) {
                        for (int pos = lo; pos < hi; ++pos)
                            or_quantize_token(c->fmt, D, c->sigma, role, pos % 16, IN_ROW(pos), blk);
                    } else if (hi == pg * 16 + 16) {
                        float* x = (float*)malloc(sizeof(float) * 16 * D);
                        for (int t = 0; t < 16; ++t) {
                            int pos = pg * 16 + t;
                            const float* r = pos < start ? staging_row(c, staging, b, h, role, t) : IN_ROW(pos);
                            memcpy(x + t * D, r, sizeof(float) * D);
                        }
                        int tier = ((uint32_t)e >> 31) & 1;
                        if (c->fmt == OR_CB2S)
                            quantize_page_cb2s(x, D, c->iters, role, c->static_ch + ((size_t)h * 2 + role) * c->n_static,
                                               c->n_static, blk);
                        else
                            or_quantize_page(tier ? OR_FP8 : page_fmt(c), D, c->sigma, c->iters, role, x, blk);
                        free(x);
                    } else {
                        for (int pos = lo; pos < hi; ++pos)
                            memcpy(staging_row(c, staging, b, h, role, pos % 16), IN_ROW(pos), sizeof(float) * D);
                    }
                }
#undef IN_ROW
            }
        seq_lens[b] = end;
    }
    return bad;
}

/* Dequantized tokens [t0, t1) of (sequence b, kv head h, role) as fp32. */
EXPORT void or_dequantize_range(const or_cfg* c, uint8_t* pool, uint8_t* tier_pool, const int32_t* page_table,
                                const int32_t* seq_lens, float* staging, int b, int h, int role, int t0, int t1,
                                float* out)
{
    int D = c->D, len = seq_lens[b];
    int paged = is_paged(c);
    float* tmp = (float*)malloc(sizeof(float) * 16 * D);
    for (int pg = t0 / 16; t1 > t0 && pg <= (t1 - 1) / 16; ++pg) {
        int full = (pg + 1) * 16 <= len;
        if (c->fmt == OR_CB2G) {
            int gr = pg / OR_GROUP;
            if ((gr + 1) * 64 <= len) {   /* quantized group: the codebook lives in its first page */
                const int32_t* row = page_table + (size_t)b * c->pages_per_seq_max;
                or_dequantize_group_page(D, block_ptr(c, pool, tier_pool, row[pg], h, role),
                                         block_ptr(c, pool, tier_pool, row[gr * OR_GROUP], h, role), role, 16, tmp);
            } else {
                for (int t = 0; t < 16; ++t)
                    memcpy(tmp + t * D, staging_row(c, staging, b, h, role, (pg % OR_GROUP) * 16 + t), sizeof(float) * D);
            }
        } else if (paged && !full) {
            for (int t = 0; t < 16; ++t) memcpy(tmp + t * D, staging_row(c, staging, b, h, role, t), sizeof(float) * D);
        } else {
            int32_t e = page_table[(size_t)b * c->pages_per_seq_max + pg];
            int tier = ((uint32_t)e >> 31) & 1;
            int ntok = full ? 16 : len - pg * 16;
            or_dequantize_block(tier ? OR_FP8 : page_fmt(c), D, block_ptr(c, pool, tier_pool, e, h, role), role,
                                ntok, tmp);
        }
        for (int t = 0; t < 16; ++t) {
            int pos = pg * 16 + t;
            if (pos >= t0 && pos < t1) memcpy(out + (size_t)(pos - t0) * D, tmp + t * D, sizeof(float) * D);
        }
    }
    free(tmp);
}

/* ------------------------------------------------------------------------- */
/* Decode attention in fp64 ([P1] "Hardware-Kernel Fusion": attention over    */
/* the dequantized cache; [P4] Flash-Decoding phase).  For sequence b and     */
/* query head h (kv head h / G, G = Hq / Hkv):                                */
/*   s_t = scale * sum_c q[c] * k[t][c],  t < seq_len                         */
/*   p   = softmax(s) (max subtracted),   o = sum_t p_t v[t]                  */
/* with q the bf16 query read exactly and k, v the values the cache stores.   */
/* An empty sequence gives o = 0.                                             */
/* ------------------------------------------------------------------------- */

EXPORT void or_attention(int G, int D, int N, const double* q, const float* k, const float* v, double scale,
                         double* out)
{
    double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
    for (int h = 0; h < G; ++h) {
        double* o = out + (size_t)h * D;
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        if (N == 0) continue;
        double mx = -INFINITY;
        for (int t = 0; t < N; ++t) {
            double acc = 0.0;
            for (int c = 0; c < D; ++c) acc += q[(size_t)h * D + c] * (double)k[(size_t)t * D + c];
            s[t] = scale * acc;
            if (s[t] > mx) mx = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < N; ++t) {
            s[t] = exp(s[t] - mx);
            l += s[t];
        }
        for (int t = 0; t < N; ++t) {
            double p = s[t] / l;
            for (int c = 0; c < D; ++c) o[c] += p * (double)v[(size_t)t * D + c];
        }
    }
    free(s);
}

/* Attention for units u in [u0, u1), u = b * Hkv + kv_head, over the paged
 * cache; q is bf16 bits [B][Hq][D]; out is fp64 [B][Hq][D].  Units are
 * independent, so they may run on `nthreads` host threads. */
EXPORT void or_decode(const or_cfg* c, uint8_t* pool, uint8_t* tier_pool, const int32_t* page_table,
                      const int32_t* seq_lens, float* staging, const uint16_t* q, int Hq, double scale,
                      double* out, int u0, int u1, int nthreads)
{
    int G = Hq / c->Hkv, D = c->D;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int u = u0; u < u1; ++u) {
        int b = u / c->Hkv, h = u % c->Hkv, N = seq_lens[b];
        float* kd = (float*)malloc(sizeof(float) * ((size_t)N * D + 1));
        float* vd = (float*)malloc(sizeof(float) * ((size_t)N * D + 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)G * D);
        or_dequantize_range(c, pool, tier_pool, page_table, seq_lens, staging, b, h, 0, 0, N, kd);
        or_dequantize_range(c, pool, tier_pool, page_table, seq_lens, staging, b, h, 1, 0, N, vd);
        for (int i = 0; i < G * D; ++i) qd[i] = or_bf16_decode(q[((size_t)b * Hq + (size_t)h * G) * D + i]);
        or_attention(G, D, N, qd, kd, vd, scale, out + ((size_t)b * Hq + (size_t)h * G) * D);
        free(kd);
        free(vd);
        free(qd);
    }
}
