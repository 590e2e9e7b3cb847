// kvq_decode.cuh -- split-K decode attention over the quantized paged cache with
// dequantization fused in.
//
// "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression",
// "Hardware-Kernel Fusion": packed codes go from HBM to shared memory and are
// expanded in registers inside the attention kernel -- no FP16 copy of the cache
// is ever written.  "Sub-5ms MoE Inference: Sub-Byte KV Quantization and Expert
// Pipelining at Scale", item 3 of "Engineering Real-Time Autonomous Workflows":
// the codes are unpacked straight into tensor-core fragment registers.  "The
// Sub-10ms Barrier: Fusing Sparse MoE Routing with FP4 KV-Cache Quantization",
// section 2 and its flash-decoding flowchart: values are dequantized only
// during the attention reduction, and the sequence is split across CTAs whose
// partial softmax states are then merged (here by the last CTA of each
// sequence and kv head to finish, or by a second kernel in the two-stage calls).
//
// Design (GB300, sm_103a):
//  * grid (splits, kv heads, sequences); a CTA owns one (sequence, kv head,
//    split) and all G query heads of that kv head; each of its W warps streams
//    its own pages (page p0 + w, p0 + w + W, ...), PPI pages per iteration,
//    with its own online-softmax state; the warps merge in shared memory.
//  * each warp runs two rings of bulk asynchronous copies (cp.async.bulk +
//    mbarrier), one copy per block: for the page formats one K stage (refilled
//    as soon as the iteration's scores are done) and one V stage (a V block is
//    read only after the K phase and the softmax of its iteration); E2M1 two
//    and two (three pages per iteration), INT4 three and two single pages; no
//    register staging, no TMA multicast.
//  * QK^T: A = K (16 tokens x 16 channels, built in registers from the codes),
//    B = Q^T (16 channels x 8 heads, fp16, loaded once).  PV: A = V^T (16
//    channels x 16 tokens, built in registers), B = P^T (fp16 hi + lo split of
//    the fp32 probabilities, so P carries ~22 bits).  mma.sync m16n8k16 with
//    fp32 accumulation; the layouts in include/kvq.h make every A register one
//    or two byte-permutes of shared-memory words.  The PPI pages of an
//    iteration are independent mma chains the scheduler interleaves; the
//    tiered format instead branches on each page's tier once, around all of
//    its steps, so that every page's steps still schedule as one block.  For
//    CB2 at G <= 4 the same products can run as fp32 FMAs instead
//    (iter_cb2_cc, kvq_config.decode_math; measured slower).
//  * CB2 outliers: a code slot holding an outlier stores code 0 (value c0).
//    The side-list's channel records go six at a time into one mma tile; the
//    correction x - c0 is applied as two mma with exact fp16 operands (+ the
//    e4m3 values, - c0 where the token mask is set) against the gathered
//    query columns (scores) or against P^T (output of those channels,
//    accumulated in shared memory with the same online-softmax rescaling as
//    the registers).  No atomics.
//  * the partial last page of page formats (fp32 staging) is done on CUDA
//    cores in fp32.
#pragma once
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kOutPrefetch = 128;     // bytes of a CB2 outlier side-list fetched with its block
constexpr float kRescaleTh = 8.0f;    // lazy rescale: p stays <= 2^8

template <int FMT>
struct Fmt {
  static constexpr bool kPaged = (FMT == KVQ_FMT_CB2_OUTLIER || FMT == KVQ_FMT_TIERED || FMT == KVQ_FMT_CB2_STATIC ||
                                  FMT == KVQ_FMT_ASYM3_OUTLIER || FMT == KVQ_FMT_CB2_GROUP4);
  static constexpr int kMain = FMT == KVQ_FMT_TIERED ? kBlkCb2 : FMT;
  static constexpr bool kGroup = kMain == kBlkCb2g;   // 4 pages share the first page's codebook
  static constexpr bool kOutliers = (kMain == kBlkInt4 || kMain == kBlkCb2 || kMain == kBlkA3 || kGroup);
  static constexpr bool kSideList = (kMain == kBlkCb2 || kMain == kBlkA3 || kGroup);   // 20-byte outlier records
  // pages per warp iteration (a whole group for the group format); E2M1's
  // lighter pages take three (three CTAs per SM; 3% faster on fp4_32k, while
  // the codebook formats lost 6-10% that way)
  static constexpr int kPPI = kMain == kBlkInt4 ? 1 : kGroup ? kGroupPages : kMain == kBlkE2m1 ? 3 : 2;
  static constexpr int kUnit = kGroup ? kGroupPages : 1;   // pages per unit of the page-to-warp assignment
};

// Bytes copied to shared memory per block.
template <int D>
__host__ __device__ constexpr int fetch_bytes(int blk) {
  return blk == kBlkInt4 ? 10 * D + 16 + 48 * int4_cap(D)
       : blk == kBlkE2m1 ? 9 * D
       : blk == kBlkCb2  ? 12 * D + kOutPrefetch
       : blk == kBlkCb2s ? 12 * D + 16 + 32 * kMaxStatic   // the copy itself takes 32 n_s
       : blk == kBlkA3   ? 10 * D + kOutPrefetch
                         : 16 * D + 16;
}
template <int FMT, int D>
__host__ __device__ constexpr int half_slot_bytes() {
  return FMT == KVQ_FMT_TIERED
             ? (fetch_bytes<D>(kBlkCb2) > fetch_bytes<D>(kBlkFp8) ? fetch_bytes<D>(kBlkCb2)
                                                                  : fetch_bytes<D>(kBlkFp8))
             : fetch_bytes<D>(Fmt<FMT>::kMain);
}

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

// Per-warp copy rings: K blocks run kK iterations ahead, V blocks kV (a V
// block is needed only after the iteration's K phase and softmax, so a
// shallower V ring still hides the fetch and leaves room for more CTAs).  The
// page formats refill their one K stage as soon as its scores are done, which
// hides the next fetch behind the softmax, PV and V corrections (measured 1.5-3%
// faster than two stages, and the smaller plan fits four CTAs per SM at G = 8).
template <int FMT>
struct Ring {
  static constexpr int kK = Fmt<FMT>::kGroup ? 1 : Fmt<FMT>::kPPI == 1 ? 3 : Fmt<FMT>::kPaged ? 1 : 2;
  static constexpr int kV = Fmt<FMT>::kGroup ? 1 : Fmt<FMT>::kPPI == 1 ? 2 : Fmt<FMT>::kPaged ? 1 : 2;
};

// Bytes of one ring stage (the blocks of one iteration, one role).  The group
// format stages [codebook 8D][page 0 codes + side-list prefix]...[page 3 ...],
// page j at 8D + j * (4D + kOutPrefetch).
template <int FMT, int D>
__host__ __device__ constexpr int group_page_bytes() { return 4 * D + kOutPrefetch; }
// Offsets of page j within a stage (its virtual block base), of its copy's
// destination, and of the copied bytes within its block.  The group format
// copies page 0 whole (codebook, codes, side-list prefix) and pages 1..3
// from their codes on; a page's virtual base puts its codes at 8D and its
// side-list at 12D, as in its block.
template <int FMT, int D>
__host__ __device__ constexpr int page_base(int j);
template <int FMT, int D>
__host__ __device__ constexpr int copy_dst(int j);
template <int FMT, int D>
__host__ __device__ constexpr int copy_src(int j) { return Fmt<FMT>::kGroup && j > 0 ? 8 * D : 0; }
template <int FMT, int D>
__host__ __device__ constexpr int stage_bytes() {
  return Fmt<FMT>::kGroup ? 8 * D + kGroupPages * group_page_bytes<FMT, D>()
                          : Fmt<FMT>::kPPI * half_slot_bytes<FMT, D>();
}

// Shared-memory plan: [mbarriers: W x (kK + kV)][qsm: D x GS fp32][zero block, page formats]
// then per warp: [K slots: kK x PPI blocks][V slots: kV x PPI blocks][meta: kK x PPI]
// [ds 16 x GS, INT4 only][psm 16 x GS][corr D x GS, formats with outliers].
// The CTA merge reuses everything after qsm, so the mbarriers sit before it.
template <int FMT>
__host__ __device__ constexpr bool has_ds() { return Fmt<FMT>::kMain == kBlkInt4; }
template <int FMT, int D>
__host__ __device__ constexpr int page_base(int j) {
  return Fmt<FMT>::kGroup ? j * group_page_bytes<FMT, D>() : j * half_slot_bytes<FMT, D>();
}
template <int FMT, int D>
__host__ __device__ constexpr int copy_dst(int j) {
  return Fmt<FMT>::kGroup ? page_base<FMT, D>(j) + copy_src<FMT, D>(j) : page_base<FMT, D>(j);
}
template <int FMT, int D>
__host__ __device__ constexpr int warp_smem_bytes(int GS) {
  return (Ring<FMT>::kK + Ring<FMT>::kV) * stage_bytes<FMT, D>() +
         align16(4 * Ring<FMT>::kK * Fmt<FMT>::kPPI) +
         (has_ds<FMT>() ? 16 * GS * 4 : 0) + 16 * GS * 4 + (Fmt<FMT>::kOutliers ? D * GS * 4 : 0);
}
// Page formats keep one zeroed block (K and V both read it) for absent pages.
// An absent page is never a tier page, so the tiered format's zero block is a
// main-format (CB2) block.
template <int FMT, int D>
__host__ __device__ constexpr int zero_block_bytes() {
  return !Fmt<FMT>::kPaged ? 0
       : Fmt<FMT>::kGroup  ? align16(stage_bytes<FMT, D>())
                           : align16(fetch_bytes<D>(Fmt<FMT>::kMain));
}
template <int FMT, int W>
__host__ __device__ constexpr int mbar_bytes() {
  return align16(8 * W * (Ring<FMT>::kK + Ring<FMT>::kV));
}
template <int FMT, int D, int W>
__host__ __device__ constexpr int cta_smem_bytes(int GS) {
  return mbar_bytes<FMT, W>() + align16(D * GS * 4) + zero_block_bytes<FMT, D>() +
         W * align16(warp_smem_bytes<FMT, D>(GS));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// ----------------------------------------------------------------------------- fragment builders
// Each builds the four A registers (f16x2) of step s for this lane from
// 32-bit shared-memory addresses.

// CB2, K role: channels x = 16s + 2q, y = x + 1 (and +8); tokens g, g + 8.
// kcb = block + 4D + 16q (the lane's codebook column).
// The codebook columns of step s (cb2_k_cols) and the expansion of the codes
// against them (cb2_k_expand) are separate so that pages sharing a codebook
// (the group format) load the columns once per step.
struct KCols {
  uint4 a, b;
};
__device__ __forceinline__ KCols cb2_k_cols(uint32_t kcb, int s) {
  return {lds128(kcb + 128 * s), lds128(kcb + 128 * s + 64)};
}
__device__ __forceinline__ void cb2_k_expand(const KCols& c, uint32_t w16, uint32_t (&a)[4]) {
  const uint32_t sel1 = (w16 & 0x3333u) | 0x4040u;
  const uint32_t sel2 = ((w16 >> 2) & 0x3333u) | 0x4040u;
  const uint4 ca = c.a, cb = c.b;
  uint32_t lo = prmt(ca.x, ca.z, sel1), hi = prmt(ca.y, ca.w, sel1);
  a[0] = prmt(lo, hi, 0x5140u);
  a[1] = prmt(lo, hi, 0x7362u);
  lo = prmt(cb.x, cb.z, sel2);
  hi = prmt(cb.y, cb.w, sel2);
  a[2] = prmt(lo, hi, 0x5140u);
  a[3] = prmt(lo, hi, 0x7362u);
}
__device__ __forceinline__ void cb2_k_frag(uint32_t kcb, uint32_t w16, int s, uint32_t (&a)[4]) {
  cb2_k_expand(cb2_k_cols(kcb, s), w16, a);
}

// CB2, V role: channels cA = 16s + g, cB = cA + 8; tokens 2q, 2q+1 (and +8).
// vcb = block + 4D + 16g.
__device__ __forceinline__ uint4 cb2_v_cols(uint32_t vcb, int s) { return lds128(vcb + 128 * s); }
__device__ __forceinline__ void cb2_v_expand(const uint4& c, uint32_t w16, uint32_t (&a)[4]) {
  const uint32_t sel1 = (w16 & 0x3333u) | 0x4400u;
  const uint32_t sel2 = ((w16 >> 2) & 0x3333u) | 0x4400u;
  uint32_t lo = prmt(c.x, c.z, sel1), hi = prmt(c.y, c.w, sel1);
  a[0] = prmt(lo, hi, 0x5140u);
  a[1] = prmt(lo, hi, 0x7362u);
  lo = prmt(c.x, c.z, sel2);
  hi = prmt(c.y, c.w, sel2);
  a[2] = prmt(lo, hi, 0x5140u);
  a[3] = prmt(lo, hi, 0x7362u);
}
__device__ __forceinline__ void cb2_v_frag(uint32_t vcb, uint32_t w16, int s, uint32_t (&a)[4]) {
  cb2_v_expand(cb2_v_cols(vcb, s), w16, a);
}

// FP8 e4m3 codes, either role: slot k = byte k of the lane's 8 bytes for step s.
__device__ __forceinline__ void fp8_frag(uint2 wd, uint32_t (&a)[4]) {
  a[0] = e4m3x2_to_f16x2(wd.x & 0xFFFFu);
  a[1] = e4m3x2_to_f16x2(wd.x >> 16);
  a[2] = e4m3x2_to_f16x2(wd.y & 0xFFFFu);
  a[3] = e4m3x2_to_f16x2(wd.y >> 16);
}

// E2M1 codes: slot k = nibble k of the lane's u32 for step s; register i holds
// slots 2i, 2i+1 = byte i.
__device__ __forceinline__ void e2m1_frag(uint32_t wd, uint32_t (&a)[4]) {
  a[0] = e2m1x2_to_f16x2(wd & 0xFFu);
  a[1] = e2m1x2_to_f16x2((wd >> 8) & 0xFFu);
  a[2] = e2m1x2_to_f16x2((wd >> 16) & 0xFFu);
  a[3] = e2m1x2_to_f16x2(wd >> 24);
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t x, uint32_t y) {
  return h2_as_u32(__hmul2(u32_as_h2(x), u32_as_h2(y)));
}

// fp32 pair -> fp16 high part and fp16 residual (together ~22 bits).
__device__ __forceinline__ void split_hilo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(x0, x1);
  float2 hf = __half22float2(h);
  hi = h2_as_u32(h);
  lo = h2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}
// INT4 codes: x = q * S + m in fp32 (per token, group of 32), as fp16 hi + lo.
// Register r holds slots 2r, 2r+1 (nibbles 2r, 2r+1 of the step's u32).
__device__ __forceinline__ float nib(uint32_t wd, int k) { return (float)((wd >> (4 * k)) & 0xFu); }
// K role: registers 0, 2 are token g (S0, M0); registers 1, 3 token g + 8 (S1, M1).
__device__ __forceinline__ void int4_k_frag(uint32_t wd, float S0, float M0, float S1, float M1,
                                            uint32_t (&ahi)[4], uint32_t (&alo)[4]) {
  split_hilo(fmaf(nib(wd, 0), S0, M0), fmaf(nib(wd, 1), S0, M0), ahi[0], alo[0]);
  split_hilo(fmaf(nib(wd, 2), S1, M1), fmaf(nib(wd, 3), S1, M1), ahi[1], alo[1]);
  split_hilo(fmaf(nib(wd, 4), S0, M0), fmaf(nib(wd, 5), S0, M0), ahi[2], alo[2]);
  split_hilo(fmaf(nib(wd, 6), S1, M1), fmaf(nib(wd, 7), S1, M1), ahi[3], alo[3]);
}
// V role: half 0 / 1 of registers 0, 1 are tokens t0 / t1; of registers 2, 3 tokens t2 / t3.
__device__ __forceinline__ void int4_v_frag(uint32_t wd, const float (&S)[4], const float (&M)[4],
                                            uint32_t (&ahi)[4], uint32_t (&alo)[4]) {
  split_hilo(fmaf(nib(wd, 0), S[0], M[0]), fmaf(nib(wd, 1), S[1], M[1]), ahi[0], alo[0]);
  split_hilo(fmaf(nib(wd, 2), S[0], M[0]), fmaf(nib(wd, 3), S[1], M[1]), ahi[1], alo[1]);
  split_hilo(fmaf(nib(wd, 4), S[2], M[2]), fmaf(nib(wd, 5), S[3], M[3]), ahi[2], alo[2]);
  split_hilo(fmaf(nib(wd, 6), S[2], M[2]), fmaf(nib(wd, 7), S[3], M[3]), ahi[3], alo[3]);
}

__device__ __forceinline__ float fp16_bits_to_float(uint32_t bits) {
  return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}

// ASYM3: a code q stands for fp16(q * S + m).  The low 2 bits come from
// words X (two steps each), the high bit from words Y (four steps each);
// register r of step s holds slots 2r (low half) and 2r + 1 (high half).
template <int D>
__device__ __forceinline__ void load_a3_words(uint32_t blk_s, int lane, uint32_t (&xw)[D / 32],
                                              uint32_t (&yw)[D / 64]) {
  if constexpr (D == 128) {
    const uint4 x = lds128(blk_s + 16 * lane);
    const uint2 y = lds64(blk_s + a3_hi_off(D) + 8 * lane);
    xw[0] = x.x; xw[1] = x.y; xw[2] = x.z; xw[3] = x.w;
    yw[0] = y.x; yw[1] = y.y;
  } else {
    const uint2 x = lds64(blk_s + 8 * lane);
    xw[0] = x.x; xw[1] = x.y;
    yw[0] = lds32(blk_s + a3_hi_off(D) + 4 * lane);
  }
}
// fp16x2 {q(2r), q(2r+1)} of step s, then fp16(q * S + m) with one rounding
// (__hfma2 is the round-to-nearest fused multiply-add).
// (s and r are loop indices of fully unrolled loops: the shifts fold to constants.)
__device__ __forceinline__ uint32_t a3_value(uint32_t xw, uint32_t yw, int S_, int R, uint32_t sc, uint32_t zp) {
  const int SH = 4 * (S_ & 3) + R;   // the high bits sit at SH and SH + 16
  const uint32_t lo = (xw >> (8 * (S_ & 1) + 2 * R)) & 0x00030003u;
  const uint32_t hi = (SH >= 2 ? (yw >> (SH - 2)) : (yw << (2 - SH))) & 0x00040004u;
  const uint32_t q1024 = lo | hi | 0x64006400u;   // fp16 1024 + q, exact
  const uint32_t q = h2_as_u32(__hsub2(u32_as_h2(q1024), u32_as_h2(0x64006400u)));
  return h2_as_u32(__hfma2(u32_as_h2(q), u32_as_h2(sc), u32_as_h2(zp)));
}
// K role: channels x = 16s + 2q, x + 1 (registers 0, 1: tokens g, g + 8) and
// x + 8, x + 9 (registers 2, 3); their S and m are 4 adjacent fp16.
template <int D>
__device__ __forceinline__ void a3_k_frag(uint32_t kb_s, const uint32_t (&xw)[D / 32], const uint32_t (&yw)[D / 64],
                                          int S_, int q4, uint32_t (&a)[4]) {
  const uint2 sc = lds64(kb_s + a3_s_off(D) + 2 * (16 * S_ + 4 * q4));
  const uint2 zp = lds64(kb_s + a3_m_off(D) + 2 * (16 * S_ + 4 * q4));
  const uint32_t x = xw[S_ >> 1], y = yw[S_ >> 2];
  a[0] = a3_value(x, y, S_, 0, sc.x, zp.x);
  a[1] = a3_value(x, y, S_, 1, sc.x, zp.x);
  a[2] = a3_value(x, y, S_, 2, sc.y, zp.y);
  a[3] = a3_value(x, y, S_, 3, sc.y, zp.y);
}
// V role: channels c = 16s + g (registers 0, 2) and c + 8 (registers 1, 3).
template <int D>
__device__ __forceinline__ void a3_v_frag(uint32_t vb_s, const uint32_t (&xw)[D / 32], const uint32_t (&yw)[D / 64],
                                          int S_, int g, uint32_t (&a)[4]) {
  const uint32_t sc = lds32(vb_s + a3_s_off(D) + 2 * (16 * S_ + 2 * g));
  const uint32_t zp = lds32(vb_s + a3_m_off(D) + 2 * (16 * S_ + 2 * g));
  // S and m of channel c (low half) and c + 8 (high half), each broadcast to both
  // halves; as half2 duplicates the fma takes them as operand selects
  const uint32_t sA = h2_as_u32(__low2half2(u32_as_h2(sc))), sB = h2_as_u32(__high2half2(u32_as_h2(sc)));
  const uint32_t mA = h2_as_u32(__low2half2(u32_as_h2(zp))), mB = h2_as_u32(__high2half2(u32_as_h2(zp)));
  const uint32_t x = xw[S_ >> 1], y = yw[S_ >> 2];
  a[0] = a3_value(x, y, S_, 0, sA, mA);
  a[1] = a3_value(x, y, S_, 1, sB, mB);
  a[2] = a3_value(x, y, S_, 2, sA, mA);
  a[3] = a3_value(x, y, S_, 3, sB, mB);
}

// ----------------------------------------------------------------------------- CB2 outlier corrections
// Side-list of a CB2 block (at 12D): {u8 n_ch, u8 total, 0, 0}, then n_ch
// 20-byte records {u8 channel, 0, u16 token mask, u8 value[16]} (e4m3 values,
// 0 where the token is not an outlier of the channel), channels ascending.
// A code slot holding an outlier stores code 0 (value c0 of its channel), so
// the correction of a channel is the sum over its outliers of (x - c0).  Both
// x (e4m3) and c0 (fp16) are exact in fp16, so it is applied as mma with exact
// operands: + the values, - c0 where the token mask is set.
//
// Records go kChunk at a time: the first chunk arrives with the block's codes
// (the prefetched bytes), later ones (rare: many channels with outliers) are
// copied from global memory into a per-warp bounce buffer, and the same code
// runs on every chunk.
constexpr int kChunk = 6;   // records per chunk
static_assert(4 + 20 * kChunk <= kOutPrefetch, "the first chunk must arrive with its block");

// {c0, c0}: fp16 bits of centroid 0 of codebook slot `slot` (the slot's (L, H)
// byte planes hold its low and high bytes at byte 0).
template <int D>
__device__ __forceinline__ uint32_t c0_bits(uint32_t blk_s, int slot) {
  const uint2 lh = lds64(blk_s + cb2_cb_off(D) + 8 * slot);
  return prmt(lh.x, lh.y, 0x4040u);
}

// {c0, c0}: the value code 0 of channel c stands for -- CB2: centroid 0;
// ASYM3: m (q = 0 gives fp16(0 * S + m) = m).
template <int D, int BLK>
__device__ __forceinline__ uint32_t code0_bits(uint32_t blk_s, int role, int c) {
  if constexpr (BLK == kBlkA3) {
    const uint32_t m = lds16(blk_s + a3_m_off(D) + 2 * a3_rho(role, c));
    return prmt(m, m, 0x1010u);
  } else if constexpr (BLK == kBlkCb2g) {   // blk_s: the group's codebook (its first page)
    const uint2 lh = lds64(blk_s + 8 * cb2_slot(role, c));
    return prmt(lh.x, lh.y, 0x4040u);
  } else {
    return c0_bits<D>(blk_s, cb2_slot(role, c));
  }
}
template <int D, int BLK>
__host__ __device__ constexpr int side_off() { return BLK == kBlkA3 ? a3_out_off(D) : cb2_out_off(D); }

// Scores of tokens g, g + 8 += sum over the chunk's channels c of
// q[h][c] * (x - c0[c]): one m16n8k8 tile, A = tokens x slots (slot i = the
// chunk's record i; slots >= nc are zero), B = Q^T gathered at the slots'
// channels.  recs: shared address of the chunk's first record.
template <int D, int NT, int BLK>
__device__ __forceinline__ void cb2_k_correct(uint32_t recs, int nc, uint32_t kb_s, uint32_t qsm_s, int G, int GS,
                                              int lane, float (&acc)[NT][4]) {
  const int g = lane >> 2, q4 = lane & 3;
  const int ia = 2 * q4;   // this lane's slots ia, ia + 1
  const bool va = ia < nc, vb = ia + 1 < nc;
  const uint32_t ra = recs + 20 * ia, rb = ra + 20;
  const uint32_t hA = va ? lds32(ra) : 0u, hB = vb ? lds32(rb) : 0u;   // {channel, 0, token mask}
  // + outlier values: a0 = tokens g, a1 = tokens g + 8 (slot ia low, ia + 1 high)
  const uint32_t x0 = (va ? lds8(ra + 4 + g) : 0u) | ((vb ? lds8(rb + 4 + g) : 0u) << 8);
  const uint32_t x1 = (va ? lds8(ra + 12 + g) : 0u) | ((vb ? lds8(rb + 12 + g) : 0u) << 8);
  const uint32_t a0 = e4m3x2_to_f16x2(x0), a1 = e4m3x2_to_f16x2(x1);
  // - c0 where flagged: shifting (mask_A | mask_B << 16) left by 7 - g puts
  // bits g / g + 8 of each mask in the sign bits of bytes 0 / 1 (A) and 2 / 3
  // (B); prmt's sign-replicate mode widens them into half masks.
  const uint32_t c01 =
      prmt(code0_bits<D, BLK>(kb_s, 0, hA & (D - 1)), code0_bits<D, BLK>(kb_s, 0, hB & (D - 1)), 0x5410u) ^ 0x80008000u;
  const uint32_t xm = prmt(hA, hB, 0x7632u) << (7 - g);
  const uint32_t n0 = c01 & prmt(xm, 0u, 0xAA88u), n1 = c01 & prmt(xm, 0u, 0xBB99u);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = nt * 8 + g;
    const float qa = (h < G && va) ? ldsf(qsm_s + 4 * ((hA & (D - 1)) * GS + h)) : 0.f;
    const float qb = (h < G && vb) ? ldsf(qsm_s + 4 * ((hB & (D - 1)) * GS + h)) : 0.f;
    const uint32_t b0 = h2_as_u32(__floats2half2_rn(qa, qb));
    mma1688(acc[nt], a0, a1, b0);
    mma1688(acc[nt], n0, n1, b0);
  }
}

// Output correction of the chunk's channels: corr[c][h] += sum_t p[t][h] *
// (x - c0[c]).  A = slots x tokens (row g = slot g; rows 8..15 are empty)
// against the page's P^T fragments; each (channel, head) is written by one lane.
template <int D, int NT, int BLK>
__device__ __forceinline__ void cb2_v_correct(uint32_t recs, int nc, uint32_t vb_s, const uint32_t (&phi)[NT][2],
                                              const uint32_t (&plo)[NT][2], uint32_t corr_s, int G, int GS,
                                              int lane) {
  const int g = lane >> 2, q4 = lane & 3;
  const int t0 = 2 * q4;
  const bool on = g < nc;   // every lane takes part in the mma; rows >= nc are zero
  const uint32_t r = recs + 20 * g;
  const uint32_t hr = on ? lds32(r) : 0u;
  const int ch = hr & (D - 1);
  const uint32_t a0 = on ? e4m3x2_to_f16x2(lds16(r + 4 + t0)) : 0u;
  const uint32_t a2 = on ? e4m3x2_to_f16x2(lds16(r + 12 + t0)) : 0u;
  // token masks: (mask << 7 - t0) / (mask << 6 - t0) hold bits t0 / t0 + 1 (and
  // + 8) in the sign bits of bytes 0 (and 1)
  const uint32_t m = hr >> 16, x = m << (7 - t0), y = m << (6 - t0);
  const uint32_t c0 = code0_bits<D, BLK>(vb_s, 1, ch) ^ 0x80008000u;
  const uint32_t n0 = c0 & prmt(x, y, 0xCC88u), n2 = c0 & prmt(x, y, 0xDD99u);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816(c, a0, 0u, a2, 0u, phi[nt][0], phi[nt][1]);
    mma16816(c, a0, 0u, a2, 0u, plo[nt][0], plo[nt][1]);
    mma16816(c, n0, 0u, n2, 0u, phi[nt][0], phi[nt][1]);
    mma16816(c, n0, 0u, n2, 0u, plo[nt][0], plo[nt][1]);
    const int h0 = nt * 8 + t0;
    const uint32_t ad = corr_s + 4 * (ch * GS + h0);
    if (on && h0 < G) sts32(ad, __float_as_uint(ldsf(ad) + c[0]));
    if (on && h0 + 1 < G) sts32(ad + 4, __float_as_uint(ldsf(ad + 4) + c[1]));
  }
}

// Copy records [base, base + nc) of a side-list from global memory into the
// warp's bounce buffer (nc <= kChunk; 5 * nc u32 words).
__device__ __forceinline__ void cb2_bounce(const uint8_t* side, int base, int nc, uint32_t bounce_s, int lane) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(side + 4 + 20 * base);
  if (lane < 5 * nc) sts32(bounce_s + 4 * lane, src[lane]);
  __syncwarp();
}

// ----------------------------------------------------------------------------- online softmax
// acc[p][nt][r]: scores in log2 units of page p for token g (r < 2) / g + 8
// (r >= 2) and head nt*8 + 2q + (r & 1), -inf for tokens that do not exist
// (the caller masks partial and absent pages).  Replaces them with p = 2^(s -
// m), raises the running max m only when a score exceeds it by more than
// kRescaleTh (so most pages skip the rescale), and updates the per-lane
// partial sums l.  Returns whether any lane changed its max (alpha holds the
// factors).
template <int PPI, int NT>
__device__ __forceinline__ bool online_softmax(float (&acc)[PPI][NT][4], float (&m)[NT][2], float (&l)[NT][2],
                                               float (&alpha)[NT][2]) {
  bool any = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mx = -INFINITY;
#pragma unroll
      for (int p = 0; p < PPI; ++p) mx = fmaxf(mx, fmaxf(acc[p][nt][j], acc[p][nt][2 + j]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const bool need = mx > m[nt][j] + kRescaleTh;
      const float mn = need ? mx : m[nt][j];
      alpha[nt][j] = need ? ex2(m[nt][j] - mn) : 1.f;
      m[nt][j] = mn;
      any |= need;
      const float mb = mn == -INFINITY ? 0.f : mn;   // no score yet: every p is 2^-inf = 0
      float sum = 0.f;
#pragma unroll
      for (int p = 0; p < PPI; ++p) {
        const float p0 = ex2(acc[p][nt][j] - mb);
        const float p1 = ex2(acc[p][nt][2 + j] - mb);
        acc[p][nt][j] = p0;
        acc[p][nt][2 + j] = p1;
        sum += p0 + p1;
      }
      l[nt][j] = l[nt][j] * alpha[nt][j] + sum;
    }
  }
  return __any_sync(0xffffffffu, any);
}

// Rescale the output accumulators (and the shared-memory outlier correction
// corr[c][h]) by alpha after a max change.
template <int D, int NT, bool kCorr, bool kO = true>
__device__ __forceinline__ void rescale_state(float (&o)[NT][D / 16][4], const float (&alpha)[NT][2],
                                              uint32_t corr_s, int G, int GS, int lane) {
  if (kO) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int s = 0; s < D / 16; ++s)
#pragma unroll
        for (int r = 0; r < 4; ++r) o[nt][s][r] *= alpha[nt][r & 1];
  }
  if (kCorr) {
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 8 * NT; ++h) {
      // alpha of head h lives in lanes with q = (h % 8) / 2, register h % 2
      const float ah = __shfl_sync(0xffffffffu, alpha[h >> 3][h & 1], (h & 7) >> 1);
      if (h < G)
        for (int c = lane; c < D; c += 32) {
          const uint32_t a = corr_s + 4 * (c * GS + h);
          sts32(a, __float_as_uint(ldsf(a) * ah));
        }
    }
    __syncwarp();
  }
}

// P (fp32, score layout) -> B fragments of P^T for the PV mma, as fp16 hi and
// lo parts.  Lane (g, q) needs P[token 2q, 2q+1 (+8)][head g]; those sit in
// lanes 8q + g/2 and 8q + g/2 + 4.
template <int NT>
__device__ __forceinline__ void p_frags(const float (&p)[NT][4], int g, int q4, uint32_t (&phi)[NT][2],
                                        uint32_t (&plo)[NT][2]) {
  const int srcA = 8 * q4 + (g >> 1), srcB = srcA + 4;
  const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    uint32_t xh, xl, yh, yl;
    split_hilo(p[nt][0], p[nt][1], xh, xl);
    split_hilo(p[nt][2], p[nt][3], yh, yl);
    phi[nt][0] = prmt(__shfl_sync(0xffffffffu, xh, srcA), __shfl_sync(0xffffffffu, xh, srcB), sel);
    phi[nt][1] = prmt(__shfl_sync(0xffffffffu, yh, srcA), __shfl_sync(0xffffffffu, yh, srcB), sel);
    plo[nt][0] = prmt(__shfl_sync(0xffffffffu, xl, srcA), __shfl_sync(0xffffffffu, xl, srcB), sel);
    plo[nt][1] = prmt(__shfl_sync(0xffffffffu, yl, srcA), __shfl_sync(0xffffffffu, yl, srcB), sel);
  }
}

// Store p into psm[t][h] (INT4 outlier corrections and the fp32 tail).
template <int NT>
__device__ __forceinline__ void store_p(const float (&p)[NT][4], float* psm, int G, int GS, int g, int q4) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = nt * 8 + 2 * q4 + j;
      if (h < G) {
        psm[g * GS + h] = p[nt][j];
        psm[(g + 8) * GS + h] = p[nt][2 + j];
      }
    }
}

// Add the INT4 K-outlier score corrections ds[t][h] to the lane's scores and clear them.
template <int NT>
__device__ __forceinline__ void apply_ds(float (&acc)[NT][4], float* ds, int G, int GS, int g, int q4) {
  __syncwarp();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = nt * 8 + 2 * q4 + j;
      if (h < G) {
        acc[nt][j] += ds[g * GS + h];
        acc[nt][2 + j] += ds[(g + 8) * GS + h];
        ds[g * GS + h] = 0.f;
        ds[(g + 8) * GS + h] = 0.f;
      }
    }
}

// Total per-token counts of tokens < ntok (16 count bytes at p).
__device__ __forceinline__ int masked_count_total(const uint8_t* p, int ntok) {
  int tot = 0;
#pragma unroll
  for (int t = 0; t < 16; ++t) tot += t < ntok ? p[t] : 0;
  return tot;
}

// Zero V^T fragment halves of tokens >= ntok (stale slots of a partial page).
__device__ __forceinline__ void mask_v_tokens(uint32_t (&a)[4], int ntok, int q4) {
  const int t0 = 2 * q4;
  const uint32_t m01 = (t0 < ntok ? 0xFFFFu : 0u) | (t0 + 1 < ntok ? 0xFFFF0000u : 0u);
  const uint32_t m23 = (t0 + 8 < ntok ? 0xFFFFu : 0u) | (t0 + 9 < ntok ? 0xFFFF0000u : 0u);
  a[0] &= m01; a[1] &= m01; a[2] &= m23; a[3] &= m23;
}

template <int D, int NT>
struct WarpState {
  float scl[NT][2];         // score scale of heads nt*8+2q, +1: softmax scale * log2(e) * 2^k_h
  float o[NT][D / 16][4];   // O^T accumulators: rows channel 16s+g (+8), cols head nt*8+2q (+1)
  float m[NT][2];           // running max (log2 units) of heads nt*8+2q, +1
  float l[NT][2];           // per-lane partial softmax sums
  // CB2_STATIC: the CTA's query at the K static channels (B fragment of the
  // m16n8k8 correction) and the output of the V static channels (rows = slots)
  uint32_t qs[NT];
  float sv[NT][4];
};
struct WarpSmem {
  const float* qsm;  // [D][GS] fp32 query of the CTA's G heads
  float* ds;         // [16][GS] INT4 K-outlier score corrections of the current page
  float* psm;        // [16][GS] probabilities of the current page (INT4, fp32 tail)
  float* corr;       // [D][GS] V-outlier output correction (rescaled with o)
  uint32_t qsm_s, corr_s;  // the same two arrays as shared-window addresses
  uint32_t bounce_s;       // CB2 side-list records beyond the prefetch (the psm area)
  int G, GS;
};

// ----------------------------------------------------------------------------- per-iteration processing
constexpr int32_t kBadEntry = 0x7FFFFFFF;  // page-table entry that failed validation
constexpr int32_t kNoPage = 0x7FFFFFFE;    // stage slot past the warp's last page

template <int FMT, int D>
__device__ __forceinline__ const uint8_t* block_src(const DecodeArgs& a, int kvh, int32_t e, int role) {
  const uint32_t u = (uint32_t)e, phys = u & 0x7FFFFFFFu;
  if (FMT == KVQ_FMT_TIERED && (u >> 31))
    return a.tier_pool + (((size_t)phys * a.Hkv + kvh) * 2 + role) * block_stride(kBlkFp8, D);
  return a.pool + (((size_t)phys * a.Hkv + kvh) * 2 + role) * block_stride(Fmt<FMT>::kMain, D);
}

// The lane's 2-bit codes of a CB2 block: one u16 per step, D/32 words.
template <int D>
__device__ __forceinline__ void load_codes(uint32_t blk_s, int lane, uint32_t (&w)[D / 32]) {
  if constexpr (D == 128) {
    const uint4 v = lds128(blk_s + 16 * lane);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = lds64(blk_s + 8 * lane);
    w[0] = v.x; w[1] = v.y;
  }
}

// Scores (in the scaled query's units) -> probabilities: each head's score
// scale st.scl undoes its query scale 2^-k_h and applies softmax_scale *
// log2(e); then the online softmax and the P^T fragments.
struct NoRescale {
  template <class A>
  __device__ __forceinline__ void operator()(const A&) const {}
};
// kO = false: the caller keeps the output in its own accumulators and
// rescales them in extra(alpha) (st.o is left alone).
template <int D, int NT, int PPI, bool kO = true, class Extra = NoRescale>
__device__ __forceinline__ void softmax_frags(WarpState<D, NT>& st, float (&acc)[PPI][NT][4], const int (&ntok)[PPI],
                                              float /*scale: in st.scl*/, const WarpSmem& sm, int lane, bool corr,
                                              uint32_t (&phi)[PPI][NT][2], uint32_t (&plo)[PPI][NT][2],
                                              Extra&& extra = Extra()) {
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int p = 0; p < PPI; ++p)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[p][nt][r] *= st.scl[nt][r & 1];
  // tokens past a partial or absent page's end: -inf (a warp-uniform branch,
  // taken only for those pages)
  bool partial = false;
#pragma unroll
  for (int p = 0; p < PPI; ++p) partial |= ntok[p] < kPage;
  if (partial) {
#pragma unroll
    for (int p = 0; p < PPI; ++p)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (g + 8 * (r >> 1) >= ntok[p]) acc[p][nt][r] = -INFINITY;
  }
  float alpha[NT][2];
  const bool rescale = online_softmax<PPI, NT>(acc, st.m, st.l, alpha);
  if (rescale) {
    if (corr) rescale_state<D, NT, true, kO>(st.o, alpha, sm.corr_s, sm.G, sm.GS, lane);
    else rescale_state<D, NT, false, kO>(st.o, alpha, sm.corr_s, sm.G, sm.GS, lane);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) st.sv[nt][r] *= alpha[nt][r & 1];
    extra(alpha);   // accumulators the caller keeps in another layout
  }
#pragma unroll
  for (int p = 0; p < PPI; ++p) p_frags<NT>(acc[p], g, q4, phi[p], plo[p]);
}

// CB2_STATIC, K side: scores[t][h] += sum_i q[h][ch_i] * x[t][ch_i] over the
// static fp16 channels -- one m16n8k8 tile, A = tokens x slots from the block,
// B = st.qs (the query at the static channels, gathered once per CTA).
template <int D, int NT>
__device__ __forceinline__ void cb2s_k_correct(uint32_t kb_s, int n_s, const uint32_t (&qs)[NT], int lane,
                                               float (&acc)[NT][4]) {
  const int g = lane >> 2, ia = 2 * (lane & 3);
  const uint32_t base = kb_s + cb2s_val_off(D) + 32 * ia + 2 * g;
  const bool va = ia < n_s, vb = ia + 1 < n_s;
  const uint32_t a0 = (va ? lds16(base) : 0u) | ((vb ? lds16(base + 32) : 0u) << 16);        // token g
  const uint32_t a1 = (va ? lds16(base + 16) : 0u) | ((vb ? lds16(base + 48) : 0u) << 16);   // token g + 8
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mma1688(acc[nt], a0, a1, qs[nt]);
}

// CB2_STATIC, V side: sv[slot][h] += sum_t p[t][h] * x[t][ch_slot] (A = slots x
// tokens, rows 8..15 empty), accumulated across pages in registers and
// rescaled with the output.
template <int D, int NT>
__device__ __forceinline__ void cb2s_v_accum(uint32_t vb_s, int n_s, const uint32_t (&phi)[NT][2],
                                             const uint32_t (&plo)[NT][2], int lane, float (&sv)[NT][4]) {
  const int g = lane >> 2, t0 = 2 * (lane & 3);
  const bool on = g < n_s;
  const uint32_t base = vb_s + cb2s_val_off(D) + 32 * g + 2 * t0;
  const uint32_t a0 = on ? lds32(base) : 0u, a2 = on ? lds32(base + 16) : 0u;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mma16816(sv[nt], a0, 0u, a2, 0u, phi[nt][0], phi[nt][1]);
    mma16816(sv[nt], a0, 0u, a2, 0u, plo[nt][0], plo[nt][1]);
  }
}

// CB2 pages (and, for the tiered format, FP8 tier pages), PPI at a time.
// kb_s / vb_s: shared addresses of the staged K / V blocks; an absent page
// points at the CTA's zero block, so it needs no masking outside the softmax.
// Each page's outlier corrections run over its side-list records in chunks of
// kChunk (a rolled loop; one chunk in the common case).
template <int FMT, int D, int NT, int PPI, class KDone, class VWait>
__device__ __forceinline__ void iter_cb2(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2],
                                         const uint32_t (&kb_s)[PPI], const uint32_t (&vb_s)[PPI],
                                         const int32_t (&ent)[PPI], const int (&ntok)[PPI], const DecodeArgs& a,
                                         int kvh, const WarpSmem& sm, int lane, KDone&& k_done, VWait&& v_wait) {
  constexpr int NS = D / 16;
  constexpr bool T = FMT == KVQ_FMT_TIERED;
  const int g = lane >> 2, q4 = lane & 3;
  bool tier[PPI];
#pragma unroll
  for (int p = 0; p < PPI; ++p) tier[p] = T && ent[p] < 0;

  constexpr bool A3 = Fmt<FMT>::kMain == kBlkA3, GRP = Fmt<FMT>::kGroup;
  constexpr int SIDE = side_off<D, Fmt<FMT>::kMain>();
  constexpr int CODES = GRP ? cb2g_code_off(D) : 0;   // codes within a page's (virtual) block
  // codebook of page p: its own block, or (group format) the group's first page
  auto kcb = [&](int p) { return GRP ? kb_s[0] : kb_s[p] + cb2_cb_off(D); };
  auto vcb = [&](int p) { return GRP ? vb_s[0] : vb_s[p] + cb2_cb_off(D); };
  float acc[PPI][NT][4];
  uint32_t kc[PPI][NS / 2], ky[PPI][A3 ? NS / 4 : 1];   // codes (ASYM3: low-bit and high-bit words)
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[p][nt][0] = acc[p][nt][1] = acc[p][nt][2] = acc[p][nt][3] = 0.f;
    if constexpr (A3) load_a3_words<D>(kb_s[p], lane, kc[p], ky[p]);
    else load_codes<D>(kb_s[p] + CODES, lane, kc[p]);
  }
  // The tiered format branches once per page on its tier, so each page's
  // steps form one block the compiler schedules freely (codebook loads
  // hoisted ahead of their use); a branch per (step, page) left small blocks
  // and measured 12% slower on the tiered workload.
  if constexpr (T) {
#pragma unroll
    for (int p = 0; p < PPI; ++p) {
      if (tier[p]) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          uint32_t ak[4];
          fp8_frag(lds64(kb_s[p] + 8 * NS * lane + 8 * s), ak);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(acc[p][nt], ak[0], ak[1], ak[2], ak[3], qf[nt][s][0], qf[nt][s][1]);
        }
        const float sk = ldsf(kb_s[p] + fp8_sc_off(D));   // the tier page's scale
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[p][nt][r] *= sk;
      } else {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          uint32_t ak[4];
          const uint32_t w16 = (s & 1) ? (kc[p][s >> 1] >> 16) : kc[p][s >> 1];
          cb2_k_frag(kcb(p) + 16 * q4, w16, s, ak);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(acc[p][nt], ak[0], ak[1], ak[2], ak[3], qf[nt][s][0], qf[nt][s][1]);
        }
      }
    }
  } else {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      KCols gcols;   // the group's codebook columns of step s, shared by its pages
      if constexpr (GRP) gcols = cb2_k_cols(kb_s[0] + 16 * q4, s);
#pragma unroll
      for (int p = 0; p < PPI; ++p) {
        uint32_t ak[4];
        const uint32_t w16 = (s & 1) ? (kc[p][s >> 1] >> 16) : kc[p][s >> 1];
        if constexpr (A3) a3_k_frag<D>(kb_s[p], kc[p], ky[p], s, q4, ak);
        else if constexpr (GRP) cb2_k_expand(gcols, w16, ak);
        else cb2_k_frag(kcb(p) + 16 * q4, w16, s, ak);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(acc[p][nt], ak[0], ak[1], ak[2], ak[3], qf[nt][s][0], qf[nt][s][1]);
      }
    }
  }
  if constexpr (FMT == KVQ_FMT_CB2_STATIC) {
#pragma unroll
    for (int p = 0; p < PPI; ++p) cb2s_k_correct<D, NT>(kb_s[p], a.n_static, st.qs, lane, acc[p]);
  }
  // outlier corrections: the first chunk (the records that arrived with the
  // block) runs without a branch -- on empty slots for a page with none, an
  // FP8 tier page or an absent one -- so it schedules with the code around
  // it; further chunks (rare) go through the rolled loop
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    if constexpr (FMT == KVQ_FMT_CB2_STATIC) break;
    const int n_ch = (T && tier[p]) ? 0 : min((int)lds8(kb_s[p] + SIDE), D);
    cb2_k_correct<D, NT, Fmt<FMT>::kMain>(kb_s[p] + SIDE + 4, min(kChunk, n_ch), GRP ? kb_s[0] : kb_s[p], sm.qsm_s,
                                          sm.G, sm.GS, lane, acc[p]);
#pragma unroll 1
    for (int base = kChunk; base < n_ch; base += kChunk) {
      cb2_bounce(block_src<FMT, D>(a, kvh, ent[p], 0) + SIDE, base, min(kChunk, n_ch - base), sm.bounce_s, lane);
      cb2_k_correct<D, NT, Fmt<FMT>::kMain>(sm.bounce_s, min(kChunk, n_ch - base), GRP ? kb_s[0] : kb_s[p], sm.qsm_s,
                                            sm.G, sm.GS, lane, acc[p]);
      __syncwarp();
    }
  }

  // Tiered: the V wait comes before the softmax and the K refill after it.
  // The copies land well ahead (the waits almost never find a block
  // missing), and the softmax then schedules with the code on either side
  // instead of between the refill's and the wait's branches: 3% on the
  // tiered workload, within noise (and not better) for the other formats.
  uint32_t phi[PPI][NT][2], plo[PPI][NT][2];
  if constexpr (T) {
    v_wait();
    softmax_frags<D, NT, PPI>(st, acc, ntok, a.scale_log2, sm, lane, Fmt<FMT>::kOutliers, phi, plo);
    k_done();   // the K blocks are no longer read
  } else {
    k_done();
    softmax_frags<D, NT, PPI>(st, acc, ntok, a.scale_log2, sm, lane, Fmt<FMT>::kOutliers, phi, plo);
    v_wait();
  }

  uint32_t vc[PPI][NS / 2], vy[PPI][A3 ? NS / 4 : 1];
  float sv[PPI];
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    if constexpr (A3) load_a3_words<D>(vb_s[p], lane, vc[p], vy[p]);
    else load_codes<D>(vb_s[p] + CODES, lane, vc[p]);
    sv[p] = (T && tier[p]) ? ldsf(vb_s[p] + fp8_sc_off(D)) : 1.f;
  }
  if constexpr (T) {   // one branch per page, as for K
#pragma unroll
    for (int p = 0; p < PPI; ++p) {
      if (tier[p]) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          uint32_t av[4];
          fp8_frag(lds64(vb_s[p] + 8 * NS * lane + 8 * s), av);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float t4[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(t4, av[0], av[1], av[2], av[3], phi[p][nt][0], phi[p][nt][1]);
            mma16816(t4, av[0], av[1], av[2], av[3], plo[p][nt][0], plo[p][nt][1]);
#pragma unroll
            for (int r = 0; r < 4; ++r) st.o[nt][s][r] = fmaf(sv[p], t4[r], st.o[nt][s][r]);
          }
        }
      } else {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          uint32_t av[4];
          const uint32_t w16 = (s & 1) ? (vc[p][s >> 1] >> 16) : vc[p][s >> 1];
          cb2_v_frag(vcb(p) + 16 * g, w16, s, av);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(st.o[nt][s], av[0], av[1], av[2], av[3], phi[p][nt][0], phi[p][nt][1]);
            mma16816(st.o[nt][s], av[0], av[1], av[2], av[3], plo[p][nt][0], plo[p][nt][1]);
          }
        }
      }
    }
  } else {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      uint4 gvcols;   // as gcols, V role
      if constexpr (GRP) gvcols = cb2_v_cols(vb_s[0] + 16 * g, s);
#pragma unroll
      for (int p = 0; p < PPI; ++p) {
        uint32_t av[4];
        const uint32_t w16 = (s & 1) ? (vc[p][s >> 1] >> 16) : vc[p][s >> 1];
        if constexpr (A3) a3_v_frag<D>(vb_s[p], vc[p], vy[p], s, g, av);
        else if constexpr (GRP) cb2_v_expand(gvcols, w16, av);
        else cb2_v_frag(vcb(p) + 16 * g, w16, s, av);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816(st.o[nt][s], av[0], av[1], av[2], av[3], phi[p][nt][0], phi[p][nt][1]);
          mma16816(st.o[nt][s], av[0], av[1], av[2], av[3], plo[p][nt][0], plo[p][nt][1]);
        }
      }
    }
  }
  if constexpr (FMT == KVQ_FMT_CB2_STATIC) {
#pragma unroll
    for (int p = 0; p < PPI; ++p) cb2s_v_accum<D, NT>(vb_s[p], a.n_static, phi[p], plo[p], lane, st.sv);
  }
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    if constexpr (FMT == KVQ_FMT_CB2_STATIC) break;
    const int n_ch = (T && tier[p]) ? 0 : min((int)lds8(vb_s[p] + SIDE), D);
    // as for K: the first chunk without a branch (empty slots write nothing)
    cb2_v_correct<D, NT, Fmt<FMT>::kMain>(vb_s[p] + SIDE + 4, min(kChunk, n_ch), GRP ? vb_s[0] : vb_s[p], phi[p],
                                          plo[p], sm.corr_s, sm.G, sm.GS, lane);
    __syncwarp();
#pragma unroll 1
    for (int base = kChunk; base < n_ch; base += kChunk) {
      cb2_bounce(block_src<FMT, D>(a, kvh, ent[p], 1) + SIDE, base, min(kChunk, n_ch - base), sm.bounce_s, lane);
      cb2_v_correct<D, NT, Fmt<FMT>::kMain>(sm.bounce_s, min(kChunk, n_ch - base), GRP ? vb_s[0] : vb_s[p], phi[p],
                                            plo[p], sm.corr_s, sm.G, sm.GS, lane);
      __syncwarp();
    }
  }
}

// ----------------------------------------------------------------------------- CUDA-core QK / PV (G <= 4)
// The same codebook pages with QK^T and PV on the FMA pipe instead of the
// tensor cores (kvq_config.decode_math = KVQ_DECODE_CUDA_CORES), for the
// small GQA groups whose heads fill only half of an m16n8 tile.  The code
// expansion is the same (cb2_k_frag / cb2_v_frag); each lane then
// multiplies its 8 values of a step in fp32:
//   QK: lane (g, q) holds K[t = g, g + 8][c = 16 s + 2q, +1, +8, +9]; partial
//       scores of its two tokens for the G heads (query rows read from the
//       fp32 query in shared memory), summed over the 4 lanes of a token;
//   PV: lane (g, q) holds V^T[c = 16 s + g, +8][t = 2q, 2q + 1, +8, +9];
//       partial outputs of its two channels for the G heads over its four
//       tokens (occ), summed over the 4 lanes once, after the page loop.
// The outlier corrections stay the exact-input mma tiles of iter_cb2.
template <int FMT, int D, int PPI, class KDone, class VWait>
__device__ __forceinline__ void iter_cb2_cc(WarpState<D, 1>& st, float (&occ)[D / 16][8], const uint32_t (&kb_s)[PPI],
                                            const uint32_t (&vb_s)[PPI], const int32_t (&ent)[PPI],
                                            const int (&ntok)[PPI], const DecodeArgs& a, int kvh, const WarpSmem& sm,
                                            int lane, KDone&& k_done, VWait&& v_wait) {
  constexpr int NS = D / 16;
  constexpr int SIDE = side_off<D, kBlkCb2>();
  const int g = lane >> 2, q4 = lane & 3;
  float sc[PPI][2][4];   // [page][token g, g + 8][head]
  uint32_t kc[PPI][NS / 2];
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int h = 0; h < 4; ++h) sc[p][i][h] = 0.f;
    load_codes<D>(kb_s[p], lane, kc[p]);
  }
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    // query rows of this lane's four channels (qsm is [D][4]: one row per channel)
    const int c0 = 16 * s + 2 * q4;
    const float4 q0 = *reinterpret_cast<const float4*>(sm.qsm + 4 * c0);
    const float4 q1 = *reinterpret_cast<const float4*>(sm.qsm + 4 * (c0 + 1));
    const float4 q8 = *reinterpret_cast<const float4*>(sm.qsm + 4 * (c0 + 8));
    const float4 q9 = *reinterpret_cast<const float4*>(sm.qsm + 4 * (c0 + 9));
#pragma unroll
    for (int p = 0; p < PPI; ++p) {
      uint32_t ak[4];
      cb2_k_frag(kb_s[p] + cb2_cb_off(D) + 16 * q4, (s & 1) ? (kc[p][s >> 1] >> 16) : kc[p][s >> 1], s, ak);
      const float2 k0 = __half22float2(u32_as_h2(ak[0]));   // token g, channels c0, c0 + 1
      const float2 k1 = __half22float2(u32_as_h2(ak[1]));   // token g + 8
      const float2 k2 = __half22float2(u32_as_h2(ak[2]));   // token g, channels c0 + 8, c0 + 9
      const float2 k3 = __half22float2(u32_as_h2(ak[3]));   // token g + 8
      const float qq[4][4] = {{q0.x, q0.y, q0.z, q0.w}, {q1.x, q1.y, q1.z, q1.w},
                              {q8.x, q8.y, q8.z, q8.w}, {q9.x, q9.y, q9.z, q9.w}};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        sc[p][0][h] = fmaf(k0.x, qq[0][h], fmaf(k0.y, qq[1][h], fmaf(k2.x, qq[2][h], fmaf(k2.y, qq[3][h], sc[p][0][h]))));
        sc[p][1][h] = fmaf(k1.x, qq[0][h], fmaf(k1.y, qq[1][h], fmaf(k3.x, qq[2][h], fmaf(k3.y, qq[3][h], sc[p][1][h]))));
      }
    }
  }
  // sum over the four lanes of a token, then the score layout of the mma path
  // (lane (g, q) holds heads 2q, 2q + 1; q >= 2 are padding heads)
  float acc[PPI][1][4];
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        sc[p][i][h] += __shfl_xor_sync(0xffffffffu, sc[p][i][h], 1);
        sc[p][i][h] += __shfl_xor_sync(0xffffffffu, sc[p][i][h], 2);
      }
    const bool lo = q4 == 0, on = q4 < 2;
    acc[p][0][0] = on ? (lo ? sc[p][0][0] : sc[p][0][2]) : 0.f;
    acc[p][0][1] = on ? (lo ? sc[p][0][1] : sc[p][0][3]) : 0.f;
    acc[p][0][2] = on ? (lo ? sc[p][1][0] : sc[p][1][2]) : 0.f;
    acc[p][0][3] = on ? (lo ? sc[p][1][1] : sc[p][1][3]) : 0.f;
  }
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    const int n_ch = min((int)lds8(kb_s[p] + SIDE), D);
#pragma unroll 1
    for (int base = 0; base < n_ch; base += kChunk) {
      uint32_t recs = kb_s[p] + SIDE + 4;
      if (base > 0) {
        cb2_bounce(block_src<FMT, D>(a, kvh, ent[p], 0) + SIDE, base, min(kChunk, n_ch - base), sm.bounce_s, lane);
        recs = sm.bounce_s;
      }
      cb2_k_correct<D, 1, kBlkCb2>(recs, min(kChunk, n_ch - base), kb_s[p], sm.qsm_s, sm.G, sm.GS, lane, acc[p]);
      __syncwarp();
    }
  }
  k_done();
  uint32_t phi[PPI][1][2], plo[PPI][1][2];
  softmax_frags<D, 1, PPI, false>(st, acc, ntok, a.scale_log2, sm, lane, true, phi, plo, [&](const float (&alpha)[1][2]) {
    // occ holds all four heads: head h's factor sits in lane (0, h / 2), register h % 2
    float ah[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) ah[h] = __shfl_sync(0xffffffffu, alpha[0][h & 1], h >> 1);
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int i = 0; i < 8; ++i) occ[s][i] *= ah[i & 3];
  });
  v_wait();
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    // probabilities of this lane's V tokens t = 2q, 2q + 1, 2q + 8, 2q + 9 for
    // every head: P[t][h] is register 2 (t >= 8) + h % 2 of lane (t % 8, h / 2)
    float pv[4][4];   // [token 2q, 2q+1, 2q+8, 2q+9][head]
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 2 * q4 + (i & 1) + 8 * (i >> 1);
        pv[i][h] = __shfl_sync(0xffffffffu, acc[p][0][2 * (i >> 1) + (h & 1)], 4 * (t & 7) + (h >> 1));
      }
    uint32_t vc[NS / 2];
    load_codes<D>(vb_s[p], lane, vc);
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      uint32_t av[4];
      cb2_v_frag(vb_s[p] + cb2_cb_off(D) + 16 * g, (s & 1) ? (vc[s >> 1] >> 16) : vc[s >> 1], s, av);
      const float2 v0 = __half22float2(u32_as_h2(av[0]));   // channel c, tokens 2q, 2q + 1
      const float2 v1 = __half22float2(u32_as_h2(av[1]));   // channel c + 8
      const float2 v2 = __half22float2(u32_as_h2(av[2]));   // channel c, tokens 2q + 8, 2q + 9
      const float2 v3 = __half22float2(u32_as_h2(av[3]));   // channel c + 8
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        occ[s][h] = fmaf(pv[0][h], v0.x, fmaf(pv[1][h], v0.y, fmaf(pv[2][h], v2.x, fmaf(pv[3][h], v2.y, occ[s][h]))));
        occ[s][4 + h] = fmaf(pv[0][h], v1.x, fmaf(pv[1][h], v1.y, fmaf(pv[2][h], v3.x, fmaf(pv[3][h], v3.y, occ[s][4 + h]))));
      }
    }
  }
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    const int n_ch = min((int)lds8(vb_s[p] + SIDE), D);
#pragma unroll 1
    for (int base = 0; base < n_ch; base += kChunk) {
      uint32_t recs = vb_s[p] + SIDE + 4;
      if (base > 0) {
        cb2_bounce(block_src<FMT, D>(a, kvh, ent[p], 1) + SIDE, base, min(kChunk, n_ch - base), sm.bounce_s, lane);
        recs = sm.bounce_s;
      }
      cb2_v_correct<D, 1, kBlkCb2>(recs, min(kChunk, n_ch - base), vb_s[p], phi[p], plo[p], sm.corr_s, sm.G, sm.GS,
                                   lane);
      __syncwarp();
    }
  }
}

// occ (lane (g, q): channels 16 s + g, +8 of every head, over its four tokens)
// summed over the 4 lanes of a channel pair and added into the output
// accumulators' layout (lane (g, q): heads 2q, 2q + 1).
template <int D>
__device__ __forceinline__ void fold_occ(WarpState<D, 1>& st, float (&occ)[D / 16][8], int lane) {
  const int q4 = lane & 3;
  const bool lo = q4 == 0, on = q4 < 2;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      occ[s][i] += __shfl_xor_sync(0xffffffffu, occ[s][i], 1);
      occ[s][i] += __shfl_xor_sync(0xffffffffu, occ[s][i], 2);
    }
    st.o[0][s][0] += on ? (lo ? occ[s][0] : occ[s][2]) : 0.f;
    st.o[0][s][1] += on ? (lo ? occ[s][1] : occ[s][3]) : 0.f;
    st.o[0][s][2] += on ? (lo ? occ[s][4] : occ[s][6]) : 0.f;
    st.o[0][s][3] += on ? (lo ? occ[s][5] : occ[s][7]) : 0.f;
  }
}

// The lane's E2M1 code words of a block: one u32 per step, NS contiguous words.
template <int D>
__device__ __forceinline__ void load_e2m1_words(uint32_t blk_s, int lane, uint32_t (&w)[D / 16]) {
#pragma unroll
  for (int i = 0; i < D / 64; ++i) {
    const uint4 v = lds128(blk_s + 4 * (D / 16) * lane + 16 * i);
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
}

// E2M1 pages (per-token format: the last page may hold fewer than 16 tokens).
template <int D, int NT, int PPI, class KDone, class VWait>
__device__ __forceinline__ void iter_e2m1(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2],
                                          const uint32_t (&kb_s)[PPI], const uint32_t (&vb_s)[PPI],
                                          const int (&ntok)[PPI], float scale, const WarpSmem& sm, int lane,
                                          KDone&& k_done, VWait&& v_wait) {
  constexpr int NS = D / 16;
  const int g = lane >> 2, q4 = lane & 3;
  float acc[PPI][NT][4];
  uint32_t kw[PPI][NS];
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[p][nt][0] = acc[p][nt][1] = acc[p][nt][2] = acc[p][nt][3] = 0.f;
    load_e2m1_words<D>(kb_s[p], lane, kw[p]);
  }
#pragma unroll
  for (int s = 0; s < NS; ++s)
#pragma unroll
    for (int p = 0; p < PPI; ++p) {
      uint32_t ak[4];
      e2m1_frag(kw[p][s], ak);
      const uint32_t sc = kb_s[p] + e2m1_sc_off(D) + 16 * s;
      const uint32_t sgs = e4m3x2_to_f16x2(lds8(sc + g) | (lds8(sc + g + 8) << 8));  // {s_g, s_g+8}
      // the token's scale in both halves: a half2 broadcast the multiply takes as an
      // operand select (byte permutes here measured 3% slower on fp4_32k)
      const __half2 sh = u32_as_h2(sgs), s0 = __low2half2(sh), s1 = __high2half2(sh);
      ak[0] = h2_as_u32(__hmul2(u32_as_h2(ak[0]), s0));
      ak[1] = h2_as_u32(__hmul2(u32_as_h2(ak[1]), s1));
      ak[2] = h2_as_u32(__hmul2(u32_as_h2(ak[2]), s0));
      ak[3] = h2_as_u32(__hmul2(u32_as_h2(ak[3]), s1));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(acc[p][nt], ak[0], ak[1], ak[2], ak[3], qf[nt][s][0], qf[nt][s][1]);
    }
  k_done();
  uint32_t phi[PPI][NT][2], plo[PPI][NT][2];
  softmax_frags<D, NT, PPI>(st, acc, ntok, scale, sm, lane, false, phi, plo);
  v_wait();
  // token masks of the page's valid slots (per-token formats: the last page may be partial)
  bool full = true;
  uint32_t m01[PPI], m23[PPI];
  uint32_t vw[PPI][NS];
#pragma unroll
  for (int p = 0; p < PPI; ++p) {
    full = full && ntok[p] == kPage;
    uint32_t a4[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
    mask_v_tokens(a4, ntok[p], q4);
    m01[p] = a4[0];
    m23[p] = a4[2];
    load_e2m1_words<D>(vb_s[p], lane, vw[p]);
  }
  auto pv_step = [&](int s, int p, bool masked) {
    uint32_t av[4];
    e2m1_frag(vw[p][s], av);
    const uint32_t sc = vb_s[p] + e2m1_sc_off(D) + 16 * s + 2 * q4;
    const uint32_t s01 = e4m3x2_to_f16x2(lds16(sc));
    const uint32_t s23 = e4m3x2_to_f16x2(lds16(sc + 8));
    av[0] = hmul2u(av[0], s01); av[1] = hmul2u(av[1], s01); av[2] = hmul2u(av[2], s23); av[3] = hmul2u(av[3], s23);
    if (masked) {
      av[0] &= m01[p]; av[1] &= m01[p]; av[2] &= m23[p]; av[3] &= m23[p];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(st.o[nt][s], av[0], av[1], av[2], av[3], phi[p][nt][0], phi[p][nt][1]);
      mma16816(st.o[nt][s], av[0], av[1], av[2], av[3], plo[p][nt][0], plo[p][nt][1]);
    }
  };
  if (full) {
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int p = 0; p < PPI; ++p) pv_step(s, p, false);
  } else {
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int p = 0; p < PPI; ++p) pv_step(s, p, true);
  }
}

// One INT4 page (per-token format; fp16 outliers in per-token slots).
template <int D, int NT, class KDone, class VWait>
__device__ __forceinline__ void iter_int4(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2], const uint8_t* kb,
                                          const uint8_t* vb, int ntok_, float scale, const WarpSmem& sm, int lane,
                                          KDone&& k_done, VWait&& v_wait) {
  constexpr int NS = D / 16, CAP = int4_cap(D), NG = D / 32;
  const int g = lane >> 2, q4 = lane & 3;
  const int ntok[1] = {ntok_};
  const uint32_t kb_s = smem_u32(kb), vb_s = smem_u32(vb);
  float acc[1][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[0][nt][0] = acc[0][nt][1] = acc[0][nt][2] = acc[0][nt][3] = 0.f;
  uint32_t kw[NS];
  load_e2m1_words<D>(kb_s, lane, kw);   // same word layout as E2M1: one u32 of nibbles per step
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int grp = s >> 1;
    const uint32_t z0 = lds32(kb_s + int4_sz_off(D) + 4 * (g * NG + grp));
    const uint32_t z1 = lds32(kb_s + int4_sz_off(D) + 4 * ((g + 8) * NG + grp));
    uint32_t ahi[4], alo[4];
    int4_k_frag(kw[s], fp16_bits_to_float(z0), fp16_bits_to_float(z0 >> 16), fp16_bits_to_float(z1),
                fp16_bits_to_float(z1 >> 16), ahi, alo);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(acc[0][nt], ahi[0], ahi[1], ahi[2], ahi[3], qf[nt][s][0], qf[nt][s][1]);
      mma16816(acc[0][nt], alo[0], alo[1], alo[2], alo[3], qf[nt][s][0], qf[nt][s][1]);
    }
  }
  // K outliers: scores[t][h] += q[h][c] * (x - m), m = the group's value of code 0
  if (ntok_ > 0 && masked_count_total(kb + int4_cnt_off(D), ntok_) > 0) {
    for (int e = lane; e < 16 * CAP; e += 32) {
      const int t = e / CAP, i = e - t * CAP;
      if (t < ntok_ && i < kb[int4_cnt_off(D) + t]) {
        const int ch = kb[int4_ch_off(D) + e] & (D - 1);
        const float x = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(kb + int4_val_off(D) + 2 * e));
        const float mz =
            fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(kb + int4_sz_off(D) + 4 * (t * NG + ch / 32) + 2));
        for (int h = 0; h < sm.G; ++h) atomicAdd(&sm.ds[t * sm.GS + h], sm.qsm[ch * sm.GS + h] * (x - mz));
      }
    }
    apply_ds<NT>(acc[0], sm.ds, sm.G, sm.GS, g, q4);
  }
  k_done();
  uint32_t phi[1][NT][2], plo[1][NT][2];
  softmax_frags<D, NT, 1>(st, acc, ntok, scale, sm, lane, true, phi, plo);
  v_wait();
  uint32_t vw[NS];
  load_e2m1_words<D>(vb_s, lane, vw);
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int grp = s >> 1;
    float S[4], M[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 2 * q4 + (i & 1) + 8 * (i >> 1);
      const uint32_t z = lds32(vb_s + int4_sz_off(D) + 4 * (t * NG + grp));
      S[i] = fp16_bits_to_float(z);
      M[i] = fp16_bits_to_float(z >> 16);
    }
    uint32_t ahi[4], alo[4];
    int4_v_frag(vw[s], S, M, ahi, alo);
    if (ntok_ < 16) {
      mask_v_tokens(ahi, ntok_, q4);
      mask_v_tokens(alo, ntok_, q4);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(st.o[nt][s], ahi[0], ahi[1], ahi[2], ahi[3], phi[0][nt][0], phi[0][nt][1]);
      mma16816(st.o[nt][s], ahi[0], ahi[1], ahi[2], ahi[3], plo[0][nt][0], plo[0][nt][1]);
      mma16816(st.o[nt][s], alo[0], alo[1], alo[2], alo[3], phi[0][nt][0], phi[0][nt][1]);
    }
  }
  if (ntok_ > 0 && masked_count_total(vb + int4_cnt_off(D), ntok_) > 0) {
    store_p<NT>(acc[0], sm.psm, sm.G, sm.GS, g, q4);
    __syncwarp();
    for (int e = lane; e < 16 * CAP; e += 32) {
      const int t = e / CAP, i = e - t * CAP;
      if (t < ntok_ && i < vb[int4_cnt_off(D) + t]) {
        const int ch = vb[int4_ch_off(D) + e] & (D - 1);
        const float x = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(vb + int4_val_off(D) + 2 * e));
        const float mz =
            fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(vb + int4_sz_off(D) + 4 * (t * NG + ch / 32) + 2));
        for (int h = 0; h < sm.G; ++h) atomicAdd(&sm.corr[ch * sm.GS + h], sm.psm[t * sm.GS + h] * (x - mz));
      }
    }
    __syncwarp();
  }
}

// The partial last page of a page format: ntail fp32 tokens in staging, on CUDA cores.
template <int D, int NT, bool kCorr>
__device__ __forceinline__ void page_tail(WarpState<D, NT>& st, const float* ks, const float* vs, int ntail,
                                          float scale, const WarpSmem& sm, int lane) {
  const int g = lane >> 2, q4 = lane & 3;
  float acc[1][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = g + 8 * (r >> 1), h = nt * 8 + 2 * q4 + (r & 1);
      float d = 0.f;
      if (t < ntail && h < sm.G)
        for (int c = 0; c < D; ++c) d = fmaf(sm.qsm[c * sm.GS + h], ks[t * D + c], d);
      acc[0][nt][r] = d;
    }
  const int ntok[1] = {ntail};
  uint32_t phi[1][NT][2], plo[1][NT][2];
  softmax_frags<D, NT, 1>(st, acc, ntok, scale, sm, lane, kCorr, phi, plo);
  store_p<NT>(acc[0], sm.psm, sm.G, sm.GS, g, q4);
  __syncwarp();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int s = 0; s < D / 16; ++s)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int c = 16 * s + g + 8 * (r >> 1), h = nt * 8 + 2 * q4 + (r & 1);
        if (h < sm.G) {
          float d = 0.f;
          for (int t = 0; t < ntail; ++t) d = fmaf(sm.psm[t * sm.GS + h], vs[t * D + c], d);
          st.o[nt][s][r] += d;
        }
      }
  __syncwarp();
}

// ----------------------------------------------------------------------------- split merge
// out[r] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the S split
// partials of the G rows r0 .. r0 + G - 1 (M = max_s m_s; 0 if no split saw a
// token).  Called by every thread of a CTA (blockDim.x a multiple of 32);
// `wts` is shared scratch of G * S floats.  For S <= 16 every thread loads its
// row's (m, l) pairs with its o columns and forms the weights itself (one
// round trip); otherwise one warp per row reduces the split maxima into
// weights first.  Either way the weighted sums of o and l run in split order.
// Shared by the combine kernel and the split kernel's fused merge, so both
// give the same bits.
__device__ __forceinline__ void merge_group(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                                            size_t r0, int G, int S, int D, void* out, int out_dtype, float* wts) {
  const int tid = threadIdx.x, nthreads = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int D4 = D / 4;
  auto store = [&](size_t o, const float (&r)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (out_dtype == KVQ_BF16) static_cast<__nv_bfloat16*>(out)[o + k] = __float2bfloat16_rn(r[k]);
      else static_cast<float*>(out)[o + k] = r[k];
    }
  };
  if (S <= 16) {
    // one round trip: each thread loads its row's S (m, l) pairs with its o
    // columns and forms the weights itself (the same values and order as below)
    for (int idx = tid; idx < G * D4; idx += nthreads) {
      const int h = idx / D4, c4 = idx % D4;
      const float4* po = reinterpret_cast<const float4*>(part_o + (r0 + h) * (size_t)S * D) + c4;
      const float2* pml = part_ml + (r0 + h) * S;
      float2 ml[16];
      float4 v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < S) {
          ml[k] = pml[k];
          v[k] = po[(size_t)k * D4];
        }
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < S) M = fmaxf(M, ml[k].x);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float L = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < S) {
          const float wgt = (ml[k].x == -INFINITY) ? 0.f : exp2f(ml[k].x - M);
          acc.x = fmaf(wgt, v[k].x, acc.x);
          acc.y = fmaf(wgt, v[k].y, acc.y);
          acc.z = fmaf(wgt, v[k].z, acc.z);
          acc.w = fmaf(wgt, v[k].w, acc.w);
          L = fmaf(wgt, ml[k].y, L);
        }
      const float r[4] = {L > 0.f ? acc.x / L : 0.f, L > 0.f ? acc.y / L : 0.f, L > 0.f ? acc.z / L : 0.f,
                          L > 0.f ? acc.w / L : 0.f};
      store((r0 + h) * D + 4 * c4, r);
    }
    return;
  }
  for (int i = tid; i < G * S; i += nthreads) wts[i] = part_ml[r0 * S + i].x;
  __syncthreads();
  // split weights 2^(m_s - M), one warp per head
  for (int h = warp; h < G; h += nthreads >> 5) {
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, wts[h * S + s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    __syncwarp();
    for (int s = lane; s < S; s += 32) {
      const float m = wts[h * S + s];
      wts[h * S + s] = (m == -INFINITY) ? 0.f : exp2f(m - M);
    }
  }
  __syncthreads();
  // outputs: a thread takes 4 adjacent columns of one row; each round keeps
  // 16 splits' o and l loads in flight; the weighted sums of o and of l run
  // in split order
  for (int idx = tid; idx < G * D4; idx += nthreads) {
    const int h = idx / D4, c4 = idx % D4;
    const float4* po = reinterpret_cast<const float4*>(part_o + (r0 + h) * (size_t)S * D) + c4;
    const float2* pml = part_ml + (r0 + h) * S;
    const float* wh = wts + h * S;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    for (int s = 0; s < S; s += 16) {
      float4 v[16];
      float l[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (s + k < S) {
          v[k] = po[(size_t)(s + k) * D4];
          l[k] = pml[s + k].y;
        }
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (s + k < S) {
          const float wgt = wh[s + k];
          acc.x = fmaf(wgt, v[k].x, acc.x);
          acc.y = fmaf(wgt, v[k].y, acc.y);
          acc.z = fmaf(wgt, v[k].z, acc.z);
          acc.w = fmaf(wgt, v[k].w, acc.w);
          L = fmaf(wgt, l[k], L);
        }
    }
    const float r[4] = {L > 0.f ? acc.x / L : 0.f, L > 0.f ? acc.y / L : 0.f, L > 0.f ? acc.z / L : 0.f,
                        L > 0.f ? acc.w / L : 0.f};
    store((r0 + h) * D + 4 * c4, r);
  }
}

// ----------------------------------------------------------------------------- split kernel
// Resident CTAs per SM the register budget is cut for (shared memory allows
// as many for G <= 8).
template <int FMT, int D, int NT, bool CC = false>
__host__ __device__ constexpr int min_ctas_per_sm() {
  return CC ? (D == 128 ? 3 : 4) : NT == 2 ? 2 : Fmt<FMT>::kMain == kBlkInt4 || Fmt<FMT>::kMain == kBlkE2m1 ? 3 : 4;
}

// CC: QK^T and PV of the codebook pages on CUDA cores (iter_cb2_cc; CB2 at G <= 4).
template <int FMT, int D, int NT, int W, bool CC = false>
__global__ void __launch_bounds__(W * 32, min_ctas_per_sm<FMT, D, NT, CC>()) decode_split_kernel(const DecodeArgs a) {
  using F = Fmt<FMT>;
  constexpr int NS = D / 16, PPI = F::kPPI, NK = Ring<FMT>::kK, NV = Ring<FMT>::kV;
  constexpr int HS = half_slot_bytes<FMT, D>();
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.G, GS = (G + 3) & ~3;

  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem) + w * (NK + NV);
  uint64_t* vbar = kbar + NK;
  uint8_t* const base = smem + mbar_bytes<FMT, W>();   // everything from here on is reused by the merge
  float* qsm = reinterpret_cast<float*>(base);
  uint8_t* zb = base + align16(D * GS * 4);
  uint8_t* wb = zb + zero_block_bytes<FMT, D>() + w * align16(warp_smem_bytes<FMT, D>(GS));
  constexpr int STG = stage_bytes<FMT, D>(), GPB = group_page_bytes<FMT, D>();
  uint8_t* kslots = wb;                    // NK K stages
  uint8_t* vslots = wb + NK * STG;         // NV V stages
  const uint32_t kslots_s = smem_u32(kslots), vslots_s = smem_u32(vslots);
  int32_t* meta = reinterpret_cast<int32_t*>(wb + (NK + NV) * STG);
  WarpSmem sm;
  sm.qsm = qsm;
  sm.ds = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(meta) + align16(4 * NK * PPI));
  sm.psm = sm.ds + (has_ds<FMT>() ? 16 * GS : 0);
  sm.corr = sm.psm + 16 * GS;
  sm.qsm_s = smem_u32(qsm);
  sm.corr_s = smem_u32(sm.corr);
  sm.bounce_s = smem_u32(sm.psm);
  sm.G = G;
  sm.GS = GS;
  const uint32_t zb_s = smem_u32(zb);

  // sequence length and this warp's first page-table entries are loaded
  // first, so their latency overlaps the query loads below
  int L = a.seq_lens[b];
  const int p0 = split * a.pps;
  auto page_of = [&](int li) {   // the sequence page of this warp's local page li
    return F::kGroup ? p0 + kGroupPages * (w + (li / kGroupPages) * W) + li % kGroupPages : p0 + w + li * W;
  };
  const int32_t* pt = a.page_table + (size_t)b * a.ppsm;
  const int spec_page = page_of(lane);
  const int win_spec = spec_page < min(p0 + a.pps, a.ppsm) ? pt[spec_page] : 0;

  // query of the CTA's G heads: fp32 in shared memory as [D][GS] (outlier
  // corrections gather its columns), fp16 B fragments in registers.  Each
  // head is scaled by a power of two 2^-k_h that puts its largest component
  // in [2^14, 2^15), so every bf16 value in range reaches the fp16 tensor-core
  // operand without overflow and, down to 2^-28 of the head's largest, without
  // loss; 2^k_h goes into that head's score scale (a power-of-two scaling
  // commutes exactly with the products and fp32 sums).
  // the per-head scales live in warp 0's probability scratch, which the
  // page loop first writes after the barrier that follows their last read
  float* const qscale = sm.psm - w * (align16(warp_smem_bytes<FMT, D>(GS)) / 4);
  const __nv_bfloat16* qg = a.q + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
  for (int i = threadIdx.x; i < GS * D; i += W * 32) {
    const int h = i / D, c = i % D;   // D is a power of two
    qsm[c * GS + h] = h < G ? __bfloat162float(qg[i]) : 0.f;
  }
  __syncthreads();
  for (int h = w; h < GS; h += W) {
    float mx = 0.f;
    for (int c = lane; c < D; c += 32) mx = fmaxf(mx, fabsf(qsm[c * GS + h]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int e = 0;
    frexpf(mx, &e);                             // mx in [2^(e-1), 2^e)
    const int k = mx > 0.f ? min(max(e - 15, -100), 100) : 0;
    if (lane == 0) qscale[h] = ldexpf(1.f, -k);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < GS * D; i += W * 32) qsm[i] *= qscale[i % GS];
  float scl[NT][2];   // score scale of heads nt*8+2q, +1 (read now: the scales' area is reused)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = nt * 8 + 2 * q4 + j;
      scl[nt][j] = h < G ? __fdiv_rn(a.scale_log2, qscale[h]) : a.scale_log2;   // exact: a power of two
    }
  for (int i = threadIdx.x; i < zero_block_bytes<FMT, D>() / 16; i += W * 32)
    reinterpret_cast<uint4*>(zb)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (has_ds<FMT>())
    for (int i = lane; i < 16 * GS; i += 32) sm.ds[i] = 0.f;
  if (F::kOutliers)
    for (int i = lane; i < D * GS; i += 32) sm.corr[i] = 0.f;
  if (lane == 0) {
    for (int j = 0; j < NK + NV; ++j) mbar_init(&kbar[j], 1);
    fence_mbar_init();
  }

  if (L > a.max_seq_len) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(a.status, KVQ_STATUS_SEQ_TOO_LONG);
    L = a.max_seq_len;
  }
  L = max(L, 0);
  const int n_all = (L + kPage - 1) / kPage;
  // pages stored as blocks (the group format quantizes whole groups)
  const int nq = F::kPaged ? (L / (kPage * F::kUnit)) * F::kUnit : n_all;
  const int p1 = min(p0 + a.pps, n_all);
  const int pq1 = min(p1, nq);
  // this warp's pages: every W-th page, or for the group format every W-th group
  int n_local;
  if constexpr (F::kGroup) {
    const int ng = max(pq1 - p0, 0) / kGroupPages;
    n_local = ng > w ? kGroupPages * ((ng - w + W - 1) / W) : 0;
  } else {
    n_local = pq1 > p0 + w ? (pq1 - p0 - w + W - 1) / W : 0;
  }
  const int n_iter = (n_local + PPI - 1) / PPI;

  // bytes copied per main-pool block (CB2_STATIC: only its n_s static channels' values)
  const int main_fetch = F::kMain == kBlkCb2s ? 12 * D + 16 + 32 * a.n_static : fetch_bytes<D>(F::kMain);

  // page-table window: lane j holds the entry of this warp's local page win_base + j
  int win_base = 0;
  int win = lane < n_local ? win_spec : 0;   // lane < n_local: a page of [p0, p1)

  // K copies of iteration `it` (local pages it*PPI .. it*PPI+PPI-1): validates
  // the page-table entries and records them in meta for the V copies and the
  // iteration itself.
  int k_issued = 0, v_issued = 0, k_waited = 0, v_waited = 0;
  auto issue_k = [&](int it) {
    if (it >= n_iter) return;
    const int slot = it % NK;
    int32_t ent[PPI];
#pragma unroll
    for (int j = 0; j < PPI; ++j) {
      const int li = it * PPI + j;
      ent[j] = kNoPage;
      if (li < n_local) {
        if (li - win_base >= 32) {
          win_base += 32;
          const int jj = win_base + lane;
          win = jj < n_local ? pt[page_of(jj)] : 0;
        }
        ent[j] = __shfl_sync(0xffffffffu, win, li - win_base);
      }
    }
    // lane j < PPI validates page j and issues its copy; lane 0 arms the
    // barrier with the total first (every lane fences its own copy against
    // the warp's earlier generic reads of the stage)
    int32_t e = kNoPage;
#pragma unroll
    for (int j = 0; j < PPI; ++j) e = lane == j ? ent[j] : e;
    uint32_t bytes = 0;
    if (lane < PPI) {
      int32_t m = kNoPage;
      if (e != kNoPage) {
        const uint32_t u = (uint32_t)e, phys = u & 0x7FFFFFFFu;
        const bool tier = (u >> 31) != 0;
        const bool ok =
            tier ? (FMT == KVQ_FMT_TIERED && phys < (uint32_t)a.num_tier_pages) : phys < (uint32_t)a.num_pages;
        if (ok) {
          m = e;
          bytes = tier ? fetch_bytes<D>(kBlkFp8) : F::kGroup ? (lane == 0 ? 8 * D + GPB : GPB) : main_fetch;
        } else {
          m = kBadEntry;
          atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        }
      }
      meta[slot * PPI + lane] = m;
    }
    const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
    if (lane == 0) {
      if (total == 0) mbar_arrive(&kbar[slot]);
      else mbar_arrive_expect_tx(&kbar[slot], total);
    }
    __syncwarp();
    if (bytes) {
      fence_proxy_async();
      bulk_g2s(kslots + slot * STG + copy_dst<FMT, D>(lane), block_src<FMT, D>(a, kvh, e, 0) + copy_src<FMT, D>(lane),
               bytes, &kbar[slot]);
    }
    __syncwarp();
    ++k_issued;
  };
  // V copies of iteration `it`; its entries were recorded by issue_k(it),
  // which ran earlier and whose meta slot is rewritten only by issue_k(it + NK).
  auto issue_v = [&](int it) {
    if (it >= n_iter) return;
    const int slot = it % NV, kslot = it % NK;
    // as issue_k: lane j < PPI copies page j
    const int32_t e = lane < PPI ? meta[kslot * PPI + lane] : kNoPage;
    const uint32_t bytes = (e == kNoPage || e == kBadEntry)       ? 0u
                           : (FMT == KVQ_FMT_TIERED && e < 0)     ? (uint32_t)fetch_bytes<D>(kBlkFp8)
                           : F::kGroup                            ? (uint32_t)(lane == 0 ? 8 * D + GPB : GPB)
                                                                  : (uint32_t)main_fetch;
    const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
    if (lane == 0) {
      if (total == 0) mbar_arrive(&vbar[slot]);
      else mbar_arrive_expect_tx(&vbar[slot], total);
    }
    __syncwarp();
    if (bytes) {
      fence_proxy_async();
      bulk_g2s(vslots + slot * STG + copy_dst<FMT, D>(lane), block_src<FMT, D>(a, kvh, e, 1) + copy_src<FMT, D>(lane),
               bytes, &vbar[slot]);
    }
    __syncwarp();
    ++v_issued;
  };

  __syncwarp();   // lane 0 initialised this warp's mbarriers
#pragma unroll 1
  for (int it = 0; it < NK; ++it) issue_k(it);
#pragma unroll 1
  for (int it = 0; it < NV; ++it) issue_v(it);

  __syncthreads();   // the scaled query
  uint32_t qf[NT][NS][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = nt * 8 + g;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const bool on = h < G;
      const int c = 16 * s + 2 * q4;
      const float x0 = on ? qsm[c * GS + h] : 0.f, x1 = on ? qsm[(c + 1) * GS + h] : 0.f;
      const float x8 = on ? qsm[(c + 8) * GS + h] : 0.f, x9 = on ? qsm[(c + 9) * GS + h] : 0.f;
      qf[nt][s][0] = h2_as_u32(__floats2half2_rn(x0, x1));
      qf[nt][s][1] = h2_as_u32(__floats2half2_rn(x8, x9));
    }
  }

  WarpState<D, NT> st;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    st.scl[nt][0] = scl[nt][0];
    st.scl[nt][1] = scl[nt][1];
#pragma unroll
    for (int s = 0; s < NS; ++s) st.o[nt][s][0] = st.o[nt][s][1] = st.o[nt][s][2] = st.o[nt][s][3] = 0.f;
    st.m[nt][0] = st.m[nt][1] = -INFINITY;
    st.l[nt][0] = st.l[nt][1] = 0.f;
    st.sv[nt][0] = st.sv[nt][1] = st.sv[nt][2] = st.sv[nt][3] = 0.f;
    st.qs[nt] = 0u;
  }
  int vch = 0;   // CB2_STATIC: the V static channel of slot g (lanes g < n_s)
  if constexpr (FMT == KVQ_FMT_CB2_STATIC) {
    const uint8_t* mk = a.static_mask + (size_t)kvh * 2 * a.n_static;   // K channels, then V channels
    const int ia = 2 * q4;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + g;
      const bool on = h < G;
      const float qa = (on && ia < a.n_static) ? qsm[(mk[ia] & (D - 1)) * GS + h] : 0.f;
      const float qb = (on && ia + 1 < a.n_static) ? qsm[(mk[ia + 1] & (D - 1)) * GS + h] : 0.f;
      st.qs[nt] = h2_as_u32(__floats2half2_rn(qa, qb));
    }
    vch = g < a.n_static ? (mk[a.n_static + g] & (D - 1)) : 0;
  }

  static_assert(!CC || (FMT == KVQ_FMT_CB2_OUTLIER && NT == 1), "CUDA-core path: CB2 pages, G <= 4");
  float occ[CC ? NS : 1][8];   // CC: per-lane partial outputs (see iter_cb2_cc)
#pragma unroll
  for (int s = 0; s < (CC ? NS : 1); ++s)
#pragma unroll
    for (int i = 0; i < 8; ++i) occ[s][i] = 0.f;

  bool timed_out = false;
#pragma unroll 1
  for (int it = 0; it < n_iter; ++it) {
    const int ks = it % NK, vs = it % NV;
    const bool ok = mbar_wait_bounded(&kbar[ks], (it / NK) & 1, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, ok)) {
      timed_out = true;
      break;
    }
    ++k_waited;
    int32_t ent[PPI];
    int ntok[PPI];
    uint32_t kb_s[PPI], vb_s[PPI];
    bool group_ok = true;
#pragma unroll
    for (int j = 0; j < PPI; ++j) {
      ent[j] = meta[ks * PPI + j];
      const int page = page_of(it * PPI + j);
      ntok[j] = (ent[j] == kBadEntry || ent[j] == kNoPage) ? 0 : (F::kPaged ? kPage : min(kPage, L - kPage * page));
      group_ok = group_ok && ntok[j] > 0;
      kb_s[j] = kslots_s + ks * STG + page_base<FMT, D>(j);
      vb_s[j] = vslots_s + vs * STG + page_base<FMT, D>(j);
      if (F::kPaged && !F::kGroup && ntok[j] == 0) kb_s[j] = vb_s[j] = zb_s;
    }
    if (F::kGroup && !group_ok) {   // a group with a bad page is left out whole
#pragma unroll
      for (int j = 0; j < PPI; ++j) {
        ntok[j] = 0;
        kb_s[j] = vb_s[j] = zb_s + page_base<FMT, D>(j);
      }
    }
    // k_done: the K slot is free, refill it; v_wait: the V blocks must have landed
    auto k_done = [&]() {
      __syncwarp();
      issue_k(it + NK);
    };
    bool v_ok = true;
    auto v_wait = [&]() {
      v_ok = __all_sync(0xffffffffu, mbar_wait_bounded(&vbar[vs], (it / NV) & 1, kWaitLimitNs));
      v_waited += v_ok;
    };
    if constexpr (CC) {
      iter_cb2_cc<FMT, D, PPI>(st, occ, kb_s, vb_s, ent, ntok, a, kvh, sm, lane, k_done, v_wait);
    } else if constexpr (F::kMain == kBlkCb2 || F::kMain == kBlkCb2s || F::kMain == kBlkA3 || F::kGroup) {
      iter_cb2<FMT, D, NT, PPI>(st, qf, kb_s, vb_s, ent, ntok, a, kvh, sm, lane, k_done, v_wait);
    } else if constexpr (F::kMain == kBlkE2m1) {
      iter_e2m1<D, NT, PPI>(st, qf, kb_s, vb_s, ntok, a.scale_log2, sm, lane, k_done, v_wait);
    } else {
      iter_int4<D, NT>(st, qf, kslots + ks * STG, vslots + vs * STG, ntok[0], a.scale_log2, sm, lane, k_done,
                       v_wait);
    }
    if (!v_ok) {
      timed_out = true;
      break;
    }
    __syncwarp();
    issue_v(it + NV);
  }
  if constexpr (CC) fold_occ<D>(st, occ, lane);
  if (timed_out) {
    if (lane == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
    // let copies still in flight land (bounded) before the CTA can exit
    for (int j = k_waited; j < k_issued; ++j) mbar_wait_bounded(&kbar[j % NK], (j / NK) & 1, kWaitLimitNs);
    for (int j = v_waited; j < v_issued; ++j) mbar_wait_bounded(&vbar[j % NV], (j / NV) & 1, kWaitLimitNs);
  }
  __syncwarp();
  if (!timed_out && lane == 0)
    for (int j = 0; j < NK + NV; ++j) mbar_inval(&kbar[j]);

  // partial last page of a page format, from fp32 staging
  // (the group format: up to kGroupPages staged pages of the partial last group)
  if (F::kPaged && !timed_out) {
    constexpr int ROWS = kPage * F::kUnit;   // staging rows per (sequence, kv head, K|V)
    const float* ks = a.staging + (((size_t)b * a.Hkv + kvh) * 2) * ROWS * D;
    for (int tp = max(nq, p0); tp < p1; ++tp)
      if ((tp - p0) % W == w) {
        const int off = (tp % F::kUnit) * kPage * D;
        page_tail<D, NT, F::kOutliers>(st, ks + off, ks + ROWS * D + off, min(kPage, L - kPage * tp), a.scale_log2, sm,
                                       lane);
      }
  }

  // ---- merge the W warps of the CTA and write the split's partial state
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      st.l[nt][j] += __shfl_xor_sync(0xffffffffu, st.l[nt][j], 4);
      st.l[nt][j] += __shfl_xor_sync(0xffffffffu, st.l[nt][j], 8);
      st.l[nt][j] += __shfl_xor_sync(0xffffffffu, st.l[nt][j], 16);
    }
  if (F::kOutliers) {
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int c = 16 * s + g + 8 * (r >> 1), h = nt * 8 + 2 * q4 + (r & 1);
          if (h < G) st.o[nt][s][r] += sm.corr[c * GS + h];
        }
  }
  __syncthreads();
  // merge area (reuses the stages): mo [W][GS][D], mm / ml [W][GS] (mm turns
  // into the warps' weights), mM / mL [GS]
  float* mo = reinterpret_cast<float*>(base + align16(D * GS * 4));
  float* mm = mo + W * GS * D;
  float* ml = mm + W * GS;
  float* mM = ml + W * GS;
  float* mL = mM + GS;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int c = 16 * s + g + 8 * (r >> 1), h = nt * 8 + 2 * q4 + (r & 1);
        if (h < G) mo[(w * GS + h) * D + c] = st.o[nt][s][r];
      }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = nt * 8 + 2 * q4 + j;
        if (h < G) {
          mm[w * GS + h] = st.m[nt][j];
          ml[w * GS + h] = st.l[nt][j];
        }
      }
  }
  if constexpr (FMT == KVQ_FMT_CB2_STATIC) {
    // the static V channels: slot g's output goes to channel vch (distinct per slot)
    __syncwarp();
    if (g < a.n_static) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = nt * 8 + 2 * q4 + j;
          if (h < G) mo[(w * GS + h) * D + vch] += st.sv[nt][j];
        }
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) M = fmaxf(M, mm[ww * GS + h]);
    float lv = 0.f;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) {
      const float mw = mm[ww * GS + h];
      const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : ex2(mw - M);
      mm[ww * GS + h] = f;
      lv = fmaf(f, ml[ww * GS + h], lv);
    }
    mM[h] = M;
    mL[h] = lv;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
    const int h = idx / D, c = idx % D;
    float ov = 0.f;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) ov = fmaf(mm[ww * GS + h], mo[(ww * GS + h) * D + c], ov);
    const size_t row = ((size_t)b * a.Hq + (size_t)kvh * G + h) * a.S + split;
    a.part_o[row * D + c] = ov;
    if (c == 0) a.part_ml[row] = make_float2(mM[h], mL[h]);
  }

  // ---- fused combine: the last CTA of this (sequence, kv head) to arrive merges the S partials
  if (a.out == nullptr) return;
  int* last = reinterpret_cast<int*>(mL + GS);
  // arrive with release semantics (the barrier orders every thread's partial
  // stores before thread 0's release); the last to arrive acquires the others'
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(&a.arrivals[(size_t)b * a.Hkv + kvh])
                 : "memory");
    *last = old == (uint32_t)(a.S - 1);
  }
  __syncthreads();
  if (!*last) return;
  merge_group(a.part_o, a.part_ml, (size_t)b * a.Hq + (size_t)kvh * G, G, a.S, D, a.out, a.out_dtype, mo);
  if (threadIdx.x == 0) a.arrivals[(size_t)b * a.Hkv + kvh] = 0u;   // ready for the next call
}

// ----------------------------------------------------------------------------- launch configuration
constexpr int kWarps = kWarpsPerCta;
struct KernelInfo {
  void* fn;
  size_t smem;
  int threads;
};

template <int FMT, int D, int NT, bool CC = false>
static KernelInfo kernel_info(int G) {
  const int GS = (G + 3) & ~3;
  const size_t plan = cta_smem_bytes<FMT, D, kWarps>(GS);
  const size_t merge = mbar_bytes<FMT, kWarps>() + align16(D * GS * 4) + (size_t)kWarps * GS * D * 4 +
                       2 * (size_t)kWarps * GS * 4 + 2 * (size_t)GS * 4 + 16;
  return {reinterpret_cast<void*>(decode_split_kernel<FMT, D, NT, kWarps, CC>), plan > merge ? plan : merge,
          kWarps * 32};
}

template <int FMT>
static KernelInfo kernel_info_fmt(int D, int G) {
  if (D == 64) return G <= 8 ? kernel_info<FMT, 64, 1>(G) : kernel_info<FMT, 64, 2>(G);
  return G <= 8 ? kernel_info<FMT, 128, 1>(G) : kernel_info<FMT, 128, 2>(G);
}

// One translation unit per format instantiates its kernels.
KernelInfo decode_kernel_int4(int D, int G);
KernelInfo decode_kernel_e2m1(int D, int G);
KernelInfo decode_kernel_cb2(int D, int G, bool cuda_cores);
KernelInfo decode_kernel_tiered(int D, int G);
KernelInfo decode_kernel_cb2s(int D, int G);
KernelInfo decode_kernel_a3(int D, int G);
KernelInfo decode_kernel_cb2g(int D, int G);

}  // namespace kvq
