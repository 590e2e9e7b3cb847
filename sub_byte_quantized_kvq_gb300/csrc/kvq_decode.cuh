// kvq_decode.cuh -- split-K decode attention over the quantized paged cache with
// dequantization fused in, and the split-combine kernel.
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
// partial softmax states a second kernel merges.
//
// Design (GB300, sm_103a):
//  * grid (splits, kv heads, sequences); a CTA owns one (sequence, kv head,
//    split) and all G query heads of that kv head; each of its W warps streams
//    its own pages (page p0 + w, p0 + w + W, ...), with its own online-softmax
//    state, and the warps merge in shared memory at the end.
//  * each warp runs an NSTAGE-deep ring of bulk asynchronous copies
//    (cp.async.bulk + mbarrier): one copy per block, K and V of a page per
//    stage; no register staging, no TMA multicast.
//  * QK^T: A = K (16 tokens x 16 channels, built in registers from the codes),
//    B = Q^T (16 channels x 8 heads, fp16, loaded once).  PV: A = V^T (16
//    channels x 16 tokens, built in registers), B = P^T (fp16 hi + lo split of
//    the fp32 probabilities, so P carries ~22 bits).  mma.sync m16n8k16 with
//    fp32 accumulation; the layouts in include/kvq.h make every A register one
//    or two byte-permutes of shared memory words.
//  * outliers: a code slot holding an outlier stores 0; each outlier adds
//    q.(x - c0) to its token's scores (K) and p.(x - c0) to a per-warp fp32
//    correction of the output (V), both through shared-memory atomics.
//  * the partial last page of page formats (fp32 staging) is done on CUDA
//    cores in fp32.
#pragma once
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kEntSmem = 64;          // CB2 entries that fit in a stage
constexpr float kRescaleTh = 8.0f;    // lazy rescale: p stays <= 2^8

template <int FMT>
struct Fmt {
  static constexpr bool kPaged = (FMT == KVQ_FMT_CB2_OUTLIER || FMT == KVQ_FMT_TIERED);
  static constexpr int kMain = FMT == KVQ_FMT_TIERED ? kBlkCb2 : FMT;
  static constexpr bool kOutliers = (kMain == kBlkInt4 || kMain == kBlkCb2);
};

// Bytes copied to shared memory per block (the kernel reads nothing else of it,
// except CB2 outlier entries past the prefetched ones).
template <int D>
__host__ __device__ constexpr int fetch_bytes(int blk) {
  return blk == kBlkInt4 ? 10 * D + 16 + 48 * int4_cap(D)
       : blk == kBlkE2m1 ? 9 * D
       : blk == kBlkCb2  ? 12 * D + 16 + 2 * kEntSmem
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

// Shared-memory plan: [qsm: D x GS fp32] then per warp:
// [stages: NSTAGE x 2 half-slots][mbar x NSTAGE][meta x NSTAGE][ds 16 x GS][psm 16 x GS][corr D x GS]
template <int FMT, int D, int NSTAGE>
__host__ __device__ constexpr int warp_smem_bytes(int GS) {
  return NSTAGE * 2 * half_slot_bytes<FMT, D>() + 8 * NSTAGE + align16(4 * NSTAGE) + 16 * GS * 4 +
         16 * GS * 4 + (Fmt<FMT>::kOutliers ? D * GS * 4 : 0);
}
template <int FMT, int D, int W, int NSTAGE>
__host__ __device__ constexpr int cta_smem_bytes(int GS) {
  return align16(D * GS * 4) + W * align16(warp_smem_bytes<FMT, D, NSTAGE>(GS));
}

// ----------------------------------------------------------------------------- fragment builders
// Each returns the four A registers (f16x2) of step s for this lane.

// CB2, K role: channels x = 16s + 2q, y = x + 1 (and +8); tokens g, g + 8.
template <int D>
__device__ __forceinline__ void cb2_k_frag(const uint8_t* kb, uint32_t w16, int s, int q4, uint32_t (&a)[4]) {
  const uint32_t sel1 = (w16 & 0x3333u) | 0x4040u;
  const uint32_t sel2 = ((w16 >> 2) & 0x3333u) | 0x4040u;
  const uint4 ca = *reinterpret_cast<const uint4*>(kb + cb2_cb_off(D) + 8 * (16 * s + 2 * q4));
  const uint4 cb = *reinterpret_cast<const uint4*>(kb + cb2_cb_off(D) + 8 * (16 * s + 2 * q4 + 8));
  uint32_t lo = prmt(ca.x, ca.z, sel1), hi = prmt(ca.y, ca.w, sel1);
  a[0] = prmt(lo, hi, 0x5140u);
  a[1] = prmt(lo, hi, 0x7362u);
  lo = prmt(cb.x, cb.z, sel2);
  hi = prmt(cb.y, cb.w, sel2);
  a[2] = prmt(lo, hi, 0x5140u);
  a[3] = prmt(lo, hi, 0x7362u);
}

// CB2, V role: channels cA = 16s + g, cB = cA + 8; tokens 2q, 2q+1 (and +8).
template <int D>
__device__ __forceinline__ void cb2_v_frag(const uint8_t* vb, uint32_t w16, int s, int g, uint32_t (&a)[4]) {
  const uint32_t sel1 = (w16 & 0x3333u) | 0x4400u;
  const uint32_t sel2 = ((w16 >> 2) & 0x3333u) | 0x4400u;
  const uint4 c = *reinterpret_cast<const uint4*>(vb + cb2_cb_off(D) + 16 * (8 * s + g));
  uint32_t lo = prmt(c.x, c.z, sel1), hi = prmt(c.y, c.w, sel1);
  a[0] = prmt(lo, hi, 0x5140u);
  a[1] = prmt(lo, hi, 0x7362u);
  lo = prmt(c.x, c.z, sel2);
  hi = prmt(c.y, c.w, sel2);
  a[2] = prmt(lo, hi, 0x5140u);
  a[3] = prmt(lo, hi, 0x7362u);
}

// FP8 e4m3 codes, either role: slot k = byte k of the lane's 8 bytes for step s.
__device__ __forceinline__ void fp8_frag(uint2 wd, uint32_t (&a)[4]) {
  a[0] = e4m3x2_to_f16x2(wd.x & 0xFFFFu);
  a[1] = e4m3x2_to_f16x2(wd.x >> 16);
  a[2] = e4m3x2_to_f16x2(wd.y & 0xFFFFu);
  a[3] = e4m3x2_to_f16x2(wd.y >> 16);
}

// E2M1 codes: slot k = nibble k of the lane's u32 for step s; register i holds
// slots 2i, 2i+1 = byte i.  sc01 / sc23: f16x2 scales for registers 0,1 / 2,3
// (K: {s_g, s_g} / {s_g8, s_g8} interleaved per register; see callers).
__device__ __forceinline__ void e2m1_frag(uint32_t wd, uint32_t (&a)[4]) {
  a[0] = e2m1x2_to_f16x2(wd & 0xFFu);
  a[1] = e2m1x2_to_f16x2((wd >> 8) & 0xFFu);
  a[2] = e2m1x2_to_f16x2((wd >> 16) & 0xFFu);
  a[3] = e2m1x2_to_f16x2(wd >> 24);
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t x, uint32_t y) {
  return h2_as_u32(__hmul2(u32_as_h2(x), u32_as_h2(y)));
}

// INT4 codes: x = q * S + m in fp32 (per token, group of 32), split into an
// fp16 high part and an fp16 residual so the tensor-core product keeps ~22 bits.
// Register r holds slots 2r, 2r+1 (nibbles 2r, 2r+1 of the step's u32).
__device__ __forceinline__ void split_hilo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(x0, x1);
  float2 hf = __half22float2(h);
  hi = h2_as_u32(h);
  lo = h2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}
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

// ----------------------------------------------------------------------------- outlier side-list helpers
// Inclusive prefix sums of 16 per-token counts held in four u32 words, one byte
// per token (sums stay below 256: at most 16 * 14 entries).
struct CountPrefix {
  uint32_t p[4];
  int total;
};
__device__ __forceinline__ CountPrefix count_prefix(uint4 c) {
  CountPrefix r;
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t carry = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r.p[i] = (w[i] + carry) * 0x01010101u;  // byte j: carry + counts 0..j of this word
    carry = r.p[i] >> 24;
  }
  r.total = (int)carry;
  return r;
}
// Token holding entry e (entries are sorted by token): number of tokens whose
// inclusive prefix is <= e.
__device__ __forceinline__ int token_of(const CountPrefix& cp, int e) {
  const uint32_t eb = (uint32_t)e * 0x01010101u;
  int t = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) t += __popc(__vcmpleu4(cp.p[i], eb)) >> 3;
  return t;
}
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  return __low2float(u32_as_h2(e4m3x2_to_f16x2(byte & 0xFFu)));
}
__device__ __forceinline__ float fp16_bits_to_float(uint32_t bits) {
  return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}

// ----------------------------------------------------------------------------- online softmax
// acc[nt][r]: scores in log2 units for token g (r < 2) / g + 8 (r >= 2) and head
// nt*8 + 2q + (r & 1).  Replaces them with p = 2^(s - m) (0 for tokens >= ntok),
// updates the running max m (raised only when a score exceeds it by more than
// kRescaleTh, so most pages skip the rescale) and the per-lane partial sums l.
// Returns whether any lane changed its max; alpha holds the rescale factors.
template <int NT>
__device__ __forceinline__ bool online_softmax(float (&acc)[NT][4], int ntok, int g, float (&m)[NT][2],
                                               float (&l)[NT][2], float (&alpha)[NT][2]) {
  const bool v0 = g < ntok, v1 = g + 8 < ntok;
  bool any = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mx = fmaxf(v0 ? acc[nt][j] : -INFINITY, v1 ? acc[nt][2 + j] : -INFINITY);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const bool need = mx > m[nt][j] + kRescaleTh;
      const float mn = need ? mx : m[nt][j];
      alpha[nt][j] = need ? exp2f(m[nt][j] - mn) : 1.f;
      m[nt][j] = mn;
      any |= need;
      const float p0 = v0 ? exp2f(acc[nt][j] - mn) : 0.f;
      const float p1 = v1 ? exp2f(acc[nt][2 + j] - mn) : 0.f;
      acc[nt][j] = p0;
      acc[nt][2 + j] = p1;
      l[nt][j] = l[nt][j] * alpha[nt][j] + p0 + p1;
    }
  }
  return __any_sync(0xffffffffu, any);
}

// Rescale the output accumulators (and the shared-memory outlier correction
// corr[c][h]) by alpha after a max change.
template <int D, int NT, bool kCorr>
__device__ __forceinline__ void rescale_state(float (&o)[NT][D / 16][4], const float (&alpha)[NT][2], float* corr,
                                              int G, int GS, int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int s = 0; s < D / 16; ++s)
#pragma unroll
      for (int r = 0; r < 4; ++r) o[nt][s][r] *= alpha[nt][r & 1];
  if (kCorr) {
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 8 * NT; ++h) {
      // alpha of head h lives in lanes with q = (h % 8) / 2, register h % 2
      const float ah = __shfl_sync(0xffffffffu, alpha[h >> 3][h & 1], (h & 7) >> 1);
      if (h < G)
        for (int c = lane; c < D; c += 32) corr[c * GS + h] *= ah;
    }
    __syncwarp();
  }
}

// P (fp32, score layout) -> B fragments of P^T for the PV mma, as an fp16 high
// part and an fp16 residual.  Lane (g, q) needs P[token 2q, 2q+1 (+8)][head g];
// those sit in lanes 8q + g/2 and 8q + g/2 + 4.
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

// Store p into psm[t][h] (for the V outlier correction and the fp32 tail).
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

// Add the K-outlier score corrections ds[t][h] to the lane's scores and clear them.
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

// ----------------------------------------------------------------------------- per-page processing
// Per-warp state and the shared-memory scratch of one warp.
template <int D, int NT>
struct WarpState {
  float o[NT][D / 16][4];   // O^T accumulators: rows channel 16s+g (+8), cols head nt*8+2q (+1)
  float m[NT][2];           // running max (log2 units) of heads nt*8+2q, +1
  float l[NT][2];           // per-lane partial softmax sums
};
struct WarpSmem {
  const float* qsm;  // [D][GS] fp32 query of the CTA's G heads
  float* ds;         // [16][GS] K-outlier score corrections of the current page
  float* psm;        // [16][GS] probabilities of the current page
  float* corr;       // [D][GS] V-outlier output correction (rescaled with o)
  int G, GS;
};

template <int D, int NT, bool kCorr>
__device__ __forceinline__ void softmax_and_frags(WarpState<D, NT>& st, float (&acc)[NT][4], int ntok, float scale,
                                                  const WarpSmem& sm, int lane, uint32_t (&phi)[NT][2],
                                                  uint32_t (&plo)[NT][2]) {
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[nt][r] *= scale;
  float alpha[NT][2];
  if (online_softmax<NT>(acc, ntok, g, st.m, st.l, alpha))
    rescale_state<D, NT, kCorr>(st.o, alpha, sm.corr, sm.G, sm.GS, lane);
  p_frags<NT>(acc, g, q4, phi, plo);
}

// K outliers of a CB2 block: scores[t][h] += q[h][c] * (x - c0[c]).
template <int D>
__device__ __forceinline__ void cb2_k_outliers(const uint8_t* kb, const uint8_t* kglob, int ent_prefetch,
                                               const WarpSmem& sm, int lane, bool& any) {
  CountPrefix cp = count_prefix(*reinterpret_cast<const uint4*>(kb + cb2_cnt_off(D)));
  cp.total = min(cp.total, 16 * kmax_outliers(D));  // a corrupt side-list never reads past its block
  any = cp.total > 0;
  for (int e = lane; e < cp.total; e += 32) {
    const uint32_t ent = e < ent_prefetch ? *reinterpret_cast<const uint16_t*>(kb + cb2_ent_off(D) + 2 * e)
                                          : __ldg(reinterpret_cast<const uint16_t*>(kglob + cb2_ent_off(D) + 2 * e));
    const int t = min(token_of(cp, e), kPage - 1), ch = ent & (D - 1);
    const uint8_t* cbp = kb + cb2_cb_off(D) + 8 * ch;  // K codebook slot = channel
    const float c0 = fp16_bits_to_float(cbp[0] | (cbp[4] << 8));
    const float delta = e4m3_to_float(ent >> 8) - c0;
    for (int h = 0; h < sm.G; ++h) atomicAdd(&sm.ds[t * sm.GS + h], sm.qsm[ch * sm.GS + h] * delta);
  }
}

// V outliers of a CB2 block: corr[c][h] += p[t][h] * (x - c0[c]).  psm must hold p.
template <int D>
__device__ __forceinline__ void cb2_v_outliers(const uint8_t* vb, const uint8_t* vglob, int ent_prefetch,
                                               const CountPrefix& cp, const WarpSmem& sm, int lane) {
  for (int e = lane; e < cp.total; e += 32) {
    const uint32_t ent = e < ent_prefetch ? *reinterpret_cast<const uint16_t*>(vb + cb2_ent_off(D) + 2 * e)
                                          : __ldg(reinterpret_cast<const uint16_t*>(vglob + cb2_ent_off(D) + 2 * e));
    const int t = min(token_of(cp, e), kPage - 1), ch = ent & (D - 1);
    const uint8_t* cbp = vb + cb2_cb_off(D) + 8 * cb2_slot(1, ch);
    const float c0 = fp16_bits_to_float(cbp[0] | (cbp[4] << 8));
    const float delta = e4m3_to_float(ent >> 8) - c0;
    for (int h = 0; h < sm.G; ++h) atomicAdd(&sm.corr[ch * sm.GS + h], sm.psm[t * sm.GS + h] * delta);
  }
}

template <int D>
__device__ __forceinline__ void load_codes(const uint8_t* p, uint32_t (&w)[D / 32]) {
  if constexpr (D == 128) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  }
}

// One CB2 page (K block kb, V block vb in shared memory; kglob/vglob the same
// blocks in global memory for entries beyond the prefetched ones).
template <int D, int NT>
__device__ __forceinline__ void page_cb2(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2], const uint8_t* kb,
                                         const uint8_t* vb, const uint8_t* kglob, const uint8_t* vglob,
                                         int ent_prefetch, float scale, const WarpSmem& sm, int lane) {
  constexpr int NS = D / 16;
  const int g = lane >> 2, q4 = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  uint32_t kc[NS / 2];
  load_codes<D>(kb + 2 * NS * lane, kc);
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    uint32_t a[4];
    cb2_k_frag<D>(kb, (s & 1) ? (kc[s >> 1] >> 16) : kc[s >> 1], s, q4, a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a[0], a[1], a[2], a[3], qf[nt][s][0], qf[nt][s][1]);
  }
  bool any_k;
  cb2_k_outliers<D>(kb, kglob, ent_prefetch, sm, lane, any_k);
  if (any_k) apply_ds<NT>(acc, sm.ds, sm.G, sm.GS, g, q4);

  uint32_t phi[NT][2], plo[NT][2];
  softmax_and_frags<D, NT, true>(st, acc, 16, scale, sm, lane, phi, plo);

  uint32_t vc[NS / 2];
  load_codes<D>(vb + 2 * NS * lane, vc);
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    uint32_t a[4];
    cb2_v_frag<D>(vb, (s & 1) ? (vc[s >> 1] >> 16) : vc[s >> 1], s, g, a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(st.o[nt][s], a[0], a[1], a[2], a[3], phi[nt][0], phi[nt][1]);
      mma16816(st.o[nt][s], a[0], a[1], a[2], a[3], plo[nt][0], plo[nt][1]);
    }
  }
  CountPrefix cpv = count_prefix(*reinterpret_cast<const uint4*>(vb + cb2_cnt_off(D)));
  cpv.total = min(cpv.total, 16 * kmax_outliers(D));
  if (cpv.total > 0) {
    store_p<NT>(acc, sm.psm, sm.G, sm.GS, g, q4);
    __syncwarp();
    cb2_v_outliers<D>(vb, vglob, ent_prefetch, cpv, sm, lane);
  }
}

// One FP8 tier page: e4m3 codes, one fp32 scale per block (scores and PV scaled in fp32).
template <int D, int NT, bool kCorr>
__device__ __forceinline__ void page_fp8(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2], const uint8_t* kb,
                                         const uint8_t* vb, float scale, const WarpSmem& sm, int lane) {
  constexpr int NS = D / 16;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    uint32_t a[4];
    fp8_frag(*reinterpret_cast<const uint2*>(kb + 8 * NS * lane + 8 * s), a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a[0], a[1], a[2], a[3], qf[nt][s][0], qf[nt][s][1]);
  }
  const float sk = *reinterpret_cast<const float*>(kb + fp8_sc_off(D));
  const float sv = *reinterpret_cast<const float*>(vb + fp8_sc_off(D));
  uint32_t phi[NT][2], plo[NT][2];
  softmax_and_frags<D, NT, kCorr>(st, acc, 16, scale * sk, sm, lane, phi, plo);
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    uint32_t a[4];
    fp8_frag(*reinterpret_cast<const uint2*>(vb + 8 * NS * lane + 8 * s), a);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float t4[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816(t4, a[0], a[1], a[2], a[3], phi[nt][0], phi[nt][1]);
      mma16816(t4, a[0], a[1], a[2], a[3], plo[nt][0], plo[nt][1]);
#pragma unroll
      for (int r = 0; r < 4; ++r) st.o[nt][s][r] = fmaf(sv, t4[r], st.o[nt][s][r]);
    }
  }
}

// Zero V^T fragment halves of tokens >= ntok (stale slots of a partial page).
__device__ __forceinline__ void mask_v_tokens(uint32_t (&a)[4], int ntok, int q4) {
  const int t0 = 2 * q4;
  const uint32_t m01 = (t0 < ntok ? 0xFFFFu : 0u) | (t0 + 1 < ntok ? 0xFFFF0000u : 0u);
  const uint32_t m23 = (t0 + 8 < ntok ? 0xFFFFu : 0u) | (t0 + 9 < ntok ? 0xFFFF0000u : 0u);
  a[0] &= m01; a[1] &= m01; a[2] &= m23; a[3] &= m23;
}

// One E2M1 page (per-token format: the last page may hold ntok < 16 tokens).
template <int D, int NT>
__device__ __forceinline__ void page_e2m1(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2], const uint8_t* kb,
                                          const uint8_t* vb, int ntok, float scale, const WarpSmem& sm, int lane) {
  constexpr int NS = D / 16;
  const int g = lane >> 2, q4 = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    uint32_t a[4];
    e2m1_frag(*reinterpret_cast<const uint32_t*>(kb + 4 * NS * lane + 4 * s), a);
    const uint8_t* sc = kb + e2m1_sc_off(D) + 16 * s;
    const uint32_t sgs = e4m3x2_to_f16x2(sc[g] | (sc[g + 8] << 8));   // {s_g, s_g+8}
    const uint32_t s0 = prmt(sgs, sgs, 0x1010u), s1 = prmt(sgs, sgs, 0x3232u);
    a[0] = hmul2u(a[0], s0); a[1] = hmul2u(a[1], s1); a[2] = hmul2u(a[2], s0); a[3] = hmul2u(a[3], s1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a[0], a[1], a[2], a[3], qf[nt][s][0], qf[nt][s][1]);
  }
  uint32_t phi[NT][2], plo[NT][2];
  softmax_and_frags<D, NT, false>(st, acc, ntok, scale, sm, lane, phi, plo);
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    uint32_t a[4];
    e2m1_frag(*reinterpret_cast<const uint32_t*>(vb + 4 * NS * lane + 4 * s), a);
    const uint8_t* sc = vb + e2m1_sc_off(D) + 16 * s + 2 * q4;
    const uint32_t s01 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sc));
    const uint32_t s23 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sc + 8));
    a[0] = hmul2u(a[0], s01); a[1] = hmul2u(a[1], s01); a[2] = hmul2u(a[2], s23); a[3] = hmul2u(a[3], s23);
    if (ntok < 16) mask_v_tokens(a, ntok, q4);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(st.o[nt][s], a[0], a[1], a[2], a[3], phi[nt][0], phi[nt][1]);
      mma16816(st.o[nt][s], a[0], a[1], a[2], a[3], plo[nt][0], plo[nt][1]);
    }
  }
}

// Total per-token counts of tokens < ntok (16 count bytes at p).
__device__ __forceinline__ int masked_count_total(const uint8_t* p, int ntok) {
  uint4 c = *reinterpret_cast<const uint4*>(p);
  uint32_t* w = reinterpret_cast<uint32_t*>(&c);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int keep = ntok - 4 * i;
    w[i] &= keep >= 4 ? 0xFFFFFFFFu : (keep <= 0 ? 0u : ((1u << (8 * keep)) - 1u));
  }
  return count_prefix(c).total;
}

// One INT4 page (per-token format; fp16 outliers in per-token slots).
template <int D, int NT>
__device__ __forceinline__ void page_int4(WarpState<D, NT>& st, const uint32_t (&qf)[NT][D / 16][2], const uint8_t* kb,
                                          const uint8_t* vb, int ntok, float scale, const WarpSmem& sm, int lane) {
  constexpr int NS = D / 16, CAP = int4_cap(D), NG = D / 32;
  const int g = lane >> 2, q4 = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int grp = s >> 1;
    const uint32_t z0 = *reinterpret_cast<const uint32_t*>(kb + int4_sz_off(D) + 4 * (g * NG + grp));
    const uint32_t z1 = *reinterpret_cast<const uint32_t*>(kb + int4_sz_off(D) + 4 * ((g + 8) * NG + grp));
    uint32_t ahi[4], alo[4];
    int4_k_frag(*reinterpret_cast<const uint32_t*>(kb + 4 * NS * lane + 4 * s), fp16_bits_to_float(z0),
                fp16_bits_to_float(z0 >> 16), fp16_bits_to_float(z1), fp16_bits_to_float(z1 >> 16), ahi, alo);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(acc[nt], ahi[0], ahi[1], ahi[2], ahi[3], qf[nt][s][0], qf[nt][s][1]);
      mma16816(acc[nt], alo[0], alo[1], alo[2], alo[3], qf[nt][s][0], qf[nt][s][1]);
    }
  }
  // K outliers: scores[t][h] += q[h][c] * (x - m), m = value of code 0 in the group
  if (masked_count_total(kb + int4_cnt_off(D), ntok) > 0) {
    for (int e = lane; e < 16 * CAP; e += 32) {
      const int t = e / CAP, i = e - t * CAP;
      if (t < ntok && i < kb[int4_cnt_off(D) + t]) {
        const int ch = kb[int4_ch_off(D) + e] & (D - 1);
        const float x = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(kb + int4_val_off(D) + 2 * e));
        const float mz = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(kb + int4_sz_off(D) + 4 * (t * NG + ch / 32) + 2));
        for (int h = 0; h < sm.G; ++h) atomicAdd(&sm.ds[t * sm.GS + h], sm.qsm[ch * sm.GS + h] * (x - mz));
      }
    }
    apply_ds<NT>(acc, sm.ds, sm.G, sm.GS, g, q4);
  }
  uint32_t phi[NT][2], plo[NT][2];
  softmax_and_frags<D, NT, true>(st, acc, ntok, scale, sm, lane, phi, plo);
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int grp = s >> 1;
    float S[4], M[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 2 * q4 + (i & 1) + 8 * (i >> 1);
      const uint32_t z = *reinterpret_cast<const uint32_t*>(vb + int4_sz_off(D) + 4 * (t * NG + grp));
      S[i] = fp16_bits_to_float(z);
      M[i] = fp16_bits_to_float(z >> 16);
    }
    uint32_t ahi[4], alo[4];
    int4_v_frag(*reinterpret_cast<const uint32_t*>(vb + 4 * NS * lane + 4 * s), S, M, ahi, alo);
    if (ntok < 16) {
      mask_v_tokens(ahi, ntok, q4);
      mask_v_tokens(alo, ntok, q4);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma16816(st.o[nt][s], ahi[0], ahi[1], ahi[2], ahi[3], phi[nt][0], phi[nt][1]);
      mma16816(st.o[nt][s], ahi[0], ahi[1], ahi[2], ahi[3], plo[nt][0], plo[nt][1]);
      mma16816(st.o[nt][s], alo[0], alo[1], alo[2], alo[3], phi[nt][0], phi[nt][1]);
    }
  }
  if (masked_count_total(vb + int4_cnt_off(D), ntok) > 0) {
    store_p<NT>(acc, sm.psm, sm.G, sm.GS, g, q4);
    __syncwarp();
    for (int e = lane; e < 16 * CAP; e += 32) {
      const int t = e / CAP, i = e - t * CAP;
      if (t < ntok && i < vb[int4_cnt_off(D) + t]) {
        const int ch = vb[int4_ch_off(D) + e] & (D - 1);
        const float x = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(vb + int4_val_off(D) + 2 * e));
        const float mz = fp16_bits_to_float(*reinterpret_cast<const uint16_t*>(vb + int4_sz_off(D) + 4 * (t * NG + ch / 32) + 2));
        for (int h = 0; h < sm.G; ++h) atomicAdd(&sm.corr[ch * sm.GS + h], sm.psm[t * sm.GS + h] * (x - mz));
      }
    }
  }
}

// The partial last page of a page format: ntail fp32 tokens in staging, on CUDA cores.
template <int D, int NT, bool kCorr>
__device__ __forceinline__ void page_tail(WarpState<D, NT>& st, const float* ks, const float* vs, int ntail,
                                          float scale, const WarpSmem& sm, int lane) {
  const int g = lane >> 2, q4 = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = g + 8 * (r >> 1), h = nt * 8 + 2 * q4 + (r & 1);
      float d = 0.f;
      if (t < ntail && h < sm.G)
        for (int c = 0; c < D; ++c) d = fmaf(sm.qsm[c * sm.GS + h], ks[t * D + c], d);
      acc[nt][r] = d;
    }
  uint32_t phi[NT][2], plo[NT][2];
  softmax_and_frags<D, NT, kCorr>(st, acc, ntail, scale, sm, lane, phi, plo);
  store_p<NT>(acc, sm.psm, sm.G, sm.GS, g, q4);
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

// ----------------------------------------------------------------------------- split kernel
constexpr int32_t kBadEntry = 0x7FFFFFFF;

template <int FMT, int D, int NT, int W, int NSTAGE>
__global__ void __launch_bounds__(W * 32) decode_split_kernel(const DecodeArgs a) {
  using F = Fmt<FMT>;
  constexpr int NS = D / 16;
  constexpr int HS = half_slot_bytes<FMT, D>();
  constexpr int kMainStride = block_stride(F::kMain, D);
  constexpr int kTierStride = block_stride(kBlkFp8, D);
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.G, GS = (G + 3) & ~3;

  float* qsm = reinterpret_cast<float*>(smem);
  uint8_t* wb = smem + align16(D * GS * 4) + w * align16(warp_smem_bytes<FMT, D, NSTAGE>(GS));
  uint8_t* stages = wb;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(wb + NSTAGE * 2 * HS);
  int32_t* meta = reinterpret_cast<int32_t*>(wb + NSTAGE * 2 * HS + 8 * NSTAGE);
  WarpSmem sm;
  sm.qsm = qsm;
  sm.ds = reinterpret_cast<float*>(wb + NSTAGE * 2 * HS + 8 * NSTAGE + align16(4 * NSTAGE));
  sm.psm = sm.ds + 16 * GS;
  sm.corr = sm.psm + 16 * GS;
  sm.G = G;
  sm.GS = GS;

  // query of the CTA's G heads, fp32 in shared memory ([D][GS]) and fp16 B fragments in registers
  const __nv_bfloat16* qg = a.q + ((size_t)b * a.Hq + (size_t)kvh * G) * D;
  for (int i = threadIdx.x; i < D * GS; i += W * 32) {
    const int c = i / GS, h = i - c * GS;
    qsm[i] = h < G ? __bfloat162float(qg[h * D + c]) : 0.f;
  }
  for (int i = lane; i < 16 * GS; i += 32) sm.ds[i] = 0.f;
  if (F::kOutliers)
    for (int i = lane; i < D * GS; i += 32) sm.corr[i] = 0.f;
  if (lane == 0) {
    for (int j = 0; j < NSTAGE; ++j) mbar_init(&mbar[j], 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint32_t qf[NT][NS][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int h = nt * 8 + g, c = 16 * s + 2 * q4;
      const bool on = h < G;
      qf[nt][s][0] = h2_as_u32(__floats2half2_rn(on ? qsm[c * GS + h] : 0.f, on ? qsm[(c + 1) * GS + h] : 0.f));
      qf[nt][s][1] = h2_as_u32(__floats2half2_rn(on ? qsm[(c + 8) * GS + h] : 0.f, on ? qsm[(c + 9) * GS + h] : 0.f));
    }

  int L = a.seq_lens[b];
  if (L > a.max_seq_len) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(a.status, KVQ_STATUS_SEQ_TOO_LONG);
    L = a.max_seq_len;
  }
  L = max(L, 0);
  const int n_all = (L + kPage - 1) / kPage;
  const int nq = F::kPaged ? L / kPage : n_all;  // pages stored as blocks
  const int p0 = split * a.pps;
  const int p1 = min(p0 + a.pps, n_all);
  const int pq1 = min(p1, nq);
  const int n_local = pq1 > p0 + w ? (pq1 - p0 - w + W - 1) / W : 0;

  WarpState<D, NT> st;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int s = 0; s < NS; ++s) st.o[nt][s][0] = st.o[nt][s][1] = st.o[nt][s][2] = st.o[nt][s][3] = 0.f;
    st.m[nt][0] = st.m[nt][1] = -INFINITY;
    st.l[nt][0] = st.l[nt][1] = 0.f;
  }

  // page-table window: lane j holds the entry of this warp's page win_base + j
  const int32_t* pt = a.page_table + (size_t)b * a.ppsm;
  int win_base = 0;
  int win = lane < n_local ? pt[p0 + w + lane * W] : 0;

  auto block_src = [&](int32_t e, int role) -> const uint8_t* {
    const uint32_t u = (uint32_t)e, phys = u & 0x7FFFFFFFu;
    if (FMT == KVQ_FMT_TIERED && (u >> 31))
      return a.tier_pool + (((size_t)phys * a.Hkv + kvh) * 2 + role) * kTierStride;
    return a.pool + (((size_t)phys * a.Hkv + kvh) * 2 + role) * kMainStride;
  };

  auto issue = [&](int i) {
    if (i >= n_local) return;
    if (i - win_base >= 32) {
      win_base += 32;
      const int j = win_base + lane;
      win = j < n_local ? pt[p0 + w + j * W] : 0;
    }
    const int32_t e = __shfl_sync(0xffffffffu, win, i - win_base);
    if (lane == 0) {
      const int slot = i % NSTAGE;
      const uint32_t u = (uint32_t)e, phys = u & 0x7FFFFFFFu;
      const bool tier = (u >> 31) != 0;
      const bool ok = tier ? (FMT == KVQ_FMT_TIERED && phys < (uint32_t)a.num_tier_pages) : phys < (uint32_t)a.num_pages;
      fence_proxy_async();
      if (!ok) {
        meta[slot] = kBadEntry;
        atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        mbar_arrive(&mbar[slot]);
      } else {
        meta[slot] = e;
        uint32_t bytes;
        if (tier) bytes = fetch_bytes<D>(kBlkFp8);
        else if (F::kMain == kBlkCb2) bytes = 12 * D + 16 + 2 * a.ent_prefetch;
        else bytes = fetch_bytes<D>(F::kMain);
        uint8_t* dst = stages + slot * 2 * HS;
        mbar_arrive_expect_tx(&mbar[slot], 2 * bytes);
        bulk_g2s(dst, block_src(e, 0), bytes, &mbar[slot]);
        bulk_g2s(dst + HS, block_src(e, 1), bytes, &mbar[slot]);
      }
    }
  };

#pragma unroll 1
  for (int i = 0; i < NSTAGE; ++i) issue(i);

  bool timed_out = false;
  int i = 0;
#pragma unroll 1
  for (; i < n_local; ++i) {
    const int slot = i % NSTAGE;
    const bool ok = mbar_wait_bounded(&mbar[slot], (i / NSTAGE) & 1, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, ok)) {
      timed_out = true;
      if (lane == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      break;
    }
    const int32_t e = meta[slot];
    if (e != kBadEntry) {
      const int page = p0 + w + i * W;
      const uint8_t* kb = stages + slot * 2 * HS;
      const uint8_t* vb = kb + HS;
      if (FMT == KVQ_FMT_TIERED && e < 0) {
        page_fp8<D, NT, true>(st, qf, kb, vb, a.scale_log2, sm, lane);
      } else if (F::kMain == kBlkCb2) {
        page_cb2<D, NT>(st, qf, kb, vb, block_src(e, 0), block_src(e, 1), a.ent_prefetch, a.scale_log2, sm, lane);
      } else if (F::kMain == kBlkE2m1) {
        page_e2m1<D, NT>(st, qf, kb, vb, min(kPage, L - kPage * page), a.scale_log2, sm, lane);
      } else {
        page_int4<D, NT>(st, qf, kb, vb, min(kPage, L - kPage * page), a.scale_log2, sm, lane);
      }
    }
    __syncwarp();
    issue(i + NSTAGE);
  }
  if (timed_out) {
    // let copies still in flight land (bounded) before the CTA can exit
    for (int j = i; j < min(i + NSTAGE, n_local); ++j) mbar_wait_bounded(&mbar[j % NSTAGE], (j / NSTAGE) & 1, kWaitLimitNs);
  }

  // partial last page of a page format, from fp32 staging
  if (F::kPaged && (L % kPage) != 0 && !timed_out) {
    const int tp = nq;
    if (tp >= p0 && tp < p1 && (tp - p0) % W == w) {
      const float* ks = a.staging + (((size_t)b * a.Hkv + kvh) * 2) * kPage * D;
      page_tail<D, NT, F::kOutliers>(st, ks, ks + kPage * D, L % kPage, a.scale_log2, sm, lane);
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
  float* mo = reinterpret_cast<float*>(smem + align16(D * GS * 4));  // [W][GS][D]
  float* mm = mo + W * GS * D;                                       // [W][GS]
  float* ml = mm + W * GS;                                           // [W][GS]
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
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
    const int h = idx / D, c = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) M = fmaxf(M, mm[ww * GS + h]);
    float ov = 0.f, lv = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < W; ++ww) {
        const float mw = mm[ww * GS + h];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        ov = fmaf(f, mo[(ww * GS + h) * D + c], ov);
        lv = fmaf(f, ml[ww * GS + h], lv);
      }
    }
    const size_t row = ((size_t)b * a.Hq + (size_t)kvh * G + h) * a.S + split;
    a.part_o[row * D + c] = ov;
    if (c == 0) a.part_ml[row] = make_float2(M, lv);
  }
}


// ----------------------------------------------------------------------------- launch configuration
constexpr int kWarps = kWarpsPerCta;
constexpr int kStages = 3;

struct KernelInfo {
  void* fn;
  size_t smem;
  int threads;
};

template <int FMT, int D, int NT>
static KernelInfo kernel_info(int G) {
  const int GS = (G + 3) & ~3;
  const size_t plan = cta_smem_bytes<FMT, D, kWarps, kStages>(GS);
  const size_t merge = align16(D * GS * 4) + (size_t)kWarps * GS * D * 4 + 2 * (size_t)kWarps * GS * 4;
  return {reinterpret_cast<void*>(decode_split_kernel<FMT, D, NT, kWarps, kStages>), plan > merge ? plan : merge,
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
KernelInfo decode_kernel_cb2(int D, int G);
KernelInfo decode_kernel_tiered(int D, int G);

}  // namespace kvq
