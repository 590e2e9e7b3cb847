// kvq_common.cuh -- block layout constants and inline-PTX helpers shared by the
// library's kernels (sm_103a).  The layout is the one include/kvq.h documents.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kPage = KVQ_PAGE_TOKENS;

// Block formats (the pool format of a cache; FP8 is the tier-1 page format).
enum BlkFmt : int { kBlkInt4 = 0, kBlkE2m1 = 1, kBlkCb2 = 2, kBlkFp8 = 3, kBlkCb2s = 4, kBlkA3 = 5, kBlkCb2g = 6 };
constexpr int kGroupPages = 4;  // CB2_GROUP4: pages sharing one codebook
constexpr int kMaxStatic = 8;   // CB2_STATIC: static fp16 channels per (kv head, K|V)

// Largest number of values of an n-vector that can lie more than 3 standard
// deviations (unbiased) from its mean: k * 9 * s^2 < (n - 1) * s^2.
__host__ __device__ constexpr int kmax_outliers(int n) { return (n - 1 + 8) / 9 - 1; }
__host__ __device__ constexpr int round_up128(int x) { return (x + 127) / 128 * 128; }
__host__ __device__ constexpr int int4_cap(int D) { return 3 * (D / 32); }

// Section offsets (bytes) within a block, per format.
__host__ __device__ constexpr int int4_sz_off(int D) { return 8 * D; }
__host__ __device__ constexpr int int4_cnt_off(int D) { return 10 * D; }
__host__ __device__ constexpr int int4_ch_off(int D) { return 10 * D + 16; }
__host__ __device__ constexpr int int4_val_off(int D) { return 10 * D + 16 + 16 * int4_cap(D); }
__host__ __device__ constexpr int e2m1_sc_off(int D) { return 8 * D; }
__host__ __device__ constexpr int cb2_cb_off(int D) { return 4 * D; }
__host__ __device__ constexpr int cb2_out_off(int D) { return 12 * D; }   // outlier side-list
__host__ __device__ constexpr int fp8_sc_off(int D) { return 16 * D; }
__host__ __device__ constexpr int cb2s_hdr_off(int D) { return 12 * D; }      // u8 n_s, u8 channel[n_s]
__host__ __device__ constexpr int cb2s_val_off(int D) { return 12 * D + 16; } // fp16 [n_s][16]
__host__ __device__ constexpr int a3_hi_off(int D) { return 4 * D; }          // high code bits
__host__ __device__ constexpr int a3_s_off(int D) { return 6 * D; }           // fp16 S by rho(c)
__host__ __device__ constexpr int a3_m_off(int D) { return 8 * D; }           // fp16 m by rho(c)
__host__ __device__ constexpr int a3_out_off(int D) { return 10 * D; }        // outlier side-list
__host__ __device__ constexpr int cb2g_code_off(int D) { return 8 * D; }      // codes (codebook at 0)
// ASYM3 position of channel c's S / m (K: 4 channels of a lane-step adjacent; V: 2).
__host__ __device__ inline int a3_rho(int role, int c) {
  return role == 0 ? 16 * (c / 16) + 4 * ((c % 8) / 2) + 2 * ((c % 16) / 8) + c % 2
                   : 16 * (c / 16) + 2 * (c % 8) + (c % 16) / 8;
}

__host__ __device__ constexpr int block_stride(int fmt, int D) {
  return fmt == kBlkInt4 ? round_up128(10 * D + 16 + 48 * int4_cap(D))
       : fmt == kBlkE2m1 ? round_up128(9 * D)
       : fmt == kBlkCb2  ? round_up128(12 * D + 4 + 20 * D)
       : fmt == kBlkCb2s ? round_up128(12 * D + 16 + 32 * kMaxStatic)
       : fmt == kBlkA3   ? round_up128(10 * D + 4 + 20 * D)
       : fmt == kBlkCb2g ? round_up128(12 * D + 4 + 20 * D)
                         : round_up128(16 * D + 16);
}

// Fragment position of element (t, c) (see include/kvq.h).
struct FragPos { int lane, step, slot; };
__host__ __device__ inline FragPos frag_pos(int role, int t, int c) {
  int j = c & 15;
  FragPos p;
  p.step = c >> 4;
  if (role == 0) {
    p.lane = 4 * (t & 7) + ((j & 7) >> 1);
    p.slot = 2 * ((t >> 3) + 2 * (j >> 3)) + (j & 1);
  } else {
    p.lane = 4 * (j & 7) + ((t & 7) >> 1);
    p.slot = 2 * ((j >> 3) + 2 * (t >> 3)) + (t & 1);
  }
  return p;
}
// CB2 codebook slot of channel c.
__host__ __device__ inline int cb2_slot(int role, int c) {
  return role == 0 ? c : 16 * (c >> 4) + 2 * (c & 7) + ((c >> 3) & 1);
}

// ----------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory loads at 32-bit shared-window addresses (immediate offsets fold
// into the instruction).  volatile keeps them after the mbarrier waits that
// publish the data.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float ldsf(uint32_t a) { return __uint_as_float(lds32(a)); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// m16n8k8 fp16 x fp16 -> fp32, D += A * B.
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(b0));
}

// m16n8k16 fp16 x fp16 -> fp32, D += A * B.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 bytes (low byte -> low half) to an f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t d;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(d) : "r"(two_bytes));
  return d;
}

// One byte holding two e2m1 nibbles (low nibble -> low half) to an f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  asm("{ .reg .b8 t; .reg .b16 w; cvt.u16.u32 w, %1; cvt.u8.u16 t, w; cvt.rn.f16x2.e2m1x2 %0, t; }"
      : "=r"(d)
      : "r"(byte));
  return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// ----------------------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Ends the life of an mbarrier; its memory may then serve another purpose.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Bulk global -> shared copy completing on `bar`.  dst, src 16-B aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, "
      "p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// try_wait that may suspend the thread for up to `hint_ns` (woken early when
// the phase completes), so waiting warps do not spin on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, "
      "p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar`, giving up after `limit_ns`.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

constexpr uint64_t kWaitLimitNs = 100ull * 1000ull * 1000ull;  // 100 ms

}  // namespace kvq
