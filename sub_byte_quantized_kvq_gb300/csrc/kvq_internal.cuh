// kvq_internal.cuh -- argument blocks and launch entry points shared between the
// library's translation units (not part of the public ABI).
#pragma once
#include "kvq_common.cuh"

namespace kvq {

// Largest split count: the split merge keeps G x S weights in the split
// kernel's shared merge area (at least 4 D + 8 floats per query head).
constexpr int kMaxSplits = 256;

struct DecodeArgs {
  const uint8_t* pool;
  const uint8_t* tier_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const float* staging;
  const __nv_bfloat16* q;
  float* part_o;    // [B][Hq][S][D]
  float2* part_ml;  // [B][Hq][S] (m in log2 units, l)
  uint32_t* status;
  int B, Hkv, Hq, G, ppsm, num_pages, num_tier_pages;
  int S, pps;       // splits, pages per split
  int max_seq_len;
  float scale_log2; // softmax_scale * log2(e)
  // Fused combine (kvq_decode_attention): the last split CTA of a (sequence,
  // kv head) to finish merges the partials into `out`.  out == nullptr: the
  // split kernel only writes partials (kvq_decode_split).
  void* out;        // [B][Hq][D] in out_dtype
  int out_dtype;    // KVQ_BF16 or KVQ_F32
  uint32_t* arrivals;  // [B][Hkv] arrival counters, zero between calls
  const uint8_t* static_mask;  // CB2_STATIC: [Hkv][2][n_static] channels
  int n_static;
  int math;         // KVQ_DECODE_TENSOR_CORES or KVQ_DECODE_CUDA_CORES (resolved, never AUTO)
};

struct AppendArgs {
  uint8_t* pool;
  uint8_t* tier_pool;
  const int32_t* page_table;
  int32_t* seq_lens;
  float* staging;
  uint32_t* status;
  const void* kv[2];
  int in_dtype;
  int t_new;
  const int32_t* t_per_seq;
  int B, Hkv, ppsm, num_pages, num_tier_pages, fmt, iters;
  double sigma;
  const uint8_t* static_mask;  // CB2_STATIC: [Hkv][2][n_static] channels
  int n_static;
};

// The split decode kernel, and the combine kernel (out_dtype KVQ_BF16 or KVQ_F32), on `st`.
cudaError_t decode_split_launch(const DecodeArgs& a, int fmt, int D, cudaStream_t st);
cudaError_t decode_combine_launch(const float* part_o, const float2* part_ml, int B, int Hkv, int Hq, int S, int D, void* out,
                                  int out_dtype, cudaStream_t st);
// Resident CTAs per SM of the split kernel for (format, head_dim, G); 0 on error.
int decode_ctas_per_sm(int fmt, int D, int G, int math);
// Warps per CTA of the split decode kernel.
constexpr int kWarpsPerCta = 4;
// Quantize-on-append launches (see kvq_quantize.cu).
cudaError_t append_launch(const AppendArgs& a, int D, cudaStream_t st);

cudaError_t select_static_launch(const void* k, const void* v, int in_dtype, int t, int Hkv, int D, int n_s,
                                 uint8_t* mask, cudaStream_t st);
// KVQ_OK for cudaSuccess; otherwise records e for kvq_last_cuda_error and
// returns KVQ_ERR_CUDA.
kvq_status cuda_status(cudaError_t e);
// kvq_decode_attention after clearing the call's arrival counters with a
// memset on `st` (validation first: an argument error enqueues nothing).
kvq_status decode_attention_zeroing_counters(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                             int32_t num_q_heads, float softmax_scale, int32_t max_seq_len,
                                             int32_t num_splits, void* out, kvq_dtype out_dtype, void* workspace,
                                             size_t workspace_bytes, cudaStream_t st);
// Dequantize tokens [t0, t1) of (seq, head, role) to fp32.
cudaError_t dequantize_launch(const kvq_config& cfg, const kvq_cache& cache, int seq, int head, int role, int t0,
                              int t1, float* out, cudaStream_t st);

}  // namespace kvq
