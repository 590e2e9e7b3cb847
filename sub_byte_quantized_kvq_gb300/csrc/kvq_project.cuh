// kvq_project.cuh -- arguments of the fused K/V projection + quantize-append
// launch (kvq_quantize.cu), shared with the ABI entry point (kvq_api.cu).
#pragma once
#include <cuda.h>

#include "kvq_internal.cuh"

namespace kvq {

// K/V projection fused with quantize-on-append: the new tokens' K and V are
// x W_k^T and x W_v^T (bf16 operands, fp32 accumulation) instead of inputs.
struct ProjArgs {
  CUtensorMap tm_x;            // x as [B * t_new][hidden], boxes of one unit of rows
  CUtensorMap tm_w[2];         // W_k, W_v as [Hkv * D][hidden], boxes of one head's rows
  AppendArgs a;                // kv[] unused
  const __nv_bfloat16* x;      // [B][t_new][hidden]
  const __nv_bfloat16* w[2];   // W_k, W_v: [Hkv * D][hidden]
  int hidden;                  // a multiple of 32
  float* kv_out;               // NULL or [2][B][t_new][Hkv][D]: the projected values
};
// Encodes p's tensor maps, then launches.
cudaError_t project_append_launch(ProjArgs& p, int D, cudaStream_t st);

}  // namespace kvq
