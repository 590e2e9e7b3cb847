// kvq_decode.cu -- the split-combine kernel and the host-side launch of the
// decode path (the split kernels live in kvq_decode.cuh, one translation unit
// per cache format).
#include "kvq_decode.cuh"

namespace kvq {

// ----------------------------------------------------------------------------- combine kernel
// One CTA per (kv head, sequence): the split merge of its G query heads.
__global__ void __launch_bounds__(128) decode_combine_kernel(const float* __restrict__ part_o,
                                                             const float2* __restrict__ part_ml, int S, int D,
                                                             int Hq, int G, void* out, int out_dtype) {
  extern __shared__ float wts[];
  merge_group(part_o, part_ml, (size_t)blockIdx.y * Hq + (size_t)blockIdx.x * G, G, S, D, out, out_dtype, wts);
}

// ----------------------------------------------------------------------------- host side
static KernelInfo pick_kernel(int fmt, int D, int G) {
  switch (fmt) {
    case KVQ_FMT_INT4_G32: return decode_kernel_int4(D, G);
    case KVQ_FMT_FP4_E2M1_S16: return decode_kernel_e2m1(D, G);
    case KVQ_FMT_CB2_OUTLIER: return decode_kernel_cb2(D, G);
    case KVQ_FMT_CB2_STATIC: return decode_kernel_cb2s(D, G);
    case KVQ_FMT_ASYM3_OUTLIER: return decode_kernel_a3(D, G);
    case KVQ_FMT_CB2_GROUP4: return decode_kernel_cb2g(D, G);
    default: return decode_kernel_tiered(D, G);
  }
}

// CTAs of the split kernel that fit on one SM (0 if the kernel cannot run).
int decode_ctas_per_sm(int fmt, int D, int G) {
  KernelInfo k = pick_kernel(fmt, D, G);
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k.fn, k.threads, k.smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t decode_split_launch(const DecodeArgs& a, int fmt, int D, cudaStream_t st) {
  KernelInfo k = pick_kernel(fmt, D, a.G);
  cudaError_t err = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem);
  if (err != cudaSuccess) return err;
  void* args[] = {const_cast<DecodeArgs*>(&a)};
  err = cudaLaunchKernel(k.fn, dim3(a.S, a.Hkv, a.B), dim3(k.threads), args, k.smem, st);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t decode_combine_launch(const float* part_o, const float2* part_ml, int B, int Hkv, int Hq, int S, int D, void* out,
                                  int out_dtype, cudaStream_t st) {
  const int G = Hq / Hkv;
  decode_combine_kernel<<<dim3(Hkv, B), 128, (size_t)(G * S + G) * sizeof(float), st>>>(part_o, part_ml, S, D, Hq, G,
                                                                                       out, out_dtype);
  return cudaGetLastError();
}

}  // namespace kvq
