// kvq_decode.cu -- the split-combine kernel and the host-side launch of the
// decode path (the split kernels live in kvq_decode.cuh, one translation unit
// per cache format).
#include "kvq_decode.cuh"

namespace kvq {

// ----------------------------------------------------------------------------- combine kernel
// out[b][h] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, M = max_s m_s (0 if no tokens).
template <typename OutT>
__global__ void __launch_bounds__(128) decode_combine_kernel(const float* __restrict__ part_o,
                                                             const float2* __restrict__ part_ml, int S, int D,
                                                             int Hq, OutT* __restrict__ out) {
  const size_t row = (size_t)blockIdx.y * Hq + blockIdx.x;
  const float2* ml = part_ml + row * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, ml[s].x);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float2 v = ml[s];
        if (v.x == -INFINITY) continue;
        const float f = exp2f(v.x - M);
        L = fmaf(f, v.y, L);
        acc = fmaf(f, part_o[(row * S + s) * D + c], acc);
      }
    }
    const float r = L > 0.f ? acc / L : 0.f;
    if constexpr (sizeof(OutT) == 2) out[row * D + c] = __float2bfloat16_rn(r);
    else out[row * D + c] = r;
  }
}

// ----------------------------------------------------------------------------- host side
static KernelInfo pick_kernel(int fmt, int D, int G) {
  switch (fmt) {
    case KVQ_FMT_INT4_G32: return decode_kernel_int4(D, G);
    case KVQ_FMT_FP4_E2M1_S16: return decode_kernel_e2m1(D, G);
    case KVQ_FMT_CB2_OUTLIER: return decode_kernel_cb2(D, G);
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

cudaError_t decode_combine_launch(const float* part_o, const float2* part_ml, int B, int Hq, int S, int D, void* out,
                                  int out_dtype, cudaStream_t st) {
  if (out_dtype == KVQ_F32)
    decode_combine_kernel<float><<<dim3(Hq, B), 128, 0, st>>>(part_o, part_ml, S, D, Hq, static_cast<float*>(out));
  else
    decode_combine_kernel<__nv_bfloat16><<<dim3(Hq, B), 128, 0, st>>>(part_o, part_ml, S, D, Hq,
                                                                        static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace kvq
