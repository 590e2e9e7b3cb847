// kvq_decode_cb2.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_cb2(int D, int G, bool cuda_cores) {
  constexpr int F = KVQ_FMT_CB2_OUTLIER;
  if (cuda_cores && G <= 4) return D == 64 ? kernel_info<F, 64, 1, true>(G) : kernel_info<F, 128, 1, true>(G);
  return kernel_info_fmt<F>(D, G);
}
}  // namespace kvq
