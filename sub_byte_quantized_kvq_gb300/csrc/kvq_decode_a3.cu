// kvq_decode_a3.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_a3(int D, int G) { return kernel_info_fmt<KVQ_FMT_ASYM3_OUTLIER>(D, G); }
}  // namespace kvq
