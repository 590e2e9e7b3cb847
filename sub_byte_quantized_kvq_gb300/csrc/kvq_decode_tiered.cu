// kvq_decode_tiered.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_tiered(int D, int G) { return kernel_info_fmt<KVQ_FMT_TIERED>(D, G); }
}  // namespace kvq
