// kvq_decode_cb2s.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_cb2s(int D, int G) { return kernel_info_fmt<KVQ_FMT_CB2_STATIC>(D, G); }
}  // namespace kvq
