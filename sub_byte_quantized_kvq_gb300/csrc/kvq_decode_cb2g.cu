// kvq_decode_cb2g.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_cb2g(int D, int G) { return kernel_info_fmt<KVQ_FMT_CB2_GROUP4>(D, G); }
}  // namespace kvq
