// kvq_decode_int4.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_int4(int D, int G) { return kernel_info_fmt<KVQ_FMT_INT4_G32>(D, G); }
}  // namespace kvq
