// kvq_decode_e2m1.cu -- instantiates the split decode kernels of one cache format.
#include "kvq_decode.cuh"

namespace kvq {
KernelInfo decode_kernel_e2m1(int D, int G) { return kernel_info_fmt<KVQ_FMT_FP4_E2M1_S16>(D, G); }
}  // namespace kvq
