// kvq_decode.cu -- the split-combine kernel and the host-side launch of the
// decode path (the split kernels live in kvq_decode.cuh, one translation unit
// per cache format).
#include <mutex>

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
static KernelInfo pick_kernel(int fmt, int D, int G, int math) {
  switch (fmt) {
    case KVQ_FMT_INT4_G32: return decode_kernel_int4(D, G);
    case KVQ_FMT_FP4_E2M1_S16: return decode_kernel_e2m1(D, G);
    case KVQ_FMT_CB2_OUTLIER: return decode_kernel_cb2(D, G, math == KVQ_DECODE_CUDA_CORES);
    case KVQ_FMT_CB2_STATIC: return decode_kernel_cb2s(D, G);
    case KVQ_FMT_ASYM3_OUTLIER: return decode_kernel_a3(D, G);
    case KVQ_FMT_CB2_GROUP4: return decode_kernel_cb2g(D, G);
    default: return decode_kernel_tiered(D, G);
  }
}

// Per-device launch facts of the split kernels, worked out once: a kernel's
// dynamic shared memory depends on the GQA group size as well as on its
// template arguments, so the attribute on each (kernel, device) is raised to
// the largest size any call has needed (on the first call of each size, not
// on every call), and the resident CTAs per SM that the split heuristic asks
// for are looked up once per (kernel, device, size).
namespace {
struct Prepared {
  void* fn;
  int dev;
  size_t smem;
  int ctas_per_sm;   // resident CTAs per SM at this size
};
struct AttrSet {
  void* fn;
  int dev;
  size_t smem;       // the attribute's current value
};
constexpr int kMaxPrepared = 512;
std::mutex g_prep_mutex;
Prepared g_prep[kMaxPrepared];
AttrSet g_attr[kMaxPrepared];
int g_nprep = 0, g_nattr = 0;

// The prepared record of kernel k on the current device (nullptr on a CUDA error).
const Prepared* prepare(const KernelInfo& k) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(g_prep_mutex);
  for (int i = 0; i < g_nprep; ++i)
    if (g_prep[i].fn == k.fn && g_prep[i].dev == dev && g_prep[i].smem == k.smem) return &g_prep[i];
  if (g_nprep == kMaxPrepared) return nullptr;
  AttrSet* at = nullptr;
  for (int i = 0; i < g_nattr; ++i)
    if (g_attr[i].fn == k.fn && g_attr[i].dev == dev) at = &g_attr[i];
  if (!at) {
    if (g_nattr == kMaxPrepared) return nullptr;
    at = &g_attr[g_nattr++];
    *at = AttrSet{k.fn, dev, 0};
  }
  if (at->smem < k.smem) {
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess)
      return nullptr;
    at->smem = k.smem;
  }
  Prepared p{k.fn, dev, k.smem, 0};
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&p.ctas_per_sm, k.fn, k.threads, k.smem) != cudaSuccess)
    return nullptr;
  g_prep[g_nprep] = p;
  return &g_prep[g_nprep++];
}
}  // namespace

// CTAs of the split kernel that fit on one SM (0 if the kernel cannot run).
int decode_ctas_per_sm(int fmt, int D, int G, int math) {
  const Prepared* p = prepare(pick_kernel(fmt, D, G, math));
  return p ? p->ctas_per_sm : 0;
}

cudaError_t decode_split_launch(const DecodeArgs& a, int fmt, int D, cudaStream_t st) {
  const KernelInfo k = pick_kernel(fmt, D, a.G, a.math);
  if (!prepare(k)) {
    const cudaError_t e = cudaGetLastError();
    return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
  }
  void* args[] = {const_cast<DecodeArgs*>(&a)};
  cudaError_t err = cudaLaunchKernel(k.fn, dim3(a.S, a.Hkv, a.B), dim3(k.threads), args, k.smem, st);
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
