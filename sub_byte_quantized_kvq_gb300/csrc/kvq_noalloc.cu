// kvq_noalloc.cu -- decode attention for callers that are not allowed to
// allocate device memory.
//
// kvq_decode_attention needs a caller-provided workspace for the fp32 split
// partials.  Some callers cannot obtain one at the moment they run decode:
// a serving loop that reserves all of its GPU memory at start-up and treats
// any later allocation as an error (cudaMalloc can also synchronise the device
// and stall every stream), code that runs inside an allocator or memory-pool
// callback where allocating again would recurse or deadlock, or a plugin whose
// host framework hands it only its input and output buffers.  For them the
// library carries one fixed scratch array of its own and reuses the ordinary
// split and combine kernels on it.
#include <mutex>

#include "kvq_internal.cuh"

// The scratch: one copy on every GPU that loads this library, alive until the
// process exits.  Host code may not use its name as an address (on the host it
// is only a stand-in for the symbol); the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch on the current device, looked up once per
// device ordinal (with that device current) and cached for the life of the
// process; nullptr if the lookup fails (the runtime's error in *err).  The
// cache is keyed by ordinal, so the entry point must not be used on a device
// after cudaDeviceReset on it.
void* scratch_on_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    if (p == nullptr) {
      *err = cudaErrorInvalidSymbol;
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}
}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                                   int32_t num_q_heads, float softmax_scale, int32_t max_seq_len,
                                                   int32_t num_splits, void* out, kvq_dtype out_dtype,
                                                   void* stream) {
  size_t need = 0;
  const kvq_status st = kvq_decode_workspace_bytes(cfg, num_q_heads, max_seq_len, num_splits, &need);
  if (st != KVQ_OK) return st;
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;  // before anything is enqueued
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_on_current_device(&err);
  if (!scratch) return kvq::cuda_status(err);
  // The scratch is shared by every cache in the process: the arrival counters
  // sit at its start, B * Hkv of them, so a call on a cache with more
  // (sequence, kv head) pairs than the last one's would find that call's
  // partials there.  This call clears its own counters on the stream before
  // the launch (a memset, which allocates nothing).
  return kvq::decode_attention_zeroing_counters(cfg, cache, q, num_q_heads, softmax_scale, max_seq_len, num_splits, out,
                                                out_dtype, scratch, (size_t)KVQ_NOALLOC_SCRATCH_BYTES,
                                                static_cast<cudaStream_t>(stream));
}
