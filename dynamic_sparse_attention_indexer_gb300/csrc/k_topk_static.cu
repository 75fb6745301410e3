// Decode top-k for callers that cannot allocate device memory.
//
// Same kernels and results as dsa_topk_select in decode mode; the only
// difference is where the scratch comes from.  Here it is a file-scope static
// device array, so the caller passes inputs and outputs only.  Callers in this
// position are, for example, a plugin running inside a serving process whose
// device memory is entirely owned by the host framework's pool and which is
// handed no allocator, or a latency-critical path that cannot afford
// cudaMalloc's implicit synchronisation and unbounded cost.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr size_t kStaticScratchBytes = DSA_TOPK_STATIC_SCRATCH_BYTES;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_topk_scratch[kStaticScratchBytes];

// Device address of g_topk_scratch per device.  In host code the array's name
// stands for a host-side shadow, not device memory, so its address must be
// looked up with the device current and never passed to a kernel directly.
void* g_scratch_addr[64] = {};
std::mutex g_scratch_mu;

dsa_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(DSA_ERR_UNSUPPORTED, "device ordinal >= 64");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || !p) return set_error(DSA_ERR_CUDA, "cudaGetSymbolAddress of the static top-k scratch failed");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_topk_select_decode_noalloc(const dsa_paged_kv* kv_, const int32_t* scores, int32_t ld,
                                                     int32_t prefix, int32_t k, int32_t* idx, int32_t* n_sel,
                                                     cudaStream_t stream) {
  dsa::KV kv{};
  size_t bytes = 0, clear_bytes = 0;
  dsa_status s = dsa::prepare_decode_topk(kv_, scores, ld, prefix, k, idx, n_sel, &kv, &bytes, &clear_bytes);
  if (s != DSA_OK) return s;
  if (bytes > dsa::kStaticScratchBytes)
    return dsa::set_error(DSA_ERR_UNSUPPORTED,
                          "decode top-k needs more scratch than the static array holds "
                          "(DSA_TOPK_STATIC_SCRATCH_BYTES); use dsa_topk_select with a workspace");
  if ((s = dsa::setup_device()) != DSA_OK) return s;
  void* base = nullptr;
  if ((s = dsa::scratch_for_current_device(&base)) != DSA_OK) return s;
  // The array keeps the previous call's contents: zero the histograms and
  // counters this call relies on (a memset, not an allocation).
  cudaError_t e = cudaMemsetAsync(base, 0, clear_bytes, stream);
  const dsa::SelState st = dsa::decode_topk_state(kv, k, prefix, base);
  if (e == cudaSuccess) e = dsa::launch_decode_hist(kv, scores, ld, prefix, k, st, stream);
  if (e == cudaSuccess) e = dsa::launch_decode_select(kv, scores, ld, prefix, k, st, idx, n_sel, stream);
  if (e != cudaSuccess) return dsa::set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return DSA_OK;
}
