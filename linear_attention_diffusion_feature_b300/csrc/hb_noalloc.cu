// hb_prefill_state_noalloc: prompt ingestion for callers that cannot call
// cudaMalloc. The split-T partial sums that hb_prefill_state keeps in a
// caller-provided workspace live here in one file-scope device array instead.
//
// The array is a module global: every GPU that loads libhb.so holds its
// HB_PREFILL_NOALLOC_SCRATCH_BYTES until the process exits. On the host its
// name only stands in for the device object, so its device address is looked
// up once per device (with that device current) and handed to the kernels as
// an ordinary pointer.
#include <map>
#include <mutex>

#include "hb_internal.cuh"

namespace hb {
namespace {

__device__ __align__(256) unsigned char g_prefill_scratch[HB_PREFILL_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;

// Device address of g_prefill_scratch on the current device, resolved on the
// first call for that device and cached afterwards.
cudaError_t scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::map<int, void*> cache;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_prefill_scratch);
  if (e != cudaSuccess) return e;
  cache[dev] = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace hb

extern "C" hb_status hb_prefill_state_noalloc(const hb_config* cfg, int32_t batch,
                                              const int32_t* slot_idx, const void* k,
                                              const void* v, int64_t total_tokens,
                                              const int64_t* cu_seqlens, int64_t max_seqlen,
                                              const void* W, float* S_pool, float* Z_pool,
                                              int32_t num_slots, int32_t accumulate,
                                              hb_stream_t stream) {
  // Every partial sum the kernels read back is written earlier in the same
  // call, so the array needs no clearing between calls.
  const size_t need = hb_prefill_workspace_size(cfg, batch, max_seqlen);
  if (need > (size_t)HB_PREFILL_NOALLOC_SCRATCH_BYTES) return HB_ERR_WORKSPACE;
  // A call that needs no scratch (another shape, a batch too large to split,
  // or arguments hb_prefill_state rejects) goes straight through.
  void* scratch = nullptr;
  if (need > 0 && hb::scratch_ptr(&scratch) != cudaSuccess) return HB_ERR_CUDA;
  return hb_prefill_state(cfg, batch, slot_idx, k, v, total_tokens, cu_seqlens, max_seqlen, W,
                          S_pool, Z_pool, num_slots, accumulate, scratch,
                          need > 0 ? (size_t)HB_PREFILL_NOALLOC_SCRATCH_BYTES : 0, stream);
}
