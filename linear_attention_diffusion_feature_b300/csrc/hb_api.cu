// The C ABI of libhb.so (include/hb.h): host-side validation, the per-device
// status word, and dispatch to the kernels. No entry point allocates memory
// or synchronises, except hb_get_device_status.
#include <math.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "hb_fast.cuh"
#include "hb_internal.cuh"
#include "hb_paged.cuh"
#include "hb_copy.cuh"
#include "hb_state16.cuh"

namespace hb {

// Device-side fault bits (kStatusBounds, kStatusTimeout). One instance per
// device context; kernels receive its device address as an argument.
__device__ unsigned g_status_word;

// Wait limit of the attend kernels' unit pipeline, in SM clocks
// (hb_set_wait_limit; process-wide).
static std::atomic<long long> g_wait_limit{1ll << 32};
long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

namespace {

std::mutex g_mu;

cudaError_t status_word_ptr(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::map<int, unsigned*> cache;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_status_word);
  if (e != cudaSuccess) return e;
  cache[dev] = static_cast<unsigned*>(p);
  *out = static_cast<unsigned*>(p);
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

hb_status check_config(const hb_config* c, Shape* s) {
  if (!c) return HB_ERR_INVALID_ARG;
  if (c->dtype != HB_DTYPE_BF16 && c->dtype != HB_DTYPE_FP32) return HB_ERR_INVALID_ARG;
  if (c->merge != HB_MERGE_SHARED_NORM && c->merge != HB_MERGE_CONVEX) return HB_ERR_INVALID_ARG;
  if (!(c->scale >= 0.f) || isinf(c->scale)) return HB_ERR_INVALID_ARG;
  if (c->num_heads < 1 || c->num_heads > 1024) return HB_ERR_UNSUPPORTED_SHAPE;
  if (c->head_dim < 16 || c->head_dim > 128 || c->head_dim % 16) return HB_ERR_UNSUPPORTED_SHAPE;
  if (c->feat_half < 8 || c->feat_half > 64 || c->feat_half % 8) return HB_ERR_UNSUPPORTED_SHAPE;
  if (c->block_len < 1 || c->block_len > 64) return HB_ERR_UNSUPPORTED_SHAPE;
  s->H = c->num_heads;
  s->d = c->head_dim;
  s->f = c->feat_half;
  s->F = 2 * c->feat_half;
  s->L = c->block_len;
  s->scale = c->scale > 0.f ? c->scale : 1.f / sqrtf((float)c->head_dim);
  s->dtype = c->dtype;
  s->merge = c->merge;
  return HB_OK;
}

// All listed pointers non-null and 16-byte aligned.
hb_status check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p) return HB_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return HB_ERR_MISALIGNED;
  return HB_OK;
}

hb_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HB_OK : HB_ERR_CUDA; }

}  // namespace

cudaError_t current_sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::map<int, int> counts;
  std::lock_guard<std::mutex> lock(g_mu);
  int& c = counts[dev];
  if (c == 0 &&
      (e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
    c = 0;
    return e;
  }
  *n = c;
  return cudaSuccess;
}

cudaError_t ensure_smem_attr(const void* fn, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::map<std::pair<const void*, int>, int> done;
  std::lock_guard<std::mutex> lock(g_mu);
  int& have = done[{fn, dev}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

}  // namespace hb

using hb::Shape;

extern "C" {

hb_status hb_feature_map(const hb_config* cfg, int64_t n_tokens, const void* x, const void* W,
                         float* phi, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (n_tokens < 0) return HB_ERR_INVALID_ARG;
  if ((r = hb::check_ptrs({W})) != HB_OK) return r;
  if (n_tokens == 0) return HB_OK;
  if ((r = hb::check_ptrs({x, phi})) != HB_OK) return r;
  if (n_tokens > (int64_t)16 * 0x7fffffff) return HB_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_feature_map_ok(s)) {
    unsigned* status = nullptr;
    if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
    return hb::from_cuda(hb::launch_feature_map_fast(s, n_tokens, x, W, phi, status, st));
  }
  return hb::from_cuda(hb::launch_feature_map_generic(s, n_tokens, x, W, phi, st));
}

hb_status hb_block_attend(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                          const void* q, const void* k, const void* v, const float* S_pool,
                          const float* Z_pool, int32_t num_slots, const void* W,
                          const float* gate_logits, void* o, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S_pool, Z_pool, W, gate_logits, o})) != HB_OK)
    return r;
  unsigned* status = nullptr;
  cudaError_t e = hb::status_word_ptr(&status);
  if (e != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_attend_step_ok(s) && hb::attend_fast_fits(s, batch, num_slots, s.L))
    return hb::from_cuda(hb::launch_attend_fast(s, batch, slot_idx, q, k, v, S_pool, Z_pool,
                                                num_slots, W, gate_logits, nullptr, o, status,
                                                st, s.L, 0, false));
  if (hb::prompt_tc_fits(s, batch, num_slots, s.L))
    // blocks of 64 tokens: the segment kernel on a one-block prompt, the
    // states only read
    return hb::from_cuda(hb::launch_prompt_tc(s, batch, slot_idx, q, k, v, s.L,
                                              const_cast<float*>(S_pool),
                                              const_cast<float*>(Z_pool), num_slots, W,
                                              gate_logits, o, status, st, false, nullptr));
  return hb::from_cuda(hb::launch_attend_generic(s, batch, slot_idx, q, k, v, S_pool, Z_pool,
                                                 num_slots, W, gate_logits, o, status, st));
}

hb_status hb_state_to_bf16(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                           const float* S_pool, void* S16_pool, int32_t num_slots,
                           hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, S_pool, S16_pool})) != HB_OK) return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_state_to_bf16(s, batch, slot_idx, S_pool, S16_pool, num_slots,
                                                status, reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_block_attend_s16(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                              const void* q, const void* k, const void* v, const void* S16_pool,
                              const float* Z_pool, int32_t num_slots, const void* W,
                              const float* gate_logits, void* o, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (!hb::fast_attend_step_ok(s)) return HB_ERR_UNSUPPORTED_SHAPE;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32 || !hb::attend_fast_fits(s, batch, num_slots, s.L))
    return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S16_pool, Z_pool, W, gate_logits, o})) != HB_OK)
    return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_attend_fast_s16(s, batch, slot_idx, q, k, v, S16_pool, Z_pool,
                                                  num_slots, W, gate_logits, o, status,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_state_to_fp8(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                          const float* S_pool, void* S8_pool, float* scale_pool,
                          int32_t num_slots, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, S_pool, S8_pool, scale_pool})) != HB_OK) return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_state_to_fp8(s, batch, slot_idx, S_pool, S8_pool, scale_pool,
                                               num_slots, status,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_block_attend_s8(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                             const void* q, const void* k, const void* v, const void* S8_pool,
                             const float* scale_pool, const float* Z_pool, int32_t num_slots,
                             const void* W, const float* gate_logits, void* o,
                             hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (!hb::fast_attend_step_ok(s)) return HB_ERR_UNSUPPORTED_SHAPE;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32 || !hb::attend_fast_fits(s, batch, num_slots, s.L))
    return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S8_pool, scale_pool, Z_pool, W, gate_logits,
                           o})) != HB_OK)
    return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_attend_fast_s8(s, batch, slot_idx, q, k, v, S8_pool,
                                                 scale_pool, Z_pool, num_slots, W, gate_logits,
                                                 o, status,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_block_attend_commit(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                                 const void* q, const void* k, const void* v, float* S_pool,
                                 float* Z_pool, int32_t num_slots, const void* W,
                                 const float* gate_logits, const int32_t* commit, void* o,
                                 hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S_pool, Z_pool, W, gate_logits, commit, o})) !=
      HB_OK)
    return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_attend_step_ok(s) && hb::attend_fast_fits(s, batch, num_slots, s.L))
    return hb::from_cuda(hb::launch_attend_fast(s, batch, slot_idx, q, k, v, S_pool, Z_pool,
                                                num_slots, W, gate_logits, commit, o, status,
                                                st, s.L, 0, false));
  if (hb::prompt_tc_fits(s, batch, num_slots, s.L))
    // blocks of 64 tokens: the segment kernel on a one-block prompt;
    // committing requests write their new state back
    return hb::from_cuda(hb::launch_prompt_tc(s, batch, slot_idx, q, k, v, s.L, S_pool, Z_pool,
                                              num_slots, W, gate_logits, o, status, st, false,
                                              commit));
  // other shapes: the attend pass reads every state, then the committing
  // requests fold their block in, in stream order
  cudaError_t e = hb::launch_attend_generic(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots,
                                            W, gate_logits, o, status, st);
  if (e != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_commit_masked_generic(s, batch, slot_idx, commit, k, v, W,
                                                        S_pool, Z_pool, num_slots, status, st));
}

hb_status hb_block_attend_commit_layers(const hb_config* cfg, int32_t n_layers, int32_t batch,
                                        const int32_t* slot_idx, const void* q, const void* k,
                                        const void* v, float* S_pool, float* Z_pool,
                                        int32_t num_slots, const void* W,
                                        const float* gate_logits, const int32_t* commit, void* o,
                                        hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (n_layers < 1 || batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  const int64_t total = (int64_t)n_layers * batch;
  if (total > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S_pool, Z_pool, W, gate_logits, o})) != HB_OK)
    return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_attend_step_ok(s) && hb::attend_fast_fits(s, (int)total, num_slots, s.L))
    return hb::from_cuda(hb::launch_attend_layers(s, n_layers, (int)total, slot_idx, q, k, v,
                                                  S_pool, Z_pool, num_slots, W, gate_logits,
                                                  commit, o, status, st));
  // other shapes: one call per layer, in layer order
  const size_t es = cfg->dtype == HB_DTYPE_BF16 ? 2 : 4;
  const size_t act = (size_t)batch * s.L * s.H * s.d * es;
  const size_t wl = (size_t)s.H * s.d * s.f * es;
  for (int l = 0; l < n_layers; ++l) {
    const size_t b0 = (size_t)l * batch;
    const char* ql = static_cast<const char*>(q) + l * act;
    const char* kl = static_cast<const char*>(k) + l * act;
    const char* vl = static_cast<const char*>(v) + l * act;
    char* ol = static_cast<char*>(o) + l * act;
    const char* Wl = static_cast<const char*>(W) + l * wl;
    const float* gl = gate_logits + (size_t)l * s.H;
    r = commit ? hb_block_attend_commit(cfg, batch, slot_idx + b0, ql, kl, vl, S_pool, Z_pool,
                                        num_slots, Wl, gl, commit + b0, ol, stream)
               : hb_block_attend(cfg, batch, slot_idx + b0, ql, kl, vl, S_pool, Z_pool,
                                 num_slots, Wl, gl, ol, stream);
    if (r != HB_OK) return r;
  }
  return HB_OK;
}

hb_status hb_block_attend_commit_s16(const hb_config* cfg, int32_t batch,
                                     const int32_t* slot_idx, const void* q, const void* k,
                                     const void* v, float* S_pool, void* S16_pool,
                                     float* Z_pool, int32_t num_slots, const void* W,
                                     const float* gate_logits, const int32_t* commit, void* o,
                                     hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (!hb::fast_attend_step_ok(s)) return HB_ERR_UNSUPPORTED_SHAPE;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32 || !hb::attend_fast_fits(s, batch, num_slots, s.L))
    return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S_pool, S16_pool, Z_pool, W, gate_logits, commit,
                           o})) != HB_OK)
    return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_attend_commit_dual(
      s, batch, slot_idx, q, k, v, S_pool, S16_pool, Z_pool, num_slots, W, gate_logits, commit, o,
      status, reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_prefill_attend(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                            const void* q, const void* k, const void* v, int64_t seq_len,
                            float* S_pool, float* Z_pool, int32_t num_slots, const void* W,
                            const float* gate_logits, int32_t accumulate, void* o,
                            hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0 || seq_len < 0) return HB_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return HB_ERR_INVALID_ARG;
  if (seq_len % s.L != 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, S_pool, Z_pool, W, gate_logits})) != HB_OK) return r;
  if (seq_len > 0 && (r = hb::check_ptrs({q, k, v, o})) != HB_OK) return r;
  if ((int64_t)batch * seq_len >= ((int64_t)1 << 31)) return HB_ERR_UNSUPPORTED_SHAPE;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (accumulate == 0 &&
      (e = hb::launch_state_zero(s, batch, slot_idx, S_pool, Z_pool, num_slots, status, st)) !=
          cudaSuccess)
    return HB_ERR_CUDA;
  if (seq_len == 0) return HB_OK;
  if (hb::prompt_tc_fits(s, batch, num_slots, seq_len))
    // one CTA per (request, head) walks the prompt in 128-token segments on
    // the tensor cores, with the state in tensor memory
    return hb::from_cuda(hb::launch_prompt_tc(s, batch, slot_idx, q, k, v, seq_len, S_pool,
                                              Z_pool, num_slots, W, gate_logits, o, status, st));
  // other shapes: an attend and a commit launch per block, in stream order
  for (int64_t row = 0; row < seq_len; row += s.L) {
    e = hb::launch_attend_generic(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, W,
                                  gate_logits, o, status, st, seq_len, row);
    if (e == cudaSuccess)
      e = hb::launch_commit_rows_generic(s, batch, slot_idx, k, v, seq_len, row, W, S_pool,
                                         Z_pool, num_slots, status, st);
    if (e != cudaSuccess) return hb::from_cuda(e);
  }
  return HB_OK;
}

namespace {

// Shape of the key/value side of a grouped-query call: Hkv heads.
hb::Shape kv_shape(const hb::Shape& s, int Hkv) {
  hb::Shape k = s;
  k.H = Hkv;
  return k;
}

// The fast attend kernel takes grouped heads when a group's share of the
// block's key/value bytes stays a whole number of 16-byte pieces.
bool fast_group_ok(int G) { return G >= 1 && 512 % G == 0; }

// Attend only, grouped heads: the tensor-core kernel for the production
// shape, else the generic one. Request b's block is rows
// b * rows_per_req + row_base .. of q, k, v and o.
cudaError_t attend_grouped(const hb::Shape& s, int Hkv, int batch, const int32_t* slot_idx,
                           const void* q, const void* k, const void* v, const float* S_pool,
                           const float* Z_pool, int num_slots, const void* Wq,
                           const float* gate, void* o, unsigned* status, cudaStream_t st,
                           int64_t rows_per_req, int64_t row_base) {
  if (hb::fast_attend_step_ok(s) && fast_group_ok(s.H / Hkv) &&
      hb::attend_fast_fits(s, batch, num_slots, rows_per_req))
    return hb::launch_attend_fast(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, Wq,
                                  gate, nullptr, o, status, st, (int)rows_per_req, (int)row_base,
                                  false, false, Hkv, nullptr);
  return hb::launch_attend_generic(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, Wq,
                                   gate, o, status, st, rows_per_req, row_base, Hkv);
}

}  // namespace

hb_status hb_block_attend_ex(const hb_config* cfg, int32_t num_kv_heads, int32_t batch,
                             const int32_t* slot_idx, const void* q, const void* k,
                             const void* v, float* S_pool, float* Z_pool, int32_t num_slots,
                             const void* Wq, const void* Wk, const float* gate_logits,
                             const int32_t* commit, void* o, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (num_kv_heads < 1 || num_kv_heads > s.H || s.H % num_kv_heads != 0)
    return HB_ERR_UNSUPPORTED_SHAPE;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, q, k, v, S_pool, Z_pool, Wq, gate_logits, o})) != HB_OK)
    return r;
  if (commit && (r = hb::check_ptrs({commit, Wk})) != HB_OK) return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int Hkv = num_kv_heads;
  const Shape skv = kv_shape(s, Hkv);
  if (commit && Hkv == s.H && Wk == Wq)  // one map, one state per head: the fused step
    return hb_block_attend_commit(cfg, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, Wq,
                                  gate_logits, commit, o, stream);
  // the attend reads every state; then, in stream order, the committing
  // requests fold their block in with the key map, one state per key/value head
  cudaError_t e = attend_grouped(s, Hkv, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, Wq,
                                 gate_logits, o, status, st, s.L, 0);
  if (e != cudaSuccess || !commit) return hb::from_cuda(e);
  if (hb::fast_state_ok(skv) && hb::commit_tc_fits(skv, batch, num_slots))
    return hb::from_cuda(hb::launch_commit_tc(skv, batch, slot_idx, k, v, Wk, S_pool, Z_pool,
                                              num_slots, status, st, commit));
  return hb::from_cuda(hb::launch_commit_masked_generic(skv, batch, slot_idx, commit, k, v, Wk,
                                                        S_pool, Z_pool, num_slots, status, st));
}

hb_status hb_prefill_attend_ex(const hb_config* cfg, int32_t num_kv_heads, int32_t batch,
                               const int32_t* slot_idx, const void* q, const void* k,
                               const void* v, int64_t seq_len, float* S_pool, float* Z_pool,
                               int32_t num_slots, const void* Wq, const void* Wk,
                               const float* gate_logits, int32_t accumulate, void* o,
                               hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0 || seq_len < 0) return HB_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return HB_ERR_INVALID_ARG;
  if (num_kv_heads < 1 || num_kv_heads > s.H || s.H % num_kv_heads != 0)
    return HB_ERR_UNSUPPORTED_SHAPE;
  if (seq_len % s.L != 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, S_pool, Z_pool, Wq, Wk, gate_logits})) != HB_OK) return r;
  if (seq_len > 0 && (r = hb::check_ptrs({q, k, v, o})) != HB_OK) return r;
  if ((int64_t)batch * seq_len >= ((int64_t)1 << 31)) return HB_ERR_UNSUPPORTED_SHAPE;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int Hkv = num_kv_heads;
  const Shape skv = kv_shape(s, Hkv);
  cudaError_t e = cudaSuccess;
  if (accumulate == 0 &&
      (e = hb::launch_state_zero(skv, batch, slot_idx, S_pool, Z_pool, num_slots, status, st)) !=
          cudaSuccess)
    return HB_ERR_CUDA;
  if (seq_len == 0) return HB_OK;
  if (Hkv == s.H && Wk == Wq && hb::prompt_tc_fits(s, batch, num_slots, seq_len))
    return hb::from_cuda(hb::launch_prompt_tc(s, batch, slot_idx, q, k, v, seq_len, S_pool,
                                              Z_pool, num_slots, Wq, gate_logits, o, status, st));
  if (Hkv == s.H && hb::fast_attend_ok(s) && hb::attend_fast_fits(s, batch, num_slots, seq_len))
    // separate maps: one CTA per (request, head) walks the prompt's blocks
    // with the state and the key map kept on chip
    return hb::from_cuda(hb::launch_attend_fast(s, batch, slot_idx, q, k, v, S_pool, Z_pool,
                                                num_slots, Wq, gate_logits, nullptr, o, status,
                                                st, (int)seq_len, 0, true, true, Hkv, Wk));
  // grouped heads or other shapes: an attend and a commit launch per block
  for (int64_t row = 0; row < seq_len; row += s.L) {
    e = attend_grouped(s, Hkv, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, Wq,
                       gate_logits, o, status, st, seq_len, row);
    if (e == cudaSuccess)
      e = hb::launch_commit_rows_generic(skv, batch, slot_idx, k, v, seq_len, row, Wk, S_pool,
                                         Z_pool, num_slots, status, st);
    if (e != cudaSuccess) return hb::from_cuda(e);
  }
  return HB_OK;
}

hb_status hb_commit_block(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                          const void* k, const void* v, const void* W, float* S_pool,
                          float* Z_pool, int32_t num_slots, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, k, v, W, S_pool, Z_pool})) != HB_OK) return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_state_ok(s))
    return hb::from_cuda(hb::launch_commit_fast(s, batch, slot_idx, k, v, W, S_pool, Z_pool,
                                                num_slots, status, st));
  return hb::from_cuda(hb::launch_state_accumulate_generic(
      s, batch, slot_idx, k, v, (int64_t)batch * s.L, nullptr, s.L, W, S_pool, Z_pool,
      num_slots, 1, status, st));
}

size_t hb_prefill_workspace_size(const hb_config* cfg, int32_t batch, int64_t max_seqlen) {
  Shape s;
  if (hb::check_config(cfg, &s) != HB_OK || batch <= 0 || max_seqlen < 0) return 0;
  return hb::fast_state_ok(s) ? hb::prefill_fast_workspace_bytes(s, batch, max_seqlen) : 0;
}

hb_status hb_prefill_state(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                           const void* k, const void* v, int64_t total_tokens,
                           const int64_t* cu_seqlens, int64_t max_seqlen, const void* W, float* S_pool, float* Z_pool,
                           int32_t num_slots, int32_t accumulate, void* workspace,
                           size_t workspace_bytes, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0 || max_seqlen < 0 || total_tokens < 0) return HB_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, cu_seqlens, W, S_pool, Z_pool})) != HB_OK) return r;
  // k/v may be absent when there are no prompt tokens at all.
  if (total_tokens > 0 && (r = hb::check_ptrs({k, v})) != HB_OK) return r;
  const size_t need = hb_prefill_workspace_size(cfg, batch, max_seqlen);
  if (need > 0) {
    if (workspace_bytes < need) return HB_ERR_WORKSPACE;
    if ((r = hb::check_ptrs({workspace})) != HB_OK) return r;
  }
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_state_ok(s))
    return hb::from_cuda(hb::launch_prefill_fast(s, batch, slot_idx, k, v, total_tokens,
                                                 cu_seqlens, max_seqlen,
                                                 W, S_pool, Z_pool, num_slots, accumulate,
                                                 workspace, status, st));
  return hb::from_cuda(hb::launch_state_accumulate_generic(s, batch, slot_idx, k, v, total_tokens,
                                                           cu_seqlens, max_seqlen, W, S_pool,
                                                           Z_pool,
                                                           num_slots, accumulate, status, st));
}

hb_status hb_state_zero(const hb_config* cfg, int32_t batch, const int32_t* slot_idx,
                        float* S_pool, float* Z_pool, int32_t num_slots, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({slot_idx, S_pool, Z_pool})) != HB_OK) return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_state_zero(s, batch, slot_idx, S_pool, Z_pool, num_slots,
                                             status, reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_state_copy(const hb_config* cfg, int32_t batch, const int32_t* src_slot,
                        const int32_t* dst_slot, float* S_pool, float* Z_pool,
                        int32_t num_slots, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || num_slots < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({src_slot, dst_slot, S_pool, Z_pool})) != HB_OK) return r;
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  return hb::from_cuda(hb::launch_state_copy(s, batch, src_slot, dst_slot, S_pool, Z_pool,
                                             num_slots, status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

size_t hb_softmax_kv_workspace_size(const hb_config* cfg, int32_t batch, int64_t max_prefix) {
  Shape s;
  if (hb::check_config(cfg, &s) != HB_OK || batch <= 0 || max_prefix < 0) return 0;
  return hb::fast_softmax_kv_ok(s) ? hb::softmax_kv_fast_workspace_bytes(s, batch, max_prefix)
                                   : 0;
}

hb_status hb_softmax_kv_attend(const hb_config* cfg, int32_t batch, const void* k_cache,
                               const void* v_cache, int64_t total_prefix,
                               const int64_t* cu_prefix, int64_t max_prefix,
                               const void* q, const void* k, const void* v, void* o,
                               void* workspace, size_t workspace_bytes, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || max_prefix < 0 || total_prefix < 0) return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({cu_prefix, q, k, v, o})) != HB_OK) return r;
  if (total_prefix > 0 && (r = hb::check_ptrs({k_cache, v_cache})) != HB_OK) return r;
  const size_t need = hb_softmax_kv_workspace_size(cfg, batch, max_prefix);
  if (need > 0) {
    if (workspace_bytes < need) return HB_ERR_WORKSPACE;
    if ((r = hb::check_ptrs({workspace})) != HB_OK) return r;
  }
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (hb::fast_softmax_kv_ok(s))
    return hb::from_cuda(hb::launch_softmax_kv_fast(s, batch, k_cache, v_cache, total_prefix,
                                                    cu_prefix,
                                                    max_prefix, q, k, v, o, workspace, status,
                                                    st));
  return hb::from_cuda(hb::launch_softmax_kv_generic(s, batch, k_cache, v_cache, total_prefix,
                                                     cu_prefix,
                                                     max_prefix, q, k, v, o, status, st));
}

hb_status hb_softmax_kv_attend_paged(const hb_config* cfg, int32_t batch, const void* k_pages,
                                     const void* v_pages, int64_t num_pages, int32_t page_tokens,
                                     const int32_t* page_table, int32_t max_pages,
                                     const int32_t* prefix_len, int64_t max_prefix, const void* q,
                                     const void* k, const void* v, void* o, void* workspace,
                                     size_t workspace_bytes, hb_stream_t stream) {
  Shape s;
  hb_status r = hb::check_config(cfg, &s);
  if (r != HB_OK) return r;
  if (batch < 0 || max_prefix < 0 || max_prefix > INT32_MAX || num_pages < 0 ||
      page_tokens <= 0 || max_pages < 0)
    return HB_ERR_INVALID_ARG;
  if (batch == 0) return HB_OK;
  if (batch > 65535 * 32) return HB_ERR_UNSUPPORTED_SHAPE;
  if ((r = hb::check_ptrs({prefix_len, q, k, v, o})) != HB_OK) return r;
  if (max_pages > 0 && (r = hb::check_ptrs({page_table})) != HB_OK) return r;
  if (num_pages > 0 && (r = hb::check_ptrs({k_pages, v_pages})) != HB_OK) return r;
  const size_t need =
      hb::softmax_kv_paged_fast_fits(s, batch, num_pages, page_tokens, max_pages)
          ? hb::softmax_kv_fast_workspace_bytes(s, batch, max_prefix)
          : 0;
  if (need > 0) {
    if (workspace_bytes < need) return HB_ERR_WORKSPACE;
    if ((r = hb::check_ptrs({workspace})) != HB_OK) return r;
  }
  unsigned* status = nullptr;
  if (hb::status_word_ptr(&status) != cudaSuccess) return HB_ERR_CUDA;
  hb::PagedKV pg;
  pg.table = page_table;
  pg.plen = prefix_len;
  pg.max_pages = max_pages;
  pg.page_tokens = page_tokens;
  pg.num_pages = num_pages;
  return hb::from_cuda(hb::launch_softmax_kv_paged(s, batch, k_pages, v_pages, pg, max_prefix, q,
                                                   k, v, o, workspace, status,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

hb_status hb_set_wait_limit(uint64_t cycles) {
  constexpr uint64_t kDefault = 1ull << 32, kMax = 1ull << 40;
  hb::g_wait_limit.store((long long)(cycles == 0 ? kDefault : (cycles > kMax ? kMax : cycles)),
                         std::memory_order_relaxed);
  return HB_OK;
}

hb_status hb_get_device_status(hb_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return HB_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, hb::g_status_word, sizeof(word)) != cudaSuccess)
    return HB_ERR_CUDA;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(hb::g_status_word, &zero, sizeof(zero)) != cudaSuccess)
      return HB_ERR_CUDA;
  }
  if (word & hb::kStatusBounds) return HB_ERR_DEVICE_BOUNDS;
  if (word & hb::kStatusTimeout) return HB_ERR_TIMEOUT;
  return HB_OK;
}

const char* hb_status_string(hb_status status) {
  switch (status) {
    case HB_OK: return "ok";
    case HB_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad enum)";
    case HB_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (H, d, f or L)";
    case HB_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case HB_ERR_CUDA: return "CUDA runtime error";
    case HB_ERR_DEVICE_BOUNDS: return "device saw an index or length out of range";
    case HB_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case HB_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

}  // extern "C"
