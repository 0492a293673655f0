// Tensor-core kernels of block-hybrid attention for the production shape
// (bf16 activations, d = 128, f = 64, F = 128, L = 32) and their dispatch
// predicates. Every other shape or dtype goes to the generic kernels.
#pragma once

#include <utility>

#include "hb_internal.cuh"

namespace hb {

inline bool production_shape(const Shape& s) {
  return s.dtype == HB_DTYPE_BF16 && s.d == 128 && s.f == 64 && s.L == 32;
}

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel in the stream finishes, and the kernel
// itself calls grid_dep_wait() before its first global memory access.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

bool fast_feature_map_ok(const Shape& s);
bool fast_attend_ok(const Shape& s);
// a decoding step (not the sequential mode): blocks of 32 or 16 tokens
bool fast_attend_step_ok(const Shape& s);
bool fast_state_ok(const Shape& s);
bool fast_softmax_kv_ok(const Shape& s);

cudaError_t launch_feature_map_fast(const Shape& s, int64_t n, const void* x, const void* W,
                                    float* phi, unsigned* status, cudaStream_t st);
// commit_mask == nullptr and !commit_all: attend only (S_pool and Z_pool are
// not written). Otherwise request b with commit_mask[b] != 0 (every request,
// with commit_all) also folds its block's k, v into its state slot after its
// output has used the old state. Request b's block is rows
// b * rows_per_req + row_base .. + L - 1 of q, k, v and o. sequential: one
// CTA per (request, head) runs all rows_per_req / L blocks of the request in
// order (each attends to the state left by the ones before, then commits;
// row_base and commit_mask unused). Hkv > 0 (attend only, Hkv divides H and
// H / Hkv is at most 16): grouped-query heads, k, v, S and Z have Hkv heads
// and query head h reads head h / (H / Hkv); W is the query map [H, d, f].
// Wk (sequential mode only): a separate key map [H, d, f] for the commits.
bool attend_fast_fits(const Shape& s, int batch, int num_slots, int64_t rows_per_req);
// Several independent layers in one launch (n_layers x the requests of one
// layer; request b takes row (b / (batch / n_layers)) * H + h of W and gate).
// commit_mask null: attend only.
cudaError_t launch_attend_layers(const Shape& s, int n_layers, int batch, const int32_t* slot_idx,
                                 const void* q, const void* k, const void* v, float* S_pool,
                                 float* Z_pool, int num_slots, const void* W, const float* gate,
                                 const int32_t* commit_mask, void* o, unsigned* status,
                                 cudaStream_t st);
cudaError_t launch_attend_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* q,
                               const void* k, const void* v, const float* S_pool,
                               const float* Z_pool, int num_slots, const void* W,
                               const float* gate, const int32_t* commit_mask, void* o,
                               unsigned* status, cudaStream_t st, int rows_per_req, int row_base,
                               bool commit_all, bool sequential = false, int Hkv = -1,
                               const void* Wk = nullptr);
// Prompts with outputs, chunked onto tcgen05 (hb_prompt_tc.cu): one CTA per
// (request, head) walks its prompt in 128-token segments with the state in
// tensor memory; q, k, v, o are [batch, seq_len, H, d], seq_len a multiple
// of L (16, 32 or 64); the slots' states are read at the start and written
// back at the end for the requests that commit (commit_all, or
// commit_mask[b] != 0). With seq_len = L it is one decoding step.
bool prompt_tc_fits(const Shape& s, int batch, int num_slots, int64_t seq_len);
cudaError_t launch_prompt_tc(const Shape& s, int batch, const int32_t* slot_idx, const void* q,
                             const void* k, const void* v, int64_t seq_len, float* S_pool,
                             float* Z_pool, int num_slots, const void* W, const float* gate,
                             void* o, unsigned* status, cudaStream_t st, bool commit_all = true,
                             const int32_t* commit_mask = nullptr);
cudaError_t launch_commit_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                               const void* v, const void* W, float* S_pool, float* Z_pool,
                               int num_slots, unsigned* status, cudaStream_t st);
// One 32-token block per (request, head), two CTAs per SM (hb_commit_fast.cu).
// With mask, only the requests with mask[b] != 0 commit.
bool commit_tc_fits(const Shape& s, int batch, int num_slots);
cudaError_t launch_commit_tc(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                             const void* v, const void* W, float* S_pool, float* Z_pool,
                             int num_slots, unsigned* status, cudaStream_t st,
                             const int32_t* mask = nullptr);
size_t prefill_fast_workspace_bytes(const Shape& s, int batch, int64_t max_seqlen);
cudaError_t launch_prefill_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                                const void* v, int64_t total_tokens, const int64_t* cu_seqlens,
                                int64_t max_seqlen,
                                const void* W, float* S_pool, float* Z_pool, int num_slots,
                                int accumulate, void* workspace, unsigned* status,
                                cudaStream_t st);
size_t softmax_kv_fast_workspace_bytes(const Shape& s, int batch, int64_t max_prefix);
cudaError_t launch_softmax_kv_fast(const Shape& s, int batch, const void* k_cache,
                                   const void* v_cache, int64_t total_prefix,
                                   const int64_t* cu_prefix,
                                   int64_t max_prefix, const void* q, const void* k,
                                   const void* v, void* o, void* workspace, unsigned* status,
                                   cudaStream_t st);

}  // namespace hb
