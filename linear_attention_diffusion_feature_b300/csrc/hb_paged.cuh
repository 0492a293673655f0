// Paged KV cache for the comparison softmax pass (hb_softmax_kv_attend_paged).
// Internal to libhb.so; the public signature is in include/hb.h.
#pragma once

#include <stdint.h>

#include "hb_internal.cuh"

namespace hb {

// A paged KV cache: token t of request b is row t % page_tokens of page
// table[b * max_pages + t / page_tokens] of a pool of num_pages pages, each
// [page_tokens][H][d]; plen[b] is the request's cached-token count.
struct PagedKV {
  const int32_t* table = nullptr;
  const int32_t* plen = nullptr;
  int max_pages = 0, page_tokens = 0;
  int64_t num_pages = 0;
};

// Any shape and page size (hb_generic.cu).
cudaError_t launch_softmax_kv_paged_generic(const Shape& s, int batch, const void* k_pages,
                                            const void* v_pages, const PagedKV& pg,
                                            int64_t max_prefix, const void* q, const void* k,
                                            const void* v, void* o, unsigned* status,
                                            cudaStream_t st);

// The TMA kernel (hb_softmax_kv_fast.cu) when the shape is the production one,
// page_tokens is a multiple of 32 and the pool fits 32-bit row coordinates;
// launch_softmax_kv_paged falls back to the generic kernel (which needs no
// workspace) otherwise.
bool softmax_kv_paged_fast_fits(const Shape& s, int batch, int64_t num_pages, int page_tokens,
                                int max_pages);
cudaError_t launch_softmax_kv_paged(const Shape& s, int batch, const void* k_pages,
                                    const void* v_pages, const PagedKV& pg, int64_t max_prefix,
                                    const void* q, const void* k, const void* v, void* o,
                                    void* workspace, unsigned* status, cudaStream_t st);

}  // namespace hb
