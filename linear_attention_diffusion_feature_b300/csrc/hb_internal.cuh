// Internal declarations shared by the translation units of libhb.so.
// Nothing here is part of the public C ABI (include/hb.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hb.h"

namespace hb {

// Bits of the per-device status word (see hb_get_device_status).
enum : unsigned { kStatusBounds = 1u, kStatusTimeout = 2u };

// Validated problem description handed to the launchers.
struct Shape {
  int H;        // heads
  int d;        // head dimension
  int f;        // width of one softmax half of phi
  int F;        // 2f
  int L;        // active-block length
  float scale;  // block softmax scale (resolved; never 0)
  int dtype;    // hb_dtype
  int merge;    // hb_merge
};

// ----------------------------------------------------------- element access
template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// log(sigmoid(a)) = -softplus(-a), finite for finite a, -inf for a = -inf.
__device__ __forceinline__ float log_sigmoid(float a) {
  return a >= 0.f ? -log1pf(expf(-a)) : a - log1pf(expf(a));
}
__device__ __forceinline__ float sigmoid(float a) {
  return a >= 0.f ? 1.f / (1.f + expf(-a)) : expf(a) / (1.f + expf(a));
}

// Gated merge of one output element, shared by every attend kernel.
//   U    = sum_j e^{s_ij - m_i} v_j   (block numerator, shifted by the row max)
//   P    = sum_j e^{s_ij - m_i}       (block denominator, same shift)
//   m    = m_i
//   n    = phi(q_i)^T S[:, col],  den = phi(q_i)^T Z
//   aux  = log(sigmoid(alpha)) for SHARED_NORM, sigmoid(g) for CONVEX
// SHARED_NORM: with lam = log(w) + m, (w e^m U + n) / (w e^m P + den) is
// evaluated as (U + e^-lam n)/(P + e^-lam den) when lam >= 0 and as
// (e^lam U + n)/(e^lam P + den) otherwise, so neither exponential overflows.
__device__ __forceinline__ float merge_out(int merge, float U, float P, float m,
                                           float n, float den, float aux) {
  if (merge == HB_MERGE_SHARED_NORM) {
    const float lam = aux + m;
    if (lam >= 0.f) {
      const float r = expf(-lam);
      return (U + r * n) / (P + r * den);
    }
    const float r = expf(lam);
    return (r * U + n) / (r * P + den);
  }
  const float soft = U / P;
  return den > 0.f ? aux * soft + (1.f - aux) * (n / den) : soft;
}

// --------------------------------------------------------------- launchers
// Generic kernels: any supported shape, bf16 or fp32 activations, fp32 FMA
// arithmetic. They are the accuracy path (HB_DTYPE_FP32) and cover shapes the
// tensor-core kernels are not built for.
cudaError_t launch_feature_map_generic(const Shape& s, int64_t n, const void* x, const void* W,
                                       float* phi, cudaStream_t st);
// Request b's block is rows b * rows_per_req + row_base .. + L - 1 of q, k, v
// and o (rows_per_req < 0 means L). Hkv > 0: grouped-query heads, k, v, S
// and Z have Hkv heads and query head h reads head h / (H / Hkv); W is the
// query map [H, d, f].
cudaError_t launch_attend_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                  const void* q, const void* k, const void* v, const float* S_pool,
                                  const float* Z_pool, int num_slots, const void* W,
                                  const float* gate, void* o, unsigned* status, cudaStream_t st,
                                  int64_t rows_per_req = -1, int64_t row_base = 0, int Hkv = -1);
// commit (cu_seqlens == nullptr: request b owns rows [b*L, b*L+L)) and prefill.
cudaError_t launch_state_accumulate_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                            const void* k, const void* v, int64_t total_tokens,
                                            const int64_t* cu_seqlens, int64_t max_seqlen,
                                            const void* W, float* S_pool, float* Z_pool,
                                            int num_slots, int accumulate, unsigned* status,
                                            cudaStream_t st);
// commit of the requests with mask[b] != 0 (rows [b*L, b*L + L) of k, v)
cudaError_t launch_commit_masked_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                         const int32_t* mask, const void* k, const void* v,
                                         const void* W, float* S_pool, float* Z_pool,
                                         int num_slots, unsigned* status, cudaStream_t st);
// commit of every request's block at rows b * rows_per_req + row_base .. + L - 1
cudaError_t launch_commit_rows_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                       const void* k, const void* v, int64_t rows_per_req,
                                       int64_t row_base, const void* W, float* S_pool,
                                       float* Z_pool, int num_slots, unsigned* status,
                                       cudaStream_t st);
cudaError_t launch_state_zero(const Shape& s, int batch, const int32_t* slot_idx, float* S_pool,
                              float* Z_pool, int num_slots, unsigned* status, cudaStream_t st);
cudaError_t launch_softmax_kv_generic(const Shape& s, int batch, const void* k_cache,
                                      const void* v_cache, int64_t total_prefix,
                                      const int64_t* cu_prefix,
                                      int64_t max_prefix, const void* q, const void* k,
                                      const void* v, void* o, unsigned* status, cudaStream_t st);

// Raises cudaFuncAttributeMaxDynamicSharedMemorySize of `fn` on the current
// device to at least `bytes` (remembered per kernel and device, so the
// runtime is asked only when the value has to grow).
cudaError_t ensure_smem_attr(const void* fn, int bytes);
// Streaming multiprocessors of the current device (cached per device).
cudaError_t current_sm_count(int* n);
// SM clocks after which a wait of the attend kernels' unit pipeline gives up
// (hb_set_wait_limit).
long long wait_limit_cycles();

}  // namespace hb
