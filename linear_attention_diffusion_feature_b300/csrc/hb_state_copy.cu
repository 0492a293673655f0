// hb_state_copy: copies per-request states between slots of one pool.
//
// A request's state S, Z is its whole summary of the blocks committed so far
// (gist.science technical summary, state-compression bullet: the states
// change only when a block is committed; pith.science review, "What carries
// the argument": S_n and Z_n are sums over the committed tokens). Copying it
// to another slot therefore snapshots the request (before it is preempted),
// restores it, or forks it into a second request with the same history.
//
// One CTA per (pair, head) moves the 64 KiB S tile (d = 128, F = 128) and Z
// with 16-byte loads and stores: a plain HBM copy, read once and written once.
//
// hb_state_to_bf16 writes the bf16 copy of listed slots' S that
// hb_block_attend_s16 reads: one CTA per (slot, head), 16-byte fp32 loads,
// round to nearest, 8-byte bf16 stores.
#include <cuda_bf16.h>

#include "hb_copy.cuh"
#include "hb_state16.cuh"

namespace hb {
namespace {

__global__ void __launch_bounds__(256)
    k_state_copy(int H, int F, int d, const int32_t* __restrict__ src,
                 const int32_t* __restrict__ dst, float* S_pool, float* Z_pool, int num_slots,
                 unsigned* status) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int from = src[b], to = dst[b];
  if (from < 0 || from >= num_slots || to < 0 || to >= num_slots) {
    if (threadIdx.x == 0 && h == 0) atomicOr(status, kStatusBounds);
    return;
  }
  if (from == to) return;
  // F * d is a multiple of 4 (F = 2f with f >= 8) and every tile starts on a
  // 16-byte boundary (the pool is 16-byte aligned)
  const size_t n4 = (size_t)F * d / 4;
  const float4* s_from =
      reinterpret_cast<const float4*>(S_pool + ((size_t)from * H + h) * F * d);
  float4* s_to = reinterpret_cast<float4*>(S_pool + ((size_t)to * H + h) * F * d);
  for (size_t i = threadIdx.x; i < n4; i += blockDim.x) s_to[i] = s_from[i];
  const float* z_from = Z_pool + ((size_t)from * H + h) * F;
  float* z_to = Z_pool + ((size_t)to * H + h) * F;
  for (int i = threadIdx.x; i < F; i += blockDim.x) z_to[i] = z_from[i];
}

__global__ void __launch_bounds__(256)
    k_state_to_bf16(int H, int F, int d, const int32_t* __restrict__ slot_idx,
                    const float* __restrict__ S_pool, __nv_bfloat16* __restrict__ S16_pool,
                    int num_slots, unsigned* status) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int slot = slot_idx[b];
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0 && h == 0) atomicOr(status, kStatusBounds);
    return;
  }
  const size_t base = ((size_t)slot * H + h) * F * d;
  const float4* from = reinterpret_cast<const float4*>(S_pool + base);
  uint2* to = reinterpret_cast<uint2*>(S16_pool + base);
  for (size_t i = threadIdx.x; i < (size_t)F * d / 4; i += blockDim.x) {
    const float4 x = from[i];
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    to[i] = w;
  }
}

}  // namespace

cudaError_t launch_state_to_bf16(const Shape& s, int batch, const int32_t* slot_idx,
                                 const float* S_pool, void* S16_pool, int num_slots,
                                 unsigned* status, cudaStream_t st) {
  k_state_to_bf16<<<dim3(batch, s.H), 256, 0, st>>>(s.H, s.F, s.d, slot_idx, S_pool,
                                                    static_cast<__nv_bfloat16*>(S16_pool),
                                                    num_slots, status);
  return cudaGetLastError();
}

cudaError_t launch_state_copy(const Shape& s, int batch, const int32_t* src, const int32_t* dst,
                              float* S_pool, float* Z_pool, int num_slots, unsigned* status,
                              cudaStream_t st) {
  k_state_copy<<<dim3(batch, s.H), 256, 0, st>>>(s.H, s.F, s.d, src, dst, S_pool, Z_pool,
                                                 num_slots, status);
  return cudaGetLastError();
}

}  // namespace hb
