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
//
// hb_state_to_fp8 writes the fp8 copy that hb_block_attend_s8 reads: per
// (slot, head), scale = max|S| / 448 (fp32, rounded to nearest) and
// code = e4m3(S / scale) (the quotient rounded to nearest in fp32, then to
// the nearest e4m3 value, ties to even, saturating at 448); a zero state
// gets scale 0 and zero codes.
#include <cuda_bf16.h>

#include "hb_copy.cuh"
#include "hb_ptx.cuh"
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

__global__ void __launch_bounds__(256)
    k_state_to_fp8(int H, int F, int d, const int32_t* __restrict__ slot_idx,
                   const float* __restrict__ S_pool, uint8_t* __restrict__ S8_pool,
                   float* __restrict__ scale_pool, int num_slots, unsigned* status) {
  __shared__ float wmax[8];
  const int b = blockIdx.x, h = blockIdx.y;
  const int slot = slot_idx[b];
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0 && h == 0) atomicOr(status, kStatusBounds);
    return;
  }
  const size_t base = ((size_t)slot * H + h) * F * d;
  const float4* from = reinterpret_cast<const float4*>(S_pool + base);
  const size_t n4 = (size_t)F * d / 4;
  float m = 0.f;
  for (size_t i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 x = from[i];
    m = fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
  const float scale = amax / 448.f;
  if (threadIdx.x == 0) scale_pool[(size_t)slot * H + h] = scale;
  uint32_t* to = reinterpret_cast<uint32_t*>(S8_pool + base);
  for (size_t i = threadIdx.x; i < n4; i += blockDim.x) {
    uint32_t w = 0u;
    if (amax > 0.f) {
      const float4 x = from[i];
      w = ptx::f32x2_to_e4m3x2(x.x / scale, x.y / scale) |
          (ptx::f32x2_to_e4m3x2(x.z / scale, x.w / scale) << 16);
    }
    to[i] = w;
  }
}

}  // namespace

cudaError_t launch_state_to_fp8(const Shape& s, int batch, const int32_t* slot_idx,
                                const float* S_pool, void* S8_pool, float* scale_pool,
                                int num_slots, unsigned* status, cudaStream_t st) {
  k_state_to_fp8<<<dim3(batch, s.H), 256, 0, st>>>(s.H, s.F, s.d, slot_idx, S_pool,
                                                   static_cast<uint8_t*>(S8_pool), scale_pool,
                                                   num_slots, status);
  return cudaGetLastError();
}

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
