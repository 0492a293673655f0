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
#include "hb_copy.cuh"

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

}  // namespace

cudaError_t launch_state_copy(const Shape& s, int batch, const int32_t* src, const int32_t* dst,
                              float* S_pool, float* Z_pool, int num_slots, unsigned* status,
                              cudaStream_t st) {
  k_state_copy<<<dim3(batch, s.H), 256, 0, st>>>(s.H, s.F, s.d, src, dst, S_pool, Z_pool,
                                                 num_slots, status);
  return cudaGetLastError();
}

}  // namespace hb
