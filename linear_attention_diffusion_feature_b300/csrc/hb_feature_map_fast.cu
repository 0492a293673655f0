// Hedgehog feature map for the production shape (bf16, d = 128, f = 64):
//   phi(x) = [softmax(x W_h), softmax(-x W_h)]
// (gist.science technical summary of arXiv 2608.06628, cross-block bullet;
// pith.science review, "What carries the argument").
//
// HBM-bound: 256 B of x in and 512 B of fp32 phi out per token and head, so
// the kernel is a plain tiled streaming pass:
//   * CTA = 64 tokens of one head; x (two 64-column SWIZZLE_128B boxes) and
//     W_h (one box) arrive by TMA on one mbarrier;
//   * warp w takes tokens 16w .. 16w + 15: u = x W_h on bf16 mma.sync with
//     fp32 accumulation (8 n-tiles x 8 k16 steps), the row max / min / sums
//     of both softmaxes reduce over the four threads of a quad with
//     shuffles, exponentials are 2^x with log2(e) folded in;
//   * each thread stores its 32 phi values as 8-byte pairs straight from
//     registers (every 32-byte sector of a row is written whole).
#include <float.h>

#include "hb_fast.cuh"
#include "hb_ptx.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kFH = 64, kF = 128;
constexpr int kTok = 64;
constexpr int kThreads = 128;
constexpr int kOffX = 0;       // 2 x [64 tokens][128 B]
constexpr int kOffW = 16384;   // [128 d rows][128 B]
constexpr int kOffBar = 32768;
constexpr int kSmemBytes = kOffBar + 16 + 1024;

struct Maps {
  CUtensorMap x;  // [n][H][d] bf16, box {64, 1, 64}
  CUtensorMap W;  // [H*d][f] bf16, box {64, 128}
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads)
    k_feature_map_fast(const __grid_constant__ Maps maps, int64_t n, int H,
                       float* __restrict__ phi, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kTok;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, 2 * 8192 + 16384);
    tma_load_3d(smem + kOffX, &maps.x, 0, h, (int)t0, bar);
    tma_load_3d(smem + kOffX + 8192, &maps.x, 64, h, (int)t0, bar);
    tma_load_2d(smem + kOffW, &maps.W, 0, h * kD, bar);
  }
  if (!mbar_wait(bar, 0)) {
    if (lane == 0) atomicOr(status, kStatusTimeout);
    return;
  }
  const uint32_t sX = smem_u32(smem + kOffX), sW = smem_u32(smem + kOffW);
  const int g = lane >> 2, t = lane & 3;

  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const int arow = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
  const int mtx = lane >> 3;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t a[4];
    const int ch = 2 * kk + (lane >> 4);
    ldsm_x4(sX + (ch >> 3) * 8192 + sw128(arow, ch & 7), a[0], a[1], a[2], a[3]);
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {  // n-tiles 2jp, 2jp + 1
      uint32_t b[4];
      const int krow = 16 * kk + (mtx & 1) * 8 + (lane & 7);
      ldsm_x4_t(sW + sw128(krow, 2 * jp + (mtx >> 1)), b[0], b[1], b[2], b[3]);
      mma_bf16(acc[2 * jp], a, b[0], b[1]);
      mma_bf16(acc[2 * jp + 1], a, b[2], b[3]);
    }
  }

  // rows g (elements 0, 1) and g + 8 (elements 2, 3) of this warp's tile
  float mx[2] = {-FLT_MAX, -FLT_MAX}, mn[2] = {FLT_MAX, FLT_MAX};
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      mx[r >> 1] = fmaxf(mx[r >> 1], acc[j][r]);
      mn[r >> 1] = fminf(mn[r >> 1], acc[j][r]);
    }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr)
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], o));
      mn[hr] = fminf(mn[hr], __shfl_xor_sync(0xffffffffu, mn[hr], o));
    }
  float ep[8][4], em[8][4], sp[2] = {0.f, 0.f}, sm[2] = {0.f, 0.f};
  const float op[2] = {-mx[0] * kLog2e, -mx[1] * kLog2e};
  const float om[2] = {mn[0] * kLog2e, mn[1] * kLog2e};
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ep[j][r] = ex2_approx(fmaf(acc[j][r], kLog2e, op[r >> 1]));   // e^{u - max}
      em[j][r] = ex2_approx(fmaf(-acc[j][r], kLog2e, om[r >> 1]));  // e^{min - u}
      sp[r >> 1] += ep[j][r];
      sm[r >> 1] += em[j][r];
    }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr)
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      sp[hr] += __shfl_xor_sync(0xffffffffu, sp[hr], o);
      sm[hr] += __shfl_xor_sync(0xffffffffu, sm[hr], o);
    }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int64_t tok = t0 + 16 * warp + g + 8 * hr;
    if (tok >= n) continue;
    const float ip = 1.f / sp[hr], im = 1.f / sm[hr];
    float* row = phi + (tok * H + h) * (int64_t)kF;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = 8 * j + 2 * t;
      *reinterpret_cast<float2*>(row + c) =
          make_float2(ep[j][2 * hr] * ip, ep[j][2 * hr + 1] * ip);
      *reinterpret_cast<float2*>(row + kFH + c) =
          make_float2(em[j][2 * hr] * im, em[j][2 * hr + 1] * im);
    }
  }
}

}  // namespace

bool fast_feature_map_ok(const Shape& s) { return production_shape(s); }

cudaError_t launch_feature_map_fast(const Shape& s, int64_t n, const void* x, const void* W,
                                    float* phi, unsigned* status, cudaStream_t st) {
  if (n >= ((int64_t)1 << 31) - kTok || (n + kTok - 1) / kTok > 0x7fffffff)
    return launch_feature_map_generic(s, n, x, W, phi, st);
  Maps maps;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)n};
    const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
    const uint32_t box[3] = {64, 1, kTok};
    if (!encode_tmap(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)kFH, (uint64_t)s.H * kD};
    const uint64_t strides[1] = {kFH * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap(&maps.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_feature_map_fast), kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((n + kTok - 1) / kTok), s.H);
  k_feature_map_fast<<<grid, kThreads, kSmemBytes, st>>>(maps, n, s.H, phi, status);
  return cudaGetLastError();
}

}  // namespace hb
