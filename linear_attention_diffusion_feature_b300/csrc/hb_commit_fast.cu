// Block commit for the production shape (bf16, d = 128, f = 64, F = 128,
// L = 32) on the 5th-generation tensor cores.
//
// Definition (pith.science review of arXiv 2608.06628, "What carries the
// argument"; gist.science technical summary, state-compression bullet: the
// state changes only when a block is committed):
//   S += sum_t phi(k_t) v_t^T,  Z += sum_t phi(k_t),  t over the L block tokens,
//   phi(k) = [softmax(k W_h), softmax(-k W_h)].
//
// One CTA per (request, head); small enough that two CTAs share an SM, so a
// commit of up to 148 requests' heads runs as a single wave:
//   warp 0     TMA: the block's k (four copies stacked into the 128 rows of
//              the MMA operand), v, W_h;
//   warp 1     owns 256 TMEM columns, issues tcgen05.mma from one thread:
//                U    [128 x 64]   = K4 W_h        (lane 32c + j = token j)
//                Sacc [128 F x 128 d] = phi^T V    (phi split hi + lo bf16)
//                Zacc [128 F x 16]    = phi^T 1
//   warps 2-5  epilogue; the warp on TMEM lane quarter c takes columns
//              16c..16c+15 of u for all 32 tokens, so the two softmaxes of a
//              token are shared by four threads (row max / sum through shared
//              memory); each writes its slice of phi(k) as bf16 hi + lo.
// The accumulator tile is staged in shared memory in the TMA SWIZZLE_128B
// layout and added into S and Z by the TMA unit (cp.reduce.async.bulk .add),
// so the old state is never read into the SM; each element receives exactly
// one add, so the result does not depend on timing.
#include <float.h>

#include "hb_fast.cuh"
#include "hb_ptx.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kFH = 64, kF = 128, kL = 32;
constexpr int kThreads = 192;

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int kOffK = 0;          // 2 d-halves x [128 rows][128 B]; rows 32c + j = token j
constexpr int kOffV = 32768;      // 2 d-halves x [32 tok][128 B]
constexpr int kOffW = 40960;      // [128 d rows][64 bf16]
constexpr int kOffPhiHi = 57344;  // 2 F-halves x [32 tok][128 B]
constexpr int kOffPhiLo = 65536;
constexpr int kOffOnes = 73728;   // [16 rows][128 B] of bf16 1.0
constexpr int kOffStats = 75776;  // max, min, sum+, sum- : [4 quarters][32 tokens] each
constexpr int kOffZst = 77824;    // [128] fp32 Z accumulator, staged for the bulk add
constexpr int kOffBar = 78336;
constexpr int kSmemBytes = kOffBar + 64 + 1024;
// The S accumulator is staged over [0, 64 KiB) once every MMA has completed:
// four SWIZZLE_128B boxes of [128 F rows][32 fp32].
constexpr int kOffStage = 0;
static_assert(kOffPhiLo == kOffStage + 65536, "staging must not reach the low phi bytes");

enum { kInFull = 0, kUFull, kPhiFull, kAccFull, kNumBars };
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColU = 0, kColZ = 128;  // U is consumed before S is written

struct Maps {
  CUtensorMap k;  // [B*L][H][d] bf16, box {64, 1, 32}
  CUtensorMap v;
  CUtensorMap W;  // [H*d][f] bf16, box {64, 128}
  CUtensorMap S;  // [slots*H*F][d] fp32, box {32, 128}
};

__device__ __forceinline__ uint32_t s_off(int k, int n) {
  return (uint32_t)((n >> 5) * 16384 + k * 128 + ((((n & 31) >> 2) ^ (k & 7)) << 4) + (n & 3) * 4);
}

// bar.red.and over the 128 epilogue threads: true if every thread passed true.
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kThreads, 2)
    k_commit_tc(const __grid_constant__ Maps maps, int H, int num_slots,
                const int32_t* __restrict__ slot_idx, const int32_t* __restrict__ mask,
                float* __restrict__ Z_pool, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  float* stats = reinterpret_cast<float*>(smem + kOffStats);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  if (mask != nullptr && mask[b] == 0) return;  // this request does not commit
  const int slot = slot_idx[b];
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBounds);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bar[kInFull], 1);
    mbar_init(&bar[kUFull], 1);
    mbar_init(&bar[kPhiFull], 4);
    mbar_init(&bar[kAccFull], 1);
    fence_mbar_init();
  }
  if (warp >= 2) {  // constant ones tile (B operand of the Z contraction)
    const uint32_t ones = smem_u32(smem + kOffOnes);
    const uint32_t one2 = 0x3F803F80u;  // two bf16 1.0
    st_shared_v4(ones + (threadIdx.x - 64) * 16, one2, one2, one2, one2);
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      prefetch_tmap(&maps.W);
      mbar_arrive_expect_tx(&bar[kInFull], 32768 + 8192 + 16384);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tma_load_3d(smem + kOffK + j * 16384 + c * 4096, &maps.k, 64 * j, h, b * kL,
                      &bar[kInFull]);
        tma_load_3d(smem + kOffV + j * 4096, &maps.v, 64 * j, h, b * kL, &bar[kInFull]);
      }
      tma_load_2d(smem + kOffW, &maps.W, 0, h * kD, &bar[kInFull]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idU = umma_idesc_bf16(128, kFH, 0, 1);
      constexpr uint32_t idS = umma_idesc_bf16(128, kD, 1, 1);
      constexpr uint32_t idZ = umma_idesc_bf16(128, 16, 1, 0);
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sW = smem_u32(smem + kOffW);
      const uint32_t sHi = smem_u32(smem + kOffPhiHi), sLo = smem_u32(smem + kOffPhiLo);
      const uint64_t dOnes = umma_desc_sw128(smem_u32(smem + kOffOnes), 0, 1024);
      bool ok = mbar_wait(&bar[kInFull], 0);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t aK = umma_desc_sw128(sK + (ks >> 2) * 16384 + (ks & 3) * 32, 0, 1024);
          const uint64_t bW = umma_desc_sw128(sW + ks * 2048, 16384, 1024);
          umma_bf16(tbase + kColU, aK, bW, idU, ks > 0 ? 1u : 0u);
        }
        umma_commit(&bar[kUFull]);
        ok = mbar_wait(&bar[kPhiFull], 0);
      }
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t aHi = umma_desc_sw128(sHi + ks * 2048, 4096, 1024);
          const uint64_t aLo = umma_desc_sw128(sLo + ks * 2048, 4096, 1024);
          const uint64_t bV = umma_desc_sw128(sV + ks * 2048, 4096, 1024);
          umma_bf16(tbase + kColS, aHi, bV, idS, ks > 0 ? 1u : 0u);
          umma_bf16(tbase + kColS, aLo, bV, idS, 1u);
          umma_bf16(tbase + kColZ, aHi, dOnes, idZ, ks > 0 ? 1u : 0u);
          umma_bf16(tbase + kColZ, aLo, dOnes, idZ, 1u);
        }
      }
      if (!ok) atomicOr(status, kStatusTimeout);
      umma_commit(&bar[kAccFull]);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;          // TMEM lane quarter of this warp
    const int tok = lane;               // token j of the block
    const uint32_t lane_bits = (uint32_t)(32 * quad) << 16;
    float* xmax = stats;
    float* xmin = stats + 128;
    float* xsp = stats + 256;
    float* xsm = stats + 384;
    bool ok = mbar_wait(&bar[kUFull], 0);
    tc_fence_after();
    float u[16];
    tmem_ld16(tbase + lane_bits + kColU + 16 * quad, u);
    tmem_wait_ld();
    float mx = -FLT_MAX, mn = FLT_MAX;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      mx = fmaxf(mx, u[i]);
      mn = fminf(mn, u[i]);
    }
    xmax[quad * 32 + tok] = mx;
    xmin[quad * 32 + tok] = mn;
    named_bar_sync(1, 128);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      mx = fmaxf(mx, xmax[q * 32 + tok]);
      mn = fminf(mn, xmin[q * 32 + tok]);
    }
    // e^{u - max} and e^{min - u} as one FMA and one ex2 each
    float ep[16], em[16], sp = 0.f, sm = 0.f;
    const float op = -mx * kLog2e, om = mn * kLog2e;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      ep[i] = ex2_approx(fmaf(u[i], kLog2e, op));
      em[i] = ex2_approx(fmaf(-u[i], kLog2e, om));
      sp += ep[i];
      sm += em[i];
    }
    xsp[quad * 32 + tok] = sp;
    xsm[quad * 32 + tok] = sm;
    named_bar_sync(1, 128);
    sp = xsp[tok] + xsp[32 + tok] + xsp[64 + tok] + xsp[96 + tok];
    sm = xsm[tok] + xsm[32 + tok] + xsm[64 + tok] + xsm[96 + tok];
    const float ip = rcp_approx(sp), im = rcp_approx(sm);  // sums >= 1 (max term e^0)
    // phi columns 16q..16q+15 of each half: two 16-byte chunks per atom row
    const uint32_t sHi = smem_u32(smem + kOffPhiHi), sLo = smem_u32(smem + kOffPhiLo);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const float* e = half ? em : ep;
      const float inv = half ? im : ip;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float p0 = e[8 * q + 2 * p] * inv, p1 = e[8 * q + 2 * p + 1] * inv;
          const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
          const float2 hf = __bfloat1622float2(hi);
          hw[p] = *reinterpret_cast<const uint32_t*>(&hi);
          lw[p] = pack_bf16(p0 - hf.x, p1 - hf.y);
        }
        const int chunk = 2 * quad + q;
        const uint32_t off = half * 4096 + tok * 128 + ((chunk ^ (tok & 7)) << 4);
        st_shared_v4(sHi + off, hw[0], hw[1], hw[2], hw[3]);
        st_shared_v4(sLo + off, lw[0], lw[1], lw[2], lw[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[kPhiFull]);

    // ---- final: row r = 32 quad + lane of Sacc (an F index) and Z_r
    ok = mbar_wait(&bar[kAccFull], 0) && ok;
    tc_fence_after();
    const int r = 32 * quad + lane;
    const uint32_t stage = smem_u32(smem + kOffStage);
#pragma unroll
    for (int part = 0; part < 4; ++part) {
      float v[32];
      tmem_ld32(tbase + lane_bits + kColS + 32 * part, v);
      tmem_wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        st_shared_v4(stage + s_off(r, 32 * part + 4 * q4), __float_as_uint(v[4 * q4]),
                     __float_as_uint(v[4 * q4 + 1]), __float_as_uint(v[4 * q4 + 2]),
                     __float_as_uint(v[4 * q4 + 3]));
    }
    reinterpret_cast<float*>(smem + kOffZst)[r] = tmem_ld1(tbase + lane_bits + kColZ);
    tmem_wait_ld();
    tc_fence_before();
    fence_proxy_async_smem();
    const bool all_ok = epilogue_all(ok);
    if (threadIdx.x == 64) {
      if (all_ok) {
        const int row = (slot * H + h) * kF;
#pragma unroll
        for (int bx = 0; bx < 4; ++bx)
          tma_reduce_add_2d(&maps.S, 32 * bx, row, smem + kOffStage + bx * 16384);
        bulk_reduce_add_f32(Z_pool + (size_t)(slot * H + h) * kF, smem + kOffZst, kF * 4);
        bulk_commit();
        bulk_wait_read();
      } else {
        atomicOr(status, kStatusTimeout);
      }
    }
  }

  __syncwarp();  // warps whose lane 0 ran a role alone reach the barrier converged
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool commit_tc_fits(const Shape& s, int batch, int num_slots) {
  return batch <= 65535 && (int64_t)batch * kL < ((int64_t)1 << 31) &&
         (int64_t)num_slots * s.H * kF < ((int64_t)1 << 31);
}

cudaError_t launch_commit_tc(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                             const void* v, const void* W, float* S_pool, float* Z_pool,
                             int num_slots, unsigned* status, cudaStream_t st,
                             const int32_t* mask) {
  Maps maps;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)batch * kL};
    const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
    const uint32_t box[3] = {64, 1, kL};
    if (!encode_tmap(&maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, box,
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
  {
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)num_slots * s.H * kF};
    const uint64_t strides[1] = {kD * 4};
    const uint32_t box[2] = {32, 128};
    if (!encode_tmap(&maps.S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, S_pool, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_commit_tc), kSmemBytes);
  if (e != cudaSuccess) return e;
  k_commit_tc<<<dim3(s.H, batch), kThreads, kSmemBytes, st>>>(maps, s.H, num_slots, slot_idx,
                                                               mask, Z_pool, status);
  return cudaGetLastError();
}

}  // namespace hb
