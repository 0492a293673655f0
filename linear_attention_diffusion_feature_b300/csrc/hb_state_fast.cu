// State commit and prompt ingestion for the production shape (bf16,
// d = 128, f = 64, F = 128) on the 5th-generation tensor cores.
//
// Definitions (pith.science review of arXiv 2608.06628, "What carries the
// argument"; gist.science technical summary, state-compression bullet):
//   S += sum_t phi(k_t) v_t^T,  Z += sum_t phi(k_t),
//   phi(k) = [softmax(k W_h), softmax(-k W_h)].
// A prompt is committed context, so ingesting it is the same sum over all of
// its tokens; the sum does not depend on how the tokens are chunked.
//
// One CTA per (request, head, token split); it streams its tokens in chunks
// of RB rows (128 for prompts, 32 for a committed block):
//   warp 0   TMA producer of k (two-stage ring of two SWIZZLE_128B boxes of
//            64 columns), W_h once; a k stage is refilled as soon as
//            U = K W_h of the chunk it held is done;
//   warp 2   TMA producer of v (same ring shape), refilled once phi^T V of
//            its chunk is done;
//   warp 1   owns TMEM (512 columns) and issues tcgen05.mma from one thread:
//              U    [128 tok x 64]  = K W_h            (A K-major, B MN-major)
//              Sacc^T [128 d x 256] += V^T [phi_hi | phi_lo]  (A, B MN-major;
//                   V is read once for both halves of the split)
//            U is double-buffered, so the next chunk's K W_h overlaps the
//            epilogue of the current one, and phi^T V runs per half-chunk
//            (tokens 0-63, then 64-127) as soon as that half of phi is
//            written;
//   warps 3-18 epilogue: four threads share a token (one TMEM lane, 16 of
//            the 64 columns of u each), exchange row max, min and sums
//            through shared memory, take both softmaxes and write phi to
//            shared memory as a bf16 pair hi + lo (phi = hi + lo to ~2^-17
//            relative), so the fp32 state meets a 1e-4 bound although the
//            tensor cores take bf16 operands; v is exact in bf16. Z is summed
//            from the same fp32 phi values in registers and reduced across
//            threads once at the end.
// At the end the epilogue reads Sacc^T (thread = column d of S, adding the
// hi and lo halves) and the Z sums, stages the tile through swizzled shared
// memory as [F][d] and writes S/Z (or a partial sum for the fixed-order split
// reduction) with coalesced 16-byte stores.
#include <float.h>

#include "hb_fast.cuh"
#include "hb_ptx.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kFH = 64, kF = 128;
constexpr int kThreads = 96 + 512;  // k producer, MMA, v producer, 16 epilogue warps

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int kOffK = 0;            // 2 stages x 2 boxes x [128 rows][128 B]
constexpr int kOffV = 65536;        // same
constexpr int kOffW = 131072;       // [128 d rows][64 bf16]
constexpr int kOffPhiHi = 147456;   // 2 atoms (F 0-63, 64-127) x [128 tok][128 B]
constexpr int kOffPhiLo = 180224;
constexpr int kOffZq = 212992;      // [4 token quarters][128 F] fp32: Z partial sums
constexpr int kOffBar = 215040;
constexpr int kOffZOld = kOffBar + 256;  // [128] fp32: Z before this call (accumulating)
constexpr int kOffX = kOffZOld + 512;    // epilogue exchange: 4 x [4 sub][128 tok] fp32
constexpr int kSmemBytes = kOffX + 8192 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory over the sm_100 per-block limit");

// mbarrier slots
enum { kKFull0 = 0, kKFull1, kKEmpty0, kKEmpty1, kVFull0, kVFull1, kVEmpty0, kVEmpty1,
       kWFull, kUFull0, kUFull1, kUEmpty0,
       kUEmpty1, kPhiFullA, kPhiFullB, kPhiEmptyA, kPhiEmptyB, kAccFull, kOldFull, kNumBars };

// TMEM columns
constexpr uint32_t kTmemCols = 512;
// S^T (lane = d) as two accumulators side by side: columns 0-127 take the
// phi hi products, 128-255 the phi lo ones (summed when read out); U is
// double-buffered in 256-383
constexpr uint32_t kColS = 0, kColU = 256;

constexpr int kPartialFloats = kF * kD + kF;  // one partial state: S then Z

struct Maps {
  CUtensorMap k;  // [rows][H][d] bf16, box {64, 1, RB}
  CUtensorMap v;
  CUtensorMap W;  // [H*d][f] bf16, box {64, 128}
};

struct Args {
  int H, num_slots, RB, splits, accumulate;
  const uint8_t* k_bytes;  // k, v base addresses (L2 prefetch of whole token rows)
  const uint8_t* v_bytes;
  int64_t total_rows, max_len;
  const int32_t* slot_idx;
  const int64_t* cu;  // nullptr: request b owns rows [b*RB, b*RB + RB)
  float* S_pool;
  float* Z_pool;
  float* ws;          // partial sums when splits > 1
  unsigned* status;
};

__device__ __forceinline__ bool unit_range(const Args& a, int b, int64_t* row0, int64_t* cnt) {
  if (a.cu) {
    *row0 = a.cu[b];
    *cnt = a.cu[b + 1] - *row0;
  } else {
    *row0 = (int64_t)b * a.RB;
    *cnt = a.RB;
  }
  const int slot = a.slot_idx[b];
  return slot >= 0 && slot < a.num_slots && *cnt >= 0 && *cnt <= a.max_len && *row0 >= 0 &&
         *row0 + *cnt <= a.total_rows;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_state_tc(const __grid_constant__ Maps maps, const __grid_constant__ Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int64_t row0, cnt;
  if (!unit_range(a, b, &row0, &cnt)) {
    if (threadIdx.x == 0 && split == 0) atomicOr(a.status, kStatusBounds);
    return;
  }
  const int slot = a.slot_idx[b];
  const int RB = a.RB;
  const int64_t n_chunks = (cnt + RB - 1) / RB;
  const int64_t c_begin = n_chunks * split / a.splits;
  const int64_t c_end = n_chunks * (split + 1) / a.splits;
  const int n_my = (int)(c_end - c_begin);

  if (threadIdx.x == 0) {
    for (int j = 0; j < 2; ++j) {
      mbar_init(&bar[kKFull0 + j], 1);
      mbar_init(&bar[kKEmpty0 + j], 1);
      mbar_init(&bar[kVFull0 + j], 1);
      mbar_init(&bar[kVEmpty0 + j], 1);
    }
    mbar_init(&bar[kWFull], 1);
    mbar_init(&bar[kUFull0], 1);
    mbar_init(&bar[kUFull1], 1);
    mbar_init(&bar[kUEmpty0], 16);
    mbar_init(&bar[kUEmpty1], 16);
    mbar_init(&bar[kPhiFullA], 8);
    mbar_init(&bar[kPhiFullB], 8);
    mbar_init(&bar[kPhiEmptyA], 1);
    mbar_init(&bar[kPhiEmptyB], 1);
    mbar_init(&bar[kAccFull], 1);
    mbar_init(&bar[kOldFull], 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  grid_dep_launch();  // the split reduction may be scheduled as SMs free up
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  // Accumulating into S/Z (a commit, or a prefill with accumulate = 1 and
  // no split) needs the old state tile. A commit has exactly one chunk, so
  // the second stage of the k/v ring is free from the start: the old rows
  // 0-63 go to the k half, rows 64-127 to the v half, fetched now so the
  // copy overlaps the whole contraction. A prompt uses both stages, so its
  // old tile is only prefetched into L2 here and copied into the k region
  // once the last MMA has finished.
  const bool add_old = a.splits == 1 && a.accumulate != 0;
  const bool commit_shape = a.cu == nullptr;
  const size_t unit_off = (size_t)slot * a.H + h;
  const float* S_old = a.S_pool + unit_off * kF * kD;
  const float* Z_old = a.Z_pool + unit_off * kF;
  uint8_t* old_lo = smem + (commit_shape ? kOffK + 32768 : kOffK);
  uint8_t* old_hi = smem + (commit_shape ? kOffV + 32768 : kOffK + 32768);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && add_old) {
      if (commit_shape) {
        mbar_arrive_expect_tx(&bar[kOldFull], 2 * 32768 + 512);
        bulk_load(old_lo, S_old, 32768, &bar[kOldFull]);
        bulk_load(old_hi, S_old + 64 * kD, 32768, &bar[kOldFull]);
        bulk_load(smem + kOffZOld, Z_old, 512, &bar[kOldFull]);
      } else {
        prefetch_l2(S_old, kF * kD * 4);
        prefetch_l2(Z_old, kF * 4);
      }
    }
    if (lane == 0 && n_my > 0) {
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      mbar_arrive_expect_tx(&bar[kWFull], 16384);
      tma_load_2d(smem + kOffW, &maps.W, 0, h * kD, &bar[kWFull]);
      // k of chunk c is loaded as soon as U = K W_h of chunk c - 2 is done
      // (it is not needed after that). Chunk c + 3 is prefetched into L2 as
      // whole token rows: the H CTAs of a request each prefetch
      // a contiguous 1/H slice of the chunk's rows of all heads, so DRAM
      // sees long contiguous reads instead of 128-byte pieces at the row
      // stride, and every head's TMA load then hits L2.
      const int64_t row_bytes = (int64_t)a.H * kD * 2;
      const int64_t slice = (int64_t)RB * kD * 2;  // = chunk bytes / H
      auto l2_rows = [&](int c) {
        if (c >= n_my) return;
        const int64_t r0 = row0 + (c_begin + c) * RB;
        const int64_t r1 = r0 + RB < row0 + cnt ? r0 + RB : row0 + cnt;
        const int64_t lo = r0 * row_bytes + h * slice;
        const int64_t hi_lim = r1 * row_bytes;
        const int64_t hi = lo + slice < hi_lim ? lo + slice : hi_lim;
        if (hi <= lo) return;
        prefetch_l2(a.k_bytes + lo, (uint32_t)(hi - lo));
        prefetch_l2(a.v_bytes + lo, (uint32_t)(hi - lo));
      };
      for (int c = 0; c < n_my; ++c) {
        const int s = c & 1, use = c >> 1;
        if (use > 0 && !mbar_wait(&bar[kKEmpty0 + s], (use - 1) & 1)) {
          atomicOr(a.status, kStatusTimeout);
          break;
        }
        const int row = (int)(row0 + (c_begin + c) * RB);
        mbar_arrive_expect_tx(&bar[kKFull0 + s], 2 * RB * 128);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem + kOffK + s * 32768 + j * 16384, &maps.k, 64 * j, h, row,
                      &bar[kKFull0 + s]);
        // the prefetches start once chunks 0 and 1 are requested, so that
        // those are served first (measured 1-2 % faster than prefetching
        // chunks 0-2 before any load)
        if (c == 1) {
          l2_rows(2);
          l2_rows(3);
          l2_rows(4);
        } else if (c > 1) {
          l2_rows(c + 3);
        }
      }
    }
  } else if (warp == 2) {
    // ----------------------------------------------------- v producer
    // v of chunk c is loaded once phi^T V of chunk c - 2 has completed
    if (lane == 0 && n_my > 0) {
      for (int c = 0; c < n_my; ++c) {
        const int s = c & 1, use = c >> 1;
        if (use > 0 && !mbar_wait(&bar[kVEmpty0 + s], (use - 1) & 1)) {
          atomicOr(a.status, kStatusTimeout);
          break;
        }
        const int row = (int)(row0 + (c_begin + c) * RB);
        mbar_arrive_expect_tx(&bar[kVFull0 + s], 2 * RB * 128);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem + kOffV + s * 32768 + j * 16384, &maps.v, 64 * j, h, row,
                      &bar[kVFull0 + s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0 && n_my > 0) {
      constexpr uint32_t idU = umma_idesc_bf16(128, kFH, 0, 1);
      // S^T [d x (F hi | F lo)] += V^T [phi_hi | phi_lo]: V is read once per
      // step for both halves of the split (M = d = 128, N = 2F = 256)
      constexpr uint32_t idS = umma_idesc_bf16(128, 2 * kF, 1, 1);
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sW = smem_u32(smem + kOffW);
      const uint32_t sHi = smem_u32(smem + kOffPhiHi);
      static_assert(kOffPhiLo == kOffPhiHi + 32768, "phi lo follows phi hi: one N = 256 operand");
      bool ok = mbar_wait(&bar[kWFull], 0);
      // Sacc += phi^T V for chunk cc, tokens 0-63 (half 0, k16 steps 0-3) as
      // soon as their phi rows are written, then tokens 64-127, so the next
      // chunk's first half can be written while the second is multiplied.
      auto mma2 = [&](int cc) -> bool {
        const int64_t valid64 = cnt - (c_begin + cc) * RB;
        const int valid = valid64 < RB ? (int)valid64 : RB;
        const int ksteps = (valid + 15) >> 4;
        const uint32_t vb = sV + (cc & 1) * 32768;
        if (!mbar_wait(&bar[kVFull0 + (cc & 1)], (cc >> 1) & 1)) return false;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (!mbar_wait(&bar[kPhiFullA + half], cc & 1)) return false;
          tc_fence_after();
          const int ks_end = ksteps < 4 * (half + 1) ? ksteps : 4 * (half + 1);
          for (int ks = 4 * half; ks < ks_end; ++ks) {
            // A = V^T (MN-major, two 64-column boxes 16 KiB apart); B = phi
            // hi then lo (MN-major, four 64-column atoms 16 KiB apart: the lo
            // buffer follows the hi buffer)
            const uint64_t aV = umma_desc_sw128(vb + ks * 2048, 16384, 1024);
            const uint64_t bP = umma_desc_sw128(sHi + ks * 2048, 16384, 1024);
            umma_bf16(tbase + kColS, aV, bP, idS, (cc == 0 && ks == 0) ? 0u : 1u);
          }
          umma_commit(&bar[kPhiEmptyA + half]);
        }
        umma_commit(&bar[kVEmpty0 + (cc & 1)]);
        return true;
      };
      for (int c = 0; ok && c < n_my; ++c) {
        const int s = c & 1;
        if (!mbar_wait(&bar[kKFull0 + s], (c >> 1) & 1)) { ok = false; break; }
        if (c >= 2 && !mbar_wait(&bar[kUEmpty0 + s], ((c >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = sK + s * 32768;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t aK = umma_desc_sw128(kb + (ks >> 2) * 16384 + (ks & 3) * 32, 0, 1024);
          const uint64_t bW = umma_desc_sw128(sW + ks * 2048, 16384, 1024);
          umma_bf16(tbase + kColU + 64 * s, aK, bW, idU, ks > 0 ? 1u : 0u);
        }
        umma_commit(&bar[kUFull0 + s]);
        umma_commit(&bar[kKEmpty0 + s]);
        if (c >= 1 && !mma2(c - 1)) { ok = false; break; }
      }
      if (ok) ok = mma2(n_my - 1);
      if (!ok) atomicOr(a.status, kStatusTimeout);
      umma_commit(&bar[kAccFull]);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // 16 warps. Warp w (3..18) reads TMEM lane quarter q = w % 4 (tokens
    // 32q .. 32q + 31 of a chunk) and column slice sub = (w - 3) / 4 (16 of
    // the 64 columns of u), so each token's two softmaxes are shared by four
    // threads that exchange row max, min and sums through shared memory.
    const int quad = warp & 3;
    const int ew = warp - 3;               // 0..15
    const int sub = ew >> 2;
    const int tok = 32 * quad + lane;      // TMEM lane = token row (chunks) = F row (final)
    const uint32_t lane_bits = (uint32_t)(32 * quad) << 16;
    const uint32_t sHi = smem_u32(smem + kOffPhiHi), sLo = smem_u32(smem + kOffPhiLo);
    float* xmax = reinterpret_cast<float*>(smem + kOffX);  // [4 sub][128 tok]
    float* xmin = xmax + 512;
    float* xsp = xmin + 512;
    float* xsm = xsp + 512;
    // Tokens 0-63 (quarters 0, 1) and 64-127 (quarters 2, 3) form two
    // independent halves with their own named barrier and phi barriers.
    const int half_id = quad >> 1;
    const int hbar = 1 + half_id;
    // Z = sum_t phi(k_t): this thread's 32 columns of phi summed over every
    // chunk it saw (same token row each time), reduced across threads at the end
    float zacc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) zacc[j] = 0.f;
    // A wait that runs out marks `ok` false for good; the threads still go
    // through every named barrier, and the vote at the first barrier of the
    // next chunk (or of the final phase) makes all of them leave together.
    bool ok = true;
    for (int c = 0; c < n_my; ++c) {
      const int s = c & 1;
      if (ok) ok = mbar_wait(&bar[kUFull0 + s], (c >> 1) & 1);
      tc_fence_after();
      float u[16];
      tmem_ld16(tbase + lane_bits + kColU + 64 * s + 16 * sub, u);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kUEmpty0 + s]);

      const int64_t valid64 = cnt - (c_begin + c) * RB;
      const int valid = valid64 < RB ? (int)valid64 : RB;
      const bool live = tok < valid;
      // Rows at or past the end of the last 16-token MMA step are never read
      // by the phi^T V contraction, so their threads skip the softmaxes.
      const bool used = tok < ((valid + 15) & ~15);
      float mx = -FLT_MAX, mn = FLT_MAX;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        mx = fmaxf(mx, u[j]);
        mn = fminf(mn, u[j]);
      }
      xmax[sub * 128 + tok] = mx;
      xmin[sub * 128 + tok] = mn;
      if (named_bar_any(hbar, 256, !ok)) break;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mx = fmaxf(mx, xmax[q * 128 + tok]);
        mn = fminf(mn, xmin[q * 128 + tok]);
      }
      // e^{u - max} as one packed FMA and one ex2 each. The other half uses
      // e^{min - u} = C / e^{u - max} with C = e^{min - max}: a reciprocal on
      // the FMA pipe instead of a second ex2, which halves the work of the
      // special-function unit. That identity needs e^{u - max} to stay a
      // normal float, so tokens whose u spans more than 60 use ex2 directly.
      float ep[16], em[16];
      float2 spp = make_float2(0.f, 0.f), smp = make_float2(0.f, 0.f);
      {
        const float2 l2e = make_float2(kLog2e, kLog2e);
        const float2 op = make_float2(-mx * kLog2e, -mx * kLog2e);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 x = fma2(make_float2(u[j], u[j + 1]), l2e, op);
          ep[j] = ex2_approx(x.x);
          ep[j + 1] = ex2_approx(x.y);
          spp = add2(spp, make_float2(ep[j], ep[j + 1]));
        }
        if (mx - mn <= 60.f) {
          const float C = ex2_approx((mn - mx) * kLog2e);
          const float2 C2 = make_float2(C, C);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float2 r = mul2(C2, rcp2_newton(make_float2(ep[j], ep[j + 1])));
            em[j] = r.x;
            em[j + 1] = r.y;
            smp = add2(smp, r);
          }
        } else {
          const float om = mn * kLog2e;
#pragma unroll
          for (int j = 0; j < 16; ++j) em[j] = ex2_approx(fmaf(-u[j], kLog2e, om));
#pragma unroll
          for (int j = 0; j < 16; j += 2) smp = add2(smp, make_float2(em[j], em[j + 1]));
        }
      }
      float sp = spp.x + spp.y, sm = smp.x + smp.y;
      xsp[sub * 128 + tok] = sp;
      xsm[sub * 128 + tok] = sm;
      named_bar_sync(hbar, 256);
      sp = (xsp[tok] + xsp[128 + tok]) + (xsp[256 + tok] + xsp[384 + tok]);
      sm = (xsm[tok] + xsm[128 + tok]) + (xsm[256 + tok] + xsm[384 + tok]);
      // (sp, sm >= 1: each sum holds its row maximum term e^0)
      const float ip = live ? rcp_approx(sp) : 0.f, im = live ? rcp_approx(sm) : 0.f;
      if (ok && c >= 1) ok = mbar_wait(&bar[kPhiEmptyA + half_id], (c - 1) & 1);
      if (used) {
        // phi columns 16 sub .. 16 sub + 15 of each half: two 16-byte chunks
        // per atom row; dead rows (live == false) are written as exact zeros
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float* e = half ? em : ep;
          const float2 inv = half ? make_float2(im, im) : make_float2(ip, ip);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const int j = 8 * q + 2 * p;
              const float2 pv = mul2(make_float2(e[j], e[j + 1]), inv);
              const float2 z = add2(make_float2(zacc[16 * half + j], zacc[16 * half + j + 1]), pv);
              zacc[16 * half + j] = z.x;
              zacc[16 * half + j + 1] = z.y;
              const __nv_bfloat162 hi = __floats2bfloat162_rn(pv.x, pv.y);
              const float2 hf = __bfloat1622float2(hi);
              hw[p] = *reinterpret_cast<const uint32_t*>(&hi);
              const float2 lo = add2(pv, make_float2(-hf.x, -hf.y));
              lw[p] = pack_bf16(lo.x, lo.y);
            }
            const int chunk = 2 * sub + q;
            const uint32_t off = half * 16384 + tok * 128 + ((chunk ^ (tok & 7)) << 4);
            st_shared_v4(sHi + off, hw[0], hw[1], hw[2], hw[3]);
            st_shared_v4(sLo + off, lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      if (used && !live) {
        // Rows past the end of the request inside the last 16-token step:
        // their phi is 0; clear v there too (chunks 2 sub, 2 sub + 1 of both
        // boxes) so foreign or fill rows cannot inject a non-finite value.
        if (ok) ok = mbar_wait(&bar[kVFull0 + s], (c >> 1) & 1);
        const uint32_t vrow = smem_u32(smem + kOffV + s * 32768) + tok * 128;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          st_shared_v4(vrow + (2 * sub + q) * 16, 0u, 0u, 0u, 0u);
          st_shared_v4(vrow + 16384 + (2 * sub + q) * 16, 0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kPhiFullA + half_id]);
    }

    // ---- final: rows 32 quad + lane of S (an F index), columns 32 sub ..
    // 32 sub + 31, and Z, staged for coalesced stores
    bool have = ok;
    if (have && n_my > 0) have = mbar_wait(&bar[kAccFull], 0);
    have = __all_sync(0xffffffffu, have);  // warp-uniform for the TMEM loads
    tc_fence_after();
    if (add_old && !commit_shape && threadIdx.x == 96) {
      // every MMA and TMA load has completed (kAccFull), so the k region is free
      mbar_arrive_expect_tx(&bar[kOldFull], 2 * 32768 + 512);
      bulk_load(old_lo, S_old, 32768, &bar[kOldFull]);
      bulk_load(old_hi, S_old + 64 * kD, 32768, &bar[kOldFull]);
      bulk_load(smem + kOffZOld, Z_old, 512, &bar[kOldFull]);
    }
    const uint32_t stage = smem_u32(smem + kOffPhiHi);  // 64 KiB, free once the MMAs are done
    {
      // The accumulator is S^T: lane = d (= tok here), columns F of the hi
      // half then of the lo half. This thread holds S[f][d] for its d and
      // f = 32 sub .. 32 sub + 31, the sum of the two halves, and writes it
      // into row f of the staged [F][d] tile (a warp's 32 d of one row are
      // 8 distinct 16-byte chunks: no bank conflict).
      const int dcol = tok;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float rh[16], rl[16];
        if (have && n_my > 0) {
          tmem_ld16(tbase + lane_bits + kColS + 32 * sub + 16 * hh, rh);
          tmem_ld16(tbase + lane_bits + kColS + kF + 32 * sub + 16 * hh, rl);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) rh[j] = rl[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int f = 32 * sub + 16 * hh + j;
          st_shared_u32(stage + f * 512 + ((((dcol >> 2) ^ (f & 31)) << 4) | ((dcol & 3) << 2)),
                        __float_as_uint(rh[j] + rl[j]));
        }
      }
    }
    // Z: reduce-scatter the 32 column sums across the warp's lanes (lane j
    // ends with column j of its slice), then add the four token quarters.
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < o; ++j) {
        const float send = upper ? zacc[j] : zacc[j + o];
        const float keep = upper ? zacc[j + o] : zacc[j];
        zacc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    float* zq = reinterpret_cast<float*>(smem + kOffZq);  // [4 quarters][128 F]
    {
      const int F = lane < 16 ? 16 * sub + lane : kFH + 16 * sub + (lane - 16);
      zq[quad * 128 + F] = zacc[0];
    }
    named_bar_sync(3, 512);
    float z = 0.f;
    if (sub == 0) z = (zq[tok] + zq[128 + tok]) + (zq[256 + tok] + zq[384 + tok]);
    tc_fence_before();
    bool have_old = true;
    if (add_old && have) have_old = mbar_wait(&bar[kOldFull], 0);
    const bool failed = named_bar_any(3, 512, !(have && have_old));
    if (failed) {
      if (threadIdx.x == 96) atomicOr(a.status, kStatusTimeout);
    } else {
      float* Sdst;
      float* Zdst;
      if (a.splits > 1) {
        float* p = a.ws + ((size_t)(b * a.H + h) * a.splits + split) * kPartialFloats;
        Sdst = p;
        Zdst = p + kF * kD;
      } else {
        Sdst = a.S_pool + unit_off * kF * kD;
        Zdst = a.Z_pool + unit_off * kF;
      }
      const uint32_t olo = smem_u32(old_lo), ohi = smem_u32(old_hi);
#pragma unroll 4
      for (int r = ew; r < kF; r += 16) {
        float4 v = ld_shared_v4f(stage + r * 512 + ((lane ^ (r & 31)) << 4));
        if (add_old) {
          const float4 o = ld_shared_v4f((r < 64 ? olo + r * 512 : ohi + (r - 64) * 512) + lane * 16);
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        reinterpret_cast<float4*>(Sdst + r * kD)[lane] = v;
      }
      if (sub == 0) {
        const float* zold = reinterpret_cast<const float*>(smem + kOffZOld);
        Zdst[tok] = add_old ? zold[tok] + z : z;
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

// Sums the split partials of each unit in split order and writes S/Z.
// Block (h, b, z) takes elements z * 256 + t, stepping by 256 * gridDim.z,
// so a few units still spread over many SMs. Launched as a programmatic
// dependent of k_state_tc: it waits for that grid before reading anything.
__global__ void __launch_bounds__(256) k_state_reduce(const __grid_constant__ Args a) {
  grid_dep_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  int64_t row0, cnt;
  if (!unit_range(a, b, &row0, &cnt)) return;  // flagged by k_state_tc
  const int slot = a.slot_idx[b];
  const float4* part =
      reinterpret_cast<const float4*>(a.ws + (size_t)(b * a.H + h) * a.splits * kPartialFloats);
  const size_t unit = (size_t)slot * a.H + h;
  float4* S = reinterpret_cast<float4*>(a.S_pool + unit * kF * kD);
  float4* Z = reinterpret_cast<float4*>(a.Z_pool + unit * kF);
  constexpr int n4 = kPartialFloats / 4;
  for (int i = blockIdx.z * blockDim.x + threadIdx.x; i < n4; i += blockDim.x * gridDim.z) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = 0; j < a.splits; ++j) {
      const float4 p = part[(size_t)j * n4 + i];
      acc.x += p.x;
      acc.y += p.y;
      acc.z += p.z;
      acc.w += p.w;
    }
    float4* dst = i < kF * kD / 4 ? S + i : Z + (i - kF * kD / 4);
    if (a.accumulate) {
      const float4 o = *dst;
      acc.x += o.x;
      acc.y += o.y;
      acc.z += o.z;
      acc.w += o.w;
    }
    *dst = acc;
  }
}

// Splits per (request, head) so that the grid fills the current device's
// SMs about once (one CTA per SM); the workspace size query and the launch
// both call this on the current device, so they agree.
int splits_for(int batch, int H, int64_t max_seqlen) {
  const int64_t units = (int64_t)batch * H;
  const int64_t chunks = (max_seqlen + 127) / 128;
  int sms = 0;
  if (current_sm_count(&sms) != cudaSuccess || sms <= 0) sms = 148;
  int64_t s = sms / (units > 0 ? units : 1);
  if (s > chunks) s = chunks;
  if (s > 64) s = 64;
  return s < 1 ? 1 : (int)s;
}

cudaError_t launch_tc(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                      const void* v, int64_t total_rows, const int64_t* cu, int64_t max_len,
                      int RB, int splits, const void* W, float* S_pool, float* Z_pool,
                      int num_slots, int accumulate, float* ws, unsigned* status,
                      cudaStream_t st) {
  Maps maps;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)total_rows};
    const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)RB};
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
  Args a;
  a.H = s.H;
  a.k_bytes = static_cast<const uint8_t*>(k);
  a.v_bytes = static_cast<const uint8_t*>(v);
  a.num_slots = num_slots;
  a.RB = RB;
  a.splits = splits;
  a.accumulate = accumulate;
  a.total_rows = total_rows;
  a.max_len = max_len;
  a.slot_idx = slot_idx;
  a.cu = cu;
  a.S_pool = S_pool;
  a.Z_pool = Z_pool;
  a.ws = ws;
  a.status = status;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_state_tc), kSmemBytes);
  if (e != cudaSuccess) return e;
  k_state_tc<<<dim3(splits, s.H, batch), kThreads, kSmemBytes, st>>>(maps, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (splits > 1) {
    // enough blocks per unit that the reduction runs on every SM
    const int64_t units = (int64_t)batch * s.H;
    int z = (int)((4 * 148 + units - 1) / units);
    z = z < 1 ? 1 : (z > 16 ? 16 : z);
    e = launch_pdl(k_state_reduce, dim3(s.H, batch, z), dim3(256), 0, st, a);
  }
  return e;
}

}  // namespace

bool fast_state_ok(const Shape& s) { return production_shape(s); }

cudaError_t launch_commit_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                               const void* v, const void* W, float* S_pool, float* Z_pool,
                               int num_slots, unsigned* status, cudaStream_t st) {
  if (commit_tc_fits(s, batch, num_slots))
    return launch_commit_tc(s, batch, slot_idx, k, v, W, S_pool, Z_pool, num_slots, status, st);
  const int64_t rows = (int64_t)batch * s.L;
  if (rows >= (int64_t)1 << 31 || batch > 65535)
    return launch_state_accumulate_generic(s, batch, slot_idx, k, v, rows, nullptr, s.L, W,
                                           S_pool, Z_pool, num_slots, 1, status, st);
  return launch_tc(s, batch, slot_idx, k, v, rows, nullptr, s.L, s.L, 1, W, S_pool, Z_pool,
                   num_slots, 1, nullptr, status, st);
}

size_t prefill_fast_workspace_bytes(const Shape& s, int batch, int64_t max_seqlen) {
  const int sp = splits_for(batch, s.H, max_seqlen);
  return sp > 1 ? (size_t)batch * s.H * sp * kPartialFloats * sizeof(float) : 0;
}

cudaError_t launch_prefill_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* k,
                                const void* v, int64_t total_tokens, const int64_t* cu_seqlens,
                                int64_t max_seqlen, const void* W, float* S_pool, float* Z_pool,
                                int num_slots, int accumulate, void* workspace, unsigned* status,
                                cudaStream_t st) {
  if (total_tokens == 0 || total_tokens >= (int64_t)1 << 31 || batch > 65535)
    return launch_state_accumulate_generic(s, batch, slot_idx, k, v, total_tokens, cu_seqlens,
                                           max_seqlen, W, S_pool, Z_pool, num_slots, accumulate,
                                           status, st);
  const int sp = splits_for(batch, s.H, max_seqlen);
  return launch_tc(s, batch, slot_idx, k, v, total_tokens, cu_seqlens, max_seqlen, 128, sp, W,
                   S_pool, Z_pool, num_slots, accumulate, static_cast<float*>(workspace), status,
                   st);
}

}  // namespace hb
