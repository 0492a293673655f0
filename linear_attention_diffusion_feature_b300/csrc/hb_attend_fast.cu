// Block-hybrid attend for the production shape (bf16, d = 128, f = 64,
// F = 128, L = 32): gist.science technical summary of arXiv 2608.06628,
// "Methodology: Block-Hybrid Attention / Architecture Design" (exact softmax
// inside the active block, Hedgehog linear read of the fixed-size state S, Z
// for committed blocks, gated merge with a shared normaliser); pith.science
// review, "What carries the argument" (the cross-block read is O(Fd) per
// query) and its comment on the Section 3.1 out(q) equation (the gate scales
// only the softmax numerator and denominator).
//
// The step is bound by the HBM read of S (64 KiB fp32 per request and head,
// 2/3 of the bytes), so the kernel is a persistent streaming pipeline:
//   * one CTA per SM, 9 warps: warp 8 is the producer, warps 0-7 compute;
//   * a two-stage shared-memory ring; each stage holds one (request, head)
//     unit: S (four 16 KiB SWIZZLE_128B TMA boxes), q, k, v (two 4 KiB boxes
//     each), W_h (16 KiB) and Z (512 B bulk copy), all arriving on one
//     mbarrier;
//   * the producer issues unit i+1's loads while the consumers compute
//     unit i; consumers release a stage through a second mbarrier;
//   * all four contractions (qW, qk^T, phi(q)S, PV) run on bf16 mma.sync with
//     fp32 accumulation; S is converted fp32 -> bf16 pairs as it is read
//     from shared memory (the swizzle makes those reads conflict-free);
//   * both softmaxes of phi and the block softmax use fp32 expf; the merge
//     is the overflow-free rescaled form in merge_out().
#include <float.h>

#include "hb_fast.cuh"
#include "hb_ptx.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kFH = 64, kF = 128, kL = 32;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;

// Stage layout (bytes from the stage base; the base is 1024-aligned).
constexpr int kOffS = 0;                    // 4 x [128 F-rows][32 fp32], SW128
constexpr int kOffQ = 65536;                // 2 x [32 tokens][64 bf16], SW128
constexpr int kOffK = kOffQ + 8192;
constexpr int kOffV = kOffK + 8192;
constexpr int kOffW = kOffV + 8192;         // [128 d-rows][64 bf16], SW128
constexpr int kOffZ = kOffW + 16384;        // [128] fp32
constexpr int kTxBytes = kOffZ + 512;       // every byte of a stage comes by TMA
constexpr int kStageStride = 107520;        // 105 KiB
// Shared buffers of the consumers.
constexpr int kOffPhi = 2 * kStageStride;   // 2 x [32][64 bf16], SW128 (phi(q) as bf16)
constexpr int kOffP = kOffPhi + 8192;       // [32][40 bf16]: e^{s - m}, 80-byte rows
constexpr int kPitchP = 80;
constexpr int kOffStats = kOffP + 32 * kPitchP;
// stats (floats): 8 partial arrays [32 rows][4 quarters], then 3 finals [32]
enum { kPMax = 0, kPMin, kSMax, kSumP, kSumM, kDenP, kDenM, kSumS, kNumPart };
constexpr int kOffFin = kOffStats + kNumPart * 32 * 4 * 4;
constexpr int kOffBar = kOffFin + 3 * 32 * 4;
constexpr int kOffMeta = kOffBar + 4 * 8;
constexpr int kSmemUsed = kOffMeta + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base to 1024
static_assert(kTxBytes <= kStageStride, "stage overflow");
static_assert(kSmemBytes <= 232448, "shared memory over the sm_100 per-block limit");

struct Maps {
  CUtensorMap S;  // [slots*H*F rows][d] fp32, box {32, 128}
  CUtensorMap q;  // [B*L][H][d] bf16, box {64, 1, 32}
  CUtensorMap k;
  CUtensorMap v;
  CUtensorMap W;  // [H*d rows][f] bf16, box {64, 128}
};

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a
// [rows][128 B] SWIZZLE_128B box.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// Byte offset of S[k][n] (fp32) in the four SW128 boxes of the stage.
__device__ __forceinline__ uint32_t s_off(int k, int n) {
  return (uint32_t)((n >> 5) * 16384 + k * 128 + ((((n & 31) >> 2) ^ (k & 7)) << 4) + (n & 3) * 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attend_fast(const __grid_constant__ Maps maps, int batch, int H, int num_slots, float scale,
                  int merge, const int32_t* __restrict__ slot_idx,
                  const float* __restrict__ S_pool, const float* __restrict__ Z_pool,
                  const float* __restrict__ gate,
                  __nv_bfloat16* __restrict__ o, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + 2;
  int* meta = reinterpret_cast<int*>(smem + kOffMeta);
  float* stats = reinterpret_cast<float*>(smem + kOffStats);
  float* fin = reinterpret_cast<float*>(smem + kOffFin);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = batch * H;

  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], kConsumerWarps);
    mbar_init(&empty[1], kConsumerWarps);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; lane 0 issues the copies. Slot indices
    // are read 32 units at a time (lane j holds the slot of local unit
    // 32w + j), and each unit's tiles are prefetched into L2 two units
    // before their TMA load is issued, so that more than one unit per SM is
    // in flight from DRAM while the consumers work.
    if (lane == 0) {
      prefetch_tmap(&maps.S);
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      prefetch_tmap(&maps.W);
    }
    const int first = blockIdx.x, stride = gridDim.x;
    const int n_local = first < units ? (units - first + stride - 1) / stride : 0;
    int win = -1, win_slot = -1;
    auto slot_of = [&](int i) -> int {  // warp-uniform i, called in increasing order
      if ((i >> 5) != win) {
        win = i >> 5;
        const int uu = first + (32 * win + lane) * stride;
        win_slot = uu < units ? slot_idx[uu / H] : -1;
      }
      return __shfl_sync(0xffffffffu, win_slot, i & 31);
    };
    auto l2_prefetch = [&](int i, int slot) {
      const int uu = first + i * stride;
      const int b = uu / H, h = uu - b * H;
      if (lane != 0 || slot < 0 || slot >= num_slots) return;
      const size_t unit = (size_t)slot * H + h;
      prefetch_l2(S_pool + unit * kF * kD, kF * kD * 4);
      prefetch_l2(Z_pool + unit * kF, kF * 4);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        prefetch_l2_3d(&maps.q, 64 * j, h, b * kL);
        prefetch_l2_3d(&maps.k, 64 * j, h, b * kL);
        prefetch_l2_3d(&maps.v, 64 * j, h, b * kL);
      }
    };
    int slot_cur = n_local > 0 ? slot_of(0) : -1;
    int slot_next = n_local > 1 ? slot_of(1) : -1;
    if (n_local > 1) l2_prefetch(1, slot_next);
    for (int i = 0; i < n_local; ++i) {
      const int s = i & 1, n = i >> 1;
      bool ok = true;
      if (lane == 0 && n > 0) ok = mbar_wait(&empty[s], (n - 1) & 1);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        break;
      }
      const int u = first + i * stride;
      const int b = u / H, h = u - b * H;
      const int slot = slot_cur;
      if (lane == 0) {
        uint8_t* st = smem + s * kStageStride;
        if (slot < 0 || slot >= num_slots) {
          atomicOr(status, kStatusBounds);
          meta[s] = 0;
          mbar_arrive(&full[s]);
        } else {
          meta[s] = 1;
          mbar_arrive_expect_tx(&full[s], kTxBytes);
          const int srow = (slot * H + h) * kF;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_load_2d(st + kOffS + j * 16384, &maps.S, 32 * j, srow, &full[s]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            tma_load_3d(st + kOffQ + j * 4096, &maps.q, 64 * j, h, b * kL, &full[s]);
            tma_load_3d(st + kOffK + j * 4096, &maps.k, 64 * j, h, b * kL, &full[s]);
            tma_load_3d(st + kOffV + j * 4096, &maps.v, 64 * j, h, b * kL, &full[s]);
          }
          tma_load_2d(st + kOffW, &maps.W, 0, h * kD, &full[s]);
          bulk_load(st + kOffZ, Z_pool + (size_t)(slot * H + h) * kF, 512, &full[s]);
        }
      }
      const int ahead = i + 2;
      const int slot_ahead = ahead < n_local ? slot_of(ahead) : -1;
      if (ahead < n_local) l2_prefetch(ahead, slot_ahead);
      slot_cur = slot_next;
      slot_next = slot_ahead;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const uint32_t sPhi = smem_u32(smem + kOffPhi);
  const uint32_t sP = smem_u32(smem + kOffP);
  auto part = [&](int which, int row, int quarter) -> float& {
    return stats[(which * 32 + row) * 4 + quarter];
  };

  int i = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
    const int s = i & 1, n = i >> 1;
    // the gate is read before the wait so its latency hides behind it
    const float gl = gate[u % H];
    if (!mbar_wait(&full[s], n & 1)) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      break;
    }
    if (meta[s]) {
      uint8_t* st = smem + s * kStageStride;
      const uint32_t sS = smem_u32(st + kOffS);
      const uint32_t sQ = smem_u32(st + kOffQ);
      const uint32_t sK = smem_u32(st + kOffK);
      const uint32_t sV = smem_u32(st + kOffV);
      const uint32_t sW = smem_u32(st + kOffW);
      const float* sZ = reinterpret_cast<const float*>(st + kOffZ);
      const int b = u / H, h = u - b * H;

      // ---- phase A: u = q W_h (16 rows x 16 cols per warp) and
      //      s = q k^T (16 rows x 8 keys per warp)
      const int mt = warp & 1, nq = warp >> 1;
      float acc_u[2][4] = {}, acc_s[4] = {};
      {
        const int arow = 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
          uint32_t a0[4], a1[4];
          {
            const int ch = 2 * kk + (lane >> 4);
            ldsm_x4(sQ + (ch >> 3) * 4096 + sw128(arow, ch & 7), a0[0], a0[1], a0[2], a0[3]);
            const int ch1 = ch + 2;
            ldsm_x4(sQ + (ch1 >> 3) * 4096 + sw128(arow, ch1 & 7), a1[0], a1[1], a1[2], a1[3]);
          }
          // k^T fragments for keys 8nq..8nq+7, two k16 steps at once
          uint32_t kb[4];
          {
            const int krow = 8 * nq + (lane & 7);
            const int ch = 2 * kk + (lane >> 3);
            ldsm_x4(sK + (ch >> 3) * 4096 + sw128(krow, ch & 7), kb[0], kb[1], kb[2], kb[3]);
          }
          mma_bf16(acc_s, a0, kb[0], kb[1]);
          mma_bf16(acc_s, a1, kb[2], kb[3]);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int k16 = kk + half;
            uint32_t wb[4];
            const int mtx = lane >> 3;
            const int krow = 16 * k16 + (mtx & 1) * 8 + (lane & 7);
            const int nch = 2 * nq + (mtx >> 1);
            ldsm_x4_t(sW + sw128(krow, nch), wb[0], wb[1], wb[2], wb[3]);
            mma_bf16(acc_u[0], half ? a1 : a0, wb[0], wb[1]);
            mma_bf16(acc_u[1], half ? a1 : a0, wb[2], wb[3]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) acc_s[r] *= scale;  // scale * log2(e): scores in base 2
      const int R0 = 16 * mt + g, R1 = R0 + 8;
      {
        float mx0 = fmaxf(fmaxf(acc_u[0][0], acc_u[0][1]), fmaxf(acc_u[1][0], acc_u[1][1]));
        float mx1 = fmaxf(fmaxf(acc_u[0][2], acc_u[0][3]), fmaxf(acc_u[1][2], acc_u[1][3]));
        float mn0 = fminf(fminf(acc_u[0][0], acc_u[0][1]), fminf(acc_u[1][0], acc_u[1][1]));
        float mn1 = fminf(fminf(acc_u[0][2], acc_u[0][3]), fminf(acc_u[1][2], acc_u[1][3]));
        float sm0 = fmaxf(acc_s[0], acc_s[1]), sm1 = fmaxf(acc_s[2], acc_s[3]);
#pragma unroll
        for (int o2 = 1; o2 < 4; o2 <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
          mn0 = fminf(mn0, __shfl_xor_sync(0xffffffffu, mn0, o2));
          mn1 = fminf(mn1, __shfl_xor_sync(0xffffffffu, mn1, o2));
          sm0 = fmaxf(sm0, __shfl_xor_sync(0xffffffffu, sm0, o2));
          sm1 = fmaxf(sm1, __shfl_xor_sync(0xffffffffu, sm1, o2));
        }
        if (t == 0) {
          part(kPMax, R0, nq) = mx0;
          part(kPMax, R1, nq) = mx1;
          part(kPMin, R0, nq) = mn0;
          part(kPMin, R1, nq) = mn1;
          part(kSMax, R0, nq) = sm0;
          part(kSMax, R1, nq) = sm1;
        }
      }
      named_bar_sync(1, kConsumers);

      // ---- phase B: exponentials, partial sums, partial phi^T Z, P = e^{s-m}
      float ep[2][4], em[2][4];
      {
        float Mp[2], Mm[2], Ms[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int R = hr ? R1 : R0;
          Mp[hr] = fmaxf(fmaxf(part(kPMax, R, 0), part(kPMax, R, 1)),
                         fmaxf(part(kPMax, R, 2), part(kPMax, R, 3)));
          Mm[hr] = -fminf(fminf(part(kPMin, R, 0), part(kPMin, R, 1)),
                          fminf(part(kPMin, R, 2), part(kPMin, R, 3)));
          Ms[hr] = fmaxf(fmaxf(part(kSMax, R, 0), part(kSMax, R, 1)),
                         fmaxf(part(kSMax, R, 2), part(kSMax, R, 3)));
        }
        float sp[2] = {0.f, 0.f}, sm[2] = {0.f, 0.f}, dp[2] = {0.f, 0.f}, dm[2] = {0.f, 0.f};
        // e^{x - M} = 2^{x log2(e) - M log2(e)}: one FMA and one ex2 each
        const float op[2] = {-Mp[0] * kLog2e, -Mp[1] * kLog2e};
        const float om[2] = {-Mm[0] * kLog2e, -Mm[1] * kLog2e};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int hr = r >> 1;
            const int c = 16 * nq + 8 * nt + 2 * t + (r & 1);
            const float x = acc_u[nt][r];
            const float e1 = ex2_approx(fmaf(x, kLog2e, op[hr]));
            const float e2 = ex2_approx(fmaf(-x, kLog2e, om[hr]));
            ep[nt][r] = e1;
            em[nt][r] = e2;
            sp[hr] += e1;
            sm[hr] += e2;
            dp[hr] = fmaf(e1, sZ[c], dp[hr]);
            dm[hr] = fmaf(e2, sZ[kFH + c], dm[hr]);
          }
        }
        float p[4], ss[2];
#pragma unroll
        for (int r = 0; r < 4; ++r) p[r] = ex2_approx(acc_s[r] - Ms[r >> 1]);
        ss[0] = p[0] + p[1];
        ss[1] = p[2] + p[3];
#pragma unroll
        for (int o2 = 1; o2 < 4; o2 <<= 1) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            sp[hr] += __shfl_xor_sync(0xffffffffu, sp[hr], o2);
            sm[hr] += __shfl_xor_sync(0xffffffffu, sm[hr], o2);
            dp[hr] += __shfl_xor_sync(0xffffffffu, dp[hr], o2);
            dm[hr] += __shfl_xor_sync(0xffffffffu, dm[hr], o2);
            ss[hr] += __shfl_xor_sync(0xffffffffu, ss[hr], o2);
          }
        }
        if (t == 0) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int R = hr ? R1 : R0;
            part(kSumP, R, nq) = sp[hr];
            part(kSumM, R, nq) = sm[hr];
            part(kDenP, R, nq) = dp[hr];
            part(kDenM, R, nq) = dm[hr];
            part(kSumS, R, nq) = ss[hr];
          }
        }
        const int key = 8 * nq + 2 * t;
        st_shared_u32(sP + R0 * kPitchP + key * 2, pack_bf16(p[0], p[1]));
        st_shared_u32(sP + R1 * kPitchP + key * 2, pack_bf16(p[2], p[3]));
      }
      named_bar_sync(1, kConsumers);

      // ---- phase C: phi(q) = e / sum -> bf16 in shared memory; row finals
      {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int R = hr ? R1 : R0;
          const float ip = 1.f / (part(kSumP, R, 0) + part(kSumP, R, 1) + part(kSumP, R, 2) +
                                  part(kSumP, R, 3));
          const float im = 1.f / (part(kSumM, R, 0) + part(kSumM, R, 1) + part(kSumM, R, 2) +
                                  part(kSumM, R, 3));
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int c = 16 * nq + 8 * nt + 2 * t;  // even column of the pair
            const int chunk = c >> 3;                // 0..7 within the 64-wide box
            const uint32_t off = sw128(R, chunk) + (c & 7) * 2;
            st_shared_u32(sPhi + off, pack_bf16(ep[nt][2 * hr] * ip, ep[nt][2 * hr + 1] * ip));
            st_shared_u32(sPhi + 4096 + off,
                          pack_bf16(em[nt][2 * hr] * im, em[nt][2 * hr + 1] * im));
          }
        }
        if (warp == 0) {
          const int R = lane;
          const float aux = merge == HB_MERGE_SHARED_NORM ? log_sigmoid(gl) : sigmoid(gl);
          float m = part(kSMax, R, 0), ps = 0.f, sp = 0.f, sm = 0.f, dp = 0.f, dm = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, part(kSMax, R, j));
            ps += part(kSumS, R, j);
            sp += part(kSumP, R, j);
            sm += part(kSumM, R, j);
            dp += part(kDenP, R, j);
            dm += part(kDenM, R, j);
          }
          // Per-row coefficients of the merge, o = cU * U + cN * num, with
          // U = sum_j e^{s_ij - m} v_j, P = ps = sum_j e^{s_ij - m}, m the row
          // max (natural units), num = phi^T S, den = phi^T Z.
          const float den = dp / sp + dm / sm;
          const float mnat = m * kLn2;
          float cU, cN;
          if (merge == HB_MERGE_SHARED_NORM) {
            // (w e^m U + num) / (w e^m P + den) with log w = aux, rescaled by
            // e^{-lam} or e^{lam} (lam = aux + m) so nothing overflows
            const float lam = aux + mnat;
            if (lam >= 0.f) {
              const float r = expf(-lam);
              cU = 1.f / (ps + r * den);
              cN = r * cU;
            } else {
              const float r = expf(lam);
              cN = 1.f / (r * ps + den);
              cU = r * cN;
            }
          } else if (den > 0.f) {
            cU = aux / ps;
            cN = (1.f - aux) / den;
          } else {  // nothing committed: the linear branch is dropped
            cU = 1.f / ps;
            cN = 0.f;
          }
          fin[R] = cU;
          fin[32 + R] = cN;
        }
      }
      named_bar_sync(1, kConsumers);

      // ---- phase D: num = phi(q) S and U = P V for columns 16w..16w+15
      float acc_n[2][2][4] = {}, acc_v[2][2][4] = {};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[2][4];
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          const int arow = 16 * m2 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ch = 2 * kk + (lane >> 4);
          ldsm_x4(sPhi + (ch >> 3) * 4096 + sw128(arow, ch & 7), a[m2][0], a[m2][1], a[m2][2],
                  a[m2][3]);
        }
        const int k0 = 16 * kk + 2 * t;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int col = 16 * warp + 8 * nt + g;
          const uint32_t b0 = pack_bf16(ld_shared_f32(sS + s_off(k0, col)),
                                        ld_shared_f32(sS + s_off(k0 + 1, col)));
          const uint32_t b1 = pack_bf16(ld_shared_f32(sS + s_off(k0 + 8, col)),
                                        ld_shared_f32(sS + s_off(k0 + 9, col)));
          mma_bf16(acc_n[0][nt], a[0], b0, b1);
          mma_bf16(acc_n[1][nt], a[1], b0, b1);
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[2][4];
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          const int arow = 16 * m2 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ch = 2 * kk + (lane >> 4);
          ldsm_x4(sP + arow * kPitchP + ch * 16, a[m2][0], a[m2][1], a[m2][2], a[m2][3]);
        }
        uint32_t vb[4];
        const int mtx = lane >> 3;
        const int vrow = 16 * kk + (mtx & 1) * 8 + (lane & 7);
        const int dch = 2 * warp + (mtx >> 1);
        ldsm_x4_t(sV + (dch >> 3) * 4096 + sw128(vrow, dch & 7), vb[0], vb[1], vb[2], vb[3]);
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          mma_bf16(acc_v[m2][0], a[m2], vb[0], vb[1]);
          mma_bf16(acc_v[m2][1], a[m2], vb[2], vb[3]);
        }
      }

      // the stage (S, V) is no longer read: hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);

      // ---- merge and store o
#pragma unroll
      for (int m2 = 0; m2 < 2; ++m2) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int R = 16 * m2 + g + 8 * hr;
          const float cU = fin[R], cN = fin[32 + R];
          __nv_bfloat16* orow = o + ((size_t)(b * kL + R) * H + h) * kD;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int c = 16 * warp + 8 * nt + 2 * t;
            const float o0 = fmaf(cU, acc_v[m2][nt][2 * hr], cN * acc_n[m2][nt][2 * hr]);
            const float o1 = fmaf(cU, acc_v[m2][nt][2 * hr + 1], cN * acc_n[m2][nt][2 * hr + 1]);
            *reinterpret_cast<__nv_bfloat162*>(orow + c) = __floats2bfloat162_rn(o0, o1);
          }
        }
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

int g_num_sms = 0;

}  // namespace

bool fast_attend_ok(const Shape& s) { return production_shape(s); }

cudaError_t launch_attend_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* q,
                               const void* k, const void* v, const float* S_pool,
                               const float* Z_pool, int num_slots, const void* W,
                               const float* gate, void* o, unsigned* status, cudaStream_t st) {
  if ((int64_t)num_slots * s.H * kF >= (int64_t)1 << 31 ||
      (int64_t)batch * kL >= (int64_t)1 << 31)
    return launch_attend_generic(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, W, gate,
                                 o, status, st);
  Maps maps;
  {
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)num_slots * s.H * kF};
    const uint64_t strides[1] = {kD * 4};
    const uint32_t box[2] = {32, 128};
    if (!encode_tmap(&maps.S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, S_pool, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)batch * kL};
    const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
    const uint32_t box[3] = {64, 1, 32};
    const void* ptrs[3] = {q, k, v};
    CUtensorMap* dst[3] = {&maps.q, &maps.k, &maps.v};
    for (int j = 0; j < 3; ++j)
      if (!encode_tmap(dst[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptrs[j], dims, strides, box,
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
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_attend_fast), kSmemBytes);
  if (e != cudaSuccess) return e;
  if (g_num_sms == 0) {
    int dev = 0, n = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    g_num_sms = n;
  }
  const int units = batch * s.H;
  const int grid = units < g_num_sms ? units : g_num_sms;
  k_attend_fast<<<grid, kThreads, kSmemBytes, st>>>(maps, batch, s.H, num_slots,
                                                    s.scale * kLog2e, s.merge,
                                                    slot_idx, S_pool, Z_pool, gate,
                                                    reinterpret_cast<__nv_bfloat16*>(o), status);
  return cudaGetLastError();
}

}  // namespace hb
