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
//   * one CTA per SM, 10 warps: warp 8 is the producer, warp 9 turns the
//     row sums into merge coefficients (and, in the committing variant,
//     stores updated states), warps 0-7 compute;
//   * a two-stage shared-memory ring; each stage holds one (request, head)
//     unit in two parts with their own mbarriers: the head (q, k, v as two
//     4 KiB SWIZZLE_128B boxes each, W_h 16 KiB, Z 512 B) and S (four 16 KiB
//     SWIZZLE_128B boxes); the feature map and block softmax run on the head
//     while S is still arriving;
//   * in the committing variant, units of committing requests come first in
//     the grid-wide order, so that every CTA gets one or two of them; such a
//     unit also forms phi(k) as bf16 hi + lo, runs dS = phi(k)^T V on
//     tcgen05 into TMEM during its state contraction, adds dS into the
//     staged S once every warp has read it, and the coefficient warp
//     TMA-stores the new S and Z;
//   * in the sequential mode (prompts with outputs) one CTA per
//     (request, head) walks the blocks of its prompt in order, the state
//     kept in the first stage's buffers and stored after the last block;
//   * launched with programmatic stream serialization: barrier set-up, TMEM
//     allocation and an L2 prefetch of the step's q, k, v and W overlap the
//     previous kernel's tail;
//   * the producer reads slot indices ahead, prefetches the tiles of the
//     next unit into L2 (deeper prefetch measured slower: it lengthens the
//     DRAM queue the TMA loads wait in), and issues unit i+1's loads while
//     the consumers compute unit i; consumers release a stage through a
//     third mbarrier as soon as S and V have been read;
//   * once q and k have been used their bytes hold the unit's feature map,
//     block probabilities and row sums;
//   * all four contractions (qW, qk^T, phi(q)S, PV) run on bf16 mma.sync with
//     fp32 accumulation. The two halves of phi(q) enter the S contraction
//     unnormalised and in separate accumulators; their normalisers, the
//     block softmax normaliser, phi(q)^T Z and the gate fold into three
//     per-row coefficients of the merge. S is converted fp32 -> bf16 pairs
//     as it is read from shared memory, two columns per 8-byte load (the
//     output columns of a warp are interleaved so that one thread's columns
//     are adjacent), conflict-free thanks to the swizzle;
//   * exponentials are 2^x on the special-function unit with log2(e) folded
//     into the operands; the shared-normaliser merge is rescaled so that
//     nothing overflows.
#include <float.h>

#include "hb_fast.cuh"
#include "hb_ptx.cuh"
#include "hb_state16.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kFH = 64, kF = 128, kL = 32;
constexpr int kConsumerWarps = 8;
// q, k, v and W of a step are prefetched into L2 ahead of the loads when
// together they take at most this many bytes
constexpr size_t kPrefetchBudget = size_t(48) << 20;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;    // warp 8
constexpr int kCoefWarp = kConsumerWarps + 1;    // warp 9: per-row merge coefficients
constexpr int kThreads = kConsumers + 64;

// Stage layout (bytes from the stage base; the base is 1024-aligned).
constexpr int kOffS = 0;                    // 4 x [128 F-rows][32 fp32], SW128
constexpr int kOffQ = 65536;                // 2 x [32 tokens][64 bf16], SW128
constexpr int kOffK = kOffQ + 8192;
constexpr int kOffV = kOffK + 8192;
constexpr int kOffW = kOffV + 8192;         // [128 d-rows][64 bf16], SW128
constexpr int kStageStride = kOffW + 16384; // 104 KiB
constexpr int kHeadBytes = 3 * 8192 + 16384;
constexpr int kSBytes = 65536;
// Consumer scratch inside the stage, valid once phase A is done with q and k:
constexpr int kOffPhi = kOffQ;              // 2 x [32][64 bf16], SW128: e^{u - max}, e^{min - u}
constexpr int kOffP = kOffK;                // [32][40 bf16]: 2^{s - m}, 80-byte rows
constexpr int kPitchP = 80;
constexpr int kOffSums = kOffK + 32 * kPitchP;  // 7 x [32 rows][4 parts] fp32
static_assert(kOffSums + 7 * 32 * 4 * 4 <= kOffV, "scratch overflows the k tile");
// Committing units only, once phase A is done with W_h: phi(k) as bf16 hi
// and lo, each 2 x [32 tokens][64 bf16] SWIZZLE_128B.
constexpr int kOffPhiKHi = kOffW;
constexpr int kOffPhiKLo = kOffW + 8192;
// Dual-copy step, committing units only, once dS has been formed: the bf16
// copy of the new S, 2 x [128 F-rows][64 bf16] SWIZZLE_128B, over the unit's
// q, k, v tiles and the first half of W_h's (all dead by then).
constexpr int kOffS16New = kOffQ;
static_assert(kOffS16New % 1024 == 0 && kOffS16New + 2 * 16384 <= kStageStride,
              "the copy's staging overflows the stage");
// Shared area after the two stages.
constexpr int kOffZ = 2 * kStageStride;     // 2 x [128] fp32 (per stage)
constexpr int kOffPart = kOffZ + 1024;      // max, min of u(q); max of s; max, min of u(k): 5 x [32][4]
constexpr int kOffZPart = kOffPart + 5 * 512;  // column sums of phi(k) per row tile: [2][128]
constexpr int kOffFin = kOffZPart + 1024;   // merge coefficients per stage: 2 x 3 x [32]
constexpr int kOffBar = kOffFin + 2 * 3 * 128;
constexpr int kOffMeta = kOffBar + 13 * 8;  // per stage: flags, slot, request, head, fp8 scale,
                                             // the head's row of W / gate (layer * H + head)
constexpr int kOffTmemSlot = kOffMeta + 48;
// committing variant: the commit mask as one bit per request, 32 per word
constexpr int kMaskWords = 1024;  // batches up to 32768 are scheduled commit-first
constexpr int kOffMaskBits = kOffTmemSlot + 16;
constexpr int kSmemUsed = kOffMaskBits + 4 * kMaskWords;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base to 1024
static_assert(kSmemBytes <= 232448, "shared memory over the sm_100 per-block limit");

enum { kSumP = 0, kSumM, kDenP, kDenM, kSumS, kSumPK, kSumMK };
enum : int { kUnitValid = 1, kUnitCommit = 2, kUnitLast = 4 };  // meta flags of a stage

struct Maps {
  const uint8_t* qkv[3];  // q, k, v base addresses (L2 prefetch of whole token rows)
  const uint8_t* w;       // W base address
  // Request b's active block is rows b * rows_per_req + row_base .. + L - 1
  // of q, k, v and o (rows_per_req = L, row_base = 0 for a decoding step;
  // the prompt length and the block's offset for chunkwise prompt
  // processing); commit_all: every request commits (commit_mask unused).
  int rows_per_req, row_base, commit_all;
  // several independent layers in one call: request b belongs to layer
  // b / reqs_per_layer, whose head h takes row layer * H + h of W and gate
  // (one layer: reqs_per_layer = batch)
  int reqs_per_layer, n_layers;
  // grouped-query heads (attend only): query head h reads k, v, S and Z of
  // head h / kv_group (1: one key/value head per query head)
  int kv_group;
  // sequential mode: the keys take their own map (maps.Wk), kept for the
  // whole walk in the second stage's S buffer, which that mode does not use
  int sep_wk;
  // SM clocks after which a wait of the unit pipeline gives up (hb_set_wait_limit);
  // the final drain of copies already issued always takes the full limit
  long long wait_limit;
  // tokens of a block: 32, or 16 (a decoding step with 16-token blocks: the
  // 32-row tiles hold the block and 16 rows past it, which take no part:
  // their keys are masked out of the block softmax, their k rows out of the
  // commit, and their outputs are not stored)
  int valid_rows;
  const uint8_t* s16;  // dual-copy step: the bf16 copies (L2 prefetch of a unit's copy)
  // fp8 attend (kS8): the scale of each (slot, head) copy, S = scale * code
  const float* s8_scale;
  CUtensorMap S;  // [slots*H*F rows][d] fp32, box {32, 128}; kS16 attend only: bf16, box {64, 128}
  CUtensorMap S16;  // dual-copy step: the bf16 copies [slots*H*F rows][d], box {64, 128}
  CUtensorMap q;  // [B*L][H][d] bf16, box {64, 1, 32}
  CUtensorMap k;
  CUtensorMap v;
  CUtensorMap W;  // [H*d rows][f] bf16, box {64, 128}: the query map (and the key map
                  // unless sep_wk)
  CUtensorMap Wk;  // sep_wk: the key map, as W
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
// Byte offset of S[k][n] (bf16 copy of the state) in the two SW128 boxes of
// the stage's S region.
__device__ __forceinline__ uint32_t s16_off(int k, int n) {
  return (uint32_t)((n >> 6) * 16384 + k * 128 + ((((n & 63) >> 3) ^ (k & 7)) << 4) +
                    (n & 7) * 2);
}
// Byte offset of code S[k][n] (fp8 copy of the state) in the SW128 box of
// the stage's S region ([128 F rows][128 codes]).
__device__ __forceinline__ uint32_t s8_off(int k, int n) {
  return (uint32_t)(k * 128 + ((((n >> 4) ^ (k & 7))) << 4) + (n & 15));
}
// Byte offset of v[key][n] (bf16) in the two SW128 boxes of the v tile.
__device__ __forceinline__ uint32_t v_off(int key, int n) {
  return (uint32_t)((n >> 6) * 4096 + key * 128 + ((((n & 63) >> 3) ^ (key & 7)) << 4) +
                    (n & 7) * 2);
}

// kSeq = true (with kCommit): one CTA per (request, head) runs the blocks of
// a prompt in order (rows j L .. j L + L - 1 of rows_per_req), each block
// attending to the state left by the blocks before it and then committed.
// The state is loaded once into the first stage's S and Z buffers, updated
// there in place after every block, and stored after the last one; only q,
// k, v and W_h go through the two-stage ring.
// kCommit = false: attend only (commit_mask is ignored; S_pool and Z_pool are
// not written). kCommit = true: requests with commit_mask[b] != 0 also fold
// their block into the state after their output has been formed.
// kS16 (attend only): S_pool is a bf16 copy of the states, each value the
// round-to-nearest of the fp32 master. The state contraction takes S as bf16
// operands rounded to nearest either way, so the output is bit-identical to
// the fp32 pool's, while a unit reads 32 KiB of state instead of 64.
// kS8 (attend only): S_pool is an fp8 (e4m3) copy of the states with one
// scale per (slot, head), S = scale * code. The codes enter the state
// contraction as f16 (exact), with phi(q) as f16 too, and the scale folds
// into the merge coefficients, so a unit reads 16 KiB of state instead of 64;
// the output is that of the attend on the dequantised state.
// kS16 with kCommit (the dual-copy step): every slot has the fp32 master in
// S_pool and its bf16 copy behind maps.S16. A request that does not commit
// reads the copy; a committing request reads the master, adds its block,
// and stores the new master and its round-to-nearest copy. The output bits
// are those of the fp32-only step whenever the copies are in step with the
// masters.
template <bool kCommit, bool kSeq = false, bool kS16 = false, bool kS8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_attend_fast(const __grid_constant__ Maps maps, int batch, int H, int num_slots, float scale,
                  int merge, const int32_t* __restrict__ slot_idx,
                  const int32_t* __restrict__ commit_mask, const float* __restrict__ S_pool,
                  float* __restrict__ Z_pool, const float* __restrict__ gate,
                  __nv_bfloat16* __restrict__ o, unsigned* status) {
  static_assert(!(kS16 && kSeq), "the sequential mode keeps the fp32 state on chip");
  static_assert(!(kS8 && (kCommit || kSeq || kS16)), "the fp8 copy is read by the attend only");
  constexpr bool kDual = kS16 && kCommit;  // the dual-copy step
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* head_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* s_full = head_full + 2;
  uint64_t* empty = head_full + 4;
  uint64_t* sums_ready = head_full + 6;  // consumers -> coefficient warp
  uint64_t* fin_ready = head_full + 8;   // coefficient warp -> consumers
  uint64_t* ds_full = head_full + 10;    // committing units: the tensor cores' dS is in TMEM
  uint64_t* s_updated = head_full + 11;  // committing units: new S, Z are in the stage
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  // units whose tiles the producer has issued (read by the final drain)
  volatile int* n_issued = reinterpret_cast<volatile int*>(smem + kOffTmemSlot + 4);
  const long long lim = maps.wait_limit;
  int* meta = reinterpret_cast<int*>(smem + kOffMeta);
  float* pmax = reinterpret_cast<float*>(smem + kOffPart);  // [32][4]
  float* pmin = pmax + 128;                                 // [32][4]
  float* smax = pmin + 128;                                 // [32][4]
  float* pmaxk = smax + 128;                                // [32][4]
  float* pmink = pmaxk + 128;                               // [32][4]
  float* zpart = reinterpret_cast<float*>(smem + kOffZPart);  // [2][128]
  float* fin_all = reinterpret_cast<float*>(smem + kOffFin);  // [stage][cU, cP, cM][32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = batch * H;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&head_full[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&empty[s], kConsumerWarps + 1);  // + the coefficient warp
      mbar_init(&sums_ready[s], kConsumerWarps);
      mbar_init(&fin_ready[s], 1);
    }
    mbar_init(ds_full, 1);
    mbar_init(&s_updated[0], kConsumerWarps);
    mbar_init(&s_updated[1], kConsumerWarps);
    fence_mbar_init();
    *n_issued = 0;
  }
  // committing variant: 128 TMEM columns hold dS = phi(k)^T V [128 F][128 d]
  if (kCommit && warp == 0) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = kCommit ? *tmem_slot : 0u;
  // The set-up above overlaps the previous kernel's tail, and so does an L2
  // prefetch of the step's q, k, v and W when together they take a modest
  // part of L2: each CTA prefetches a 1/grid share. A prefetch reads nothing
  // into the SM, and L2 is where the previous kernel's writes land, so this
  // is safe before the wait. Every load and store of global memory comes
  // after grid_dep_wait().
  if (warp == kProducerWarp && lane == 0) {
    const size_t q_bytes = (size_t)batch * maps.rows_per_req * H * kD * 2;
    const size_t kv_bytes = q_bytes / maps.kv_group;  // k, v have H / kv_group heads
    const size_t w_bytes = (size_t)maps.n_layers * H * kD * kFH * 2;
    if (q_bytes + 2 * kv_bytes + w_bytes <= kPrefetchBudget) {
      const uint8_t* base[4] = {maps.qkv[0], maps.qkv[1], maps.qkv[2], maps.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const size_t bytes = j == 0 ? q_bytes : j < 3 ? kv_bytes : w_bytes;
        // 16-byte aligned share of this CTA, issued in pieces of <= 32 KiB
        const size_t share = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
        size_t lo = (size_t)blockIdx.x * share;
        const size_t hi = lo + share < bytes ? lo + share : bytes;
        for (; lo < hi; lo += 32768) {
          const size_t n = (hi - lo < 32768 ? hi - lo : 32768) & ~size_t(15);
          if (n > 0) prefetch_l2(base[j] + lo, (uint32_t)n);
        }
      }
    }
  }
  grid_dep_wait();
  grid_dep_launch();
  int ds_issued = 0;  // thread 0: dS MMAs issued (committing units)
  // units of this CTA: every gridDim.x-th (request, head) unit, or in the
  // sequential mode the blocks of its (request, head)
  const int n_units_cta =
      kSeq ? maps.rows_per_req / kL
           : ((int)blockIdx.x < units ? (units - (int)blockIdx.x + (int)gridDim.x - 1) /
                                            (int)gridDim.x
                                      : 0);

  if (warp == kCoefWarp) {
    // ------------------------------------------------- merge coefficients
    // Lane R computes row R of the unit's merge, o = cU U + cP num+ + cM num-
    // (U = sum_j e^{s_ij - m} v_j; num+- the contractions of the unnormalised
    // halves of phi(q) with S), from the row sums the consumers leave in the
    // stage, while the consumers run the state contraction.
    uint32_t su_phase[2] = {0u, 0u};  // parity of s_updated per stage
    for (int i = 0; i < n_units_cta; ++i) {
      const int s = i & 1, n = i >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&sums_ready[s], n & 1, lim))) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        break;
      }
      const int h = meta[6 + s];
      const float gl = gate[meta[10 + s]];
      if (meta[s] & kUnitValid) {
        const float* sums = reinterpret_cast<const float*>(smem + s * kStageStride + kOffSums);
        float* fin = fin_all + s * 96;
        const int R = lane;
        const float4 a = *reinterpret_cast<const float4*>(sums + (kSumP * 32 + R) * 4);
        const float4 c = *reinterpret_cast<const float4*>(sums + (kSumM * 32 + R) * 4);
        const float4 d = *reinterpret_cast<const float4*>(sums + (kDenP * 32 + R) * 4);
        const float4 e = *reinterpret_cast<const float4*>(sums + (kDenM * 32 + R) * 4);
        const float4 f = *reinterpret_cast<const float4*>(sums + (kSumS * 32 + R) * 4);
        const float4 m4 = *reinterpret_cast<const float4*>(smax + R * 4);
        // (approximate reciprocals and exponentials: ~1e-7 relative, far
        // below what a bf16 output can show)
        const float sp = (a.x + a.y) + (a.z + a.w), sm = (c.x + c.y) + (c.z + c.w);
        const float ps = (f.x + f.y) + (f.z + f.w);
        const float isp = rcp_approx(sp), ism = rcp_approx(sm);
        const float den = ((d.x + d.y) + (d.z + d.w)) * isp + ((e.x + e.y) + (e.z + e.w)) * ism;
        const float m2 = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));  // row max, base 2
        float cU, cN;
        if (merge == HB_MERGE_SHARED_NORM) {
          // (w e^m U + num) / (w e^m P + den) with log w = log sigmoid(alpha),
          // rescaled by e^{-lam} or e^{lam} (lam = log w + m) so nothing overflows
          const float lam2 = log_sigmoid(gl) * kLog2e + m2;  // lam in base 2
          if (lam2 >= 0.f) {
            const float r = ex2_approx(-lam2);
            cU = rcp_approx(fmaf(r, den, ps));
            cN = r * cU;
          } else {
            const float r = ex2_approx(lam2);
            cN = rcp_approx(fmaf(r, ps, den));
            cU = r * cN;
          }
        } else {
          const float w = sigmoid(gl);
          if (den > 0.f) {
            cU = w * rcp_approx(ps);
            cN = (1.f - w) * rcp_approx(den);
          } else {  // nothing committed: the linear branch is dropped
            cU = rcp_approx(ps);
            cN = 0.f;
          }
        }
        // (fp8 copy: the contraction used the codes, S = scale * code)
        const float sc = kS8 ? __int_as_float(meta[8 + s]) : 1.f;
        fin[R] = cU;
        fin[32 + R] = cN * isp * sc;
        fin[64 + R] = cN * ism * sc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&fin_ready[s]);
      if (kSeq) {
        // the prompt's last block: store the state once the consumers have
        // updated it; every block: the row sums have been read
        if (meta[s] & kUnitLast) {
          const bool ok = mbar_wait(&s_updated[s], su_phase[s], lim);
          su_phase[s] ^= 1u;
          if (lane == 0) {
            if (ok) {
              const int uslot = meta[2 + s];
              const int row = (uslot * H + h) * kF;
#pragma unroll
              for (int bx = 0; bx < 4; ++bx)
                tma_store_2d(&maps.S, 32 * bx, row, smem + kOffS + bx * 16384);
              bulk_store(Z_pool + (size_t)(uslot * H + h) * kF, smem + kOffZ, kF * 4);
              bulk_commit();
              bulk_wait_read();
            } else {
              atomicOr(status, kStatusTimeout);
            }
          }
        }
        if (lane == 0) mbar_arrive(&empty[s]);
      } else if (kCommit && (meta[s] & kUnitCommit)) {
        // the consumers have written the new S and Z into the stage: store
        // them (TMA), and hand the stage back on their behalf once the store
        // has read it (not after a wait that ran out: the stage's loads may
        // still be landing, so it is never refilled)
        const bool ok = mbar_wait(&s_updated[s], su_phase[s], lim);
        su_phase[s] ^= 1u;
        if (lane == 0) {
          if (ok) {
            const int uslot = meta[2 + s];
            const int row = (uslot * H + h) * kF;
            uint8_t* st = smem + s * kStageStride;
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
              tma_store_2d(&maps.S, 32 * bx, row, st + kOffS + bx * 16384);
            if (kDual) {
              // the new state's bf16 copy, staged in the unit's dead head tiles
#pragma unroll
              for (int bx = 0; bx < 2; ++bx)
                tma_store_2d(&maps.S16, 64 * bx, row, st + kOffS16New + bx * 16384);
            }
            bulk_store(Z_pool + (size_t)(uslot * H + h) * kF, smem + kOffZ + s * 512, kF * 4);
            bulk_commit();
            bulk_wait_read();
            mbar_arrive_cnt(&empty[s], kConsumerWarps + 1);
          } else {
            atomicOr(status, kStatusTimeout);
          }
        }
      } else if (lane == 0) {
        mbar_arrive(&empty[s]);  // the row sums in the stage have been read
      }
    }
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; lane 0 issues the copies. A unit's q, k,
    // v and W_h do not depend on its state slot, so the first unit's are
    // issued before its slot index is read; the slots of later units are
    // read 32 at a time, a window ahead, and each unit's tiles are
    // prefetched into L2 one unit before their TMA load is issued.
    if (lane == 0) {
      prefetch_tmap(&maps.S);
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      prefetch_tmap(&maps.W);
    }
    const int first = blockIdx.x, stride = gridDim.x;
    const int n_local = n_units_cta;
    if (kSeq) {
      // this CTA's (request, head); its blocks in order, the state with the
      // first one only
      const int b = (int)blockIdx.x / H, h = (int)blockIdx.x - b * H;
      const int slot = slot_idx[b];
      const bool bad = slot < 0 || slot >= num_slots;
      if (lane == 0 && bad) atomicOr(status, kStatusBounds);
      const size_t slice = (size_t)kL * kD * 2;
      for (int i = 0; i < n_local; ++i) {
        const int s = i & 1, n = i >> 1;
        bool ok = true;
        if (lane == 0 && n > 0) ok = mbar_wait(&empty[s], (n - 1) & 1, lim);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          if (lane == 0) atomicOr(status, kStatusTimeout);
          break;
        }
        if (lane == 0) {
          *n_issued = i + 1;
          uint8_t* st = smem + s * kStageStride;
          const int row = b * maps.rows_per_req + i * kL;
          mbar_expect_tx(&head_full[s], kHeadBytes);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            tma_load_3d(st + kOffQ + j * 4096, &maps.q, 64 * j, h, row, &head_full[s]);
            tma_load_3d(st + kOffK + j * 4096, &maps.k, 64 * j, h, row, &head_full[s]);
            tma_load_3d(st + kOffV + j * 4096, &maps.v, 64 * j, h, row, &head_full[s]);
          }
          const int wh = (b / maps.reqs_per_layer) * H + h;
          tma_load_2d(st + kOffW, &maps.W, 0, wh * kD, &head_full[s]);
          meta[4 + s] = b;
          meta[6 + s] = h;
          meta[10 + s] = wh;
          if (bad) {
            meta[s] = 0;
            mbar_arrive(&head_full[s]);
            mbar_arrive(&s_full[s]);
          } else {
            meta[s] = kUnitValid | kUnitCommit | (i == n_local - 1 ? kUnitLast : 0);
            meta[2 + s] = slot;
            if (i == 0) {
              if (maps.sep_wk) {  // the key map, kept for the whole walk
                mbar_expect_tx(&head_full[s], 16384);
                tma_load_2d(smem + kStageStride + kOffS, &maps.Wk, 0, wh * kD, &head_full[s]);
              }
              mbar_expect_tx(&head_full[s], 512);
              bulk_load(smem + kOffZ, Z_pool + (size_t)(slot * H + h) * kF, 512, &head_full[s]);
              mbar_arrive(&head_full[s]);
              mbar_arrive_expect_tx(&s_full[s], kSBytes);
              const int srow = (slot * H + h) * kF;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_2d(smem + kOffS + j * 16384, &maps.S, 32 * j, srow, &s_full[s]);
            } else {
              mbar_arrive(&head_full[s]);
              mbar_arrive(&s_full[s]);
            }
          }
          if (i + 2 < n_local) {
            // the block two ahead: its rows of all heads are contiguous, so
            // the CTAs of this request each prefetch a 1/H slice of them
            const size_t off = ((size_t)b * maps.rows_per_req + (size_t)(i + 2) * kL) * H * kD * 2 +
                               (size_t)h * slice;
#pragma unroll
            for (int j = 0; j < 3; ++j) prefetch_l2(maps.qkv[j] + off, (uint32_t)slice);
          }
        }
        __syncwarp();
      }
    } else {
    // Unit schedule. Position p = first + i * stride of the grid-wide order
    // is this CTA's i-th unit. Committing requests are heavier (their state
    // is also updated and stored), so in the committing variant their units
    // take the first positions, which spreads them evenly over the CTAs;
    // then come the other requests', each group in request order, heads
    // innermost. The mask is kept as bits in shared memory.
    uint32_t* mask_bits = reinterpret_cast<uint32_t*>(smem + kOffMaskBits);
    const int mask_words = (batch + 31) >> 5;
    const bool all_commit = kCommit && maps.commit_all != 0;
    const bool commit_first = kCommit && !all_commit && mask_words <= kMaskWords;
    int n_commit = 0;  // committing requests
    if (commit_first) {
      // eight words per round, their loads issued back to back, so the scan
      // costs one memory round trip for batches up to 256
      for (int w0 = 0; w0 < mask_words; w0 += 8) {
        int f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 32 * (w0 + j) + lane;
          f[j] = (w0 + j < mask_words && r < batch) ? commit_mask[r] : 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t bits = __ballot_sync(0xffffffffu, f[j] != 0);
          if (lane == 0 && w0 + j < mask_words) mask_bits[w0 + j] = bits;
          n_commit += __popc(bits);
        }
      }
      __syncwarp();
    }
    const int commit_units = all_commit ? units : n_commit * H;
    // Lane j describes local unit 32 W + j of window W. Its request comes
    // from a per-lane cursor over the mask bits for each flag value (a
    // lane's units have increasing positions, so the cursors only move
    // forward); -1 if the mask no longer holds that many (it changed while
    // this kernel ran).
    int cw[2] = {0, 0}, cbefore[2] = {0, 0};
    auto nth_request = [&](int want, int r) -> int {
      for (;;) {
        if (cw[want] >= mask_words) return -1;
        const int w = cw[want];
        uint32_t bits = mask_bits[w];
        if (!want) {
          const int left = batch - 32 * w;
          bits = ~bits & (left >= 32 ? 0xffffffffu : (1u << left) - 1u);
        }
        const int cnt = __popc(bits);
        if (cbefore[want] + cnt > r) {
          for (int t = r - cbefore[want]; t > 0; --t) bits &= bits - 1u;
          return 32 * w + __ffs(bits) - 1;
        }
        cbefore[want] += cnt;
        ++cw[want];
      }
    };
    struct Window {
      int b, h, flags;  // flags: kUnitCommit, or -1 for a request the mask lost
      int slot;
      float scale;      // fp8 copy: the unit's scale
    };
    // fills this lane's entry of window W and issues its slot load
    auto fill_window = [&](int W) -> Window {
      Window wd{0, 0, 0, -1, 1.f};
      const int i = 32 * W + lane;
      if (i >= n_local) return wd;
      const int p = first + i * stride;
      int r;
      if (p < commit_units) {
        r = p / H;
        wd.h = p - r * H;
        wd.b = all_commit ? r : nth_request(1, r);
        wd.flags = kUnitCommit;
      } else {
        r = (p - commit_units) / H;
        wd.h = p - commit_units - r * H;
        wd.b = commit_first ? nth_request(0, r) : r;
        wd.flags = (kCommit && !commit_first && commit_mask[wd.b] != 0) ? kUnitCommit : 0;
      }
      if (wd.b < 0) {  // flagged through the slot; nothing is written for it
        wd.b = 0;
        wd.flags = -1;
      } else {
        wd.slot = slot_idx[wd.b];
        if (kS8 && wd.slot >= 0 && wd.slot < num_slots)
          wd.scale = maps.s8_scale[(size_t)wd.slot * (H / maps.kv_group) + wd.h / maps.kv_group];
      }
      return wd;
    };
    Window win_cur = fill_window(0), win_next = fill_window(1);
    int win_base = 0;  // window index of win_cur
    // fields of local unit i (warp-uniform, within the two windows held)
    auto unit_b = [&](int i) {
      return __shfl_sync(0xffffffffu, (i >> 5) == win_base ? win_cur.b : win_next.b, i & 31);
    };
    auto unit_h = [&](int i) {
      return __shfl_sync(0xffffffffu, (i >> 5) == win_base ? win_cur.h : win_next.h, i & 31);
    };
    auto unit_flags = [&](int i) {
      return __shfl_sync(0xffffffffu, (i >> 5) == win_base ? win_cur.flags : win_next.flags,
                         i & 31);
    };
    auto unit_slot = [&](int i) {
      return __shfl_sync(0xffffffffu, (i >> 5) == win_base ? win_cur.slot : win_next.slot,
                         i & 31);
    };
    auto unit_scale = [&](int i) {
      return __shfl_sync(0xffffffffu, (i >> 5) == win_base ? win_cur.scale : win_next.scale,
                         i & 31);
    };
    auto issue_head = [&](int i) {
      const int s = i & 1;
      const int b = unit_b(i), h = unit_h(i);
      const int g = h / maps.kv_group;  // key/value head
      uint8_t* st = smem + s * kStageStride;
      if (lane == 0) {
        *n_issued = i + 1;  // issue_state(i) always follows
        mbar_expect_tx(&head_full[s], kHeadBytes);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int row = b * maps.rows_per_req + maps.row_base;
          tma_load_3d(st + kOffQ + j * 4096, &maps.q, 64 * j, h, row, &head_full[s]);
          tma_load_3d(st + kOffK + j * 4096, &maps.k, 64 * j, g, row, &head_full[s]);
          tma_load_3d(st + kOffV + j * 4096, &maps.v, 64 * j, g, row, &head_full[s]);
        }
        tma_load_2d(st + kOffW, &maps.W, 0, ((b / maps.reqs_per_layer) * H + h) * kD,
                    &head_full[s]);
      }
    };
    auto issue_state = [&](int i) {
      const int s = i & 1;
      const int b = unit_b(i), h = unit_h(i);
      const int hs = h / maps.kv_group;  // the state's head
      const int Hs = H / maps.kv_group;
      const int flags = unit_flags(i), slot = unit_slot(i);
      const float scale = kS8 ? unit_scale(i) : 1.f;
      uint8_t* st = smem + s * kStageStride;
      if (lane == 0) {
        meta[4 + s] = b;
        meta[6 + s] = h;
        meta[8 + s] = __float_as_int(scale);
        meta[10 + s] = (b / maps.reqs_per_layer) * H + h;
        if (flags < 0 || slot < 0 || slot >= num_slots) {
          atomicOr(status, kStatusBounds);
          meta[s] = 0;
          mbar_arrive(&head_full[s]);
          mbar_arrive(&s_full[s]);
        } else {
          meta[s] = kUnitValid | flags;
          meta[2 + s] = slot;
          mbar_expect_tx(&head_full[s], 512);
          bulk_load(smem + kOffZ + s * 512, Z_pool + (size_t)(slot * Hs + hs) * kF, 512,
                    &head_full[s]);
          mbar_arrive(&head_full[s]);
          const int srow = (slot * Hs + hs) * kF;
          if (kS8) {
            // the fp8 copy: one SWIZZLE_128B box of [128 F rows][128 codes]
            mbar_arrive_expect_tx(&s_full[s], kSBytes / 4);
            tma_load_2d(st + kOffS, &maps.S, 0, srow, &s_full[s]);
          } else if (kS16 && !(kDual && (flags & kUnitCommit))) {
            // the bf16 copy (a dual-copy step's committing unit reads the master)
            mbar_arrive_expect_tx(&s_full[s], kSBytes / 2);
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d(st + kOffS + j * 16384, kDual ? &maps.S16 : &maps.S, 64 * j, srow,
                          &s_full[s]);
          } else {
            mbar_arrive_expect_tx(&s_full[s], kSBytes);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(st + kOffS + j * 16384, &maps.S, 32 * j, srow, &s_full[s]);
          }
        }
      }
    };
    auto l2_prefetch = [&](int i) {
      const int b = unit_b(i), h = unit_h(i), slot = unit_slot(i), flags = unit_flags(i);
      if (lane != 0 || slot < 0 || slot >= num_slots) return;
      const int G = maps.kv_group;
      const size_t unit = (size_t)slot * (H / G) + h / G;
      if (kDual && !(flags & kUnitCommit))
        prefetch_l2(maps.s16 + unit * kF * kD * 2, kF * kD * 2);
      else {
        // bytes per state value in S_pool: fp8 copy 1, bf16 copy 2, fp32 4
        constexpr int kSv = kS8 ? 1 : (kS16 && !kDual) ? 2 : 4;
        prefetch_l2(reinterpret_cast<const uint8_t*>(S_pool) + unit * kF * kD * kSv, kF * kD * kSv);
      }
      prefetch_l2(Z_pool + unit * kF, kF * 4);
      // the request's block of q, k, v is one contiguous range of L rows of
      // all heads; the CTAs working on its heads at the same time each
      // prefetch a 1/H slice of it, so DRAM reads it as one long run
      // (k and v have H / G heads: their block is G times smaller)
      const size_t slice = (size_t)maps.valid_rows * kD * 2;  // = q block bytes / H
      const size_t row0 = (size_t)b * maps.rows_per_req + maps.row_base;
      prefetch_l2(maps.qkv[0] + row0 * H * kD * 2 + (size_t)h * slice, (uint32_t)slice);
      const size_t kv_slice = slice / G;
      const size_t kv_off = row0 * (H / G) * kD * 2 + (size_t)h * kv_slice;
#pragma unroll
      for (int j = 1; j < 3; ++j) prefetch_l2(maps.qkv[j] + kv_off, (uint32_t)kv_slice);
    };
    // Both stages are free at the start. Unit 0 goes out first and whole;
    // unit 1's head follows, but its state only once unit 0's has landed,
    // so that DRAM serves unit 0 first and its computation starts early.
    // Later units are prefetched into L2 one unit ahead of their TMA loads.
    if (n_local > 0) {
      issue_head(0);
      issue_state(0);
    }
    if (n_local > 1) {
      issue_head(1);
      if (lane == 0) mbar_wait(&s_full[0], 0, lim);  // a wait that runs out only delays
      __syncwarp();
      issue_state(1);
    }
    if (n_local > 2) l2_prefetch(2);
    for (int i = 2; i < n_local; ++i) {
      const int s = i & 1, n = i >> 1;
      if ((i >> 5) != win_base) {  // move on to the next window
        win_cur = win_next;
        ++win_base;
        win_next = fill_window(win_base + 1);
      }
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&empty[s], (n - 1) & 1, lim);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        break;
      }
      issue_head(i);
      issue_state(i);
      if (i + 1 < n_local) l2_prefetch(i + 1);
    }
    }  // non-sequential producer
  } else {

  // -------------------------------------------------------------- consumers
  // Warp w: row tile mt = w & 1 (rows 16 mt .. 16 mt + 15), column quarter
  // nq = w >> 1 of u = q W_h (16 of 64 columns) and keys 8 nq .. 8 nq + 7 of
  // the block scores; in phase D, output columns 16 w .. 16 w + 15 of both
  // row tiles, interleaved: physical column 16 w + 2 c + j is column c of
  // n-tile j.
  const int g = lane >> 2, t = lane & 3;
  const int mt = warp & 1, nq = warp >> 1;
  const int c0 = 16 * warp;

  // A wait that runs out does not leave the loop on its own: the warp goes on
  // to the next named barrier, which also votes, and all warps leave
  // together (a warp left behind at a named barrier would never return).
  int i = 0;
  bool aborted = false, late_fail = false;
  uint32_t cm_phase = 0;  // parity of ds_full for the next committing unit
  for (; i < n_units_cta; ++i) {
    const int s = i & 1, n = i >> 1;
    const bool head_ok = mbar_wait(&head_full[s], n & 1, lim);
    uint8_t* st = smem + s * kStageStride;
    // the sequential mode keeps one state, in the first stage's buffers
    const uint32_t sS = smem_u32(kSeq ? smem + kOffS : st + kOffS);
    const uint32_t sQ = smem_u32(st + kOffQ);
    const uint32_t sK = smem_u32(st + kOffK);
    const uint32_t sV = smem_u32(st + kOffV);
    const uint32_t sW = smem_u32(st + kOffW);
    const uint32_t sPhi = smem_u32(st + kOffPhi);
    const uint32_t sP = smem_u32(st + kOffP);
    float* sums = reinterpret_cast<float*>(st + kOffSums);  // [7][32][4]
    float* sZ = reinterpret_cast<float*>(smem + kOffZ + (kSeq ? 0 : s * 512));
    const int b = meta[4 + s], h = meta[6 + s];
    const int R0 = 16 * mt + g, R1 = R0 + 8;
    // stage flags, valid once the head has landed (the producer writes them
    // before it arrives on head_full)
    const int flags = meta[s];
    const bool cm = kCommit && (flags & kUnitCommit) != 0;  // this unit also commits its block

    // ---- phase A: u = q W_h (16 rows x 16 cols per warp) and
    //      s = q k^T (16 rows x 8 keys per warp); for a committing unit also
    //      u_k = k W_h
    float acc_u[2][4] = {}, acc_s[4] = {}, acc_uk[2][4] = {};
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
        uint32_t ka0[4], ka1[4];  // k rows as the A operand (committing units)
        if (cm) {
          const int ch = 2 * kk + (lane >> 4);
          ldsm_x4(sK + (ch >> 3) * 4096 + sw128(arow, ch & 7), ka0[0], ka0[1], ka0[2], ka0[3]);
          const int ch1 = ch + 2;
          ldsm_x4(sK + (ch1 >> 3) * 4096 + sw128(arow, ch1 & 7), ka1[0], ka1[1], ka1[2], ka1[3]);
        }
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
          if (cm) {
            uint32_t wk[4] = {wb[0], wb[1], wb[2], wb[3]};
            if (kSeq && maps.sep_wk)  // the key map, in the second stage's S buffer
              ldsm_x4_t(smem_u32(smem + kStageStride + kOffS) + sw128(krow, nch), wk[0], wk[1],
                        wk[2], wk[3]);
            mma_bf16(acc_uk[0], half ? ka1 : ka0, wk[0], wk[1]);
            mma_bf16(acc_uk[1], half ? ka1 : ka0, wk[2], wk[3]);
          }
        }
      }
    }
    const int vrows = maps.valid_rows;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      acc_s[r] *= scale;  // scale * log2(e): scores in base 2
      if (8 * nq + 2 * t + (r & 1) >= vrows) acc_s[r] = -INFINITY;  // a key past the block
    }
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
        pmax[R0 * 4 + nq] = mx0;
        pmax[R1 * 4 + nq] = mx1;
        pmin[R0 * 4 + nq] = mn0;
        pmin[R1 * 4 + nq] = mn1;
        smax[R0 * 4 + nq] = sm0;
        smax[R1 * 4 + nq] = sm1;
      }
      if (cm) {
        float kx0 = fmaxf(fmaxf(acc_uk[0][0], acc_uk[0][1]), fmaxf(acc_uk[1][0], acc_uk[1][1]));
        float kx1 = fmaxf(fmaxf(acc_uk[0][2], acc_uk[0][3]), fmaxf(acc_uk[1][2], acc_uk[1][3]));
        float kn0 = fminf(fminf(acc_uk[0][0], acc_uk[0][1]), fminf(acc_uk[1][0], acc_uk[1][1]));
        float kn1 = fminf(fminf(acc_uk[0][2], acc_uk[0][3]), fminf(acc_uk[1][2], acc_uk[1][3]));
#pragma unroll
        for (int o2 = 1; o2 < 4; o2 <<= 1) {
          kx0 = fmaxf(kx0, __shfl_xor_sync(0xffffffffu, kx0, o2));
          kx1 = fmaxf(kx1, __shfl_xor_sync(0xffffffffu, kx1, o2));
          kn0 = fminf(kn0, __shfl_xor_sync(0xffffffffu, kn0, o2));
          kn1 = fminf(kn1, __shfl_xor_sync(0xffffffffu, kn1, o2));
        }
        if (t == 0) {
          pmaxk[R0 * 4 + nq] = kx0;
          pmaxk[R1 * 4 + nq] = kx1;
          pmink[R0 * 4 + nq] = kn0;
          pmink[R1 * 4 + nq] = kn1;
        }
      }
    }
    // q and k are no longer read after this barrier
    if (named_bar_any(1, kConsumers, !head_ok || late_fail)) {
      if (threadIdx.x == 0) atomicOr(status, kStatusTimeout);
      aborted = true;
      break;
    }

    // ---- phase B: unnormalised exponentials of both halves of phi(q), their
    //      partial sums and partial dot products with Z; P = 2^{s - m}; for a
    //      committing unit also the exponentials of both halves of phi(k)
    float ekp[2][4], ekm[2][4];
    if (cm) {
      float okp[2], okm[2], skp[2] = {0.f, 0.f}, skm[2] = {0.f, 0.f};
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int R = hr ? R1 : R0;
        const float4 a = *reinterpret_cast<const float4*>(pmaxk + R * 4);
        const float4 c = *reinterpret_cast<const float4*>(pmink + R * 4);
        okp[hr] = -fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)) * kLog2e;
        okm[hr] = fminf(fminf(c.x, c.y), fminf(c.z, c.w)) * kLog2e;
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float x = acc_uk[nt][r];
          ekp[nt][r] = ex2_approx(fmaf(x, kLog2e, okp[r >> 1]));
          ekm[nt][r] = ex2_approx(fmaf(-x, kLog2e, okm[r >> 1]));
          skp[r >> 1] += ekp[nt][r];
          skm[r >> 1] += ekm[nt][r];
        }
#pragma unroll
      for (int o2 = 1; o2 < 4; o2 <<= 1)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          skp[hr] += __shfl_xor_sync(0xffffffffu, skp[hr], o2);
          skm[hr] += __shfl_xor_sync(0xffffffffu, skm[hr], o2);
        }
      if (t == 0) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int R = hr ? R1 : R0;
          sums[(kSumPK * 32 + R) * 4 + nq] = skp[hr];
          sums[(kSumMK * 32 + R) * 4 + nq] = skm[hr];
        }
      }
    }
    {
      float op[2], om[2], Ms[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int R = hr ? R1 : R0;
        const float4 a = *reinterpret_cast<const float4*>(pmax + R * 4);
        const float4 c = *reinterpret_cast<const float4*>(pmin + R * 4);
        const float4 f = *reinterpret_cast<const float4*>(smax + R * 4);
        op[hr] = -fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)) * kLog2e;
        om[hr] = fminf(fminf(c.x, c.y), fminf(c.z, c.w)) * kLog2e;
        Ms[hr] = fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w));
      }
      float sp[2] = {0.f, 0.f}, sm[2] = {0.f, 0.f}, dp[2] = {0.f, 0.f}, dm[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * nq + 8 * nt + 2 * t;
        const float2 zp = *reinterpret_cast<const float2*>(sZ + c);
        const float2 zm = *reinterpret_cast<const float2*>(sZ + kFH + c);
        float ep[4], em[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int hr = r >> 1;
          const float x = acc_u[nt][r];
          ep[r] = ex2_approx(fmaf(x, kLog2e, op[hr]));   // e^{u - max u}
          em[r] = ex2_approx(fmaf(-x, kLog2e, om[hr]));  // e^{min u - u}
          sp[hr] += ep[r];
          sm[hr] += em[r];
          dp[hr] = fmaf(ep[r], (r & 1) ? zp.y : zp.x, dp[hr]);
          dm[hr] = fmaf(em[r], (r & 1) ? zm.y : zm.x, dm[hr]);
        }
        const uint32_t off0 = sw128(R0, c >> 3) + (c & 7) * 2;
        const uint32_t off1 = sw128(R1, c >> 3) + (c & 7) * 2;
        // (the fp8 copy's contraction runs on f16 operands)
        auto pk = [](float lo, float hi) { return kS8 ? pack_f16(lo, hi) : pack_bf16(lo, hi); };
        st_shared_u32(sPhi + off0, pk(ep[0], ep[1]));
        st_shared_u32(sPhi + off1, pk(ep[2], ep[3]));
        st_shared_u32(sPhi + 4096 + off0, pk(em[0], em[1]));
        st_shared_u32(sPhi + 4096 + off1, pk(em[2], em[3]));
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
          sums[(kSumP * 32 + R) * 4 + nq] = sp[hr];
          sums[(kSumM * 32 + R) * 4 + nq] = sm[hr];
          sums[(kDenP * 32 + R) * 4 + nq] = dp[hr];
          sums[(kDenM * 32 + R) * 4 + nq] = dm[hr];
          sums[(kSumS * 32 + R) * 4 + nq] = ss[hr];
        }
      }
      const int key = 8 * nq + 2 * t;
      st_shared_u32(sP + R0 * kPitchP + key * 2, pack_bf16(p[0], p[1]));
      st_shared_u32(sP + R1 * kPitchP + key * 2, pack_bf16(p[2], p[3]));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sums_ready[s]);  // row sums are in the stage
    named_bar_sync(1, kConsumers);

    // ---- committing unit: phi(k) = e / sum as bf16 hi + lo (phi = hi + lo to
    //      about 2^-17 relative, so S meets a 1e-4 bound) for the state update,
    //      and the column sums of phi(k) over this warp's 16 tokens for Z
    if (cm) {
      const uint32_t sKHi = smem_u32(st + kOffPhiKHi), sKLo = smem_u32(st + kOffPhiKLo);
      float ip[2], im[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int R = hr ? R1 : R0;
        const float4 a = *reinterpret_cast<const float4*>(sums + (kSumPK * 32 + R) * 4);
        const float4 c = *reinterpret_cast<const float4*>(sums + (kSumMK * 32 + R) * 4);
        ip[hr] = rcp_approx((a.x + a.y) + (a.z + a.w));  // ~1e-7 relative
        im[hr] = rcp_approx((c.x + c.y) + (c.z + c.w));
        if (R >= vrows) ip[hr] = im[hr] = 0.f;  // a row past the block: phi(k) = 0
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * nq + 8 * nt + 2 * t;
        float colp[2] = {0.f, 0.f}, colm[2] = {0.f, 0.f};
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int R = hr ? R1 : R0;
          const float p0 = ekp[nt][2 * hr] * ip[hr], p1 = ekp[nt][2 * hr + 1] * ip[hr];
          const float m0 = ekm[nt][2 * hr] * im[hr], m1 = ekm[nt][2 * hr + 1] * im[hr];
          colp[0] += p0;
          colp[1] += p1;
          colm[0] += m0;
          colm[1] += m1;
          const __nv_bfloat162 hp = __floats2bfloat162_rn(p0, p1);
          const __nv_bfloat162 hm = __floats2bfloat162_rn(m0, m1);
          const float2 fp = __bfloat1622float2(hp), fm = __bfloat1622float2(hm);
          const uint32_t off = sw128(R, c >> 3) + (c & 7) * 2;
          st_shared_u32(sKHi + off, *reinterpret_cast<const uint32_t*>(&hp));
          st_shared_u32(sKHi + 4096 + off, *reinterpret_cast<const uint32_t*>(&hm));
          st_shared_u32(sKLo + off, pack_bf16(p0 - fp.x, p1 - fp.y));
          st_shared_u32(sKLo + 4096 + off, pack_bf16(m0 - fm.x, m1 - fm.y));
        }
        // sum over the 8 row groups g of this warp (lanes with the same t)
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          colp[0] += __shfl_xor_sync(0xffffffffu, colp[0], o2);
          colp[1] += __shfl_xor_sync(0xffffffffu, colp[1], o2);
          colm[0] += __shfl_xor_sync(0xffffffffu, colm[0], o2);
          colm[1] += __shfl_xor_sync(0xffffffffu, colm[1], o2);
        }
        if (g == 0) {
          zpart[mt * 128 + c] = colp[0];
          zpart[mt * 128 + c + 1] = colp[1];
          zpart[mt * 128 + kFH + c] = colm[0];
          zpart[mt * 128 + kFH + c + 1] = colm[1];
        }
      }
      // dS = phi(k)^T V on the tensor cores (M = F = 128, N = d = 128,
      // K = 32 tokens, phi(k) as hi and lo; both operands MN-major in shared
      // memory), running while this unit's state contraction and merge go on
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, kConsumers);
      if (threadIdx.x == 0) {
        tc_fence_after();
        constexpr uint32_t idS = umma_idesc_bf16(128, kD, 1, 1);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t aHi = umma_desc_sw128(sKHi + ks * 2048, 4096, 1024);
          const uint64_t aLo = umma_desc_sw128(sKLo + ks * 2048, 4096, 1024);
          const uint64_t bV = umma_desc_sw128(sV + ks * 2048, 4096, 1024);
          umma_bf16(tbase, aHi, bV, idS, ks > 0 ? 1u : 0u);
          umma_bf16(tbase, aLo, bV, idS, 1u);
        }
        umma_commit(ds_full);
        ++ds_issued;
      }
    }

    // ---- phase D: num+- = e+- S and U = P V for columns 16w .. 16w + 15
    // (a unit with a bad slot, flagged by the producer, runs on stale bytes
    // and writes nothing)
    const bool s_ok = mbar_wait(&s_full[s], n & 1, lim);
    const int valid = meta[s];  // read before the stage is handed back
    float acc_p[2][2][4] = {}, acc_m[2][2][4] = {}, acc_v[2][2][4] = {};
    {
      const int col = c0 + 2 * g;  // and col + 1: columns g of n-tiles 0 and 1
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
        uint32_t b00, b01, b10, b11;
        if (kS8) {
          // codes S[k][col], S[k][col + 1] share a 16-bit word; regroup by
          // column ({S[k][c], S[k + 1][c]}) and widen to f16 pairs
          const uint32_t h0 = ld_shared_u16(sS + s8_off(k0, col));
          const uint32_t h1 = ld_shared_u16(sS + s8_off(k0 + 1, col));
          const uint32_t h8 = ld_shared_u16(sS + s8_off(k0 + 8, col));
          const uint32_t h9 = ld_shared_u16(sS + s8_off(k0 + 9, col));
          const uint32_t p01 = __byte_perm(h0, h1, 0x5140), p89 = __byte_perm(h8, h9, 0x5140);
          b00 = e4m3x2_to_f16x2(p01);
          b10 = e4m3x2_to_f16x2(p01 >> 16);
          b01 = e4m3x2_to_f16x2(p89);
          b11 = e4m3x2_to_f16x2(p89 >> 16);
        } else if (kS16 && !cm) {
          // the same operands as below: S[k][col], S[k][col + 1] share a word
          const uint32_t w0 = ld_shared_u32(sS + s16_off(k0, col));
          const uint32_t w1 = ld_shared_u32(sS + s16_off(k0 + 1, col));
          const uint32_t w8 = ld_shared_u32(sS + s16_off(k0 + 8, col));
          const uint32_t w9 = ld_shared_u32(sS + s16_off(k0 + 9, col));
          b00 = __byte_perm(w0, w1, 0x5410);
          b01 = __byte_perm(w8, w9, 0x5410);
          b10 = __byte_perm(w0, w1, 0x7632);
          b11 = __byte_perm(w8, w9, 0x7632);
        } else {
          const float2 r0 = ld_shared_v2f(sS + s_off(k0, col));
          const float2 r1 = ld_shared_v2f(sS + s_off(k0 + 1, col));
          const float2 r8 = ld_shared_v2f(sS + s_off(k0 + 8, col));
          const float2 r9 = ld_shared_v2f(sS + s_off(k0 + 9, col));
          b00 = pack_bf16(r0.x, r1.x);
          b01 = pack_bf16(r8.x, r9.x);
          b10 = pack_bf16(r0.y, r1.y);
          b11 = pack_bf16(r8.y, r9.y);
        }
        float (&acc)[2][2][4] = kk < 4 ? acc_p : acc_m;
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          if (kS8) {
            mma_f16(acc[m2][0], a[m2], b00, b01);
            mma_f16(acc[m2][1], a[m2], b10, b11);
          } else {
            mma_bf16(acc[m2][0], a[m2], b00, b01);
            mma_bf16(acc[m2][1], a[m2], b10, b11);
          }
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int key = 16 * kk + 2 * t;
        const uint32_t w0 = ld_shared_u32(sV + v_off(key, col));
        const uint32_t w1 = ld_shared_u32(sV + v_off(key + 1, col));
        const uint32_t w8 = ld_shared_u32(sV + v_off(key + 8, col));
        const uint32_t w9 = ld_shared_u32(sV + v_off(key + 9, col));
        const uint32_t b00 = __byte_perm(w0, w1, 0x5410), b01 = __byte_perm(w8, w9, 0x5410);
        const uint32_t b10 = __byte_perm(w0, w1, 0x7632), b11 = __byte_perm(w8, w9, 0x7632);
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          uint32_t a[4];
          const int arow = 16 * m2 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ch = 2 * kk + (lane >> 4);
          ldsm_x4(sP + arow * kPitchP + ch * 16, a[0], a[1], a[2], a[3]);
          mma_bf16(acc_v[m2][0], a, b00, b01);
          mma_bf16(acc_v[m2][1], a, b10, b11);
        }
      }
    }
    // the stage is no longer read: hand it back to the producer (a
    // committing unit keeps it until its new S has been stored)
    // (only once this lane has seen the stage's loads land: after a wait that
    // ran out, the stage is never handed back, so no copy is issued into it
    // while an earlier one may still be landing)
    bool release_ok = s_ok;
    if (kSeq && cm) {
      // the stage's V and phi(k) are read by the dS MMA; once it is done,
      // the stage (q, k, v, W_h) is free: the state lives elsewhere
      const bool ds_ok = mbar_wait(ds_full, cm_phase, lim);
      cm_phase ^= 1u;
      if (!ds_ok) {
        late_fail = true;
        release_ok = false;
        if (lane == 0) atomicOr(status, kStatusTimeout);
      }
    }
    __syncwarp();
    if (lane == 0 && (kSeq || !cm) && release_ok) mbar_arrive(&empty[s]);
    if (!s_ok) {
      late_fail = true;  // voted on at the next unit's first barrier
      if (lane == 0) atomicOr(status, kStatusTimeout);
    }
    if (!(valid & kUnitValid)) continue;
    if (!mbar_wait(&fin_ready[s], n & 1, lim)) {
      late_fail = true;
      if (lane == 0) atomicOr(status, kStatusTimeout);
    }
    const float* fin = fin_all + s * 96;

    // ---- merge and store o: thread holds columns c0 + 4t .. c0 + 4t + 3
#pragma unroll
    for (int m2 = 0; m2 < 2; ++m2) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int R = 16 * m2 + g + 8 * hr;
        const float cU = fin[R], cP = fin[32 + R], cM = fin[64 + R];
        float ov[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = q & 1, e = 2 * hr + (q >> 1);
          ov[q] = fmaf(cU, acc_v[m2][j][e], fmaf(cP, acc_p[m2][j][e], cM * acc_m[m2][j][e]));
        }
        uint2 pk;
        pk.x = pack_bf16(ov[0], ov[1]);
        pk.y = pack_bf16(ov[2], ov[3]);
        const size_t orow =
            (size_t)b * maps.rows_per_req + (kSeq ? i * kL : maps.row_base) + R;
        if (R < vrows) *reinterpret_cast<uint2*>(o + (orow * H + h) * kD + c0 + 4 * t) = pk;
      }
    }

    // ---- committing unit (after its output used the old state):
    //      S += phi(k)^T V with phi(k) = hi + lo, Z += sum_t phi(k_t); the new
    //      state is written over the old one in the stage and stored by TMA.
    //      Warp w produces F rows 16w .. 16w + 15, all 128 columns.
    if (cm) {
      // dS rows F = 32 (w % 4) + lane (this warp's TMEM lane quarter),
      // columns 64 (w / 4) .. 64 (w / 4) + 63, added to the staged old S,
      // once every warp's state contraction has finished reading it
      named_bar_sync(1, kConsumers);
      if (!kSeq) {
        const bool ds_ok = mbar_wait(ds_full, cm_phase, lim);
        cm_phase ^= 1u;
        if (!ds_ok) {
          late_fail = true;
          if (lane == 0) atomicOr(status, kStatusTimeout);
        }
      }
      tc_fence_after();
      const int F = 32 * (warp & 3) + lane;
      const int n0 = 64 * (warp >> 2);
      const uint32_t lane_bits = (uint32_t)(32 * (warp & 3)) << 16;
      const uint32_t sS16New = smem_u32(st + kOffS16New);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float r[32];
        tmem_ld32(tbase + lane_bits + n0 + 32 * part, r);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const int n = n0 + 32 * part + 4 * q4;
          const uint32_t a = sS + s_off(F, n);
          const float4 old = ld_shared_v4f(a);
          const float4 nw = make_float4(old.x + r[4 * q4], old.y + r[4 * q4 + 1],
                                        old.z + r[4 * q4 + 2], old.w + r[4 * q4 + 3]);
          st_shared_v4(a, __float_as_uint(nw.x), __float_as_uint(nw.y), __float_as_uint(nw.z),
                       __float_as_uint(nw.w));
          if (kDual)  // the copy: round to nearest, as hb_state_to_bf16 does
            st_shared_v2u(sS16New + s16_off(F, n), pack_bf16(nw.x, nw.y), pack_bf16(nw.z, nw.w));
        }
      }
      tc_fence_before();
      if (threadIdx.x < kF) sZ[threadIdx.x] += zpart[threadIdx.x] + zpart[128 + threadIdx.x];
      // the coefficient warp stores the new state and releases the stage
      // (sequential mode: stores it after the prompt's last block)
      if (!kSeq || (flags & kUnitLast)) {
        fence_proxy_async_smem();
        __syncwarp();
        // (not after the stage's state load ran out: the coefficient warp's
        // wait then runs out too, and the stage is never refilled)
        if (lane == 0 && s_ok) mbar_arrive(&s_updated[s]);
      }
    }
  }
  (void)aborted;
  }  // consumers

  // Every warp has left its loop (each wait is bounded), so the producer has
  // issued everything it will. A stage is refilled only after its previous
  // loads were seen to land, so only the last unit issued into each stage can
  // still have copies in flight: wait for those (full limit) so that no copy
  // lands in the shared memory of an exited CTA, and for the last dS MMA
  // before its tensor memory is freed.
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = *n_issued;
    for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) {
      mbar_wait(&head_full[j & 1], (j >> 1) & 1);
      mbar_wait(&s_full[j & 1], (j >> 1) & 1);
    }
    if (kCommit && ds_issued > 0) mbar_wait(ds_full, (uint32_t)(ds_issued - 1) & 1u);
  }
  if (kCommit && warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

}  // namespace

bool fast_attend_ok(const Shape& s) { return production_shape(s); }

bool fast_attend_step_ok(const Shape& s) {
  Shape s32 = s;
  s32.L = kL;
  return production_shape(s32) && (s.L == kL || s.L == 16);
}

bool attend_fast_fits(const Shape& s, int batch, int num_slots, int64_t rows_per_req) {
  return (int64_t)num_slots * s.H * kF < ((int64_t)1 << 31) &&
         (int64_t)batch * rows_per_req < ((int64_t)1 << 31);
}

namespace {

// Every entry point: S_pool is the fp32 pool, or with state_bf16 and no
// commit its bf16 copy (attend only). S16_pool (dual-copy step, with a
// commit mask): the bf16 copies beside the fp32 masters in S_pool.
cudaError_t launch_attend_impl(const Shape& s, int batch, const int32_t* slot_idx, const void* q,
                               const void* k, const void* v, const void* S_pool,
                               const float* Z_pool, int num_slots, const void* W,
                               const float* gate, const int32_t* commit_mask, void* o,
                               unsigned* status, cudaStream_t st, int rows_per_req, int row_base,
                               bool commit_all, bool sequential, bool state_bf16,
                               void* S16_pool = nullptr, int Hkv = -1,
                               const void* Wk = nullptr, const float* s8_scale = nullptr,
                               int n_layers = 1) {
  const bool dual = S16_pool != nullptr;
  // the fp8 copy (with its per-(slot, head) scales) is read by the attend only
  const bool fp8 = s8_scale != nullptr;
  if (fp8 && (commit_mask || commit_all || sequential || dual || state_bf16))
    return cudaErrorInvalidValue;
  if (Hkv <= 0) Hkv = s.H;
  // grouped heads in the attend-only kernels; a separate key map in the
  // sequential mode
  if (s.H % Hkv != 0 || (Hkv != s.H && (commit_mask || commit_all || sequential || dual)))
    return cudaErrorInvalidValue;
  const bool sep_wk = Wk != nullptr && Wk != W;
  if (sep_wk && !sequential) return cudaErrorInvalidValue;
  // blocks of 16 tokens in a decoding step; prompts walk 32-token blocks
  if (sequential ? s.L != kL : (s.L != kL && s.L != 16)) return cudaErrorInvalidValue;
  // independent layers: batch = n_layers x the requests of one layer
  if (n_layers < 1 || batch % n_layers != 0 || (n_layers > 1 && sequential))
    return cudaErrorInvalidValue;
  Maps maps;
  maps.n_layers = n_layers;
  maps.reqs_per_layer = batch > 0 ? batch / n_layers : 1;
  maps.valid_rows = sequential ? kL : s.L;
  maps.kv_group = s.H / Hkv;
  maps.sep_wk = sep_wk ? 1 : 0;
  maps.s16 = static_cast<const uint8_t*>(S16_pool);
  maps.s8_scale = s8_scale;
  maps.rows_per_req = rows_per_req;
  maps.wait_limit = wait_limit_cycles();
  maps.row_base = row_base;
  maps.commit_all = commit_all ? 1 : 0;
  maps.qkv[0] = static_cast<const uint8_t*>(q);
  maps.qkv[1] = static_cast<const uint8_t*>(k);
  maps.qkv[2] = static_cast<const uint8_t*>(v);
  maps.w = static_cast<const uint8_t*>(W);
  {
    // bytes per value: fp32 master 4, bf16 copy 2, fp8 copy 1; a box row is
    // 128 bytes (SWIZZLE_128B) of 128 F rows
    const int vb = fp8 ? 1 : state_bf16 ? 2 : 4;
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)num_slots * Hkv * kF};
    const uint64_t strides[1] = {(uint64_t)kD * vb};
    const uint32_t box[2] = {(uint32_t)(128 / vb), 128};
    const CUtensorMapDataType dt = fp8          ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : state_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (!encode_tmap(&maps.S, dt, 2, S_pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    maps.S16 = maps.S;  // unused unless dual
  }
  if (dual) {
    const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)num_slots * s.H * kF};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box[2] = {64u, 128};
    if (!encode_tmap(&maps.S16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, S16_pool, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // q with H heads; k, v with Hkv
    const uint32_t box[3] = {64, 1, 32};
    const void* ptrs[3] = {q, k, v};
    CUtensorMap* dst[3] = {&maps.q, &maps.k, &maps.v};
    for (int j = 0; j < 3; ++j) {
      const uint64_t heads = j == 0 ? (uint64_t)s.H : (uint64_t)Hkv;
      const uint64_t dims[3] = {(uint64_t)kD, heads, (uint64_t)batch * rows_per_req};
      const uint64_t strides[2] = {kD * 2, heads * kD * 2};
      if (!encode_tmap(dst[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptrs[j], dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
  }
  {
    const uint64_t dims[2] = {(uint64_t)kFH, (uint64_t)n_layers * s.H * kD};
    const uint64_t strides[1] = {kFH * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap(&maps.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    maps.Wk = maps.W;
    if (sep_wk && !encode_tmap(&maps.Wk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wk, dims, strides,
                               box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  auto* kernel = dual         ? k_attend_fast<true, false, true>
                 : fp8        ? k_attend_fast<false, false, false, true>
                 : state_bf16 ? k_attend_fast<false, false, true>
                 : sequential ? k_attend_fast<true, true>
                 : (commit_mask || commit_all) ? k_attend_fast<true> : k_attend_fast<false>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  int num_sms = 0;
  if ((e = current_sm_count(&num_sms)) != cudaSuccess) return e;
  const int units = batch * s.H;
  // persistent grid over the units, or one CTA per (request, head) walking
  // its prompt's blocks in order
  const int grid = sequential ? units : (units < num_sms ? units : num_sms);
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, maps, batch, s.H,
                    num_slots, s.scale * kLog2e, s.merge, slot_idx, commit_mask,
                    static_cast<const float*>(S_pool), const_cast<float*>(Z_pool), gate,
                    reinterpret_cast<__nv_bfloat16*>(o), status);
}

}  // namespace

cudaError_t launch_attend_commit_dual(const Shape& s, int batch, const int32_t* slot_idx,
                                      const void* q, const void* k, const void* v, float* S_pool,
                                      void* S16_pool, float* Z_pool, int num_slots, const void* W,
                                      const float* gate, const int32_t* commit_mask, void* o,
                                      unsigned* status, cudaStream_t st) {
  return launch_attend_impl(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, W, gate,
                            commit_mask, o, status, st, s.L, 0, false, false, false, S16_pool);
}

cudaError_t launch_attend_fast(const Shape& s, int batch, const int32_t* slot_idx, const void* q,
                               const void* k, const void* v, const float* S_pool,
                               const float* Z_pool, int num_slots, const void* W,
                               const float* gate, const int32_t* commit_mask, void* o,
                               unsigned* status, cudaStream_t st, int rows_per_req, int row_base,
                               bool commit_all, bool sequential, int Hkv, const void* Wk) {
  return launch_attend_impl(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, W, gate,
                            commit_mask, o, status, st, rows_per_req, row_base, commit_all,
                            sequential, false, nullptr, Hkv, Wk);
}

cudaError_t launch_attend_layers(const Shape& s, int n_layers, int batch, const int32_t* slot_idx,
                                 const void* q, const void* k, const void* v, float* S_pool,
                                 float* Z_pool, int num_slots, const void* W, const float* gate,
                                 const int32_t* commit_mask, void* o, unsigned* status,
                                 cudaStream_t st) {
  return launch_attend_impl(s, batch, slot_idx, q, k, v, S_pool, Z_pool, num_slots, W, gate,
                            commit_mask, o, status, st, s.L, 0, false, false, false, nullptr, -1,
                            nullptr, nullptr, n_layers);
}

cudaError_t launch_attend_fast_s16(const Shape& s, int batch, const int32_t* slot_idx,
                                   const void* q, const void* k, const void* v,
                                   const void* S16_pool, const float* Z_pool, int num_slots,
                                   const void* W, const float* gate, void* o, unsigned* status,
                                   cudaStream_t st) {
  return launch_attend_impl(s, batch, slot_idx, q, k, v, S16_pool, Z_pool, num_slots, W, gate,
                            nullptr, o, status, st, s.L, 0, false, false, true);
}

cudaError_t launch_attend_fast_s8(const Shape& s, int batch, const int32_t* slot_idx,
                                  const void* q, const void* k, const void* v,
                                  const void* S8_pool, const float* scale_pool,
                                  const float* Z_pool, int num_slots, const void* W,
                                  const float* gate, void* o, unsigned* status,
                                  cudaStream_t st) {
  return launch_attend_impl(s, batch, slot_idx, q, k, v, S8_pool, Z_pool, num_slots, W, gate,
                            nullptr, o, status, st, s.L, 0, false, false, false, nullptr, -1,
                            nullptr, scale_pool);
}

}  // namespace hb
