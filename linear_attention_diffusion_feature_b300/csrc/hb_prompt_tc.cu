// Prompt with outputs for the production shape (bf16, d = 128, f = 64,
// F = 128, L = 32), chunked onto the 5th-generation tensor cores.
//
// What is computed (gist.science technical summary of arXiv 2608.06628,
// "Methodology: Block-Hybrid Attention / Architecture Design", all four
// bullets; pith.science review, "What carries the argument"): the prompt is
// a sequence of L-token blocks; block j attends with exact softmax inside
// itself and linearly to the state of blocks 0 .. j - 1, and is then
// committed: S += sum_t phi(k_t) v_t^T, Z += sum_t phi(k_t).
//
// The state after block j - 1 is the state at the start of the block's
// 128-token segment plus the sums over the segment's earlier blocks, and
// phi(q)^T sum_t phi(k_t) v_t^T = sum_t (phi(q) . phi(k_t)) v_t. So one
// segment of four blocks needs only dense 128 x 128 products:
//   U_q = Q W,  U_k = K W           (then the two softmaxes: phi(Q), phi(K))
//   Sc  = Q K^T                      (block scores; the 32 x 32 diagonal blocks are used)
//   A   = phi(Q) phi(K)^T            (weights of the segment's earlier blocks)
//   O2  = phi(Q) S_start             (the linear read of the state at segment start)
//   S  += phi(K)^T V                 (phi(K) as bf16 hi + lo; the fp32 state stays in TMEM)
//   O1  = C V,  C = cU * P (own block) + cN * A (earlier blocks), 0 elsewhere
//   o   = O1 + cN * O2
// with the per-row merge coefficients cU, cN of the gated merge (shared
// normaliser or convex). Every product runs as tcgen05.mma with M = 128 and
// an fp32 accumulator in tensor memory; the state lives in tensor memory for
// the whole prompt, with a bf16 copy in shared memory as the operand of the
// next segment's read.
//
// One CTA per (request, head), 18 warps: warp 0 loads (TMA), warp 1 owns
// tensor memory and issues every MMA from one thread, warps 2-17 are the
// epilogue (thread = token row of the segment x one quarter of the columns).
#include <float.h>

#include "hb_fast.cuh"
#include "hb_ptx.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kFH = 64, kF = 128, kSeg = 128;  // four 32-token blocks per segment
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // loader, MMA issuer, epilogue

// Shared memory (bytes from a 1024-aligned base). Every 128-row bf16 tile is
// two SWIZZLE_128B boxes of [128 rows][64 columns] (16 KiB each).
constexpr int kOffW = 0;                 // W_h [d rows][f]
constexpr int kOffQ = 16384;             // Q, then phi(Q)
constexpr int kOffK = kOffQ + 32768;     // K, then phi(K) hi
constexpr int kOffKlo = kOffK + 32768;   // phi(K) lo, then C, then the outputs o
constexpr int kOffV = kOffKlo + 32768;   // V, two buffers
constexpr int kOffS16 = kOffV + 65536;   // bf16 copy of the state [F rows][d]
constexpr int kOffX = kOffS16 + 32768;   // exchange: 4 arrays of [4 quarters][128 rows] fp32
constexpr int kOffXden = kOffX + 8192;   // [4][128]: phi(q) . Z partial sums
constexpr int kOffXm = kOffXden + 2048;  // [4][128]: partial row max of the own block's scores
constexpr int kOffXP = kOffXm + 2048;    // [4][128]: the matching partial sums
constexpr int kOffZ = kOffXP + 2048;     // [128]: Z
constexpr int kOffZq = kOffZ + 512;      // [4][128]: the segment's column sums of phi(K)
constexpr int kOffBar = kOffZq + 2048;
constexpr int kNumBars = 16;
constexpr int kSmemUsed = kOffBar + kNumBars * 8 + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory over the sm_100 per-block limit");

enum { kBarW = 0, kBarQ, kBarK, kBarV0, kBarV1, kBarUq, kBarUk, kBarPhi, kBarL, kBarC, kBarO,
       kBarE, kBarSc, kBarUpd, kBarPhiQ, kBarDone };

// tensor-memory columns (512 allocated; lane = row of every accumulator)
constexpr uint32_t kColM = 0;    // the state S [F][d], fp32, for the whole prompt
constexpr uint32_t kColU = 128;  // O2 (128)
constexpr uint32_t kColS = 256;  // block scores; later O1
constexpr uint32_t kColA = 384;  // U_q (64) and U_k (64); later phi(Q) phi(K)^T

struct Maps {
  CUtensorMap q, k, v;  // [B*T rows][H][d] bf16, box {64, 1, 128}
  CUtensorMap W;        // [H*d rows][f] bf16, box {64, 128}
  CUtensorMap o;        // [B][T][H][d] bf16, box {64, 1, 128, 1}: stores clip at T
};

// Shared -> global copy of one box of a 4-D tensor map (bulk async-group).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, int x, int y, int z, int w,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          map),
      "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(src))
      : "memory");
}

struct Args {
  int H, num_slots, merge;
  // request b's final state is written back when commit_all or
  // commit_mask[b] != 0 (otherwise the slot is only read)
  int commit_all;
  const int32_t* commit_mask;
  int64_t T;  // prompt length (a multiple of 32)
  float scale_log2;
  const int32_t* slot_idx;
  float* S_pool;
  float* Z_pool;
  const float* gate;
  __nv_bfloat16* o;
  const uint8_t* qkv[3];  // base addresses for L2 prefetch
  unsigned* status;
  long long wait_limit;  // pipeline waits (hb_set_wait_limit); drains take the default
};

// K-major operand: 16-element step ks of the contraction within two boxes
// of [128 rows][64 columns].
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int ks) {
  return umma_desc_sw128(base + (ks >> 2) * 16384 + (ks & 3) * 32, 0, 1024);
}
// MN-major operand: 16 contraction rows per step, 64-column boxes 16 KiB apart.
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int ks) {
  return umma_desc_sw128(base + ks * 2048, 16384, 1024);
}
// Byte offset of 16-byte chunk c (0..15 over the 128 columns) of row r in a
// two-box tile.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// kBL: the block length L (16, 32 or 64), a divisor of the 128-token
// segment; row r of a segment is in block r / kBL.
// 18 warps put five on two of the four sub-partitions, whose 16 Ki
// registers then allow at most 102 per thread: capped at 96.
template <int kBL>
__global__ void __maxnreg__(96)
    k_prompt_tc(const __grid_constant__ Maps maps, const __grid_constant__ Args a) {
  static_assert(kBL == 16 || kBL == 32 || kBL == 64, "block length");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = (int)blockIdx.x / a.H, h = (int)blockIdx.x - b * a.H;
  const int slot = a.slot_idx[b];
  if (slot < 0 || slot >= a.num_slots) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
    return;
  }
  const int n_seg = (int)((a.T + kSeg - 1) / kSeg);
  const size_t unit = (size_t)slot * a.H + h;
  const bool commits = a.commit_all != 0 || (a.commit_mask != nullptr && a.commit_mask[b] != 0);

  if (threadIdx.x == 0) {
    mbar_init(&bar[kBarW], 1);
    mbar_init(&bar[kBarQ], 1);
    mbar_init(&bar[kBarK], 1);
    mbar_init(&bar[kBarV0], 1);
    mbar_init(&bar[kBarV1], 1);
    mbar_init(&bar[kBarUq], 1);
    mbar_init(&bar[kBarUk], 1);
    mbar_init(&bar[kBarPhi], kEpiWarps);
    mbar_init(&bar[kBarL], 1);
    mbar_init(&bar[kBarC], kEpiWarps);
    mbar_init(&bar[kBarO], 1);
    mbar_init(&bar[kBarE], kEpiWarps);
    mbar_init(&bar[kBarSc], 1);
    mbar_init(&bar[kBarUpd], 1);
    mbar_init(&bar[kBarPhiQ], kEpiWarps);
    mbar_init(&bar[kBarDone], 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t sW = smem_u32(smem + kOffW), sQ = smem_u32(smem + kOffQ);
  const uint32_t sK = smem_u32(smem + kOffK), sKlo = smem_u32(smem + kOffKlo);
  const uint32_t sV = smem_u32(smem + kOffV), sS16 = smem_u32(smem + kOffS16);

  if (warp == 0) {
    // ------------------------------------------------------------- loader
    if (lane == 0) {
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      prefetch_tmap(&maps.W);
      mbar_arrive_expect_tx(&bar[kBarW], 16384);
      tma_load_2d(smem + kOffW, &maps.W, 0, h * kD, &bar[kBarW]);
      const int64_t base_row = (int64_t)b * a.T;
      // a segment's rows of all heads are contiguous: this CTA prefetches a
      // 1/H slice of them into L2, the request's other heads the rest
      auto l2 = [&](int s) {
        if (s >= n_seg) return;
        const int64_t r0 = base_row + (int64_t)s * kSeg;
        const int64_t rows = a.T - (int64_t)s * kSeg < kSeg ? a.T - (int64_t)s * kSeg : kSeg;
        const size_t bytes = (size_t)rows * kD * 2;  // = rows * H * d * 2 / H
        const size_t off = (size_t)r0 * a.H * kD * 2 + (size_t)h * bytes;
#pragma unroll
        for (int j = 0; j < 3; ++j) prefetch_l2(a.qkv[j] + off, (uint32_t)bytes);
      };
      int n_q = 0, n_k = 0, n_v0 = 0, n_v1 = 0;  // loads issued, for the final drain
      auto load_q = [&](int s) {
        const int row = (int)(base_row + (int64_t)s * kSeg);
        ++n_q;
        mbar_arrive_expect_tx(&bar[kBarQ], 32768);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem + kOffQ + j * 16384, &maps.q, 64 * j, h, row, &bar[kBarQ]);
      };
      auto load_k = [&](int s) {
        const int row = (int)(base_row + (int64_t)s * kSeg);
        ++n_k;
        mbar_arrive_expect_tx(&bar[kBarK], 32768);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem + kOffK + j * 16384, &maps.k, 64 * j, h, row, &bar[kBarK]);
      };
      auto load_v = [&](int s) {
        const int row = (int)(base_row + (int64_t)s * kSeg);
        uint64_t* vb = &bar[kBarV0 + (s & 1)];
        if (s & 1) ++n_v1; else ++n_v0;
        mbar_arrive_expect_tx(vb, 32768);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem + kOffV + (s & 1) * 32768 + j * 16384, &maps.v, 64 * j, h, row, vb);
      };
      if (n_seg > 0) {
        load_q(0);
        load_k(0);
        load_v(0);
        if (n_seg > 1) load_v(1);
        l2(1);
        l2(2);
      }
      for (int s = 1; s < n_seg; ++s) {
        // phi(Q) of the segment before, over its Q, has been read once its
        // A and O2 are done; phi(K) once its state update is done too; its
        // V buffer once O1 is done
        if (!mbar_wait(&bar[kBarL], (s - 1) & 1, a.wait_limit)) {
          atomicOr(a.status, kStatusTimeout);
          break;
        }
        load_q(s);
        if (!mbar_wait(&bar[kBarUpd], (s - 1) & 1, a.wait_limit)) {
          atomicOr(a.status, kStatusTimeout);
          break;
        }
        load_k(s);
        l2(s + 2);
        if (s + 1 < n_seg) {
          if (!mbar_wait(&bar[kBarO], (s - 1) & 1, a.wait_limit)) {
            atomicOr(a.status, kStatusTimeout);
            break;
          }
          load_v(s + 1);
        }
      }
      // no copy may land in the shared memory of an exited CTA: wait for the
      // last one issued on each barrier (immediate when already consumed)
      if (n_q > 0) mbar_wait(&bar[kBarQ], (n_q - 1) & 1);
      if (n_k > 0) mbar_wait(&bar[kBarK], (n_k - 1) & 1);
      if (n_v0 > 0) mbar_wait(&bar[kBarV0], (n_v0 - 1) & 1);
      if (n_v1 > 0) mbar_wait(&bar[kBarV1], (n_v1 - 1) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0 && n_seg > 0) {
      constexpr uint32_t idU = umma_idesc_bf16(128, kFH, 0, 1);  // A K-major, B MN-major
      constexpr uint32_t idKK = umma_idesc_bf16(128, 128, 0, 0);  // both K-major
      constexpr uint32_t idKM = umma_idesc_bf16(128, 128, 0, 1);  // A K-major, B MN-major
      constexpr uint32_t idMM = umma_idesc_bf16(128, 128, 1, 1);  // both MN-major
      const long long lim = a.wait_limit;
      // U_q = Q W and U_k = K W of segment s, into the A columns, each
      // issued once its operand has landed
      auto issue_u = [&](int s) -> bool {
        if (!mbar_wait(&bar[kBarQ], s & 1, lim)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tbase + kColA, desc_k(sQ, ks), desc_mn(sW, ks), idU, ks > 0 ? 1u : 0u);
        umma_commit(&bar[kBarUq]);
        if (!mbar_wait(&bar[kBarK], s & 1, lim)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tbase + kColA + 64, desc_k(sK, ks), desc_mn(sW, ks), idU, ks > 0 ? 1u : 0u);
        umma_commit(&bar[kBarUk]);
        return true;
      };
      // Segment s's U_q is issued once the A columns are free (segment
      // s - 1's C is written) and its Q has landed (loaded once s - 1's A and
      // O2 have read phi(Q)); U_k once its K has landed (after s - 1's state
      // update). Both run while the epilogue forms s - 1's outputs; the
      // scores Sc wait for those outputs to be read (the S columns) and run
      // while the epilogue forms s's feature maps, which overwrite Q and K
      // only after Sc has read them.
      bool ok = mbar_wait(&bar[kBarW], 0, lim);
      if (ok) ok = issue_u(0);
      for (int s = 0; ok && s < n_seg; ++s) {
        const uint32_t vb = sV + (s & 1) * 32768;
        if (s > 0 && !(ok = mbar_wait(&bar[kBarE], (s - 1) & 1, lim))) break;  // O1, O2 of s - 1 read
        tc_fence_after();
        // Sc = Q K^T
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tbase + kColS, desc_k(sQ, ks), desc_k(sK, ks), idKK, ks > 0 ? 1u : 0u);
        umma_commit(&bar[kBarSc]);
        // phi(Q) written by the epilogue: O2 = phi(Q) S_start runs while it
        // forms phi(K)
        if (!(ok = mbar_wait(&bar[kBarPhiQ], s & 1, lim))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tbase + kColU, desc_k(sQ, ks), desc_mn(sS16, ks), idKM, ks > 0 ? 1u : 0u);
        // phi(K) written; V landed
        ok = mbar_wait(&bar[kBarPhi], s & 1, lim);
        if (ok) ok = mbar_wait(&bar[kBarV0 + (s & 1)], (s >> 1) & 1, lim);
        if (!ok) break;
        tc_fence_after();
        // A = phi(Q) phi(K)^T (with O2, what the epilogue's merge needs);
        // then S += phi(K)^T V (hi + lo), which runs while it forms C
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tbase + kColA, desc_k(sQ, ks), desc_k(sK, ks), idKK, ks > 0 ? 1u : 0u);
        umma_commit(&bar[kBarL]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          umma_bf16(tbase + kColM, desc_mn(sK, ks), desc_mn(vb, ks), idMM, 1u);
          umma_bf16(tbase + kColM, desc_mn(sKlo, ks), desc_mn(vb, ks), idMM, 1u);
        }
        umma_commit(&bar[kBarUpd]);
        // C written by the epilogue (over the state copy O2 has read): O1 = C V
        if (!(ok = mbar_wait(&bar[kBarC], s & 1, lim))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tbase + kColS, desc_k(sS16, ks), desc_mn(vb, ks), idKM, ks > 0 ? 1u : 0u);
        umma_commit(&bar[kBarO]);
        // the next segment's U (A has been read; its Q, K load after L)
        if (s + 1 < n_seg && !(ok = issue_u(s + 1))) break;
      }
      if (!ok) atomicOr(a.status, kStatusTimeout);
      // every MMA issued has completed before tensor memory is freed
      umma_commit(&bar[kBarDone]);
      mbar_wait(&bar[kBarDone], 0);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // Thread: row r = 32 quad + lane of the segment (a token; for the state,
    // an F index) and column quarter sub (16 of the 64 columns of u, or 32 of
    // the 128 columns of the other accumulators). Row r's block in the
    // segment is r / 32 = quad.
    const int quad = warp & 3, ew = warp - 2, sub = ew >> 2;
    const int r = 32 * quad + lane;
    const uint32_t lane_bits = (uint32_t)(32 * quad) << 16;
    float* xa = reinterpret_cast<float*>(smem + kOffX);
    float* xb = xa + 512;
    float* xc = xb + 512;
    float* xd = xc + 512;
    float* xden = reinterpret_cast<float*>(smem + kOffXden);
    float* xm = reinterpret_cast<float*>(smem + kOffXm);
    float* xP = reinterpret_cast<float*>(smem + kOffXP);
    float* Zs = reinterpret_cast<float*>(smem + kOffZ);
    float* zq = reinterpret_cast<float*>(smem + kOffZq);
    const float gl = a.gate[h];
    bool ok = true;

    // the state at the start of the prompt: fp32 into tensor memory, its
    // bf16 copy into shared memory, Z into shared memory
    {
      const float4* src = reinterpret_cast<const float4*>(a.S_pool + unit * kF * kD + r * kD + 32 * sub);
      float v32[32];
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 t = src[q4];
        v32[4 * q4] = t.x;
        v32[4 * q4 + 1] = t.y;
        v32[4 * q4 + 2] = t.z;
        v32[4 * q4 + 3] = t.w;
      }
      tmem_st32(tbase + lane_bits + kColM + 32 * sub, v32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        st_shared_v4(sS16 + tile_off(r, 4 * sub + q4), pack_bf16(v32[8 * q4], v32[8 * q4 + 1]),
                     pack_bf16(v32[8 * q4 + 2], v32[8 * q4 + 3]),
                     pack_bf16(v32[8 * q4 + 4], v32[8 * q4 + 5]),
                     pack_bf16(v32[8 * q4 + 6], v32[8 * q4 + 7]));
      if (sub == 0) Zs[r] = a.Z_pool[unit * kF + r];
      tmem_wait_st();
    }

    for (int s = 0; s < n_seg; ++s) {
      const int64_t valid64 = a.T - (int64_t)s * kSeg;
      const int valid = valid64 < kSeg ? (int)valid64 : kSeg;
      const bool live = r < valid;
      // ---- E1: the feature maps of the segment's queries and keys
      if (ok) ok = mbar_wait(&bar[kBarUq], s & 1, a.wait_limit);
      tc_fence_after();
      float u[16];
      // phi(x) = [softmax(u), softmax(-u)] over the 64 columns of u, shared
      // by the four threads of the row: row max, min and sums exchanged
      float ph[32];
      auto softmaxes = [&]() {
        // the row's max and min first (its four threads' partial ones
        // exchanged), so every exponential is taken against the row's own
        // bound and the sums need no rescaling; then the sums are exchanged
        float mx = -FLT_MAX, mn = FLT_MAX;
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          mx = fmax3(mx, u[j], u[j + 1]);
          mn = fmin3(mn, u[j], u[j + 1]);
        }
        xa[sub * 128 + r] = mx;
        xb[sub * 128 + r] = mn;
        named_bar_sync(1, 32 * kEpiWarps);
        mx = fmax3(fmax3(mx, xa[r], xa[128 + r]), xa[256 + r], xa[384 + r]);
        mn = fmin3(fmin3(mn, xb[r], xb[128 + r]), xb[256 + r], xb[384 + r]);
        const float opx = -mx * kLog2e, omn = mn * kLog2e;
        float sp = 0.f, sm = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          ph[j] = ex2_approx(fmaf(u[j], kLog2e, opx));
          ph[16 + j] = ex2_approx(fmaf(u[j], -kLog2e, omn));
          sp += ph[j];
          sm += ph[16 + j];
        }
        xc[sub * 128 + r] = sp;
        xd[sub * 128 + r] = sm;
        named_bar_sync(1, 32 * kEpiWarps);
        // row totals of e^{u - max} and e^{min - u} (each >= 1), in a fixed order
        const float tp = (xc[r] + xc[128 + r]) + (xc[256 + r] + xc[384 + r]);
        const float tm = (xd[r] + xd[128 + r]) + (xd[256 + r] + xd[384 + r]);
        const float cp = rcp_approx(tp), cm = rcp_approx(tm);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          ph[j] *= cp;
          ph[16 + j] *= cm;
        }
        // slot reuse: xa and xb are written again only after the second
        // barrier (every thread has read them before it), xc and xd only
        // after the next call's first barrier (likewise)
      };
      // queries: phi(Q) (bf16) over Q, and phi(q) . Z of this thread's columns
      tmem_ld16(tbase + lane_bits + kColA + 16 * sub, u);
      tmem_wait_ld();
      softmaxes();
      // Q and K are overwritten below: the scores Sc must have read them
      if (ok) ok = mbar_wait(&bar[kBarSc], s & 1, a.wait_limit);
      tc_fence_after();
      {
        float den = 0.f;
        const float4* zp = reinterpret_cast<const float4*>(Zs + 16 * sub);
        const float4* zm = reinterpret_cast<const float4*>(Zs + kFH + 16 * sub);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 a4 = zp[j4], b4 = zm[j4];
          const int j = 4 * j4;
          den = fmaf(ph[j], a4.x, fmaf(ph[16 + j], b4.x, den));
          den = fmaf(ph[j + 1], a4.y, fmaf(ph[17 + j], b4.y, den));
          den = fmaf(ph[j + 2], a4.z, fmaf(ph[18 + j], b4.z, den));
          den = fmaf(ph[j + 3], a4.w, fmaf(ph[19 + j], b4.w, den));
        }
        xden[sub * 128 + r] = den;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int j = 16 * half + 8 * q;
            // F columns 64 half + 16 sub + 8 q .. + 7: chunk 8 half + 2 sub + q
            st_shared_v4(sQ + tile_off(r, 8 * half + 2 * sub + q), pack_bf16(ph[j], ph[j + 1]),
                         pack_bf16(ph[j + 2], ph[j + 3]), pack_bf16(ph[j + 4], ph[j + 5]),
                         pack_bf16(ph[j + 6], ph[j + 7]));
          }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarPhiQ]);
      // keys: phi(K) as hi + lo over K and in the lo buffer (rows past the
      // prompt are zero, so they add nothing). The lo buffer held the
      // previous segment's outputs: their store has read it before this
      // thread reaches the next barrier, and every write follows that one.
      if (threadIdx.x == 64) bulk_wait_read();
      if (ok) ok = mbar_wait(&bar[kBarUk], s & 1, a.wait_limit);
      tc_fence_after();
      tmem_ld16(tbase + lane_bits + kColA + 64 + 16 * sub, u);
      tmem_wait_ld();
      softmaxes();
      if (!live) {
#pragma unroll
        for (int j = 0; j < 32; ++j) ph[j] = 0.f;
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t wh[4], wl[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int j = 16 * half + 8 * q + 2 * p;
            const __nv_bfloat162 hi = __floats2bfloat162_rn(ph[j], ph[j + 1]);
            const float2 hf = __bfloat1622float2(hi);
            wh[p] = *reinterpret_cast<const uint32_t*>(&hi);
            wl[p] = pack_bf16(ph[j] - hf.x, ph[j + 1] - hf.y);
          }
          const uint32_t off = tile_off(r, 8 * half + 2 * sub + q);
          st_shared_v4(sK + off, wh[0], wh[1], wh[2], wh[3]);
          st_shared_v4(sKlo + off, wl[0], wl[1], wl[2], wl[3]);
        }
      }
      // the segment's column sums of phi(K) over this warp's 32 rows: lane j
      // ends with column j of this thread's 32 (reduce-scatter), then by
      // quarter into zq in a fixed order
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) {
        const bool upper = (lane & o2) != 0;
#pragma unroll
        for (int j = 0; j < o2; ++j) {
          const float send = upper ? ph[j] : ph[j + o2];
          const float keep = upper ? ph[j + o2] : ph[j];
          ph[j] = keep + __shfl_xor_sync(0xffffffffu, send, o2);
        }
      }
      zq[quad * 128 + (lane < 16 ? 16 * sub + lane : kFH + 16 * sub + lane - 16)] = ph[0];
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarPhi]);

      // ---- E3: block softmax, weights of the earlier blocks, merge
      //      coefficients, C (over the state copy, which O2 has read)
      if (ok) ok = mbar_wait(&bar[kBarL], s & 1, a.wait_limit);
      tc_fence_after();
      // This thread's 32 keys (32 sub .. 32 sub + 31 of the segment): key j
      // is in block kb = (32 sub + j) / kBL; it is the row's own block
      // (block softmax) when kb == r / kBL, an earlier block (linear weight
      // from A) when kb < r / kBL, and a later one (0) otherwise. v holds the
      // scores (base 2) of own-block keys and A of earlier ones.
      const int rb = r / kBL;
      float v32[32];
      float m_t = -FLT_MAX, P_t = 0.f, part = 0.f;
      // kBL >= 32: one block per 32 keys, so the class is the warp's (no
      // per-key selection); kBL = 16: two blocks per quarter, per-key masks
      const int kbw = (32 * sub) / kBL;
      const bool w_own = kBL >= 32 && kbw == rb, w_early = kBL >= 32 && kbw < rb;
      uint32_t own = 0u, early = 0u;  // kBL = 16: bit j is key j's class
      if constexpr (kBL >= 32) {
        if (w_own || w_early) {
          tmem_ld32(tbase + lane_bits + (w_own ? kColS : kColA) + 32 * sub, v32);
          tmem_wait_ld();
        }
        if (w_own) {  // P = 2^{s - m} over the own block's keys held here
          float mr = -FLT_MAX;
#pragma unroll
          for (int j = 0; j < 32; j += 2) mr = fmax3(mr, v32[j], v32[j + 1]);
          m_t = mr * a.scale_log2;  // the scale is positive: max of scaled = scaled max
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v32[j] = ex2_approx(fmaf(v32[j], a.scale_log2, -m_t));
            P_t += v32[j];
          }
        } else if (w_early) {
#pragma unroll
          for (int j = 0; j < 32; ++j) part += v32[j];
        }
      } else {
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          float sc[16], aw[16];
          tmem_ld16(tbase + lane_bits + kColS + 32 * sub + 16 * hk, sc);
          tmem_ld16(tbase + lane_bits + kColA + 32 * sub + 16 * hk, aw);
          tmem_wait_ld();
          const int kb = 2 * sub + hk;
#pragma unroll
          for (int j = 0; j < 16; ++j) v32[16 * hk + j] = kb == rb ? sc[j] : aw[j];
          if (kb == rb) own |= 0xffffu << (16 * hk);
          else if (kb < rb) early |= 0xffffu << (16 * hk);
        }
        // own-block keys: local max and sum, merged across the quarters below
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((own >> j) & 1u) {
            v32[j] *= a.scale_log2;
            m_t = fmaxf(m_t, v32[j]);
          }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((own >> j) & 1u) {
            v32[j] = ex2_approx(v32[j] - m_t);
            P_t += v32[j];
          } else if ((early >> j) & 1u) {
            part += v32[j];
          }
        }
      }
      xm[sub * 128 + r] = m_t;
      xP[sub * 128 + r] = P_t;
      xa[sub * 128 + r] = part;
      named_bar_sync(1, 32 * kEpiWarps);
      // Z takes the segment's keys (every thread used Z for this segment in
      // E1; the column sums zq are complete since the barrier)
      if (sub == 0) {
        Zs[r] += (zq[r] + zq[128 + r]) + (zq[256 + r] + zq[384 + r]);
        if (s + 1 == n_seg && ok && commits) a.Z_pool[unit * kF + r] = Zs[r];
      }
      // row r's merge coefficients (its four threads compute the same): the
      // own block's max m2 and sum P (kBL = 32: one quarter holds the whole
      // block; otherwise merged exactly over the quarters that hold a part)
      float dn = (xden[r] + xden[128 + r]) + (xden[256 + r] + xden[384 + r]);
      dn += (xa[r] + xa[128 + r]) + (xa[256 + r] + xa[384 + r]);
      float m2, P, own_scale;
      if constexpr (kBL == 32) {
        m2 = xm[quad * 128 + r];
        P = xP[quad * 128 + r];
        own_scale = 1.f;
      } else {
        m2 = -FLT_MAX;
#pragma unroll
        for (int q = 0; q < 4; ++q) m2 = fmaxf(m2, xm[q * 128 + r]);
        P = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (xP[q * 128 + r] > 0.f) P = fmaf(xP[q * 128 + r], ex2_approx(xm[q * 128 + r] - m2), P);
        own_scale = P_t > 0.f ? ex2_approx(m_t - m2) : 0.f;
      }
      float cU, cN;
      if (a.merge == HB_MERGE_SHARED_NORM) {
        const float lam2 = log_sigmoid(gl) * kLog2e + m2;
        if (lam2 >= 0.f) {
          const float rr = ex2_approx(-lam2);
          cU = rcp_approx(fmaf(rr, dn, P));
          cN = rr * cU;
        } else {
          const float rr = ex2_approx(lam2);
          cN = rcp_approx(fmaf(rr, P, dn));
          cU = rr * cN;
        }
      } else {
        const float w = sigmoid(gl);
        if (dn > 0.f) {
          cU = w * rcp_approx(P);
          cN = (1.f - w) * rcp_approx(dn);
        } else {
          cU = rcp_approx(P);
          cN = 0.f;
        }
      }
      if constexpr (kBL >= 32) {
        // C = cU P on the own block, cN A on earlier ones, 0 on later ones
        const float c = w_own ? cU * own_scale : w_early ? cN : 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w4[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int j = 8 * q4 + 2 * p;
            w4[p] = (w_own || w_early) ? pack_bf16(c * v32[j], c * v32[j + 1]) : 0u;
          }
          st_shared_v4(sS16 + tile_off(r, 4 * sub + q4), w4[0], w4[1], w4[2], w4[3]);
        }
      } else {
        const float cu = cU * own_scale;
        float cj[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          cj[j] = ((own >> j) & 1u) ? cu * v32[j] : ((early >> j) & 1u) ? cN * v32[j] : 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = 8 * q4;
          st_shared_v4(sS16 + tile_off(r, 4 * sub + q4), pack_bf16(cj[j], cj[j + 1]),
                       pack_bf16(cj[j + 2], cj[j + 3]), pack_bf16(cj[j + 4], cj[j + 5]),
                       pack_bf16(cj[j + 6], cj[j + 7]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarC]);

      // ---- E4: the state after this segment (its S update is done), then
      //      o = O1 + cN O2 for this thread's 32 columns of row r
      // The state is read (and, after the last segment, stored) while O1
      // runs; its bf16 copy for the next segment's O2 goes over C once O1
      // has read C
      if (ok) ok = mbar_wait(&bar[kBarUpd], s & 1, a.wait_limit);
      tc_fence_after();
      {
        float st[32];
        tmem_ld32(tbase + lane_bits + kColM + 32 * sub, st);
        tmem_wait_ld();
        if (s + 1 < n_seg) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(st[2 * j], st[2 * j + 1]);
          if (ok) ok = mbar_wait(&bar[kBarO], s & 1, a.wait_limit);
          tc_fence_after();
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(sS16 + tile_off(r, 4 * sub + q4), pk[4 * q4], pk[4 * q4 + 1],
                         pk[4 * q4 + 2], pk[4 * q4 + 3]);
        } else {
          if (ok && commits) {
            float4* dst = reinterpret_cast<float4*>(a.S_pool + unit * kF * kD + r * kD + 32 * sub);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(st[4 * q4], st[4 * q4 + 1], st[4 * q4 + 2], st[4 * q4 + 3]);
          }
          if (ok) ok = mbar_wait(&bar[kBarO], s & 1, a.wait_limit);
          tc_fence_after();
        }
      }

#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float o1[16], o2[16];
        tmem_ld16(tbase + lane_bits + kColS + 32 * sub + 16 * hf, o1);
        tmem_ld16(tbase + lane_bits + kColU + 32 * sub + 16 * hf, o2);
        tmem_wait_ld();
        const float2 cN2 = make_float2(cN, cN);
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int j = 8 * q2;
          uint32_t w4[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 ov = fma2(make_float2(o2[j + 2 * p], o2[j + 2 * p + 1]), cN2,
                                   make_float2(o1[j + 2 * p], o1[j + 2 * p + 1]));
            w4[p] = pack_bf16(ov.x, ov.y);
          }
          // d columns 32 sub + 16 hf + 8 q2 .. + 7: chunk 4 sub + 2 hf + q2
          st_shared_v4(sKlo + tile_off(r, 4 * sub + 2 * hf + q2), w4[0], w4[1], w4[2], w4[3]);
        }
      }
      // the segment's outputs: two TMA stores (rows past the prompt are
      // clipped by the map), left in flight: the next segment waits for
      // them to have read the lo buffer only before it writes phi(K) there
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 32 * kEpiWarps);
      if (threadIdx.x == 64 && ok) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_store_4d(&maps.o, 64 * j, h, s * kSeg, b, smem + kOffKlo + j * 16384);
        bulk_commit();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarE]);
    }
    if (threadIdx.x == 64) {
      bulk_wait_read();  // the last outputs' store has read shared memory
      if (!ok) atomicOr(a.status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncwarp();  // warps whose lane 0 ran a role alone reach the barrier converged
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

bool prompt_tc_fits(const Shape& s, int batch, int num_slots, int64_t seq_len) {
  return s.dtype == HB_DTYPE_BF16 && s.d == kD && s.f == kFH &&
         (s.L == 16 || s.L == 32 || s.L == 64) && seq_len % s.L == 0 &&
         (int64_t)batch * seq_len >= kSeg && (int64_t)batch * s.H <= (1 << 30) &&
         (int64_t)batch * seq_len < ((int64_t)1 << 31) &&
         (int64_t)num_slots * s.H * kF < ((int64_t)1 << 31);
}

cudaError_t launch_prompt_tc(const Shape& s, int batch, const int32_t* slot_idx, const void* q,
                             const void* k, const void* v, int64_t seq_len, float* S_pool,
                             float* Z_pool, int num_slots, const void* W, const float* gate,
                             void* o, unsigned* status, cudaStream_t st, bool commit_all,
                             const int32_t* commit_mask) {
  Maps maps;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)batch * seq_len};
    const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
    const uint32_t box[3] = {64, 1, kSeg};
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
  {
    const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)seq_len, (uint64_t)batch};
    const uint64_t strides[3] = {kD * 2, (uint64_t)s.H * kD * 2,
                                 (uint64_t)seq_len * s.H * kD * 2};
    const uint32_t box[4] = {64, 1, kSeg, 1};
    if (!encode_tmap(&maps.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, o, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  Args a;
  a.H = s.H;
  a.num_slots = num_slots;
  a.merge = s.merge;
  a.T = seq_len;
  a.scale_log2 = s.scale * ptx::kLog2e;
  a.slot_idx = slot_idx;
  a.S_pool = S_pool;
  a.Z_pool = Z_pool;
  a.gate = gate;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.qkv[0] = static_cast<const uint8_t*>(q);
  a.qkv[1] = static_cast<const uint8_t*>(k);
  a.qkv[2] = static_cast<const uint8_t*>(v);
  a.status = status;
  a.wait_limit = wait_limit_cycles();
  a.commit_all = commit_all ? 1 : 0;
  a.commit_mask = commit_mask;
  auto* kernel = s.L == 16 ? k_prompt_tc<16> : s.L == 64 ? k_prompt_tc<64> : k_prompt_tc<32>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<dim3(batch * s.H), kThreads, kSmemBytes, st>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace hb
