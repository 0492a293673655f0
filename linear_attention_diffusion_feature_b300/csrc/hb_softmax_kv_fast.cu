// Full-prefix softmax attention of the active block over a KV cache, for the
// production shape (bf16, d = 128, L = 32). This is the comparison path: the
// cost that block-hybrid attention removes (arXiv 2608.06628 abstract: every
// denoising step of a blockwise diffusion LM still attends to all previous
// blocks; gist.science technical summary, problem statement). Query i of
// request b attends, unmasked, to the request's P_b cached keys followed by
// the L keys of its own block:
//   o_i = sum_j e^{s_ij} v_j / sum_j e^{s_ij},   s_ij = scale q_i . k_j.
//
// Split-KV ("flash-decoding") layout, sized for HBM streaming:
//   * grid (split, head, request); each CTA takes a contiguous range of
//     64-key tiles of its request (prefix tiles, then one 32-key tile of the
//     block itself);
//   * warp 4 is a TMA producer feeding a 3-stage ring of K and V tiles
//     (SWIZZLE_128B boxes of [64 keys][64 dims]); two CTAs fit on an SM;
//   * warps 0-3 compute: warp w owns query rows 16(w&1)..+15 and keys
//     32(w>>1)..+31 of every tile, with its own running max and sum
//     (online softmax in base 2), Q in registers, S = QK^T and O += PV on
//     bf16 mma.sync with fp32 accumulation; the score fragments turn into
//     the PV operand in registers;
//   * the two key halves merge in shared memory at the end; a CTA that holds
//     the whole key range writes o, otherwise it writes (m, l, O) partials
//     that k_softmax_kv_combine merges in split order.
//
// Paged cache (kPaged): the cached tokens live in pages of page_tokens rows
// of a shared pool (PagedAttention, Kwon et al., SOSP 2023; gist.science
// technical summary, "Key Contributions", implementation bullet: the serving
// kernel keeps the state next to paged KV caches). Token t of request b is
// row t mod page_tokens of page page_table[b][t / page_tokens]. With
// page_tokens a multiple of 32, each 64-key tile is two 32-row TMA boxes,
// each inside one page. Every page id a CTA needs is checked before the first
// load, and the V rows of a tile past the request's last token are zeroed in
// registers, so unused slots of a page are never read into a sum (they may
// hold anything, NaN included).
#include <float.h>
#include <math.h>

#include "hb_fast.cuh"
#include "hb_paged.cuh"
#include "hb_ptx.cuh"

namespace hb {
namespace {

using namespace ptx;

constexpr int kD = 128, kL = 32;
constexpr int kKT = 64;     // keys per tile
constexpr int kStages = 3;
constexpr int kWarps = 4;   // compute warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kMaxSplits = 64;

constexpr int kOffQ = 0;                      // 2 boxes x [32 rows][128 B]
constexpr int kOffStage = 8192;               // K: 2 x [64][128 B], V: same
constexpr int kStageBytes = 32768;
constexpr int kOffV = 16384;                  // V within a stage
constexpr int kOffBar = kOffStage + kStages * kStageBytes;
constexpr int kSmemBytes = kOffBar + 128 + 1024;
// Paged: the page ids of a CTA's key range, read once when they are checked.
constexpr int kPageCache = 1024;
constexpr int kOffPages = kOffBar + 128;
constexpr int kSmemBytesPaged = kOffPages + 4 * kPageCache + 1024;
constexpr int kPartFloats = kL * kD + 2 * kL;  // O [32][128], m [32], l [32]

struct Maps {
  CUtensorMap kc;  // [total_prefix][H][d], box {64, 1, 64}; paged: [pages * page_tokens][H][d], box {64, 1, 32}
  CUtensorMap vc;
  CUtensorMap q;   // [B*L][H][d], box {64, 1, 32}
  CUtensorMap k;
  CUtensorMap v;
};

struct Args {
  int H, splits;
  int64_t total_prefix, max_prefix;
  float scale_log2;  // scale * log2(e)
  const int64_t* cu;
  __nv_bfloat16* o;
  float* ws;
  unsigned* status;
  // paged cache only
  const int32_t* page_table;  // [batch][max_pages]
  const int32_t* plen;        // [batch] cached tokens per request
  int max_pages, page_tokens;
  int64_t num_pages;
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <bool kPaged>
__device__ __forceinline__ bool prefix_range(const Args& a, int b, int64_t* p0, int64_t* P) {
  if constexpr (kPaged) {
    *p0 = 0;
    *P = a.plen[b];
    return *P >= 0 && *P <= a.max_prefix &&
           (*P + a.page_tokens - 1) / a.page_tokens <= a.max_pages;
  } else {
    *p0 = a.cu[b];
    *P = a.cu[b + 1] - *p0;
    return *P >= 0 && *P <= a.max_prefix && *p0 >= 0 && *p0 + *P <= a.total_prefix;
  }
}

// True on every thread of the block when each page holding cached tokens
// [tok_lo, tok_hi) of request b lies in the pool. All threads must call it.
// With `cache` set, the id of the range's j-th page is also kept in
// cache[j] for j < kPageCache (visible to the whole block on return).
__device__ __forceinline__ bool pages_in_pool(const Args& a, int b, int64_t tok_lo,
                                              int64_t tok_hi, int32_t* cache = nullptr) {
  int bad = 0;
  if (tok_lo < tok_hi) {
    const int64_t first = tok_lo / a.page_tokens, last = (tok_hi - 1) / a.page_tokens;
    const int32_t* row = a.page_table + (size_t)b * a.max_pages;
    for (int64_t j = first + threadIdx.x; j <= last; j += blockDim.x) {
      const int32_t id = row[j];
      bad |= id < 0 || id >= a.num_pages;
      if (cache && j - first < kPageCache) cache[j - first] = id;
    }
  }
  return !__syncthreads_or(bad);
}

template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 2)
    k_softmax_kv_fast(const __grid_constant__ Maps maps, const __grid_constant__ Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = qbar + 1;
  uint64_t* empty = full + kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int64_t p0, P;
  if (!prefix_range<kPaged>(a, b, &p0, &P)) {
    if (threadIdx.x == 0 && split == 0) atomicOr(a.status, kStatusBounds);
    return;
  }
  const int n_pre = (int)((P + kKT - 1) / kKT);
  const int n_t = n_pre + 1;
  const int t_begin = (int)((int64_t)n_t * split / a.splits);
  const int t_end = (int)((int64_t)n_t * (split + 1) / a.splits);
  const int n_my = t_end - t_begin;
  int32_t* s_pages = reinterpret_cast<int32_t*>(smem + kOffPages);  // paged only
  int64_t first_page = 0;
  if constexpr (kPaged) {
    const int64_t lo = min((int64_t)t_begin * kKT, P), hi = min((int64_t)t_end * kKT, P);
    first_page = lo / a.page_tokens;
    if (!pages_in_pool(a, b, lo, hi, s_pages)) {
      if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
      return;
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(qbar, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&maps.q);
      if (n_pre > 0) {
        prefetch_tmap(&maps.kc);
        prefetch_tmap(&maps.vc);
      }
      mbar_arrive_expect_tx(qbar, 2 * 4096);
      tma_load_3d(smem + kOffQ, &maps.q, 0, h, b * kL, qbar);
      tma_load_3d(smem + kOffQ + 4096, &maps.q, 64, h, b * kL, qbar);
      // paged: page (relative to first_page) and row within it of the next
      // 32-token piece, advanced without a division per piece
      int pg_rel = 0, pg_off = 0;
      if (kPaged && t_begin < n_pre) {
        const int64_t tok = (int64_t)t_begin * kKT;
        pg_rel = (int)(tok / a.page_tokens - first_page);
        pg_off = (int)(tok % a.page_tokens);
      }
      for (int i = 0; i < n_my; ++i) {
        const int s = i % kStages, n = i / kStages;
        if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
          atomicOr(a.status, kStatusTimeout);
          break;
        }
        const int t = t_begin + i;
        uint8_t* st = smem + kOffStage + s * kStageBytes;
        if (t < n_pre && kPaged) {
          // one 32-row box per page piece; the second half only when the
          // request has a token there
          const int64_t tok0 = (int64_t)t * kKT;
          const int halves = P - tok0 > 32 ? 2 : 1;
          mbar_arrive_expect_tx(&full[s], halves * 4 * 4096);
          for (int c = 0; c < halves; ++c) {
            const int32_t page = pg_rel < kPageCache
                                     ? s_pages[pg_rel]
                                     : a.page_table[(size_t)b * a.max_pages + first_page + pg_rel];
            const int row = page * a.page_tokens + pg_off;
            pg_off += 32;
            if (pg_off == a.page_tokens) {
              pg_off = 0;
              ++pg_rel;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              tma_load_3d(st + j * 8192 + c * 4096, &maps.kc, 64 * j, h, row, &full[s]);
              tma_load_3d(st + kOffV + j * 8192 + c * 4096, &maps.vc, 64 * j, h, row, &full[s]);
            }
          }
        } else if (t < n_pre) {
          const int row = (int)(p0 + (int64_t)t * kKT);
          mbar_arrive_expect_tx(&full[s], 4 * 8192);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            tma_load_3d(st + j * 8192, &maps.kc, 64 * j, h, row, &full[s]);
            tma_load_3d(st + kOffV + j * 8192, &maps.vc, 64 * j, h, row, &full[s]);
          }
        } else {
          mbar_arrive_expect_tx(&full[s], 4 * 4096);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            tma_load_3d(st + j * 8192, &maps.k, 64 * j, h, b * kL, &full[s]);
            tma_load_3d(st + kOffV + j * 8192, &maps.v, 64 * j, h, b * kL, &full[s]);
          }
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------------- compute
  const int g = lane >> 2, t4 = lane & 3;
  const int mrow = warp & 1, khalf = warp >> 1;
  const int key0 = 32 * khalf;
  bool ok = mbar_wait(qbar, 0);
  if (!ok && lane == 0) atomicOr(a.status, kStatusTimeout);
  uint32_t qa[8][4];
  {
    const uint32_t sQ = smem_u32(smem + kOffQ);
    const int arow = 16 * mrow + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int ch = 2 * kk + (lane >> 4);
      ldsm_x4(sQ + (ch >> 3) * 4096 + sw128(arow, ch & 7), qa[kk][0], qa[kk][1], qa[kk][2],
              qa[kk][3]);
    }
  }
  float oacc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int i = 0; ok && i < n_my; ++i) {
    const int s = i % kStages, n = i / kStages;
    if (!mbar_wait(&full[s], n & 1)) {
      if (lane == 0) atomicOr(a.status, kStatusTimeout);
      break;
    }
    const int t = t_begin + i;
    const int valid = t < n_pre ? (int)min((int64_t)kKT, P - (int64_t)t * kKT) : kL;
    if (key0 < valid) {
      const uint32_t sK = smem_u32(smem + kOffStage + s * kStageBytes);
      const uint32_t sV = sK + kOffV;
      // scores of 16 rows x this warp's 32 keys
      float sc[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; kk += 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b0, b1, b2, b3;
          const int krow = key0 + 8 * j + (lane & 7);
          const int ch = 2 * kk + (lane >> 3);
          ldsm_x4(sK + (ch >> 3) * 8192 + sw128(krow, ch & 7), b0, b1, b2, b3);
          mma_bf16(sc[j], qa[kk], b0, b1);
          mma_bf16(sc[j], qa[kk + 1], b2, b3);
        }
      }
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int key = key0 + 8 * j + 2 * t4 + (r & 1);
          const float x = key < valid ? sc[j][r] * a.scale_log2 : -INFINITY;
          sc[j][r] = x;
          mx[r >> 1] = fmaxf(mx[r >> 1], x);
        }
      }
      float alpha[2], sum[2] = {0.f, 0.f};
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
        mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
        const float m_new = fmaxf(m_r[hr], mx[hr]);  // finite: key0 < valid
        alpha[hr] = ex2_approx(m_r[hr] - m_new);      // 0 on the first tile
        m_r[hr] = m_new;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float p = ex2_approx(sc[j][r] - m_r[r >> 1]);
          sc[j][r] = p;
          sum[r >> 1] += p;
        }
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        sum[hr] += __shfl_xor_sync(0xffffffffu, sum[hr], 1);
        sum[hr] += __shfl_xor_sync(0xffffffffu, sum[hr], 2);
        l_r[hr] = l_r[hr] * alpha[hr] + sum[hr];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        oacc[j][0] *= alpha[0];
        oacc[j][1] *= alpha[0];
        oacc[j][2] *= alpha[1];
        oacc[j][3] *= alpha[1];
      }
      // O += P V over this warp's 32 keys (two k16 steps)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * ks][0], sc[2 * ks][1]);
        pa[1] = pack_bf16(sc[2 * ks][2], sc[2 * ks][3]);
        pa[2] = pack_bf16(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
        pa[3] = pack_bf16(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
        const int mtx = lane >> 3;
        const int vrow = key0 + 16 * ks + (mtx & 1) * 8 + (lane & 7);
        // Paged: this lane's V operand holds keys kb, kb + 1 (first register
        // of each pair) and kb + 8, kb + 9 (second); rows past the request's
        // last token are zeroed so that a page's unused slots never enter
        // the sum, whatever they hold.
        uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
        if constexpr (kPaged) {
          const int kb = key0 + 16 * ks + 2 * t4;
          mk0 = (kb < valid ? 0x0000ffffu : 0u) | (kb + 1 < valid ? 0xffff0000u : 0u);
          mk1 = (kb + 8 < valid ? 0x0000ffffu : 0u) | (kb + 9 < valid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t v0, v1, v2, v3;
          const int dch = 2 * np + (mtx >> 1);
          ldsm_x4_t(sV + (dch >> 3) * 8192 + sw128(vrow, dch & 7), v0, v1, v2, v3);
          if constexpr (kPaged) {
            v0 &= mk0;
            v1 &= mk1;
            v2 &= mk0;
            v3 &= mk1;
          }
          mma_bf16(oacc[2 * np], pa, v0, v1);
          mma_bf16(oacc[2 * np + 1], pa, v2, v3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- merge the two key halves of each row block. The first barrier makes
  // sure every warp is done with the last tile before its stage is reused.
  named_bar_sync(1, kWarps * 32);
  float* xo = reinterpret_cast<float*>(smem + kOffStage) + mrow * (16 * kD + 128);
  float* xm = xo + 16 * kD;  // [2][32]: rows g and g + 8, indexed by lane
  float* xl = xm + 64;
  if (khalf == 1) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) xo[(j * 4 + r) * 32 + lane] = oacc[j][r];
    xm[lane] = m_r[0];
    xm[32 + lane] = m_r[1];
    xl[lane] = l_r[0];
    xl[32 + lane] = l_r[1];
  }
  named_bar_sync(1, kWarps * 32);
  if (khalf == 1) return;
  float f0[2], f1[2], l[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const float m1 = xm[32 * hr + lane], l1 = xl[32 * hr + lane];
    const float m = fmaxf(m_r[hr], m1);
    f0[hr] = m_r[hr] == -INFINITY ? 0.f : ex2_approx(m_r[hr] - m);
    f1[hr] = m1 == -INFINITY ? 0.f : ex2_approx(m1 - m);
    l[hr] = l_r[hr] * f0[hr] + l1 * f1[hr];
    m_r[hr] = m;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r)
      oacc[j][r] = oacc[j][r] * f0[r >> 1] + xo[(j * 4 + r) * 32 + lane] * f1[r >> 1];

  const int R0 = 16 * mrow + g;
  if (a.splits == 1) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int R = R0 + 8 * hr;
      const float inv = 1.f / l[hr];
      __nv_bfloat16* orow = a.o + ((size_t)(b * kL + R) * a.H + h) * kD;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<__nv_bfloat162*>(orow + 8 * j + 2 * t4) =
            __floats2bfloat162_rn(oacc[j][2 * hr] * inv, oacc[j][2 * hr + 1] * inv);
    }
  } else {
    float* part = a.ws + ((size_t)(b * a.H + h) * a.splits + split) * kPartFloats;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int R = R0 + 8 * hr;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<float2*>(part + R * kD + 8 * j + 2 * t4) =
            make_float2(oacc[j][2 * hr], oacc[j][2 * hr + 1]);
      if (t4 == 0) {
        part[kL * kD + R] = m_r[hr];
        part[kL * kD + kL + R] = l[hr];
      }
    }
  }
}

// Merges the split partials of each (request, head) in split order. A
// request that k_softmax_kv_fast flagged gets no output.
template <bool kPaged>
__global__ void __launch_bounds__(256) k_softmax_kv_combine(const __grid_constant__ Args a) {
  const int h = blockIdx.x, b = blockIdx.y;
  int64_t p0, P;
  if (!prefix_range<kPaged>(a, b, &p0, &P)) return;
  if constexpr (kPaged) {
    if (!pages_in_pool(a, b, 0, P)) return;
  }
  __shared__ float wgt[kMaxSplits][kL];
  __shared__ float inv[kL];
  const float* base = a.ws + (size_t)(b * a.H + h) * a.splits * kPartFloats;
  if (threadIdx.x < kL) {
    const int R = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, base[(size_t)s * kPartFloats + kL * kD + R]);
    float sum = 0.f;
    for (int s = 0; s < a.splits; ++s) {
      const float m = base[(size_t)s * kPartFloats + kL * kD + R];
      const float w = m == -INFINITY ? 0.f : ex2_approx(m - M);
      wgt[s][R] = w;
      sum += w * base[(size_t)s * kPartFloats + kL * kD + kL + R];
    }
    inv[R] = 1.f / sum;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kL * kD / 2; e += blockDim.x) {
    const int R = (2 * e) / kD, c = (2 * e) % kD;
    float x = 0.f, y = 0.f;
    for (int s = 0; s < a.splits; ++s) {
      const float2 v = *reinterpret_cast<const float2*>(base + (size_t)s * kPartFloats + R * kD + c);
      x = fmaf(wgt[s][R], v.x, x);
      y = fmaf(wgt[s][R], v.y, y);
    }
    *reinterpret_cast<__nv_bfloat162*>(a.o + ((size_t)(b * kL + R) * a.H + h) * kD + c) =
        __floats2bfloat162_rn(x * inv[R], y * inv[R]);
  }
}

int num_sms() {
  int n = 0;
  return current_sm_count(&n) == cudaSuccess && n > 0 ? n : 148;
}

// Splits per (request, head): at most one wave of two CTAs per SM (rounded
// down, so that no CTA waits for a second wave), at most one split per
// 64-key tile.
int kv_splits(int batch, int H, int64_t max_prefix) {
  const int64_t units = (int64_t)batch * H;
  const int64_t tiles = (max_prefix + kKT - 1) / kKT + 1;
  int64_t s = 2 * (int64_t)num_sms() / (units > 0 ? units : 1);
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : (int)s;
}

bool fast_kv_fits(int batch, int64_t total_prefix) {
  return batch <= 65535 && total_prefix < ((int64_t)1 << 31) &&
         (int64_t)batch * kL < ((int64_t)1 << 31);
}

// q, k, v of the active blocks: [batch * L][H][d], box {64, 1, 32}.
bool encode_block_maps(Maps* m, const Shape& s, int batch, const void* q, const void* k,
                       const void* v) {
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, (uint64_t)batch * kL};
  const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
  const uint32_t box[3] = {64, 1, 32};
  const void* ptrs[3] = {q, k, v};
  CUtensorMap* dst[3] = {&m->q, &m->k, &m->v};
  for (int j = 0; j < 3; ++j)
    if (!encode_tmap(dst[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptrs[j], dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  return true;
}

// Cached keys and values: `rows` rows of [H][d], boxes of `box_rows` rows.
bool encode_cache_maps(Maps* m, const Shape& s, const void* kc, const void* vc, uint64_t rows,
                       uint32_t box_rows) {
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)s.H, rows};
  const uint64_t strides[2] = {kD * 2, (uint64_t)s.H * kD * 2};
  const uint32_t box[3] = {64, 1, box_rows};
  return encode_tmap(&m->kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kc, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_tmap(&m->vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, vc, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool kPaged>
cudaError_t run(const Maps& maps, const Args& a, int H, int batch, cudaStream_t st) {
  const int smem = kPaged ? kSmemBytesPaged : kSmemBytes;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_softmax_kv_fast<kPaged>), smem);
  if (e != cudaSuccess) return e;
  k_softmax_kv_fast<kPaged><<<dim3(a.splits, H, batch), kThreads, smem, st>>>(maps, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.splits > 1) {
    k_softmax_kv_combine<kPaged><<<dim3(H, batch), 256, 0, st>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

Args common_args(const Shape& s, int batch, int64_t max_prefix, void* o, void* workspace,
                 unsigned* status) {
  Args a{};
  a.H = s.H;
  a.splits = kv_splits(batch, s.H, max_prefix);
  a.max_prefix = max_prefix;
  a.scale_log2 = s.scale * kLog2e;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.ws = static_cast<float*>(workspace);
  a.status = status;
  return a;
}

}  // namespace

bool fast_softmax_kv_ok(const Shape& s) { return production_shape(s); }

size_t softmax_kv_fast_workspace_bytes(const Shape& s, int batch, int64_t max_prefix) {
  const int sp = kv_splits(batch, s.H, max_prefix);
  return sp > 1 ? (size_t)batch * s.H * sp * kPartFloats * sizeof(float) : 0;
}

cudaError_t launch_softmax_kv_fast(const Shape& s, int batch, const void* k_cache,
                                   const void* v_cache, int64_t total_prefix,
                                   const int64_t* cu_prefix, int64_t max_prefix, const void* q,
                                   const void* k, const void* v, void* o, void* workspace,
                                   unsigned* status, cudaStream_t st) {
  if (!fast_kv_fits(batch, total_prefix))
    return launch_softmax_kv_generic(s, batch, k_cache, v_cache, total_prefix, cu_prefix,
                                     max_prefix, q, k, v, o, status, st);
  Maps maps;
  // With no cached rows at all no prefix tile is ever loaded; the block
  // tensors then stand in so that the maps stay encodable.
  const bool none = total_prefix == 0;
  if (!encode_block_maps(&maps, s, batch, q, k, v) ||
      !encode_cache_maps(&maps, s, none ? k : k_cache, none ? v : v_cache,
                         none ? (uint64_t)batch * kL : (uint64_t)total_prefix, kKT))
    return cudaErrorInvalidValue;
  Args a = common_args(s, batch, max_prefix, o, workspace, status);
  a.total_prefix = total_prefix;
  a.cu = cu_prefix;
  return run<false>(maps, a, s.H, batch, st);
}

bool softmax_kv_paged_fast_fits(const Shape& s, int batch, int64_t num_pages, int page_tokens,
                                int max_pages) {
  return production_shape(s) && page_tokens > 0 && page_tokens % 32 == 0 && batch <= 65535 &&
         num_pages >= 0 && num_pages * (int64_t)page_tokens < ((int64_t)1 << 31) &&
         (int64_t)batch * max_pages < ((int64_t)1 << 31) &&
         (int64_t)batch * kL < ((int64_t)1 << 31);
}

cudaError_t launch_softmax_kv_paged(const Shape& s, int batch, const void* k_pages,
                                    const void* v_pages, const PagedKV& pg, int64_t max_prefix,
                                    const void* q, const void* k, const void* v, void* o,
                                    void* workspace, unsigned* status, cudaStream_t st) {
  if (!softmax_kv_paged_fast_fits(s, batch, pg.num_pages, pg.page_tokens, pg.max_pages))
    return launch_softmax_kv_paged_generic(s, batch, k_pages, v_pages, pg, max_prefix, q, k, v,
                                           o, status, st);
  Maps maps;
  // An empty pool is never read (every request with a cached token is
  // flagged); the block tensors then stand in for it.
  const bool none = pg.num_pages == 0;
  if (!encode_block_maps(&maps, s, batch, q, k, v) ||
      !encode_cache_maps(&maps, s, none ? k : k_pages, none ? v : v_pages,
                         none ? (uint64_t)batch * kL : (uint64_t)(pg.num_pages * pg.page_tokens),
                         32))
    return cudaErrorInvalidValue;
  Args a = common_args(s, batch, max_prefix, o, workspace, status);
  a.page_table = pg.table;
  a.plen = pg.plen;
  a.max_pages = pg.max_pages;
  a.page_tokens = pg.page_tokens;
  a.num_pages = pg.num_pages;
  return run<true>(maps, a, s.H, batch, st);
}

}  // namespace hb
