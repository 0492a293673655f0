// Generic CUDA kernels of block-hybrid attention: any supported shape
// (d <= 128, f <= 64, L <= 64), bf16 or fp32 activations, fp32 FMA arithmetic
// in a fixed order. They serve the fp32 accuracy mode and every shape the
// tensor-core kernels are not specialised for.
//
// Definitions followed (arXiv 2608.06628 as summarised on gist.science,
// "Technical Summary / Architecture Design", and in the pith.science review,
// "What carries the argument"):
//   phi(x)  = [softmax(x W_h), softmax(-x W_h)]
//   S      += sum_t phi(k_t) v_t^T,  Z += sum_t phi(k_t)     (commit / prefill)
//   o_i     = merge(block softmax over the L active tokens, phi(q_i)^T S, phi(q_i)^T Z)
#include <float.h>

#include "hb_internal.cuh"
#include "hb_paged.cuh"

namespace hb {
namespace {

constexpr int kThreads = 256;

// Softmax of +u (sign = 0) or -u (sign = 1) over the f entries u[0..f) held
// in shared memory, computed by one warp; writes out[0..f).
__device__ __forceinline__ void warp_half_softmax(const float* u, int f, int sign, float* out) {
  const int lane = threadIdx.x & 31;
  const float sg = sign ? -1.f : 1.f;
  float mx = -FLT_MAX;
  for (int c = lane; c < f; c += 32) mx = fmaxf(mx, sg * u[c]);
  mx = warp_max(mx);
  float sum = 0.f;
  for (int c = lane; c < f; c += 32) sum += expf(sg * u[c] - mx);
  sum = warp_sum(sum);
  const float inv = 1.f / sum;
  for (int c = lane; c < f; c += 32) out[c] = expf(sg * u[c] - mx) * inv;
}

// ------------------------------------------------------------- feature map
// grid (ceil(n / TOK), H), block 128. Shared: W_h [d][f], x tile [TOK][d],
// u tile [TOK][f] (fp32).
template <typename T>
__global__ void __launch_bounds__(128) k_feature_map_generic(int64_t n, int H, int d, int f,
                                                             const T* __restrict__ x,
                                                             const T* __restrict__ W,
                                                             float* __restrict__ phi) {
  constexpr int TOK = 16;
  extern __shared__ float smem[];
  float* sW = smem;
  float* sx = sW + d * f;
  float* su = sx + TOK * d;
  const int h = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * TOK;
  const int ntok = (int)min((int64_t)TOK, n - t0);
  for (int i = threadIdx.x; i < d * f; i += blockDim.x) sW[i] = to_f32(W[(size_t)h * d * f + i]);
  for (int i = threadIdx.x; i < ntok * d; i += blockDim.x) {
    const int t = i / d, a = i - t * d;
    sx[i] = to_f32(x[((t0 + t) * H + h) * (int64_t)d + a]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ntok * f; i += blockDim.x) {
    const int t = i / f, c = i - t * f;
    float acc = 0.f;
    for (int a = 0; a < d; ++a) acc = fmaf(sx[t * d + a], sW[a * f + c], acc);
    su[i] = acc;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int t = warp; t < ntok; t += nwarps) {
    float* out = phi + ((t0 + t) * H + h) * (int64_t)(2 * f);
    warp_half_softmax(su + t * f, f, 0, out);
    warp_half_softmax(su + t * f, f, 1, out + f);
  }
}

// ------------------------------------------------- commit / prefill (state)
// grid (batch, H), block 256. Each thread owns up to kMaxE entries of the
// F x d state in registers (entry e = tid + 256 m) and, if tid < F, one
// entry of Z. Tokens stream through shared memory in chunks of CH.
constexpr int kMaxE = 64;  // 128 * 128 / 256

template <typename T>
__global__ void __launch_bounds__(kThreads) k_state_accumulate_generic(
    int H, int d, int f, int L, const int32_t* __restrict__ slot_idx,
    const int32_t* __restrict__ mask, const T* __restrict__ k,
    const T* __restrict__ v, int64_t total_tokens, const int64_t* __restrict__ cu_seqlens,
    int64_t max_seqlen, int64_t row_stride, int64_t row_base,
    const T* __restrict__ W, float* __restrict__ S_pool, float* __restrict__ Z_pool,
    int num_slots, int accumulate, unsigned* status) {
  constexpr int CH = 16;
  const int F = 2 * f;
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (mask && mask[b] == 0) return;  // request b does not commit
  const int slot = slot_idx[b];
  int64_t row0, cnt;
  if (cu_seqlens) {
    row0 = cu_seqlens[b];
    cnt = cu_seqlens[b + 1] - row0;
  } else {  // block b is rows b * row_stride + row_base .. + L - 1
    row0 = (int64_t)b * row_stride + row_base;
    cnt = L;
  }
  if (slot < 0 || slot >= num_slots || cnt < 0 || cnt > max_seqlen || row0 < 0 ||
      row0 + cnt > total_tokens) {
    if (tid == 0) atomicOr(status, kStatusBounds);
    return;
  }
  extern __shared__ float smem[];
  float* sW = smem;             // [d][f]
  float* sk = sW + d * f;       // [CH][d]
  float* sv = sk + CH * d;      // [CH][d]
  float* su = sv + CH * d;      // [CH][f]
  float* sphi = su + CH * f;    // [CH][F]
  for (int i = tid; i < d * f; i += kThreads) sW[i] = to_f32(W[(size_t)h * d * f + i]);

  const int nE = F * d;
  float acc[kMaxE];
#pragma unroll
  for (int m = 0; m < kMaxE; ++m) acc[m] = 0.f;
  float zacc = 0.f;

  for (int64_t c0 = 0; c0 < cnt; c0 += CH) {
    const int nt = (int)min((int64_t)CH, cnt - c0);
    __syncthreads();  // previous chunk fully consumed (and sW written)
    for (int i = tid; i < nt * d; i += kThreads) {
      const int t = i / d, a = i - t * d;
      const int64_t g = ((row0 + c0 + t) * H + h) * (int64_t)d + a;
      sk[i] = to_f32(k[g]);
      sv[i] = to_f32(v[g]);
    }
    __syncthreads();
    for (int i = tid; i < nt * f; i += kThreads) {
      const int t = i / f, c = i - t * f;
      float u = 0.f;
      for (int a = 0; a < d; ++a) u = fmaf(sk[t * d + a], sW[a * f + c], u);
      su[i] = u;
    }
    __syncthreads();
    for (int t = tid >> 5; t < nt; t += kThreads / 32) {
      warp_half_softmax(su + t * f, f, 0, sphi + t * F);
      warp_half_softmax(su + t * f, f, 1, sphi + t * F + f);
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMaxE; ++m) {
      const int e = tid + kThreads * m;
      if (e < nE) {
        const int i = e / d, j = e - i * d;
        float a = acc[m];
        for (int t = 0; t < nt; ++t) a = fmaf(sphi[t * F + i], sv[t * d + j], a);
        acc[m] = a;
      }
    }
    if (tid < F)
      for (int t = 0; t < nt; ++t) zacc += sphi[t * F + tid];
  }

  float* S = S_pool + ((size_t)slot * H + h) * (size_t)F * d;
  float* Z = Z_pool + ((size_t)slot * H + h) * (size_t)F;
#pragma unroll
  for (int m = 0; m < kMaxE; ++m) {
    const int e = tid + kThreads * m;
    if (e < nE) S[e] = accumulate ? S[e] + acc[m] : acc[m];
  }
  if (tid < F) Z[tid] = accumulate ? Z[tid] + zacc : zacc;
}

// ------------------------------------------------------------------ attend
// grid (batch, H), block 256. Shared (fp32): q, k, v [L][d], W_h [d][f],
// phi [L][F], scratch [L][max(L, f)], Z [F], row stats.
// Each thread owns up to kMaxO output entries (e = tid + 256 m, i = e / d,
// j = e % d) and accumulates the block numerator and phi(q)^T S for them;
// S is read straight from global memory, column j by consecutive threads.
constexpr int kMaxO = 32;  // 64 * 128 / 256

template <typename T>
__global__ void __launch_bounds__(kThreads) k_attend_generic(
    int H, int d, int f, int L, float scale, int merge, const int32_t* __restrict__ slot_idx,
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ S_pool, const float* __restrict__ Z_pool, int num_slots,
    const T* __restrict__ W, const float* __restrict__ gate, T* __restrict__ o, unsigned* status,
    int64_t row_stride, int64_t row_base, int Hkv) {
  const int F = 2 * f;
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  // grouped-query heads: query head h reads key/value head g (k, v, S, Z)
  const int g = h / (H / Hkv);
  const int slot = slot_idx[b];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0) atomicOr(status, kStatusBounds);
    return;
  }
  extern __shared__ float smem[];
  float* sq = smem;
  float* sk = sq + L * d;
  float* sv = sk + L * d;
  float* sW = sv + L * d;
  float* sphi = sW + d * f;
  float* sscr = sphi + L * F;                 // [L][max(L, f)]
  const int scr_ld = L > f ? L : f;
  float* sZ = sscr + L * scr_ld;
  float* s_m = sZ + F;                        // row max of the block scores
  float* s_P = s_m + L;                       // row sum of e^{s - m}
  float* s_den = s_P + L;                     // phi(q)^T Z

  const size_t tok_stride = (size_t)H * d, kv_tok_stride = (size_t)Hkv * d;
  // request b's block: rows b * row_stride + row_base .. + L - 1
  const size_t row0 = (size_t)b * row_stride + row_base;
  const size_t base = (row0 * H + h) * d;
  const size_t kv_base = (row0 * Hkv + g) * d;
  for (int i = tid; i < L * d; i += kThreads) {
    const int t = i / d, a = i - t * d;
    sq[i] = to_f32(q[base + t * tok_stride + a]);
    sk[i] = to_f32(k[kv_base + t * kv_tok_stride + a]);
    sv[i] = to_f32(v[kv_base + t * kv_tok_stride + a]);
  }
  for (int i = tid; i < d * f; i += kThreads) sW[i] = to_f32(W[(size_t)h * d * f + i]);
  const float* S = S_pool + ((size_t)slot * Hkv + g) * (size_t)F * d;
  const float* Zg = Z_pool + ((size_t)slot * Hkv + g) * (size_t)F;
  for (int i = tid; i < F; i += kThreads) sZ[i] = Zg[i];
  __syncthreads();

  // u = q W_h, then phi(q) row by row.
  for (int i = tid; i < L * f; i += kThreads) {
    const int t = i / f, c = i - t * f;
    float u = 0.f;
    for (int a = 0; a < d; ++a) u = fmaf(sq[t * d + a], sW[a * f + c], u);
    sscr[t * scr_ld + c] = u;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int t = warp; t < L; t += kThreads / 32) {
    warp_half_softmax(sscr + t * scr_ld, f, 0, sphi + t * F);
    warp_half_softmax(sscr + t * scr_ld, f, 1, sphi + t * F + f);
    __syncwarp();
    float dn = 0.f;
    for (int c = lane; c < F; c += 32) dn = fmaf(sphi[t * F + c], sZ[c], dn);
    dn = warp_sum(dn);
    if (lane == 0) s_den[t] = dn;
  }
  __syncthreads();

  // Block scores s_ij = scale q_i . k_j (no mask), then row max and e^{s-m}.
  for (int e = tid; e < L * L; e += kThreads) {
    const int i = e / L, j = e - i * L;
    float s = 0.f;
    for (int a = 0; a < d; ++a) s = fmaf(sq[i * d + a], sk[j * d + a], s);
    sscr[i * scr_ld + j] = s * scale;
  }
  __syncthreads();
  for (int i = warp; i < L; i += kThreads / 32) {
    float mx = -FLT_MAX;
    for (int j = lane; j < L; j += 32) mx = fmaxf(mx, sscr[i * scr_ld + j]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j < L; j += 32) {
      const float p = expf(sscr[i * scr_ld + j] - mx);
      sscr[i * scr_ld + j] = p;
      sum += p;
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      s_m[i] = mx;
      s_P[i] = sum;
    }
  }
  __syncthreads();

  const float gl = gate[h];
  const float aux = merge == HB_MERGE_SHARED_NORM ? log_sigmoid(gl) : sigmoid(gl);
  const int nE = L * d;
  float accN[kMaxO];
#pragma unroll
  for (int m = 0; m < kMaxO; ++m) accN[m] = 0.f;
  // phi(q)^T S: column j of S is read once per thread, for all its rows i.
  for (int c = 0; c < F; ++c) {
#pragma unroll
    for (int m = 0; m < kMaxO; ++m) {
      const int e = tid + kThreads * m;
      if (e < nE) {
        const int i = e / d, j = e - i * d;
        accN[m] = fmaf(sphi[i * F + c], __ldg(S + (size_t)c * d + j), accN[m]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kMaxO; ++m) {
    const int e = tid + kThreads * m;
    if (e < nE) {
      const int i = e / d, j = e - i * d;
      float u = 0.f;
      for (int t = 0; t < L; ++t) u = fmaf(sscr[i * scr_ld + t], sv[t * d + j], u);
      const float out = merge_out(merge, u, s_P[i], s_m[i], accN[m], s_den[i], aux);
      o[base + i * tok_stride + j] = from_f32<T>(out);
    }
  }
}

// ---------------------------------------------------- softmax over KV cache
// grid (batch, H), block 256. Flash-style online softmax over the request's
// prefix keys followed by its block keys, in chunks of KC keys. The cache is
// packed per request (cu_prefix) or paged (pg.table set): cached token t of
// request b is then row t % page_tokens of page table[b][t / page_tokens].
template <typename T>
__global__ void __launch_bounds__(kThreads) k_softmax_kv_generic(
    int H, int d, int L, float scale, const T* __restrict__ k_cache, const T* __restrict__ v_cache,
    int64_t total_prefix, const int64_t* __restrict__ cu_prefix, int64_t max_prefix, const T* __restrict__ q,
    const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ o, unsigned* status,
    PagedKV pg) {
  constexpr int KC = 64;
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  int64_t p0, P;
  bool bad;
  if (pg.table) {
    p0 = 0;
    P = pg.plen[b];
    bad = P < 0 || P > max_prefix || (P + pg.page_tokens - 1) / pg.page_tokens > pg.max_pages;
  } else {
    p0 = cu_prefix[b];
    P = cu_prefix[b + 1] - p0;
    bad = P < 0 || P > max_prefix || p0 < 0 || p0 + P > total_prefix;
  }
  if (!bad && pg.table) {
    // every page the request's tokens occupy must lie in the pool
    int out = 0;
    const int32_t* row = pg.table + (size_t)b * pg.max_pages;
    for (int64_t j = tid; j < (P + pg.page_tokens - 1) / pg.page_tokens; j += blockDim.x)
      out |= row[j] < 0 || row[j] >= pg.num_pages;
    bad = __syncthreads_or(out) != 0;
  }
  if (bad) {
    if (tid == 0) atomicOr(status, kStatusBounds);
    return;
  }
  extern __shared__ float smem[];
  float* sq = smem;             // [L][d]
  float* sk = sq + L * d;       // [KC][d]
  float* sv = sk + KC * d;      // [KC][d]
  float* ss = sv + KC * d;      // [L][KC]
  float* s_m = ss + L * KC;     // running max
  float* s_l = s_m + L;         // running sum
  float* s_a = s_l + L;         // rescale factor of this chunk

  const size_t tok_stride = (size_t)H * d;
  const size_t base = ((size_t)b * L * H + h) * d;
  for (int i = tid; i < L * d; i += kThreads) {
    const int t = i / d, a = i - t * d;
    sq[i] = to_f32(q[base + t * tok_stride + a]);
  }
  for (int i = tid; i < L; i += kThreads) {
    s_m[i] = -FLT_MAX;
    s_l[i] = 0.f;
  }
  const int nE = L * d;
  float acc[kMaxO];
#pragma unroll
  for (int m = 0; m < kMaxO; ++m) acc[m] = 0.f;

  const int64_t total = P + L;
  const int warp = tid >> 5, lane = tid & 31;
  for (int64_t c0 = 0; c0 < total; c0 += KC) {
    const int nk = (int)min((int64_t)KC, total - c0);
    __syncthreads();
    for (int i = tid; i < nk * d; i += kThreads) {
      const int t = i / d, a = i - t * d;
      const int64_t key = c0 + t;
      float kk, vv;
      if (key < P) {
        const int64_t r = pg.table ? (int64_t)pg.table[(size_t)b * pg.max_pages + key / pg.page_tokens] *
                                             pg.page_tokens + key % pg.page_tokens
                                   : p0 + key;
        const size_t g = ((size_t)r * H + h) * d + a;
        kk = to_f32(k_cache[g]);
        vv = to_f32(v_cache[g]);
      } else {
        const size_t g = base + (size_t)(key - P) * tok_stride + a;
        kk = to_f32(k[g]);
        vv = to_f32(v[g]);
      }
      sk[i] = kk;
      sv[i] = vv;
    }
    __syncthreads();
    for (int e = tid; e < L * nk; e += kThreads) {
      const int i = e / nk, j = e - i * nk;
      float s = 0.f;
      for (int a = 0; a < d; ++a) s = fmaf(sq[i * d + a], sk[j * d + a], s);
      ss[i * KC + j] = s * scale;
    }
    __syncthreads();
    for (int i = warp; i < L; i += kThreads / 32) {
      float mx = -FLT_MAX;
      for (int j = lane; j < nk; j += 32) mx = fmaxf(mx, ss[i * KC + j]);
      mx = warp_max(mx);
      const float m_old = s_m[i];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (int j = lane; j < nk; j += 32) {
        const float p = expf(ss[i * KC + j] - m_new);
        ss[i * KC + j] = p;
        sum += p;
      }
      sum = warp_sum(sum);
      __syncwarp();
      if (lane == 0) {
        const float a = expf(m_old - m_new);
        s_a[i] = a;
        s_l[i] = s_l[i] * a + sum;
        s_m[i] = m_new;
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMaxO; ++m) {
      const int e = tid + kThreads * m;
      if (e < nE) {
        const int i = e / d, j = e - i * d;
        float a = acc[m] * s_a[i];
        for (int t = 0; t < nk; ++t) a = fmaf(ss[i * KC + t], sv[t * d + j], a);
        acc[m] = a;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < kMaxO; ++m) {
    const int e = tid + kThreads * m;
    if (e < nE) {
      const int i = e / d, j = e - i * d;
      o[base + i * tok_stride + j] = from_f32<T>(acc[m] / s_l[i]);
    }
  }
}

// --------------------------------------------------------------- state zero
__global__ void k_state_zero(int H, int F, int d, const int32_t* __restrict__ slot_idx,
                             float* __restrict__ S_pool, float* __restrict__ Z_pool,
                             int num_slots, unsigned* status) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int slot = slot_idx[b];
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBounds);
    return;
  }
  float4* S = reinterpret_cast<float4*>(S_pool + ((size_t)slot * H + h) * (size_t)F * d);
  for (int i = threadIdx.x; i < F * d / 4; i += blockDim.x) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  float* Z = Z_pool + ((size_t)slot * H + h) * (size_t)F;
  for (int i = threadIdx.x; i < F; i += blockDim.x) Z[i] = 0.f;
}

template <typename Fn>
cudaError_t prepare(Fn* fn, size_t smem) {
  return ensure_smem_attr(reinterpret_cast<const void*>(fn), (int)smem);
}

}  // namespace

cudaError_t launch_feature_map_generic(const Shape& s, int64_t n, const void* x, const void* W,
                                       float* phi, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)s.d * s.f + 16 * s.d + 16 * s.f);
  const dim3 grid((unsigned)((n + 15) / 16), s.H);
  cudaError_t e;
  if (s.dtype == HB_DTYPE_BF16) {
    auto* fn = k_feature_map_generic<__nv_bfloat16>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, 128, smem, st>>>(n, s.H, s.d, s.f, (const __nv_bfloat16*)x,
                                (const __nv_bfloat16*)W, phi);
  } else {
    auto* fn = k_feature_map_generic<float>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, 128, smem, st>>>(n, s.H, s.d, s.f, (const float*)x, (const float*)W, phi);
  }
  return cudaGetLastError();
}

static cudaError_t state_accumulate_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                            const int32_t* mask,
                                            const void* k, const void* v, int64_t total_tokens,
                                            const int64_t* cu_seqlens, int64_t max_seqlen,
                                            const void* W, float* S_pool, float* Z_pool,
                                            int num_slots, int accumulate, unsigned* status,
                                            cudaStream_t st, int64_t row_stride = -1,
                                            int64_t row_base = 0) {
  if (row_stride < 0) row_stride = s.L;
  constexpr int CH = 16;
  const size_t smem =
      sizeof(float) * ((size_t)s.d * s.f + 2 * CH * s.d + CH * s.f + CH * s.F);
  const dim3 grid(batch, s.H);
  const int64_t maxlen = cu_seqlens ? max_seqlen : (int64_t)s.L;
  cudaError_t e;
  if (s.dtype == HB_DTYPE_BF16) {
    auto* fn = k_state_accumulate_generic<__nv_bfloat16>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(s.H, s.d, s.f, s.L, slot_idx, mask, (const __nv_bfloat16*)k,
                                     (const __nv_bfloat16*)v, total_tokens, cu_seqlens, maxlen,
                                     row_stride, row_base, (const __nv_bfloat16*)W, S_pool, Z_pool,
                                     num_slots, accumulate, status);
  } else {
    auto* fn = k_state_accumulate_generic<float>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(s.H, s.d, s.f, s.L, slot_idx, mask, (const float*)k,
                                     (const float*)v, total_tokens, cu_seqlens, maxlen,
                                     row_stride, row_base, (const float*)W,
                                     S_pool, Z_pool, num_slots, accumulate, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_state_accumulate_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                            const void* k, const void* v, int64_t total_tokens,
                                            const int64_t* cu_seqlens, int64_t max_seqlen,
                                            const void* W, float* S_pool, float* Z_pool,
                                            int num_slots, int accumulate, unsigned* status,
                                            cudaStream_t st) {
  return state_accumulate_generic(s, batch, slot_idx, nullptr, k, v, total_tokens, cu_seqlens,
                                  max_seqlen, W, S_pool, Z_pool, num_slots, accumulate, status,
                                  st);
}

cudaError_t launch_commit_masked_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                         const int32_t* mask, const void* k, const void* v,
                                         const void* W, float* S_pool, float* Z_pool,
                                         int num_slots, unsigned* status, cudaStream_t st) {
  return state_accumulate_generic(s, batch, slot_idx, mask, k, v, (int64_t)batch * s.L, nullptr,
                                  s.L, W, S_pool, Z_pool, num_slots, 1, status, st);
}

cudaError_t launch_commit_rows_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                       const void* k, const void* v, int64_t rows_per_req,
                                       int64_t row_base, const void* W, float* S_pool,
                                       float* Z_pool, int num_slots, unsigned* status,
                                       cudaStream_t st) {
  return state_accumulate_generic(s, batch, slot_idx, nullptr, k, v, (int64_t)batch * rows_per_req,
                                  nullptr, s.L, W, S_pool, Z_pool, num_slots, 1, status, st,
                                  rows_per_req, row_base);
}

cudaError_t launch_attend_generic(const Shape& s, int batch, const int32_t* slot_idx,
                                  const void* q, const void* k, const void* v, const float* S_pool,
                                  const float* Z_pool, int num_slots, const void* W,
                                  const float* gate, void* o, unsigned* status, cudaStream_t st,
                                  int64_t rows_per_req, int64_t row_base, int Hkv) {
  if (rows_per_req < 0) rows_per_req = s.L;
  if (Hkv <= 0) Hkv = s.H;
  const int scr_ld = s.L > s.f ? s.L : s.f;
  const size_t smem = sizeof(float) * ((size_t)3 * s.L * s.d + s.d * s.f + s.L * s.F +
                                       s.L * scr_ld + s.F + 3 * s.L);
  const dim3 grid(batch, s.H);
  cudaError_t e;
  if (s.dtype == HB_DTYPE_BF16) {
    auto* fn = k_attend_generic<__nv_bfloat16>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(s.H, s.d, s.f, s.L, s.scale, s.merge, slot_idx,
                                     (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                     (const __nv_bfloat16*)v, S_pool, Z_pool, num_slots,
                                     (const __nv_bfloat16*)W, gate, (__nv_bfloat16*)o, status,
                                     rows_per_req, row_base, Hkv);
  } else {
    auto* fn = k_attend_generic<float>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(s.H, s.d, s.f, s.L, s.scale, s.merge, slot_idx,
                                     (const float*)q, (const float*)k, (const float*)v, S_pool,
                                     Z_pool, num_slots, (const float*)W, gate, (float*)o, status,
                                     rows_per_req, row_base, Hkv);
  }
  return cudaGetLastError();
}

static cudaError_t softmax_kv_generic(const Shape& s, int batch, const void* k_cache,
                                      const void* v_cache, int64_t total_prefix,
                                      const int64_t* cu_prefix, int64_t max_prefix, const void* q,
                                      const void* k, const void* v, void* o, unsigned* status,
                                      cudaStream_t st, const PagedKV& pg);

cudaError_t launch_softmax_kv_generic(const Shape& s, int batch, const void* k_cache,
                                      const void* v_cache, int64_t total_prefix,
                                      const int64_t* cu_prefix,
                                      int64_t max_prefix, const void* q, const void* k,
                                      const void* v, void* o, unsigned* status, cudaStream_t st) {
  return softmax_kv_generic(s, batch, k_cache, v_cache, total_prefix, cu_prefix, max_prefix, q, k,
                            v, o, status, st, PagedKV{});
}

static cudaError_t softmax_kv_generic(const Shape& s, int batch, const void* k_cache,
                                      const void* v_cache, int64_t total_prefix,
                                      const int64_t* cu_prefix, int64_t max_prefix, const void* q,
                                      const void* k, const void* v, void* o, unsigned* status,
                                      cudaStream_t st, const PagedKV& pg) {
  constexpr int KC = 64;
  const size_t smem = sizeof(float) * ((size_t)s.L * s.d + 2 * KC * s.d + s.L * KC + 3 * s.L);
  const dim3 grid(batch, s.H);
  cudaError_t e;
  if (s.dtype == HB_DTYPE_BF16) {
    auto* fn = k_softmax_kv_generic<__nv_bfloat16>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(s.H, s.d, s.L, s.scale, (const __nv_bfloat16*)k_cache,
                                     (const __nv_bfloat16*)v_cache, total_prefix, cu_prefix,
                                     max_prefix,
                                     (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                     (const __nv_bfloat16*)v, (__nv_bfloat16*)o, status, pg);
  } else {
    auto* fn = k_softmax_kv_generic<float>;
    if ((e = prepare(fn, smem)) != cudaSuccess) return e;
    fn<<<grid, kThreads, smem, st>>>(s.H, s.d, s.L, s.scale, (const float*)k_cache,
                                     (const float*)v_cache, total_prefix, cu_prefix, max_prefix,
                                     (const float*)q, (const float*)k, (const float*)v,
                                     (float*)o, status, pg);
  }
  return cudaGetLastError();
}

cudaError_t launch_softmax_kv_paged_generic(const Shape& s, int batch, const void* k_pages,
                                            const void* v_pages, const PagedKV& pg,
                                            int64_t max_prefix, const void* q, const void* k,
                                            const void* v, void* o, unsigned* status,
                                            cudaStream_t st) {
  return softmax_kv_generic(s, batch, k_pages, v_pages, 0, nullptr, max_prefix, q, k, v, o,
                            status, st, pg);
}

cudaError_t launch_state_zero(const Shape& s, int batch, const int32_t* slot_idx, float* S_pool,
                              float* Z_pool, int num_slots, unsigned* status, cudaStream_t st) {
  k_state_zero<<<dim3(batch, s.H), 256, 0, st>>>(s.H, s.F, s.d, slot_idx, S_pool, Z_pool,
                                                 num_slots, status);
  return cudaGetLastError();
}

}  // namespace hb
