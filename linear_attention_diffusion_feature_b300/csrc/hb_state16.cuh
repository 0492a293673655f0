// Reduced-precision copies of the state pool for the attend's read: bf16
// (hb_state_to_bf16, hb_block_attend_s16) and fp8 with a scale per (slot,
// head) (hb_state_to_fp8, hb_block_attend_s8). Internal to libhb.so; the
// public signatures are in include/hb.h.
//
// The attend's state contraction takes S as bf16 operands rounded to nearest
// from the fp32 state, so a copy holding exactly those rounded values gives
// bit-identical outputs while the read of S halves. The fp32 pool stays the
// master that commits and prompt ingestion update.
#pragma once

#include "hb_internal.cuh"

namespace hb {

// S16[slot] = round-to-nearest bf16 of S[slot] for the listed slots; a slot
// outside [0, num_slots) is skipped and flagged (hb_state_copy.cu).
cudaError_t launch_state_to_bf16(const Shape& s, int batch, const int32_t* slot_idx,
                                 const float* S_pool, void* S16_pool, int num_slots,
                                 unsigned* status, cudaStream_t st);

// hb_block_attend on the bf16 copy (production shape only; hb_attend_fast.cu).
cudaError_t launch_attend_fast_s16(const Shape& s, int batch, const int32_t* slot_idx,
                                   const void* q, const void* k, const void* v,
                                   const void* S16_pool, const float* Z_pool, int num_slots,
                                   const void* W, const float* gate, void* o, unsigned* status,
                                   cudaStream_t st);

// The fp8 (e4m3) copy with one scale per (slot, head): scale = max|S| / 448,
// code = e4m3(S / scale) for the listed slots; a slot outside
// [0, num_slots) is skipped and flagged (hb_state_copy.cu).
cudaError_t launch_state_to_fp8(const Shape& s, int batch, const int32_t* slot_idx,
                                const float* S_pool, void* S8_pool, float* scale_pool,
                                int num_slots, unsigned* status, cudaStream_t st);

// hb_block_attend on the fp8 copy (production shape only; hb_attend_fast.cu).
cudaError_t launch_attend_fast_s8(const Shape& s, int batch, const int32_t* slot_idx,
                                  const void* q, const void* k, const void* v,
                                  const void* S8_pool, const float* scale_pool,
                                  const float* Z_pool, int num_slots, const void* W,
                                  const float* gate, void* o, unsigned* status,
                                  cudaStream_t st);

// hb_block_attend_commit with the bf16 copies beside the fp32 masters:
// requests that do not commit read their copy, committing ones read the
// master and store the new master and its copy (production shape only;
// hb_attend_fast.cu).
cudaError_t launch_attend_commit_dual(const Shape& s, int batch, const int32_t* slot_idx,
                                      const void* q, const void* k, const void* v, float* S_pool,
                                      void* S16_pool, float* Z_pool, int num_slots, const void* W,
                                      const float* gate, const int32_t* commit_mask, void* o,
                                      unsigned* status, cudaStream_t st);

}  // namespace hb
