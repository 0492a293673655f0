// Slot-to-slot copy of per-request states (hb_state_copy). Internal to
// libhb.so; the public signature is in include/hb.h.
#pragma once

#include "hb_internal.cuh"

namespace hb {

// S and Z of slot src[b] are copied to slot dst[b] for every b < batch; a
// pair with a slot outside [0, num_slots) is skipped and flagged.
cudaError_t launch_state_copy(const Shape& s, int batch, const int32_t* src, const int32_t* dst,
                              float* S_pool, float* Z_pool, int num_slots, unsigned* status,
                              cudaStream_t st);

}  // namespace hb
