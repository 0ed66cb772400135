// Host-side helpers shared by the library's translation units: device
// properties, argument checks and tensor-map encoding.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/twell.h"

namespace twell {

// Properties of the current device, cached per device ordinal.
struct DeviceInfo {
  int ordinal = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  int max_smem_optin = 0;
};

// Returns false if the current device cannot be queried.
bool current_device(DeviceInfo* out);

// TWELL_OK if the current device is an sm_103 part, else
// TWELL_ERR_UNSUPPORTED (or TWELL_ERR_CUDA if it cannot be queried).
twell_status require_sm103(DeviceInfo* info);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validate a TwELL descriptor against the expected T and F.
twell_status check_twell(const twell_t* h, int32_t T, int32_t F, bool need_spill_n);

// Validate a hybrid descriptor against the expected T and F.
twell_status check_hybrid(const hybrid_t* h, int32_t T, int32_t F);

// 2-D bf16 tensor map over a row-major [outer][inner] array whose rows are
// `pitch` elements apart (pitch = inner when 0), box [box_outer][box_inner],
// 128-byte swizzle, zero fill out of bounds.
twell_status make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner,
                               uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                               uint64_t pitch = 0);

// 2-D tensor map of 1-byte (u8), 2-byte (bf16) or 4-byte (fp32) elements over a row-major
// [outer][inner] array with rows `pitch_bytes` apart (a multiple of 16), box
// [box_outer][box_inner], zero fill out of bounds.  `swizzle` = 0 (none) or
// the span in bytes (32, 64, 128): in shared memory, the 16-byte chunk index
// within each span is XORed with address bits 7 and up (as many bits as the
// span has chunk-index bits); the inner box must fit in the span.
twell_status make_tmap_2d(CUtensorMap* map, int elem_bytes, const void* base, uint64_t inner,
                          uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                          uint64_t pitch_bytes, int swizzle);

}  // namespace twell
