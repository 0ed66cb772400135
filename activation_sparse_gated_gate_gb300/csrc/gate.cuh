// Internal interface between the gate entry point and its decode-size
// kernel (gate_decode.cu).
#pragma once

#include "common.cuh"

namespace twell {

// True when the decode-size gate kernel handles T tokens of width D
// (1 <= T <= 256 and at least two K blocks of 64 to split).
bool gate_decode_supported(int32_t T, int32_t D);

// The up + down projection of twell_ffn_decode: with y, fused into the
// decode-size gate kernel (y [T][D] fp32, zeroed by the caller on the
// stream); with y NULL the kernel only prefetches the active neurons' W_u
// and W_d rows into L2 for the CUDA-core forward that follows it.
struct DecodeFfn {
  const uint16_t* Wu_t;  // [F][D] bf16
  const uint16_t* Wd;    // [F][D] bf16
  float* y;
  // with y NULL: [T][D] fp32 the kernel zeroes (NULL: none) for the forward
  // that follows, which adds into it
  float* y_zero;
};

// Enqueue the decode-size gate kernel (the caller has validated the
// arguments and zeroed out->spill_n on `s`; the kernel stores every word of
// out->block_bits itself).  With `ffn` not NULL the kernel also prefetches
// the active neurons' W_u and W_d rows into L2 and, when ffn->y is not NULL,
// adds every active entry's (h u) W_d[j, :] into it.
twell_status launch_gate_decode(const DeviceInfo& dev, const uint16_t* x, const uint16_t* Wg_t,
                                int32_t T, int32_t D, int32_t F, const twell_t* out,
                                float* z_debug, int32_t* status_dev, uint64_t wait_ns,
                                const DecodeFfn* ffn, cudaStream_t s);

}  // namespace twell
