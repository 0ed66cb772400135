// Power-of-two gradient scaling of the fp16 tensor-core backward.
//
// The backward feeds dy and the sparse gradients dz, du to the tensor cores
// as fp16, whose normal range (2^-14 .. 65504) is far narrower than fp32's:
// a gradient of a loss averaged over many tokens can lie wholly below it.
// The operands are therefore multiplied by s = 2^-e, with 2^(e-1) <= v < 2^e
// for v the largest magnitude of dy, so that the largest scaled dy lies in
// [0.5, 1), and the fp32 products are multiplied by 2^e on the way out.
// The L1 coefficient lambda enters the scaled dz as s lambda; v is at least
// 2^-14 lambda, which keeps s lambda below 2^14 (dy far below lambda then
// scales to less than [0.5, 1)).  Both factors are powers of two: apart from
// values that leave the fp16 range (reported with TWELL_FLAG_RANGE) the
// scaling rounds nothing.
#pragma once

#include <cstdint>

namespace twell {

// v = max(*amax_bits as a non-negative float, |floor_v|): s = 2^-e (inverse:
// 2^e) with e as above, limited to [-125, 126]; 1 for v = 0 or v not finite.
__device__ __forceinline__ float pow2_scale(const uint32_t* amax_bits, float floor_v,
                                            bool inverse) {
  uint32_t v = __float_as_uint(fabsf(floor_v));
  const uint32_t a = *amax_bits;
  if (a > v) v = a;
  const int E = static_cast<int>(v >> 23);
  if (v == 0u || E >= 255) return 1.0f;
  int e = E - 126;
  if (e < -125) e = -125;
  if (e > 126) e = 126;
  return __uint_as_float(static_cast<uint32_t>(127 + (inverse ? e : -e)) << 23);
}

}  // namespace twell
