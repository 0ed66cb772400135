// FP32 FMA throughput probe: the denominator of the CUDA-core kernels'
// arithmetic roofline.  Each thread runs 16 independent register-resident
// multiply-add chains (acc = acc * a + b) for `iters` rounds, as scalar FFMA
// or as packed two-lane fma.rn.f32x2, and writes the sum of its chains so
// the compiler keeps every FMA.  The caller times the launch (CUDA events on
// `stream`); flops = 2 * 16 * iters * threads, threads as returned.
#include "common.cuh"

namespace twell {
namespace {

constexpr int kChains = 16;
constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads)
    fma_probe_kernel(float* out, int iters, float a, float b) {
  float acc[kChains];
#pragma unroll
  for (int i = 0; i < kChains; ++i) acc[i] = 1e-3f * static_cast<float>(threadIdx.x + i);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kChains; ++i) acc[i] = fmaf(acc[i], a, b);
  }
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kChains; ++i) s += acc[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kProbeThreads)
    fma2_probe_kernel(float* out, int iters, float a, float b) {
  unsigned long long acc[kChains / 2];
#pragma unroll
  for (int i = 0; i < kChains / 2; ++i) {
    const float lo = 1e-3f * static_cast<float>(threadIdx.x + 2 * i);
    const float hi = 1e-3f * static_cast<float>(threadIdx.x + 2 * i + 1);
    acc[i] = (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
  }
  const unsigned long long av =
      (static_cast<unsigned long long>(__float_as_uint(a)) << 32) | __float_as_uint(a);
  const unsigned long long bv =
      (static_cast<unsigned long long>(__float_as_uint(b)) << 32) | __float_as_uint(b);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kChains / 2; ++i)
      asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[i]) : "l"(av), "l"(bv));
  }
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kChains / 2; ++i)
    s += __uint_as_float(static_cast<uint32_t>(acc[i])) +
         __uint_as_float(static_cast<uint32_t>(acc[i] >> 32));
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace
}  // namespace twell

extern "C" twell_status twell_probe_fma(int32_t packed, int32_t iters, float* out,
                                        size_t out_len, int64_t* threads, void* stream) {
  using namespace twell;
  if (iters < 1 || out == nullptr || threads == nullptr || !aligned16(out))
    return TWELL_ERR_INVALID;
  DeviceInfo dev;
  twell_status st = require_sm103(&dev);
  if (st != TWELL_OK) return st;
  // two 512-thread CTAs per SM: 32 warps, 8 per sub-partition
  const int blocks = 2 * dev.sm_count;
  const size_t n = static_cast<size_t>(blocks) * kProbeThreads;
  if (out_len < n) return TWELL_ERR_INVALID;
  *threads = static_cast<int64_t>(n);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (packed)
    fma2_probe_kernel<<<blocks, kProbeThreads, 0, s>>>(out, iters, 0.999f, 1e-3f);
  else
    fma_probe_kernel<<<blocks, kProbeThreads, 0, s>>>(out, iters, 0.999f, 1e-3f);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
