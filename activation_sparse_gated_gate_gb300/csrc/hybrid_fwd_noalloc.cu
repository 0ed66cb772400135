// hybrid_ffn_fwd_noalloc: the hybrid training forward with its workspace in
// a fixed device array owned by this library, for callers that cannot
// allocate device memory themselves -- for example a serving or training
// loop whose memory budget is fixed before it starts, a host program that
// embeds the library without access to a device allocator, or code that must
// not call cudaMalloc because that call can synchronise the device.
//
// The array is a file-scope __device__ variable of kScratchBytes, so every
// GPU on which the library is loaded holds it until the process exits.  Host
// code cannot use the variable's name as a device address (on the host it
// names a stand-in), so the first call on each device asks the runtime for
// the array's device address with cudaGetSymbolAddress, with that device
// current, and caches it together with the device's current context; that
// first call should therefore come before any stream capture.  A context
// torn down and created again (cudaDeviceReset, or the primary context
// released and retained) reloads the library's module at another address,
// so a call that finds a different current context looks the address up
// again (that call, too, should not be made under stream capture).  All
// calls share the one array and it keeps the contents
// of the last call; hybrid_ffn_fwd writes every workspace byte it later
// reads, so nothing has to start at zero.  Calls that may overlap on the GPU
// (different streams, or different host threads) race on the array.
#include <mutex>

#include "hybrid.cuh"

namespace twell {
namespace {

constexpr size_t kScratchBytes = size_t{64} << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
CUcontext g_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;

// The calling thread's current context (driver API, reached through the
// runtime's entry-point query so the library does not link libcuda), or
// nullptr if it cannot be read.
CUcontext current_context() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  });
  CUcontext c = nullptr;
  if (g_ctx_get == nullptr || g_ctx_get(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

}  // namespace
}  // namespace twell

extern "C" twell_status hybrid_ffn_fwd(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                                       const uint16_t* Wd, int32_t D, float* y, float* u_ell,
                                       float* U_dense, void* ws, size_t ws_bytes,
                                       int32_t* status_dev, void* stream);

extern "C" twell_status hybrid_ffn_fwd_noalloc(const uint16_t* x, const hybrid_t* h,
                                               const uint16_t* Wu_t, const uint16_t* Wd,
                                               int32_t D, float* y, float* u_ell,
                                               float* U_dense, int32_t* status_dev,
                                               void* stream) {
  using namespace twell;
  if (h == nullptr || h->T < 0 || h->F <= 0 || D <= 0 || h->cap < 1 || h->max_dense < 0)
    return TWELL_ERR_INVALID;
  const size_t need =
      h->max_dense > 0 ? ws_layout(1, h->T, D, h->F, h->cap, h->max_dense).bytes : 0;
  if (need > kScratchBytes) return TWELL_ERR_UNSUPPORTED;  // workspace above 64 MiB
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return TWELL_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const CUcontext ctx = current_context();
    if (g_addr[dev] == nullptr || ctx == nullptr || ctx != g_ctx[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return TWELL_ERR_CUDA;
      g_addr[dev] = p;
      // the lookup makes the device's primary context current if the thread
      // had none yet, so the context is read again after it
      g_ctx[dev] = current_context();
    }
    scratch = g_addr[dev];
  }
  return hybrid_ffn_fwd(x, h, Wu_t, Wd, D, y, u_ell, U_dense, scratch, kScratchBytes,
                        status_dev, stream);
}
