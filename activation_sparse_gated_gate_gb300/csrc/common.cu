// Host-side helpers and the library-wide entry points (status strings,
// version).
#include "common.cuh"

#include <mutex>

namespace twell {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::mutex g_info_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool current_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_info_mu);
  DeviceInfo& d = g_info[dev];
  if (d.ordinal != dev) {
    DeviceInfo n;
    n.ordinal = dev;
    if (cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               dev) != cudaSuccess)
      return false;
    d = n;
  }
  *out = d;
  return true;
}

twell_status require_sm103(DeviceInfo* info) {
  if (!current_device(info)) return TWELL_ERR_CUDA;
  if (info->cc_major != 10 || info->cc_minor != 3) return TWELL_ERR_UNSUPPORTED;
  return TWELL_OK;
}

twell_status check_twell(const twell_t* h, int32_t T, int32_t F, bool need_spill_n) {
  if (h == nullptr) return TWELL_ERR_INVALID;
  if (h->T != T || h->F != F || h->tile != TWELL_TILE) return TWELL_ERR_INVALID;
  if (h->width < 1 || h->width > TWELL_TILE) return TWELL_ERR_INVALID;
  if (h->spill_cap < 0) return TWELL_ERR_INVALID;
  if (T == 0) return TWELL_OK;
  if (!h->val || !h->col || !h->cnt || !h->spill_slot) return TWELL_ERR_INVALID;
  if (need_spill_n && !h->spill_n) return TWELL_ERR_INVALID;
  if (h->spill_cap > 0 && (!h->spill_rt || !h->spill_val || !aligned16(h->spill_val)))
    return TWELL_ERR_INVALID;
  if (!aligned16(h->val) || !aligned16(h->col) || !aligned16(h->cnt) ||
      !aligned16(h->spill_slot))
    return TWELL_ERR_INVALID;
  return TWELL_OK;
}

twell_status make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner,
                               uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                               uint64_t pitch) {
  return make_tmap_2d(map, 2, base, inner, outer, box_inner, box_outer,
                      (pitch ? pitch : inner) * 2, 128);
}

twell_status make_tmap_2d(CUtensorMap* map, int elem_bytes, const void* base, uint64_t inner,
                          uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                          uint64_t pitch_bytes, int swizzle) {
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4) return TWELL_ERR_INVALID;
  CUtensorMapSwizzle sw;
  switch (swizzle) {
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return TWELL_ERR_INVALID;
  }
  if (swizzle && box_inner * static_cast<uint32_t>(elem_bytes) > static_cast<uint32_t>(swizzle))
    return TWELL_ERR_INVALID;
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return TWELL_ERR_CUDA;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(
      map,
      elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
      : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                        : CU_TENSOR_MAP_DATA_TYPE_UINT8,
      2,
      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TWELL_OK : TWELL_ERR_INVALID;
}

}  // namespace twell

extern "C" const char* twell_status_string(twell_status s) {
  switch (s) {
    case TWELL_OK:
      return "TWELL_OK";
    case TWELL_ERR_INVALID:
      return "TWELL_ERR_INVALID: bad argument, nothing enqueued";
    case TWELL_ERR_UNSUPPORTED:
      return "TWELL_ERR_UNSUPPORTED: device is not sm_103 or a size limit is exceeded";
    case TWELL_ERR_CUDA:
      return "TWELL_ERR_CUDA: a CUDA call failed while enqueuing";
  }
  return "unknown twell_status";
}

extern "C" int32_t twell_version(void) { return (0 << 16) | 1; }
