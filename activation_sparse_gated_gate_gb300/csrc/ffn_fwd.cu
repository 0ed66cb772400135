// Fused up + down projection driven by the TwELL gate ("Sparser, Faster,
// Lighter Transformer Language Models", section 2.B.2: one kernel does the
// up and down projections from the TwELL gate activations, computing dot
// products only for the nonzero elements and keeping DRAM traffic low).
//
// One warp per token row t.  x_t and the fp32 accumulator of y_t live in
// registers, spread over the 32 lanes in 16-byte chunks (lane l holds chunks
// l, l+32, ...).  The warp walks the row's TwELL tiles (the counts of 32
// tiles are read at once and the non-empty ones found with a ballot); for
// every active (j, h) it gathers neuron j's rows W_u^T[j] and W_d[j] (2*D
// contiguous bf16 each, 16-byte vector loads, coalesced across the warp),
// forms u = x_t . W_u[:, j] with a butterfly reduction and accumulates
// (h u) W_d[j, :] in fp32.
#include "common.cuh"

namespace twell {
namespace {

struct FfnParams {
  const uint16_t* x;
  const uint16_t* Wu_t;
  const uint16_t* Wd;
  float* y;
  const float* val;
  const uint8_t* col;
  const uint8_t* cnt;
  const int32_t* spill_slot;
  const float* spill_val;
  int32_t spill_cap;
  int32_t T, D, n_t, W;
  int32_t* status;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// NC = 16-byte chunks per lane (D <= 256 * NC).  EXACT: D == 256 * NC, so
// every lane owns every one of its chunks and no predicate is needed.
template <int NC, bool EXACT>
struct RowState {
  uint32_t x[NC][4];   // x_t, bf16 pairs
  float acc[NC][8];    // y_t accumulator

  __device__ __forceinline__ bool own(int i, int lane, int nch) const {
    return EXACT || (lane + 32 * i) < nch;
  }

  // u = x_t . W_u[:, j];  y_t += (h u) W_d[j, :]
  __device__ __forceinline__ void nonzero(const FfnParams& p, int j, float h, int lane,
                                          int nch) {
    const uint16_t* wu = p.Wu_t + static_cast<size_t>(j) * p.D;
    const uint16_t* wd = p.Wd + static_cast<size_t>(j) * p.D;
    uint4 a[NC], b[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      if (own(i, lane, nch)) {
        a[i] = ldg16(wu + 8 * (lane + 32 * i));
        b[i] = ldg16(wd + 8 * (lane + 32 * i));
      } else {
        a[i] = make_uint4(0, 0, 0, 0);
        b[i] = make_uint4(0, 0, 0, 0);
      }
    }
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      const uint32_t av[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        part = fmaf(bf16lo(x[i][e]), bf16lo(av[e]), part);
        part = fmaf(bf16hi(x[i][e]), bf16hi(av[e]), part);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float s = h * part;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      const uint32_t bv[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[i][2 * e] = fmaf(s, bf16lo(bv[e]), acc[i][2 * e]);
        acc[i][2 * e + 1] = fmaf(s, bf16hi(bv[e]), acc[i][2 * e + 1]);
      }
    }
  }
};

template <int NC, bool EXACT>
__global__ void __launch_bounds__(256) ffn_fwd_kernel(const FfnParams p) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nch = p.D >> 3;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < p.T; t += warps) {
    RowState<NC, EXACT> st;
    const uint16_t* xr = p.x + static_cast<size_t>(t) * p.D;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      uint4 v = st.own(i, lane, nch) ? ldg16(xr + 8 * (lane + 32 * i)) : make_uint4(0, 0, 0, 0);
      st.x[i][0] = v.x;
      st.x[i][1] = v.y;
      st.x[i][2] = v.z;
      st.x[i][3] = v.w;
#pragma unroll
      for (int e = 0; e < 8; ++e) st.acc[i][e] = 0.0f;
    }

    const size_t row_rt = static_cast<size_t>(t) * p.n_t;
    for (int kb = 0; kb < p.n_t; kb += 32) {
      const int k = kb + lane;
      const int c = k < p.n_t ? p.cnt[row_rt + k] : 0;
      uint32_t m = __ballot_sync(0xffffffffu, c > 0);
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const int kt = kb + src;
        const int cc = __shfl_sync(0xffffffffu, c, src);
        const size_t rt = row_rt + kt;
        if (cc <= p.W) {
          // slots: lane s holds slot s of this (row, tile)
          for (int s0 = 0; s0 < cc; s0 += 32) {
            const int s = s0 + lane;
            int jl = 0;
            float hl = 0.0f;
            if (s < cc) {
              jl = p.col[rt * p.W + s];
              hl = p.val[rt * p.W + s];
            }
            const int n = min(32, cc - s0);
            for (int qq = 0; qq < n; ++qq) {
              const int j = kt * TWELL_TILE + __shfl_sync(0xffffffffu, jl, qq);
              const float h = __shfl_sync(0xffffffffu, hl, qq);
              st.nonzero(p, j, h, lane, nch);
            }
          }
        } else {
          const int slot = p.spill_slot[rt];
          if (slot < 0 || slot >= p.spill_cap) {
            if (lane == 0 && p.status) atomicOr(p.status, TWELL_FLAG_SPILL_FULL);
            continue;
          }
          const float* sl = p.spill_val + static_cast<size_t>(slot) * TWELL_TILE;
#pragma unroll 1
          for (int g = 0; g < TWELL_TILE / 32; ++g) {
            const float hv = sl[g * 32 + lane];
            // stored values are ReLU outputs: positive means active
            uint32_t mm = __ballot_sync(0xffffffffu, hv > 0.0f);
            while (mm) {
              const int qq = __ffs(mm) - 1;
              mm &= mm - 1;
              const float h = __shfl_sync(0xffffffffu, hv, qq);
              st.nonzero(p, kt * TWELL_TILE + g * 32 + qq, h, lane, nch);
            }
          }
        }
      }
    }

    float* yr = p.y + static_cast<size_t>(t) * p.D;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      if (st.own(i, lane, nch)) {
        float4* o = reinterpret_cast<float4*>(yr + 8 * (lane + 32 * i));
        o[0] = make_float4(st.acc[i][0], st.acc[i][1], st.acc[i][2], st.acc[i][3]);
        o[1] = make_float4(st.acc[i][4], st.acc[i][5], st.acc[i][6], st.acc[i][7]);
      }
    }
  }
}

template <int NC>
twell_status launch_nc(const FfnParams& p, const DeviceInfo& dev, cudaStream_t s) {
  const bool exact = p.D == 256 * NC;
  const int threads = 256;
  const long long want = (static_cast<long long>(p.T) * 32 + threads - 1) / threads;
  const int grid = static_cast<int>(want < 65535LL * 8 ? want : 65535LL * 8);
  (void)dev;
  if (exact)
    ffn_fwd_kernel<NC, true><<<grid, threads, 0, s>>>(p);
  else
    ffn_fwd_kernel<NC, false><<<grid, threads, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace
}  // namespace twell

extern "C" twell_status twell_ffn_fwd(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                                      const uint16_t* Wd, int32_t D, float* y,
                                      int32_t* status_dev, void* stream) {
  using namespace twell;
  if (h == nullptr) return TWELL_ERR_INVALID;
  const int32_t T = h->T, F = h->F;
  if (T < 0 || F <= 0 || F % TWELL_TILE != 0 || D <= 0 || D % 8 != 0) return TWELL_ERR_INVALID;
  twell_status st = check_twell(h, T, F, false);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  if (!x || !Wu_t || !Wd || !y) return TWELL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(y))
    return TWELL_ERR_INVALID;
  if (D > 256 * 12) return TWELL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;

  FfnParams p;
  p.x = x;
  p.Wu_t = Wu_t;
  p.Wd = Wd;
  p.y = y;
  p.val = h->val;
  p.col = h->col;
  p.cnt = h->cnt;
  p.spill_slot = h->spill_slot;
  p.spill_val = h->spill_val;
  p.spill_cap = h->spill_cap;
  p.T = T;
  p.D = D;
  p.n_t = F / TWELL_TILE;
  p.W = h->width;
  p.status = status_dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch ((D + 255) / 256) {
    case 1: return launch_nc<1>(p, dev, s);
    case 2: return launch_nc<2>(p, dev, s);
    case 3: return launch_nc<3>(p, dev, s);
    case 4: return launch_nc<4>(p, dev, s);
    case 5: return launch_nc<5>(p, dev, s);
    case 6: return launch_nc<6>(p, dev, s);
    case 7: return launch_nc<7>(p, dev, s);
    case 8: return launch_nc<8>(p, dev, s);
    case 9: return launch_nc<9>(p, dev, s);
    case 10: return launch_nc<10>(p, dev, s);
    case 11: return launch_nc<11>(p, dev, s);
    case 12: return launch_nc<12>(p, dev, s);
    default: return TWELL_ERR_UNSUPPORTED;
  }
}
