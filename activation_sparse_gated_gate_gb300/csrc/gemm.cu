// tcgen05 GEMM for the dense-overflow rows of the hybrid training format
// ("Sparser, Faster, Lighter Transformer Language Models", section 2.B.3:
// overflow rows are routed to a dense backup, whose contractions run here on
// the tensor cores), plus the transpose / gather kernels preparing its
// operands.
//
// C[M][N] = sum over K segments of A_s[M][K_s] * B_s[N][K_s]^T, bf16 inputs,
// fp32 accumulation in TMEM.  Same warp layout as the gate kernel: a TMA
// producer warp, an MMA-issuing warp, four epilogue warps, two TMEM
// accumulator buffers, persistent CTAs.  K segments let one accumulator sum
// the bf16 hi and lo halves of an fp32 operand (v = hi + lo with |lo| <=
// 2^-9 |v|, so hi*B + lo*B carries v*B with a relative error near 2^-17);
// the row count may be a device value (number of overflow rows), in which
// case row tiles past it are skipped by every role.  Every wait is bounded
// (about a second); one that runs out sets TWELL_FLAG_TIMEOUT, and before the
// CTA frees its TMEM and exits its MMAs complete (a commit waited for) and
// its TMA loads land (a bounded 100 us wait).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bounds.cuh"
#include "gemm.cuh"
#include "ptx.cuh"
#include "scale.cuh"

namespace twell {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;

template <int BN, int STAGES>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 256 + 1024;
};

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float bf16_val(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void split(float v, uint16_t& hi, uint16_t& lo) {
  hi = bf16_bits(v);
  lo = bf16_bits(v - bf16_val(hi));
}

// Epilogue of one 32-column chunk of tile row m (global), columns
// n0 .. n0+31; `full` when all 32 columns are inside N.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& p, int m, int n0,
                                               const uint32_t (&r)[32], bool full) {
  const int N = p.N;
  if ((EPI == EPI_STORE || EPI == EPI_ADD) && p.row_idx && p.row_limit &&
      !in_bounds(p.row_idx[m], p.row_limit, p.status))
    return;
  if ((EPI == EPI_STORE || EPI == EPI_ADD) && p.ksplit > 1) {
    const int64_t row = p.row_idx ? p.row_idx[m] : m;
    float* c = p.C + row * p.ldc + n0;
    if (full) {
      float4* c4 = reinterpret_cast<float4*>(c);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        atomicAdd(c4 + i, make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                      __uint_as_float(r[4 * i + 2]),
                                      __uint_as_float(r[4 * i + 3])));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < N) atomicAdd(c + i, __uint_as_float(r[i]));
    }
  } else if (EPI == EPI_STORE || EPI == EPI_ADD) {
    const int64_t row = p.row_idx ? p.row_idx[m] : m;
    float* c = p.C + row * p.ldc + n0;
    if (full) {
      float4* c4 = reinterpret_cast<float4*>(c);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 v = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                               __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        if (EPI == EPI_ADD) {
          const float4 o = c4[i];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        c4[i] = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (n0 + i < N) {
          const float v = __uint_as_float(r[i]);
          c[i] = EPI == EPI_ADD ? c[i] + v : v;
        }
      }
    }
  } else if (EPI == EPI_UP) {
    const int64_t off = static_cast<int64_t>(m) * N + n0;
    const float* h = p.H + off;
    float* uo = p.U_out + off;
    uint16_t* hi = p.S_out + static_cast<int64_t>(m) * p.lds + n0;
    uint16_t* lo = hi + N;
    if (full && (N & 7) == 0 && (p.lds & 7) == 0) {  // 16-byte vectors (row offsets stay 32-byte aligned)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float4 h0 = reinterpret_cast<const float4*>(h)[2 * g];
        const float4 h1 = reinterpret_cast<const float4*>(h)[2 * g + 1];
        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint16_t h_a, l_a, h_b, l_b;
          split(hv[2 * e] * __uint_as_float(r[8 * g + 2 * e]), h_a, l_a);
          split(hv[2 * e + 1] * __uint_as_float(r[8 * g + 2 * e + 1]), h_b, l_b);
          wh[e] = h_a | (static_cast<uint32_t>(h_b) << 16);
          wl[e] = l_a | (static_cast<uint32_t>(l_b) << 16);
        }
        reinterpret_cast<float4*>(uo)[2 * g] =
            make_float4(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1]),
                        __uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3]));
        reinterpret_cast<float4*>(uo)[2 * g + 1] =
            make_float4(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5]),
                        __uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7]));
        reinterpret_cast<uint4*>(hi)[g] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        reinterpret_cast<uint4*>(lo)[g] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (full || n0 + i < N) {
          const float u = __uint_as_float(r[i]);
          uo[i] = u;
          uint16_t a_hi, a_lo;
          split(h[i] * u, a_hi, a_lo);
          hi[i] = a_hi;
          lo[i] = a_lo;
        }
      }
    }
  } else {  // EPI_DA
    const int64_t off = static_cast<int64_t>(m) * N + n0;
    const float* h = p.H + off;
    const float* u = p.U_in + off;
    uint16_t* s = p.S_out + static_cast<int64_t>(m) * p.lds + n0;
    auto da_at = [&](int i, float hv, float uv, uint16_t& zh, uint16_t& zl, uint16_t& wh,
                     uint16_t& wl) {
      const float da = __uint_as_float(r[i]);
      split(hv > 0.0f ? fmaf(da, uv, p.lambda) : 0.0f, zh, zl);
      split(da * hv, wh, wl);
    };
    if (full && (N & 7) == 0 && (p.lds & 7) == 0) {  // 16-byte vectors
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float4 h0 = reinterpret_cast<const float4*>(h)[2 * g];
        const float4 h1 = reinterpret_cast<const float4*>(h)[2 * g + 1];
        const float4 u0 = reinterpret_cast<const float4*>(u)[2 * g];
        const float4 u1 = reinterpret_cast<const float4*>(u)[2 * g + 1];
        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        uint32_t w[4][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint16_t a[4], b[4];
          da_at(8 * g + 2 * e, hv[2 * e], uv[2 * e], a[0], a[1], a[2], a[3]);
          da_at(8 * g + 2 * e + 1, hv[2 * e + 1], uv[2 * e + 1], b[0], b[1], b[2], b[3]);
#pragma unroll
          for (int q = 0; q < 4; ++q) w[q][e] = a[q] | (static_cast<uint32_t>(b[q]) << 16);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          reinterpret_cast<uint4*>(s + q * N)[g] = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (full || n0 + i < N) {
          uint16_t zh, zl, wh, wl;
          da_at(i, h[i], u[i], zh, zl, wh, wl);
          s[i] = zh;
          s[i + N] = zl;
          s[i + 2 * N] = wh;
          s[i + 3 * N] = wl;
        }
      }
    }
  }
}

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs p, int num_m, int num_n) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  uint64_t* drain = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // abort path: MMA drain
  volatile uint32_t* aborted = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // extents known only on the device (rows and K lengths of this call)
  const int M_act = p.M_dyn ? min(p.M, *p.M_dyn) : p.M;
  int kb_seg[kGemmMaxSeg];
  int total_kb = 0;
#pragma unroll
  for (int s = 0; s < kGemmMaxSeg; ++s) {
    int len = 0;
    if (s < p.nseg) {
      len = p.seg[s].len;
      if (p.seg[s].len_dyn) len = min(len, *p.seg[s].len_dyn);
    }
    kb_seg[s] = len > 0 ? (len + BK - 1) / BK : 0;
    total_kb += kb_seg[s];
  }
  // only the row tiles that hold rows of this call: with the row count a
  // device value (overflow rows) the launch covers the maximum, and a unit
  // numbering over all of them left whole CTAs without work (152 CTAs and 8
  // row tiles of which 4 were present: every CTA's units fell in the same row
  // tile, so half the SMs sat idle)
  const int num_m_act = min(num_m, (M_act + BM - 1) / BM);
  const int num_tiles = num_m_act * num_n;
  const int ksplit = p.ksplit > 1 ? p.ksplit : 1;
  const int num_units = num_tiles * ksplit;
  const int kb_chunk = (total_kb + ksplit - 1) / ksplit;
  // unit -> (tile, k-block range); every role skips the same units
  auto unit_range = [&](int u, int& m_blk, int& n_blk, int& kb0, int& kb1) {
    const int tile = u % num_tiles;
    const int ks = u / num_tiles;
    m_blk = tile % num_m_act;
    n_blk = tile / num_m_act;
    kb0 = ks * kb_chunk;
    kb1 = min(total_kb, kb0 + kb_chunk);
    return m_blk * BM < M_act && kb0 < kb1;
  };

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kGemmMaxSeg; ++s) {
      if (s < p.nseg) {
        ptx::prefetch_tmap(&maps.a[p.seg[s].map_a]);
        ptx::prefetch_tmap(&maps.b[p.seg[s].map_b]);
      }
    }
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 128);
    }
    ptx::mbar_init(drain, 1);
    *aborted = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (total_kb > 0) {
    if (warp == 0) {
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
          int m_blk, n_blk, kb0, kb1;
          if (!unit_range(u, m_blk, n_blk, kb0, kb1)) continue;
          int seg_first = 0;  // global index of the segment's first k block
          for (int s = 0; s < p.nseg; seg_first += kb_seg[s], ++s) {
            const CUtensorMap* ma = &maps.a[p.seg[s].map_a];
            const CUtensorMap* mb = &maps.b[p.seg[s].map_b];
            const int lo = max(kb0 - seg_first, 0);
            const int hi = min(kb1 - seg_first, kb_seg[s]);
            for (int kb = lo; kb < hi; ++kb) {
              if (!ptx::mbar_wait(&empty[stage], phase ^ 1u)) {
                { if (p.status) atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
                goto done;
              }
              ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
              ptx::tma_load_2d(sA + stage * C::A_BYTES, ma, &full[stage], kb * BK, m_blk * BM);
              ptx::tma_load_2d(sB + stage * C::B_BYTES, mb, &full[stage], kb * BK, n_blk * BN);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
          int m_blk, n_blk, kb0, kb1;
          if (!unit_range(u, m_blk, n_blk, kb0, kb1)) continue;
          const int acc = local & 1;
          const uint32_t acc_phase = (local >> 1) & 1;
          ++local;
          if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u)) {
            { if (p.status) atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          bool first = true;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!ptx::mbar_wait(&full[stage], phase)) {
              { if (p.status) atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
              goto done;
            }
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_u32(sA + stage * C::A_BYTES);
            const uint32_t b_addr = ptx::smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              ptx::mma_bf16(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + kk * 32),
                            ptx::sdesc_kmajor_sw128(b_addr + kk * 32), idesc, first ? 0u : 1u);
              first = false;
            }
            ptx::mma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          ptx::mma_commit(&tfull[acc]);
        }
      }
    } else {
      const int q = warp & 3;
      const int row = q * 32 + lane;
      int local = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        int m_blk, n_blk, kb0, kb1;
        if (!unit_range(u, m_blk, n_blk, kb0, kb1)) continue;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        ++local;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&tfull[acc], acc_phase))) {
          if (lane == 0) { if (p.status) atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        ptx::tc_fence_after();
        const int m = m_blk * BM + row;
        const bool valid = m < M_act;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int n0 = n_blk * BN + c * 32;
          if (n0 >= p.N) break;  // uniform over the CTA
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(
              tmem_base + static_cast<uint32_t>(acc * BN + c * 32) +
                  (static_cast<uint32_t>(q * 32) << 16),
              r);
          ptx::tmem_wait_ld();
          if (valid) epilogue_chunk<EPI>(p, m, n0, r, n0 + 32 <= p.N);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[acc]);
      }
    }
  }

done:
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (*aborted) {
    // a wait gave up: every MMA this CTA issued completes (the MMA thread
    // commits to a barrier of its own and waits for it) and the TMA loads
    // already issued land (bounded waits) before the TMEM is freed
    if (warp == 1 && lane == 0) {
      ptx::tc_fence_after();
      ptx::mma_commit(drain);
      ptx::mbar_wait(drain, 0);
    }
    if (threadIdx.x == 0) ptx::spin_ns(100000);
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int STAGES, int EPI>
twell_status launch(const GemmMaps& maps, const GemmArgs& a, const DeviceInfo& dev,
                    cudaStream_t s) {
  using Cc = Cfg<BN, STAGES>;
  static_assert(Cc::SMEM <= 232448, "shared memory budget");
  auto kern = gemm_kernel<BN, STAGES, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cc::SMEM) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  const int num_m = (a.M + BM - 1) / BM;
  const int num_n = (a.N + BN - 1) / BN;
  const int units = num_m * num_n * (a.ksplit > 1 ? a.ksplit : 1);
  if (units == 0) return TWELL_OK;
  const int grid = units < dev.sm_count ? units : dev.sm_count;
  kern<<<grid, kThreads, Cc::SMEM, s>>>(maps, a, num_m, num_n);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

template <int BN, int STAGES>
twell_status launch_epi(const GemmMaps& maps, const GemmArgs& a, const DeviceInfo& dev,
                        cudaStream_t s) {
  switch (a.epi) {
    case EPI_STORE: return launch<BN, STAGES, EPI_STORE>(maps, a, dev, s);
    case EPI_ADD: return launch<BN, STAGES, EPI_ADD>(maps, a, dev, s);
    case EPI_UP: return launch<BN, STAGES, EPI_UP>(maps, a, dev, s);
    case EPI_DA: return launch<BN, STAGES, EPI_DA>(maps, a, dev, s);
  }
  return TWELL_ERR_INVALID;
}

// ------------------------------------------------------------- transposes

template <int MODE>
__global__ void __launch_bounds__(256) transpose_kernel(const TransposeArgs a) {
  __shared__ float tile[32][33];
  const int R_act = a.R_dyn ? min(a.R, *a.R_dyn) : a.R;
  const int c0 = blockIdx.x * 32;
  const int r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty + 8 * i;
    const int c = c0 + tx;
    float v = 0.0f;
    if (r < R_act && c < a.C) {
      const int64_t sr =
          a.row_idx ? (a.row_limit ? clamp_index(a.row_idx[r], a.row_limit, a.status)
                                   : static_cast<long long>(a.row_idx[r]))
                    : r;
      if (MODE == 0) {
        v = bf16_val(static_cast<const uint16_t*>(a.src)[sr * a.lds + c]);
      } else {
        v = static_cast<const float*>(a.src)[sr * a.lds + c];
        if (MODE == 2) v *= a.src2[static_cast<int64_t>(r) * a.lds2 + c];
      }
    }
    tile[ty + 8 * i][tx] = v;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c0 + ty + 8 * i;
    const int r = r0 + tx;
    if (c < a.C && r < a.R_pad) {
      const float v = tile[tx][ty + 8 * i];
      const int64_t o = static_cast<int64_t>(c) * a.ldo + r;
      if (MODE == 0) {
        a.out_hi[o] = bf16_bits(v);
      } else {
        uint16_t hi, lo;
        split(v, hi, lo);
        a.out_hi[o] = hi;
        a.out_lo[o] = lo;
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(256) gather_kernel(const GatherArgs a) {
  const int R_act = a.R_dyn ? min(a.R, *a.R_dyn) : a.R;
  const int R_out = a.pad > 0 ? min(a.R, (R_act + a.pad - 1) / a.pad * a.pad) : R_act;
  const int per_row = (MODE == 1 || MODE == 3) ? a.C / 4 : a.C / 8;
  const long long total = static_cast<long long>(R_out) * per_row;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(v / per_row);
    const int q = static_cast<int>(v % per_row);
    if (i >= R_act) {  // zero padding rows
      if (MODE == 1 || MODE == 3) {
        uint16_t* o = a.out + static_cast<int64_t>(i) * a.ldo + 4 * q;
        reinterpret_cast<uint2*>(o)[0] = make_uint2(0u, 0u);
        reinterpret_cast<uint2*>(o + a.C)[0] = make_uint2(0u, 0u);
      } else {
        reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(i) * a.ldo)[q] =
            make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    const int64_t sr =
        a.row_idx ? (a.row_limit ? clamp_index(a.row_idx[i], a.row_limit, a.status)
                                 : static_cast<long long>(a.row_idx[i]))
                  : i;
    if (MODE == 3) {
      const float4 x =
          reinterpret_cast<const float4*>(static_cast<const float*>(a.src) + sr * a.lds)[q];
      const float sc = a.amax ? pow2_scale(a.amax, a.amax_floor, false) : 1.0f;
      const float f[4] = {sc * x.x, sc * x.y, sc * x.z, sc * x.w};
      uint32_t h[4], l[4];
      bool over = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        over |= fabsf(f[e]) > 65504.0f;
        const __half hv = __float2half_rn(f[e]);
        h[e] = __half_as_ushort(hv);
        l[e] = __half_as_ushort(__float2half_rn(f[e] - __half2float(hv)));
      }
      if (over && a.status) atomicOr(a.status, TWELL_FLAG_RANGE);
      uint16_t* o = a.out + static_cast<int64_t>(i) * a.ldo + 4 * q;
      reinterpret_cast<uint2*>(o)[0] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
      reinterpret_cast<uint2*>(o + a.C)[0] = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
    } else if (MODE == 4) {
      float f[8];
      {
        const uint4 x = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.src) +
                                                       sr * a.lds)[q];
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = __uint_as_float(wv[e] << 16);
          f[2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
        }
      }
      uint32_t w[4];
      bool over = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        over |= fabsf(f[2 * e]) > 65504.0f || fabsf(f[2 * e + 1]) > 65504.0f;
        w[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(f[2 * e]))) |
               (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(f[2 * e + 1]))) << 16);
      }
      if (over && a.status) atomicOr(a.status, TWELL_FLAG_RANGE);
      reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(i) * a.ldo)[q] =
          make_uint4(w[0], w[1], w[2], w[3]);
    } else if (MODE == 2) {
      const float4* s =
          reinterpret_cast<const float4*>(static_cast<const float*>(a.src) + sr * a.lds) + 2 * q;
      const float4 x0 = s[0], x1 = s[1];
      const float f[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = bf16_bits(f[2 * e]) | (static_cast<uint32_t>(bf16_bits(f[2 * e + 1])) << 16);
      reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(i) * a.ldo)[q] =
          make_uint4(w[0], w[1], w[2], w[3]);
    } else if (MODE == 0) {
      const uint4 x = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.src) +
                                                     sr * a.lds)[q];
      reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(i) * a.ldo)[q] = x;
    } else {
      const float4 x =
          reinterpret_cast<const float4*>(static_cast<const float*>(a.src) + sr * a.lds)[q];
      uint16_t h[4], l[4];
      split(x.x, h[0], l[0]);
      split(x.y, h[1], l[1]);
      split(x.z, h[2], l[2]);
      split(x.w, h[3], l[3]);
      uint16_t* o = a.out + static_cast<int64_t>(i) * a.ldo + 4 * q;
      reinterpret_cast<uint2*>(o)[0] =
          make_uint2(h[0] | (static_cast<uint32_t>(h[1]) << 16),
                     h[2] | (static_cast<uint32_t>(h[3]) << 16));
      reinterpret_cast<uint2*>(o + a.C)[0] =
          make_uint2(l[0] | (static_cast<uint32_t>(l[1]) << 16),
                     l[2] | (static_cast<uint32_t>(l[3]) << 16));
    }
  }
}

}  // namespace

twell_status gemm_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                      int64_t pitch, bool is_b_wide) {
  return make_tmap_bf16_2d(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                           BK, is_b_wide ? 256 : BM, static_cast<uint64_t>(pitch));
}

int gemm_ksplit(int64_t tiles, int64_t k, const DeviceInfo& dev) {
  const int64_t kb = (k + BK - 1) / BK;
  int64_t split = (kb + 63) / 64;
  while (split * 2 <= kb && tiles * split < 2 * dev.sm_count) split *= 2;
  if (split > kb) split = kb;
  return static_cast<int>(split < 1 ? 1 : split);
}

namespace {
__global__ void __launch_bounds__(256) zero_rows_kernel(float* C, int64_t ldc,
                                                        const int32_t* row_idx, int32_t R,
                                                        const int32_t* R_dyn, int32_t N,
                                                        int32_t row_limit, int32_t* status) {
  const int R_act = R_dyn ? min(R, *R_dyn) : R;
  const int i = blockIdx.x;
  if (i >= R_act) return;
  if (row_idx && row_limit && !in_bounds(row_idx[i], row_limit, status)) return;
  float* row = C + static_cast<int64_t>(row_idx ? row_idx[i] : i) * ldc;
  for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] = 0.0f;
}
}  // namespace

twell_status zero_rows(float* C, int64_t ldc, const int32_t* row_idx, int32_t R,
                       const int32_t* R_dyn, int32_t N, cudaStream_t s, int32_t row_limit,
                       int32_t* status) {
  if (R <= 0) return TWELL_OK;
  zero_rows_kernel<<<R, 256, 0, s>>>(C, ldc, row_idx, R, R_dyn, N, row_limit, status);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

twell_status gemm_run(const GemmMaps& maps, const GemmArgs& a, bool wide_n,
                      const DeviceInfo& dev, cudaStream_t s) {
  if (a.nseg < 1 || a.nseg > kGemmMaxSeg || a.M < 0 || a.N <= 0) return TWELL_ERR_INVALID;
  if (a.ksplit > 1 && (a.epi == EPI_UP || a.epi == EPI_DA)) return TWELL_ERR_INVALID;
  if (a.M == 0) return TWELL_OK;
  return wide_n ? launch_epi<256, 4>(maps, a, dev, s) : launch_epi<128, 6>(maps, a, dev, s);
}

twell_status transpose_run(int mode, const TransposeArgs& a, cudaStream_t s) {
  if (a.C <= 0 || a.R_pad <= 0) return TWELL_OK;
  dim3 grid((a.C + 31) / 32, (a.R_pad + 31) / 32);
  switch (mode) {
    case 0: transpose_kernel<0><<<grid, 256, 0, s>>>(a); break;
    case 1: transpose_kernel<1><<<grid, 256, 0, s>>>(a); break;
    case 2: transpose_kernel<2><<<grid, 256, 0, s>>>(a); break;
    default: return TWELL_ERR_INVALID;
  }
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

namespace {
__global__ void __launch_bounds__(256) amax_kernel(const float4* src, int64_t n4, uint32_t* out) {
  uint32_t m = 0u;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = src[i];
    m = max(m, max(max(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y))),
                   max(__float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w)))));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(out, m);
}
}  // namespace

twell_status amax_run(const float* src, int64_t n, uint32_t* out, cudaStream_t s) {
  if (cudaMemsetAsync(out, 0, sizeof(uint32_t), s) != cudaSuccess) return TWELL_ERR_CUDA;
  const int64_t n4 = n / 4;
  if (n4 <= 0) return TWELL_OK;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > 1216) blocks = 1216;  // 8 per SM
  amax_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(reinterpret_cast<const float4*>(src), n4,
                                                       out);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

twell_status gather_run(int mode, const GatherArgs& a, cudaStream_t s) {
  if (a.R <= 0) return TWELL_OK;
  const long long per_row = (mode == 1 || mode == 3) ? a.C / 4 : a.C / 8;
  long long blocks = (static_cast<long long>(a.R) * per_row + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  if (mode == 0)
    gather_kernel<0><<<static_cast<int>(blocks), 256, 0, s>>>(a);
  else if (mode == 1)
    gather_kernel<1><<<static_cast<int>(blocks), 256, 0, s>>>(a);
  else if (mode == 2)
    gather_kernel<2><<<static_cast<int>(blocks), 256, 0, s>>>(a);
  else if (mode == 3)
    gather_kernel<3><<<static_cast<int>(blocks), 256, 0, s>>>(a);
  else if (mode == 4)
    gather_kernel<4><<<static_cast<int>(blocks), 256, 0, s>>>(a);
  else
    return TWELL_ERR_INVALID;
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace twell
