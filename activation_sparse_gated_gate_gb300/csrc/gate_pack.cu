// Gate GEMM z = x W_g with the TwELL epilogue ("Sparser, Faster, Lighter
// Transformer Language Models", section 2.B.1: TwELL is materialised at the
// end of the dense kernel computing h_g = ReLU(x W_g), so no separate
// conversion kernel and no global round trip of h; news article "Sakana AI
// and NVIDIA TwELL boosts LLM training speed by 21.9%", epilogue paragraph:
// horizontal tiles sized to the matmul tile).
//
// Persistent tcgen05 kernel, one CTA per SM, 6 warps:
//   warp 0      TMA producer (one elected thread): x and Wg_t tiles of
//               BK = 64 (128 B rows, 128B swizzle) into a STAGES-deep ring
//   warp 1      TMEM allocator and MMA issuer (one thread): 128 x BN x 16
//               bf16 MMAs accumulating fp32 in TMEM, two accumulator buffers
//   warps 2..5  epilogue: each thread owns one output row of the 128-row
//               tile, reads its 128 fp32 z of a slice from TMEM at once
//               (four tcgen05.ld 32x32b), and packs the slice straight into
//               TwELL: a 32-bit mask of z > 0 per 32-column chunk, a walk over
//               its set bits (ascending columns), the chunk staged in a
//               private shared-memory row (XOR-swizzled by 16-byte chunk) only
//               when it has entries; spilled slices are written from the
//               registers already loaded.
// The accumulator is double-buffered so the epilogue of tile i overlaps the
// MMAs of tile i+1.
//
// Every pipeline wait is bounded (by default about 1 s; twell_gate_pack_
// wait_limit sets another bound).  A role whose wait runs out sets
// TWELL_FLAG_TIMEOUT, marks the CTA aborted and leaves its loop; the other
// roles' waits then run out too.  Before the TMEM is freed, an aborted CTA
// drains what it already issued: the producer waits for the last TMA load
// of every stage it filled, the MMA issuer commits to a barrier of its own
// and waits for all its MMAs; both waits use the fixed 1 s bound.  The
// epilogue's TMEM loads complete before it moves on, so no copy or MMA is in
// flight when the CTA deallocates and exits.
#include <atomic>

#include "common.cuh"
#include "fused.cuh"
#include "gate.cuh"
#include "ptx.cuh"

namespace twell {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
// twell_ffn_decode: the projection stays in the gate kernel up to this many
// tokens (measured at d_model 2048, d_ff 8192, 0.5 %: the one-kernel step wins
// at T = 1 and 4 and ties at 16), and for rows wider than the CUDA-core fused
// kernel takes
constexpr int32_t kDecodeProjectMaxT = 8;
constexpr int32_t kGateDecodeMaxT = 192;  // twell_gate_pack: the decode kernel up to here
constexpr int32_t kFusedMaxD = 256 * 12;

std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

struct GatePackParams {
  int32_t T, D, F, n_t, W;
  int32_t num_m, num_n, num_kb, num_tiles;
  float* val;
  uint8_t* col;
  uint8_t* cnt;
  int32_t* spill_slot;
  int32_t spill_cap;
  int32_t* spill_n;
  int32_t* spill_rt;
  float* spill_val;
  uint32_t* block_bits;  // optional [num_m][F / 32]
  float* z_debug;
  int32_t* status;
  uint64_t wait_ns;  // bound on each pipeline wait
};

template <int BN, int STAGES>
struct GateCfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = 256;
  static constexpr int STAGING = 128 * 128;  // a 32-column chunk per epilogue thread
  static constexpr int SMEM = STAGES * STAGE_BYTES + STAGING + BAR_BYTES + 1024;
};

__device__ __forceinline__ void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// A pipeline wait under the call's bound (short bounds are checked on every
// retry, the default one every 64).
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return limit_ns >= kDefaultWaitNs ? ptx::mbar_wait(bar, parity, limit_ns)
                                    : ptx::mbar_wait_strict(bar, parity, limit_ns);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gate_pack_kernel(const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_w, const GatePackParams p) {
  using Cfg = GateCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint8_t* staging = smem + STAGES * Cfg::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile uint32_t* aborted = tmem_slot + 1;
  uint64_t* drain = reinterpret_cast<uint64_t*>(tmem_slot + 2);
  uint32_t n_loads = 0;  // TMA stage fills issued (producer thread)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_x);
    ptx::prefetch_tmap(&tmap_w);
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
    ptx::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
        const int m_blk = tile / p.num_n;
        const int n_blk = tile % p.num_n;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!pipe_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
            flag(p.status, TWELL_FLAG_TIMEOUT);
            *aborted = 1u;
            goto done;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          ptx::tma_load_2d(sA + stage * Cfg::A_BYTES, &tmap_x, &full[stage], kb * BK,
                           m_blk * BM);
          ptx::tma_load_2d(sB + stage * Cfg::B_BYTES, &tmap_w, &full[stage], kb * BK,
                           n_blk * BN);
          ++n_loads;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!pipe_wait(&tempty[acc], acc_phase ^ 1u, p.wait_ns)) {
          flag(p.status, TWELL_FLAG_TIMEOUT);
          *aborted = 1u;
          goto done;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!pipe_wait(&full[stage], phase, p.wait_ns)) {
            flag(p.status, TWELL_FLAG_TIMEOUT);
            *aborted = 1u;
            goto done;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(sA + stage * Cfg::A_BYTES);
          const uint32_t b_addr = ptx::smem_u32(sB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // advancing K by 16 bf16 = 32 bytes inside the 128-byte swizzle row
            ptx::mma_bf16(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + kk * 32),
                          ptx::sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
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
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;       // row of the 128-row tile
    const int W = p.W;
    int local = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
      const int m_blk = tile / p.num_n;
      const int n_blk = tile % p.num_n;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      // the decision must be warp-uniform: tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, pipe_wait(&tfull[acc], acc_phase, p.wait_ns))) {
        if (lane == 0) {
          flag(p.status, TWELL_FLAG_TIMEOUT);
          *aborted = 1u;
        }
        goto done;
      }
      ptx::tc_fence_after();
      const int t = m_blk * BM + row;
      const bool valid = t < p.T;
      uint8_t* my_stage = staging + row * 128;
#pragma unroll 1
      for (int sub = 0; sub < BN / TWELL_TILE; ++sub) {
        const int kt = n_blk * (BN / TWELL_TILE) + sub;
        if (kt >= p.n_t) break;  // uniform over the CTA
        const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN + sub * TWELL_TILE) +
                               (static_cast<uint32_t>(q * 32) << 16);
        const size_t rt = static_cast<size_t>(valid ? t : 0) * p.n_t + kt;
        float* vrow = p.val + rt * W;
        uint8_t* crow = p.col + rt * W;
        uint32_t r[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) ptx::tmem_ld_32x32b_x32(taddr + ch * 32, r[ch]);
        ptx::tmem_wait_ld();
        // bitmask of the positive gates of each 32-column chunk of the row
        uint32_t mk[4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t m = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (__uint_as_float(r[ch][i]) > 0.0f) m |= 1u << i;
          mk[ch] = valid ? m : 0u;
        }
        if (p.block_bits) {
          // OR over the warp's 32 rows, one atomic per word and warp
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t any = __reduce_or_sync(0xffffffffu, mk[ch]);
            if (lane == 0 && any)
              atomicOr(p.block_bits + static_cast<size_t>(m_blk) * (p.F / 32) + kt * 4 + ch, any);
          }
        }
        int c = 0;
        if (valid) {
          if (p.z_debug) {
            float4* zd = reinterpret_cast<float4*>(p.z_debug + static_cast<size_t>(t) * p.F +
                                                   kt * TWELL_TILE);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
#pragma unroll
              for (int i = 0; i < 8; ++i)
                zd[ch * 8 + i] = make_float4(
                    __uint_as_float(r[ch][4 * i]), __uint_as_float(r[ch][4 * i + 1]),
                    __uint_as_float(r[ch][4 * i + 2]), __uint_as_float(r[ch][4 * i + 3]));
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t m = mk[ch];
            if (m == 0u) continue;
            const int n = __popc(m);
            if (c < W) {
              // stage the chunk, then store its actives in column order
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(my_stage + ((j ^ (row & 7)) << 4)) =
                    make_uint4(r[ch][4 * j], r[ch][4 * j + 1], r[ch][4 * j + 2],
                               r[ch][4 * j + 3]);
              uint32_t mm = m;
              for (int e = c; e < W && mm != 0u; ++e) {
                const int i = __ffs(mm) - 1;
                mm &= mm - 1u;
                vrow[e] = *reinterpret_cast<const float*>(
                    my_stage + ((((i >> 2) ^ (row & 7)) << 4) | ((i & 3) << 2)));
                crow[e] = static_cast<uint8_t>(ch * 32 + i);
              }
            }
            c += n;
          }
          p.cnt[rt] = static_cast<uint8_t>(c);
        }
        const bool spill = valid && c > W;
        if (spill) {
          const int slot = atomicAdd(p.spill_n, 1);
          p.spill_slot[rt] = slot;
          if (slot < p.spill_cap) {
            p.spill_rt[slot] = static_cast<int32_t>(rt);
            float4* dst = reinterpret_cast<float4*>(p.spill_val +
                                                    static_cast<size_t>(slot) * TWELL_TILE);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float e[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float v = __uint_as_float(r[ch][4 * i + k]);
                  e[k] = v > 0.0f ? v : 0.0f;
                }
                dst[ch * 8 + i] = make_float4(e[0], e[1], e[2], e[3]);
              }
          } else {
            flag(p.status, TWELL_FLAG_SPILL_FULL);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
    }
  }

done:
  __syncwarp();  // lanes idle during the producer / MMA loops rejoin lane 0
  ptx::tc_fence_before();
  __syncthreads();
  if (*aborted) {  // read after the barrier: the same value in every thread
    if (warp == 0 && lane == 0) {
      // the last fill of each stage: n_loads fills went round the ring in
      // order, stage s got (n_loads - s + STAGES - 1) / STAGES of them
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t n_s = (n_loads + STAGES - 1 - s) / STAGES;
        if (n_s > 0 && !ptx::mbar_wait(&full[s], (n_s - 1) & 1u)) break;
      }
    }
    if (warp == 1 && lane == 0) {
      ptx::tc_fence_after();
      ptx::mma_commit(drain);  // arrives once every MMA this thread issued is done
      ptx::mbar_wait(drain, 0);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

template <int BN, int STAGES>
twell_status launch(const DeviceInfo& dev, const CUtensorMap& mx, const CUtensorMap& mw,
                    const GatePackParams& p, cudaStream_t stream) {
  using Cfg = GateCfg<BN, STAGES>;
  static_assert(Cfg::SMEM <= 232448, "shared memory budget");
  auto kern = gate_pack_kernel<BN, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  const int grid = p.num_tiles < dev.sm_count ? p.num_tiles : dev.sm_count;
  kern<<<grid, kThreads, Cfg::SMEM, stream>>>(mx, mw, p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace
}  // namespace twell

extern "C" twell_status twell_gate_pack(const uint16_t* x, const uint16_t* Wg_t, int32_t T,
                                        int32_t D, int32_t F, const twell_t* out,
                                        float* z_debug, int32_t* status_dev, void* stream) {
  using namespace twell;
  if (T < 0 || D <= 0 || F <= 0 || D % 8 != 0 || F % TWELL_TILE != 0) return TWELL_ERR_INVALID;
  twell_status st = check_twell(out, T, F, true);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  if (!x || !Wg_t || !aligned16(x) || !aligned16(Wg_t)) return TWELL_ERR_INVALID;
  if (z_debug && !aligned16(z_debug)) return TWELL_ERR_INVALID;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GatePackParams p;
  p.T = T;
  p.D = D;
  p.F = F;
  p.n_t = F / TWELL_TILE;
  p.W = out->width;
  p.num_m = (T + BM - 1) / BM;
  p.num_kb = (D + BK - 1) / BK;
  p.val = out->val;
  p.col = out->col;
  p.cnt = out->cnt;
  p.spill_slot = out->spill_slot;
  p.spill_cap = out->spill_cap;
  p.spill_n = out->spill_n;
  p.spill_rt = out->spill_rt;
  p.spill_val = out->spill_val;
  p.block_bits = out->block_bits;
  p.z_debug = z_debug;
  p.status = status_dev;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);

  if (cudaMemsetAsync(out->spill_n, 0, sizeof(int32_t), s) != cudaSuccess) return TWELL_ERR_CUDA;

  // Decode-sized batches: the split-K kernel with the tokens as the MMA's N
  // (every TwELL tile on a 2-CTA cluster, W_g streamed once; it stores every
  // block-bitmap word itself).  Above 192 tokens its packing epilogue (16
  // tokens per step and set) outweighs the stream, and the batch kernel is
  // the faster (d_model 2048, d_ff 8192, graph replay: 23.7 against 25.7 us
  // at T = 224 and 256, equal at 128-192, 19.6 against 21.6 us at T = 96).
  if (gate_decode_supported(T, D) && T <= kGateDecodeMaxT)
    return launch_gate_decode(dev, x, Wg_t, T, D, F, out, z_debug, status_dev, p.wait_ns,
                              nullptr, s);

  if (out->block_bits &&
      cudaMemsetAsync(out->block_bits, 0,
                      static_cast<size_t>(p.num_m) * (F / 32) * sizeof(uint32_t), s) !=
          cudaSuccess)
    return TWELL_ERR_CUDA;

  // Wide tiles (N = 256, two TwELL tiles per accumulator) when they still
  // give every SM work; N = 128 otherwise (few token rows).
  const int tiles256 = p.num_m * ((F + 255) / 256);
  const bool wide = tiles256 >= dev.sm_count;
  const int BN = wide ? 256 : 128;
  p.num_n = (F + BN - 1) / BN;
  p.num_tiles = p.num_m * p.num_n;

  CUtensorMap mx, mw;
  if ((st = make_tmap_bf16_2d(&mx, x, D, T, BK, BM)) != TWELL_OK) return st;
  if ((st = make_tmap_bf16_2d(&mw, Wg_t, D, F, BK, BN)) != TWELL_OK) return st;
  return wide ? launch<256, 4>(dev, mx, mw, p, s) : launch<128, 6>(dev, mx, mw, p, s);
}

extern "C" twell_status twell_ffn_decode(const uint16_t* x, const uint16_t* Wg_t,
                                         const uint16_t* Wu_t, const uint16_t* Wd, int32_t T,
                                         int32_t D, int32_t F, const twell_t* out, float* y,
                                         float* z_debug, int32_t* status_dev, void* stream) {
  using namespace twell;
  if (T < 0 || D <= 0 || F <= 0 || D % 8 != 0 || F % TWELL_TILE != 0) return TWELL_ERR_INVALID;
  twell_status st = check_twell(out, T, F, true);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  if (!x || !Wg_t || !Wu_t || !Wd || !y || !status_dev) return TWELL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(Wg_t) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(y))
    return TWELL_ERR_INVALID;
  if (z_debug && !aligned16(z_debug)) return TWELL_ERR_INVALID;
  if (!gate_decode_supported(T, D)) return TWELL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(out->spill_n, 0, sizeof(int32_t), s) != cudaSuccess) return TWELL_ERR_CUDA;
  const uint64_t wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  // A few tokens: the projection inside the gate kernel (each entry adds a
  // whole row of y with atomics, cheap while entries are few).  More: the
  // gate kernel prefetches the active rows into L2 and the CUDA-core fused
  // kernel, which sums several entries per warp before its atomics, follows.
  if (T <= kDecodeProjectMaxT || D > kFusedMaxD) {
    if (cudaMemsetAsync(y, 0, static_cast<size_t>(T) * D * sizeof(float), s) != cudaSuccess)
      return TWELL_ERR_CUDA;
    const DecodeFfn ffn{Wu_t, Wd, y, nullptr};
    return launch_gate_decode(dev, x, Wg_t, T, D, F, out, z_debug, status_dev, wait_ns, &ffn,
                              s);
  }
  // (the gate kernel also zeroes y for the forward, which adds into it)
  const DecodeFfn prefetch{Wu_t, Wd, nullptr, y};
  if ((st = launch_gate_decode(dev, x, Wg_t, T, D, F, out, z_debug, status_dev, wait_ns,
                               &prefetch, s)) != TWELL_OK)
    return st;
  return ffn_fwd_twell(x, out, Wu_t, Wd, D, y, status_dev, s, true);
}

extern "C" uint64_t twell_gate_pack_wait_limit(uint64_t ns) {
  return twell::g_wait_ns.exchange(ns == 0 ? twell::kDefaultWaitNs : ns);
}
