// Gate GEMM z = x W_g with the TwELL epilogue for decode-sized batches
// ("Sparser, Faster, Lighter Transformer Language Models", section 2.B.1:
// TwELL is written in the epilogue of the gate matmul, with no separate
// conversion kernel and no round trip of h through global memory; the
// paper's kernel is a matrix-vector product at this size).
//
// With a few hundred tokens or fewer the gate is a stream of W_g (2 D F
// bytes) and the token-row tiling of the batch kernel leaves most SMs idle
// (one CTA per 128-neuron tile, 64 CTAs at d_ff 8192).  Here the operands
// swap roles and K is split:
//   * one 2-CTA cluster per TwELL tile of 128 neurons; CTA rank r of the
//     cluster runs half of the K blocks, so 2 * F / 128 CTAs stream W_g once;
//   * the MMA is z^T = W_g^T x^T: M = 128 neurons (the W_g tile, K-major by
//     TMA), N = the tokens rounded up to 16 (the x tile, rows past T read as
//     zeros), fp32 accumulation in TMEM (lane = neuron, column = token);
//   * each CTA walks its K blocks from a starting block that differs from
//     tile to tile (and wraps around), so the loads in flight at any moment
//     cover many column offsets of W_g instead of one 128-byte segment of
//     rows exactly 2 D bytes apart, which kept the DRAM at a fifth of its
//     bandwidth when every CTA walked K in step;
//   * rank 1 reads its partial sums from TMEM into its (then idle) stage
//     buffers as token rows; after a cluster barrier rank 0 adds them to its
//     own through distributed shared memory, writes the sums as token rows
//     of 128 values into its own stage buffers, and one epilogue thread per
//     token packs its row into TwELL exactly as the batch kernel does
//     (ascending slots, true count, fp32 spill slice when the count exceeds
//     W); each word of the block bitmaps is one warp's ballot over its 32
//     neurons, stored by that warp alone (so the bitmap needs no zeroing).
// Roles per CTA: warp 0 TMA producer, warp 1 TMEM allocation and MMA issue,
// warps 2-5 epilogue (warp w reads TMEM lanes 32 (w mod 4) .. + 31).
//
// Waits: every mbarrier wait is bounded (the call's bound, by default about
// 1 s) and a CTA whose wait runs out sets TWELL_FLAG_TIMEOUT, drains the
// TMA loads and MMAs it issued (waits of at most 1 s), skips its epilogue and
// still reaches both cluster barriers, which every thread of both CTAs
// passes on every path: the first publishes rank 1's partial sums, the
// second keeps rank 1's shared memory alive until rank 0 has read it.
#include "common.cuh"
#include "gate.cuh"
#include "ptx.cuh"

namespace twell {
namespace {

constexpr int DM = 128;              // neurons per CTA tile = one TwELL tile
constexpr int DK = 64;               // K block: 128-byte rows, 128B swizzle
constexpr int kThreads = 192;        // producer, MMA issuer, four epilogue warps
constexpr int kA = DM * DK * 2;      // W_g tile of a stage (16 KB)
constexpr int kMaxStages = 8;
constexpr int kRowBytes = DM * 4;    // one token's 128 fp32 values
constexpr int kBarBytes = 256;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

struct DecParams {
  int32_t T, D, F, n_t, W;
  int32_t N;          // token columns of the MMA: T rounded up to 16 (16..256)
  int32_t nkb;        // K blocks
  int32_t kb_split;   // first K block of rank 1
  int32_t stages, stage_bytes, region;  // region: bytes of the stage area
  uint32_t tmem_cols;
  float* val;
  uint8_t* col;
  uint8_t* cnt;
  int32_t* spill_slot;
  int32_t spill_cap;
  int32_t* spill_n;
  int32_t* spill_rt;
  float* spill_val;
  uint32_t* block_bits;
  float* z_debug;
  int32_t* status;
  uint64_t wait_ns;
};

__device__ __forceinline__ void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return limit_ns >= kDefaultWaitNs ? ptx::mbar_wait(bar, parity, limit_ns)
                                    : ptx::mbar_wait_strict(bar, parity, limit_ns);
}

// Byte offset of neuron n in the staged row of token slot tl: 16-byte
// chunks XOR-permuted by tl & 7, so one thread per row reading chunk c meets
// fewer bank conflicts, and a warp writing consecutive neurons of one row
// meets none.
__device__ __forceinline__ uint32_t zoff(int tl, int n) {
  return static_cast<uint32_t>(tl) * kRowBytes +
         ((static_cast<uint32_t>((n >> 2) ^ (tl & 7)) << 4) | (static_cast<uint32_t>(n & 3) << 2));
}

// TwELL packing of token t's 128 gate values (staged row tl of zt) for
// column tile `tile`: ascending active columns, the first W in the slots,
// the true count, and the ReLU'd slice in the spill list when the count
// exceeds W.
__device__ __forceinline__ void pack_row(const DecParams& p, const uint8_t* zt, int tl, int t,
                                         int tile) {
  const uint8_t* row = zt + static_cast<size_t>(tl) * kRowBytes;
  const size_t rt = static_cast<size_t>(t) * p.n_t + tile;
  uint32_t mk[4] = {0u, 0u, 0u, 0u};
  float* zd = p.z_debug ? p.z_debug + static_cast<size_t>(t) * p.F + tile * DM : nullptr;
#pragma unroll
  for (int c4 = 0; c4 < DM / 4; ++c4) {
    const float4 v = *reinterpret_cast<const float4*>(row + ((c4 ^ (tl & 7)) << 4));
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (e[k] > 0.0f) mk[c4 >> 3] |= 1u << ((4 * c4 + k) & 31);
    if (zd) reinterpret_cast<float4*>(zd)[c4] = v;
  }
  const int W = p.W;
  float* vrow = p.val + rt * W;
  uint8_t* crow = p.col + rt * W;
  int c = 0;
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    const uint32_t m = mk[ch];
    if (m == 0u) continue;
    uint32_t mm = m;
    for (int e = c; e < W && mm != 0u; ++e) {
      const int n = ch * 32 + __ffs(mm) - 1;
      mm &= mm - 1u;
      vrow[e] = *reinterpret_cast<const float*>(zt + zoff(tl, n));
      crow[e] = static_cast<uint8_t>(n);
    }
    c += __popc(m);
  }
  p.cnt[rt] = static_cast<uint8_t>(c);
  if (c > W) {
    const int slot = atomicAdd(p.spill_n, 1);
    p.spill_slot[rt] = slot;
    if (slot < p.spill_cap) {
      p.spill_rt[slot] = static_cast<int32_t>(rt);
      float4* dst = reinterpret_cast<float4*>(p.spill_val + static_cast<size_t>(slot) * DM);
#pragma unroll 8
      for (int c4 = 0; c4 < DM / 4; ++c4) {
        const float4 v = *reinterpret_cast<const float4*>(row + ((c4 ^ (tl & 7)) << 4));
        dst[c4] = make_float4(v.x > 0.0f ? v.x : 0.0f, v.y > 0.0f ? v.y : 0.0f,
                              v.z > 0.0f ? v.z : 0.0f, v.w > 0.0f ? v.w : 0.0f);
      }
    } else {
      flag(p.status, TWELL_FLAG_SPILL_FULL);
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gate_decode_kernel(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w, const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* region = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(region + p.region);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* aborted = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int tile = static_cast<int>(blockIdx.x >> 1);
  const int kb0 = rank == 0 ? 0 : p.kb_split;
  const int nloc = (rank == 0 ? p.kb_split : p.nkb) - kb0;   // K blocks of this CTA
  const int rot = nloc > 0 ? (tile * 7 + static_cast<int>(rank) * 3) % nloc : 0;
  const int S = p.stages;
  uint32_t n_loads = 0;  // stage fills issued (producer thread)

  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_x);
    ptx::prefetch_tmap(&tmap_w);
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(drain, 1);
    *aborted = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, p.tmem_cols);
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
      for (int i = 0; i < nloc; ++i) {
        const int kb = kb0 + (i + rot < nloc ? i + rot : i + rot - nloc);
        if (!pipe_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
          flag(p.status, TWELL_FLAG_TIMEOUT);
          *aborted = 1u;
          break;
        }
        uint8_t* st = region + static_cast<size_t>(stage) * p.stage_bytes;
        ptx::mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(p.stage_bytes));
        ptx::tma_load_2d(st, &tmap_w, &full[stage], kb * DK, tile * DM);
        ptx::tma_load_2d(st + kA, &tmap_x, &full[stage], kb * DK, 0);
        ++n_loads;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(DM, p.N);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < nloc; ++i) {
        if (!pipe_wait(&full[stage], phase, p.wait_ns)) {
          flag(p.status, TWELL_FLAG_TIMEOUT);
          *aborted = 1u;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_addr = ptx::smem_u32(region + static_cast<size_t>(stage) * p.stage_bytes);
        const uint32_t b_addr = a_addr + kA;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          ptx::mma_bf16(tmem_base, ptx::sdesc_kmajor_sw128(a_addr + kk * 32),
                        ptx::sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                        (i > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) ptx::mma_commit(tfull);
    }
  } else {
    // epilogue warps: the accumulator is complete (the decision is
    // warp-uniform; tcgen05.ld below is warp-collective)
    if (!__all_sync(0xffffffffu, pipe_wait(tfull, 0, p.wait_ns)) && lane == 0) {
      flag(p.status, TWELL_FLAG_TIMEOUT);
      *aborted = 1u;
    }
  }

  __syncwarp();  // lanes idle during the producer / MMA loops rejoin lane 0
  ptx::tc_fence_before();
  __syncthreads();
  const bool aborted_here = *aborted != 0u;  // the same value in every thread
  if (aborted_here) {
    if (warp == 0 && lane == 0) {
      // the last fill of each stage: fills went round the ring in order
      for (int s = 0; s < S; ++s) {
        const uint32_t n_s = (n_loads + S - 1 - s) / S;
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

  const int q = warp & 3;           // TMEM lane quarter of this warp
  const int n = q * 32 + lane;      // neuron of the tile (epilogue threads)
  const bool epi = warp >= 2;
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  if (epi && rank == 1 && !aborted_here) {
    // partial sums as token rows (plain layout) in the idle stage buffers
    ptx::tc_fence_after();
    for (int c = 0; c < p.N; c += 16) {
      uint32_t r[16];
      ptx::tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(c), r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<float*>(region + static_cast<size_t>(c + j) * kRowBytes + n * 4) =
            __uint_as_float(r[j]);
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // rank 1's partial sums and abort flag are visible

  if (epi && rank == 0) {
    const uint32_t peer_aborted =
        ptx::ld_cluster_u32(ptx::mapa(ptx::smem_u32(const_cast<uint32_t*>(aborted)), 1));
    if (!aborted_here && peer_aborted == 0u) {
      ptx::tc_fence_after();
      const uint32_t part1 = ptx::mapa(ptx::smem_u32(region), 1);
      uint8_t* zt = region;  // rank 0's own stage buffers are idle now
      const int tl_own = (warp - 2) * 32 + lane;
      for (int tb = 0; tb < p.N; tb += DM) {
        const int nb = min(DM, p.N - tb);
        bool any = false;
        for (int c = tb; c < tb + nb; c += 16) {
          // the partner's 16 partial sums first (one round trip for all),
          // then this CTA's from TMEM
          float pv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pv[j] = ptx::ld_cluster_f32(part1 + static_cast<uint32_t>((c + j) * kRowBytes + n * 4));
          uint32_t r[16];
          ptx::tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(c), r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c + j;
            const float v = __uint_as_float(r[j]) + pv[j];
            *reinterpret_cast<float*>(zt + zoff(t - tb, n)) = v;
            any |= t < p.T && v > 0.0f;
          }
        }
        if (p.block_bits) {
          // this warp alone produces the word: stored, not OR-ed (no zeroing)
          const uint32_t word = __ballot_sync(0xffffffffu, any);
          if (lane == 0)
            p.block_bits[static_cast<size_t>(tb / DM) * (p.F / 32) + tile * 4 + q] = word;
        }
        ptx::bar_sync(1, 128);  // the block's rows are staged
        const int t = tb + tl_own;
        if (tl_own < nb && t < p.T) pack_row(p, zt, tl_own, t, tile);
        ptx::bar_sync(1, 128);  // rows read before the next block overwrites them
      }
    }
  }
  ptx::cluster_sync();  // rank 1's shared memory stays until rank 0 has read it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace

bool gate_decode_supported(int32_t T, int32_t D) {
  return T >= 1 && T <= 256 && (D + DK - 1) / DK >= 2;
}

twell_status launch_gate_decode(const DeviceInfo& dev, const uint16_t* x, const uint16_t* Wg_t,
                                int32_t T, int32_t D, int32_t F, const twell_t* out,
                                float* z_debug, int32_t* status_dev, uint64_t wait_ns,
                                cudaStream_t s) {
  if (!gate_decode_supported(T, D)) return TWELL_ERR_UNSUPPORTED;
  DecParams p;
  p.T = T;
  p.D = D;
  p.F = F;
  p.n_t = F / TWELL_TILE;
  p.W = out->width;
  p.N = (T + 15) / 16 * 16;
  p.nkb = (D + DK - 1) / DK;
  p.kb_split = (p.nkb + 1) / 2;
  p.stage_bytes = kA + p.N * DK * 2;
  const int budget = (dev.max_smem_optin < 232448 ? dev.max_smem_optin : 232448) - 1024 -
                     kBarBytes;
  const int need_rows = (p.N > DM ? p.N : DM) * kRowBytes;  // exchange / staging rows
  int stages = budget / p.stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return TWELL_ERR_UNSUPPORTED;
  p.stages = stages;
  p.region = stages * p.stage_bytes > need_rows ? stages * p.stage_bytes : need_rows;
  if (p.region > budget) return TWELL_ERR_UNSUPPORTED;
  p.tmem_cols = 32;
  while (p.tmem_cols < static_cast<uint32_t>(p.N)) p.tmem_cols <<= 1;
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
  p.wait_ns = wait_ns;

  CUtensorMap mx, mw;
  twell_status st;
  if ((st = make_tmap_bf16_2d(&mw, Wg_t, D, F, DK, DM)) != TWELL_OK) return st;
  if ((st = make_tmap_bf16_2d(&mx, x, D, T, DK, static_cast<uint32_t>(p.N))) != TWELL_OK)
    return st;
  const int smem = p.region + kBarBytes + 1024;
  if (cudaFuncSetAttribute(gate_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return TWELL_ERR_CUDA;
  gate_decode_kernel<<<2 * p.n_t, kThreads, smem, s>>>(mx, mw, p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace twell
