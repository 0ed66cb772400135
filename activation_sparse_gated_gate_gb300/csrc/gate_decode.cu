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
//   * the producer issues the first round of stage fills right after it
//     initialises the barriers, before the block-wide sync and the TMEM
//     allocation;
//   * the tokens are split between the two CTAs in 16-column chunks (rank 0
//     the first half, rank 1 the rest): each CTA reads from TMEM the partial
//     sums of the partner's tokens and stores them straight into the
//     partner's exchange rows (one row of 128 fp32 per token, a region of
//     its own, never a stage buffer) with remote shared-memory stores, and
//     after one cluster barrier adds the partner's rows to its own partial
//     sums;
//   * packing is warp-parallel: two sets of four epilogue warps take
//     alternate chunks of 16 tokens; for a chunk each warp of the set (32
//     neurons, one per lane) takes one ballot per token, the set's four warps
//     exchange the ballots through shared memory, and each active lane
//     writes its value to slot (active neurons before it in the tile) when
//     that is below W, so the slots hold the first W active columns in
//     ascending order; the true count and, when it exceeds W, the ReLU'd
//     fp32 slice in the spill list are written as by the batch kernel;
//   * each block-bitmap word (one per 128-token block and 32 neurons) is the
//     OR of the ballots of that quarter's warps (a shared-memory word each
//     CTA clears in its prologue): rank 1 hands its part of block 0 to rank 0
//     with a remote store, and each word is stored once (no zeroing).
// Roles per CTA: warp 0 TMA producer, warp 1 TMEM allocation and MMA issue,
// warps 2-9 epilogue (warp w reads TMEM lanes 32 (w mod 4) .. + 31).
//
// Waits: every mbarrier wait is bounded (the call's bound, by default about
// 1 s) and a CTA whose wait runs out sets TWELL_FLAG_TIMEOUT, drains the
// TMA loads and MMAs it issued (waits of at most 1 s), skips its epilogue,
// tells the partner (which then skips its packing too) and still passes
// every cluster barrier phase, which every thread of both CTAs reaches on
// every path: the first (arrived at after the prologue, waited for before
// the first remote store) guarantees the partner has started, the second
// publishes the exchanged partial sums, the third the block-bitmap words.
#include "bounds.cuh"
#include "common.cuh"
#include "gate.cuh"
#include "ptx.cuh"

namespace twell {
namespace {

constexpr int DM = 128;              // neurons per CTA tile = one TwELL tile
constexpr int DK = 64;               // K block: 128-byte rows, 128B swizzle
constexpr int kThreads = 320;        // producer, MMA issuer, two sets of four epilogue warps
constexpr int kA = DM * DK * 2;      // W_g tile of a stage (16 KB)
constexpr int kMaxStages = 8;
constexpr int kRowBytes = DM * 4;    // one token's 128 fp32 values
// barrier area, byte offsets: full[8] 0, empty[8] 64, tfull 128, drain 136,
// TMEM address 144, abort flag 148, partner's abort flag 152, rank 1's
// block-0 words 160, this CTA's block words [2 blocks][4 quarters] 192,
// entry count 224, ballots [2 sets][2][16 tokens][4 quarters] 256, spill
// slots [2 sets][2][16] 1280
constexpr int kBarBytes = 2048;
constexpr int kEntryBytes = 8;       // (token * 128 + neuron, gate value) of an active entry
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

struct DecParams {
  int32_t T, D, F, n_t, W;
  int32_t N;          // token columns of the MMA: T rounded up to 16 (16..256)
  int32_t nkb;        // K blocks
  int32_t kb_split;   // first K block of rank 1
  int32_t stages, stage_bytes, region;  // region: bytes of the stage area
  int32_t half;       // tokens of rank 0 (16-column chunks, rounded up); rank 1 has N - half
  int32_t xch_bytes;  // exchange rows: half * 512
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
  // fused up + down projection (twell_ffn_decode); y NULL skips it
  const uint16_t* x;
  const uint16_t* Wu_t;
  const uint16_t* Wd;
  float* y;
  float* y_zero;      // prefetch mode: y of the forward that follows, zeroed here
};

__device__ __forceinline__ void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return limit_ns >= kDefaultWaitNs ? ptx::mbar_wait(bar, parity, limit_ns)
                                    : ptx::mbar_wait_strict(bar, parity, limit_ns);
}

// The eight bf16 of a 16-byte chunk as fp32 (exact: a bf16 is the top half
// of its fp32).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* f) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(u[k] << 16);
    f[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
  }
}

// Sum of the eight products of two 16-byte bf16 chunks, in fp32 (in order).
__device__ __forceinline__ float dot8_bf16(const uint4 a, const uint4 b) {
  float fa[8], fb[8];
  bf16x8_to_f32(a, fa);
  bf16x8_to_f32(b, fb);
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s = fmaf(fa[k], fb[k], s);
  return s;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gate_decode_kernel(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w, const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* region = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* xch = region + p.region;  // the partner's partial sums of this CTA's tokens
  uint8_t* bars = xch + p.xch_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bars);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 144);
  volatile uint32_t* aborted = reinterpret_cast<volatile uint32_t*>(bars + 148);
  volatile uint32_t* peer_aborted = reinterpret_cast<volatile uint32_t*>(bars + 152);
  uint32_t* bx = reinterpret_cast<uint32_t*>(bars + 160);
  uint32_t* bacc = reinterpret_cast<uint32_t*>(bars + 192);
  int32_t* n_ent = reinterpret_cast<int32_t*>(bars + 224);
  // active entries of this CTA's tokens (fused projection), in the stage
  // buffers once the MMAs are done
  uint2* ent = reinterpret_cast<uint2*>(region);
  uint32_t* masks = reinterpret_cast<uint32_t*>(bars + 256);
  int32_t* sslot = reinterpret_cast<int32_t*>(bars + 1280);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int tile = static_cast<int>(blockIdx.x >> 1);
  const int kb0 = rank == 0 ? 0 : p.kb_split;
  const int nloc = (rank == 0 ? p.kb_split : p.nkb) - kb0;   // K blocks of this CTA
  const int rot = nloc > 0 ? (tile * 7 + static_cast<int>(rank) * 3) % nloc : 0;
  const int S = p.stages;
  uint32_t n_loads = 0;  // stage fills issued (producer thread)
  int stage = 0;
  uint32_t phase = 0;

  auto fill = [&](int i) {
    const int kb = kb0 + (i + rot < nloc ? i + rot : i + rot - nloc);
    uint8_t* st = region + static_cast<size_t>(stage) * p.stage_bytes;
    ptx::mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(p.stage_bytes));
    ptx::tma_load_2d(st, &tmap_w, &full[stage], kb * DK, tile * DM);
    ptx::tma_load_2d(st + kA, &tmap_x, &full[stage], kb * DK, 0);
    ++n_loads;
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  };

  const int first = nloc < S ? nloc : S;  // fills that need no free stage
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
    for (int i = 0; i < 8; ++i) bacc[i] = 0u;
    *n_ent = 0;
    ptx::fence_mbar_init();
    for (int i = 0; i < first; ++i) fill(i);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // this CTA has started (waited for before the first remote store); no
  // ordering: the partner writes only words this CTA never writes, and a
  // releasing arrive would also wait for the fills issued above
  ptx::cluster_arrive_relaxed();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int i = first; i < nloc; ++i) {
        if (!pipe_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
          flag(p.status, TWELL_FLAG_TIMEOUT);
          *aborted = 1u;
          break;
        }
        fill(i);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(DM, p.N);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; i < nloc; ++i) {
        if (!pipe_wait(&full[st], ph, p.wait_ns)) {
          flag(p.status, TWELL_FLAG_TIMEOUT);
          *aborted = 1u;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_addr = ptx::smem_u32(region + static_cast<size_t>(st) * p.stage_bytes);
        const uint32_t b_addr = a_addr + kA;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          ptx::mma_bf16(tmem_base, ptx::sdesc_kmajor_sw128(a_addr + kk * 32),
                        ptx::sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                        (i > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&empty[st]);
        if (++st == S) {
          st = 0;
          ph ^= 1u;
        }
      }
      if (ok) ptx::mma_commit(tfull);
    }
  } else {
    // epilogue warps: first, in prefetch mode, zero this CTA's share of the
    // forward's y while W_g streams (the forward adds into y); then wait
    // until the accumulator is complete (the decision is warp-uniform;
    // tcgen05.ld below is warp-collective)
    if (p.y_zero) {
      const size_t n4 = static_cast<size_t>(p.T) * p.D / 4;
      float4* y4 = reinterpret_cast<float4*>(p.y_zero);
      const size_t nthr = static_cast<size_t>(gridDim.x) * (kThreads - 64);
      for (size_t i = static_cast<size_t>(blockIdx.x) * (kThreads - 64) + (threadIdx.x - 64);
           i < n4; i += nthr)
        y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
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
  const int set = (warp - 2) >> 2;  // epilogue set: takes every other 16-token chunk
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  const int own0 = rank == 0 ? 0 : p.half;     // this CTA's tokens: [own0, own1)
  const int own1 = rank == 0 ? p.half : p.N;
  const int oth0 = rank == 0 ? p.half : 0;     // the partner's
  const int oth1 = rank == 0 ? p.N : p.half;
  const uint32_t peer = rank ^ 1u;

  ptx::cluster_wait();  // the partner has started: its shared memory may be written
  if (epi) {
    if (!aborted_here) {
      // the partner's tokens: partial sums into its exchange rows
      ptx::tc_fence_after();
      const uint32_t rx = ptx::mapa(ptx::smem_u32(xch), peer) + static_cast<uint32_t>(n * 4);
      for (int c = oth0 + 16 * set; c < oth1; c += 32) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(c), r);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          ptx::st_cluster_u32(rx + static_cast<uint32_t>((c - oth0 + j) * kRowBytes), r[j]);
      }
    }
    if (warp == 2 && lane == 0)
      ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(const_cast<uint32_t*>(peer_aborted)), peer),
                          aborted_here ? 1u : 0u);
  }
  ptx::tc_fence_before();
  ptx::cluster_arrive();
  ptx::cluster_wait();  // the partner's partial sums and abort flag are here

  const bool go = !aborted_here && *peer_aborted == 0u;  // the same value in every thread
  if (epi && !go) {
    // nothing is packed: the tile's counts of this CTA's tokens say so, so
    // a consumer of the TwELL (the CUDA-core kernel that twell_ffn_decode
    // runs next, for one) finds it empty rather than undefined
    const int t = own0 + (warp - 2) * 32 + lane;
    if (t < own1 && t < p.T) p.cnt[static_cast<size_t>(t) * p.n_t + tile] = 0;
  }
  if (epi && go) {
    ptx::tc_fence_after();
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t bar_id = 1u + static_cast<uint32_t>(set);
    uint32_t bw0 = 0u, bw1 = 0u;  // this warp's block-bitmap words (blocks 0 and 1)
    int par = 0;
    for (int c = own0 + 16 * set; c < own1; c += 32, par ^= 1) {
      uint32_t r[16];
      ptx::tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(c), r);
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j] = *reinterpret_cast<const float*>(xch + (c - own0 + j) * kRowBytes + n * 4);
      ptx::tmem_wait_ld();
      uint32_t* mk = masks + (set * 2 + par) * 64;  // [token j][warp quarter]
      int32_t* ss = sslot + (set * 2 + par) * 16;
      uint32_t m[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        v[j] += __uint_as_float(r[j]);
        m[j] = __ballot_sync(0xffffffffu, c + j < p.T && v[j] > 0.0f);
        if (lane == j) mk[j * 4 + q] = m[j];
        if (c + j < 128) bw0 |= m[j];
        else bw1 |= m[j];
      }
      if (p.z_debug) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c + j < p.T) p.z_debug[static_cast<size_t>(c + j) * p.F + tile * DM + n] = v[j];
      }
      ptx::bar_sync(bar_id, 128);  // the four warps' ballots of these 16 tokens
      // lane j < 16: token c + j's active count and the active neurons of
      // the warps before this one
      int cnt_j = 0, base_j = 0;
      if (lane < 16) {
        const uint4 w = *reinterpret_cast<const uint4*>(mk + lane * 4);
        const int a0 = __popc(w.x), a1 = __popc(w.y), a2 = __popc(w.z), a3 = __popc(w.w);
        cnt_j = a0 + a1 + a2 + a3;
        base_j = (q > 0 ? a0 : 0) + (q > 1 ? a1 : 0) + (q > 2 ? a2 : 0);
      }
      const bool real = lane < 16 && c + lane < p.T;
      const uint32_t spills = __ballot_sync(0xffffffffu, real && cnt_j > p.W);
      if (q == 0 && real) {
        const size_t rt = static_cast<size_t>(c + lane) * p.n_t + tile;
        p.cnt[rt] = static_cast<uint8_t>(cnt_j);
        if (cnt_j > p.W) {
          const int slot = atomicAdd(p.spill_n, 1);
          p.spill_slot[rt] = slot;
          if (slot < p.spill_cap) p.spill_rt[slot] = static_cast<int32_t>(rt);
          else flag(p.status, TWELL_FLAG_SPILL_FULL);
          ss[lane] = slot;
        }
      }
      int e[16];  // this lane's slot for each token (all shuffles issued together)
#pragma unroll
      for (int j = 0; j < 16; ++j) e[j] = __shfl_sync(0xffffffffu, base_j, j) + __popc(m[j] & lt);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (((m[j] >> lane) & 1u) && e[j] < p.W) {
          const size_t o = (static_cast<size_t>(c + j) * p.n_t + tile) * p.W + e[j];
          p.val[o] = v[j];
          p.col[o] = static_cast<uint8_t>(n);
        }
      }
      if (p.Wu_t) {
        // the chunk's active neurons: their W_u and W_d rows on their way to
        // L2, read next by the projection (in this kernel, or the CUDA-core
        // forward right after it); with the projection here, every active
        // entry (slots and spill alike) into the CTA's list
        uint32_t mine = 0u;
#pragma unroll
        for (int j = 0; j < 16; ++j) mine |= m[j];
        if (p.y) {
          int pre[16], tot = 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            pre[j] = tot;
            tot += __popc(m[j]);
          }
          if (tot > 0) {
            int base = 0;
            if (lane == 0) base = atomicAdd(n_ent, tot);
            base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if ((m[j] >> lane) & 1u) {
                const int idx = base + pre[j] + __popc(m[j] & lt);
                if (in_bounds(idx, (own1 - own0) * DM, p.status))
                  ent[idx] =
                      make_uint2(static_cast<uint32_t>((c + j) * DM + n), __float_as_uint(v[j]));
              }
            }
          }
        }
        if ((mine >> lane) & 1u) {
          const size_t roff = (static_cast<size_t>(tile) * DM + n) * p.D;
          ptx::prefetch_l2_bulk(p.Wu_t + roff, static_cast<uint32_t>(p.D) * 2u);
          ptx::prefetch_l2_bulk(p.Wd + roff, static_cast<uint32_t>(p.D) * 2u);
        }
      }
      if (spills != 0u) {
        ptx::bar_sync(bar_id, 128);  // the spill slots of these tokens are published
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if ((spills >> j) & 1u) {
            const int slot = ss[j];
            if (slot < p.spill_cap)
              p.spill_val[static_cast<size_t>(slot) * DM + n] = v[j] > 0.0f ? v[j] : 0.0f;
          }
        }
      }
    }
    if (lane == 0) {
      if (bw0 != 0u) atomicOr(&bacc[q], bw0);
      if (bw1 != 0u) atomicOr(&bacc[4 + q], bw1);
    }
  }
  if (epi) ptx::bar_sync(3, 256);  // both sets' block words and entries are in
  if (epi && go && p.y) {
    // fused projection: each epilogue warp takes whole entries in turn;
    // u = x_t . W_u[:, j] over 16-byte chunks of the rows (lane-strided),
    // reduced across the warp, then y_t += (h u) W_d[j, :] with float4
    // atomics (y zeroed by the call)
    const int nE = *n_ent;
    const int nq = p.D / 8;
    const uint4* x4 = reinterpret_cast<const uint4*>(p.x);
    const uint4* wu4 = reinterpret_cast<const uint4*>(p.Wu_t);
    const uint4* wd4 = reinterpret_cast<const uint4*>(p.Wd);
    for (int ei = warp - 2; ei < nE; ei += 8) {
      const uint2 en = ent[ei];
      const int t = static_cast<int>(en.x / DM);
      const size_t j = static_cast<size_t>(tile) * DM + en.x % DM;
      const uint4* xr = x4 + static_cast<size_t>(t) * nq;
      const uint4* ur = wu4 + j * nq;
      const uint4* dr = wd4 + j * nq;
      float u = 0.0f;
      for (int q0 = 0; q0 < nq; q0 += 256) {
        uint4 xa[8], wa[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int q = q0 + 32 * i + lane;
          if (q < nq) {
            xa[i] = __ldg(xr + q);
            wa[i] = __ldg(ur + q);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (q0 + 32 * i + lane < nq) u += dot8_bf16(xa[i], wa[i]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
      const float a = __uint_as_float(en.y) * u;
      float* yr = p.y + static_cast<size_t>(t) * p.D;
      for (int q0 = 0; q0 < nq; q0 += 256) {
        uint4 wa[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int q = q0 + 32 * i + lane;
          if (q < nq) wa[i] = __ldg(dr + q);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int q = q0 + 32 * i + lane;
          if (q < nq) {
            float f[8];
            bf16x8_to_f32(wa[i], f);
            float4* o = reinterpret_cast<float4*>(yr + 8 * q);
            atomicAdd(o, make_float4(a * f[0], a * f[1], a * f[2], a * f[3]));
            atomicAdd(o + 1, make_float4(a * f[4], a * f[5], a * f[6], a * f[7]));
          }
        }
      }
    }
  }
  // block words: rank 0's tokens all lie in block 0, rank 1's in block 0
  // and / or block 1; rank 1's part of block 0 goes to rank 0
  if (epi && rank == 1 && set == 0 && lane == 0)
    ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(bx + q), 0), bacc[q]);
  ptx::cluster_arrive();
  ptx::cluster_wait();  // rank 1's words are here; neither CTA's memory is read afterwards
  if (epi && set == 0 && go && lane == 0 && p.block_bits) {
    if (rank == 0) p.block_bits[tile * 4 + q] = bacc[q] | bx[q];
    else if (p.N > DM) p.block_bits[static_cast<size_t>(p.F / 32) + tile * 4 + q] = bacc[4 + q];
  }
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
                                const DecodeFfn* ffn, cudaStream_t s) {
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
  p.half = (p.N / 16 + 1) / 2 * 16;
  p.xch_bytes = p.half * kRowBytes;
  const int budget = (dev.max_smem_optin < 232448 ? dev.max_smem_optin : 232448) - 1024 -
                     kBarBytes - p.xch_bytes;
  int stages = budget / p.stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return TWELL_ERR_UNSUPPORTED;
  p.stages = stages;
  p.region = stages * p.stage_bytes;
  // the entry list of the fused projection: at most every neuron of every
  // token of rank 0 (the larger half)
  if (ffn && ffn->y && p.region < p.half * DM * kEntryBytes) return TWELL_ERR_UNSUPPORTED;
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
  p.x = x;
  p.Wu_t = ffn ? ffn->Wu_t : nullptr;
  p.Wd = ffn ? ffn->Wd : nullptr;
  p.y = ffn ? ffn->y : nullptr;
  p.y_zero = ffn && !ffn->y ? ffn->y_zero : nullptr;

  CUtensorMap mx, mw;
  twell_status st;
  if ((st = make_tmap_bf16_2d(&mw, Wg_t, D, F, DK, DM)) != TWELL_OK) return st;
  if ((st = make_tmap_bf16_2d(&mx, x, D, T, DK, static_cast<uint32_t>(p.N))) != TWELL_OK)
    return st;
  const int smem = p.region + p.xch_bytes + kBarBytes + 1024;
  if (cudaFuncSetAttribute(gate_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return TWELL_ERR_CUDA;
  gate_decode_kernel<<<2 * p.n_t, kThreads, smem, s>>>(mx, mw, p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace twell
