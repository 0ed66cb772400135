// tcgen05 kernels over the ELL part of the hybrid training format ("Sparser,
// Faster, Lighter Transformer Language Models", section 2.B.3).
//
// One persistent, warp-specialised kernel per mode (see tc_ell.cuh), tiles
// of 128 x 256 outputs, K in blocks of 64:
//   warp 0      TMA producer: the dense operands, and for the expanded modes
//               the weight or activation rows as an N-major operand (four
//               64 x 64 boxes, one 128-byte swizzle atom column each)
//   warp 1      TMEM allocation and the MMA issue (one thread)
//   warps 2-5   epilogue, one TMEM lane quarter each, two accumulators in
//               flight
//   warps 6-21  (expanded modes) four groups of four warps, taking the stages
//               in turn, write the fp16 A tile of a stage from the raw ELL
//               slots: zero it and scatter the entries whose column falls in
//               the K block, then fence to the async proxy and arrive.  They
//               issue no global loads of their own, so the proxy fence has no
//               loads in flight to wait for.
//   warp 22     (expanded modes) TMA producer of the raw ELL slots (columns
//               and fp16 values of the rows of the stage) into a ring of
//               their own, freed by the expansion warps: the raw data runs
//               ahead of the A/B stages, which the MMA frees.
// Shared-memory stages: [A 16 KB][B 32 KB] x 4, plus the raw ring (ROWS:
// 2 slots of 128 rows, one per 128-column tile = two K blocks; TRANS: 4
// slots of 64 rows, one per K block).
//
// The sampled epilogue stages each 32-column accumulator chunk in a private
// shared-memory row per thread (XOR-swizzled by 16-byte chunk) and walks the
// row's ELL entries of the tile in column order, so every entry reads its
// accumulator once.
//
// Every wait is bounded (about a second); a wait that runs out sets
// TWELL_FLAG_TIMEOUT and the CTA leaves its loops; before it frees its TMEM
// and exits, every MMA it issued completes (a commit to a barrier of its
// own, waited for) and the TMA loads it issued land (a bounded 100 us wait:
// their completion barrier may no longer complete once another role left).
#include <cuda_fp16.h>

#include "gemm.cuh"
#include "ptx.cuh"
#include "scale.cuh"
#include "bounds.cuh"
#include "tc_ell.cuh"

namespace twell {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int kExpandBar = 1;     // named barriers 1 .. kGroups: the expansion groups
constexpr int kGroups = 4;        // expansion groups of four warps, taking stages in turn
constexpr int kRawWarp = 6 + 4 * kGroups;

constexpr int RAW_COLS = 4096;  // raw slot: columns of <= 128 rows x C <= 32, then values

template <int MODE>
struct TcCfg {
  static constexpr bool SAMPLE = MODE <= TC_SAMPLE_DA;
  static constexpr int STAGES = 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGING = SAMPLE ? 128 * 128 : 0;
  static constexpr int RAW_ROWS = MODE == TC_ROWS ? 128 : 64;
  static constexpr int RAW_SLOT = SAMPLE ? 0 : RAW_COLS + RAW_ROWS * 2 * 32;
  static constexpr int RAW_SLOTS = SAMPLE ? 0 : (MODE == TC_ROWS ? 2 : 4);
  static constexpr int THREADS = SAMPLE ? 192 : 32 * (kRawWarp + 1);
  static constexpr int SMEM =
      STAGES * STAGE_BYTES + STAGING + RAW_SLOTS * RAW_SLOT + 512 + 1024;
};

// fp16 bits of v; a |v| beyond the fp16 range sets TWELL_FLAG_RANGE
__device__ __forceinline__ uint16_t f16_bits(float v, int32_t* status) {
  if (fabsf(v) > 65504.0f) atomicOr(status, TWELL_FLAG_RANGE);
  return __half_as_ushort(__float2half_rn(v));
}

// Per-unit decomposition shared by every role.  Returns 0 (nothing to do),
// 1 (a tile with K blocks [kb0, kb1)) or 2 (a TRANS tile with an empty K
// range: its output is zero).
// With ks = 2 K parts per tile, unit u is part u % 2 of tile u / 2; the parts
// split the K blocks in halves (ROWS: at an even block, as a raw ELL slot
// covers two) and one of them may be empty.
struct Units {
  int num_m, num_n, total_kb, kb_per_seg;
  int n_rows;
  int ks;
  __device__ int info(int u, int mode, int& m_blk, int& n_blk, int& kb0, int& kb1) const {
    const int t = u / ks, part = u - t * ks;
    m_blk = t / num_n;
    n_blk = t % num_n;
    int mid = total_kb / 2;
    if (mode == TC_ROWS) mid &= ~1;
    kb0 = ks == 1 || part == 0 ? 0 : mid;
    kb1 = ks == 1 || part == 1 ? total_kb : mid;
    if (mode != TC_TRANS && m_blk * BM >= n_rows) return 0;
    if (total_kb == 0) return mode == TC_TRANS ? 2 : 0;
    return kb1 > kb0 ? 1 : 0;
  }
};

template <int MODE>
__global__ void __launch_bounds__(TcCfg<MODE>::THREADS, 1)
    tc_ell_kernel(const __grid_constant__ TcMaps maps, const TcArgs p, int num_m, int num_n) {
  using Cfg = TcCfg<MODE>;
  constexpr int ST = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* staging = smem + ST * Cfg::STAGE_BYTES;
  uint8_t* raw = staging + Cfg::STAGING;
  uint64_t* full = reinterpret_cast<uint64_t*>(raw + Cfg::RAW_SLOTS * Cfg::RAW_SLOT);
  uint64_t* ready = full + ST;
  uint64_t* empty = ready + ST;
  uint64_t* tfull = empty + ST;
  uint64_t* tempty = tfull + 2;
  uint64_t* raw_full = tempty + 2;
  uint64_t* raw_empty = raw_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_empty + 4);
  uint64_t* drain = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // abort path: MMA drain
  volatile uint32_t* aborted = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int C = p.C;

  Units U;
  U.num_m = num_m;
  U.num_n = num_n;
  U.n_rows = min(*p.n_rows, p.rows_cap);
  U.ks = p.ksplit > 1 ? 2 : 1;
  if (MODE == TC_ROWS) {
    U.kb_per_seg = p.F / BK;
    U.total_kb = p.nseg * U.kb_per_seg;
  } else if (MODE == TC_TRANS) {
    U.kb_per_seg = (U.n_rows + BK - 1) / BK;
    U.total_kb = p.nseg * U.kb_per_seg;
  } else {
    U.kb_per_seg = p.D / BK;
    U.total_kb = p.nseg * U.kb_per_seg;
  }
  const int num_units = num_m * num_n * U.ks;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < ST; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&ready[s], 4);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 128);
    }
    for (int r = 0; r < 4; ++r) {
      ptx::mbar_init(&raw_full[r], 1);
      // ROWS: both expansion groups read each slot (one half of the tile each)
      ptx::mbar_init(&raw_empty[r], MODE == TC_ROWS ? 8 : 4);  // ROWS: the two groups of a tile
    }
    ptx::mbar_init(drain, 1);
    *aborted = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 2 * BN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        int m_blk, n_blk, kb0, kb1;
        if (U.info(u, MODE, m_blk, n_blk, kb0, kb1) != 1) continue;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u)) {
            { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          if (Cfg::SAMPLE) {
            const int seg = kb / U.kb_per_seg;
            const int kl = kb - seg * U.kb_per_seg;
            ptx::mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
            ptx::tma_load_2d(sA, &maps.a[seg], &full[stage], kl * BK, m_blk * BM);
            ptx::tma_load_2d(sB, &maps.b[0], &full[stage], kl * BK, n_blk * BN);
          } else {
            const int seg = kb / U.kb_per_seg;
            const int kl = kb - seg * U.kb_per_seg;
            const int n_base = n_blk * BN;
            int atoms = (p.D - n_base) / 64;
            if (atoms > 4) atoms = 4;
            ptx::mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(atoms * 8192));
            for (int q = 0; q < atoms; ++q)
              ptx::tma_load_2d(sB + q * 8192, &maps.b[seg], &full[stage], n_base + 64 * q,
                               kl * BK);
          }
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = p.f16_ops ? ptx::idesc_f16_f32(BM, BN, false, !Cfg::SAMPLE)
                                   : ptx::idesc_bf16_f32(BM, BN, false, !Cfg::SAMPLE);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        int m_blk, n_blk, kb0, kb1;
        if (U.info(u, MODE, m_blk, n_blk, kb0, kb1) != 1) continue;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        ++local;
        if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u)) {
          { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool first = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase) ||
              (!Cfg::SAMPLE && !ptx::mbar_wait(&ready[stage], phase))) {
            { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = Cfg::SAMPLE ? ptx::sdesc_kmajor_sw128(b_addr + kk * 32)
                                            : ptx::sdesc_mnmajor_sw128(b_addr + kk * 2048,
                                                                       8192, 1024);
            ptx::mma_bf16(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + kk * 32), bd, idesc,
                          first ? 0u : 1u);
            first = false;
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        ptx::mma_commit(&tfull[acc]);
      }
    }
  } else if (warp == kRawWarp) {
    // ------------------------------------------- raw ELL slots (TMA) ring
    if (!Cfg::SAMPLE && lane == 0) {
      int slot = 0;
      uint32_t rphase = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        int m_blk, n_blk, kb0, kb1;
        if (U.info(u, MODE, m_blk, n_blk, kb0, kb1) != 1) continue;
        // ROWS: one raw slot per tile (two K blocks); TRANS: one per K block
        for (int kb = kb0; kb < kb1; kb += (MODE == TC_ROWS ? 2 : 1)) {
          if (!ptx::mbar_wait(&raw_empty[slot], rphase ^ 1u)) {
            { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          const int seg = kb / U.kb_per_seg;
          const int kl = kb - seg * U.kb_per_seg;
          const int kt = MODE == TC_ROWS ? (kl >> 1) : m_blk;
          const int row0 = MODE == TC_ROWS ? m_blk * BM : kl * BK;
          uint8_t* sr = raw + slot * Cfg::RAW_SLOT;
          ptx::mbar_arrive_expect_tx(&raw_full[slot],
                                     static_cast<uint32_t>(Cfg::RAW_ROWS * 3 * C));
          ptx::tma_load_2d(sr, &maps.cols, &raw_full[slot], kt * C, row0);
          ptx::tma_load_2d(sr + RAW_COLS, &maps.vals[seg], &raw_full[slot], kt * C, row0);
          if (++slot == Cfg::RAW_SLOTS) {
            slot = 0;
            rphase ^= 1u;
          }
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------- ELL expansion into A tiles
    // kGroups groups of four warps take the stages in turn (group g the
    // stages with sequence number = g mod kGroups), so each has kGroups MMA
    // stage times per tile.
    if (!Cfg::SAMPLE) {
      const int grp = (warp - 6) >> 2;
      const int x = (threadIdx.x - 192) & 127;  // thread within the group
      const uint32_t rr = static_cast<uint32_t>(x & 63);
      const uint32_t bar_id = kExpandBar + static_cast<uint32_t>(grp);
      int stage = 0, slot = 0, seq = 0;
      uint32_t phase = 0, rphase = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        int m_blk, n_blk, kb0, kb1;
        if (U.info(u, MODE, m_blk, n_blk, kb0, kb1) != 1) continue;
        for (int kb = kb0; kb < kb1; ++kb, ++seq) {
          const int kl = kb % U.kb_per_seg;
          // last use of the raw slot: ROWS, the second half of the tile (or
          // the unit's last K block); TRANS, every K block
          const bool slot_done = MODE == TC_TRANS || (kl & 1) == 1 || kb + 1 == kb1;
          if (seq % kGroups == grp) {
            const bool ok = ptx::mbar_wait(&empty[stage], phase ^ 1u) &&
                            ptx::mbar_wait(&raw_full[slot], rphase);
            if (MODE == TC_TRANS ? ptx::bar_any(bar_id, 128, !ok)
                                 : !__all_sync(0xffffffffu, ok)) {
              if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
              goto done;
            }
            uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
            const uint8_t* sr = raw + slot * Cfg::RAW_SLOT;
            const uint16_t* rv = reinterpret_cast<const uint16_t*>(sr + RAW_COLS);
            // Zero the A tile with contiguous 512-byte warp stores (conflict
            // free): ROWS, each warp its own 32 rows (4 KB); TRANS, the whole
            // tile across the group.
            if (MODE == TC_ROWS) {
              uint4* z = reinterpret_cast<uint4*>(sA + (x >> 5) * 4096) + lane;
#pragma unroll
              for (int j = 0; j < 8; ++j) z[32 * j] = make_uint4(0u, 0u, 0u, 0u);
              __syncwarp();  // the warp's rows are zero before its lanes scatter into them
            } else {
              uint4* z = reinterpret_cast<uint4*>(sA) + x;
#pragma unroll
              for (int j = 0; j < 8; ++j) z[128 * j] = make_uint4(0u, 0u, 0u, 0u);
              ptx::bar_sync(bar_id, 128);  // the tile is zero before any scatter
            }
            // Slots of this thread, loaded with 16-byte reads: ROWS, row x of
            // the tile (C / 16 groups of 16 slots); TRANS, K row rr of the
            // block, slot group x / 64.  Rows past the ELL rows read as
            // 0xff columns.  Each 4-slot word is skipped when no lane of the
            // warp has an entry of this A tile in it.
            const int ngroups = MODE == TC_ROWS ? C / 16 : 1;
            const int g0 = MODE == TC_ROWS ? 0 : (x >> 6) * 16;
            const int srow = MODE == TC_ROWS ? x : static_cast<int>(rr);
            const bool live = MODE == TC_ROWS
                                  ? m_blk * BM + x < U.n_rows
                                  : (kl * BK + static_cast<int>(rr) < U.n_rows && g0 < C);
            const uint32_t half = static_cast<uint32_t>(kl & 1);
            // chunk j of a raw row lies at chunk j ^ (the row's address bits
            // 7..): columns (32-byte rows, C == 32) (row >> 2) & 1; values
            // (2C-byte rows) (row >> 1) & 3 for C == 32, (row >> 2) & 1 for 16
            const int cswz = C == 32 ? (srow >> 2) & 1 : 0;
            const int vswz = C == 32 ? (srow >> 1) & 3 : (srow >> 2) & 1;
            for (int gi = 0; gi < ngroups; ++gi) {
              const int cj = (g0 >> 4) + gi;  // 16-slot group = column chunk
              const uint4 cv =
                  *reinterpret_cast<const uint4*>(sr + srow * C + 16 * (cj ^ cswz));
              const uint8_t* vr = reinterpret_cast<const uint8_t*>(rv) + 2 * srow * C;
              const uint4 v0 = *reinterpret_cast<const uint4*>(vr + 16 * ((2 * cj) ^ vswz));
              const uint4 v1 = *reinterpret_cast<const uint4*>(vr + 16 * ((2 * cj + 1) ^ vswz));
              const uint32_t cw[4] = {live ? cv.x : ~0u, live ? cv.y : ~0u, live ? cv.z : ~0u,
                                      live ? cv.w : ~0u};
              const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                // 0xff per slot byte that is an entry of this A tile
                const uint32_t hit =
                    MODE == TC_ROWS ? __vcmpeq4(cw[q] & 0xc0c0c0c0u, half ? 0x40404040u : 0u)
                                    : __vcmpltu4(cw[q], 0x80808080u);
                if (!__any_sync(0xffffffffu, hit != 0u)) continue;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                  if (!((hit >> (8 * b)) & 1u)) continue;
                  const int e = 4 * q + b;
                  const uint32_t c = (cw[q] >> (8 * b)) & 0xffu;
                  const uint16_t v = static_cast<uint16_t>(vw[e >> 1] >> (16 * (e & 1)));
                  if (MODE == TC_ROWS) {
                    // A row x, K = column c of the stage's half
                    const uint32_t k = c & 63u;
                    *reinterpret_cast<uint16_t*>(
                        sA + x * 128 + ((((k >> 3) ^ (x & 7)) << 4) | ((k & 7) << 1))) = v;
                  } else {
                    // A row c (neuron of the tile), K = ELL row rr of the block
                    *reinterpret_cast<uint16_t*>(
                        sA + c * 128 + ((((rr >> 3) ^ (c & 7u)) << 4) | ((rr & 7) << 1))) = v;
                  }
                }
              }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(&ready[stage]);
              if (MODE == TC_ROWS || slot_done) ptx::mbar_arrive(&raw_empty[slot]);
            }
          }
          if (slot_done) {
            if (++slot == Cfg::RAW_SLOTS) {
              slot = 0;
              rphase ^= 1u;
            }
          }
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const float lambda_s =
        p.amax ? p.lambda * pow2_scale(p.amax, p.amax_floor, false) : p.lambda;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    uint8_t* my_stage = staging + r * 128;
    int local = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      int m_blk, n_blk, kb0, kb1;
      const int kind = U.info(u, MODE, m_blk, n_blk, kb0, kb1);
      if (kind == 0) continue;
      if (MODE == TC_TRANS && kind == 2) {  // no ELL rows: the product is zero
        float* o = p.out + static_cast<int64_t>(m_blk * BM + r) * p.ldo + n_blk * BN;
        for (int n = 0; n < BN && n_blk * BN + n < p.D; n += 4)
          *reinterpret_cast<float4*>(o + n) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      ++local;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&tfull[acc], acc_phase))) {
        if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
        goto done;
      }
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if (Cfg::SAMPLE) {
        // Row r of the tile is ELL row i.  Per (row, tile) the thread loads
        // the C column indices, the h values (and for SAMPLE_DA the saved
        // u) with 16-byte loads at once, then walks its slots for each
        // 32-column accumulator chunk: slot s is an entry of chunk c iff
        // s < count and its column's bits 5-6 equal c (columns ascending).
        // Groups of four slots that no lane of the warp needs are skipped.
        const int i = m_blk * BM + r;
        const bool valid = i < U.n_rows;
#pragma unroll 1
        for (int t2 = 0; t2 < 2; ++t2) {
          const int kt = n_blk * 2 + t2;
          if (kt >= p.n_t) break;  // uniform
          const size_t rt = static_cast<size_t>(valid ? i : 0) * p.n_t + kt;
          const size_t base = rt * static_cast<size_t>(C);
          const int cnt = valid ? p.ell_cnt[rt] : 0;
          uint32_t cw[8];
          float hv[32], uv[32];
          {
            const uint4* cp = reinterpret_cast<const uint4*>(p.ell_col + base);
            const float4* hp = reinterpret_cast<const float4*>(p.ell_val + base);
            const float4* up = reinterpret_cast<const float4*>(p.u_ell + base);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const uint4 c4 = (g == 0 || C == 32) ? __ldg(cp + g) : make_uint4(~0u, ~0u, ~0u, ~0u);
              cw[4 * g] = c4.x;
              cw[4 * g + 1] = c4.y;
              cw[4 * g + 2] = c4.z;
              cw[4 * g + 3] = c4.w;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const bool in = q < 4 || C == 32;
              const float4 h4 = in ? __ldg(hp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
              hv[4 * q] = h4.x;
              hv[4 * q + 1] = h4.y;
              hv[4 * q + 2] = h4.z;
              hv[4 * q + 3] = h4.w;
              if (MODE == TC_SAMPLE_DA) {
                const float4 u4 = in ? __ldg(up + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                uv[4 * q] = u4.x;
                uv[4 * q + 1] = u4.y;
                uv[4 * q + 2] = u4.z;
                uv[4 * q + 3] = u4.w;
              }
            }
          }
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(t2 * 128 + c * 32), v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(my_stage + ((j ^ (r & 7)) << 4)) =
                  make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              // 0xff per slot byte of word q that is an entry of chunk c
              const uint32_t w = cw[q];
              const uint32_t in_chunk = __vcmpeq4(w & 0xe0e0e0e0u, static_cast<uint32_t>(c) *
                                                                   0x20202020u);
              const uint32_t live = (4 * q < cnt) ? in_chunk : 0u;
              if (!__any_sync(0xffffffffu, live != 0u)) continue;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const int sidx = 4 * q + b;
                if (sidx >= cnt || !((live >> (8 * b)) & 1u)) continue;
                const int cl = (w >> (8 * b)) & 31;
                const float val = *reinterpret_cast<const float*>(
                    my_stage + ((((cl >> 2) ^ (r & 7)) << 4) | ((cl & 3) << 2)));
                const size_t pos = base + sidx;
                if (MODE == TC_SAMPLE_U) {
                  p.u_ell[pos] = val;
                  p.a_ell[pos] = f16_bits(hv[sidx] * val, p.status);
                } else {
                  const float dz = fmaf(val, uv[sidx], lambda_s);
                  const uint16_t dz_hi = f16_bits(dz, p.status);
                  p.dz_ell[pos] = dz_hi;
                  if (p.dz_lo_ell)
                    p.dz_lo_ell[pos] = __half_as_ushort(
                        __float2half_rn(dz - __half2float(__ushort_as_half(dz_hi))));
                  p.du_ell[pos] = f16_bits(val * hv[sidx], p.status);
                  p.a_ell[pos] = f16_bits(hv[sidx] * uv[sidx], p.status);
                }
              }
            }
          }
        }
      } else {
        int64_t orow = 0;
        bool valid = true;
        if (MODE == TC_ROWS) {
          const int i = m_blk * BM + r;
          valid = i < U.n_rows;
          orow = valid ? p.row_idx[i] : 0;
          if (valid && p.row_limit && !in_bounds(orow, p.row_limit, p.status)) {
            valid = false;
            orow = 0;
          }
        } else {
          orow = m_blk * BM + r;
        }
        float* o = p.out + orow * p.ldo + n_blk * BN;
        const float osc = p.amax ? pow2_scale(p.amax, p.amax_floor, true) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          if (n_blk * BN + c * 32 >= p.D) break;  // uniform
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), v);
          ptx::tmem_wait_ld();
          if (valid) {
            float4* o4 = reinterpret_cast<float4*>(o + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 q = make_float4(osc * __uint_as_float(v[4 * j]),
                                           osc * __uint_as_float(v[4 * j + 1]),
                                           osc * __uint_as_float(v[4 * j + 2]),
                                           osc * __uint_as_float(v[4 * j + 3]));
              // two K parts add into the zeroed output: 0 + a + b is the same
              // sum in either order, so repeats stay bit-identical
              if (U.ks > 1)
                atomicAdd(o4 + j, q);
              else
                o4[j] = q;
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
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
    ptx::tmem_dealloc(tmem_base, 2 * BN);
  }
}

template <int MODE>
twell_status tc_launch(const TcMaps& maps, const TcArgs& a, const DeviceInfo& dev,
                       cudaStream_t s) {
  using Cfg = TcCfg<MODE>;
  static_assert(Cfg::SMEM <= 232448, "shared memory budget");
  auto kern = tc_ell_kernel<MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  const int num_m = MODE == TC_TRANS ? a.F / BM : (a.rows_cap + BM - 1) / BM;
  const int num_n = MODE <= TC_SAMPLE_DA ? (a.F + BN - 1) / BN : (a.D + BN - 1) / BN;
  long long units = static_cast<long long>(num_m) * num_n;
  if (units == 0) return TWELL_OK;
  // TRANS, and ROWS over several segments, with fewer than eight tiles per
  // SM: two K parts per tile, so the last, partial round of tiles costs half
  // a tile, for a zeroed output and atomic additions.  Measured at the
  // 2B-class layer (648 TRANS tiles, 1125 ROWS tiles on 152 SMs): backward
  // 5.16 -> 5.03 ms; the forward's one-segment ROWS lost more to the zeroing
  // and the atomics than it gained (1.31 -> 1.33 ms), so it keeps one part.
  TcArgs ak = a;
  ak.ksplit = 1;
  if (!Cfg::SAMPLE && (MODE == TC_TRANS || a.nseg > 1) && units < 8LL * dev.sm_count) {
    ak.ksplit = 2;
    units *= 2;
    if (MODE == TC_TRANS) {
      if (cudaMemset2DAsync(a.out, static_cast<size_t>(a.ldo) * 4, 0,
                            static_cast<size_t>(a.D) * 4, static_cast<size_t>(a.F), s) !=
          cudaSuccess)
        return TWELL_ERR_CUDA;
    } else {
      twell_status st = zero_rows(a.out, a.ldo, a.row_idx, a.rows_cap, a.n_rows, a.D, s,
                                  a.row_limit, a.status);
      if (st != TWELL_OK) return st;
    }
  }
  const int grid = static_cast<int>(units < dev.sm_count ? units : dev.sm_count);
  kern<<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(maps, ak, num_m, num_n);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace

bool tc_supported(int32_t D, int32_t F, int32_t C) {
  return D > 0 && D % 64 == 0 && F > 0 && F % TWELL_TILE == 0 && (C == 16 || C == 32);
}

twell_status tc_map_a(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t D,
                      int64_t pitch) {
  return make_tmap_2d(m, 2, base, D, rows, BK, BM, (pitch ? pitch : D) * 2, 128);
}

twell_status tc_map_w_kmajor(CUtensorMap* m, const uint16_t* base, int64_t F, int64_t D) {
  return make_tmap_2d(m, 2, base, D, F, BK, BN, D * 2, 128);
}

twell_status tc_map_mn(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t D,
                       int64_t pitch) {
  return make_tmap_2d(m, 2, base, D, rows, 64, BK, (pitch ? pitch : D) * 2, 128);
}

// Raw ELL boxes land swizzled so that a thread reading its own row's 16-byte
// chunks hits distinct bank groups: columns (C bytes per row) with the 32-byte
// swizzle when C == 32, values (2 C bytes per row) with the 2 C-byte swizzle.
twell_status tc_map_cols(CUtensorMap* m, const uint8_t* base, int64_t rows, int64_t n_t,
                         int64_t C, int box_rows) {
  return make_tmap_2d(m, 1, base, n_t * C, rows, static_cast<uint32_t>(C),
                      static_cast<uint32_t>(box_rows), n_t * C, C == 32 ? 32 : 0);
}

twell_status tc_map_vals(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t n_t,
                         int64_t C, int box_rows) {
  return make_tmap_2d(m, 2, base, n_t * C, rows, static_cast<uint32_t>(C),
                      static_cast<uint32_t>(box_rows), n_t * C * 2, static_cast<int>(2 * C));
}

twell_status tc_run(const TcMaps& maps, const TcArgs& a, const DeviceInfo& dev,
                    cudaStream_t s) {
  if (!tc_supported(a.D, a.F, a.C) || a.n_t != a.F / TWELL_TILE || a.rows_cap < 0 ||
      !a.n_rows || !a.status)
    return TWELL_ERR_INVALID;
  switch (a.mode) {
    case TC_SAMPLE_U:
    case TC_SAMPLE_DA:
      if (a.nseg < 1 || a.nseg > 2) return TWELL_ERR_INVALID;
      return a.mode == TC_SAMPLE_U ? tc_launch<TC_SAMPLE_U>(maps, a, dev, s)
                                   : tc_launch<TC_SAMPLE_DA>(maps, a, dev, s);
    case TC_ROWS:
      if (a.nseg < 1 || a.nseg > kTcMaxSeg) return TWELL_ERR_INVALID;
      return tc_launch<TC_ROWS>(maps, a, dev, s);
    case TC_TRANS:
      if (a.nseg < 1 || a.nseg > kTcMaxSeg) return TWELL_ERR_INVALID;
      return tc_launch<TC_TRANS>(maps, a, dev, s);
  }
  return TWELL_ERR_INVALID;
}

}  // namespace twell
