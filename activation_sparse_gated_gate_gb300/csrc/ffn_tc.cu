// Tensor-core (union-gather) variant of the fused up + down projection from
// a TwELL gate ("Sparser, Faster, Lighter Transformer Language Models",
// section 2.B.2: the up and down projections are computed only for the
// gate's active neurons, with the kernels built to keep the tensor cores
// busy).
//
// The rows of a block of 128 tokens share one gathered operand: the union U
// of their active neurons (ascending).  The forward is then two dense
// tcgen05 GEMMs over that union alone:
//   up    u = x_blk . W_u[:, U]          (128 x |U|, K = D, bf16), and in the
//         epilogue a = fp16(h u) at each row's own active neurons, 0 at the
//         other union positions, written to a [T][Fp] fp16 scratch matrix in
//         union-position order
//   down  y_blk = a_blk . W_d[U, :]      (128 x D, K = |U|, fp16 operands:
//         W_d converted into the workspace), fp32 out
// (fp16 for the down GEMM: a bf16 a = h u adds up to 2^-8 |h u| per term,
// which over 30-40 terms of a row exceeded 2e-2 * RMS(y); fp16 adds 2^-11.)
// The union's weight rows are gathered into the 128-byte-swizzled operand
// tiles by four warps with 16-byte cp.async copies (each copy lands where a
// TMA box with that swizzle would put it); the token tiles (x, a) come by
// TMA.
//
// Optionally (twell_ffn_fwd_tc_sorted) token blocks are formed by activity,
// not by position: the work of a block
// is set by its union, and the union of 128 tokens grows with their summed
// activity in a concave way (1 - prod(1 - p_t) per neuron), so blocks of
// tokens with similar counts of active neurons have a smaller total union
// than blocks of consecutive tokens wherever the per-token activity varies
// (a heavy-tailed batch: 55 % of d_ff per block instead of 73 % in the
// 1.5B-class workload).  Two small kernels sort the tokens, stably, by a
// logarithmic bucket of their active count (eight buckets per octave) into a
// permutation; the union-bitmap kernel also copies x into that order for the
// up GEMM's TMA tiles, the down epilogue writes each y row to its token, and the rest of
// the pipeline works on token positions.  In a batch whose tokens are about
// equally active the sort gains nothing and costs its kernels, so the plain
// entry point keeps blocks of consecutive tokens.
//
// A block whose union is nearly every neuron runs dense: U is then every
// neuron in order, its weight tiles are contiguous and come by TMA (about
// 1.26 times the tensor-pipe rate of the row gathers).
//
// The union bitmap of each block comes from the gate kernel (TwELL
// block_bits, blocks of consecutive tokens only) or from a small kernel over
// the TwELL entries of its tokens; a scan kernel turns it into U (padded
// with neuron 0 to a multiple of 256), the per-word position prefix and the
// list of (block, 256-position chunk) units of the up GEMM.  The up epilogue
// finds its row's entries in the chunk from the TwELL itself while the
// chunk's MMAs run.
//
// Both GEMMs: one persistent CTA per SM, tiles of 128 x 256 outputs, K in
// blocks of 64, four shared-memory stages [A 16 KB][B 32 KB].  A CTA takes
// its units (tiles) one at a time from a ticket counter of the launch, not a
// fixed share: unit costs differ (dense or gathered weight tiles, union
// sizes, heavy rows in the up epilogue), and a fixed round-robin share left
// the average SM idle for a quarter of the sorted call's up GEMM at the
// 1.5B-class layer (max / mean active cycles 1.28; with tickets 1.12, the
// call 526 -> 497 us).  The producer claims the next unit near the end of
// the current one and hands its record to the other roles through a ring of
// unit records in shared memory.  Roles:
//   warp 0      TMA producer of the A tiles, unit tickets
//   warp 1      TMEM allocation (two 256-column accumulators) and MMA issue
//   warps 2-9   epilogue: two sets of four warps, one TMEM lane quarter per
//               warp; set s writes columns 128 s .. 128 s + 127 of the tile
//   warps 10-17 B gather: four groups of two warps, group g filling stage g
//               (32 copies per thread), marking it full once its copies
//               have landed and it has fenced them to the async proxy
// Every wait is bounded (about a second); a wait that runs out sets
// TWELL_FLAG_TIMEOUT and the CTA leaves its loops; before it frees its TMEM
// and exits, every MMA it issued completes (a commit to a barrier of its
// own, waited for) and the TMA loads it issued land (a bounded 100 us wait:
// their completion barrier may no longer complete once another role left).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bounds.cuh"
#include "fused.cuh"
#include "ptx.cuh"
#include "tc_ell.cuh"

namespace twell {
namespace {

constexpr int UG_BM = 128;
constexpr int UG_BN = 256;
constexpr int UG_BK = 64;
constexpr int UG_ST = 4;
constexpr int UG_A = UG_BM * UG_BK * 2;
constexpr int UG_B = UG_BN * UG_BK * 2;
constexpr int UG_STAGE = UG_A + UG_B;
constexpr int UG_GROUP = 64;            // threads of a gather group (one per stage)
constexpr int UG_EPI = 256;             // epilogue threads: two sets of four warps
constexpr int UG_GATHER0 = 64 + UG_EPI; // first thread of the gather groups
constexpr int UG_THREADS = UG_GATHER0 + UG_ST * UG_GROUP;
constexpr int UG_HSLOTS = 16;           // up epilogue: gate values staged per row and set
constexpr int UG_RING = 8;              // unit records in flight between the roles
// arrivals that free a unit-ring slot: the MMA thread, each gather warp, each epilogue warp
constexpr int UG_RING_READERS = 1 + UG_ST * UG_GROUP / 32 + UG_EPI / 32;
// A block whose union holds at least this percentage of the neurons runs as
// a dense block (every neuron, weight tiles by TMA instead of row gathers).
// Measured at the 1.5B-class layer: a dense block costs about 1 / 1.26 of a
// gathered block of the same width, so the whole tile wins from a union of
// about 80 % (thresholds 60 / 70 / 80 % / never: sorted call 529 / 514 / 513 /
// 531 us, and 70 % made the plain call's 72 % unions slower, 632 against 571).
#ifndef UG_DENSE_PCT
#define UG_DENSE_PCT 80
#endif

// Shared memory: [stages][output staging: 8 epilogue warps x one 32 x 32
// chunk][barriers and the unit ring 512 B][up: gate-value slots 2 sets x 128
// rows x UG_HSLOTS fp32]
template <int MODE>
struct UgSmem {
  static constexpr int STG_BUF = MODE == 0 ? 32 * 32 * 2 : 32 * 32 * 4;
  static constexpr int STG = UG_ST * UG_STAGE;
  static constexpr int BARS = STG + 8 * STG_BUF;
  static constexpr int SLOTS = BARS + 512;
  static constexpr int BYTES = SLOTS + (MODE == 0 ? 2 * UG_BM * UG_HSLOTS * 4 : 0) + 1024;
};
constexpr int UG_PREP_THREADS = 256;
constexpr int UG_ROWS_PER_CTA = 16;     // preparation: rows per CTA
constexpr int UG_MAX_F = 32768;         // bitmap words <= 4 per preparation thread

enum { UG_UP = 0, UG_DOWN = 1 };

struct UgArgs {
  // TwELL gate
  const float* val;
  const uint8_t* col;
  const uint8_t* cnt;
  const int32_t* spill_slot;
  const float* spill_val;
  int32_t spill_cap;
  int32_t T, D, F, Fp, nw, n_t, W, n_m, nj, nN;
  const uint16_t* Wu_t;
  const uint16_t* Wd;   // bf16 (converted by ug_f16_kernel)
  uint16_t* Wd16;       // fp16 copy in the workspace (the down GEMM's B)
  float* y;
  // workspace
  int32_t* ctr;     // [0]: units of the up GEMM; [1], [2]: next-unit tickets of the up and
                    // down GEMMs (zero before the launch)
  uint32_t* gbm;    // [n_m][gbm_pitch] union bitmap of each block (F / 32 words used)
  int32_t gbm_pitch;
  int32_t* nU;      // [n_m] union sizes (a dense block: F)
  int8_t* dense;    // [n_m] 1: the block's union is every neuron (see UG_DENSE_PCT)
  int32_t dense_min;  // union size from which a block runs dense (0: never)
  int32_t* Ulist;   // [n_m][Fp] union neurons, ascending, padded with 0
  int32_t* units;   // [n_m * nj] up-GEMM units (block * nj + chunk)
  int32_t* wpre;    // [n_m][nw] union position of each bitmap word's first bit
  uint16_t* abuf;   // [T][Fp] a = fp16(h u) in union-position order
  // token order (sorted variant): position i holds token perm[i]; NULL:
  // position i is token i
  int32_t* perm;    // [T]
  uint8_t* keys;    // [T] activity bucket of each token
  int32_t* hist;    // [n_sort][UG_NBUCKET] bucket counts, then start positions
  int32_t n_sort;   // sort CTAs (UG_SORT_THREADS tokens each)
  const uint16_t* x;  // [T][D] bf16, token order
  uint16_t* xp;       // [T][D] bf16, position order (the up GEMM's A)
  int32_t* status;
};

constexpr int UG_SORT_THREADS = 1024;  // tokens per sort CTA
constexpr int UG_NBUCKET = 128;        // activity buckets (eight per octave)

struct UgLayout {
  size_t ctr, gbm, nU, dense, Ulist, units, wpre, abuf, wd16, perm, keys, hist, xp, bytes;
  int64_t Fp, nw, n_m, nj, n_sort;
};

inline size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

UgLayout ug_layout(int64_t T, int64_t D, int64_t F, bool sorted) {
  UgLayout L{};
  L.Fp = (F + 255) / 256 * 256;
  L.nw = L.Fp / 32;
  L.n_m = (T + UG_BM - 1) / UG_BM;
  L.nj = L.Fp / 256;
  size_t o = 0;
  L.ctr = o;
  o += 256;
  L.gbm = o;
  o = up256(o + static_cast<size_t>(L.n_m) * L.nw * 4);
  L.nU = o;
  o = up256(o + L.n_m * 4);
  L.dense = o;
  o = up256(o + L.n_m);
  L.Ulist = o;
  o = up256(o + static_cast<size_t>(L.n_m) * L.Fp * 4);
  L.units = o;
  o = up256(o + static_cast<size_t>(L.n_m) * L.nj * 4);
  L.wpre = o;
  o = up256(o + static_cast<size_t>(L.n_m) * L.nw * 4);
  L.abuf = o;
  o = up256(o + static_cast<size_t>(T) * L.Fp * 2);
  L.wd16 = o;
  o = up256(o + static_cast<size_t>(F) * D * 2);
  L.n_sort = (T + UG_SORT_THREADS - 1) / UG_SORT_THREADS;
  if (!sorted) {
    L.perm = L.keys = L.hist = L.xp = 0;
    L.bytes = o;
    return L;
  }
  L.perm = o;
  o = up256(o + static_cast<size_t>(T) * 4);
  L.keys = o;
  o = up256(o + static_cast<size_t>(T));
  L.hist = o;
  o = up256(o + static_cast<size_t>(L.n_sort) * UG_NBUCKET * 4);
  L.xp = o;
  o = up256(o + static_cast<size_t>(T) * D * 2);
  L.bytes = o;
  return L;
}

// ------------------------------------------------------------ preparation
//   ug_key_kernel, ug_place_kernel  sort the tokens into positions (see the
//                   header).
//   ug_bits_kernel  (grid: blocks x 8 CTAs of 16 positions) ORs every active
//                   neuron of its positions' tokens into the block's union
//                   bitmap (shared memory, then global atomics into the
//                   zeroed [n_m][nw] bitmap); in sorted order it also copies
//                   its positions' x rows into position order.
//   ug_scan_kernel  (one CTA per block) takes the exclusive prefix of the
//                   bitmap words' popcounts -- a neuron's union position is
//                   the prefix of its word plus the set bits below it in the
//                   word -- and writes it, U (ascending, padded with neuron
//                   0), |U| and the block's up-GEMM units.
// A (row, tile) whose spill slice is missing is skipped
// (TWELL_FLAG_SPILL_FULL), as in the fused CUDA-core kernel.
template <typename Fn>
__device__ __forceinline__ void ug_walk_pair(const UgArgs& p, size_t rt, int k, bool flag_missing,
                                             Fn&& fn) {
  const int c = p.cnt[rt];
  if (c == 0 || !in_bounds(c, TWELL_TILE + 1, p.status)) return;
  if (c <= p.W) {
    const uint8_t* cp = p.col + rt * p.W;
    const float* vp = p.val + rt * p.W;
    for (int s = 0; s < c; ++s) {
      const int n = k * TWELL_TILE + tile_col(cp[s]);
      if (in_bounds(n, p.F, p.status)) fn(n, vp[s]);
    }
  } else {
    const int sl = p.spill_slot[rt];
    if (sl < 0 || sl >= p.spill_cap) {
      if (flag_missing) atomicOr(p.status, TWELL_FLAG_SPILL_FULL);
      return;
    }
    const float* sv = p.spill_val + static_cast<size_t>(sl) * TWELL_TILE;
    for (int cc = 0; cc < TWELL_TILE; ++cc) {
      const float v = sv[cc];
      if (v > 0.0f) fn(k * TWELL_TILE + cc, v);
    }
  }
}

// Activity bucket of a token with n active neurons: eight buckets per octave
// of n + 1 (n + 1 < 8 exactly), monotone in n.
__device__ __forceinline__ int ug_bucket(int n) {
  const int v = n + 1;
  const int e = 31 - __clz(v);
  const int b = e < 3 ? v : 8 * (e - 2) + ((v >> (e - 3)) & 7);
  return min(b, UG_NBUCKET - 1);
}

// One thread per token: its bucket (from the TwELL counts of its row) into
// keys[t], and the CTA's bucket counts into hist[cta][*].
__global__ void __launch_bounds__(UG_SORT_THREADS) ug_key_kernel(const UgArgs p) {
  __shared__ int h[UG_NBUCKET];
  for (int i = threadIdx.x; i < UG_NBUCKET; i += UG_SORT_THREADS) h[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * UG_SORT_THREADS + threadIdx.x;
  if (t < p.T) {
    const uint8_t* row = p.cnt + static_cast<size_t>(t) * p.n_t;
    int n = 0;
    if ((p.n_t & 15) == 0 && (reinterpret_cast<uintptr_t>(p.cnt) & 15) == 0) {
      for (int k = 0; k < p.n_t; k += 16) {
        const uint4 w4 = __ldg(reinterpret_cast<const uint4*>(row + k));
        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t s2 = (ws[e] & 0x00ff00ffu) + ((ws[e] >> 8) & 0x00ff00ffu);
          n += static_cast<int>((s2 & 0xffffu) + (s2 >> 16));
        }
      }
    } else if ((p.n_t & 3) == 0) {
      for (int k = 0; k < p.n_t; k += 4) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(row + k));
        const uint32_t s2 = (w & 0x00ff00ffu) + ((w >> 8) & 0x00ff00ffu);
        n += static_cast<int>((s2 & 0xffffu) + (s2 >> 16));
      }
    } else {
      for (int k = 0; k < p.n_t; ++k) n += row[k];
    }
    const int b = ug_bucket(n);
    p.keys[t] = static_cast<uint8_t>(b);
    atomicAdd(&h[b], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < UG_NBUCKET; i += UG_SORT_THREADS)
    p.hist[static_cast<size_t>(blockIdx.x) * UG_NBUCKET + i] = h[i];
}

// One thread per token: its position = the start of its bucket in its sort
// CTA (the tokens of lower buckets, then those of its bucket in earlier sort
// CTAs, both from the per-CTA histograms) + the tokens of the same bucket
// before it in the CTA (warp match and per-warp counts), so the order is
// stable.
__global__ void __launch_bounds__(UG_SORT_THREADS) ug_place_kernel(const UgArgs p) {
  constexpr int kWarps = UG_SORT_THREADS / 32;
  __shared__ int wc[kWarps][UG_NBUCKET];
  __shared__ int start[UG_NBUCKET];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kWarps * UG_NBUCKET; i += UG_SORT_THREADS)
    wc[i / UG_NBUCKET][i % UG_NBUCKET] = 0;
  if (warp < UG_NBUCKET / 32) {
    // bucket b = 32 warp + lane: its total over all sort CTAs and its count
    // in the CTAs before this one, then the exclusive prefix of the totals
    const int b = warp * 32 + lane;
    int total = 0, before = 0;
    for (int c = 0; c < p.n_sort; ++c) {
      const int v = p.hist[static_cast<size_t>(c) * UG_NBUCKET + b];
      total += v;
      if (c < static_cast<int>(blockIdx.x)) before += v;
    }
    int incl = total;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    wc[0][b] = incl;  // the warps' inclusive sums, combined below
    start[b] = before - total;
  }
  __syncthreads();
  if (warp < UG_NBUCKET / 32) {
    const int b = warp * 32 + lane;
    int lower = 0;  // totals of the earlier warps' buckets
    for (int w = 0; w < warp; ++w) lower += wc[0][w * 32 + 31];
    start[b] += wc[0][b] + lower;  // = exclusive prefix of totals + before
  }
  __syncthreads();
  for (int i = threadIdx.x; i < UG_NBUCKET; i += UG_SORT_THREADS) wc[0][i] = 0;
  __syncthreads();
  const int t = blockIdx.x * UG_SORT_THREADS + threadIdx.x;
  const bool valid = t < p.T;
  const int b = valid ? p.keys[t] : UG_NBUCKET;  // an out-of-range key for the tail
  const uint32_t same = __match_any_sync(0xffffffffu, b);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (valid && rank == 0) wc[warp][b] = __popc(same);
  __syncthreads();
  // exclusive prefix over the warps, per bucket
  for (int i = threadIdx.x; i < UG_NBUCKET; i += UG_SORT_THREADS) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = wc[w][i];
      wc[w][i] = run;
      run += v;
    }
  }
  __syncthreads();
  if (valid) {
    const int pos = start[b] + wc[warp][b] + rank;
    if (in_bounds(pos, p.T, p.status)) p.perm[pos] = t;
  }
}

__global__ void __launch_bounds__(UG_PREP_THREADS) ug_bits_kernel(const UgArgs p) {
  extern __shared__ uint32_t psm[];
  const int nw = p.nw;
  uint32_t* bm = psm;
  const int m = blockIdx.x;
  const int r0 = m * UG_BM + blockIdx.y * UG_ROWS_PER_CTA;
  const int rows = min(UG_ROWS_PER_CTA, p.T - r0);
  if (rows <= 0) return;
  for (int i = threadIdx.x; i < nw; i += UG_PREP_THREADS) bm[i] = 0u;
  if (p.xp) {
    // sorted order: the CTA's positions' x rows, xp[i] = x[perm[i]], for the
    // up GEMM's TMA tiles (16-byte steps, four loads in flight per thread
    // before their stores; bandwidth-bound, it overlaps the latency-bound
    // walk below across the CTAs of an SM)
    constexpr int kInFlight = 4;
    const int per_row = p.D / 8;
    const int n = rows * per_row;
    uint4* xp4 = reinterpret_cast<uint4*>(p.xp + static_cast<size_t>(r0) * p.D);
    for (int i0 = threadIdx.x; i0 < n; i0 += kInFlight * UG_PREP_THREADS) {
      uint4 v[kInFlight];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int i = i0 + u * UG_PREP_THREADS;
        if (i < n) {
          const int r = i / per_row;
          const int t = static_cast<int>(clamp_index(p.perm[r0 + r], p.T, p.status));
          v[u] = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * p.D) +
                       (i - r * per_row));
        }
      }
      // rows r0.. of xp are contiguous: position i of the CTA's rows is xp4[i]
#pragma unroll
      for (int u = 0; u < kInFlight; ++u)
        if (i0 + u * UG_PREP_THREADS < n) xp4[i0 + u * UG_PREP_THREADS] = v[u];
    }
  }
  __syncthreads();
  const int n_t = p.n_t;
  for (int q = threadIdx.x; q < rows * n_t; q += UG_PREP_THREADS) {
    const int tok = p.perm ? p.perm[r0 + q / n_t] : r0 + q / n_t;
    if (!in_bounds(tok, p.T, p.status)) continue;
    ug_walk_pair(p, static_cast<size_t>(tok) * n_t + q % n_t, q % n_t, true,
                 [&](int n, float) { atomicOr(&bm[n >> 5], 1u << (n & 31)); });
  }
  __syncthreads();
  uint32_t* g = p.gbm + static_cast<size_t>(m) * p.gbm_pitch;
  for (int i = threadIdx.x; i < nw; i += UG_PREP_THREADS)
    if (bm[i]) atomicOr(&g[i], bm[i]);
}

__global__ void __launch_bounds__(UG_PREP_THREADS) ug_scan_kernel(const UgArgs p) {
  extern __shared__ uint32_t psm[];
  const int nw = p.nw;
  uint32_t* bm = psm;                            // [nw]
  int* wpre = reinterpret_cast<int*>(psm + nw);  // [nw]
  __shared__ int wsum[UG_PREP_THREADS / 32];
  __shared__ int s_total, s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.x;
  const uint32_t* g = p.gbm + static_cast<size_t>(m) * p.gbm_pitch;
  for (int i = tid; i < nw; i += UG_PREP_THREADS) bm[i] = i < p.F / 32 ? g[i] : 0u;
  __syncthreads();

  // exclusive prefix of the words' popcounts, four words per thread
  int c[4], v = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int w = 4 * tid + e;
    c[e] = w < nw ? __popc(bm[w]) : 0;
    v += c[e];
  }
  const int mine = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int s = lane < UG_PREP_THREADS / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += o;
    }
    if (lane < UG_PREP_THREADS / 32) wsum[lane] = s;
    if (lane == UG_PREP_THREADS / 32 - 1) s_total = s;
  }
  __syncthreads();
  int ex = v - mine + (warp > 0 ? wsum[warp - 1] : 0);
  int32_t* wg = p.wpre + static_cast<size_t>(m) * nw;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int w = 4 * tid + e;
    if (w < nw) {
      wpre[w] = ex;
      wg[w] = ex;
    }
    ex += c[e];
  }
  // a union this large runs as a dense block: every neuron, in order, so
  // its weight rows are contiguous and come by TMA instead of row gathers
  const bool dense = p.dense_min > 0 && s_total >= p.dense_min;
  const int nU = dense ? p.F : s_total;
  const int chunks = (nU + 255) >> 8;
  if (tid == 0) {
    p.nU[m] = nU;
    p.dense[m] = dense ? 1 : 0;
    s_base = chunks > 0 ? atomicAdd(p.ctr, chunks) : 0;
  }
  __syncthreads();
  int32_t* Ul = p.Ulist + static_cast<size_t>(m) * p.Fp;
  if (dense) {
    for (int i = tid; i < chunks * 256; i += UG_PREP_THREADS) Ul[i] = i < p.F ? i : 0;
  } else {
    for (int w = tid; w < nw; w += UG_PREP_THREADS) {
      uint32_t bits = bm[w];
      int r = wpre[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        Ul[r++] = 32 * w + b;
      }
    }
    for (int i = nU + tid; i < chunks * 256; i += UG_PREP_THREADS) Ul[i] = 0;
  }
  for (int jn = tid; jn < chunks; jn += UG_PREP_THREADS) p.units[s_base + jn] = m * p.nj + jn;
}

// bf16 -> fp16 copy of W_d for the down GEMM (8 values per thread and step;
// exact for |w| in fp16's normal range, |w| >= 2^-14; a |w| above 65504
// becomes inf and sets TWELL_FLAG_RANGE).
__global__ void __launch_bounds__(256) ug_f16_kernel(const uint16_t* __restrict__ src,
                                                     uint16_t* __restrict__ dst, size_t n8,
                                                     int32_t* status) {
  bool over = false;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16);
      const float hi = __uint_as_float(w[k] & 0xffff0000u);
      over |= fabsf(lo) > 65504.0f || fabsf(hi) > 65504.0f;
      o[k] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
             (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
    }
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (over) atomicOr(status, TWELL_FLAG_RANGE);
}

// --------------------------------------------------------------- the GEMMs
struct UgUnit {
  int m, j, kb;  // token block, output chunk (up: union chunk; down: D tile), K blocks
  int n0;        // first output column (down) or union position (up) of the tile
};

template <int MODE>
__device__ __forceinline__ UgUnit ug_unit(const UgArgs& p, int u) {
  UgUnit r;
  if (MODE == UG_UP) {
    const int code = p.units[u];
    r.m = code / p.nj;
    r.j = code - r.m * p.nj;
    r.kb = p.D / UG_BK;
  } else {
    r.m = u / p.nN;
    r.j = u - r.m * p.nN;
    r.kb = (p.nU[r.m] + UG_BK - 1) / UG_BK;
  }
  r.n0 = UG_BN * r.j;
  return r;
}

// v[i] for a run-time i in [0, 32) without indexing a register array: a
// five-level select tree.
__device__ __forceinline__ uint32_t select32(const uint32_t (&v)[32], int i) {
  uint32_t a[16], b[8], c[4], d[2];
#pragma unroll
  for (int k = 0; k < 16; ++k) a[k] = (i & 1) ? v[2 * k + 1] : v[2 * k];
#pragma unroll
  for (int k = 0; k < 8; ++k) b[k] = (i & 2) ? a[2 * k + 1] : a[2 * k];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = (i & 4) ? b[2 * k + 1] : b[2 * k];
#pragma unroll
  for (int k = 0; k < 2; ++k) d[k] = (i & 8) ? c[2 * k + 1] : c[2 * k];
  return (i & 16) ? d[1] : d[0];
}

// Entries (neuron, gate value) of the TwELL tiles [k0, k1] of the row whose
// (row, tile) pairs start at rtb, in ascending neuron order, for width WV
// (8 or 16): B tiles' counts, then all their slots (16-byte loads; slots past
// the count are loaded, not used), are loaded before any entry is used.
template <int WV, int B, typename Fn>
__device__ __forceinline__ void walk_tiles(const UgArgs& p, size_t rtb, int k0, int k1, Fn&& fn) {
  for (int k = k0; k <= k1; k += B) {
    int cn[B];
#pragma unroll
    for (int b = 0; b < B; ++b) cn[b] = k + b <= k1 ? p.cnt[rtb + k + b] : 0;
    uint32_t cw[B][WV / 4];
    float vs[B][WV];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const size_t rt = rtb + k + b;
      const bool in = cn[b] > 0 && cn[b] <= WV;
      if (WV == 16) {
        const uint4 c4 = in ? __ldg(reinterpret_cast<const uint4*>(p.col + rt * 16))
                            : make_uint4(0u, 0u, 0u, 0u);
        cw[b][0] = c4.x;
        cw[b][1] = c4.y;
        cw[b][WV / 4 - 2] = c4.z;
        cw[b][WV / 4 - 1] = c4.w;
      } else {
        const uint2 c2 =
            in ? __ldg(reinterpret_cast<const uint2*>(p.col + rt * 8)) : make_uint2(0u, 0u);
        cw[b][0] = c2.x;
        cw[b][WV / 4 - 1] = c2.y;
      }
#pragma unroll
      for (int g4 = 0; g4 < WV / 4; ++g4) {
        const float4 v4 = in ? __ldg(reinterpret_cast<const float4*>(p.val + rt * WV) + g4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        vs[b][4 * g4] = v4.x;
        vs[b][4 * g4 + 1] = v4.y;
        vs[b][4 * g4 + 2] = v4.z;
        vs[b][4 * g4 + 3] = v4.w;
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (cn[b] == 0) continue;
      if (cn[b] > WV) {  // spilled: the slice's positive values
        ug_walk_pair(p, rtb + k + b, k + b, false, fn);
        continue;
      }
#pragma unroll
      for (int e = 0; e < WV; ++e)
        if (e < cn[b]) {
          const int n =
              (k + b) * TWELL_TILE + tile_col((cw[b][e >> 2] >> (8 * (e & 3))) & 0xffu);
          if (in_bounds(n, p.F, p.status)) fn(n, vs[b][e]);
        }
    }
  }
}

// Gate value of row t at neuron n read from the TwELL (0 if inactive or in a
// missing spill slice): the slow path for rows with many entries in a chunk.
__device__ __forceinline__ float twell_h_at(const UgArgs& p, int t, int n) {
  const size_t rt = static_cast<size_t>(t) * p.n_t + (n >> 7);
  const int col = n & (TWELL_TILE - 1);
  const int c = p.cnt[rt];
  if (c <= p.W) {
    for (int s = 0; s < c; ++s)
      if (p.col[rt * p.W + s] == col) return p.val[rt * p.W + s];
    return 0.0f;
  }
  const int sl = p.spill_slot[rt];
  if (sl < 0 || sl >= p.spill_cap) return 0.0f;
  return p.spill_val[static_cast<size_t>(sl) * TWELL_TILE + col];
}

template <int MODE>
__global__ void __launch_bounds__(UG_THREADS, 1)
    ug_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_out,
                   const __grid_constant__ CUtensorMap map_b, const UgArgs p) {
  using SM = UgSmem<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::BARS);
  uint64_t* empty = full + UG_ST;
  uint64_t* tfull = empty + UG_ST;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  uint64_t* drain = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // abort path: MMA drain
  volatile uint32_t* aborted = tmem_slot + 1;
  // unit ring: the producer publishes each unit's record, every other role
  // reads it (barrier area bytes 128 .. 383)
  uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + SM::BARS + 128);
  uint64_t* rempty = rfull + UG_RING;
  UgUnit* ring = reinterpret_cast<UgUnit*>(smem + SM::BARS + 256);
  float* hslots = reinterpret_cast<float*>(smem + SM::SLOTS);  // up: [2][128][UG_HSLOTS]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < UG_ST; ++s) {
      ptx::mbar_init(&full[s], 1 + UG_GROUP);  // the A producer's expect_tx + a gather group
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], UG_EPI);
    }
    for (int r = 0; r < UG_RING; ++r) {
      ptx::mbar_init(&rfull[r], 1);
      ptx::mbar_init(&rempty[r], UG_RING_READERS);
    }
    ptx::mbar_init(drain, 1);
    *aborted = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 2 * UG_BN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------- TMA producer (A)
    // It also hands out the work: units go to CTAs in the order they ask,
    // from a ticket counter of the launch (the costs of units differ: dense
    // or gathered weight tiles, union sizes, rows with many entries in the
    // up epilogue), and each unit's record goes to the other roles through
    // the unit ring.  The down GEMM takes its units last to first: blocks of
    // activity-sorted tokens come in ascending activity, so the largest
    // unions go first.  A unit index past the count ends every role's loop.
    if (lane == 0) {
      const int num_units = MODE == UG_UP ? *p.ctr : p.n_m * p.nN;
      int* ticket = p.ctr + 1 + MODE;
      int stage = 0;
      uint32_t phase = 0;
      int rs = 0;
      uint32_t rph = 0;
      auto unit_of = [&](int tk) {
        return tk < num_units ? ug_unit<MODE>(p, MODE == UG_DOWN ? num_units - 1 - tk : tk)
                              : UgUnit{-1, 0, 0, 0};
      };
      // a unit's record into the next ring slot (false: the wait ran out)
      auto publish = [&](const UgUnit& V) {
        if (!ptx::mbar_wait(&rempty[rs], rph ^ 1u)) return false;
        ring[rs] = V;
        ptx::mbar_arrive(&rfull[rs]);
        if (++rs == UG_RING) {
          rs = 0;
          rph ^= 1u;
        }
        return true;
      };
      UgUnit Un = unit_of(atomicAdd(ticket, 1));
      bool published = false;  // Un is in the ring already
      for (;;) {
        const UgUnit U = Un;
        if (!published && !publish(U)) {
          { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        published = false;
        if (U.m < 0) break;
        // The next unit is claimed ten tiles before this unit's last is
        // issued (late, so that a CTA holds a unit in reserve only briefly:
        // a reserved unit can leave other CTAs idle at the end), and its
        // record is read and published three tiles later.  The producer runs
        // stages ahead of the MMA, so neither latency reaches it, and the
        // gather groups know the next unit before their last stage of this
        // one and load its neuron ids while that stage lands.
        const int kb_claim = U.kb > 10 ? U.kb - 10 : 0;
        const int kb_read = U.kb > 7 ? U.kb - 7 : (U.kb > 1 ? 1 : 0);
        int tk = 0;
        if (U.kb == 0) Un = unit_of(atomicAdd(ticket, 1));
        for (int kb = 0; kb < U.kb; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u)) {
            { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], UG_A);
          ptx::tma_load_2d(smem + stage * UG_STAGE, &map_a, &full[stage], kb * UG_BK,
                           U.m * UG_BM);
          if (++stage == UG_ST) {
            stage = 0;
            phase ^= 1u;
          }
          if (kb == kb_claim) tk = atomicAdd(ticket, 1);
          if (kb == kb_read) {
            Un = unit_of(tk);
            if (!publish(Un)) {
              { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
              goto done;
            }
            published = true;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      // up: bf16 x and W_u; down: fp16 a and W_d
      constexpr uint32_t idesc = MODE == UG_UP ? ptx::idesc_bf16_f32(UG_BM, UG_BN, false, false)
                                               : ptx::idesc_f16_f32(UG_BM, UG_BN, false, true);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      int rs = 0;
      uint32_t rph = 0;
      for (;;) {
        if (!ptx::mbar_wait(&rfull[rs], rph)) {
          { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        const UgUnit U = ring[rs];
        ptx::mbar_arrive(&rempty[rs]);
        if (++rs == UG_RING) {
          rs = 0;
          rph ^= 1u;
        }
        if (U.m < 0) break;
        if (U.kb == 0) continue;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        ++local;
        if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u)) {
          { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * UG_BN);
        for (int kb = 0; kb < U.kb; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase)) {
            { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + stage * UG_STAGE);
          const uint32_t b_addr = a_addr + UG_A;
#pragma unroll
          for (int kk = 0; kk < UG_BK / 16; ++kk) {
            const uint64_t bd = MODE == UG_UP
                                    ? ptx::sdesc_kmajor_sw128(b_addr + kk * 32)
                                    : ptx::sdesc_mnmajor_sw128(b_addr + kk * 2048, 8192, 1024);
            ptx::mma_bf16(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + kk * 32), bd, idesc,
                          (kb | kk) ? 1u : 0u);
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == UG_ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        ptx::mma_commit(&tfull[acc]);
      }
    }
  } else if (warp >= UG_GATHER0 / 32) {
    // --------------------------------------------------------- B gather
    // Group grp (64 threads) fills stage grp, i.e. the K blocks whose stage
    // sequence number is grp mod 4: wait for the stage to be free, issue 32
    // copies per thread, wait for them, fence them to the async proxy and
    // arrive on the stage's full barrier.  The four groups keep all four
    // stages in flight.
    // up:   B = W_u^T rows of 256 union neurons x 64 K, K-major: neuron row
    //       n at n * 128 bytes, its 16-byte chunk c at chunk c ^ (n & 7).
    //       Thread g copies chunk g & 7 of rows (g >> 3) + 8 i.
    // down: B = W_d rows of 64 union neurons (K) x 256 outputs, N-major in
    //       four 64-column boxes of 8 KB: K row k of box b at b * 8192 +
    //       k * 128, chunk c at chunk c ^ (k & 7).  Thread g copies chunk
    //       g & 7 of box (g >> 3) & 3 of K rows (g >> 5) + 2 i; chunks past
    //       D are zero-filled.
    const int grp = (threadIdx.x - UG_GATHER0) / UG_GROUP;
    const int g = (threadIdx.x - UG_GATHER0) % UG_GROUP;
    const int cj = g & 7;
    uint8_t* sBp = smem + grp * UG_STAGE + UG_A;
    const uint32_t sB = ptx::smem_u32(sBp);
    uint64_t* fb = &full[grp];
    uint64_t* eb = &empty[grp];
    int seq = 0;
    int ids[32];
    int ids_for = -1;  // up: the unit (ring sequence number) whose neuron ids are in ids[]
    int rs = 0;
    uint32_t rph = 0;
    int nu = 0;              // units taken from the ring
    bool have_next = false;  // up: the next unit, taken early, is in Un
    UgUnit Un{};
    // the next unit from the ring (warp-uniform; false: the wait ran out)
    auto take = [&](UgUnit& out) {
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&rfull[rs], rph))) return false;
      out = ring[rs];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&rempty[rs]);
      if (++rs == UG_RING) {
        rs = 0;
        rph ^= 1u;
      }
      ++nu;
      return true;
    };
    // up: the next unit into Un and its neuron ids into ids[]
    auto take_next = [&]() {
      if (!take(Un)) return false;
      have_next = true;
      if (Un.m >= 0) {
        const int32_t* Uln = p.Ulist + static_cast<size_t>(Un.m) * p.Fp;
#pragma unroll
        for (int i = 0; i < 32; ++i) ids[i] = __ldg(Uln + Un.j * 256 + (g >> 3) + 8 * i);
        ids_for = nu;
      }
      return true;
    };
    for (;;) {
      UgUnit U;
      if (have_next) {
        U = Un;
        have_next = false;
      } else if (!take(U)) {
        if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
        goto done;
      }
      if (U.m < 0) break;
      const int cur = nu;
      if (U.kb == 0) continue;
      const int32_t* Ul = p.Ulist + static_cast<size_t>(U.m) * p.Fp;
      // first K block of this unit that is this group's
      int kb = (grp - seq) & (UG_ST - 1);
      const int seq0 = seq;
      seq += U.kb;
      if (kb >= U.kb) continue;
      if (p.dense[U.m]) {
        // a dense block's tile: its B rows are contiguous (union position =
        // neuron), one TMA box per stage (up: 256 neurons x 64 K of W_u^T;
        // down: four 64 x 64 boxes of W_d16) issued by the group's first
        // thread; the group still makes its 64 arrivals
        for (; kb < U.kb; kb += UG_ST) {
          const uint32_t phase = static_cast<uint32_t>((seq0 + kb) / UG_ST) & 1u;
          if (!ptx::mbar_wait(eb, phase ^ 1u)) {
            { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
            goto done;
          }
          if (g == 0) {
            ptx::mbar_arrive_expect_tx(fb, UG_B);
            if (MODE == UG_UP) {
              ptx::tma_load_2d(sBp, &map_b, fb, kb * UG_BK, U.n0);
            } else {
#pragma unroll
              for (int b4 = 0; b4 < 4; ++b4)
                ptx::tma_load_2d(sBp + b4 * 8192, &map_b, fb, U.n0 + 64 * b4, kb * UG_BK);
            }
          } else {
            ptx::mbar_arrive(fb);
          }
        }
        continue;
      }
      int col = 0;
      uint32_t nbytes = 16;
      if (MODE == UG_UP) {
        if (ids_for != cur) {
#pragma unroll
          for (int i = 0; i < 32; ++i) ids[i] = __ldg(Ul + U.j * 256 + (g >> 3) + 8 * i);
        }
      } else {
        col = U.n0 + 64 * ((g >> 3) & 3) + 8 * cj;
        nbytes = col < p.D ? 16u : 0u;
        if (col >= p.D) col = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) ids[i] = __ldg(Ul + kb * UG_BK + (g >> 5) + 2 * i);
      }
      for (; kb < U.kb; kb += UG_ST) {
        const uint32_t phase = static_cast<uint32_t>((seq0 + kb) / UG_ST) & 1u;
        if (!ptx::mbar_wait(eb, phase ^ 1u)) {
          { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        if (MODE == UG_UP) {
          const uint32_t dst0 = sB + (g >> 3) * 128 + ((cj ^ (g >> 3)) << 4);
          const size_t koff = static_cast<size_t>(kb) * UG_BK + 8 * cj;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            ptx::cp_async16(dst0 + i * 1024,
                            p.Wu_t + static_cast<size_t>(clamp_index(ids[i], p.F, p.status)) * p.D +
                                koff);
        } else {
          const uint32_t box = sB + ((g >> 3) & 3) * 8192;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int k = (g >> 5) + 2 * i;
            ptx::cp_async16(
                box + k * 128 + ((cj ^ (k & 7)) << 4),
                p.Wd16 + static_cast<size_t>(clamp_index(ids[i], p.F, p.status)) * p.D + col,
                nbytes);
          }
          if (kb + UG_ST < U.kb) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              ids[i] = __ldg(Ul + (kb + UG_ST) * UG_BK + (g >> 5) + 2 * i);
          }
        }
        ptx::cp_async_commit();
        // This group's last stage of an up unit: the next unit's neuron ids
        // are loaded while the stage lands (the copies read their addresses
        // at issue) when the producer has already published that unit, else
        // once the stage is marked full, before the group's next stage is free.
        const bool last = MODE == UG_UP && kb + UG_ST >= U.kb;
        const bool early = last && __all_sync(0xffffffffu, ptx::mbar_try_wait(&rfull[rs], rph));
        if (early && !take_next()) {
          if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(fb);
        if (last && !early && !take_next()) {
          if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
          goto done;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int set = (warp - 2) >> 2;  // column half of the tile
    uint8_t* buf = smem + SM::STG + (warp - 2) * SM::STG_BUF;
    int local = 0;
    int rs = 0;
    uint32_t rph = 0;
    for (;;) {
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&rfull[rs], rph))) {
        if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
        goto done;
      }
      const UgUnit U = ring[rs];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&rempty[rs]);
      if (++rs == UG_RING) {
        rs = 0;
        rph ^= 1u;
      }
      if (U.m < 0) break;
      const int pos = U.m * UG_BM + r;  // position of this row
      const bool valid = pos < p.T;
      const int t = !valid ? 0
                    : p.perm ? static_cast<int>(clamp_index(p.perm[pos], p.T, p.status))
                             : pos;
      if (MODE == UG_DOWN && U.kb == 0) {  // no active neuron in the block: y rows are zero
        if (valid) {
          float* o = p.y + static_cast<size_t>(t) * p.D + U.n0 + 128 * set;
          for (int n = 0; n < 128 && U.n0 + 128 * set + n < p.D; n += 4)
            *reinterpret_cast<float4*>(o + n) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      ++local;
      // Up: the row's active positions in this set's half of the chunk
      // (positions ps .. ps + 127 of U, ps = 256 j + 128 set, i.e. neurons
      // U[ps] .. U[last]) as four mask words, and the gate values of the
      // first UG_HSLOTS of them (ascending) in the row's shared-memory slots.
      // They come from the row's TwELL tiles that cover those neurons, four
      // tiles' counts and slots loaded at a time, while the chunk's MMAs run.
      uint32_t mq[4] = {0u, 0u, 0u, 0u};
      float* myslot = hslots + (set * UG_BM + r) * UG_HSLOTS;
      const int32_t* Ul = p.Ulist + static_cast<size_t>(U.m) * p.Fp;
      const int ps = 256 * U.j + 128 * set;
      if (MODE == UG_UP && valid) {
        const int nUm = __ldg(p.nU + U.m);
        if (ps < nUm) {
          const int lo_n = __ldg(Ul + ps);
          const int hi_n = __ldg(Ul + min(ps + 127, nUm - 1));
          const uint32_t* bmr = p.gbm + static_cast<size_t>(U.m) * p.gbm_pitch;
          const int32_t* wpr = p.wpre + static_cast<size_t>(U.m) * p.nw;
          const bool dense_blk = p.dense[U.m] != 0;
          int nset = 0;
          auto add = [&](int n, float h) {
            if (n < lo_n || n > hi_n) return;
            const int w = n >> 5;
            const int pos = dense_blk ? n - ps
                                    : __ldg(wpr + w) +
                                          __popc(__ldg(bmr + w) & ((1u << (n & 31)) - 1u)) - ps;
            const uint32_t bit = 1u << (pos & 31);
            const uint32_t wsel = pos >> 5;  // a select per word, not an index
#pragma unroll
            for (int k = 0; k < 4; ++k) mq[k] |= (wsel == static_cast<uint32_t>(k) ? bit : 0u);
            if (nset < UG_HSLOTS) myslot[nset] = h;
            ++nset;
          };
          const size_t rtb = static_cast<size_t>(t) * p.n_t;
          const int k0 = lo_n >> 7, k1 = hi_n >> 7;
          if (p.W == 8) {
            walk_tiles<8, 4>(p, rtb, k0, k1, add);
          } else if (p.W == 16) {
            walk_tiles<16, 2>(p, rtb, k0, k1, add);
          } else {
            for (int k = k0; k <= k1; ++k) ug_walk_pair(p, rtb + k, k, false, add);
          }
        }
      }
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&tfull[acc], acc_phase))) {
        if (lane == 0) { atomicOr(p.status, TWELL_FLAG_TIMEOUT); *aborted = 1u; }
        goto done;
      }
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * UG_BN + 128 * set) +
                             (static_cast<uint32_t>(q * 32) << 16);
      // Output chunks of 32 columns go through the warp's staging buffer:
      // each lane writes its row with the swizzle of the output tensor map
      // (16-byte chunk j of row r at chunk j ^ (address bits 7..)),
      // conflict-free, and lane 0 stores the warp's 32 x 32 box with one TMA
      // store (rows past T are clipped); the buffer is reused once that
      // store has read it.
      const int row0 = U.m * UG_BM + q * 32;
      // chunks of this set (down: the tile may end before the second half)
      const int nch = MODE == UG_UP ? 4 : max(0, min(128, p.D - U.n0 - 128 * set) / 32);
      if (nch == 0) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[acc]);
      }
      int rank = 0;  // up: active positions of the row consumed so far
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), v);
        ptx::tmem_wait_ld();
        if (c == nch - 1) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&tempty[acc]);
        }
        if (lane == 0) ptx::bulk_wait_read<0>();
        __syncwarp();
        if (MODE == UG_UP) {
          uint32_t mc = mq[0];
#pragma unroll
          for (int i = 0; i < 3; ++i) mq[i] = mq[i + 1];
          // 64-byte rows, 64-byte swizzle: chunk j of row lane at j ^ ((lane >> 1) & 3).
          // The row is zeroed, then each active position gets its bf16 a;
          // the loop runs as often as the busiest lane of the warp needs.
          uint8_t* my_row = buf + lane * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(my_row + 16 * j) = make_uint4(0u, 0u, 0u, 0u);
          const int sw = (lane >> 1) & 3;
          while (__any_sync(0xffffffffu, mc != 0u)) {
            if (mc != 0u) {
              const int i = __ffs(mc) - 1;
              mc &= mc - 1u;
              const float hv = rank < UG_HSLOTS
                                   ? myslot[rank]
                                   : twell_h_at(p, t, __ldg(Ul + ps + 32 * c + i));
              ++rank;
              const float a = hv * __uint_as_float(select32(v, i));
              if (fabsf(a) > 65504.0f) atomicOr(p.status, TWELL_FLAG_RANGE);
              *reinterpret_cast<uint16_t*>(my_row + ((((i >> 3) ^ sw)) << 4) + (i & 7) * 2) =
                  __half_as_ushort(__float2half_rn(a));
            }
          }
        } else {
          // 128-byte rows, 128-byte swizzle: chunk j of row lane at j ^ (lane & 7)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          if (p.perm) {
            // rows in sorted order go to their tokens: the staged box is read
            // back four rows per pass, eight lanes per row (one 16-byte chunk
            // each), so every store writes four whole 128-byte row segments
            __syncwarp();
            const int sub = lane >> 3;   // row within the pass
            const int ch = lane & 7;     // chunk of the row
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = 4 * i + sub;  // row of the warp's box
              const int tr = __shfl_sync(0xffffffffu, t, rr);
              const bool vr = __shfl_sync(0xffffffffu, valid ? 1 : 0, rr) != 0;
              const uint4 w = *reinterpret_cast<const uint4*>(buf + rr * 128 +
                                                              ((ch ^ (rr & 7)) << 4));
              if (vr)
                reinterpret_cast<uint4*>(p.y + static_cast<size_t>(tr) * p.D + U.n0 +
                                         128 * set + 32 * c)[ch] = w;
            }
            __syncwarp();  // the buffer is rewritten by the next chunk
            continue;
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&map_out, buf, U.n0 + 128 * set + 32 * c, row0);
          ptx::bulk_commit();
        }
      }
    }
  }

done:
  // the epilogue's TMA stores have finished before the CTA's shared memory goes away
  if (warp >= 2 && warp < UG_GATHER0 / 32 && lane == 0) ptx::bulk_wait_all();
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
    ptx::tmem_dealloc(tmem_base, 2 * UG_BN);
  }
}

template <int MODE>
twell_status ug_launch(const CUtensorMap& map, const CUtensorMap& map_out,
                       const CUtensorMap& map_b, const UgArgs& a, int max_units,
                       const DeviceInfo& dev, cudaStream_t s) {
  constexpr int SMEM = UgSmem<MODE>::BYTES;
  static_assert(SMEM <= 232448, "shared memory budget");
  auto kern = ug_gemm_kernel<MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  if (max_units <= 0) return TWELL_OK;
  const int grid = max_units < dev.sm_count ? max_units : dev.sm_count;
  kern<<<grid, UG_THREADS, SMEM, s>>>(map, map_out, map_b, a);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace

size_t ffn_tc_workspace_bytes(int64_t T, int64_t D, int64_t F, bool sorted) {
  return ug_layout(T, D, F, sorted).bytes;
}

}  // namespace twell

extern "C" twell_status twell_to_f16(const uint16_t* src, uint16_t* dst, size_t n,
                                     int32_t* status_dev, void* stream) {
  using namespace twell;
  if (n == 0) return TWELL_OK;
  if (!src || !dst || !status_dev || n % 8 != 0 || !aligned16(src) || !aligned16(dst))
    return TWELL_ERR_INVALID;
  DeviceInfo dev;
  twell_status st;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  const size_t n8 = n / 8;
  const size_t want = (n8 + 255) / 256;
  const size_t cap = 4u * static_cast<size_t>(dev.sm_count);
  ug_f16_kernel<<<static_cast<int>(want < cap ? want : cap), 256, 0,
                  static_cast<cudaStream_t>(stream)>>>(src, dst, n8, status_dev);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

namespace twell {
namespace {

twell_status ffn_tc_run(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                        const uint16_t* Wd, const uint16_t* Wd_f16, int32_t D, float* y,
                        void* ws, size_t ws_bytes, int32_t* status_dev, void* stream,
                        bool sorted) {
  if (h == nullptr) return TWELL_ERR_INVALID;
  const int32_t T = h->T, F = h->F;
  if (T < 0 || F <= 0 || F % TWELL_TILE != 0 || D <= 0 || D % UG_BK != 0)
    return TWELL_ERR_INVALID;
  if (F > UG_MAX_F) return TWELL_ERR_UNSUPPORTED;
  twell_status st = check_twell(h, T, F, false);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  if (!x || !Wu_t || !Wd || !y || !status_dev || !ws) return TWELL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(y) ||
      (Wd_f16 && !aligned16(Wd_f16)) || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return TWELL_ERR_INVALID;
  const UgLayout L = ug_layout(T, D, F, sorted);
  if (ws_bytes < L.bytes) return TWELL_ERR_INVALID;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  uint8_t* w = static_cast<uint8_t*>(ws);
  UgArgs a{};
  a.val = h->val;
  a.col = h->col;
  a.cnt = h->cnt;
  a.spill_slot = h->spill_slot;
  a.spill_val = h->spill_val;
  a.spill_cap = h->spill_cap;
  a.T = T;
  a.D = D;
  a.F = F;
  a.Fp = static_cast<int32_t>(L.Fp);
  a.nw = static_cast<int32_t>(L.nw);
  a.n_t = F / TWELL_TILE;
  a.W = h->width;
  a.n_m = static_cast<int32_t>(L.n_m);
  a.nj = static_cast<int32_t>(L.nj);
  a.nN = (D + UG_BN - 1) / UG_BN;
  a.Wu_t = Wu_t;
  a.Wd = Wd;
  a.y = y;
  a.ctr = reinterpret_cast<int32_t*>(w + L.ctr);
  // the gate kernel's block bitmaps when the TwELL has them and the blocks
  // are its blocks of consecutive tokens, else our own
  const bool own_bits = sorted || h->block_bits == nullptr;
  a.gbm = own_bits ? reinterpret_cast<uint32_t*>(w + L.gbm) : h->block_bits;
  a.gbm_pitch = own_bits ? static_cast<int32_t>(L.nw) : F / 32;
  a.nU = reinterpret_cast<int32_t*>(w + L.nU);
  a.dense = reinterpret_cast<int8_t*>(w + L.dense);
  a.dense_min = static_cast<int32_t>((static_cast<int64_t>(F) * UG_DENSE_PCT + 99) / 100);
  a.Ulist = reinterpret_cast<int32_t*>(w + L.Ulist);
  a.units = reinterpret_cast<int32_t*>(w + L.units);
  a.wpre = reinterpret_cast<int32_t*>(w + L.wpre);
  a.abuf = reinterpret_cast<uint16_t*>(w + L.abuf);
  a.perm = sorted ? reinterpret_cast<int32_t*>(w + L.perm) : nullptr;
  a.keys = sorted ? w + L.keys : nullptr;
  a.hist = sorted ? reinterpret_cast<int32_t*>(w + L.hist) : nullptr;
  a.n_sort = static_cast<int32_t>(L.n_sort);
  a.x = x;
  a.xp = sorted ? reinterpret_cast<uint16_t*>(w + L.xp) : nullptr;
  // the caller's fp16 copy of W_d, or one made in the workspace below
  a.Wd16 = Wd_f16 ? const_cast<uint16_t*>(Wd_f16) : reinterpret_cast<uint16_t*>(w + L.wd16);
  a.status = status_dev;

  // operand maps (box 64 x 128, 128-byte swizzle) and output maps (box
  // 32 x 32: a in bf16 with the 64-byte swizzle, y in fp32 with 128)
  CUtensorMap map_x, map_a, map_as, map_y, map_wu, map_wd;
  if ((st = tc_map_a(&map_x, sorted ? a.xp : x, T, D, 0)) != TWELL_OK) return st;
  if ((st = tc_map_a(&map_a, a.abuf, T, L.Fp, 0)) != TWELL_OK) return st;
  if ((st = make_tmap_2d(&map_as, 2, a.abuf, L.Fp, T, 32, 32, L.Fp * 2, 64)) != TWELL_OK)
    return st;
  if ((st = make_tmap_2d(&map_y, 4, y, D, T, 32, 32, static_cast<uint64_t>(D) * 4, 128)) !=
      TWELL_OK)
    return st;
  // dense blocks' weight tiles: W_u^T 256 neurons x 64 K (K-major), W_d16
  // 64 neurons x 64 outputs (N-major), both with the 128-byte swizzle
  if ((st = make_tmap_2d(&map_wu, 2, Wu_t, D, F, UG_BK, UG_BN, static_cast<uint64_t>(D) * 2,
                         128)) != TWELL_OK)
    return st;
  if ((st = make_tmap_2d(&map_wd, 2, a.Wd16, D, F, 64, UG_BK, static_cast<uint64_t>(D) * 2,
                         128)) != TWELL_OK)
    return st;

  // the counter and our block bitmaps are adjacent: one memset clears both
  if (cudaMemsetAsync(w + L.ctr, 0, own_bits ? L.nU - L.ctr : 256, s) != cudaSuccess)
    return TWELL_ERR_CUDA;
  if (sorted) {
    // token order, then x in that order
    ug_key_kernel<<<a.n_sort, UG_SORT_THREADS, 0, s>>>(a);
    ug_place_kernel<<<a.n_sort, UG_SORT_THREADS, 0, s>>>(a);
  }
  const dim3 pgrid(a.n_m, UG_BM / UG_ROWS_PER_CTA);
  if (own_bits) {
    ug_bits_kernel<<<pgrid, UG_PREP_THREADS, static_cast<size_t>(L.nw) * 4, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  }
  ug_scan_kernel<<<a.n_m, UG_PREP_THREADS, static_cast<size_t>(L.nw) * 8, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  if (!Wd_f16) {
    const size_t n8 = static_cast<size_t>(F) * D / 8;  // D % 64 == 0
    const size_t want = (n8 + 255) / 256;
    const size_t cap = 4u * static_cast<size_t>(dev.sm_count);
    ug_f16_kernel<<<static_cast<int>(want < cap ? want : cap), 256, 0, s>>>(Wd, a.Wd16, n8,
                                                                           status_dev);
    if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  }
  if ((st = ug_launch<UG_UP>(map_x, map_as, map_wu, a, a.n_m * a.nj, dev, s)) != TWELL_OK)
    return st;
  return ug_launch<UG_DOWN>(map_a, map_y, map_wd, a, a.n_m * a.nN, dev, s);
}

}  // namespace
}  // namespace twell

extern "C" twell_status twell_ffn_fwd_tc(const uint16_t* x, const twell_t* h,
                                         const uint16_t* Wu_t, const uint16_t* Wd,
                                         const uint16_t* Wd_f16, int32_t D, float* y, void* ws,
                                         size_t ws_bytes, int32_t* status_dev, void* stream) {
  return twell::ffn_tc_run(x, h, Wu_t, Wd, Wd_f16, D, y, ws, ws_bytes, status_dev, stream,
                           false);
}

extern "C" twell_status twell_ffn_fwd_tc_sorted(const uint16_t* x, const twell_t* h,
                                                const uint16_t* Wu_t, const uint16_t* Wd,
                                                const uint16_t* Wd_f16, int32_t D, float* y,
                                                void* ws, size_t ws_bytes, int32_t* status_dev,
                                                void* stream) {
  return twell::ffn_tc_run(x, h, Wu_t, Wd, Wd_f16, D, y, ws, ws_bytes, status_dev, stream,
                           true);
}
