// TwELL -> hybrid conversion ("Sparser, Faster, Lighter Transformer Language
// Models", section 2.B.3: during training the per-row nonzero count varies a
// lot, so rows with few nonzeros are kept in a compact ELL matrix and
// overflow rows are routed to a dense backup; a custom kernel converts
// TwELL to this hybrid format).
//
// Four launches on the caller's stream, no host round trip:
//   classify  one warp per row: overflow iff some tile count > C; the flag
//             is parked in row_map[t]
//   scan      one CTA: exclusive scans of the ELL / dense flags in token
//             order give every row its place; writes row_map, ell_rows,
//             dense_rows, n_ell, n_dense (deterministic)
//   ell_fill  one warp per ELL row (grid sized by T, rows past n_ell exit):
//             lane k copies tile k's count and entries (slots, or the spill
//             slice when W < count <= C); with W == C (16 or 32) whole
//             16-byte chunks of slots instead (ell_copy)
//   dense_fill one CTA per dense row: thread j writes ReLU(z) of column j
//             from the slots or the spill slice (coalesced row writes)
#include "bounds.cuh"
#include "common.cuh"

namespace twell {
namespace {

constexpr int kScanThreads = 1024;

struct HybParams {
  // TwELL input
  const float* val;
  const uint8_t* col;
  const uint8_t* cnt;
  const int32_t* spill_slot;
  const float* spill_val;
  int32_t spill_cap;
  int32_t W;
  // hybrid output
  int32_t T, n_t, F, C, max_dense;
  int32_t* n_ell;
  int32_t* n_dense;
  int32_t* row_map;
  int32_t* ell_rows;
  float* ell_val;
  uint8_t* ell_col;
  uint8_t* ell_cnt;
  int32_t* dense_rows;
  float* dense_h;
  int32_t* status;
};

__global__ void __launch_bounds__(256) classify_kernel(const HybParams p) {
  const int lane = threadIdx.x & 31;
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= p.T) return;
  const uint8_t* row = p.cnt + t * p.n_t;
  bool over = false;
  for (int k = lane; k < p.n_t; k += 32) over |= row[k] > p.C;
  over = __any_sync(0xffffffffu, over);
  if (lane == 0) p.row_map[t] = over ? 1 : 0;
}

__global__ void __launch_bounds__(kScanThreads) scan_kernel(const HybParams p) {
  __shared__ int32_t part[kScanThreads];
  const int tid = threadIdx.x;
  const int per = (p.T + kScanThreads - 1) / kScanThreads;
  const int t0 = tid * per;
  const int t1 = min(p.T, t0 + per);
  int n_over = 0;
  for (int t = t0; t < t1; ++t) n_over += p.row_map[t];
  part[tid] = n_over;
  __syncthreads();
  // Hillis-Steele inclusive scan of the per-thread overflow counts
  for (int d = 1; d < kScanThreads; d <<= 1) {
    const int v = tid >= d ? part[tid - d] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int dense_pos = part[tid] - n_over;                 // overflow rows before t0
  int ell_pos = (t0 < p.T ? t0 : p.T) - dense_pos;    // ELL rows before t0
  for (int t = t0; t < t1; ++t) {
    if (p.row_map[t]) {
      if (dense_pos < p.max_dense) p.dense_rows[dense_pos] = t;
      p.row_map[t] = -(dense_pos + 1);
      ++dense_pos;
    } else {
      p.ell_rows[ell_pos] = t;
      p.row_map[t] = ell_pos;
      ++ell_pos;
    }
  }
  if (tid == kScanThreads - 1) {
    const int total_dense = part[kScanThreads - 1];
    *p.n_dense = total_dense;
    *p.n_ell = p.T - total_dense;
    if (total_dense > p.max_dense && p.status) atomicOr(p.status, TWELL_FLAG_DENSE_FULL);
  }
}

__global__ void __launch_bounds__(256) ell_fill_kernel(const HybParams p) {
  const int lane = threadIdx.x & 31;
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (i >= *p.n_ell) return;
  const int t = p.ell_rows[i];
  if (!in_bounds(t, p.T, p.status)) return;  // warp-uniform
  const size_t src_rt = static_cast<size_t>(t) * p.n_t;
  const size_t dst_rt = static_cast<size_t>(i) * p.n_t;
  for (int k = lane; k < p.n_t; k += 32) {
    int c = min(static_cast<int>(p.cnt[src_rt + k]), p.C);  // <= C for an ELL row
    int slot = -1;
    if (c > p.W) {
      slot = p.spill_slot[src_rt + k];
      if (slot < 0 || slot >= p.spill_cap) {
        // the gate kernel found no room for this slice: the tile is stored
        // empty (count 0, every slot padding) so that no reader follows a
        // column the slots do not hold
        if (p.status) atomicOr(p.status, TWELL_FLAG_SPILL_FULL);
        c = 0;
      }
    }
    float* dv = p.ell_val + (dst_rt + k) * p.C;
    uint8_t* dc = p.ell_col + (dst_rt + k) * p.C;
    // padding slots: column sentinel 0xff (whole rows of 16 bytes first,
    // entries overwrite theirs below)
    if ((p.C & 15) == 0) {
      for (int s = (c & ~15); s < p.C; s += 16)
        *reinterpret_cast<uint4*>(dc + s) = make_uint4(~0u, ~0u, ~0u, ~0u);
    } else {
      for (int s = c; s < p.C; ++s) dc[s] = 0xffu;
    }
    int s = 0;
    if (c > 0 && c <= p.W) {
      const float* sv = p.val + (src_rt + k) * p.W;
      const uint8_t* sc = p.col + (src_rt + k) * p.W;
      for (; s < c; ++s) {
        dv[s] = sv[s];
        dc[s] = static_cast<uint8_t>(tile_col(sc[s]));
      }
    } else if (c > 0) {
      const float* sl = p.spill_val + static_cast<size_t>(slot) * TWELL_TILE;
      for (int cc = 0; cc < TWELL_TILE && s < c; ++cc) {
        const float v = sl[cc];
        if (v > 0.0f) {
          dv[s] = v;
          dc[s] = static_cast<uint8_t>(cc);
          ++s;
        }
      }
      // a slice with fewer positive values than its count leaves the rest
      // of its slots as padding
      for (int r = s; r < c; ++r) dc[r] = 0xffu;
    }
    // the count is the number of entries written, stored last
    p.ell_cnt[dst_rt + k] = static_cast<uint8_t>(s);
  }
}

// ell_fill for W == C (16 or 32) and 16-byte aligned slot arrays, the
// training setting, where a tile's slots are its ELL entries: whole 16-byte
// chunks instead of one slot at a time.  One warp per ELL row, a group of
// eight lanes per tile, four tiles at a time: lane j copies value chunk j
// (slots 4j .. 4j+3) when it holds entries, and lanes j < C / 16 write column
// chunk j with the slots at and past the count set to the padding sentinel.
template <int C>
__global__ void __launch_bounds__(256) ell_copy_kernel(const HybParams p) {
  const int lane = threadIdx.x & 31;
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (i >= *p.n_ell) return;
  const int t = p.ell_rows[i];
  if (!in_bounds(t, p.T, p.status)) return;  // warp-uniform
  const size_t src_rt = static_cast<size_t>(t) * p.n_t;
  const size_t dst_rt = static_cast<size_t>(i) * p.n_t;
  const int j = lane & 7;
  for (int k = lane >> 3; k < p.n_t; k += 4) {
    const int c = min(static_cast<int>(p.cnt[src_rt + k]), C);  // <= C for an ELL row
    if (j < C / 4 && 4 * j < c)
      reinterpret_cast<uint4*>(p.ell_val + (dst_rt + k) * C)[j] =
          __ldg(reinterpret_cast<const uint4*>(p.val + (src_rt + k) * C) + j);
    if (j < C / 16) {
      const uint4 w = 16 * j < c
                          ? __ldg(reinterpret_cast<const uint4*>(p.col + (src_rt + k) * C) + j)
                          : make_uint4(0u, 0u, 0u, 0u);
      uint32_t o[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t r = 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int slot = 16 * j + 4 * q + b;
          const uint32_t v = slot < c ? (static_cast<uint32_t>(tile_col((o[q] >> (8 * b)) & 0xffu)) & 0xffu)
                                      : 0xffu;
          r |= v << (8 * b);
        }
        o[q] = r;
      }
      reinterpret_cast<uint4*>(p.ell_col + (dst_rt + k) * C)[j] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (j == 0) p.ell_cnt[dst_rt + k] = static_cast<uint8_t>(c);
  }
}

__global__ void __launch_bounds__(256) dense_fill_kernel(const HybParams p) {
  const int i = blockIdx.x;
  const int n = min(*p.n_dense, p.max_dense);
  if (i >= n) return;
  const int t = p.dense_rows[i];
  if (!in_bounds(t, p.T, p.status)) return;  // CTA-uniform
  const size_t rt0 = static_cast<size_t>(t) * p.n_t;
  float* out = p.dense_h + static_cast<size_t>(i) * p.F;
  for (int j = threadIdx.x; j < p.F; j += blockDim.x) {
    const int k = j / TWELL_TILE;
    const int cc = j % TWELL_TILE;
    const int c = p.cnt[rt0 + k];
    float v = 0.0f;
    if (c > p.W) {
      const int slot = p.spill_slot[rt0 + k];
      if (slot >= 0 && slot < p.spill_cap)
        v = p.spill_val[static_cast<size_t>(slot) * TWELL_TILE + cc];
      else if (cc == 0 && p.status)
        atomicOr(p.status, TWELL_FLAG_SPILL_FULL);
    } else {
      const uint8_t* sc = p.col + (rt0 + k) * p.W;
      const float* sv = p.val + (rt0 + k) * p.W;
      for (int s = 0; s < min(c, p.W); ++s)
        if (sc[s] == cc) v = sv[s];
    }
    out[j] = v;
  }
}

}  // namespace

twell_status check_hybrid(const hybrid_t* h, int32_t T, int32_t F) {
  if (h == nullptr) return TWELL_ERR_INVALID;
  if (h->T != T || h->F != F || h->tile != TWELL_TILE) return TWELL_ERR_INVALID;
  if (h->cap < 1 || h->cap > TWELL_TILE || h->max_dense < 0) return TWELL_ERR_INVALID;
  if (T == 0) return TWELL_OK;
  if (!h->n_ell || !h->n_dense || !h->row_map || !h->ell_rows || !h->ell_val || !h->ell_col ||
      !h->ell_cnt)
    return TWELL_ERR_INVALID;
  if (h->max_dense > 0 && (!h->dense_rows || !h->dense_h || !aligned16(h->dense_h)))
    return TWELL_ERR_INVALID;
  if (!aligned16(h->ell_val) || !aligned16(h->row_map) || !aligned16(h->ell_rows) ||
      !aligned16(h->ell_col) || !aligned16(h->ell_cnt))
    return TWELL_ERR_INVALID;
  return TWELL_OK;
}

}  // namespace twell

extern "C" twell_status twell_to_hybrid(const twell_t* h, const hybrid_t* out,
                                        int32_t* status_dev, void* stream) {
  using namespace twell;
  if (h == nullptr || out == nullptr) return TWELL_ERR_INVALID;
  twell_status st = check_twell(h, h->T, h->F, false);
  if (st != TWELL_OK) return st;
  if ((st = check_hybrid(out, h->T, h->F)) != TWELL_OK) return st;
  if (h->T == 0) return TWELL_OK;
  if (!status_dev) return TWELL_ERR_INVALID;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  HybParams p;
  p.val = h->val;
  p.col = h->col;
  p.cnt = h->cnt;
  p.spill_slot = h->spill_slot;
  p.spill_val = h->spill_val;
  p.spill_cap = h->spill_cap;
  p.W = h->width;
  p.T = h->T;
  p.F = h->F;
  p.n_t = h->F / TWELL_TILE;
  p.C = out->cap;
  p.max_dense = out->max_dense;
  p.n_ell = out->n_ell;
  p.n_dense = out->n_dense;
  p.row_map = out->row_map;
  p.ell_rows = out->ell_rows;
  p.ell_val = out->ell_val;
  p.ell_col = out->ell_col;
  p.ell_cnt = out->ell_cnt;
  p.dense_rows = out->dense_rows;
  p.dense_h = out->dense_h;
  p.status = status_dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int warp_blocks = static_cast<int>((static_cast<long long>(p.T) * 32 + 255) / 256);
  classify_kernel<<<warp_blocks, 256, 0, s>>>(p);
  scan_kernel<<<1, kScanThreads, 0, s>>>(p);
  const bool chunks = p.W == p.C && aligned16(h->val) && aligned16(h->col);
  if (chunks && p.C == 32)
    ell_copy_kernel<32><<<warp_blocks, 256, 0, s>>>(p);
  else if (chunks && p.C == 16)
    ell_copy_kernel<16><<<warp_blocks, 256, 0, s>>>(p);
  else
    ell_fill_kernel<<<warp_blocks, 256, 0, s>>>(p);
  if (p.max_dense > 0) dense_fill_kernel<<<p.max_dense, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
