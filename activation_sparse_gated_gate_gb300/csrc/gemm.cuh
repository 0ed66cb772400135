// Internal building blocks for the dense-overflow rows of the hybrid
// training format: a tcgen05 GEMM with selectable epilogues, and transpose /
// row-gather kernels that prepare its bf16 operands.
#pragma once

#include "common.cuh"

namespace twell {

constexpr int kGemmMaxSeg = 4;

// One K segment of C = sum_s A_s B_s^T: A_s rows come from tensor map
// maps.a[map_a] (K-major, [M][K_s]), B_s rows from maps.b[map_b] ([N][K_s]).
// K_s = len, or min(len, *len_dyn) when len_dyn is set (a device count).
// Columns past K_s must read as zero (each map's inner extent ends there).
struct GemmSeg {
  int32_t map_a;
  int32_t map_b;
  int32_t len;
  const int32_t* len_dyn;
};

enum GemmEpi : int32_t {
  EPI_STORE = 0,  // C[row(m)][n] = acc
  EPI_ADD = 1,    // C[row(m)][n] += acc
  EPI_UP = 2,     // u = acc: U_out[m][n] = u; a = H[m][n] u split into bf16
                  // S_out[m][n] (hi) and S_out[m][N + n] (lo)
  EPI_DA = 3      // da = acc, h = H[m][n], u = U_in[m][n]: du = da h,
                  // dz = h > 0 ? da u + lambda : 0; bf16 splits into S_out row m:
                  // [dz hi | dz lo | du hi | du lo], N columns each
};

struct GemmArgs {
  int32_t M, N;
  // K split into ksplit contiguous ranges of k blocks, each accumulated in
  // TMEM on its own and added into C with fp32 atomics (EPI_STORE then needs
  // C zeroed first).  Shorter tensor-core accumulations keep the fp32
  // accumulator error small and give small-M products more parallelism.
  // EPI_UP / EPI_DA need ksplit == 1.
  int32_t ksplit;
  const int32_t* M_dyn;  // rows present = min(M, *M_dyn) when set
  int32_t nseg;
  GemmSeg seg[kGemmMaxSeg];
  int32_t epi;
  float* C;
  int64_t ldc;
  const int32_t* row_idx;  // STORE / ADD: output row of tile row m (identity when null)
  int32_t row_limit;       // rows of C that row_idx may name (0: unchecked; checked only
                           // in the bounds-checking build)
  const float* H;          // [M][N]
  const float* U_in;       // [M][N]
  float* U_out;            // [M][N]
  uint16_t* S_out;         // bf16 splits, row pitch lds
  int64_t lds;
  float lambda;
  int32_t* status;
};

struct GemmMaps {
  CUtensorMap a[kGemmMaxSeg];
  CUtensorMap b[kGemmMaxSeg];
};

// K-major bf16 operand map over rows of `rows` x `cols` (pitch elements per
// row) with the GEMM's box; `cols` ends the K extent (zero fill beyond).
twell_status gemm_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                      int64_t pitch, bool is_b_wide);

twell_status gemm_run(const GemmMaps& maps, const GemmArgs& a, bool wide_n,
                      const DeviceInfo& dev, cudaStream_t s);

// Split factor for a product of `tiles` output tiles over `k` total columns:
// at most 64 k blocks (4096 columns) per accumulation, and enough units to
// give every SM two.
int gemm_ksplit(int64_t tiles, int64_t k, const DeviceInfo& dev);

// C[row_idx[i]][0..N) = 0 for i < min(R, *R_dyn).
// (row_limit: rows of C that row_idx may name, 0 unchecked; checked only in
// the bounds-checking build, with TWELL_FLAG_BOUNDS in *status)
twell_status zero_rows(float* C, int64_t ldc, const int32_t* row_idx, int32_t R,
                       const int32_t* R_dyn, int32_t N, cudaStream_t s, int32_t row_limit = 0,
                       int32_t* status = nullptr);

// out_hi[c][r] (and out_lo[c][r]) = transposed, bf16-split value v(r, c) for
// r < R_act (= min(R, *R_dyn)), zeros for R_act <= r < R_pad, c < C:
//   MODE 0  v = src_bf16[row(r)][c]                     (bf16 copy, out_lo unused)
//   MODE 1  v = src_f32[row(r)][c], hi = bf16(v), lo = bf16(v - hi)
//   MODE 2  v = src_f32[r][c] * src2[r][c], split as MODE 1
struct TransposeArgs {
  const void* src;
  int64_t lds;
  const int32_t* row_idx;
  const float* src2;
  int64_t lds2;
  int32_t R, C, R_pad;
  const int32_t* R_dyn;
  uint16_t* out_hi;
  uint16_t* out_lo;
  int64_t ldo;
  int32_t row_limit;  // rows of src that row_idx may name (0: unchecked)
  int32_t* status;    // TWELL_FLAG_BOUNDS in the bounds-checking build
};
twell_status transpose_run(int mode, const TransposeArgs& a, cudaStream_t s);

// out[i][:] = src[row_idx[i]][:] for i < R_act = min(R, *R_dyn):
//   MODE 0  bf16 rows of C elements (C % 8 == 0), out pitch ldo
//   MODE 1  fp32 rows split into bf16 [hi (C) | lo (C)], out pitch ldo
//   MODE 2  fp32 rows rounded to bf16 (C % 8 == 0), out pitch ldo
//   MODE 3  fp32 rows -> fp16 [hi | lo] (C % 4 == 0), out pitch ldo >= 2C;
//           with amax set the rows are first multiplied by the power-of-two
//           gradient scale of scale.cuh
//   MODE 4  bf16 rows converted to fp16 (C % 8 == 0), out pitch ldo
//   (modes 3 and 4 set TWELL_FLAG_RANGE in *status, when given, for a value
//   beyond the fp16 range)
// With pad > 0, rows R_act <= i < min(R, R_act rounded up to pad) are
// written as zeros.
struct GatherArgs {
  const void* src;
  int64_t lds;
  const int32_t* row_idx;
  int32_t row_limit;  // rows of src that row_idx may name (0: unchecked)
  int32_t R, C;
  const int32_t* R_dyn;
  uint16_t* out;
  int64_t ldo;
  int32_t pad;
  int32_t* status;
  const uint32_t* amax;
  float amax_floor;
};
twell_status gather_run(int mode, const GatherArgs& a, cudaStream_t s);

// *out = the bits of max_i |src[i]| over n floats (n % 4 == 0, src 16-byte
// aligned); NaN compares above every number.  Two launches (a clear, then a
// grid-stride maximum with one atomic per warp).
twell_status amax_run(const float* src, int64_t n, uint32_t* out, cudaStream_t s);

}  // namespace twell
