// Tensor-core products over the ELL part of the hybrid training format
// ("Sparser, Faster, Lighter Transformer Language Models", section 2.B.3:
// dense-to-sparse and sparse-to-dense matmuls of the forward and backward
// passes over the hybrid format).
//
// A variant of the CUDA-core ELL kernels for the dense activation regimes of
// training, where every 128-token block touches every neuron tile: the ELL
// values are expanded tile by tile in shared memory into fp16 MMA operands,
// and the dense-to-sparse products are full tcgen05 tiles of which only the
// ELL entries are kept.  Operands in bf16 or fp16 (the sparse values written
// as fp16), fp32 accumulation in TMEM.
#pragma once

#include "common.cuh"

namespace twell {

enum TcMode : int32_t {
  // acc = X_ell W_u (M = ELL rows, N = F, K = D); at the ELL entries (i, j):
  // u_ell = acc, a_ell = fp16(h acc)
  TC_SAMPLE_U = 0,
  // acc = sum_s dY_s W_d^T (M = ELL rows, N = F, K = D per segment; the
  // segments are the fp16 hi and lo halves of s dy); at the entries, in
  // fp16: du = acc h, dz = acc u + s lambda (hi in dz_ell and, when
  // dz_lo_ell is set, lo), a = h u
  TC_SAMPLE_DA = 1,
  // out[row_idx[i]][:] = sum_s E_s[i][:] W_s (M = ELL rows, N = D, K = F per
  // segment, up to 3 segments), E_s = ELL values vals_s expanded to dense
  // fp16 rows, W_s [F][D]
  TC_ROWS = 2,
  // out[j][:] = sum_s sum_i E_s[i][j] B_s[i][:] (M = F, N = D, K = ELL rows
  // per segment), E_s the ELL values vals_s expanded, B_s [rows][D] fp16 (the
  // gathered x or dy rows)
  TC_TRANS = 3
};

constexpr int kTcMaxSeg = 3;

struct TcMaps {
  CUtensorMap a[2];             // SAMPLE: dense A [rows][D] per segment, box 64 x 128
  CUtensorMap b[kTcMaxSeg];     // SAMPLE: W [F][D] box 64 x 256 (b[0], every segment);
                                // ROWS / TRANS: [K][D] box 64 x 64 per segment
  CUtensorMap cols;             // ROWS / TRANS: u8 ELL columns [rows][n_t C], box C x (128|64)
  CUtensorMap vals[kTcMaxSeg];  // ROWS / TRANS: fp16 ELL values [rows][n_t C] per segment
};

struct TcArgs {
  int32_t mode;
  int32_t rows_cap;        // rows of the ELL arrays (host bound)
  const int32_t* n_rows;   // ELL rows present (device)
  int32_t n_t, C, D, F;
  int32_t nseg;            // SAMPLE: 1 or 2 A segments; ROWS / TRANS: 1..3
  // SAMPLE epilogues
  const uint8_t* ell_col;
  const uint8_t* ell_cnt;
  const float* ell_val;
  float* u_ell;            // SAMPLE_U out, SAMPLE_DA in
  uint16_t* a_ell;         // fp16 h u, out of both
  uint16_t* dz_ell;        // SAMPLE_DA out: fp16(dz)
  uint16_t* dz_lo_ell;     // SAMPLE_DA out (optional): fp16(dz - fp16(dz))
  uint16_t* du_ell;        // SAMPLE_DA out: fp16(du)
  float lambda;
  // The A and B tiles of every segment are fp16 (else bf16).  The values the
  // SAMPLE epilogues write are fp16 either way; one beyond the fp16 range
  // sets TWELL_FLAG_RANGE.
  int32_t f16_ops;
  // Gradient scaling (scale.cuh), when amax is set: SAMPLE_DA's accumulator
  // is s da (dy scaled by s), and it writes s dz = acc u + s lambda and
  // s du = acc h; ROWS and TRANS multiply their accumulators by 1 / s.
  const uint32_t* amax;
  float amax_floor;
  // ROWS / TRANS epilogues
  float* out;
  int64_t ldo;
  const int32_t* row_idx;  // ROWS: output row of ELL row i
  int32_t row_limit;       // rows of out that row_idx may name (0: unchecked)
  int32_t* status;
  // ROWS / TRANS, set by the launch: K parts per tile (1 or 2); with 2, each
  // part adds its product into out, which the launch zeroes first
  int32_t ksplit;
};

// Tensor maps of the operands (box shapes as listed in TcMaps).
// `pitch` = elements between rows (D when 0).
twell_status tc_map_a(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t D,
                      int64_t pitch = 0);
twell_status tc_map_w_kmajor(CUtensorMap* m, const uint16_t* base, int64_t F, int64_t D);
twell_status tc_map_mn(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t D,
                       int64_t pitch = 0);
// ELL columns / values ([rows][n_t][C]; padding slots of the columns hold
// 0xff), box C x box_rows (128 for ROWS, 64 for TRANS).
twell_status tc_map_cols(CUtensorMap* m, const uint8_t* base, int64_t rows, int64_t n_t,
                         int64_t C, int box_rows);
twell_status tc_map_vals(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t n_t,
                         int64_t C, int box_rows);

// Shapes the kernels accept: D % 64 == 0, F % 128 == 0, C in {16, 32}.
bool tc_supported(int32_t D, int32_t F, int32_t C);

twell_status tc_run(const TcMaps& maps, const TcArgs& a, const DeviceInfo& dev, cudaStream_t s);

}  // namespace twell
