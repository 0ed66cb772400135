// Internal interface of the fused gather kernel (TwELL inference forward and
// the ELL rows of the hybrid training forward).
#pragma once

#include "common.cuh"

namespace twell {

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
  int32_t G;           // column tiles per work unit
  int32_t upr;         // units per token row, ceil(n_t / G)
  int32_t split;       // rows split over several units: accumulate with atomics
  int32_t stages;      // P
  int32_t warp_bytes;  // shared memory per warp
  int32_t* status;
  // ELL mode (hybrid training forward): rows are the ELL rows of a hybrid
  // (count *n_rows, token ell_rows[i]); u is saved at every ELL slot
  const int32_t* n_rows;
  const int32_t* ell_rows;
  float* u_save;
  // y is zero on the stream already (split rows then skip their memset)
  int32_t y_zeroed;
};

struct Entry {
  int32_t j;    // neuron
  float h;      // gate value
  int32_t pos;  // ELL slot (ELL mode) where u is saved
};

// Launch the fused up+down kernel: TwELL rows (ell = false) or the ELL rows
// of a hybrid (ell = true; n_rows / ell_rows / u_save set, W = C, no spill).
twell_status launch_fused(const FfnParams& p, const DeviceInfo& dev, cudaStream_t s, bool ell);

// twell_ffn_fwd with its arguments already checked by the caller except the
// TwELL's; `y_zeroed`: y [T][D] is zero on `s` already (the decode step's
// gate kernel zeroes it), so no memset precedes the kernel.
twell_status ffn_fwd_twell(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                           const uint16_t* Wd, int32_t D, float* y, int32_t* status_dev,
                           cudaStream_t s, bool y_zeroed);

// Workspace bytes of twell_ffn_fwd_tc (sorted: twell_ffn_fwd_tc_sorted) for T
// rows, width D and F gate columns.
size_t ffn_tc_workspace_bytes(int64_t T, int64_t D, int64_t F, bool sorted);

}  // namespace twell
