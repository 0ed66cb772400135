// Workspace layouts of the hybrid training forward and backward (one
// definition used by the entry points and by twell_workspace_size).
#pragma once

#include "common.cuh"

namespace twell {

struct WsLayout {
  size_t bytes = 0;
  // tensor-core ELL path: gathered x / dy rows, fp16 ELL values and
  // weights, the gradient scale's maximum
  size_t xe = 0, dye = 0, ae = 0, dze = 0, dzl = 0, due = 0, wg16 = 0, wu16 = 0, wd16 = 0,
         amax = 0;
  // forward
  size_t xo = 0, wdT = 0, asplit = 0;
  // backward
  size_t cnt = 0, offs = 0, cursor = 0, records = 0, dys = 0, g = 0, wgT = 0, wuT = 0;
  size_t xoT = 0, dyT_hi = 0, dyT_lo = 0, dzT_hi = 0, dzT_lo = 0, duT_hi = 0, duT_lo = 0,
         aoT_hi = 0, aoT_lo = 0;
  int64_t mpad = 0;  // max_dense rounded up to the GEMM K block (64)
};

// One ELL-entry record of the backward, stored per neuron (CSC order).
struct BwdRecord {
  int32_t t;   // token
  float dz;    // dL/dz at (t, j)
  float du;    // dL/du at (t, j)
  float a;     // h * u at (t, j)
};

inline size_t ws_take(size_t* cur, size_t n) {
  const size_t off = (*cur + 255) & ~static_cast<size_t>(255);
  *cur = off + n;
  return off;
}

inline WsLayout ws_layout(int op, int64_t T, int64_t D, int64_t F, int64_t cap,
                          int64_t max_dense) {
  WsLayout w;
  size_t cur = 0;
  const int64_t n_t = F / TWELL_TILE;
  w.mpad = (max_dense + 63) / 64 * 64;
  if (op == 3 || op == 4) {
    w.xe = ws_take(&cur, T * D * 2);
    w.ae = ws_take(&cur, T * n_t * cap * 2);
    w.wd16 = ws_take(&cur, F * D * 2);
  }
  if (op == 4) {
    w.dye = ws_take(&cur, T * 2 * D * 2);  // fp16 [hi | lo] rows
    w.dze = ws_take(&cur, T * n_t * cap * 2);
    w.dzl = ws_take(&cur, T * n_t * cap * 2);
    w.due = ws_take(&cur, T * n_t * cap * 2);
    w.wg16 = ws_take(&cur, F * D * 2);
    w.wu16 = ws_take(&cur, F * D * 2);
    w.amax = ws_take(&cur, 4);
  }
  if (op == 1 || op == 3) {
    w.xo = ws_take(&cur, max_dense * D * 2);
    w.wdT = ws_take(&cur, D * F * 2);
    w.asplit = ws_take(&cur, max_dense * 2 * F * 2);
  } else if (op == 2 || op == 4) {
    if (op == 2) {
      w.cnt = ws_take(&cur, F * 4);
      w.offs = ws_take(&cur, (F + 1) * 4);
      w.cursor = ws_take(&cur, F * 4);
      w.records = ws_take(&cur, T * n_t * cap * sizeof(BwdRecord));
    }
    w.xo = ws_take(&cur, max_dense * D * 2);
    w.dys = ws_take(&cur, max_dense * 2 * D * 2);
    w.g = ws_take(&cur, max_dense * 4 * F * 2);
    w.wgT = ws_take(&cur, D * F * 2);
    w.wuT = ws_take(&cur, D * F * 2);
    w.xoT = ws_take(&cur, D * w.mpad * 2);
    w.dyT_hi = ws_take(&cur, D * w.mpad * 2);
    w.dyT_lo = ws_take(&cur, D * w.mpad * 2);
    w.dzT_hi = ws_take(&cur, F * w.mpad * 2);
    w.dzT_lo = ws_take(&cur, F * w.mpad * 2);
    w.duT_hi = ws_take(&cur, F * w.mpad * 2);
    w.duT_lo = ws_take(&cur, F * w.mpad * 2);
    w.aoT_hi = ws_take(&cur, F * w.mpad * 2);
    w.aoT_lo = ws_take(&cur, F * w.mpad * 2);
  }
  w.bytes = (cur + 255) & ~static_cast<size_t>(255);
  return w;
}

// Dense overflow rows of the hybrid forward / backward (tensor cores with
// bf16 hi/lo operand splits), shared by the CUDA-core and tensor-core entry
// points; `w` is the workspace laid out by L.
twell_status dense_rows_fwd(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                            const uint16_t* Wd, int32_t D, float* y, float* U_dense,
                            uint8_t* w, const WsLayout& L, int32_t* status_dev,
                            const DeviceInfo& dev, cudaStream_t s);
twell_status dense_rows_bwd(const uint16_t* x, const hybrid_t* h, const float* U_dense,
                            const uint16_t* Wg_t, const uint16_t* Wu_t, const uint16_t* Wd,
                            int32_t D, const float* dy, float l1_coeff, float* dx, float* dWg_t,
                            float* dWu_t, float* dWd, uint8_t* w, const WsLayout& L,
                            int32_t* status_dev, const DeviceInfo& dev, cudaStream_t s);

}  // namespace twell
