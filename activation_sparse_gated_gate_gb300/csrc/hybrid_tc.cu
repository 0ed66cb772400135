// Tensor-core entry points of the hybrid training forward and backward
// ("Sparser, Faster, Lighter Transformer Language Models", section 2.B.3:
// the hybrid format's sparse-to-dense and dense-to-sparse matmuls; the L1
// coefficient from the news article "Sakana AI and NVIDIA TwELL boosts LLM
// training speed by 21.9%", recipe list).
//
// ELL rows, forward:
//   Xe = x[ell rows] (bf16 gather)
//   SAMPLE_U   u = Xe W_u at the ELL entries -> u_ell, a = bf16(h u)
//   ROWS       y[ell rows] = E(a) W_d
// ELL rows, backward:
//   Xe = x[ell rows] (bf16), dYe = dy[ell rows] split into bf16 hi | lo
//             (rows up to the next multiple of 64 zero-filled: the K tail of
//             TRANS)
//   SAMPLE_DA  da = dYe_hi W_d^T + dYe_lo W_d^T at the entries -> dz = da u +
//              lambda (bf16 hi and lo), du = da h, a = h u (bf16)
//   ROWS       dx[ell rows] = E(dz_hi) W_g^T + E(dz_lo) W_g^T + E(du) W_u^T
//   TRANS x3   dW_g^T = E(dz_hi)^T Xe + E(dz_lo)^T Xe, dW_u^T = E(du)^T Xe,
//              dW_d = E(a_hi)^T dYe_hi + E(a_lo)^T dYe_hi + E(a_hi)^T dYe_lo
// dy and dz keep their low halves: a column of W_g with large entries for
// every neuron (a bias feature) sums dz into dx, where a single bf16
// rounding of each term would dominate the column's error, and dz = da u is
// the most heavy-tailed of the sparse values (a product of two roughly
// normal factors), so in dW_g a few large terms can carry the rounding of
// an element.  In dW_d both factors are activations; their low halves (the
// a_lo dy_lo product is below fp32 resolution and left out) keep the
// heavy-tailed terms that dominate some elements from carrying a bf16
// rounding each.
// E(v) = the ELL values expanded to dense bf16 tiles in shared memory.
// Dense overflow rows: the shared tensor-core path with hi/lo splits, which
// writes its dx rows and adds its weight-gradient terms after TRANS.
#include "hybrid.cuh"
#include "gemm.cuh"
#include "tc_ell.cuh"

namespace twell {
namespace {

twell_status tc_common_checks(const hybrid_t* h, int32_t D, int32_t* T_out) {
  if (h == nullptr) return TWELL_ERR_INVALID;
  const int32_t T = h->T, F = h->F;
  if (T < 0 || F <= 0 || F % TWELL_TILE != 0 || D <= 0 || D % 8 != 0) return TWELL_ERR_INVALID;
  twell_status st = check_hybrid(h, T, F);
  if (st != TWELL_OK) return st;
  if (!tc_supported(D, F, h->cap)) return TWELL_ERR_UNSUPPORTED;
  *T_out = T;
  return TWELL_OK;
}

twell_status gather_rows(int mode, const void* src, const hybrid_t* h, int32_t D, uint16_t* out,
                         cudaStream_t s) {
  GatherArgs g{};
  g.src = src;
  g.lds = D;
  g.row_idx = h->ell_rows;
  g.R = h->T;
  g.C = D;
  g.R_dyn = h->n_ell;
  g.out = out;
  g.ldo = mode == 1 ? 2 * static_cast<int64_t>(D) : D;
  g.pad = 64;
  return gather_run(mode, g, s);
}

TcArgs tc_args(int mode, const hybrid_t* h, int32_t D, int32_t* status_dev) {
  TcArgs a{};
  a.mode = mode;
  a.rows_cap = h->T;
  a.n_rows = h->n_ell;
  a.n_t = h->F / TWELL_TILE;
  a.C = h->cap;
  a.D = D;
  a.F = h->F;
  a.nseg = 1;
  a.ell_col = h->ell_col;
  a.ell_cnt = h->ell_cnt;
  a.ell_val = h->ell_val;
  a.status = status_dev;
  return a;
}

}  // namespace
}  // namespace twell

extern "C" twell_status hybrid_ffn_fwd_tc(const uint16_t* x, const hybrid_t* h,
                                          const uint16_t* Wu_t, const uint16_t* Wd, int32_t D,
                                          float* y, float* u_ell, float* U_dense, void* ws,
                                          size_t ws_bytes, int32_t* status_dev, void* stream) {
  using namespace twell;
  int32_t T = 0;
  twell_status st = tc_common_checks(h, D, &T);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  const int32_t F = h->F, C = h->cap, n_t = F / TWELL_TILE;
  const WsLayout L = ws_layout(3, T, D, F, C, h->max_dense);
  if (!x || !Wu_t || !Wd || !y || !u_ell || !status_dev || !ws || ws_bytes < L.bytes)
    return TWELL_ERR_INVALID;
  if (h->max_dense > 0 && !U_dense) return TWELL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(y) ||
      !aligned16(u_ell) || (U_dense && !aligned16(U_dense)) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return TWELL_ERR_INVALID;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Xe = reinterpret_cast<uint16_t*>(w + L.xe);
  uint16_t* Ae = reinterpret_cast<uint16_t*>(w + L.ae);

  if ((st = gather_rows(0, x, h, D, Xe, s)) != TWELL_OK) return st;
  {  // u at the ELL entries, a = bf16(h u)
    TcMaps m;
    if ((st = tc_map_a(&m.a[0], Xe, T, D)) != TWELL_OK) return st;
    if ((st = tc_map_w_kmajor(&m.b[0], Wu_t, F, D)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_SAMPLE_U, h, D, status_dev);
    a.u_ell = u_ell;
    a.a_ell = Ae;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  {  // y[ell rows] = E(a) W_d
    TcMaps m;
    if ((st = tc_map_cols(&m.cols, h->ell_col, T, n_t, C, 128)) != TWELL_OK) return st;
    if ((st = tc_map_vals(&m.vals[0], Ae, T, n_t, C, 128)) != TWELL_OK) return st;
    if ((st = tc_map_mn(&m.b[0], Wd, F, D)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_ROWS, h, D, status_dev);
    a.out = y;
    a.ldo = D;
    a.row_idx = h->ell_rows;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  if (h->max_dense == 0) return TWELL_OK;
  return dense_rows_fwd(x, h, Wu_t, Wd, D, y, U_dense, w, L, status_dev, dev, s);
}

extern "C" twell_status hybrid_ffn_bwd_tc(const uint16_t* x, const hybrid_t* h,
                                          const float* u_ell, const float* U_dense,
                                          const uint16_t* Wg_t, const uint16_t* Wu_t,
                                          const uint16_t* Wd, int32_t D, const float* dy,
                                          float l1_coeff, float* dx, float* dWg_t,
                                          float* dWu_t, float* dWd, void* ws, size_t ws_bytes,
                                          int32_t* status_dev, void* stream) {
  using namespace twell;
  int32_t T = 0;
  twell_status st = tc_common_checks(h, D, &T);
  if (st != TWELL_OK) return st;
  const int32_t F = h->F, C = h->cap, n_t = F / TWELL_TILE;
  if (!Wg_t || !Wu_t || !Wd || !dWg_t || !dWu_t || !dWd || !status_dev) return TWELL_ERR_INVALID;
  if (!aligned16(Wg_t) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(dWg_t) ||
      !aligned16(dWu_t) || !aligned16(dWd))
    return TWELL_ERR_INVALID;
  const WsLayout L = ws_layout(4, T, D, F, C, h->max_dense);
  if (T > 0) {
    if (!x || !dy || !dx || !u_ell || !ws || ws_bytes < L.bytes) return TWELL_ERR_INVALID;
    if (h->max_dense > 0 && !U_dense) return TWELL_ERR_INVALID;
    if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(u_ell) ||
        (U_dense && !aligned16(U_dense)) || (reinterpret_cast<uintptr_t>(ws) & 255u))
      return TWELL_ERR_INVALID;
  }
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {  // no tokens: every gradient is zero
    const size_t wbytes = static_cast<size_t>(F) * D * sizeof(float);
    if (cudaMemsetAsync(dWg_t, 0, wbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dWu_t, 0, wbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dWd, 0, wbytes, s) != cudaSuccess)
      return TWELL_ERR_CUDA;
    return TWELL_OK;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Xe = reinterpret_cast<uint16_t*>(w + L.xe);
  uint16_t* dYe = reinterpret_cast<uint16_t*>(w + L.dye);
  uint16_t* Ae = reinterpret_cast<uint16_t*>(w + L.ae);
  uint16_t* Al = reinterpret_cast<uint16_t*>(w + L.ale);
  uint16_t* dZe = reinterpret_cast<uint16_t*>(w + L.dze);
  uint16_t* dZl = reinterpret_cast<uint16_t*>(w + L.dzl);
  uint16_t* dUe = reinterpret_cast<uint16_t*>(w + L.due);
  const int64_t D2 = 2 * static_cast<int64_t>(D);

  if ((st = gather_rows(0, x, h, D, Xe, s)) != TWELL_OK) return st;
  if ((st = gather_rows(1, dy, h, D, dYe, s)) != TWELL_OK) return st;
  {  // da at the ELL entries -> dz (hi, lo), du, a
    TcMaps m;
    if ((st = tc_map_a(&m.a[0], dYe, T, D, D2)) != TWELL_OK) return st;
    if ((st = tc_map_a(&m.a[1], dYe + D, T, D, D2)) != TWELL_OK) return st;
    if ((st = tc_map_w_kmajor(&m.b[0], Wd, F, D)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_SAMPLE_DA, h, D, status_dev);
    a.nseg = 2;
    a.u_ell = const_cast<float*>(u_ell);
    a.a_ell = Ae;
    a.a_lo_ell = Al;
    a.dz_ell = dZe;
    a.dz_lo_ell = dZl;
    a.du_ell = dUe;
    a.lambda = l1_coeff;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  {  // dx[ell rows] = E(dz_hi) W_g^T + E(dz_lo) W_g^T + E(du) W_u^T
    TcMaps m;
    if ((st = tc_map_mn(&m.b[0], Wg_t, F, D)) != TWELL_OK) return st;
    if ((st = tc_map_mn(&m.b[1], Wg_t, F, D)) != TWELL_OK) return st;
    if ((st = tc_map_mn(&m.b[2], Wu_t, F, D)) != TWELL_OK) return st;
    if ((st = tc_map_cols(&m.cols, h->ell_col, T, n_t, C, 128)) != TWELL_OK) return st;
    const uint16_t* segv[3] = {dZe, dZl, dUe};
    for (int q = 0; q < 3; ++q)
      if ((st = tc_map_vals(&m.vals[q], segv[q], T, n_t, C, 128)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_ROWS, h, D, status_dev);
    a.nseg = 3;
    a.out = dx;
    a.ldo = D;
    a.row_idx = h->ell_rows;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  {  // weight gradients of the ELL rows (overwrite)
    struct Job {
      int nseg;
      const uint16_t* vals[3];
      const uint16_t* b[3];
      int64_t pitch;
      float* out;
    };
    const Job jobs[3] = {{2, {dZe, dZl, nullptr}, {Xe, Xe, nullptr}, D, dWg_t},
                         {1, {dUe, nullptr, nullptr}, {Xe, nullptr, nullptr}, D, dWu_t},
                         {3, {Ae, Al, Ae}, {dYe, dYe, dYe + D}, D2, dWd}};
    for (const Job& jb : jobs) {
      TcMaps m;
      TcArgs a = tc_args(TC_TRANS, h, D, status_dev);
      a.nseg = jb.nseg;
      if ((st = tc_map_cols(&m.cols, h->ell_col, T, n_t, C, 64)) != TWELL_OK) return st;
      for (int q = 0; q < jb.nseg; ++q) {
        if ((st = tc_map_mn(&m.b[q], jb.b[q], T, D, jb.pitch)) != TWELL_OK) return st;
        if ((st = tc_map_vals(&m.vals[q], jb.vals[q], T, n_t, C, 64)) != TWELL_OK) return st;
      }
      a.out = jb.out;
      a.ldo = D;
      if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
    }
  }
  if (h->max_dense == 0) return TWELL_OK;
  return dense_rows_bwd(x, h, U_dense, Wg_t, Wu_t, Wd, D, dy, l1_coeff, dx, dWg_t, dWu_t, dWd, w,
                        L, status_dev, dev, s);
}
