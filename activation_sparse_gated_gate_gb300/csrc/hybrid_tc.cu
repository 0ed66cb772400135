// Tensor-core entry points of the hybrid training forward and backward
// ("Sparser, Faster, Lighter Transformer Language Models", section 2.B.3:
// the hybrid format's sparse-to-dense and dense-to-sparse matmuls; the L1
// coefficient from the news article "Sakana AI and NVIDIA TwELL boosts LLM
// training speed by 21.9%", recipe list).
//
// ELL rows, forward:
//   Xe = x[ell rows] (bf16 gather)
//   SAMPLE_U   u = Xe W_u at the ELL entries -> u_ell, a = fp16(h u)
//   ROWS       y[ell rows] = E(a) W_d16                         (fp16 operands)
// ELL rows, backward (every operand fp16; s = the power-of-two gradient
// scale of scale.cuh, from max(max |dy|, 2^-14 lambda)):
//   Xe = fp16(x[ell rows]), dYe = s dy[ell rows] as fp16 hi | lo (rows up
//             to the next multiple of 64 zero-filled: the K tail of TRANS)
//   SAMPLE_DA  s da = dYe_hi W_d16^T + dYe_lo W_d16^T at the entries ->
//              s dz = s da u + s lambda (fp16 hi and lo), s du = s da h, a = h u
//   ROWS       dx[ell rows] = (E(s dz_hi) W_g16^T + E(s dz_lo) W_g16^T +
//              E(s du) W_u16^T) / s
//   TRANS x3   dW_g^T = E(s dz)^T Xe / s, dW_u^T = E(s du)^T Xe / s,
//              dW_d = E(a)^T dYe_hi / s
// E(v) = the ELL values expanded to dense fp16 tiles in shared memory;
// W_*16 = fp16 copies of the weights, made in the workspace by each call.
// fp16 rounds each operand to 2^-11 relative (bf16: 2^-8) over a range that
// covers activations and weights and, after the scaling, gradients; a value
// that leaves it sets TWELL_FLAG_RANGE.  A single fp16 segment per product
// replaces the bf16 hi + lo pairs a bf16 operand needs for the same error,
// except on the way to dx: a column of W_g with large entries for every
// neuron (a bias feature) sums a token's dz into one element of dx, where
// even fp16's rounding of each term, or the rounding of the token's dy that
// every da of the token shares, can reach a few percent of dx's RMS, so dz
// (in dx) and dy (in da) keep fp16 low halves (2^-22).
// Dense overflow rows: the shared tensor-core path with bf16 hi/lo splits,
// which writes its dx rows and adds its weight-gradient terms after TRANS.
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
                         cudaStream_t s, int32_t* status = nullptr,
                         const uint32_t* amax = nullptr, float amax_floor = 0.0f) {
  GatherArgs g{};
  g.status = status;
  g.amax = amax;
  g.amax_floor = amax_floor;
  g.src = src;
  g.lds = D;
  g.row_idx = h->ell_rows;
  g.row_limit = h->T;
  g.R = h->T;
  g.C = D;
  g.R_dyn = h->n_ell;
  g.out = out;
  g.ldo = mode == 3 ? 2 * static_cast<int64_t>(D) : D;
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
  uint16_t* Wd16 = reinterpret_cast<uint16_t*>(w + L.wd16);
  const size_t FD = static_cast<size_t>(F) * D;

  if ((st = twell_to_f16(Wd, Wd16, FD, status_dev, s)) != TWELL_OK) return st;
  if ((st = gather_rows(0, x, h, D, Xe, s)) != TWELL_OK) return st;
  {  // u at the ELL entries, a = fp16(h u)
    TcMaps m;
    if ((st = tc_map_a(&m.a[0], Xe, T, D)) != TWELL_OK) return st;
    if ((st = tc_map_w_kmajor(&m.b[0], Wu_t, F, D)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_SAMPLE_U, h, D, status_dev);
    a.u_ell = u_ell;
    a.a_ell = Ae;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  {  // y[ell rows] = E(a) W_d16
    TcMaps m;
    if ((st = tc_map_cols(&m.cols, h->ell_col, T, n_t, C, 128)) != TWELL_OK) return st;
    if ((st = tc_map_vals(&m.vals[0], Ae, T, n_t, C, 128)) != TWELL_OK) return st;
    if ((st = tc_map_mn(&m.b[0], Wd16, F, D)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_ROWS, h, D, status_dev);
    a.f16_ops = 1;
    a.out = y;
    a.ldo = D;
    a.row_idx = h->ell_rows;
    a.row_limit = h->T;
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
  uint16_t* dZe = reinterpret_cast<uint16_t*>(w + L.dze);
  uint16_t* dZl = reinterpret_cast<uint16_t*>(w + L.dzl);
  uint16_t* dUe = reinterpret_cast<uint16_t*>(w + L.due);
  uint16_t* Wg16 = reinterpret_cast<uint16_t*>(w + L.wg16);
  uint16_t* Wu16 = reinterpret_cast<uint16_t*>(w + L.wu16);
  uint16_t* Wd16 = reinterpret_cast<uint16_t*>(w + L.wd16);
  uint32_t* amax = reinterpret_cast<uint32_t*>(w + L.amax);
  const size_t FD = static_cast<size_t>(F) * D;
  const float floor_v = l1_coeff * 0x1p-14f;  // s lambda < 2^14

  if ((st = twell_to_f16(Wg_t, Wg16, FD, status_dev, s)) != TWELL_OK) return st;
  if ((st = twell_to_f16(Wu_t, Wu16, FD, status_dev, s)) != TWELL_OK) return st;
  if ((st = twell_to_f16(Wd, Wd16, FD, status_dev, s)) != TWELL_OK) return st;
  if ((st = amax_run(dy, static_cast<int64_t>(T) * D, amax, s)) != TWELL_OK) return st;
  if ((st = gather_rows(4, x, h, D, Xe, s, status_dev)) != TWELL_OK) return st;
  if ((st = gather_rows(3, dy, h, D, dYe, s, status_dev, amax, floor_v)) != TWELL_OK) return st;
  const int64_t D2 = 2 * static_cast<int64_t>(D);
  {  // s da at the ELL entries -> s dz, s du, a
    TcMaps m;
    if ((st = tc_map_a(&m.a[0], dYe, T, D, D2)) != TWELL_OK) return st;
    if ((st = tc_map_a(&m.a[1], dYe + D, T, D, D2)) != TWELL_OK) return st;
    if ((st = tc_map_w_kmajor(&m.b[0], Wd16, F, D)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_SAMPLE_DA, h, D, status_dev);
    a.nseg = 2;
    a.f16_ops = 1;
    a.amax = amax;
    a.amax_floor = floor_v;
    a.u_ell = const_cast<float*>(u_ell);
    a.a_ell = Ae;
    a.dz_ell = dZe;
    a.dz_lo_ell = dZl;
    a.du_ell = dUe;
    a.lambda = l1_coeff;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  {  // dx[ell rows] = (E(s dz_hi) W_g16^T + E(s dz_lo) W_g16^T + E(s du) W_u16^T) / s
    TcMaps m;
    if ((st = tc_map_mn(&m.b[0], Wg16, F, D)) != TWELL_OK) return st;
    if ((st = tc_map_mn(&m.b[1], Wg16, F, D)) != TWELL_OK) return st;
    if ((st = tc_map_mn(&m.b[2], Wu16, F, D)) != TWELL_OK) return st;
    if ((st = tc_map_cols(&m.cols, h->ell_col, T, n_t, C, 128)) != TWELL_OK) return st;
    const uint16_t* segv[3] = {dZe, dZl, dUe};
    for (int q = 0; q < 3; ++q)
      if ((st = tc_map_vals(&m.vals[q], segv[q], T, n_t, C, 128)) != TWELL_OK) return st;
    TcArgs a = tc_args(TC_ROWS, h, D, status_dev);
    a.nseg = 3;
    a.f16_ops = 1;
    a.amax = amax;
    a.amax_floor = floor_v;
    a.out = dx;
    a.ldo = D;
    a.row_idx = h->ell_rows;
    a.row_limit = h->T;
    if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
  }
  {  // weight gradients of the ELL rows (overwrite)
    struct Job {
      const uint16_t* vals;
      const uint16_t* b;
      int64_t pitch;
      float* out;
    };
    const Job jobs[3] = {{dZe, Xe, D, dWg_t}, {dUe, Xe, D, dWu_t}, {Ae, dYe, D2, dWd}};
    for (const Job& jb : jobs) {
      TcMaps m;
      TcArgs a = tc_args(TC_TRANS, h, D, status_dev);
      a.f16_ops = 1;
      a.amax = amax;
      a.amax_floor = floor_v;
      if ((st = tc_map_cols(&m.cols, h->ell_col, T, n_t, C, 64)) != TWELL_OK) return st;
      if ((st = tc_map_mn(&m.b[0], jb.b, T, D, jb.pitch)) != TWELL_OK) return st;
      if ((st = tc_map_vals(&m.vals[0], jb.vals, T, n_t, C, 64)) != TWELL_OK) return st;
      a.out = jb.out;
      a.ldo = D;
      if ((st = tc_run(m, a, dev, s)) != TWELL_OK) return st;
    }
  }
  if (h->max_dense == 0) return TWELL_OK;
  return dense_rows_bwd(x, h, U_dense, Wg_t, Wu_t, Wd, D, dy, l1_coeff, dx, dWg_t, dWu_t, dWd, w,
                        L, status_dev, dev, s);
}
