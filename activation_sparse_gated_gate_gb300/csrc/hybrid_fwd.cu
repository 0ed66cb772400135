// Hybrid training forward ("Sparser, Faster, Lighter Transformer Language
// Models", section 2.B.3: sparse-to-dense and dense-to-sparse matmuls over
// the hybrid format in the forward pass).
//
// ELL rows: the fused gather kernel in ELL mode computes, per active (t, j),
// u = x_t . W_u[:, j] (the dense-to-sparse product, saved per ELL slot for
// the backward) and y_t += (h u) W_d[j, :] (the sparse-to-dense product).
// Dense overflow rows, on the tensor cores:
//   Xo = x[dense rows]                                       (gather)
//   U  = Xo W_u        G1, epilogue: save U, a = h * U split to bf16 hi/lo
//   y[dense rows] = a W_d = a_hi W_d + a_lo W_d              G2 (W_d^T staged,
//                  K split in ranges of <= 4096 summed with fp32 atomics)
#include "fused.cuh"
#include "gemm.cuh"
#include "hybrid.cuh"

extern "C" size_t twell_workspace_size(int32_t op, int32_t T, int32_t D, int32_t F,
                                       int32_t cap, int32_t max_dense) {
  if (op == TWELL_WS_FFN_FWD_TC || op == TWELL_WS_FFN_FWD_TC_SORTED)
    return T < 0 || D <= 0 || F <= 0
               ? 0
               : twell::ffn_tc_workspace_bytes(T, D, F, op == TWELL_WS_FFN_FWD_TC_SORTED);
  if (op < 1 || op > 4 || T < 0 || D <= 0 || F <= 0 || cap < 1 || max_dense < 0) return 0;
  return twell::ws_layout(op, T, D, F, cap, max_dense).bytes;
}

namespace twell {

twell_status dense_rows_fwd(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                            const uint16_t* Wd, int32_t D, float* y, float* U_dense,
                            uint8_t* w, const WsLayout& L, int32_t* status_dev,
                            const DeviceInfo& dev, cudaStream_t s) {
  const int32_t F = h->F;
  twell_status st;
  uint16_t* Xo = reinterpret_cast<uint16_t*>(w + L.xo);
  uint16_t* WdT = reinterpret_cast<uint16_t*>(w + L.wdT);
  uint16_t* As = reinterpret_cast<uint16_t*>(w + L.asplit);
  const int32_t MD = h->max_dense;

  GatherArgs g{};
  g.src = x;
  g.lds = D;
  g.row_idx = h->dense_rows;
  g.row_limit = h->T;
  g.R = MD;
  g.C = D;
  g.R_dyn = h->n_dense;
  g.out = Xo;
  g.ldo = D;
  if ((st = gather_run(0, g, s)) != TWELL_OK) return st;

  TransposeArgs tr{};
  tr.src = Wd;
  tr.lds = D;
  tr.R = F;
  tr.C = D;
  tr.R_pad = F;
  tr.out_hi = WdT;
  tr.ldo = F;
  if ((st = transpose_run(0, tr, s)) != TWELL_OK) return st;

  // G1: U = Xo W_u  (A = Xo [MD][D], B = Wu_t [F][D])
  {
    const int num_m = (MD + 127) / 128;
    const bool wide = static_cast<long long>(num_m) * ((F + 255) / 256) >= dev.sm_count;
    GemmMaps maps;
    if ((st = gemm_map(&maps.a[0], Xo, MD, D, D, false)) != TWELL_OK) return st;
    if ((st = gemm_map(&maps.b[0], Wu_t, F, D, D, wide)) != TWELL_OK) return st;
    GemmArgs a{};
    a.M = MD;
    a.N = F;
    a.M_dyn = h->n_dense;
    a.nseg = 1;
    a.seg[0] = GemmSeg{0, 0, D, nullptr};
    a.epi = EPI_UP;
    a.H = h->dense_h;
    a.U_out = U_dense;
    a.S_out = As;
    a.lds = 2 * static_cast<int64_t>(F);
    a.status = status_dev;
    if ((st = gemm_run(maps, a, wide, dev, s)) != TWELL_OK) return st;
  }
  // G2: y[dense rows] = a_hi W_d + a_lo W_d  (A = a halves [MD][F], B = W_d^T [D][F])
  {
    const int num_m = (MD + 127) / 128;
    const bool wide = static_cast<long long>(num_m) * ((D + 255) / 256) >= dev.sm_count;
    GemmMaps maps;
    if ((st = gemm_map(&maps.a[0], As, MD, F, 2 * static_cast<int64_t>(F), false)) != TWELL_OK)
      return st;
    if ((st = gemm_map(&maps.a[1], As + F, MD, F, 2 * static_cast<int64_t>(F), false)) !=
        TWELL_OK)
      return st;
    if ((st = gemm_map(&maps.b[0], WdT, D, F, F, wide)) != TWELL_OK) return st;
    GemmArgs a{};
    a.M = MD;
    a.N = D;
    a.M_dyn = h->n_dense;
    a.nseg = 2;
    a.seg[0] = GemmSeg{0, 0, F, nullptr};
    a.seg[1] = GemmSeg{1, 0, F, nullptr};
    a.epi = EPI_STORE;
    a.C = y;
    a.ldc = D;
    a.row_idx = h->dense_rows;
    a.row_limit = h->T;
    a.status = status_dev;
    a.ksplit = gemm_ksplit(static_cast<int64_t>(num_m) * ((D + (wide ? 255 : 127)) /
                                                           (wide ? 256 : 128)),
                           2 * static_cast<int64_t>(F), dev);
    if ((st = zero_rows(y, D, h->dense_rows, MD, h->n_dense, D, s, h->T, status_dev)) != TWELL_OK) return st;
    if ((st = gemm_run(maps, a, wide, dev, s)) != TWELL_OK) return st;
  }
  return TWELL_OK;
}

}  // namespace twell

extern "C" twell_status hybrid_ffn_fwd(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                                       const uint16_t* Wd, int32_t D, float* y, float* u_ell,
                                       float* U_dense, void* ws, size_t ws_bytes,
                                       int32_t* status_dev, void* stream) {
  using namespace twell;
  if (h == nullptr) return TWELL_ERR_INVALID;
  const int32_t T = h->T, F = h->F;
  if (T < 0 || F <= 0 || F % TWELL_TILE != 0 || D <= 0 || D % 8 != 0) return TWELL_ERR_INVALID;
  twell_status st = check_hybrid(h, T, F);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  const WsLayout L = ws_layout(1, T, D, F, h->cap, h->max_dense);
  if (!x || !Wu_t || !Wd || !y || !u_ell || !status_dev) return TWELL_ERR_INVALID;
  if (h->max_dense > 0 && (!U_dense || !ws || ws_bytes < L.bytes)) return TWELL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(y) ||
      !aligned16(u_ell) || (U_dense && !aligned16(U_dense)) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return TWELL_ERR_INVALID;
  if (D > 256 * 12) return TWELL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // ELL rows
  FfnParams p{};
  p.x = x;
  p.Wu_t = Wu_t;
  p.Wd = Wd;
  p.y = y;
  p.val = h->ell_val;
  p.col = h->ell_col;
  p.cnt = h->ell_cnt;
  p.T = T;
  p.D = D;
  p.n_t = F / TWELL_TILE;
  p.W = h->cap;
  p.status = status_dev;
  p.n_rows = h->n_ell;
  p.ell_rows = h->ell_rows;
  p.u_save = u_ell;
  if ((st = launch_fused(p, dev, s, true)) != TWELL_OK) return st;
  if (h->max_dense == 0) return TWELL_OK;

  // dense overflow rows
  return dense_rows_fwd(x, h, Wu_t, Wd, D, y, U_dense, static_cast<uint8_t*>(ws), L,
                        status_dev, dev, s);
}
