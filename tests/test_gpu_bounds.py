"""The bounds-checking build (libtwell_bounds.so, compiled with
-DTWELL_BOUNDS_CHECK): every data-dependent index the kernels gather from or
scatter to (neurons read from TwELL and ELL columns, counts used as loop
bounds, spill slots, row maps, per-neuron record offsets, union positions)
is range-checked and an index outside its buffer sets TWELL_FLAG_BOUNDS
instead of being used.  This stands in for a memory checker on this pool.

The small parity cases of the inference and training paths (the one-kernel
decode forward among them) run through that
build: no index falls outside its buffer (the flag stays clear) and every
result equals the normal build's (bit for bit where the kernels are
deterministic, to fp32 rounding where they add with atomics).  One TwELL
whose column names a neuron past d_ff is then fed to the checking build only:
the flag is set and the access is redirected, never made."""
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import workloads
from _gpu import ensure_built, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import os
    if torch.cuda.is_available() and not os.path.exists(tw.BOUNDS_LIB_PATH):
        from activation_sparse_gated_gate_gb300 import build
        build.build(variants=("bounds",))


def _inference(w, d, spill_cap=None):
    h = tw.TwELL(w.T, w.F, w.width, spill_cap=spill_cap)
    z = torch.empty((w.T, w.F), dtype=torch.float32, device="cuda")
    tw.twell_gate_pack(d["x"], d["Wg_t"], h, z_debug=z)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    # the tensor-core forwards take d_model in multiples of 64
    tc = w.D % 64 == 0
    y_tc = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"]) if tc else y
    y_tcs = tw.twell_ffn_fwd_tc_sorted(d["x"], h, d["Wu_t"], d["Wd"]) if tc else y
    # the one-kernel decode forward (decode batches; its own TwELL)
    dec = w.T <= 256 and w.D > 64
    hd = tw.TwELL(w.T, w.F, w.width, spill_cap=spill_cap)
    y_dec = tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], hd) if dec else y
    torch.cuda.synchronize()
    if dec:
        assert int(hd.status.item()) & tw.FLAG_BOUNDS == 0
    return h, z, y, (y_tc, y_tcs), y_dec


def _slots(h):
    cnt = h.cnt.long()
    used = torch.arange(h.width, device="cuda")[None, None, :] < torch.clamp(
        cnt, max=h.width)[:, :, None]
    return cnt, torch.where(used, h.col.long(), -1), torch.where(used, h.val, 0.0)


@pytest.mark.parametrize("T,D,F,p,W,cap", [
    (77, 72, 384, 0.10, 8, None),      # decode-size gate kernel, ragged D
    (300, 512, 2048, 0.02, 8, None),   # batch gate kernel
    (200, 128, 1024, 0.50, 8, None),   # heavy spilling
    (64, 128, 1024, 0.50, 8, 4),       # spill list exhausted (its own flag only)
])
def test_inference_under_bounds_checks(T, D, F, p, W, cap):
    w = workloads.random_small(T, D, F, p, W, seed=T + 7)
    d = upload(w)
    h0, z0, y0, yt0, yd0 = _inference(w, d, cap)
    s0 = int(h0.status.item())
    with tw.library(tw.BOUNDS_LIB_PATH):
        h1, z1, y1, yt1, yd1 = _inference(w, d, cap)
    s1 = int(h1.status.item())
    assert s1 & tw.FLAG_BOUNDS == 0
    assert s1 == s0
    torch.testing.assert_close(z1, z0, rtol=0, atol=0)
    for a, b in zip(_slots(h1), _slots(h0)):
        torch.testing.assert_close(a, b, rtol=0, atol=0)
    torch.testing.assert_close(h1.block_bits, h0.block_bits, rtol=0, atol=0)
    if s0 != 0:
        # a full spill list: which slices got a slot depends on the order of
        # atomics, and the rows without one are undefined, so y is not compared
        return
    # the decode forward adds rows with atomics in any order (up to F terms
    # per element): equal to fp32 rounding of the largest terms
    torch.testing.assert_close(yd1, yd0, rtol=1e-5, atol=1e-5 * float(yd0.abs().max()))
    # few-row calls split rows over warps and add partial sums with atomics
    torch.testing.assert_close(y1, y0, rtol=1e-5, atol=1e-6)
    if w.D % 64 == 0:
        for a, b in zip(yt1, yt0):
            torch.testing.assert_close(a, b, rtol=0, atol=0)


def _training(w, d, tc):
    h = tw.TwELL(w.T, w.F, w.width)
    tw.twell_gate_pack(d["x"], d["Wg_t"], h)
    hyb = tw.Hybrid(w.T, w.F, w.cap, 256)
    tw.twell_to_hybrid(h, hyb)
    fwd, bwd = ((tw.hybrid_ffn_fwd_tc, tw.hybrid_ffn_bwd_tc) if tc
                else (tw.hybrid_ffn_fwd, tw.hybrid_ffn_bwd))
    y, u_ell, U_dense = fwd(d["x"], hyb, d["Wu_t"], d["Wd"])
    dy = torch.from_numpy(w.dy).cuda()
    grads = bwd(d["x"], hyb, u_ell, U_dense, d["Wg_t"], d["Wu_t"], d["Wd"], dy, w.l1_coeff)
    torch.cuda.synchronize()
    return h, hyb, y, grads


@pytest.mark.parametrize("tc", [False, True])
def test_training_under_bounds_checks(tc):
    w = workloads.make_training("bounds-checked training", 1000, 256, 2048, 0.05, 0.03, 0.4, 16,
                                2e-5, seed=12)
    d = upload(w)
    h0, hyb0, y0, g0 = _training(w, d, tc)
    with tw.library(tw.BOUNDS_LIB_PATH):
        h1, hyb1, y1, g1 = _training(w, d, tc)
    for st in (h1.status, hyb1.status):
        assert int(st.item()) & tw.FLAG_BOUNDS == 0
    assert int(hyb1.status.item()) == int(hyb0.status.item()) == 0
    assert hyb1.n_dense == hyb0.n_dense > 0
    n_ell = hyb0.n_ell
    assert hyb1.n_ell == n_ell
    torch.testing.assert_close(hyb1.ell_cnt[:n_ell], hyb0.ell_cnt[:n_ell], rtol=0, atol=0)
    torch.testing.assert_close(hyb1.row_map, hyb0.row_map, rtol=0, atol=0)
    # dense rows and weight gradients sum with atomics: equal to fp32 rounding
    torch.testing.assert_close(y1, y0, rtol=1e-5, atol=1e-6)
    for a, b in zip(g1, g0):
        scale = float(b.abs().max())
        torch.testing.assert_close(a, b, rtol=1e-4, atol=1e-5 * scale)


def test_column_past_d_ff_is_caught():
    # A valid TwELL, then one (row, tile) of the last tile rewritten to hold a
    # single entry whose column (0xFF) names neuron F + 127.  Only the
    # checking build sees it: the fused kernel flags TWELL_FLAG_BOUNDS and
    # gathers row 0 in its place.
    w = workloads.random_small(64, 256, 1024, 0.02, 8, seed=3)
    d = upload(w)
    with tw.library(tw.BOUNDS_LIB_PATH):
        h = tw.TwELL(w.T, w.F, w.width)
        tw.twell_gate_pack(d["x"], d["Wg_t"], h)
        torch.cuda.synchronize()
        assert int(h.status.item()) == 0
        k = w.F // 128 - 1
        h.cnt[5, k] = 1
        h.col[5, k, 0] = 0xFF
        h.val[5, k, 0] = 1.0
        tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
        torch.cuda.synchronize()
        assert int(h.status.item()) & tw.FLAG_BOUNDS


def test_undefined_column_stays_in_tile_in_the_normal_build():
    # The normal build reads a column byte as its low seven bits, so a TwELL
    # left undefined (a gate call whose wait ran out) cannot name a neuron
    # outside its tile: the column 0xFF of the last tile acts as 127 (neuron
    # F - 1) in both forwards, exactly as a stored 127 does.
    w = workloads.random_small(64, 256, 1024, 0.02, 8, seed=3)
    d = upload(w)
    ys = []
    for colbyte in (0xFF, 0x7F):
        h = tw.TwELL(w.T, w.F, w.width)
        tw.twell_gate_pack(d["x"], d["Wg_t"], h)
        torch.cuda.synchronize()
        k = w.F // 128 - 1
        h.cnt[5, k] = 1
        h.col[5, k, 0] = colbyte
        h.val[5, k, 0] = 1.0
        ys.append((tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"]),
                   tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])))
        torch.cuda.synchronize()
        assert int(h.status.item()) == 0
    (a_cc, a_tc), (b_cc, b_tc) = ys
    torch.testing.assert_close(a_cc, b_cc, rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(a_tc, b_tc, rtol=0, atol=0)
