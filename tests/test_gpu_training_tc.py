"""GPU parity of the tensor-core variants of the hybrid training forward and
backward (hybrid_ffn_fwd_tc / hybrid_ffn_bwd_tc) through the C-ABI, against
the dense fp64 oracle.

Bars: the spec bar, max-abs <= 2e-2 * RMS(reference) per tensor, and
a statistical bug-catching bar, RMS(error) <= 5e-3 * RMS(reference).  The
variant feeds the sparse values (h u, dz, du), the weights, x and dy to the
tensor cores as fp16 (dy, dz and du multiplied by a power-of-two gradient
scale), each with a relative rounding error below 2^-11, so a product of a
few such factors summed over many independent terms has an error RMS well
below 1e-3 of the result's RMS; a wrong index, sign, scale or dropped term
gives errors of the order of the RMS itself."""
import numpy as np
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import oracle
import workloads
from _gpu import assert_ns_tol, ensure_built, rms, run_pack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _bars(got, ref, names, scales=None, stat=5e-3):
    for i, (g, r, n) in enumerate(zip(got, ref, names)):
        scale = rms(r) if scales is None else scales[i]
        err = float(np.max(np.abs(g - r)))
        assert err <= 2e-2 * scale, f"{n}: max-abs {err:.3e} > 2e-2*RMS {2e-2 * scale:.3e}"
        e_rms = rms(g - r)
        assert e_rms <= stat * scale, f"{n}: error RMS {e_rms:.3e} > {stat}*RMS"


def _training(T, D, F, p, frac, pd, cap, seed=0):
    return workloads.make_training(f"train {T}x{D}x{F}", T, D, F, p, frac, pd, cap,
                                   2e-5, seed=seed)


def _hybrid(w, max_dense):
    d, h, z = run_pack(w)
    hyb = tw.Hybrid(w.T, w.F, w.cap, max_dense)
    tw.twell_to_hybrid(h, hyb)
    torch.cuda.synchronize()
    return d, h, hyb, z


def _run(w, max_dense, l1, dy=None, bwd=True):
    d, h, hyb, z = _hybrid(w, max_dense)
    y, u_ell, U_dense = tw.hybrid_ffn_fwd_tc(d["x"], hyb, d["Wu_t"], d["Wd"])
    grads = None
    if bwd:
        dyt = torch.from_numpy(w.dy if dy is None else dy).cuda()
        grads = tw.hybrid_ffn_bwd_tc(d["x"], hyb, u_ell, U_dense, d["Wg_t"], d["Wu_t"],
                                     d["Wd"], dyt, l1)
    torch.cuda.synchronize()
    assert int(hyb.status.item()) == 0
    zg = z.cpu().numpy()
    out = {"y": y, "u_ell": u_ell, "U_dense": U_dense, "hyb": hyb, "zg": zg, "d": d}
    if grads is not None:
        out["grads"] = [g.cpu().numpy().astype(np.float64) for g in grads]
    return out


TC_SMALL = [
    # T, D, F, mean density, dense fraction, dense density, C, max_dense
    (512, 128, 1024, 0.05, 0.05, 0.4, 16, 512),
    (1000, 256, 2048, 0.05, 0.03, 0.4, 32, 256),   # ragged T, several row tiles
    (700, 320, 1152, 0.06, 0.0, 0.4, 32, 64),      # no dense rows; D not a multiple of 256
    (300, 64, 384, 0.08, 0.10, 0.5, 16, 300),      # odd tile count, one K block
]
NAMES = ("dx", "dWg_t", "dWu_t", "dWd")


@pytest.mark.parametrize("T,D,F,p,frac,pd,cap,md", TC_SMALL)
def test_tc_fwd_parity(T, D, F, p, frac, pd, cap, md):
    w = _training(T, D, F, p, frac, pd, cap, seed=T + 1)
    r = _run(w, md, 2e-5, bwd=False)
    act = r["zg"] > 0
    y_ref = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd, active=act)
    y = r["y"].cpu().numpy().astype(np.float64)
    _bars([y], [y_ref], ("y",))
    # u at the ELL entries: fp32 accumulation of exact bf16 products
    hyb = r["hyb"]
    n_ell = hyb.n_ell
    if n_ell:
        X = oracle.bf16_to_f64(w.x)
        U = oracle.bf16_to_f64(w.Wu_t)
        rows = hyb.ell_rows[:n_ell].cpu().numpy()
        cnt = hyb.ell_cnt[:n_ell].cpu().numpy().astype(np.int64)
        col = hyb.ell_col[:n_ell].cpu().numpy().astype(np.int64)
        ue = r["u_ell"][:n_ell].cpu().numpy().astype(np.float64)
        for i in range(0, n_ell, max(1, n_ell // 64)):
            ks, ss = np.nonzero(np.arange(hyb.cap)[None, :] < cnt[i][:, None])
            js = ks * 128 + col[i, ks, ss]
            uref = U[js] @ X[rows[i]]
            bound = w.D * 2.0 ** -24 * (np.abs(U[js]) @ np.abs(X[rows[i]])) + 1e-30
            assert (np.abs(ue[i, ks, ss] - uref) <= bound).all(), f"u at ELL row {i}"


@pytest.mark.parametrize("T,D,F,p,frac,pd,cap,md", TC_SMALL)
def test_tc_bwd_parity(T, D, F, p, frac, pd, cap, md):
    w = _training(T, D, F, p, frac, pd, cap, seed=T + 2)
    r = _run(w, md, 2e-5)
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 2e-5, active=r["zg"] > 0)
    _bars(r["grads"], ref, NAMES)


def test_tc_all_rows_dense():
    # every row overflows C: no ELL rows, the weight-gradient tiles have an
    # empty K range and must come out as the dense rows' terms alone
    w = _training(256, 128, 512, 0.5, 0.0, 0.5, 16, seed=5)
    r = _run(w, 256, 2e-5)
    assert r["hyb"].n_ell == 0 and r["hyb"].n_dense == 256
    act = r["zg"] > 0
    y_ref = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd, active=act)
    assert_ns_tol(r["y"].cpu().numpy().astype(np.float64), y_ref, "y")
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 2e-5, active=act)
    _bars(r["grads"], ref, NAMES)


@pytest.mark.parametrize("lam", [2e-5, 1.0])
def test_tc_l1_term_alone(lam):
    # dy = 0: da = 0, so dz = lambda exactly and du = 0 at every active
    # entry: dx_t = lambda sum_{active j} W_g[:, j], dW_g^T[j] = lambda
    # sum_{active t} x_t.  The ELL rows carry fp16(s lambda) (one relative
    # rounding <= 2^-11 shared by every term; s a power of two) and fp16
    # copies of W_g and x (exact for magnitudes >= 2^-14, else an absolute
    # error <= 2^-25), the dense rows bf16 hi + lo halves, and fp32 sums add
    # at most about 2^-15 relative over these term counts, so |err| <= 2^-10
    # lambda sum |terms| + 2^-24 lambda (number of terms) elementwise (ELL
    # and dense-row terms may cancel in the reference); dW_u = dW_d = 0
    # exactly
    w = _training(400, 128, 1024, 0.05, 0.05, 0.4, 16, seed=11)
    r = _run(w, 400, lam, dy=np.zeros_like(w.dy))
    got = r["grads"]
    act = (r["zg"] > 0).astype(np.float64)
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, np.zeros_like(w.dy), lam,
                              active=act > 0)
    X = oracle.bf16_to_f64(w.x)
    G = oracle.bf16_to_f64(w.Wg_t)
    bounds = (2.0 ** -10 * lam * (act @ np.abs(G)) + 2.0 ** -24 * lam * act.sum(1)[:, None],
              2.0 ** -10 * lam * (act.T @ np.abs(X)) + 2.0 ** -24 * lam * act.sum(0)[:, None])
    for g, rf, b, n in zip(got[:2], ref[:2], bounds, NAMES[:2]):
        err = np.abs(g - rf)
        assert (err <= b + 1e-5 * np.max(np.abs(rf))).all(), n
    assert np.abs(got[0]).max() > 0
    assert not got[2].any() and not got[3].any()


def test_tc_lambda_zero_is_plain_gradient():
    w = _training(300, 128, 1024, 0.05, 0.05, 0.4, 16, seed=12)
    r = _run(w, 300, 0.0)
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 0.0, active=r["zg"] > 0)
    _bars(r["grads"], ref, NAMES)


def test_tc_agrees_with_cuda_core_path():
    # both entry points on the same hybrid: same dense rows (identical
    # code), ELL rows within the fp16 operand rounding of each other
    w = _training(600, 256, 1024, 0.05, 0.03, 0.4, 32, seed=13)
    d, h, hyb, z = _hybrid(w, 128)
    dyt = torch.from_numpy(w.dy).cuda()
    outs = []
    for fwd, bwd in ((tw.hybrid_ffn_fwd, tw.hybrid_ffn_bwd),
                     (tw.hybrid_ffn_fwd_tc, tw.hybrid_ffn_bwd_tc)):
        y, u_ell, U_dense = fwd(d["x"], hyb, d["Wu_t"], d["Wd"])
        g = bwd(d["x"], hyb, u_ell, U_dense, d["Wg_t"], d["Wu_t"], d["Wd"], dyt, 2e-5)
        torch.cuda.synchronize()
        outs.append([t.cpu().numpy().astype(np.float64) for t in (y, u_ell, *g)])
    n_ell = hyb.n_ell
    cnt = hyb.ell_cnt[:n_ell].cpu().numpy()
    used = np.arange(hyb.cap)[None, None, :] < cnt[:, :, None]
    ua, ub = outs[0][1][:n_ell], outs[1][1][:n_ell]
    assert np.max(np.abs(np.where(used, ua - ub, 0))) <= 1e-4 * np.max(np.abs(ua))
    dense = hyb.dense_rows[:hyb.n_dense].cpu().numpy()
    np.testing.assert_allclose(outs[1][0][dense], outs[0][0][dense], rtol=1e-5, atol=1e-5)
    for a, b, n in zip(outs[0][2:], outs[1][2:], NAMES):
        assert rms(a - b) <= 5e-3 * rms(a), n


@pytest.mark.parametrize("c,lam", [(1e-12, 0.0), (1e-12, 2e-17), (1e-10, 2e-5), (1e3, 2e-5)])
def test_tc_gradient_scale(c, lam):
    # dy far below fp16's normal range (a loss averaged over many tokens),
    # far above it (where unscaled dz = da u + lambda would overflow fp16),
    # or far below the L1 coefficient (the scale then follows 2^-14 lambda
    # and dy scales to below [0.5, 1)): the power-of-two scale keeps every
    # fp16 operand in range, so the same bars hold for every gradient,
    # including dW_u and dW_d, which depend on dy alone
    w = _training(500, 128, 1024, 0.05, 0.05, 0.4, 16, seed=14)
    dy = (w.dy.astype(np.float64) * c).astype(np.float32)
    r = _run(w, 128, lam, dy=dy)
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, dy, lam, active=r["zg"] > 0)
    _bars(r["grads"], ref, NAMES)


def _random_cases(n, seed=2026):
    # seeded shapes: ragged T, D a multiple of 64, any tile count, both
    # capacities, with and without dense rows, three L1 coefficients and dy
    # spread over 15 decades (the gradient scale's range)
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        c = dict(T=int(rng.integers(64, 2600)), D=int(rng.choice([64, 128, 192, 256, 320, 512])),
                 F=128 * int(rng.integers(2, 17)), C=int(rng.choice([16, 32])),
                 p=float(rng.uniform(0.02, 0.09)), frac=float(rng.choice([0.0, 0.02, 0.08])),
                 pd=float(rng.uniform(0.35, 0.5)), lam=float(rng.choice([0.0, 2e-5, 1e-3])),
                 sc=float(10 ** rng.uniform(-12, 3)), seed=len(out) + 100)
        try:
            workloads.make_training("check", c["T"], c["D"], c["F"], c["p"], c["frac"], c["pd"],
                                    c["C"], c["lam"], seed=c["seed"])
        except ValueError:  # no base density gives the mean
            continue
        out.append(c)
    return out


@pytest.mark.parametrize("c", _random_cases(6), ids=lambda c: f"T{c['T']}D{c['D']}F{c['F']}C{c['C']}")
def test_tc_random_shapes(c):
    w = workloads.make_training("check", c["T"], c["D"], c["F"], c["p"], c["frac"], c["pd"],
                                c["C"], c["lam"], seed=c["seed"])
    dy = (w.dy.astype(np.float64) * c["sc"]).astype(np.float32)
    r = _run(w, w.T, c["lam"], dy=dy)
    act = r["zg"] > 0
    y_ref = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd, active=act)
    _bars([r["y"].cpu().numpy().astype(np.float64)], [y_ref], ("y",))
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, dy, c["lam"], active=act)
    _bars(r["grads"], ref, NAMES)


def test_tc_fp16_range_flag():
    # x multiplied by 2^20: u and h u grow past fp16's 65504 in the forward,
    # and x itself in the backward's fp16 copy; both calls report it
    w = _training(256, 128, 512, 0.05, 0.0, 0.4, 16, seed=15)
    d, h, hyb, z = _hybrid(w, 64)
    xb = d["x"] * 2.0 ** 20
    y, u_ell, U_dense = tw.hybrid_ffn_fwd_tc(xb, hyb, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(hyb.status.item()) & tw.FLAG_RANGE
    hyb.status.zero_()
    tw.hybrid_ffn_bwd_tc(xb, hyb, u_ell, U_dense, d["Wg_t"], d["Wu_t"], d["Wd"],
                         torch.from_numpy(w.dy).cuda(), 2e-5)
    torch.cuda.synchronize()
    assert int(hyb.status.item()) & tw.FLAG_RANGE


def test_tc_unsupported_shapes():
    w = _training(128, 72, 256, 0.05, 0.0, 0.4, 16, seed=3)   # D % 64 != 0
    d, h, hyb, z = _hybrid(w, 16)
    with pytest.raises(tw.TwellError, match="UNSUPPORTED"):
        tw.hybrid_ffn_fwd_tc(d["x"], hyb, d["Wu_t"], d["Wd"])
    w = _training(128, 64, 256, 0.02, 0.0, 0.4, 8, seed=3)    # C = 8
    d, h, hyb, z = _hybrid(w, 16)
    with pytest.raises(tw.TwellError, match="UNSUPPORTED"):
        tw.hybrid_ffn_fwd_tc(d["x"], hyb, d["Wu_t"], d["Wd"])


def test_tc_training_config_reduced():
    w = workloads.config(3, T=2048)
    r = _run(w, 128, w.l1_coeff)
    act = r["zg"] > 0
    y_ref = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd, active=act)
    _bars([r["y"].cpu().numpy().astype(np.float64)], [y_ref], ("y",))
    ref = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, w.l1_coeff, active=act)
    _bars(r["grads"], ref, NAMES)


def test_tc_training_config_full_size():
    """The 2B-class training step at full size (T=16384, D=2304, F=9216,
    C=32) in the bench's launch configuration; y and dx on sampled token
    rows (dense rows among them), the weight gradients on sampled neurons.
    The max-abs bar uses each full tensor's RMS; the statistical bar the
    sample's."""
    w = workloads.config(3)
    d, h, z = run_pack(w)
    hyb = tw.Hybrid(w.T, w.F, w.cap, 1024)
    tw.twell_to_hybrid(h, hyb)
    y, u_ell, U_dense = tw.hybrid_ffn_fwd_tc(d["x"], hyb, d["Wu_t"], d["Wd"])
    dyt = torch.from_numpy(w.dy).cuda()
    grads = tw.hybrid_ffn_bwd_tc(d["x"], hyb, u_ell, U_dense, d["Wg_t"], d["Wu_t"], d["Wd"],
                                 dyt, w.l1_coeff)
    torch.cuda.synchronize()
    assert int(hyb.status.item()) == 0 and int(h.status.item()) == 0
    rng = np.random.default_rng(4)
    dense = hyb.dense_rows[:hyb.n_dense].cpu().numpy()
    rows = np.sort(np.concatenate([rng.choice(w.T, 40, replace=False), dense[:8]]))
    ridx = torch.as_tensor(rows, device="cuda")
    zr = z[ridx].cpu().numpy()
    yg = y[ridx].cpu().numpy().astype(np.float64)
    yref = oracle.ffn_forward(w.x[rows], w.Wg_t, w.Wu_t, w.Wd, active=zr > 0)
    dxg = grads[0][ridx].cpu().numpy().astype(np.float64)
    dxref = oracle.ffn_backward_dx_rows(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, w.l1_coeff, rows,
                                        active_rows=zr > 0)
    full_rms = [float(torch.sqrt((t.double() ** 2).mean())) for t in (y, grads[0])]
    for g, r_, n, s in zip((yg, dxg), (yref, dxref), ("y", "dx"), full_rms):
        assert np.max(np.abs(g - r_)) <= 2e-2 * s, n
        assert rms(g - r_) <= 5e-3 * rms(r_), n
    neurons = np.sort(rng.choice(w.F, 24, replace=False))
    nidx = torch.as_tensor(neurons, device="cuda")
    zc = z[:, nidx].cpu().numpy()
    refw = oracle.ffn_backward_dw_cols(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, w.l1_coeff, neurons,
                                       active_cols=zc > 0)
    for g, r_, n in zip(grads[1:], refw, NAMES[1:]):
        s = float(torch.sqrt((g.double() ** 2).mean()))
        gw = g[nidx].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(gw - r_)) <= 2e-2 * s, n
        assert rms(gw - r_) <= 5e-3 * rms(r_), n
