"""Pins of the oracle's training-step gradients: a hand-worked example,
central finite differences of the loss, and the L1 closed form."""
import numpy as np
import pytest

import oracle
import workloads
from _golden import bf16_bits, load


def test_backward_hand_example():
    g = load("ffn_tiny.json")
    x, Wg, Wu, Wd = (bf16_bits(g[k]) for k in ("x", "Wg_t", "Wu_t", "Wd"))
    dx, dg, du, dd = oracle.ffn_backward(x, Wg, Wu, Wd, np.array(g["dy"], float), g["l1_coeff"])
    np.testing.assert_array_equal(dx, np.array(g["dx"], float))
    np.testing.assert_array_equal(dg, np.array(g["dWg_t"], float))
    np.testing.assert_array_equal(du, np.array(g["dWu_t"], float))
    np.testing.assert_array_equal(dd, np.array(g["dWd"], float))
    X, G, U, Dn = (oracle.bf16_to_f64(a) for a in (x, Wg, Wu, Wd))
    assert oracle.training_loss(X, G, U, Dn, np.array(g["dy"], float), g["l1_coeff"]) == g["loss"]


def _fd_case(seed, T=3, D=4, F=6, margin=1e-3):
    rng = np.random.default_rng(seed)
    while True:
        X = rng.standard_normal((T, D))
        G = rng.standard_normal((F, D))
        if np.min(np.abs(X @ G.T)) > margin * 50:
            break
    U = rng.standard_normal((F, D))
    Dn = rng.standard_normal((F, D))
    dY = rng.standard_normal((T, D))
    return X, G, U, Dn, dY


@pytest.mark.parametrize("seed,lam", [(0, 0.0), (1, 2e-5), (2, 0.7), (3, 1.0)])
def test_backward_finite_differences(seed, lam):
    X, G, U, Dn, dY = _fd_case(seed)
    grads = oracle.ffn_backward_f64(X, G, U, Dn, dY, lam)
    args = [X, G, U, Dn]
    eps = 1e-6
    for which in range(4):
        num = np.zeros_like(args[which])
        for idx in np.ndindex(args[which].shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (oracle.training_loss(*plus, dY, lam)
                        - oracle.training_loss(*minus, dY, lam)) / (2 * eps)
        np.testing.assert_allclose(grads[which], num, rtol=1e-6, atol=1e-7,
                                   err_msg=f"grad {which}")


def test_l1_closed_form_with_zero_dy():
    # dy = 0: only the L1 term acts.  dx_t = lam * sum_j [z_tj > 0] W_g[:, j],
    # dW_g[:, j] = lam * sum_t [z_tj > 0] x_t, dW_u = dW_d = 0
    w = workloads.random_small(6, 64, 256, 0.1, 8, seed=21)
    X, G = oracle.bf16_to_f64(w.x), oracle.bf16_to_f64(w.Wg_t)
    act = (X @ G.T) > 0
    for lam in (2e-5, 1.0):
        dx, dg, du, dd = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd,
                                             np.zeros((6, 64)), lam)
        for t in range(6):
            np.testing.assert_allclose(dx[t], lam * G[act[t]].sum(0), rtol=1e-12, atol=1e-15)
        for j in range(256):
            np.testing.assert_allclose(dg[j], lam * X[act[:, j]].sum(0), rtol=1e-12,
                                       atol=1e-15)
        assert not du.any() and not dd.any()


def test_restrictions_match_full():
    w = workloads.random_small(10, 64, 256, 0.1, 8, seed=22, dy=True, l1_coeff=0.3)
    full = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 0.3)
    rows = [1, 4, 9]
    np.testing.assert_allclose(
        oracle.ffn_backward_dx_rows(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 0.3, rows),
        full[0][rows], rtol=1e-12, atol=1e-14)
    nz = [0, 7, 100, 255]
    dg, du, dd = oracle.ffn_backward_dw_cols(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 0.3, nz)
    np.testing.assert_allclose(dg, full[1][nz], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(du, full[2][nz], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dd, full[3][nz], rtol=1e-12, atol=1e-14)


def test_inactive_entries_get_no_gradient():
    # a neuron that is never active has zero dW_g, dW_u, dW_d rows
    w = workloads.random_small(8, 64, 256, 0.1, 8, seed=23, dy=True, l1_coeff=0.5)
    act = oracle.gate_preact(w.x, w.Wg_t) > 0
    dead = np.nonzero(~act.any(axis=0))[0]
    assert len(dead) > 0
    _, dg, du, dd = oracle.ffn_backward(w.x, w.Wg_t, w.Wu_t, w.Wd, w.dy, 0.5)
    assert not dg[dead].any() and not du[dead].any() and not dd[dead].any()


def test_stack_chain_rule_finite_differences():
    # two residual layers without stream rounding: the chained gradients of
    # stack_forward_backward match central differences of the stack's loss
    rng = np.random.default_rng(21)
    T, D, F = 3, 8, 16

    def bits(a):
        return oracle.f32_to_bf16(a.astype(np.float32))

    x = bits(rng.standard_normal((T, D)))
    layers = [tuple(bits(rng.standard_normal((F, D)) * 0.4) for _ in range(3)) for _ in range(2)]
    dy = rng.standard_normal((T, D))
    lam = 0.05
    out, dx0, grads = oracle.stack_forward_backward(x, layers, dy, lam, round_inputs=False)
    ws = [[oracle.bf16_to_f64(w) for w in layer] for layer in layers]

    def loss(X0, ws):
        X = X0
        total = 0.0
        for G, U, Dn in ws:
            z = X @ G.T
            total += lam * np.sum(np.where(z > 0, z, 0.0))
            y = oracle.ffn_forward_f64(X, G, U, Dn)
            y[:, -1] = 0.0
            X = X + y
        return total + float(np.sum(X * dy))

    X0 = oracle.bf16_to_f64(x)
    eps = 1e-6
    for (t, d) in [(0, 0), (1, 3), (2, 7)]:
        Xp, Xm = X0.copy(), X0.copy()
        Xp[t, d] += eps
        Xm[t, d] -= eps
        fd = (loss(Xp, ws) - loss(Xm, ws)) / (2 * eps)
        assert abs(fd - dx0[t, d]) <= 1e-5 * max(1.0, abs(fd))
    for l in range(2):
        for k in range(3):
            for (j, d) in [(0, 0), (5, 2), (15, 7)]:
                wp = [list(w) for w in ws]
                wm = [list(w) for w in ws]
                wp[l][k] = ws[l][k].copy()
                wm[l][k] = ws[l][k].copy()
                wp[l][k][j, d] += eps
                wm[l][k][j, d] -= eps
                fd = (loss(X0, wp) - loss(X0, wm)) / (2 * eps)
                assert abs(fd - grads[l][k][j, d]) <= 1e-5 * max(1.0, abs(fd)), (l, k, j, d)


def test_stack_rounded_inputs_straight_through_finite_differences():
    # round_inputs=True (the default): each layer input is the stream rounded
    # to bf16 and the backward passes through the rounding as the identity.
    # Pin: freeze each layer's rounding offset c_l = bf16(x_l) - x_l at the
    # base point (bf16 by torch's CPU conversion, not the oracle's), so the
    # layer input is x_l + c_l.  That surrogate equals the rounded stack at
    # the base point and its exact gradient is the straight-through one, so
    # the oracle's forward matches it there and its gradients match central
    # differences of it.
    import torch
    rng = np.random.default_rng(31)
    T, D, F = 4, 8, 16

    def bits(a):
        return oracle.f32_to_bf16(a.astype(np.float32))

    x = bits(rng.standard_normal((T, D)))
    layers = [tuple(bits(rng.standard_normal((F, D)) * 0.4) for _ in range(3))
              for _ in range(3)]
    dy = rng.standard_normal((T, D))
    lam = 0.05
    out, dx0, grads = oracle.stack_forward_backward(x, layers, dy, lam)
    ws = [[oracle.bf16_to_f64(w) for w in layer] for layer in layers]
    X0 = oracle.bf16_to_f64(x)

    def torch_bf16(a):
        return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(
            torch.float64).numpy()

    # offsets at the base point
    offs = []
    X = X0
    for G, U, Dn in ws:
        offs.append(torch_bf16(X) - X)
        y = oracle.ffn_forward_f64(X + offs[-1], G, U, Dn)
        y[:, -1] = 0.0
        X = X + y
    assert np.abs(X - out).max() <= 1e-12 * max(1.0, np.abs(out).max())
    # at least one layer input really was rounded
    assert max(np.abs(c).max() for c in offs[1:]) > 0

    def loss(X0, ws):
        X = X0
        total = 0.0
        for (G, U, Dn), c in zip(ws, offs):
            A = X + c
            z = A @ G.T
            total += lam * np.sum(np.where(z > 0, z, 0.0))
            y = oracle.ffn_forward_f64(A, G, U, Dn)
            y[:, -1] = 0.0
            X = X + y
        return total + float(np.sum(X * dy))

    eps = 1e-6
    for (t, d) in [(0, 0), (1, 3), (3, 6)]:
        Xp, Xm = X0.copy(), X0.copy()
        Xp[t, d] += eps
        Xm[t, d] -= eps
        fd = (loss(Xp, ws) - loss(Xm, ws)) / (2 * eps)
        assert abs(fd - dx0[t, d]) <= 1e-5 * max(1.0, abs(fd))
    for l in range(3):
        for k in range(3):
            for (j, d) in [(0, 0), (7, 2), (15, 6)]:
                wp = [list(w) for w in ws]
                wm = [list(w) for w in ws]
                wp[l][k] = ws[l][k].copy()
                wm[l][k] = ws[l][k].copy()
                wp[l][k][j, d] += eps
                wm[l][k][j, d] -= eps
                fd = (loss(X0, wp) - loss(X0, wm)) / (2 * eps)
                assert abs(fd - grads[l][k][j, d]) <= 1e-5 * max(1.0, abs(fd)), (l, k, j, d)
