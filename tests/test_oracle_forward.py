"""Pins of the oracle's gated-FFN forward: a hand-worked example, brute
force scalar loops, the dense == sparse identity, and closed forms."""
import numpy as np
import pytest

import oracle
import workloads
from _golden import bf16_bits, load


def test_forward_hand_example():
    g = load("ffn_tiny.json")
    x, Wg, Wu, Wd = (bf16_bits(g[k]) for k in ("x", "Wg_t", "Wu_t", "Wd"))
    np.testing.assert_array_equal(oracle.gate_preact(x, Wg), np.array(g["z"], float))
    np.testing.assert_array_equal(oracle.ffn_forward(x, Wg, Wu, Wd), np.array(g["y"], float))
    np.testing.assert_array_equal(oracle.ffn_forward_sparse(x, Wg, Wu, Wd),
                                  np.array(g["y"], float))


def _brute(x, Wg, Wu, Wd):
    X, G, U, Dn = (oracle.bf16_to_f64(a) for a in (x, Wg, Wu, Wd))
    T, D = X.shape
    F = G.shape[0]
    y = np.zeros((T, D))
    for t in range(T):
        for j in range(F):
            z = 0.0
            u = 0.0
            for i in range(D):
                z += X[t, i] * G[j, i]
                u += X[t, i] * U[j, i]
            if z > 0:
                for d in range(D):
                    y[t, d] += z * u * Dn[j, d]
    return y


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_forward_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    T, D, F = 3, 5, 7
    x = workloads.to_bf16(rng.standard_normal((T, D)))
    Wg, Wu, Wd = (workloads.to_bf16(rng.standard_normal((F, D))) for _ in range(3))
    np.testing.assert_allclose(oracle.ffn_forward(x, Wg, Wu, Wd), _brute(x, Wg, Wu, Wd),
                               rtol=1e-12, atol=1e-12)


def test_dense_equals_sparse():
    w = workloads.random_small(9, 64, 256, 0.1, 8, seed=3)
    yd = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd)
    ys = oracle.ffn_forward_sparse(w.x, w.Wg_t, w.Wu_t, w.Wd)
    assert np.max(np.abs(yd - ys)) <= 1e-12 * max(1.0, np.max(np.abs(yd)))


def test_zero_active_gives_zero():
    w = workloads.make_uniform("none", 6, 64, 256, 1e-12, 8, seed=4)
    assert (oracle.gate_preact(w.x, w.Wg_t) <= 0).all()
    assert not oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd).any()


def test_all_active_is_bilinear_form():
    # every z > 0: ReLU is the identity and y_t = sum_j z_tj u_tj W_d[j]
    rng = np.random.default_rng(6)
    T, D, F = 4, 8, 16
    x = workloads.to_bf16(np.abs(rng.standard_normal((T, D))) + 0.1)
    Wg = workloads.to_bf16(np.abs(rng.standard_normal((F, D))) + 0.1)
    Wu = workloads.to_bf16(rng.standard_normal((F, D)))
    Wd = workloads.to_bf16(rng.standard_normal((F, D)))
    X, G, U, Dn = (oracle.bf16_to_f64(a) for a in (x, Wg, Wu, Wd))
    assert (X @ G.T > 0).all()
    # computed through the scalar identity y = sum_j (x.g_j)(x.u_j) d_j
    ref = np.zeros((T, D))
    for t in range(T):
        for j in range(F):
            ref[t] += np.dot(X[t], G[j]) * np.dot(X[t], U[j]) * Dn[j]
    np.testing.assert_allclose(oracle.ffn_forward(x, Wg, Wu, Wd), ref, rtol=1e-12, atol=1e-12)


def test_single_active_neuron_closed_form():
    # x_t = e_t (one-hot) makes z_tj = Wg_t[j, t]; only neuron j=t has a
    # positive gate entry in column t, so y_t = Wg_t[t,t] * Wu_t[t,t] * Wd[t]
    T, D, F = 4, 4, 8
    X = np.eye(T, D)
    G = -np.ones((F, D))
    for t in range(T):
        G[t, t] = 0.5 * (t + 1)
    rng = np.random.default_rng(7)
    U = np.round(rng.standard_normal((F, D)) * 8) / 8
    Dn = np.round(rng.standard_normal((F, D)) * 8) / 8
    x, Wg, Wu, Wd = (workloads.to_bf16(a) for a in (X, G, U, Dn))
    y = oracle.ffn_forward(x, Wg, Wu, Wd)
    for t in range(T):
        np.testing.assert_array_equal(y[t], G[t, t] * U[t, t] * Dn[t])


def test_forward_rows_is_row_restriction():
    w = workloads.random_small(10, 64, 256, 0.05, 8, seed=8)
    full = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd)
    rows = [0, 3, 9]
    np.testing.assert_array_equal(oracle.ffn_forward_rows(w.x, w.Wg_t, w.Wu_t, w.Wd, rows),
                                  full[rows])


def test_active_override():
    w = workloads.random_small(5, 64, 256, 0.2, 8, seed=9)
    z = oracle.gate_preact(w.x, w.Wg_t)
    act = z > 0
    np.testing.assert_array_equal(oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd, active=act),
                                  oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd))
    none = np.zeros_like(act)
    assert not oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd, active=none).any()
