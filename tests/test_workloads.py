"""The seeded synthetic inputs reach the densities their recipe states."""
import numpy as np
import pytest

import oracle
import workloads


@pytest.mark.parametrize("idx,T,target,tol", [
    (0, 64, 0.05, 0.01),
    (1, 256, 0.01, 0.0015),
    (2, 512, 0.01, 0.003),
    (4, 256, 0.005, 0.001),
])
def test_density(idx, T, target, tol):
    w = workloads.config(idx, T=T)
    z = oracle.gate_preact(w.x, w.Wg_t)
    assert abs((z > 0).mean() - target) < tol


def test_training_rows():
    w = workloads.config(3, T=1024)
    z = oracle.gate_preact(w.x, w.Wg_t)
    dens = (z > 0).mean(axis=1)
    heavy = dens > 0.2
    assert abs(heavy.sum() - round(0.03 * 1024)) <= 0
    assert abs(dens.mean() - 0.05) < 0.004
    tw = oracle.twell_pack(z.astype(np.float32), 128, 32)
    over = (tw.cnt > 32).any(axis=1)
    np.testing.assert_array_equal(over, heavy)
    assert w.dy.shape == (1024, 2304) and w.dy.dtype == np.float32


def test_prefix_nesting_and_determinism():
    a = workloads.config(4, T=4)
    b = workloads.config(4, T=16)
    np.testing.assert_array_equal(a.x, b.x[:4])
    np.testing.assert_array_equal(a.Wg_t, b.Wg_t)
    c = workloads.config(4, T=16)
    np.testing.assert_array_equal(b.x, c.x)
