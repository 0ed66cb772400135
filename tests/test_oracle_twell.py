"""Pins of the oracle's TwELL pack/unpack and hybrid conversion: a
hand-worked fixture, scalar loops, invariants, crafted counts."""
import numpy as np
import pytest

import oracle
import workloads
from _golden import f32, load


def test_pack_hand_example():
    g = load("twell_tiny.json")
    z = f32(g["z"])
    tw = oracle.twell_pack(z, g["tile"], g["width"])
    np.testing.assert_array_equal(tw.cnt, np.array(g["cnt"]))
    for key, slots in g["slots"].items():
        t, k = map(int, key.split(","))
        for s, (c, v) in enumerate(slots):
            assert tw.col[t, k, s] == c and tw.val[t, k, s] == np.float32(v), (key, s)
    assert set(tw.spill) == {tuple(map(int, k.split(","))) for k in g["spill"]}
    for key, sl in g["spill"].items():
        np.testing.assert_array_equal(tw.spill[tuple(map(int, key.split(",")))],
                                      np.array(sl, np.float32))
    np.testing.assert_array_equal(oracle.twell_unpack(tw), np.array(g["unpacked"], np.float32))


def test_hybrid_hand_example():
    g = load("twell_tiny.json")
    tw = oracle.twell_pack(f32(g["z"]), g["tile"], g["width"])
    h2 = oracle.to_hybrid(tw, 2)
    e = g["hybrid_cap2"]
    assert list(h2.ell_rows) == e["ell_rows"] and list(h2.dense_rows) == e["dense_rows"]
    assert list(h2.row_map) == e["row_map"]
    np.testing.assert_array_equal(h2.dense_h[0], np.array(g["unpacked"][0], np.float32))
    h4 = oracle.to_hybrid(tw, 4)
    e = g["hybrid_cap4"]
    assert list(h4.ell_rows) == e["ell_rows"] and list(h4.dense_rows) == e["dense_rows"]
    assert list(h4.row_map) == e["row_map"]
    got = [[int(h4.ell_col[0, 2, s]), float(h4.ell_val[0, 2, s])] for s in range(4)]
    assert got == e["row0_tile2"]


def _z(T, F, p, seed, dtype=np.float32):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, F)) - 1.5
    return z.astype(dtype)


@pytest.mark.parametrize("width", [1, 8, 16])
def test_pack_matches_scalar_loops(width):
    z = _z(5, 512, 0.1, 11)
    z[1, 0:128] = 1.0     # a full tile
    z[2, 128:256] = -1.0  # an empty tile
    a = oracle.twell_pack(z, 128, width)
    b = oracle.twell_pack_loops(z, 128, width)
    np.testing.assert_array_equal(a.cnt, b.cnt)
    np.testing.assert_array_equal(a.col, b.col)
    np.testing.assert_array_equal(a.val, b.val)
    assert set(a.spill) == set(b.spill)
    for k in a.spill:
        np.testing.assert_array_equal(a.spill[k], b.spill[k])


@pytest.mark.parametrize("width", [8, 16, 32])
def test_pack_invariants(width):
    z = _z(40, 1024, 0.1, 12)
    z[3] += 3.0   # a dense-ish row to force spills
    tw = oracle.twell_pack(z, 128, width)
    assert tw.cnt.sum() == (z > 0).sum()
    assert (tw.cnt <= 128).all()
    for t in range(tw.T):
        for k in range(tw.n_t):
            m = min(int(tw.cnt[t, k]), width)
            cols = tw.col[t, k, :m]
            assert (np.diff(cols) > 0).all() and (cols < 128).all()
            # the slots are exactly the first m active columns of the tile
            act = np.nonzero(z[t, k * 128:(k + 1) * 128] > 0)[0]
            np.testing.assert_array_equal(cols, act[:m])
    assert set(tw.spill) == {(t, k) for t, k in zip(*np.nonzero(tw.cnt > width))}
    assert len(tw.spill) > 0
    exp = np.where(z > 0, z, np.float32(0))
    np.testing.assert_array_equal(oracle.twell_unpack(tw), exp)


def test_pack_crafted_counts():
    W = 8
    T, F = 7, 256
    z = -np.ones((T, F), np.float32)
    counts = [0, 1, W, W + 1, 32, 33, 128]
    for t, c in enumerate(counts):
        # tile 0: c actives spread over it, including its first and last
        # column once c >= 2 (c = 1 uses the last column)
        cols = np.linspace(0, 127, c).round().astype(int) if c > 1 else np.array([127] * c, dtype=int)
        assert len(np.unique(cols)) == c
        z[t, cols] = 0.5 + t
    tw = oracle.twell_pack(z, 128, W)
    np.testing.assert_array_equal(tw.cnt[:, 0], counts)
    np.testing.assert_array_equal(tw.cnt[:, 1], 0)
    assert set(tw.spill) == {(t, 0) for t, c in enumerate(counts) if c > W}
    h = oracle.to_hybrid(tw, 32)
    assert list(h.dense_rows) == [t for t, c in enumerate(counts) if c > 32]
    assert list(h.ell_rows) == [t for t, c in enumerate(counts) if c <= 32]


def test_pack_fp64_decision_precision():
    # a positive fp64 value that underflows to 0 in fp32 is still active
    z = np.full((1, 128), -1.0)
    z[0, 5] = 1e-300
    tw = oracle.twell_pack(z, 128, 8)
    assert tw.cnt[0, 0] == 1 and tw.col[0, 0, 0] == 5


@pytest.mark.parametrize("cap,width", [(32, 32), (16, 8), (8, 16)])
def test_hybrid_invariants(cap, width):
    z = _z(64, 1024, 0.05, 13) + 0.3
    z[[5, 17, 40]] += 2.0   # overflow rows
    tw = oracle.twell_pack(z, 128, width)
    h = oracle.to_hybrid(tw, cap)
    T = tw.T
    assert len(h.ell_rows) + len(h.dense_rows) == T
    assert sorted(np.concatenate([h.ell_rows, h.dense_rows]).tolist()) == list(range(T))
    assert (np.diff(h.ell_rows) > 0).all() and (np.diff(h.dense_rows) > 0).all()
    for i, t in enumerate(h.ell_rows):
        assert h.row_map[t] == i
    for i, t in enumerate(h.dense_rows):
        assert h.row_map[t] == -(i + 1)
    over = (tw.cnt > cap).any(axis=1)
    assert set(h.dense_rows) == set(np.nonzero(over)[0])
    nnz_ell = int(h.ell_cnt.sum())
    nnz_dense = int((h.dense_h > 0).sum())
    assert nnz_ell + nnz_dense == int((z > 0).sum())
    # ELL entries rebuild the same gate rows as the TwELL
    full = oracle.twell_unpack(tw)
    for i, t in enumerate(h.ell_rows):
        row = np.zeros(tw.F, np.float32)
        for k in range(tw.n_t):
            c = int(h.ell_cnt[i, k])
            row[k * 128 + h.ell_col[i, k, :c]] = h.ell_val[i, k, :c]
        np.testing.assert_array_equal(row, full[t])
    np.testing.assert_array_equal(h.dense_h, full[h.dense_rows])


def test_twell_forward_close_to_dense():
    # y from the TwELL of fp32-rounded z differs from the fp64 dense y only
    # by that rounding: |dy_t| <= 2^-23 * sum_j |h_tj u_tj W_d[j]|
    w = workloads.random_small(12, 128, 512, 0.05, 4, seed=14)
    z = oracle.gate_preact(w.x, w.Wg_t)
    tw = oracle.twell_pack(z, 128, 4)
    assert len(tw.spill) > 0
    y_tw = oracle.ffn_forward_twell(w.x, tw, w.Wu_t, w.Wd)
    y = oracle.ffn_forward(w.x, w.Wg_t, w.Wu_t, w.Wd)
    X, U, Dn = (oracle.bf16_to_f64(a) for a in (w.x, w.Wu_t, w.Wd))
    bound = 2.0 ** -23 * (np.abs(np.where(z > 0, z, 0) * (X @ U.T)) @ np.abs(Dn)) + 1e-15
    assert (np.abs(y_tw - y) <= bound).all()
