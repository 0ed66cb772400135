"""Roofline arithmetic of bench.py against hand-computed values of the
method's algorithmic work (no GPU)."""
import pytest

import bench


def test_updown_bytes_and_fractions_0p5b_class():
    # T=8192, D=1536, F=6144, nnz=501951, every neuron active somewhere:
    # x 25.17 MB + y (fp32) 50.33 MB + W_u/W_d rows 37.75 MB + 5 B per entry
    # 2.51 MB + counts 0.39 MB
    T, D, F, nnz = 8192, 1536, 6144, 501951
    b = bench.updown_bytes(T, D, F, nnz, F)
    assert b == 2 * T * D + 4 * T * D + 4 * F * D + 5 * nnz + T * (F // 128)
    assert b == pytest.approx(116.149e6, rel=1e-5)
    r = bench.updown_roofline(T, D, F, nnz, F, 0.200, 6784.5, 80.0, 1906.6, 64 * 4428)
    t_hbm = b / 6784.5e9
    t_fma = 4 * D * nnz / 80e12
    assert r["hbm"]["frac"] == pytest.approx(t_hbm / 200e-6)
    assert r["alu"]["frac"] == pytest.approx(t_fma / 200e-6)
    assert r["bound"] == "alu" and r["binding"]["t_us"] == pytest.approx(t_fma * 1e6)
    assert r["union_tensor_frac"] == pytest.approx(4 * 128 * D * 64 * 4428 / 200e-6 / 1906.6e12)


def test_updown_decode_is_hbm_bound():
    # one token, ~41 active neurons of 8192: bytes dominate
    r = bench.updown_roofline(1, 2048, 8192, 41, 41, 0.010, 6784.5, 80.0)
    assert r["bound"] == "hbm"
    assert r["binding"]["frac"] == pytest.approx(r["hbm"]["frac"])
    assert "union_tensor_frac" not in r


def test_gate_bound_switches_from_tensor_to_hbm():
    big = bench.gate_roofline(8192, 1536, 6144, 501951, 0.1, 6784.5, 1906.6)
    assert big["bound"] == "tensor"
    assert big["frac"] == pytest.approx(2 * 8192 * 1536 * 6144 / 0.1e-3 / 1906.6e12)
    one = bench.gate_roofline(1, 2048, 8192, 41, 0.02, 6784.5, 1906.6)
    assert one["bound"] == "hbm"
    nbytes = 2 * 2048 + 2 * 8192 * 2048 + 5 * 41 + 64
    assert one["frac"] == pytest.approx(nbytes / 6784.5e9 / 0.02e-3)


def test_train_rooflines_count_sparse_and_dense_work():
    D, F, T = 2304, 9216, 16384
    ms = {"twell_gate_pack": 0.43, "twell_to_hybrid": 0.18, "hybrid_ffn_fwd": 1.3,
          "hybrid_ffn_bwd": 5.2}
    r = bench.train_rooflines(D, F, T, 7_000_000, 492, 7_550_000, ms, 6784.5, 80.0, 1906.6)
    f = r["hybrid_ffn_fwd"]
    assert f["sparse_flops"] == 4 * D * 7_000_000
    assert f["dense_flops"] == 2 * 2 * 492 * D * F
    b = r["hybrid_ffn_bwd"]
    assert b["sparse_flops"] == 12 * D * 7_000_000
    assert b["dense_flops"] == 6 * 2 * 492 * D * F
    t = b["t_alu_us"] + b["t_tensor_us"]
    assert b["frac"] == pytest.approx(max(t, b["t_hbm_us"]) / 5200)
    assert r["twell_gate_pack"]["bound"] == "tensor"


def test_decode_roofline_counts_the_whole_step_once():
    # T=64 tokens of the decode layer (d_model 2048, d_ff 8192), 2600 active
    # entries over 2245 neurons: x in, W_g, the active neurons' W_u/W_d rows,
    # y out (fp32) and the TwELL written; HBM binds at this size
    T, D, F, nnz, na = 64, 2048, 8192, 2600, 2245
    r = bench.decode_roofline(T, D, F, nnz, na, 0.020, 6784.5, 80.0, 1906.6)
    nbytes = 2 * T * D + 2 * F * D + 4 * na * D + 4 * T * D + 5 * nnz + T * (F // 128)
    assert r["bytes"] == nbytes
    assert r["bound"] == "hbm"
    assert r["binding"]["frac"] == pytest.approx(nbytes / 6784.5e9 / 20e-6)
    assert r["tensor"]["frac"] == pytest.approx(2 * T * D * F / 1906.6e12 / 20e-6)
    assert r["alu"]["frac"] == pytest.approx(4 * D * nnz / 80e12 / 20e-6)


def test_iter_launches():
    # gate + (forward + step) for the three batch forwards: 1 + (3+4) + (6+7) + (1+2);
    # the decode step is at most two kernels (gate, then the CUDA-core forward)
    assert bench.iter_launches(("tc", "tcs", "cc")) == 24
    assert bench.iter_launches(("tc", "tcs", "cc", "dec"), 64) == 26
    assert bench.iter_launches(("tc", "tcs", "cc", "dec"), 4) == 25
