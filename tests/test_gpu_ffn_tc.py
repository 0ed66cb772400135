"""GPU parity of the tensor-core (union-gather) fused forward,
twell_ffn_fwd_tc, through the C-ABI: against the fp64 oracle fed the gate
kernel's own fp32 pre-activations (spec bar max-abs <= 2e-2 * RMS plus
an RMS bar), against an elementwise worst-case bound for its arithmetic
(h u rounded to fp16, W_d converted to fp16, fp32 tensor-core sums), and
against the CUDA-core fused kernel."""
import numpy as np
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import oracle
import workloads
from _gpu import assert_ns_tol, ensure_built, rms, run_pack, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def check_y_tc(yg, w, zg, rows=None):
    """``yg``: the kernel's y for token rows ``rows``; ``zg``: the gate
    kernel's fp32 pre-activations of those rows (the activation decision).

    1. Spec bar against the dense fp64 definition:
       max-abs <= 2e-2 * RMS(reference), and RMS(error) <= 5e-3 * RMS.
    2. Elementwise bound against the oracle's TwELL-form forward (same gate
       values), with S_a = sum_j |h_j u_j| |W_d[j]|, S_u = sum_j |h_j| B_j
       |W_d[j]|, B = |x| |W_u|:  a = fp16(h u) is off by at most
       2^-11 |h u| + 2^-25 (round to nearest, 11 significant bits, subnormal
       spacing 2^-24) after u's fp32 tensor-core sum (D terms, 2^-23 each
       allowing truncating adds); W_d's fp16 copy is exact down to 2^-14 and
       off by at most 2^-25 below; y's fp32 sum over at most F union
       positions adds F 2^-23 S_a:
         |err| <= 1.01 (2^-11 S_a + D 2^-23 S_u) + F 2^-22 S_a
                  + 2^-24 (sum_j |W_d[j]| + sum_j |h_j u_j|)   (active j).
    """
    rows = np.arange(w.T) if rows is None else np.asarray(rows)
    x = w.x[rows]
    ref_tw = oracle.twell_pack(zg, 128, w.width)
    y_tw = oracle.ffn_forward_twell(x, ref_tw, w.Wu_t, w.Wd)
    act = zg > 0
    y_dense = oracle.ffn_forward(x, w.Wg_t, w.Wu_t, w.Wd, active=act)
    err, tol = assert_ns_tol(yg, y_dense, "y vs dense fp64 oracle")
    assert rms(yg - y_dense) <= 5e-3 * rms(y_dense) + 1e-30
    X, U, Dn = (oracle.bf16_to_f64(a) for a in (x, w.Wu_t, w.Wd))
    u = X @ U.T
    B = np.abs(X) @ np.abs(U).T
    h = np.where(act, zg.astype(np.float64), 0.0)
    Dabs = np.abs(Dn)
    S_a = (np.abs(h * u)) @ Dabs
    S_u = (np.abs(h) * B) @ Dabs
    tiny = act.astype(np.float64) @ Dabs + np.abs(h * u).sum(axis=1, keepdims=True)
    b = (1.01 * (2.0 ** -11 * S_a + w.D * 2.0 ** -23 * S_u) + w.F * 2.0 ** -22 * S_a
         + 2.0 ** -24 * tiny + 1e-30)
    e = np.abs(yg - y_tw)
    assert (e <= b).all(), f"max excess {float((e - b).max()):.3e}"
    return y_tw


CASES = [
    # T, D, F, density, W
    (1, 64, 128, 0.05, 8),
    (128, 256, 1024, 0.05, 16),
    (300, 512, 2048, 0.02, 8),      # ragged last block
    (1024, 1536, 6144, 0.01, 8),    # the 0.5B-class layer on 1024 tokens
    (200, 128, 1024, 0.50, 8),      # heavy spilling, unions near F
    (129, 192, 640, 0.05, 1),       # W = 1; D < 256: one ragged output tile; F not a multiple of 256
    (64, 256, 512, 0.2, 128),       # W = tile
    (700, 320, 1152, 0.03, 8),      # D = 320: a full and a ragged output tile
    (10240, 320, 512, 0.05, 8),     # 160 down tiles: the partial last wave split in halves,
                                    # ragged tiles among them
]


@pytest.mark.parametrize("T,D,F,p,W", CASES)
def test_ffn_fwd_tc_parity(T, D, F, p, W):
    w = workloads.random_small(T, D, F, p, W, seed=T + D + 1)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    check_y_tc(y.cpu().numpy().astype(np.float64), w, z.cpu().numpy())


@pytest.mark.parametrize("T,D,F,p,W", [CASES[2], CASES[4], CASES[5], CASES[7]])
def test_without_block_bits(T, D, F, p, W):
    """A TwELL without the gate kernel's block bitmaps: the forward builds
    the unions itself, with the same result bit for bit."""
    w = workloads.random_small(T, D, F, p, W, seed=T + D + 1)
    d = upload(w)
    h1 = tw.TwELL(w.T, w.F, W, block_bits=False)
    z = torch.empty((w.T, w.F), dtype=torch.float32, device="cuda")
    tw.twell_gate_pack(d["x"], d["Wg_t"], h1, z_debug=z)
    _, h2, _ = run_pack(w, d)
    y1 = tw.twell_ffn_fwd_tc(d["x"], h1, d["Wu_t"], d["Wd"])
    y2 = tw.twell_ffn_fwd_tc(d["x"], h2, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h1.status.item()) == 0
    assert torch.equal(y1, y2)
    check_y_tc(y1.cpu().numpy().astype(np.float64), w, z.cpu().numpy())


def test_precomputed_f16_weights():
    """twell_to_f16 rounds like numpy's float32 -> float16 conversion, and a
    caller-made fp16 W_d gives the same y, bit for bit, as the call's own."""
    w = workloads.random_small(300, 256, 1024, 0.05, 8, seed=17)
    d, h, z = run_pack(w)
    wd16 = tw.twell_to_f16(d["Wd"])
    torch.cuda.synchronize()
    ref = workloads.bf16_to_f64(w.Wd).astype(np.float32).astype(np.float16)
    np.testing.assert_array_equal(wd16.cpu().numpy().view(np.uint16), ref.view(np.uint16))
    y1 = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    y2 = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"], Wd_f16=wd16)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_agrees_with_cuda_core_kernel_and_repeats_bit_exact():
    w = workloads.random_small(512, 512, 2048, 0.03, 8, seed=11)
    d, h, z = run_pack(w)
    y1 = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    y2 = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    y0 = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    # both are within their bounds of the same TwELL-form value; the gap is
    # the fp16 rounding of h u (relative 2^-11 per term, random signs)
    a, b = y1.cpu().numpy().astype(np.float64), y0.cpu().numpy().astype(np.float64)
    assert rms(a - b) <= 5e-4 * rms(b)
    check_y_tc(a, w, z.cpu().numpy())


def test_blocks_without_active_neurons():
    # rows 128..255 (one whole block) and the last rows get a large bias
    # input, so no gate there is positive: their y rows must be exactly 0
    w = workloads.random_small(400, 256, 1024, 0.05, 8, seed=12)
    big = workloads.to_bf16(np.array([1000.0]))[0]
    w.x[128:256, w.D - 1] = big
    w.x[390:, w.D - 1] = big
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.cnt[128:256].sum()) == 0 and int(h.cnt[390:].sum()) == 0
    yc = y.cpu().numpy()
    assert not yc[128:256].any() and not yc[390:].any()
    check_y_tc(yc.astype(np.float64), w, z.cpu().numpy())


def test_zero_active_everywhere():
    w = workloads.make_uniform("none", 300, 256, 512, 1e-9, 8, seed=13)
    d, h, z = run_pack(w)
    y = torch.full((w.T, w.D), float("nan"), device="cuda")
    tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"], y=y)
    torch.cuda.synchronize()
    assert int(h.cnt.sum()) == 0
    assert not y.any()


def test_stale_workspace_is_harmless():
    # the workspace holds NaN bytes from a previous user: every value the
    # kernels read is written first or masked
    w = workloads.random_small(333, 256, 1024, 0.05, 8, seed=14)
    d, h, z = run_pack(w)
    nbytes = tw.twell_workspace_size(tw.WS_FFN_FWD_TC, w.T, w.D, w.F, 0, 0)
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    y = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"], ws=ws.view(torch.uint8))
    torch.cuda.synchronize()
    check_y_tc(y.cpu().numpy().astype(np.float64), w, z.cpu().numpy())


def test_fp16_range_exceeded_sets_flag():
    # inputs 300x larger make |h u| ~ 1e5 > 65504: the fp16 operand of the
    # down GEMM cannot hold it and the call says so
    w = workloads.random_small(256, 256, 512, 0.05, 8, seed=16)
    xs = workloads.bf16_to_f64(w.x)
    xs[:, :-1] *= 300.0
    w.x = workloads.to_bf16(xs)
    d, h, z = run_pack(w)
    tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) & tw.FLAG_RANGE


def test_spill_capacity_exhausted_sets_flag():
    w = workloads.random_small(64, 128, 1024, 0.5, 8, seed=15)
    d, h, z = run_pack(w, spill_cap=4)
    tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) & tw.FLAG_SPILL_FULL


def test_unsupported_shapes_are_rejected():
    x = torch.zeros((16, 72), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 72), dtype=torch.bfloat16, device="cuda")
    h = tw.TwELL(16, 128, 8)
    tw.twell_gate_pack(x, W, h)
    with pytest.raises(tw.TwellError):
        tw.twell_ffn_fwd_tc(x, h, W, W)  # D not a multiple of 64
    ws = torch.empty((16,), dtype=torch.uint8, device="cuda")
    x2 = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tw.TwellError):
        tw.twell_ffn_fwd_tc(x2, h, W2, W2, ws=ws)  # workspace too small


def test_empty_batch_is_noop():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    h = tw.TwELL(0, 128, 8)
    tw.twell_gate_pack(x, W, h)
    y = tw.twell_ffn_fwd_tc(x, h, W, W)
    torch.cuda.synchronize()
    assert y.shape == (0, 64)


def _sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    rows = rng.choice(T, size=min(n, T), replace=False)
    return np.sort(np.concatenate([rows, [0, T - 1]]))


@pytest.mark.parametrize("idx", [1, 2])
def test_config_full_size(idx):
    """The inference layers at full size (0.5B- and 1.5B-class), checked on
    sampled rows (each row depends on its own token and gate alone)."""
    w = workloads.config(idx)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    rows = _sample_rows(w.T, 64, idx + 100)
    ri = torch.as_tensor(rows, device="cuda")
    zg = z[ri].cpu().numpy()
    check_y_tc(y[ri].cpu().numpy().astype(np.float64), w, zg, rows)


# ------------------------------------------- blocks grouped by activity (sorted)

def _tc_sorted(d, h, w):
    return tw.twell_ffn_fwd_tc_sorted(d["x"], h, d["Wu_t"], d["Wd"])


@pytest.mark.parametrize("T,D,F,p,W", CASES)
def test_ffn_fwd_tc_sorted_parity(T, D, F, p, W):
    w = workloads.random_small(T, D, F, p, W, seed=T + D + 1)
    d, h, z = run_pack(w)
    y = _tc_sorted(d, h, w)
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    check_y_tc(y.cpu().numpy().astype(np.float64), w, z.cpu().numpy())


def test_sorted_heavy_tail_repeats_and_agrees_with_token_order():
    # per-token activity spread like the 1.5B-class workload (lognormal
    # threshold offsets): the sorted blocks give the same y as blocks of
    # consecutive tokens up to fp16 rounding of h u, and repeats are equal
    w = workloads.make_heavy_tail("heavy-tail small", 3000, 256, 2048, 0.01, 16, seed=4)
    d, h, z = run_pack(w)
    y1 = _tc_sorted(d, h, w)
    y2 = _tc_sorted(d, h, w)
    y0 = tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    assert torch.equal(y1, y2)
    assert float((y1 - y0).norm() / y0.norm()) <= 2e-3
    check_y_tc(y1.cpu().numpy().astype(np.float64), w, z.cpu().numpy())


def test_sorted_spill_capacity_exhausted_sets_flag():
    w = workloads.random_small(256, 128, 1024, 0.5, 8, seed=5)
    d, h, z = run_pack(w, spill_cap=4)
    _tc_sorted(d, h, w)
    torch.cuda.synchronize()
    assert int(h.status.item()) & tw.FLAG_SPILL_FULL


def test_sorted_full_size_heavy_tail_layer():
    # the 1.5B-class layer at full size in the bench's launch configuration,
    # checked on sampled rows
    w = workloads.config(2)
    d, h, z = run_pack(w)
    y = _tc_sorted(d, h, w)
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    rng = np.random.default_rng(2)
    rows = np.sort(np.concatenate([rng.choice(w.T, 96, replace=False), [0, w.T - 1]]))
    idx = torch.as_tensor(rows, device="cuda")
    check_y_tc(y[idx].cpu().numpy().astype(np.float64), w, z[idx].cpu().numpy(), rows)
