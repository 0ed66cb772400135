"""GPU parity of the inference path through the C-ABI: the gate GEMM with
TwELL epilogue (bit-exact packing against the oracle fed the kernel's own
fp32 gate pre-activations) and the fused up+down kernel (against the fp64
oracle, max-abs error <= 2e-2 * RMS of the reference)."""
import numpy as np
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import oracle
import workloads
from _gpu import (assert_twell_equal, check_y, ensure_built, fetch_twell, run_pack, upload,
                  z_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check_z(w, z, rows=None):
    zg = z.cpu().numpy() if rows is None else z[torch.as_tensor(rows, device=z.device)].cpu().numpy()
    X = w.x if rows is None else w.x[rows]
    ref = oracle.gate_preact(X, w.Wg_t)
    bound = z_bound(w, rows)
    bad = np.abs(zg.astype(np.float64) - ref) > bound
    assert not bad.any(), f"{bad.sum()} gate values outside the fp32 accumulation bound"
    return zg


SMALL = [
    # T, D, F, density, W
    (1, 64, 128, 0.05, 8),
    (77, 72, 384, 0.10, 8),       # ragged T, D not a multiple of 64, odd tile count
    (128, 256, 1024, 0.05, 16),
    (300, 512, 2048, 0.02, 8),
    (1024, 1536, 6144, 0.01, 8),  # enough tiles for the 256-wide variant
    (200, 128, 1024, 0.50, 8),    # heavy spilling
    (129, 192, 640, 0.05, 1),     # W = 1
    (64, 256, 512, 0.2, 128),     # W = tile: never spills
]


@pytest.mark.parametrize("T,D,F,p,W", SMALL)
def test_gate_pack_bit_exact(T, D, F, p, W):
    w = workloads.random_small(T, D, F, p, W, seed=T + D)
    _, h, z = run_pack(w)
    torch.cuda.synchronize()
    zg = _check_z(w, z)
    ref = oracle.twell_pack(zg, 128, W)
    g = fetch_twell(h)
    assert_twell_equal(g, ref)
    assert g["spill_n"] == len(ref.spill)
    assert int(h.status.item()) == 0


def block_bits_reference(zg):
    """Per block of 128 rows, bit i of word w set iff column 32 w + i has a
    positive gate in some row of the block (the TwELL block bitmap)."""
    T, F = zg.shape
    nb = (T + 127) // 128
    act = np.zeros((nb * 128, F), dtype=bool)
    act[:T] = zg > 0
    anyb = act.reshape(nb, 128, F).any(axis=1).reshape(nb, F // 32, 32)
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (anyb.astype(np.uint64) * weights).sum(axis=2).astype(np.uint32)


@pytest.mark.parametrize("T,D,F,p,W", SMALL)
def test_gate_pack_block_bits_bit_exact(T, D, F, p, W):
    w = workloads.random_small(T, D, F, p, W, seed=T + D)
    _, h, z = run_pack(w)
    torch.cuda.synchronize()
    zg = _check_z(w, z)
    got = h.block_bits.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, block_bits_reference(zg))


@pytest.mark.parametrize("T,D,F,p,W", SMALL)
def test_ffn_fwd_parity(T, D, F, p, W):
    w = workloads.random_small(T, D, F, p, W, seed=T + D)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    check_y(y.cpu().numpy().astype(np.float64), w, z.cpu().numpy())
    assert int(h.status.item()) == 0


def test_zero_active():
    w = workloads.make_uniform("none", 100, 256, 512, 1e-9, 8, seed=3)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.cnt.sum()) == 0
    assert not y.any()


def test_all_active_equals_dense_library_gemm():
    # density ~1 with W = 128: TwELL holds the dense gate; y must match the
    # dense gated FFN evaluated with torch's fp64 CPU matmul
    w = workloads.make_uniform("all", 96, 128, 256, 0.999999, 128, seed=4)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    X, G, U, Dn = (torch.from_numpy(oracle.bf16_to_f64(a)) for a in (w.x, w.Wg_t, w.Wu_t, w.Wd))
    ref = ((torch.relu(X @ G.T) * (X @ U.T)) @ Dn).numpy()
    S = (torch.relu(X @ G.T) * (X @ U.T)).abs().numpy() @ Dn.abs().numpy()
    assert (h.cnt.cpu().numpy() >= 120).all()
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 1e-4 * S + 1e-30).all()
    check_y(y.cpu().numpy().astype(np.float64), w, z.cpu().numpy())


@pytest.mark.parametrize("T", [64, 300])  # decode-size and batch gate kernels
def test_spill_count_between_packs(T):
    """Packs that spill, then none, then again, into one TwELL (through
    twell_gate_pack and, at decode sizes, twell_ffn_decode) each report
    their own spill count: the count starts from zero on every call."""
    heavy = workloads.random_small(T, 256, 1024, 0.4, 4, seed=T + 11)
    light = workloads.random_small(T, 256, 1024, 0.004, 4, seed=T + 12)
    dh, dl = upload(heavy), upload(light)
    h = tw.TwELL(T, 1024, 4)
    calls = [lambda d: tw.twell_gate_pack(d["x"], d["Wg_t"], h)]
    if T <= 256:
        calls.append(lambda d: tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h))
    for call in calls:
        for d in (dh, dl, dh, dl):
            call(d)
            torch.cuda.synchronize()
            expect = int((h.cnt.cpu().numpy() > 4).sum())
            assert int(h.spill_n.item()) == expect
            assert expect > 0 if d is dh else True
    assert int(h.status.item()) == 0


def test_spill_capacity_exhausted_sets_flag():
    w = workloads.random_small(64, 128, 1024, 0.5, 8, seed=5)
    d, h, z = run_pack(w, spill_cap=4)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) & tw.FLAG_SPILL_FULL
    ref = oracle.twell_pack(z.cpu().numpy(), 128, 8)
    g = fetch_twell(h)
    assert g["spill_n"] == len(ref.spill) > 4
    np.testing.assert_array_equal(g["cnt"], ref.cnt)
    assert len(g["spill"]) == 4
    for k, sl in g["spill"].items():
        np.testing.assert_array_equal(sl, ref.spill[k])


@pytest.mark.parametrize("T,D,F", [(300, 4096, 2048),    # narrow tiles, 64 K steps
                                    (1280, 1024, 4096),   # wide tiles, several per CTA
                                    (64, 4096, 2048)])    # decode kernel: split-K clusters
def test_gate_pack_wait_timeout_sets_flag_then_recovers(T, D, F):
    # A 2 ns bound on the gate kernel's pipeline waits: they run out, the
    # kernel sets TWELL_FLAG_TIMEOUT, drains the loads and MMAs it issued and
    # returns; the same call under the default bound then packs exactly.
    w = workloads.random_small(T, D, F, 0.05, 8, seed=T + 1)
    d = upload(w)
    h = tw.TwELL(T, F, 8)
    torch.cuda.synchronize()
    prev = tw.twell_gate_pack_wait_limit(2)
    try:
        tw.twell_gate_pack(d["x"], d["Wg_t"], h)
        torch.cuda.synchronize()
    finally:
        tw.twell_gate_pack_wait_limit(prev)
    assert prev == 1_000_000_000
    assert int(h.status.item()) & tw.FLAG_TIMEOUT
    _, h2, z = run_pack(w, d)
    torch.cuda.synchronize()
    assert int(h2.status.item()) == 0
    zg = _check_z(w, z)
    assert_twell_equal(fetch_twell(h2), oracle.twell_pack(zg, 128, 8))


def test_ffn_decode_wait_timeout_sets_flag_then_recovers():
    # the same 2 ns bound on the one-kernel decode step: its waits run out,
    # it flags TWELL_FLAG_TIMEOUT, drains and skips the packing and the
    # projection; the next call under the default bound is exact
    w = workloads.random_small(64, 4096, 2048, 0.05, 8, seed=65)
    d = upload(w)
    h = tw.TwELL(w.T, w.F, 8)
    torch.cuda.synchronize()
    prev = tw.twell_gate_pack_wait_limit(2)
    try:
        tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h)
        torch.cuda.synchronize()
    finally:
        tw.twell_gate_pack_wait_limit(prev)
    assert int(h.status.item()) & tw.FLAG_TIMEOUT
    h2 = tw.TwELL(w.T, w.F, 8)
    z = torch.empty((w.T, w.F), dtype=torch.float32, device="cuda")
    y = tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h2, z_debug=z)
    torch.cuda.synchronize()
    assert int(h2.status.item()) == 0
    zg = _check_z(w, z)
    assert_twell_equal(fetch_twell(h2), oracle.twell_pack(zg, 128, 8))
    check_y(y.cpu().numpy().astype(np.float64), w, zg)


def test_empty_batch_is_noop():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    h = tw.TwELL(0, 128, 8)
    tw.twell_gate_pack(x, W, h)
    y = tw.twell_ffn_fwd(x, h, W, W)
    torch.cuda.synchronize()
    assert y.shape == (0, 64)


def test_side_stream_and_repeat():
    w = workloads.random_small(256, 256, 1024, 0.05, 8, seed=6)
    s = torch.cuda.Stream()
    d = upload(w)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        h = tw.TwELL(w.T, w.F, 8)
        tw.twell_gate_pack(d["x"], d["Wg_t"], h, stream=s)
        y1 = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"], stream=s)
        tw.twell_gate_pack(d["x"], d["Wg_t"], h, stream=s)
        y2 = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"], stream=s)
    s.synchronize()
    # rows split over several warps (few tokens) accumulate with float
    # atomics, so repeats agree to fp32 rounding rather than bit for bit
    torch.testing.assert_close(y1, y2, rtol=1e-5, atol=1e-6)
    check_y(y2.cpu().numpy().astype(np.float64), w, tw_z(w, d))


def tw_z(w, d):
    """The kernel's fp32 gate pre-activations for all rows (z_debug)."""
    h = tw.TwELL(w.T, w.F, w.width)
    z = torch.empty((w.T, w.F), dtype=torch.float32, device="cuda")
    tw.twell_gate_pack(d["x"], d["Wg_t"], h, z_debug=z)
    return z.cpu().numpy()


# ------------------------------------------------------------ full-size configs

def _sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    rows = rng.choice(T, size=min(n, T), replace=False)
    return np.sort(np.concatenate([rows, [0, T - 1]]))


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_config_full_size(idx):
    """The bench's launch configuration at the config's full size; packing
    and y checked on sampled rows (each row depends on its token alone)."""
    w = workloads.config(idx)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    rows = _sample_rows(w.T, 96, idx)
    zg = _check_z(w, z, rows)
    assert_twell_equal(fetch_twell(h), oracle.twell_pack(zg, 128, w.width), rows)
    yg = y[torch.as_tensor(rows, device="cuda")].cpu().numpy().astype(np.float64)
    check_y(yg, w, zg, rows)
    # invariant at full size: total count equals the number of positive z
    assert int(h.cnt.to(torch.int64).sum()) == int((z > 0).sum())


@pytest.mark.parametrize("T", workloads.DECODE_T)
def test_decode_sweep(T):
    w = workloads.config(4, T=T)
    d, h, z = run_pack(w)
    y = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    zg = _check_z(w, z)
    assert_twell_equal(fetch_twell(h), oracle.twell_pack(zg, 128, w.width))
    check_y(y.cpu().numpy().astype(np.float64), w, zg)


# ------------------------------------------------- fused decode-sized forward

DECODE_FUSED = [
    # T, D, F, density, W
    (1, 256, 1024, 0.05, 8),
    (16, 2048, 1024, 0.01, 8),    # long rows: several 16-byte chunks per lane
    (77, 72, 384, 0.10, 8),       # ragged T; D of two K blocks, not a multiple of 64
    (129, 192, 640, 0.05, 1),     # W = 1; rank 1's tokens in both 128-token blocks
    (200, 128, 1024, 0.50, 8),    # heavy spilling: every active entry still in y
    (256, 512, 2048, 0.02, 16),   # the largest decode batch
    (256, 2048, 256, 0.50, 8),    # half of all entries active: 8192 entries per CTA
]


@pytest.mark.parametrize("T,D,F,p,W", DECODE_FUSED)
def test_ffn_decode_parity(T, D, F, p, W):
    # one kernel: the TwELL bit-exact as twell_gate_pack packs it, y against
    # the dense fp64 definition on the kernel's own fp32 gate decisions
    w = workloads.random_small(T, D, F, p, W, seed=T + 3)
    d = upload(w)
    h = tw.TwELL(T, F, W)
    z = torch.empty((T, F), dtype=torch.float32, device="cuda")
    y = tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h, z_debug=z)
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    zg = _check_z(w, z)
    assert_twell_equal(fetch_twell(h), oracle.twell_pack(zg, 128, W))
    np.testing.assert_array_equal(h.block_bits.cpu().numpy().view(np.uint32),
                                  block_bits_reference(zg))
    check_y(y.cpu().numpy().astype(np.float64), w, zg)
    # the same TwELL through the separate fused kernel: equal to fp32 rounding
    y2 = tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"])
    torch.cuda.synchronize()
    scale = float(y2.abs().max()) + 1e-30
    assert float((y - y2).abs().max()) <= 1e-5 * scale


def test_ffn_decode_full_spill_list_drops_nothing():
    # up to 8 tokens the projection runs in the gate kernel: with a spill
    # list of 4 slices the TwELL flags the overflow, but y still sums every
    # positive gate value (the entries come from z, not from the list)
    w = workloads.random_small(8, 128, 1024, 0.5, 8, seed=5)
    d = upload(w)
    h = tw.TwELL(w.T, w.F, 8, spill_cap=4)
    z = torch.empty((w.T, w.F), dtype=torch.float32, device="cuda")
    y = tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h, z_debug=z)
    torch.cuda.synchronize()
    assert int(h.status.item()) == tw.FLAG_SPILL_FULL
    zg = _check_z(w, z)
    check_y(y.cpu().numpy().astype(np.float64), w, zg)


def test_ffn_decode_limits():
    w = workloads.random_small(257, 128, 256, 0.05, 8, seed=1)
    d = upload(w)
    with pytest.raises(tw.TwellError):
        tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], tw.TwELL(257, 256, 8))
    x0 = d["x"][:0]
    y0 = tw.twell_ffn_decode(x0, d["Wg_t"], d["Wu_t"], d["Wd"], tw.TwELL(0, 256, 8))
    assert y0.shape == (0, 128)
    # repeated calls (y zeroed by each) agree to fp32 rounding
    h = tw.TwELL(100, 256, 8)
    x1 = d["x"][:100]
    ya = tw.twell_ffn_decode(x1, d["Wg_t"], d["Wu_t"], d["Wd"], h).clone()
    yb = tw.twell_ffn_decode(x1, d["Wg_t"], d["Wu_t"], d["Wd"], h)
    torch.cuda.synchronize()
    assert float((ya - yb).abs().max()) <= 1e-5 * (float(ya.abs().max()) + 1e-30)


@pytest.mark.parametrize("T", workloads.DECODE_T)
def test_ffn_decode_sweep(T):
    w = workloads.config(4, T=T)
    d = upload(w)
    h = tw.TwELL(T, w.F, w.width)
    z = torch.empty((T, w.F), dtype=torch.float32, device="cuda")
    y = tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h, z_debug=z)
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    zg = _check_z(w, z)
    assert_twell_equal(fetch_twell(h), oracle.twell_pack(zg, 128, w.width))
    check_y(y.cpu().numpy().astype(np.float64), w, zg)
