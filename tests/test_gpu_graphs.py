"""Every inference call is safe to capture in a CUDA graph and replay (the
way a decode loop runs it, and the way the bench times it): the library
keeps no host-side state that a replay would reuse wrongly (tensor maps
encode buffer addresses, which stay; memsets and workspaces are on the
stream).  A step -- the gate and one forward, or the one-kernel decode
step -- is captured on a side stream with inputs A, the inputs are then
overwritten in place with inputs B, and the replay must give what direct
calls on B give: the TwELL bit for bit, y bit for bit where the kernels are
deterministic and to fp32 rounding where they add with atomics."""
import numpy as np
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import workloads
from _gpu import ensure_built, fetch_twell, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(side)  # per-call setup (kernel attributes) outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn(side)
    torch.cuda.synchronize()
    return g


def _step(kind, d, h, y, ws, wd16):
    def run(s):
        if kind == "dec":
            tw.twell_ffn_decode(d["x"], d["Wg_t"], d["Wu_t"], d["Wd"], h, y=y, stream=s)
            return
        tw.twell_gate_pack(d["x"], d["Wg_t"], h, stream=s)
        if kind == "cc":
            tw.twell_ffn_fwd(d["x"], h, d["Wu_t"], d["Wd"], y=y, stream=s)
        else:
            tw.twell_ffn_fwd_tc(d["x"], h, d["Wu_t"], d["Wd"], y=y, ws=ws, Wd_f16=wd16,
                                stream=s, sorted_rows=kind == "tcs")
    return run


CASES = [
    # T, D, F, density, W, forwards
    (300, 512, 2048, 0.02, 8, ("tc", "tcs", "cc")),      # batch gate kernel
    (64, 256, 1024, 0.05, 8, ("tc", "tcs", "cc", "dec")),  # decode gate kernel
    (1, 2048, 1024, 0.02, 8, ("cc", "dec")),             # one token
]


def _same_twell(a, b, W):
    """The unique content of two fetched TwELLs: counts, the first min(cnt, W)
    slots, every spill slice (which slot holds a slice is free)."""
    np.testing.assert_array_equal(a["cnt"], b["cnt"])
    used = np.arange(W)[None, None, :] < np.minimum(a["cnt"], W)[:, :, None]
    np.testing.assert_array_equal(np.where(used, a["col"], -1), np.where(used, b["col"], -1))
    np.testing.assert_array_equal(np.where(used, a["val"], 0), np.where(used, b["val"], 0))
    assert set(a["spill"]) == set(b["spill"])
    for key, sl in a["spill"].items():
        np.testing.assert_array_equal(sl, b["spill"][key])


def _direct(kind, d, T, D, F, W, wd16):
    """y and TwELL of direct calls (fresh buffers) on the inputs d."""
    op = tw.WS_FFN_FWD_TC_SORTED if kind == "tcs" else tw.WS_FFN_FWD_TC
    ws = (torch.empty((tw.twell_workspace_size(op, T, D, F, 0, 0),), dtype=torch.uint8,
                      device="cuda") if kind in ("tc", "tcs") else None)
    h = tw.TwELL(T, F, W)
    y = torch.empty((T, D), dtype=torch.float32, device="cuda")
    _step(kind, d, h, y, ws, wd16)(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(h.status.item()) == 0
    return y, fetch_twell(h)


@pytest.mark.parametrize("T,D,F,p,W,kinds", CASES)
def test_graph_replay_matches_direct_calls(T, D, F, p, W, kinds):
    wa = workloads.random_small(T, D, F, p, W, seed=T + 101)
    wb = workloads.random_small(T, D, F, p, W, seed=T + 202)
    da, db = upload(wa), upload(wb)
    wd16_a, wd16_b = tw.twell_to_f16(da["Wd"]), tw.twell_to_f16(db["Wd"])
    for kind in kinds:
        op = tw.WS_FFN_FWD_TC_SORTED if kind == "tcs" else tw.WS_FFN_FWD_TC
        ws = (torch.empty((tw.twell_workspace_size(op, T, D, F, 0, 0),), dtype=torch.uint8,
                          device="cuda") if kind in ("tc", "tcs") else None)
        d = {k: v.clone() for k, v in da.items()}
        wd16 = wd16_a.clone()
        h = tw.TwELL(T, F, W)
        y = torch.empty((T, D), dtype=torch.float32, device="cuda")
        g = _capture(_step(kind, d, h, y, ws, wd16))
        y_a = y.clone()  # the capture's warm-up call ran on A
        # inputs B in the captured buffers (weights too), then replay
        for k in d:
            d[k].copy_(db[k])
        wd16.copy_(wd16_b)
        g.replay()
        torch.cuda.synchronize()
        assert int(h.status.item()) == 0
        y_b, tw_b = _direct(kind, db, T, D, F, W, wd16_b)
        _same_twell(fetch_twell(h), tw_b, W)
        if kind in ("tc", "tcs"):
            torch.testing.assert_close(y, y_b, rtol=0, atol=0)
        else:
            # atomics (split rows, the one-kernel step): fp32 rounding
            scale = float(y_b.abs().max()) + 1e-30
            assert float((y - y_b).abs().max()) <= 1e-5 * scale
        assert float((y - y_a).abs().max()) > 1e-3 * float(y_a.abs().max())
