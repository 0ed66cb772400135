"""hybrid_ffn_fwd_noalloc: the hybrid forward without a workspace argument,
for callers that cannot allocate device memory themselves (a fixed memory
budget, no access to a device allocator, or no cudaMalloc because it can
synchronise the device).  Its workspace is the library's 64 MiB device
array.  Checked through the C ABI against hybrid_ffn_fwd (which takes a
caller workspace) on two calls in a row: the shared array keeps the first
call's contents, and the second call must not depend on them.  This file is
collected last so a run stopping at its first failure has run every other
test."""
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import workloads
from _gpu import ensure_built, run_pack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _hybrid_case(w, max_dense):
    d, h, z = run_pack(w)
    hyb = tw.Hybrid(w.T, w.F, w.cap, max_dense)
    tw.twell_to_hybrid(h, hyb)
    return d, hyb


def test_noalloc_matches_workspace_entry_point_twice():
    # The target case, and a different, larger one (another seed, wider
    # d_model, more and denser overflow rows) that fills more of the shared
    # array with other values first: the second call's results must not
    # depend on what the first call left there.
    w = workloads.make_training("no-alloc case", 1000, 256, 2048, 0.05, 0.03, 0.4, 16, 2e-5,
                                seed=21)
    w0 = workloads.make_training("no-alloc filler", 1500, 512, 2048, 0.06, 0.08, 0.5, 16,
                                 2e-5, seed=5)
    d0, hyb0 = _hybrid_case(w0, 512)
    d, hyb = _hybrid_case(w, 256)
    assert (tw.twell_workspace_size(tw.WS_HYBRID_FWD, w0.T, w0.D, w0.F, w0.cap, 512)
            > tw.twell_workspace_size(tw.WS_HYBRID_FWD, w.T, w.D, w.F, w.cap, 256))
    y_ref, u_ref, U_ref = tw.hybrid_ffn_fwd(d["x"], hyb, d["Wu_t"], d["Wd"])
    y0_ref, _, _ = tw.hybrid_ffn_fwd(d0["x"], hyb0, d0["Wu_t"], d0["Wd"])
    torch.cuda.synchronize()
    n_ell, n_dense = hyb.n_ell, min(hyb.n_dense, hyb.max_dense)
    assert n_dense > 0 and hyb0.n_dense > n_dense
    cnt = hyb.ell_cnt[:n_ell].long()
    used = torch.arange(w.cap, device="cuda")[None, None, :] < cnt[:, :, None]
    # first call: the filler case, itself checked
    y0, _, _ = tw.hybrid_ffn_fwd_noalloc(d0["x"], hyb0, d0["Wu_t"], d0["Wd"])
    torch.cuda.synchronize()
    assert int(hyb0.status.item()) == 0
    torch.testing.assert_close(y0, y0_ref, rtol=1e-5, atol=1e-6)
    # then the target case twice in a row
    for _ in range(2):
        y, u_ell, U_dense = tw.hybrid_ffn_fwd_noalloc(d["x"], hyb, d["Wu_t"], d["Wd"])
        torch.cuda.synchronize()
        assert int(hyb.status.item()) == 0
        # dense rows of y sum split-K partials with atomics: equal to fp32 rounding
        torch.testing.assert_close(y, y_ref, rtol=1e-5, atol=1e-6)
        torch.testing.assert_close(u_ell[:n_ell][used], u_ref[:n_ell][used], rtol=0, atol=0)
        torch.testing.assert_close(U_dense[:n_dense], U_ref[:n_dense], rtol=0, atol=0)


def test_noalloc_rejects_workspace_above_limit():
    # W_d^T alone needs D * F * 2 bytes = 72 MiB here, above the 64 MiB array
    T, D, F = 4, 3072, 12288
    assert tw.twell_workspace_size(tw.WS_HYBRID_FWD, T, D, F, 8, 4) > 64 << 20
    x = torch.zeros((T, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((F, D), dtype=torch.bfloat16, device="cuda")
    hyb = tw.Hybrid(T, F, 8, 4)
    with pytest.raises(tw.TwellError) as e:
        tw.hybrid_ffn_fwd_noalloc(x, hyb, W, W)
    assert e.value.code == 2  # TWELL_ERR_UNSUPPORTED
