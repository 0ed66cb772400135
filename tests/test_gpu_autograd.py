"""GPU checks of the torch.autograd wrapper (activation_sparse_gated_gate_gb300.
autograd): one layer against the direct C-ABI calls, and a two-layer
residual stack against the oracle's chained fp64 composition."""
import numpy as np
import pytest
import torch

import activation_sparse_gated_gate_gb300 as tw
import oracle
import workloads
from _gpu import ensure_built, rms
from activation_sparse_gated_gate_gb300.autograd import SparseFFNStack, SparseGatedFFNFunction

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).cuda()


@pytest.mark.parametrize("tensor_cores", [True, False])
def test_function_matches_direct_calls(tensor_cores):
    w = workloads.make_training("ag", 600, 128, 1024, 0.05, 0.03, 0.4, 16, 2e-5, seed=31)
    x, Wg, Wu, Wd = (_dev(a) for a in (w.x, w.Wg_t, w.Wu_t, w.Wd))
    dy = torch.from_numpy(w.dy).cuda()
    # direct calls
    h = tw.TwELL(w.T, w.F, w.cap)
    tw.twell_gate_pack(x, Wg, h)
    hyb = tw.Hybrid(w.T, w.F, w.cap, 128)
    tw.twell_to_hybrid(h, hyb)
    fwd = tw.hybrid_ffn_fwd_tc if tensor_cores else tw.hybrid_ffn_fwd
    bwd = tw.hybrid_ffn_bwd_tc if tensor_cores else tw.hybrid_ffn_bwd
    y0, u, U = fwd(x, hyb, Wu, Wd)
    g0 = bwd(x, hyb, u, U, Wg, Wu, Wd, dy, 2e-5)
    # through autograd
    leaves = [t.clone().requires_grad_(True) for t in (x, Wg, Wu, Wd)]
    sink = []
    y1 = SparseGatedFFNFunction.apply(*leaves, 2e-5, w.cap, 128, tensor_cores, sink)
    (y1 * dy).sum().backward()
    torch.cuda.synchronize()
    assert all(int(s.item()) == 0 for s in sink)
    torch.testing.assert_close(y1, y0, rtol=1e-5, atol=1e-5)
    for g_auto, g_dir in zip([t.grad for t in leaves], g0):
        # autograd hands gradients back in the parameters' bf16
        torch.testing.assert_close(g_auto.float(), g_dir.to(torch.bfloat16).float(),
                                   rtol=1e-2, atol=1e-3)


def test_two_layer_stack_against_oracle():
    T, D, F, C = 512, 128, 1024, 16
    layers = []
    for l in range(2):
        wl = workloads.make_training(f"stack{l}", T, D, F, 0.05, 0.03, 0.4, C, 2e-5, seed=40 + l)
        layers.append((wl.Wg_t, wl.Wu_t, wl.Wd))
        if l == 0:
            w0 = wl
    stack = SparseFFNStack([tuple(_dev(a) for a in layer) for layer in layers], l1_coeff=2e-5,
                           cap=C, max_dense=T, tensor_cores=True)
    x = _dev(w0.x).requires_grad_(True)
    dy = torch.from_numpy(w0.dy).cuda()
    out = stack(x)
    (out * dy).sum().backward()
    torch.cuda.synchronize()
    assert stack.status_flags() == 0
    # The reference takes the kernel's layer inputs (the fp32 stream rounded
    # to bf16) and gate decisions (z exported by the gate kernel on the same
    # inputs): gradients through ReLU layers jump where a gate straddles zero,
    # and tiny stream differences would move a few gates across it.
    inputs, actives = [], []
    s_l = _dev(w0.x).float()
    for l in range(2):
        a_l = s_l.to(torch.bfloat16)
        inputs.append(a_l.view(torch.int16).cpu().numpy().view(np.uint16))
        h = tw.TwELL(T, F, C)
        z = torch.empty((T, F), dtype=torch.float32, device="cuda")
        tw.twell_gate_pack(a_l, stack.Wg[l].detach().to(torch.bfloat16).contiguous(), h,
                           z_debug=z)
        actives.append(z.cpu().numpy() > 0)
        with torch.no_grad():
            y = SparseGatedFFNFunction.apply(a_l, stack.Wg[l], stack.Wu[l], stack.Wd[l], 2e-5, C,
                                             T, True, None)
            y[:, -1] = 0.0
            s_l = s_l + y
    ref_out, _, ref_grads = oracle.stack_forward_backward(w0.x, layers, w0.dy, 2e-5,
                                                          inputs=inputs, actives=actives)
    # the layers' contribution out - x
    x0 = oracle.bf16_to_f64(w0.x)
    got = out.detach().cpu().numpy().astype(np.float64) - x0
    ref = ref_out - x0
    assert np.max(np.abs(got - ref)) <= 2e-2 * rms(ref)
    assert rms(got - ref) <= 5e-3 * rms(ref)
    # fp32 master weights: fp32 gradients
    params = [(stack.Wg[l], stack.Wu[l], stack.Wd[l]) for l in range(2)]
    for l in range(2):
        for p, r, n in zip(params[l], ref_grads[l], ("dWg_t", "dWu_t", "dWd")):
            g = p.grad.float().cpu().numpy().astype(np.float64)
            assert np.max(np.abs(g - r)) <= 2e-2 * rms(r), (l, n)
            assert rms(g - r) <= 5e-3 * rms(r), (l, n)
