"""torch.autograd wrapper of the hybrid training path ("Sparser, Faster,
Lighter Transformer Language Models", section 2.B.3; the L1 coefficient from
the news article "Sakana AI and NVIDIA TwELL boosts LLM training speed by
21.9%", recipe list).

``SparseGatedFFNFunction`` runs one activation-sparse gated FFN layer
through the C-ABI: the gate GEMM with the TwELL epilogue, the TwELL -> hybrid
conversion and the hybrid forward; its backward is the hybrid backward with
the L1 term on h.  ``SparseFFNStack`` chains layers with residual additions.
Argument marshalling only: every step runs in libtwell's kernels, on torch's
current stream, with nothing read back.

Weights may be bf16 or fp32 master copies (cast to bf16 for the kernels on
every call); their gradients come back from the library in fp32 and are
returned in the weights' own dtype, as autograd requires, so fp32 masters keep
fp32 gradients.  The activation stream x is bf16 (its gradient too).
"""
from __future__ import annotations

import torch

from . import (Hybrid, TwELL, hybrid_ffn_bwd, hybrid_ffn_bwd_tc, hybrid_ffn_fwd,
               hybrid_ffn_fwd_tc, twell_gate_pack, twell_to_hybrid)


class SparseGatedFFNFunction(torch.autograd.Function):
    """y = (ReLU(x W_g) * (x W_u)) W_d through TwELL and the hybrid format.

    Inputs: x [T][D] bf16, Wg_t / Wu_t / Wd [F][D] bf16 or fp32; ``l1_coeff`` adds
    l1_coeff * sum(h) to the loss; ``cap`` is the ELL capacity per 128-column
    tile (rows above it in some tile go to the dense backup, at most
    ``max_dense`` of them); ``tensor_cores`` selects hybrid_ffn_*_tc.
    Returns y [T][D] fp32.  The device status words of the call (TwELL and
    hybrid) are appended to ``status_sink`` when it is a list."""

    @staticmethod
    def forward(ctx, x, Wg_t, Wu_t, Wd, l1_coeff, cap, max_dense, tensor_cores, status_sink):
        T, _ = x.shape
        F = Wg_t.shape[0]
        w16 = [w if w.dtype == torch.bfloat16 else w.to(torch.bfloat16).contiguous()
               for w in (Wg_t, Wu_t, Wd)]
        # with the TwELL width equal to the ELL capacity, a (row, tile) spills
        # only in rows that overflow to the dense backup: max_dense * n_t
        # spill slices suffice (more rows than that set TWELL_FLAG_DENSE_FULL)
        h = TwELL(T, F, cap, spill_cap=max(1, max_dense) * (F // 128), device=x.device)
        twell_gate_pack(x, w16[0], h)
        hyb = Hybrid(T, F, cap, max_dense, device=x.device)
        twell_to_hybrid(h, hyb)
        fwd = hybrid_ffn_fwd_tc if tensor_cores else hybrid_ffn_fwd
        y, u_ell, U_dense = fwd(x, hyb, w16[1], w16[2])
        ctx.save_for_backward(x, *w16, u_ell, U_dense)
        ctx.w_dtypes = (Wg_t.dtype, Wu_t.dtype, Wd.dtype)
        ctx.hyb = hyb
        ctx.l1 = float(l1_coeff)
        ctx.tc = bool(tensor_cores)
        if status_sink is not None:
            status_sink.extend([h.status, hyb.status])
        return y

    @staticmethod
    def backward(ctx, dy):
        x, Wg_t, Wu_t, Wd, u_ell, U_dense = ctx.saved_tensors
        bwd = hybrid_ffn_bwd_tc if ctx.tc else hybrid_ffn_bwd
        dx, dWg, dWu, dWd = bwd(x, ctx.hyb, u_ell, U_dense, Wg_t, Wu_t, Wd,
                                dy.float().contiguous(), ctx.l1)
        dt = ctx.w_dtypes
        return (dx.to(x.dtype), dWg.to(dt[0]), dWu.to(dt[1]), dWd.to(dt[2]),
                None, None, None, None, None)


class SparseFFNStack(torch.nn.Module):
    """L residual blocks x <- x + FFN_l(bf16(x)): the residual stream and its
    gradient stay fp32; each layer's input is the stream rounded to bf16.

    Parameters are fp32 master copies of the given weights (gradients in
    fp32); the kernels see them rounded to bf16 on every call.

    ``bias_feature``: when set, feature D - 1 of x is a constant bias input
    (the gate's threshold feature, as in the synthetic workloads) and the
    residual update leaves it unchanged, so every layer sees the same
    activation-density control."""

    def __init__(self, weights, l1_coeff=2e-5, cap=32, max_dense=1024, tensor_cores=True,
                 bias_feature=True):
        super().__init__()
        self.Wg = torch.nn.ParameterList(torch.nn.Parameter(w[0].float()) for w in weights)
        self.Wu = torch.nn.ParameterList(torch.nn.Parameter(w[1].float()) for w in weights)
        self.Wd = torch.nn.ParameterList(torch.nn.Parameter(w[2].float()) for w in weights)
        self.l1 = l1_coeff
        self.cap = cap
        self.max_dense = max_dense
        self.tc = tensor_cores
        self.bias_feature = bias_feature
        self.last_status = []

    def forward(self, x):
        """x [T][D] (any float dtype) -> the fp32 stream after the last layer."""
        self.last_status = []
        s = x.float()
        for Wg, Wu, Wd in zip(self.Wg, self.Wu, self.Wd):
            y = SparseGatedFFNFunction.apply(s.to(torch.bfloat16), Wg, Wu, Wd, self.l1, self.cap,
                                             self.max_dense, self.tc, self.last_status)
            if self.bias_feature:
                y = torch.cat([y[:, :-1], torch.zeros_like(y[:, -1:])], dim=1)
            s = s + y
        return s

    def status_flags(self) -> int:
        """OR of the device status words of the last forward (synchronises)."""
        flags = 0
        for s in self.last_status:
            flags |= int(s.item())
        return flags
