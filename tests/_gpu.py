"""Helpers for the GPU parity tests: upload seeded inputs, run the library
through its C-ABI binding, and bring results back in the oracle's form."""
import numpy as np
import torch

import activation_sparse_gated_gate_gb300 as tw
import oracle


def ensure_built():
    if not torch.cuda.is_available():
        return
    import os
    if not os.path.exists(tw.LIB_PATH):
        from activation_sparse_gated_gate_gb300 import build
        build.build()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).cuda()


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def upload(w):
    return {k: dev_bf16(getattr(w, k)) for k in ("x", "Wg_t", "Wu_t", "Wd")}


def run_pack(w, d=None, spill_cap=None, z_debug=True, stream=None):
    d = d or upload(w)
    h = tw.TwELL(w.T, w.F, w.width, spill_cap=spill_cap)
    z = torch.empty((w.T, w.F), dtype=torch.float32, device="cuda") if z_debug else None
    tw.twell_gate_pack(d["x"], d["Wg_t"], h, z_debug=z, stream=stream)
    return d, h, z


def fetch_twell(h):
    """GPU TwELL -> dict(cnt, col, val, spill {(t,k): slice}, slot, spill_n)."""
    cnt = h.cnt.cpu().numpy().astype(np.int64)
    col = h.col.cpu().numpy().astype(np.int64)
    val = h.val.cpu().numpy()
    slot = h.spill_slot.cpu().numpy()
    spill_n = int(h.spill_n.item())
    sv = h.spill_val.cpu().numpy()
    srt = h.spill_rt.cpu().numpy()
    spill = {}
    for t, k in zip(*np.nonzero(cnt > h.width)):
        s = int(slot[t, k])
        if 0 <= s < h.spill_cap:
            assert srt[s] == t * h.n_t + k
            spill[(int(t), int(k))] = sv[s]
    return dict(cnt=cnt, col=col, val=val, spill=spill, slot=slot, spill_n=spill_n)


def assert_twell_equal(g, ref: oracle.TwELL, rows=None):
    """Bit-exact comparison of the unique content: counts, the first
    min(cnt, W) slots and every spill slice (padding slots are free).
    With ``rows``, GPU row rows[i] is compared with ``ref`` row i (``ref``
    packed from those rows only)."""
    rows = np.arange(ref.T) if rows is None else np.asarray(rows)
    W = ref.width
    np.testing.assert_array_equal(g["cnt"][rows], ref.cnt)
    s = np.arange(W)[None, None, :]
    used = s < np.minimum(ref.cnt, W)[:, :, None]
    np.testing.assert_array_equal(np.where(used, g["col"][rows], -1),
                                  np.where(used, ref.col, -1))
    np.testing.assert_array_equal(np.where(used, g["val"][rows], 0),
                                  np.where(used, ref.val, 0))
    pos = {int(t): i for i, t in enumerate(rows)}
    got = {(pos[t], k) for (t, k) in g["spill"] if t in pos}
    assert got == set(ref.spill)
    for (t, k), sl in g["spill"].items():
        if t in pos:
            np.testing.assert_array_equal(sl, ref.spill[(pos[t], k)])


def z_bound(w, rows=None):
    """Bound on |z_fp32 - z_exact|: fp32 accumulation of D exact products,
    D * 2^-24 * sum_i |x_i w_i| (plus the subnormal floor)."""
    X = oracle.bf16_to_f64(w.x if rows is None else w.x[rows])
    G = oracle.bf16_to_f64(w.Wg_t)
    return w.D * 2.0 ** -24 * (np.abs(X) @ np.abs(G).T) + 1e-30


def rms(a):
    return float(np.sqrt(np.mean(np.square(a)))) if a.size else 0.0


def assert_ns_tol(got, ref, what=""):
    """Output tolerance: max-abs error <= 2e-2 * RMS(reference)."""
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    tol = 2e-2 * rms(ref)
    assert err <= tol, f"{what}: max-abs {err:.3e} > 2e-2*RMS {tol:.3e}"
    return err, tol


def check_y(yg, w, zg, rows=None):
    """Check the kernel's fp32 output y for token rows ``rows`` (all by
    default); ``zg`` holds the kernel's fp32 gate pre-activations of those
    rows, so both sides take the activation decision in fp32.

    1. Spec bar against the dense fp64 definition:
       max-abs <= 2e-2 * RMS(reference).
    2. Elementwise worst-case fp32 bounds (gamma_n = n * 2^-24 per summed
       term, any summation order), with A = |x||W_g|, B = |x||W_u|:
       against the oracle's TwELL-form forward (same fp32 gate values)
         |err| <= (D + F + 2) 2^-24 * sum_j |h_j| B_j |W_d[j]|
       and against the dense fp64 definition, plus the gate's own fp32
       rounding  D 2^-24 * sum_j A_j |u_j| |W_d[j]|.
    """
    rows = np.arange(w.T) if rows is None else np.asarray(rows)
    x = w.x[rows]
    ref_tw = oracle.twell_pack(zg, 128, w.width)
    y_tw = oracle.ffn_forward_twell(x, ref_tw, w.Wu_t, w.Wd)
    X, G, U, Dn = (oracle.bf16_to_f64(a) for a in (x, w.Wg_t, w.Wu_t, w.Wd))
    act = zg > 0
    y_dense = oracle.ffn_forward(x, w.Wg_t, w.Wu_t, w.Wd, active=act)
    assert_ns_tol(yg, y_dense, "y vs dense fp64 oracle")
    Xa = np.abs(X)
    A = Xa @ np.abs(G).T
    B = Xa @ np.abs(U).T
    u = X @ U.T
    Dabs = np.abs(Dn)
    S2 = (np.where(act, np.abs(zg), 0.0) * B) @ Dabs
    Sz = (np.where(act, A, 0.0) * np.abs(u)) @ Dabs
    eps = 2.0 ** -24
    b_tw = (w.D + w.F + 2) * eps * S2 + eps * np.abs(y_tw) + 1e-30
    e1 = np.abs(yg - y_tw)
    assert (e1 <= b_tw).all(), f"TwELL-form: max excess {float((e1 - b_tw).max()):.3e}"
    b_d = b_tw + w.D * eps * Sz
    e2 = np.abs(yg - y_dense)
    assert (e2 <= b_d).all(), f"dense: max excess {float((e2 - b_d).max()):.3e}"
    return y_tw
