"""CPU oracle for the activation-sparse gated FFN with TwELL.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The library
(``activation_sparse_gated_gate_gb300``) never calls it, and this package
never imports the library: the two share no code.

Plain and slow on purpose: numpy in fp64, library matmuls as steps, no
blocking or fusion beyond what the definitions state.

Sources ("Sparser, Faster, Lighter Transformer Language Models", gist.science
summary of arXiv 2603.23198, and the MarkTechPost-derived news article
"Sakana AI and NVIDIA TwELL boosts LLM training speed by 21.9%"):

* Gated FFN with ReLU in place of SiLU so the gate has exact zeros
  (news article, bullet list of the two recipe changes; paper section 2.A),
  gate activations h_g = ReLU(x W_g) (paper section 2.B.1).  The up and down
  projections follow the standard gated MLP: y = (h_g * (x W_u)) W_d
  (paper section 2.B.2: fused up and down projections using h_g).
* TwELL: the gate columns are cut into horizontal tiles the width of the
  matmul tile; each (row, tile) keeps its own nonzeros (paper section 2.B.1;
  news article, epilogue paragraph).
* Hybrid training format: rows with few nonzeros in a compact ELL matrix,
  overflow rows in a dense backup (paper section 2.B.3).
* L1 penalty on the FFN activations with coefficient 2e-5 (news article,
  recipe list; paper section 4, accuracy bullet).

Readings where the pages are silent (each listed in the design notes):
  active iff z > 0 in the precision the decision is taken in (NaN, +0 and -0
  inactive); slots hold active columns in ascending order; slot values are z
  at the gate accumulator's precision (fp32), since rounding them to bf16
  alone costs up to ~2% of RMS(y) against the dense definition; a (row,
  tile) with more actives than the width W keeps its true count, its first W
  actives in the slots, and its whole 128-wide fp32 slice ReLU(z) in a spill
  list; a row goes to the dense backup iff some tile count exceeds the ELL
  capacity C; the L1 term adds lambda to dL/dh at active entries.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against hand-derived fixtures (``tests/golden/``), brute-force loops on tiny
inputs, central finite differences, closed forms and invariants.
"""

from __future__ import annotations

import dataclasses

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> float (the oracle's own; round to nearest, ties to even)
# ---------------------------------------------------------------------------


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    with np.errstate(invalid="ignore"):
        return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(
            np.float32).astype(np.float64)


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns, round to nearest, ties to even.

    The 16 low bits of the fp32 pattern are dropped after adding half an ulp
    of bf16, plus one more when the kept part is odd (ties to even).  NaN is
    mapped to a quiet NaN so rounding cannot turn it into infinity.
    """
    f = np.ascontiguousarray(f, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), r)
    return r


def relu(z: np.ndarray) -> np.ndarray:
    """ReLU with the active test z > 0; inactive entries are +0."""
    return np.where(z > 0, z, 0.0)


# ---------------------------------------------------------------------------
# Dense definitions (paper section 2.B: h_g = ReLU(x W_g); fused up/down)
# ---------------------------------------------------------------------------


def gate_preact(x, Wg_t):
    """z = x W_g in fp64.  ``x`` [T][D], ``Wg_t`` = W_g^T [F][D], both bf16
    bits.  Products of two bf16 values are exact in fp64."""
    return bf16_to_f64(x) @ bf16_to_f64(Wg_t).T


def ffn_forward_f64(X, G, U, Dn, active=None):
    """y = (ReLU(x W_g) * (x W_u)) W_d on fp64 arrays, the plain gated FFN
    with the ReLU gate (news article recipe list; paper sections 2.A and
    2.B).  ``G``, ``U`` are W_g^T, W_u^T and ``Dn`` is W_d, all [F][D].

    ``active`` optionally overrides the activation decision z > 0 (a boolean
    [T][F] array taken in another precision); values stay fp64.
    """
    z = X @ G.T
    act = (z > 0) if active is None else active
    h = np.where(act, z, 0.0)
    u = X @ U.T
    return (h * u) @ Dn


def ffn_forward(x, Wg_t, Wu_t, Wd, active=None):
    """``ffn_forward_f64`` on bf16 bit-pattern inputs; returns y [T][D] fp64."""
    return ffn_forward_f64(bf16_to_f64(x), bf16_to_f64(Wg_t), bf16_to_f64(Wu_t),
                           bf16_to_f64(Wd), active)


def ffn_forward_rows(x, Wg_t, Wu_t, Wd, rows):
    """``ffn_forward`` restricted to the token rows ``rows`` (each row of the
    gated FFN depends on that token alone)."""
    return ffn_forward(np.asarray(x)[np.asarray(rows)], Wg_t, Wu_t, Wd)


def ffn_forward_sparse(x, Wg_t, Wu_t, Wd):
    """The same output computed only over active neurons: for each token,
    for each j with z_tj > 0, u = x_t . W_u[:, j] and
    y_t += (h_tj u) W_d[j, :] (paper section 2.B.2: dot products only for
    the nonzero elements).  Must equal ``ffn_forward`` up to fp64 rounding."""
    X = bf16_to_f64(x)
    G = bf16_to_f64(Wg_t)
    U = bf16_to_f64(Wu_t)
    Dn = bf16_to_f64(Wd)
    y = np.zeros((X.shape[0], Dn.shape[1]))
    for t in range(X.shape[0]):
        z = G @ X[t]
        for j in np.nonzero(z > 0)[0]:
            u = float(U[j] @ X[t])
            y[t] += (z[j] * u) * Dn[j]
    return y


# ---------------------------------------------------------------------------
# TwELL (paper section 2.B.1; news article, epilogue paragraph)
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class TwELL:
    """Tile-wise ELL of a [T][F] gate activation.

    cnt  [T][n_t]     number of active entries of row t in column tile k
    col  [T][n_t][W]  local column (0..tile-1) of slot s, valid for s < min(cnt, W)
    val  [T][n_t][W]  fp32 z at that column
    spill  dict (t, k) -> [tile] fp32 ReLU(z) for every (t, k) with cnt > W
    """
    T: int
    F: int
    tile: int
    width: int
    cnt: np.ndarray
    col: np.ndarray
    val: np.ndarray
    spill: dict

    @property
    def n_t(self):
        return self.F // self.tile


def twell_pack(z, tile, width):
    """Pack the gate activation ReLU(z) into TwELL.

    ``z`` is the gate pre-activation in the precision the activation
    decision is taken in (fp32 from a kernel, or fp64).  For every row t and
    column tile k = [k*tile, (k+1)*tile): list the columns with z > 0 in
    ascending order; cnt is the list's length; the first min(cnt, W) go to
    the slots with value z (fp32); if cnt > W the whole slice ReLU(z) (fp32)
    is kept in the spill list.
    """
    z = np.asarray(z)
    T, F = z.shape
    assert F % tile == 0
    n_t = F // tile
    # the decision is taken in z's own precision; values are rounded from fp32
    act = z.reshape(T, n_t, tile) > 0
    zt = z.astype(np.float32).reshape(T, n_t, tile)
    cnt = act.sum(axis=2).astype(np.int64)
    # stable sort puts the active columns first, in ascending order
    order = np.argsort(~act, axis=2, kind="stable")
    col = np.zeros((T, n_t, width), np.int64)
    val = np.zeros((T, n_t, width), np.float32)
    take = min(width, tile)
    col[:, :, :take] = order[:, :, :take]
    val[:, :, :take] = np.take_along_axis(zt, order[:, :, :take], axis=2)
    s = np.arange(width)[None, None, :]
    valid = s < np.minimum(cnt, width)[:, :, None]
    col = np.where(valid, col, 0)
    val = np.where(valid, val, np.float32(0)).astype(np.float32)
    spill = {}
    relu = np.where(act, zt, np.float32(0.0)).astype(np.float32)
    for t, k in zip(*np.nonzero(cnt > width)):
        spill[(int(t), int(k))] = relu[t, k].copy()
    return TwELL(T, F, tile, width, cnt, col, val, spill)


def twell_pack_loops(z, tile, width):
    """``twell_pack`` written as scalar loops (small inputs only)."""
    z = np.asarray(z, dtype=np.float32)
    T, F = z.shape
    n_t = F // tile
    cnt = np.zeros((T, n_t), np.int64)
    col = np.zeros((T, n_t, width), np.int64)
    val = np.zeros((T, n_t, width), np.float32)
    spill = {}
    for t in range(T):
        for k in range(n_t):
            c = 0
            for j in range(tile):
                v = z[t, k * tile + j]
                if v > 0:
                    if c < width:
                        col[t, k, c] = j
                        val[t, k, c] = v
                    c += 1
            cnt[t, k] = c
            if c > width:
                spill[(t, k)] = np.array([z[t, k * tile + j] if z[t, k * tile + j] > 0 else 0.0
                                          for j in range(tile)], np.float32)
    return TwELL(T, F, tile, width, cnt, col, val, spill)


def twell_unpack(tw: TwELL):
    """Dense [T][F] fp32 gate activation rebuilt from slots and spill.
    unpack(pack(z)) equals ReLU(z) (fp32) exactly."""
    h = np.zeros((tw.T, tw.n_t, tw.tile), np.float32)
    s = np.arange(tw.width)[None, None, :]
    in_slots = (s < tw.cnt[:, :, None]) & (tw.cnt <= tw.width)[:, :, None]
    t_i, k_i, s_i = np.nonzero(in_slots)
    h[t_i, k_i, tw.col[t_i, k_i, s_i]] = tw.val[t_i, k_i, s_i]
    for (t, k), sl in tw.spill.items():
        h[t, k] = sl
    return h.reshape(tw.T, tw.F)


def twell_entries(tw: TwELL, t):
    """(global column, fp32 value) of every stored active entry of row t, in
    ascending column order, taken from slots or the spill slice (a spill
    slice entry is active iff its value is > 0)."""
    out = []
    for k in range(tw.n_t):
        c = int(tw.cnt[t, k])
        base = k * tw.tile
        if c > tw.width:
            sl = tw.spill[(t, k)]
            for j in range(tw.tile):
                if sl[j] > 0:
                    out.append((base + j, float(sl[j])))
        else:
            for s in range(c):
                out.append((base + int(tw.col[t, k, s]), float(tw.val[t, k, s])))
    return out


def ffn_forward_twell(x, tw: TwELL, Wu_t, Wd, rows=None):
    """Fused up+down projection driven by a TwELL gate (paper section
    2.B.2): for each row t and each stored nonzero (j, h):
    u = x_t . W_u[:, j]; y_t += (h u) W_d[j, :].  fp64 arithmetic on the
    stored fp32 h values.  Returns y for ``rows`` (default all)."""
    X = bf16_to_f64(x)
    U = bf16_to_f64(Wu_t)
    Dn = bf16_to_f64(Wd)
    rows = range(tw.T) if rows is None else rows
    rows = list(rows)
    y = np.zeros((len(rows), Dn.shape[1]))
    for i, t in enumerate(rows):
        ent = twell_entries(tw, t)
        if not ent:
            continue
        js = np.array([e[0] for e in ent])
        hs = np.array([e[1] for e in ent], np.float64)
        u = U[js] @ X[t]
        y[i] = (hs * u) @ Dn[js]
    return y


# ---------------------------------------------------------------------------
# Hybrid training format (paper section 2.B.3)
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Hybrid:
    """ELL rows (no tile count above capacity C) and dense overflow rows.

    ell_rows   ascending token indices of the ELL part
    dense_rows ascending token indices of the dense backup
    row_map    [T]: i >= 0 -> ELL row i; i < 0 -> dense row -(i+1)
    ell_cnt    [n_ell][n_t], ell_col / ell_val [n_ell][n_t][C] (fp32 values)
    dense_h    [n_dense][F] fp32 ReLU(z)
    """
    T: int
    F: int
    tile: int
    cap: int
    ell_rows: np.ndarray
    dense_rows: np.ndarray
    row_map: np.ndarray
    ell_cnt: np.ndarray
    ell_col: np.ndarray
    ell_val: np.ndarray
    dense_h: np.ndarray


def to_hybrid(tw: TwELL, cap):
    """TwELL -> hybrid.  A row overflows iff some tile count exceeds the
    capacity C (a count equal to C stays in ELL).  ELL rows keep their
    entries, ascending, in C slots per tile; overflow rows get their whole
    dense gate row; both lists are in ascending token order."""
    over = (tw.cnt > cap).any(axis=1)
    ell_rows = np.nonzero(~over)[0]
    dense_rows = np.nonzero(over)[0]
    row_map = np.zeros(tw.T, np.int64)
    row_map[ell_rows] = np.arange(len(ell_rows))
    row_map[dense_rows] = -(np.arange(len(dense_rows)) + 1)
    n_t = tw.n_t
    ell_cnt = tw.cnt[ell_rows].copy()
    ell_col = np.zeros((len(ell_rows), n_t, cap), np.int64)
    ell_val = np.zeros((len(ell_rows), n_t, cap), np.float32)
    # entries held in the TwELL slots (count <= W) ...
    m = min(cap, tw.width)
    s = np.arange(m)[None, None, :]
    keep = (s < ell_cnt[:, :, None]) & (ell_cnt <= tw.width)[:, :, None]
    ell_col[:, :, :m] = np.where(keep, tw.col[ell_rows][:, :, :m], 0)
    ell_val[:, :, :m] = np.where(keep, tw.val[ell_rows][:, :, :m], 0)
    # ... and those held in a spill slice (W < count <= C, only when C > W)
    for i, t in enumerate(ell_rows):
        for k in np.nonzero(ell_cnt[i] > tw.width)[0]:
            sl = tw.spill[(int(t), int(k))]
            js = np.nonzero(sl > 0)[0]
            ell_col[i, k, :len(js)] = js
            ell_val[i, k, :len(js)] = sl[js]
    full = twell_unpack(tw)
    dense_h = full[dense_rows]
    return Hybrid(tw.T, tw.F, tw.tile, cap, ell_rows, dense_rows, row_map, ell_cnt,
                  ell_col, ell_val, dense_h)


# ---------------------------------------------------------------------------
# Training step gradients (paper section 2.B.3 forward/backward; L1 term from
# the news article recipe list and paper section 4)
# ---------------------------------------------------------------------------


def ffn_backward_f64(X, G, U, Dn, dY, l1_coeff, active=None):
    """Gradients of L = sum(y * dy) + l1_coeff * sum(h) for the gated FFN
    y = (h * u) W_d, h = ReLU(z), z = x W_g, u = x W_u, on fp64 arrays.

    With a = h * u:  da = dy W_d^T;  du = da * h;  dh = da * u + lambda;
    dz = dh where active else 0;  dx = dz W_g^T + du W_u^T;
    dW_g = x^T dz;  dW_u = x^T du;  dW_d = a^T dy.

    ``G``, ``U`` are W_g^T, W_u^T and ``Dn`` is W_d, all [F][D]; the weight
    gradients come back in the same neuron-major layout.  ``active``
    optionally overrides z > 0 (a boolean [T][F] decision taken in another
    precision).  Returns dx [T][D], dWg_t, dWu_t, dWd [F][D].
    """
    z = X @ G.T
    act = (z > 0) if active is None else active
    h = np.where(act, z, 0.0)
    u = X @ U.T
    a = h * u
    da = dY @ Dn.T
    du = da * h
    dz = np.where(act, da * u + l1_coeff, 0.0)
    return dz @ G + du @ U, dz.T @ X, du.T @ X, a.T @ dY


def ffn_backward(x, Wg_t, Wu_t, Wd, dy, l1_coeff, active=None):
    """``ffn_backward_f64`` on bf16 inputs (``dy`` fp32 or fp64)."""
    return ffn_backward_f64(bf16_to_f64(x), bf16_to_f64(Wg_t), bf16_to_f64(Wu_t),
                            bf16_to_f64(Wd), np.asarray(dy, dtype=np.float64), l1_coeff,
                            active)


def ffn_backward_dx_rows(x, Wg_t, Wu_t, Wd, dy, l1_coeff, rows, active_rows=None):
    """dx for the token rows ``rows`` only: dx_t depends on token t alone, so
    this is the dense definition applied to those rows."""
    rows = np.asarray(rows)
    return ffn_backward_f64(bf16_to_f64(np.asarray(x)[rows]), bf16_to_f64(Wg_t),
                            bf16_to_f64(Wu_t), bf16_to_f64(Wd),
                            np.asarray(dy, dtype=np.float64)[rows], l1_coeff, active_rows)[0]


def ffn_backward_dw_cols(x, Wg_t, Wu_t, Wd, dy, l1_coeff, neurons, active_cols=None):
    """Rows ``neurons`` of dWg_t, dWu_t and dWd: the gradients of neuron j
    depend on that neuron's weights alone, so this is the dense definition
    applied to the FFN restricted to those neurons."""
    n = np.asarray(neurons)
    _, dg, du, dd = ffn_backward_f64(bf16_to_f64(x), bf16_to_f64(np.asarray(Wg_t)[n]),
                                     bf16_to_f64(np.asarray(Wu_t)[n]),
                                     bf16_to_f64(np.asarray(Wd)[n]),
                                     np.asarray(dy, dtype=np.float64), l1_coeff, active_cols)
    return dg, du, dd


def training_loss(X, G, U, Dn, dY, l1_coeff):
    """The scalar L = sum(y * dy) + l1_coeff * sum(ReLU(z)) on fp64 arrays,
    whose gradients ``ffn_backward_f64`` returns (finite-difference pin)."""
    y = ffn_forward_f64(X, G, U, Dn)
    z = X @ G.T
    return float(np.sum(y * dY) + l1_coeff * np.sum(np.where(z > 0, z, 0.0)))


def stack_forward_backward(x, layers, dy, l1_coeff, bias_feature=True, round_inputs=True,
                           inputs=None, actives=None):
    """A residual stack of gated FFN layers, x_{l+1} = x_l + y_l with
    y_l = FFN_l(a_l), and the gradients of
    L = sum(x_L * dy) + l1_coeff * sum_l sum(h_l).

    ``x`` bf16 bits [T][D]; ``layers`` a list of (Wg_t, Wu_t, Wd) bf16 bits.
    The stream x_l is kept in fp64; each layer's input a_l is x_l rounded to
    bf16 (``round_inputs``), or the bf16 bits ``inputs[l]`` when given; with
    ``bias_feature`` the last feature of y_l is dropped (feature D - 1 stays
    the constant gate-threshold input).  ``actives`` (boolean [T][F] per
    layer) optionally replaces the z > 0 decisions, so a ReLU kink that two
    computations straddle does not make their gradients differ by O(1).
    The backward treats the rounding of a_l as the identity and chains the
    single-layer gradients of ``ffn_backward_f64`` in reverse order:
    dL/dx_l = dL/dx_{l+1} + dx(layer l, dy = dL/dx_{l+1} without the bias
    feature).  Returns (x_L [T][D] fp64, dL/dx_0, [(dWg_t, dWu_t, dWd)])."""
    X = bf16_to_f64(x)
    ws = [tuple(bf16_to_f64(w) for w in layer) for layer in layers]
    As = []
    for i, (G, U, Dn) in enumerate(ws):
        if inputs is not None:
            A = bf16_to_f64(inputs[i])
        elif round_inputs:
            A = bf16_to_f64(f32_to_bf16(X.astype(np.float32)))
        else:
            A = X
        As.append(A)
        y = ffn_forward_f64(A, G, U, Dn, None if actives is None else actives[i])
        if bias_feature:
            y[:, -1] = 0.0
        X = X + y
    g = np.asarray(dy, dtype=np.float64).copy()
    grads = [None] * len(ws)
    for i in range(len(ws) - 1, -1, -1):
        G, U, Dn = ws[i]
        dyl = g.copy()
        if bias_feature:
            dyl[:, -1] = 0.0
        dx, dg, du, dd = ffn_backward_f64(As[i], G, U, Dn, dyl, l1_coeff,
                                          None if actives is None else actives[i])
        grads[i] = (dg, du, dd)
        g = g + dx
    return X, g, grads
