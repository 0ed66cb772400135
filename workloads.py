"""Seeded synthetic inputs for the activation-sparse gated FFN (TwELL) workloads.

This module is the only code shared by the CPU oracle (``oracle/``) and the
GPU path's tests and benchmark.  It draws random numbers and builds the
per-config sparsity construction; it holds none of the method's arithmetic
(no gate product, no ReLU, no packing).

The pages ("Sparser, Faster, Lighter Transformer Language Models", section 4)
measure trained 0.5B-2B Transformer++ models on FineWeb.  Neither the dataset
nor the weights exist here, so these inputs stand in for them: they take the
layer shapes of those model classes and set the gate density through a
constant "bias" input feature whose gate weight is a negative threshold.

Recipe (all configs):
  * ``rng = numpy.random.default_rng(seed)`` (PCG64), values drawn in fp64
    and rounded to bf16 (round-to-nearest-even through fp32).
  * Draw order: Wg_t, Wu_t, Wd, then x, then the per-config extras, then dy.
    Drawing the weights first keeps them identical across the decode sweep,
    and x is prefix-nested across T.
  * Storage is neuron-major: ``Wg_t = W_g^T``, ``Wu_t = W_u^T`` (both
    [F][D]) and ``Wd = W_d`` ([F][D]); x is [T][D].
  * Wg_t, Wu_t ~ N(0, 1/D); Wd ~ N(0, 1/F); x ~ N(0, 1).
  * Feature D-1 of x is the bias feature.  The gate pre-activation without
    it has variance sigma^2 = (D-1)/D, so a threshold tau gives
    P(z > 0) = 1 - Phi(tau / sigma).

bf16 tensors are returned as ``numpy.uint16`` bit patterns.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

TILE = 128

# ---------------------------------------------------------------------------
# bf16 helpers for input construction only (the oracle has its own).
# ---------------------------------------------------------------------------


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE) bit patterns as uint16."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _norm_ppf(q: float) -> float:
    from scipy.special import ndtri

    return float(ndtri(q))


def _norm_sf(x):
    from scipy.special import ndtr

    return 1.0 - ndtr(x)


def threshold_for_density(p: float, d_model: int) -> float:
    """tau with P(N(0, (D-1)/D) > tau) = p."""
    sigma = math.sqrt((d_model - 1) / d_model)
    return _norm_ppf(1.0 - p) * sigma


def lognormal_offset_base(mean_density: float, d_model: int, s: float = 0.5) -> float:
    """t0 such that E_o[P(z > t0 + o)] = mean_density, o ~ LogNormal(0, s).

    Solved by bisection on a fixed Gauss-Hermite quadrature, so the value is
    reproducible on any host.
    """
    sigma = math.sqrt((d_model - 1) / d_model)
    nodes, weights = np.polynomial.hermite_e.hermegauss(200)
    weights = weights / weights.sum()
    offs = np.exp(s * nodes)

    def mean_p(t0):
        return float(np.sum(weights * _norm_sf((t0 + offs) / sigma)))

    lo, hi = -10.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mean_p(mid) > mean_density:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Workload:
    name: str
    T: int
    D: int
    F: int
    width: int                 # TwELL slots per (row, tile)
    x: np.ndarray              # [T][D] bf16 bits
    Wg_t: np.ndarray           # [F][D] bf16 bits
    Wu_t: np.ndarray           # [F][D] bf16 bits
    Wd: np.ndarray             # [F][D] bf16 bits
    dy: np.ndarray | None = None   # [T][D] fp32 (training configs)
    cap: int | None = None         # hybrid ELL capacity (training configs)
    l1_coeff: float = 0.0
    tile: int = TILE
    note: str = ""

    @property
    def n_t(self) -> int:
        return self.F // self.tile


_WEIGHT_CACHE: dict = {}


def _weights(rng, D, F, seed=None):
    """Draw Wg_t, Wu_t, Wd (first draws of a fresh generator).  With ``seed``
    given, the draw and the generator state after it are cached per
    (seed, D, F), so repeated configs in one process skip the draw."""
    key = (seed, D, F)
    if seed is not None and key in _WEIGHT_CACHE:
        w, state = _WEIGHT_CACHE[key]
        rng.bit_generator.state = state
        return tuple(a.copy() for a in w)
    Wg_t = _to_bf16_bits(rng.standard_normal((F, D)) / math.sqrt(D))
    Wu_t = _to_bf16_bits(rng.standard_normal((F, D)) / math.sqrt(D))
    Wd = _to_bf16_bits(rng.standard_normal((F, D)) / math.sqrt(F))
    if seed is not None:
        _WEIGHT_CACHE.clear()
        _WEIGHT_CACHE[key] = ((Wg_t, Wu_t, Wd), rng.bit_generator.state)
        return Wg_t.copy(), Wu_t.copy(), Wd.copy()
    return Wg_t, Wu_t, Wd


def make_uniform(name, T, D, F, density, width, seed=0, weights=None):
    """Uniform gate density through the bias feature (x[:, D-1] = 1,
    Wg_t[:, D-1] = -tau)."""
    rng = np.random.default_rng(seed)
    Wg_t, Wu_t, Wd = _weights(rng, D, F, seed) if weights is None else weights
    Wg_t = Wg_t.copy()
    tau = threshold_for_density(density, D)
    Wg_t[:, D - 1] = _to_bf16_bits(np.array([-tau]))[0]
    x = rng.standard_normal((T, D))
    x[:, D - 1] = 1.0
    return Workload(name, T, D, F, width, _to_bf16_bits(x), Wg_t, Wu_t, Wd,
                    note=f"uniform density {density}, tau={tau:.5f}")


def make_heavy_tail(name, T, D, F, mean_density, width, seed=0, s=0.5):
    """Per-token threshold tau_t = t0 + o_t, o_t ~ LogNormal(0, s) (additive
    offset), t0 solved so the mean density is ``mean_density``."""
    rng = np.random.default_rng(seed)
    Wg_t, Wu_t, Wd = _weights(rng, D, F, seed)
    Wg_t[:, D - 1] = _to_bf16_bits(np.array([-1.0]))[0]
    x = rng.standard_normal((T, D))
    t0 = lognormal_offset_base(mean_density, D, s)
    o = rng.lognormal(0.0, s, size=T)
    x[:, D - 1] = t0 + o
    return Workload(name, T, D, F, width, _to_bf16_bits(x), Wg_t, Wu_t, Wd,
                    note=f"heavy-tailed per-token threshold t0={t0:.4f} + LogNormal(0,{s})")


def make_training(name, T, D, F, mean_density, dense_frac, dense_density, cap,
                  l1_coeff=2e-5, seed=0):
    """Training workload: a fraction ``dense_frac`` of rows (chosen at random)
    gets density ``dense_density``, far above the ELL capacity; the other rows
    get the base density that makes the overall mean ``mean_density``."""
    rng = np.random.default_rng(seed)
    Wg_t, Wu_t, Wd = _weights(rng, D, F, seed)
    Wg_t[:, D - 1] = _to_bf16_bits(np.array([-1.0]))[0]
    x = rng.standard_normal((T, D))
    n_dense = int(round(dense_frac * T))
    dense_rows = rng.choice(T, n_dense, replace=False) if n_dense else np.zeros(0, np.int64)
    p_base = (mean_density * T - dense_density * n_dense) / (T - n_dense)
    if not 0.0 < p_base < 1.0:
        raise ValueError(f"no base density gives mean {mean_density} (base {p_base})")
    tau_b = threshold_for_density(p_base, D)
    tau_d = threshold_for_density(dense_density, D)
    x[:, D - 1] = tau_b
    x[dense_rows, D - 1] = tau_d
    dy = rng.standard_normal((T, D)).astype(np.float32)
    return Workload(name, T, D, F, cap, _to_bf16_bits(x), Wg_t, Wu_t, Wd, dy=dy,
                    cap=cap, l1_coeff=l1_coeff,
                    note=(f"{n_dense} rows at density {dense_density} (tau={tau_d:.4f}), "
                          f"others at {p_base:.5f} (tau={tau_b:.4f})"))


DECODE_T = (1, 4, 16, 64, 256)


def config(idx: int, seed: int = 0, T: int | None = None) -> Workload:
    """The five workloads.  ``T`` overrides the token count (a prefix of the
    same draw for configs whose x is drawn after the weights)."""
    if idx == 0:
        return make_uniform("gated-MLP T=64 D=256 F=1024 5% W=16", T or 64, 256, 1024,
                            0.05, 16, seed)
    if idx == 1:
        return make_uniform("0.5B-class T=8192 D=1536 F=6144 1% W=8", T or 8192, 1536, 6144,
                            0.01, 8, seed)
    if idx == 2:
        return make_heavy_tail("1.5B-class T=16384 D=2048 F=8192 mean 1% heavy-tail W=16",
                               T or 16384, 2048, 8192, 0.01, 16, seed)
    if idx == 3:
        return make_training("2B-class training T=16384 D=2304 F=9216 5% (3% rows dense) C=32",
                             T or 16384, 2304, 9216, 0.05, 0.03, 0.40, 32, 2e-5, seed)
    if idx == 4:
        return make_uniform(f"decode T={T or 1} D=2048 F=8192 0.5% W=8", T or 1, 2048, 8192,
                            0.005, 8, seed)
    raise ValueError(idx)


def random_small(T, D, F, density, width, seed=0, dy=False, cap=None, l1_coeff=0.0):
    """Small uniform-density case for parity tests (any T, D, F)."""
    w = make_uniform(f"small T={T} D={D} F={F} p={density} W={width}", T, D, F, density,
                     width, seed)
    if dy:
        rng = np.random.default_rng(seed + 1000)
        w.dy = rng.standard_normal((T, D)).astype(np.float32)
        w.cap = cap if cap is not None else width
        w.l1_coeff = l1_coeff
    return w


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (for building fixtures; exact)."""
    return _bf16_bits_to_f64(b)


def to_bf16(a: np.ndarray) -> np.ndarray:
    """Round values to bf16 bit patterns (for building fixtures)."""
    return _to_bf16_bits(a)
